"""Seeded input generators: determinism, prefix property, moments, rounding."""
import numpy as np
import pytest

import synth


def test_deterministic_and_prefix():
    a = synth.normal(5, 0, (1000,))
    b = synth.normal(5, 0, (1000,))
    assert np.array_equal(a, b)
    assert not np.array_equal(a, synth.normal(6, 0, (1000,)))
    assert not np.array_equal(a, synth.normal(5, 1, (1000,)))
    u = synth.uniform01(9, 2, 5000)
    assert np.array_equal(u[:100], synth.uniform01(9, 2, 100))


def test_splitmix64_reference_value():
    # splitmix64's published test vector: seeding the state with 0 and taking
    # one step yields 0xE220A8397B1DCDAF.
    z = synth._mix(np.array([0x9E3779B97F4A7C15], dtype=np.uint64))[0]
    assert int(z) == 0xE220A8397B1DCDAF


def test_moments():
    z = synth.normal(1, 0, (200000,))
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01
    u = synth.uniform(1, 1, (200000,), -1, 1)
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 0.01
    k = synth.small_ints(3, 0, (10000,))
    assert set(np.unique(k).tolist()) == set(range(-3, 4))


def test_rounding_matches_torch():
    import torch
    v = synth.normal(2, 0, (4096,)) * 3
    s16, e16 = synth.round_to(v, "f16")
    assert np.array_equal(s16.view(np.uint16),
                          torch.from_numpy(v.astype(np.float32)).half().numpy().view(np.uint16))
    assert np.array_equal(e16, s16.astype(np.float64))
    sb, eb = synth.round_to(v, "bf16")
    assert sb.dtype == torch.bfloat16
    assert np.array_equal(eb, torch.from_numpy(v.astype(np.float32)).bfloat16().double().numpy())


def test_workloads_table():
    w = synth.WORKLOADS
    assert w["tiny"].out_hw() == (32, 32)
    assert w["stem"].out_hw() == (112, 112)
    assert w["vgg"].flops() == 2 * 64 * 512 * 28 * 28 * 512 * 9
    assert w["sweep_k3_s2"].out_hw() == (32, 32)
    assert w["sweep_k11"].pad == 5
    # Table I of the im2win paper: output sizes of the twelve layers (p = 0).
    outs = {1: 55, 2: 56, 3: 111, 4: 109, 5: 20, 6: 10, 7: 222, 8: 110, 9: 54, 10: 26, 11: 12, 12: 5}
    for i, o in outs.items():
        assert w[f"cv{i}"].out_hw() == (o, o), i
        assert w[f"cv{i}"].N == 256
    d = synth.make_inputs(w["tiny"], "f32")
    assert d["X"].shape == (1, 16, 32, 32) and d["X"].dtype == np.float32
    small = synth.make_inputs(w["resnet_stage1"], "f16", N=2)
    assert small["X"].shape[0] == 2


@pytest.mark.parametrize("name", ["resnet_stage1", "stem"])
def test_batch_prefix_consistency(name):
    wl = synth.WORKLOADS[name]
    a = synth.make_inputs(wl, "f32", N=1)
    b = synth.make_inputs(wl, "f32", N=2)
    assert np.array_equal(a["X"][0], b["X"][0])
