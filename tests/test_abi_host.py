"""Host-side checks of the C ABI: the library loads without a GPU, exports
every function ``include/conv2d.h`` declares, and its descriptor, workspace
and argument checks behave as documented.  No kernel is launched here."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def capi():
    from dense_convolution_gb300 import build, capi
    build.build()
    capi.load()
    return capi


def _declared():
    src = open(os.path.join(ROOT, "include", "conv2d.h")).read()
    return sorted(set(re.findall(r"\b(conv2d_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(capi):
    import ctypes
    names = _declared()
    assert len(names) == len(capi.EXPORTED)
    assert set(names) == set(capi.EXPORTED)
    L = ctypes.CDLL(capi.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(capi):
    for s in range(8):
        assert capi.conv2d_status_string(s)
    assert capi.conv2d_status_string(99) == "unknown status"


@pytest.mark.parametrize("args", [
    (0, 3, 8, 8, 4, 3, 3, 1, 1), (1, 0, 8, 8, 4, 3, 3, 1, 1), (1, 3, 8, 8, 4, 3, 3, 0, 1),
    (1, 3, 8, 8, 4, 3, 3, 1, -1), (1, 3, 2, 2, 4, 5, 5, 1, 0), (1, 3, 8, 8, 4, 0, 3, 1, 0),
])
def test_bad_geometry(capi, args):
    with pytest.raises(capi.Conv2dError) as e:
        capi.conv2d_desc_create(*args, "f32", "auto")
    assert e.value.status == capi.ERR_BAD_PARAM


def test_dtype_algo_mismatch(capi):
    with pytest.raises(capi.Conv2dError) as e:
        capi.conv2d_desc_create(1, 8, 8, 8, 8, 3, 3, 1, 1, "f16", "im2win_fp32_cc")
    assert e.value.status == capi.ERR_BAD_PARAM
    with pytest.raises(capi.Conv2dError) as e:
        capi.conv2d_desc_create(1, 8, 8, 8, 8, 3, 3, 1, 1, "f32", "implicit_tc")
    assert e.value.status == capi.ERR_BAD_PARAM
    with pytest.raises(capi.Conv2dError) as e:
        capi.conv2d_desc_create(1, 8, 8, 8, 8, 3, 3, 1, 1, 7, "auto")
    assert e.value.status == capi.ERR_BAD_PARAM


def test_out_dims_floor_rule(capi):
    d = capi.conv2d_desc_create(2, 64, 224, 224, 64, 7, 7, 2, 0, "f32", "auto")
    try:
        assert capi.conv2d_out_dims(d) == (109, 109)     # Table I, cv4
    finally:
        capi.conv2d_desc_destroy(d)


def test_auto_choices_and_workspace(capi):
    cases = {
        # name: (shape, dtype, expected algo)
        "resnet_f16": ((32, 64, 56, 56, 64, 3, 3, 1, 1), "f16", "padded_tc"),
        "k1_f16": ((16, 128, 64, 64, 128, 1, 1, 1, 0), "f16", "implicit_tc"),
        "k3s2_f16": ((16, 128, 64, 64, 128, 3, 3, 2, 1), "f16", "implicit_tc"),
        "k3_f16": ((16, 128, 64, 64, 128, 3, 3, 1, 1), "f16", "padded_tc"),
        "k5_f16": ((16, 128, 64, 64, 128, 5, 5, 1, 2), "f16", "implicit_tc"),
        "stem_f16": ((32, 3, 224, 224, 64, 7, 7, 2, 3), "f16", "im2win_tc"),
        "vgg_bf16": ((64, 512, 28, 28, 512, 3, 3, 1, 1), "bf16", "implicit_tc"),
        "resnet_f32": ((32, 64, 56, 56, 64, 3, 3, 1, 1), "f32", "im2win_fp32_cc"),
    }
    for name, (shape, dt, algo) in cases.items():
        d = capi.conv2d_desc_create(*shape, dt, "auto")
        try:
            assert capi.conv2d_get_algo(d) == algo, name
            N, Ci, H, W, Co, Kh, Kw, s, p = shape
            Ho = (H + 2 * p - Kh) // s + 1
            ws = capi.conv2d_workspace_size(d)
            elem = 4 if dt == "f32" else 2
            im2win_tensor = N * Ci * Ho * (W + 2 * p) * Kh * elem
            if Kh == Kw == 1 and s == 1 and p == 0 and Ci % 8 == 0 and (H * W) % 8 == 0 and dt != "f32":
                # 1x1 layer: one GEMM on the caller's tensors, no workspace, one launch.
                assert ws == 0, name
                assert capi.conv2d_launches_per_call(d) == 1
                continue
            assert ws > 0
            if algo == "padded_tc":
                ci8 = (Ci + 7) // 8 * 8
                wq = (W + 2 * p + 3) // 4 * 4
                assert ws >= N * (H + 2 * p) * wq * ci8 * 2    # zero-padded channels-last copy of X
            if algo == "implicit_tc":
                ci8 = (Ci + 7) // 8 * 8
                assert ws >= N * H * W * ci8 * 2          # channels-last copy of X
                # The copy never exceeds the im2win tensor (equal for 1x1 layers);
                # the repacked filter comes on top.
                packed = Co * Kh * Kw * ((ci8 + 63) // 64 * 64) * 2
                assert ws <= im2win_tensor + packed + 1024
        finally:
            capi.conv2d_desc_destroy(d)


def test_nhwc_layout_drops_input_copy(capi):
    d = capi.conv2d_desc_create(8, 64, 28, 28, 64, 3, 3, 1, 1, "f16", "implicit_tc")
    try:
        nchw = capi.conv2d_workspace_size(d)
        capi.conv2d_desc_set_input_layout(d, "nhwc")
        nhwc = capi.conv2d_workspace_size(d)
        assert nhwc == 64 * 9 * 64 * 2                   # packed filter only
        assert nchw > nhwc
        with pytest.raises(capi.Conv2dError):
            capi.conv2d_desc_set_input_layout(d, 5)
    finally:
        capi.conv2d_desc_destroy(d)
    d = capi.conv2d_desc_create(8, 64, 28, 28, 64, 3, 3, 1, 1, "f32", "auto")
    try:
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_input_layout(d, "nhwc")
        assert e.value.status == capi.ERR_UNSUPPORTED
    finally:
        capi.conv2d_desc_destroy(d)


def test_fwd_argument_checks_before_launch(capi):
    # These return before any CUDA call, so fake addresses are safe here.
    d = capi.conv2d_desc_create(1, 8, 16, 16, 8, 3, 3, 1, 1, "f32", "im2win_fp32_cc")
    try:
        ws = capi.conv2d_workspace_size(d)
        A = 1 << 20
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_fwd(d, 0, A, A, A, ws)
        assert e.value.status == capi.ERR_NULL_PTR
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_fwd(d, A + 4, A, A, A, ws)
        assert e.value.status == capi.ERR_MISALIGNED
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_fwd(d, A, A, A, A, ws - 1)
        assert e.value.status == capi.ERR_WORKSPACE_TOO_SMALL
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_fwd(d, A, A, A, 0, ws)
        assert e.value.status == capi.ERR_NULL_PTR
    finally:
        capi.conv2d_desc_destroy(d)


def test_padded_algo_limits(capi):
    # Stride-1 only; NCHW input only.
    with pytest.raises(capi.Conv2dError) as e:
        capi.conv2d_desc_create(2, 64, 16, 16, 64, 3, 3, 2, 1, "f16", "padded_tc")
    assert e.value.status == capi.ERR_UNSUPPORTED
    d = capi.conv2d_desc_create(2, 64, 16, 16, 64, 3, 3, 1, 1, "f16", "padded_tc")
    try:
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_input_layout(d, "nhwc")
        assert e.value.status == capi.ERR_UNSUPPORTED
        assert capi.conv2d_launches_per_call(d) == 3
    finally:
        capi.conv2d_desc_destroy(d)


def test_destroy_null_is_ok(capi):
    capi.conv2d_desc_destroy(0)


@pytest.mark.parametrize("shape,dtype,gemm", [
    ((16, 128, 64, 64, 128, 1, 1, 1, 0), "f16", True),     # the 1x1 sweep layer
    ((2, 72, 10, 12, 17, 1, 1, 1, 0), "bf16", True),      # Ci, H*W multiples of 8, any Co
    ((2, 12, 10, 12, 17, 1, 1, 1, 0), "f16", False),      # Ci % 8 != 0: the TMA row pitch
    ((2, 64, 5, 5, 64, 1, 1, 1, 0), "f16", False),        # H*W % 8 != 0
    ((2, 64, 8, 8, 64, 1, 1, 2, 0), "f16", False),        # stride 2
    ((2, 64, 8, 8, 64, 1, 1, 1, 1), "f16", False),        # padded 1x1
])
def test_one_by_one_gemm_selection(capi, shape, dtype, gemm):
    d = capi.conv2d_desc_create(*shape, dtype, "implicit_tc")
    try:
        ws = capi.conv2d_workspace_size(d)
        n = capi.conv2d_launches_per_call(d)
        if gemm:
            assert ws == 0 and n == 1
        else:
            assert ws > 0 and n == 3
        # An NHWC input (Ci % 8 == 0 only) never takes the in-place GEMM, which
        # reads X as [ci][pixels]: filter repack + implicit contraction.
        if shape[1] % 8 == 0:
            capi.conv2d_desc_set_input_layout(d, "nhwc")
            assert capi.conv2d_launches_per_call(d) == 2
    finally:
        capi.conv2d_desc_destroy(d)


def test_fwd_host_argument_checks_before_copy(capi):
    # These return before any copy or launch, so fake addresses are safe here.
    d = capi.conv2d_desc_create(1, 8, 16, 16, 8, 3, 3, 1, 1, "f16", "implicit_tc")
    try:
        ws = capi.conv2d_workspace_size(d)
        A = 1 << 20
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_fwd_host(d, 0, A, A, A, A, A, A, ws)
        assert e.value.status == capi.ERR_NULL_PTR
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_fwd_host(d, A, A, A, A, A, 0, A, ws)
        assert e.value.status == capi.ERR_NULL_PTR
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_fwd_host(d, A, A, A, A + 8, A, A, A, ws)
        assert e.value.status == capi.ERR_MISALIGNED
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_fwd_host(d, A, A, A, A, A, A, A, ws - 1)
        assert e.value.status == capi.ERR_WORKSPACE_TOO_SMALL
    finally:
        capi.conv2d_desc_destroy(d)


def test_static_workspace_size_getter(capi):
    # The binding reads the size from the library, which reports the header's value.
    assert capi.conv2d_static_workspace_bytes() == 64 << 20
    assert capi.STATIC_WORKSPACE_BYTES == 64 << 20


def test_output_dtype_and_bias_setters(capi):
    d16 = capi.conv2d_desc_create(1, 8, 8, 8, 8, 3, 3, 1, 1, "f16", "auto")
    d32 = capi.conv2d_desc_create(1, 8, 8, 8, 8, 3, 3, 1, 1, "f32", "auto")
    try:
        capi.conv2d_desc_set_output_dtype(d16, "f32")      # fp32 sum of 16-bit inputs
        capi.conv2d_desc_set_output_dtype(d16, "f16")      # back to the input type
        for desc, bad in ((d16, "bf16"), (d32, "f16"), (d32, "bf16")):
            with pytest.raises(capi.Conv2dError) as e:
                capi.conv2d_desc_set_output_dtype(desc, bad)
            assert e.value.status == capi.ERR_BAD_PARAM
        capi.conv2d_desc_set_bias(d16, 0)                  # no bias
        capi.conv2d_desc_set_bias(d16, 0x10002)            # 2-byte aligned is enough for 16-bit values
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_bias(d16, 0x10001)
        assert e.value.status == capi.ERR_MISALIGNED
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_bias(d32, 0x10002)
        assert e.value.status == capi.ERR_MISALIGNED
        capi.conv2d_desc_set_bias(d16, 0)
    finally:
        capi.conv2d_desc_destroy(d16)
        capi.conv2d_desc_destroy(d32)


@pytest.mark.parametrize("shape,dtype", [((32, 64, 56, 56, 64, 3, 3, 1, 1), "f16"),
                                         ((64, 512, 28, 28, 512, 3, 3, 1, 1), "bf16"),
                                         ((1, 13, 11, 13, 17, 3, 5, 1, 2), "f16"),
                                         ((2, 64, 16, 16, 130, 1, 1, 1, 0), "f16")])
def test_implicit_nchw_needs_only_the_packed_filter(capi, shape, dtype):
    """The implicit GEMM that reads NCHW X in the contraction kernel: workspace =
    the repacked filter, two launches; stride > 1, NHWC input and fp32 are refused."""
    N, Ci, H, W, Co, Kh, Kw, s, p = shape
    d = capi.conv2d_desc_create(*shape, dtype, "implicit_nchw_tc")
    try:
        ci8 = (Ci + 7) // 8 * 8
        assert capi.conv2d_workspace_size(d) == Co * Kh * Kw * ((ci8 + 63) // 64 * 64) * 2
        assert capi.conv2d_launches_per_call(d) == 2
        assert capi.conv2d_get_algo(d) == "implicit_nchw_tc"
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_input_layout(d, "nhwc")
        assert e.value.status == capi.ERR_UNSUPPORTED
    finally:
        capi.conv2d_desc_destroy(d)
    for bad, status in (((N, Ci, H, W, Co, Kh, Kw, 2, p), "f16"), (shape, "f32")):
        with pytest.raises(capi.Conv2dError):
            capi.conv2d_desc_create(*bad, status, "implicit_nchw_tc")


def test_tuning_knobs_ranges(capi):
    d = capi.conv2d_desc_create(1, 8, 8, 8, 8, 3, 3, 1, 1, "f16", "auto")
    try:
        for knob, good, bad in (("stages", (0, 1, 2, 8), (-1, 9)), ("sync_copies", (0, 1), (2, -1)),
                                ("raster", (0, 1, 2), (3, -1)), ("no_resident", (0, 1), (2,)),
                                ("split", (0, 1, 0), (2,)), ("epi_groups", (0, 2, 3, 0), (1, 4, -1)),
                                ("tile_n", (0, 64, 128, 176, 256, 0), (32, 192, -1))):
            for v in good:
                capi.conv2d_desc_set_tuning(d, knob, v)
            for v in bad:
                with pytest.raises(capi.Conv2dError) as e:
                    capi.conv2d_desc_set_tuning(d, knob, v)
                assert e.value.status == capi.ERR_BAD_PARAM
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_tuning(d, 7, 0)
        assert e.value.status == capi.ERR_BAD_PARAM
    finally:
        capi.conv2d_desc_destroy(d)


def test_winograd_descriptor(capi):
    """F(2x2, 3x3): 3x3 stride-1 fp32 only; workspace = transformed filter
    (16 values per (output channel rounded to 64, input channel rounded to 8))."""
    d = capi.conv2d_desc_create(2, 13, 9, 11, 70, 3, 3, 1, 1, "f32", "winograd_fp32_cc")
    try:
        assert capi.conv2d_workspace_size(d) == 128 * 16 * 16 * 4
        assert capi.conv2d_launches_per_call(d) == 2
        assert capi.conv2d_get_algo(d) == "winograd_fp32_cc"
    finally:
        capi.conv2d_desc_destroy(d)
    for shape, dt, status in (((1, 8, 9, 9, 8, 5, 5, 1, 2), "f32", capi.ERR_UNSUPPORTED),
                              ((1, 8, 9, 9, 8, 3, 3, 2, 1), "f32", capi.ERR_UNSUPPORTED),
                              ((1, 8, 9, 9, 8, 3, 3, 1, 1), "f16", capi.ERR_BAD_PARAM)):
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_create(*shape, dt, "winograd_fp32_cc")
        assert e.value.status == status


@pytest.mark.parametrize("shape,dtype,algo", [((32, 64, 56, 56, 64, 3, 3, 1, 1), "f16", "padded_tc"),
                                              ((64, 512, 28, 28, 512, 3, 3, 1, 1), "f16", "implicit_tc"),
                                              ((16, 128, 64, 64, 128, 1, 1, 1, 0), "f16", "implicit_tc"),
                                              ((32, 64, 56, 56, 64, 3, 3, 1, 1), "f32", "im2win_fp32_cc"),
                                              ((32, 64, 56, 56, 64, 3, 3, 1, 1), "f32", "winograd_fp32_cc"),
                                              ((32, 64, 56, 56, 64, 3, 3, 1, 1), "f16", "implicit_nchw_tc")])
def test_prepacked_filter_workspace_and_launches(capi, shape, dtype, algo):
    """Pre-packing moves the packed filter out of the workspace and drops the
    repack launch (the 1x1 GEMM has neither)."""
    d = capi.conv2d_desc_create(*shape, dtype, algo)
    try:
        ws0, n0 = capi.conv2d_workspace_size(d), capi.conv2d_launches_per_call(d)
        packed = capi.conv2d_packed_filter_bytes(d)
        assert packed > 0
        capi.conv2d_desc_set_filter_prepacked(d, True)
        ws1, n1 = capi.conv2d_workspace_size(d), capi.conv2d_launches_per_call(d)
        if n0 == 1:     # 1x1 GEMM: the filter is read as given, nothing to drop
            assert (ws1, n1) == (ws0, n0) == (0, 1)
        else:
            assert n1 == n0 - 1 and ws1 <= ws0 - packed
        capi.conv2d_desc_set_filter_prepacked(d, False)
        assert capi.conv2d_workspace_size(d) == ws0
        assert capi.load().conv2d_desc_set_filter_prepacked(d, 2) == capi.ERR_BAD_PARAM
    finally:
        capi.conv2d_desc_destroy(d)


def test_split_tail_workspace(capi):
    """The opt-in split tail reserves its partial sums at the end of the
    workspace; switching it off gives the space back."""
    d = capi.conv2d_desc_create(64, 512, 28, 28, 512, 3, 3, 1, 1, "f16", "implicit_tc")
    try:
        without = capi.conv2d_workspace_size(d)
        assert without == 64 * 28 * 28 * 512 * 2 + 512 * 9 * 512 * 2
        capi.conv2d_desc_set_tuning(d, "split", 1)
        with_split = capi.conv2d_workspace_size(d)
        assert with_split > without
        capi.conv2d_desc_set_tuning(d, "split", 0)
        assert capi.conv2d_workspace_size(d) == without
    finally:
        capi.conv2d_desc_destroy(d)


def test_tile_width_knob_limits(capi):
    """176-wide tiles exist on the implicit, padded and im2win sources only
    and not with the split tail; the workspace does not depend on the width."""
    d = capi.conv2d_desc_create(4, 64, 28, 28, 512, 3, 3, 1, 1, "f16", "implicit_tc")
    try:
        ws = capi.conv2d_workspace_size(d)
        for v in (64, 128, 176, 256, 0):
            capi.conv2d_desc_set_tuning(d, "tile_n", v)
            assert capi.conv2d_workspace_size(d) == ws
        capi.conv2d_desc_set_tuning(d, "tile_n", 176)
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_tuning(d, "split", 1)
        assert e.value.status == capi.ERR_UNSUPPORTED
        capi.conv2d_desc_set_tuning(d, "tile_n", 0)
        capi.conv2d_desc_set_tuning(d, "split", 1)
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_tuning(d, "tile_n", 176)
        assert e.value.status == capi.ERR_UNSUPPORTED
    finally:
        capi.conv2d_desc_destroy(d)
    d = capi.conv2d_desc_create(2, 64, 28, 28, 512, 3, 3, 1, 1, "f16", "implicit_nchw_tc")
    try:
        with pytest.raises(capi.Conv2dError) as e:
            capi.conv2d_desc_set_tuning(d, "tile_n", 176)
        assert e.value.status == capi.ERR_UNSUPPORTED
        capi.conv2d_desc_set_tuning(d, "tile_n", 128)
    finally:
        capi.conv2d_desc_destroy(d)
