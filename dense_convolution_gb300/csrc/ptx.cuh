// Inline-PTX wrappers for sm_103a: mbarrier, bulk/tensor TMA copies, tcgen05
// (MMA, TMEM allocation and loads) and the bounded waits every kernel uses.
// Encodings follow the public PTX ISA (tcgen05 matrix/instruction descriptor
// tables, cp.async.bulk.tensor tile and im2col modes).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace conv2d_gb300 {

// ---------------------------------------------------------------- status word
// Bit set in the library's device status word when a bounded wait expires.
// Host code reads and clears it through conv2d_device_status().
constexpr uint32_t kStatusTimeout = 1u;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per wait, then give up

// One status word per translation unit (internal linkage, so no relocatable
// device code is needed); each unit exports a host reader.
static __device__ uint32_t g_device_status = 0;

// Limit of the pipeline waits (mbar_wait), default kWaitLimitNs.  The host can
// lower it (wait_limit_set) so that a test sees waits give up; the waits that
// let in-flight copies and MMAs finish before a CTA exits (mbar_drain_wait)
// always use kWaitLimitNs.
static __constant__ uint64_t g_wait_limit_ns = kWaitLimitNs;

// Set this translation unit's pipeline-wait limit for kernels launched on
// `st` after this call (0, or anything above the default, gives the default:
// the limit can only be lowered, so every wait stays bounded).
static inline cudaError_t wait_limit_set(cudaStream_t st, uint64_t ns) {
    static uint64_t v;   // the copy reads the source when the stream reaches it
    v = (ns == 0 || ns > kWaitLimitNs) ? kWaitLimitNs : ns;
    cudaError_t e = cudaMemcpyToSymbolAsync(g_wait_limit_ns, &v, sizeof(v), 0, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    return e;
}

// Read and clear this translation unit's status word (synchronises `st`).
static inline cudaError_t status_read_clear(cudaStream_t st, uint32_t* out) {
    uint32_t v = 0, z = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_device_status, sizeof(v), 0, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e == cudaSuccess && v != 0) {
        e = cudaMemcpyToSymbolAsync(g_device_status, &z, sizeof(z), 0, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    *out = v;
    return e;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- dependent launch
// Allow the next kernel in the stream to start launching (no-op without PDL).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the preceding kernel has completed and its writes are visible
// (no-op when this kernel was not launched as a dependent).
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the same condition (never suspends the thread).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Gives up after
// kWaitLimitNs, or early once *abort (shared memory) is set by another role;
// on a timeout it records kStatusTimeout in the device status word and sets
// *abort so that the other warps of the CTA stop too.  Returns false when the
// wait did not complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
    const uint64_t limit = g_wait_limit_ns;
    if (limit >= kWaitLimitNs) {
        // Default limit: try_wait may suspend the thread for a hardware time
        // slice, which covers nearly every pipeline wait; the clock is read
        // only once 256 slices have passed, and then every 256 more.
        bool started = false;
        uint64_t t0 = 0;
        for (uint32_t i = 1;; ++i) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((i & 255u) == 0) {
                if (*abort) return false;
                const uint64_t t = global_timer_ns();
                if (!started) {
                    started = true;
                    t0 = t;
                } else if (t - t0 > limit) {
                    atomicOr(&g_device_status, kStatusTimeout);
                    *abort = 1;
                    return false;
                }
            }
        }
    }
    // A lowered limit: poll without suspending and test the clock every time,
    // so that even a wait of a few nanoseconds can expire.
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_test_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > limit) {
            atomicOr(&g_device_status, kStatusTimeout);
            *abort = 1;
            return false;
        }
    }
}

// Wait used after an abort, for copies or MMAs this CTA already issued to
// complete before it exits: no abort test, fixed limit kWaitLimitNs (then the
// status word is set and the wait gives up).
__device__ __forceinline__ bool mbar_drain_wait(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
            atomicOr(&g_device_status, kStatusTimeout);
            return false;
        }
    }
}

// Wait until a 64-bit flag in global memory (written by another CTA of this
// grid) holds `value`.  Bounded like mbar_wait: gives up after the wait
// limit, or once *abort is set, recording kStatusTimeout on a timeout.
__device__ __forceinline__ bool flag_wait(const unsigned long long* flag, unsigned long long value,
                                          volatile int* abort) {
    const volatile unsigned long long* f = flag;
    if (*f == value) return true;
    const uint64_t t0 = global_timer_ns();
    const uint64_t limit = g_wait_limit_ns;
    for (uint32_t i = 1;; ++i) {
        if (*f == value) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > limit) {
                atomicOr(&g_device_status, kStatusTimeout);
                *abort = 1;
                return false;
            }
        }
        __nanosleep(64);
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

// Four 8x8 matrices of 16-bit elements from shared memory, transposed: lane
// 8i + j gives the address of row j of matrix i (16 bytes); thread t receives
// in r[i] the transposed matrix's row t/4, elements 2(t%4) and 2(t%4)+1.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}
// Four 8x8 matrices of 16-bit elements to shared memory: lane 8i + j gives the
// address of row j of matrix i (16 bytes); thread t supplies in r[i] row t/4,
// elements 2(t%4) and 2(t%4)+1.
__device__ __forceinline__ void stsm_x4(uint32_t addr, const uint32_t (&r)[4]) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ void st_shared_b32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Tiled TMA store of a shared-memory box to global memory (bulk-group
// completion).  Elements of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Wait until every committed bulk store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c0, int c1,
                                            int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}

// im2col-mode load of a 4-D channels-innermost tensor (C, W, H, N): a column
// of pixels walked W-then-H-then-N inside the map's bounding box, starting at
// (w, h, n), each pixel read at (w + off_w, h + off_h), channels [c, c+box).
__device__ __forceinline__ void tma_load_im2col_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int c,
                                                   int w, int h, int n, uint16_t off_w, uint16_t off_h) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.im2col.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], {%7, %8};" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c), "r"(w), "r"(h), "r"(n), "h"(off_w), "h"(off_h)
        : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (fp16 or bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on an mbarrier when all previously issued tcgen05 ops of this
// thread have completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor, K-major operand in the 128-byte swizzle
// layout written by a TMA box whose rows are 128 bytes: 8-row groups are
// 1024 bytes apart (stride byte offset); the leading byte offset is unused
// for this layout; bit 46 is the descriptor version; swizzle code 2 = 128B.
// An operand may start r rows into a 1024-byte-aligned tile (the halo tiles
// of the padded path): the swizzle phase is taken from the absolute shared
// memory address, the same rule TMA uses when it writes the tile, so the
// base-offset field (bits 49-51) stays 0.  Measured: setting it to r gives
// wrong products, leaving it 0 is bit-exact.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Shared-memory matrix descriptor for an MN-major operand in the 128-byte
// swizzle, as a TMA box 64 elements (128 bytes) wide along M/N and K rows
// deep writes it: 8 K rows (1024 bytes) per swizzle atom; the next 64-wide
// M/N block of the operand lies mn_block_bytes further on.  A K step of 16
// advances the start address by 2048 bytes.  (Measured on GB300 against a
// host product; the stride fields are read as LBO = the M/N block stride and
// SBO = the 8-row K-group stride.)
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t saddr, uint32_t mn_block_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((mn_block_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation, both operands
// K-major: D format (bits 4-5) = F32, A/B format (bits 7-9 / 10-12) = F16 or
// BF16, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_f16(bool bf16, int M, int N) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// 32 lanes x 32 consecutive 32-bit TMEM columns -> 32 registers per thread
// (thread i of the warp gets lane base+i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also returns the AND of `pred` over the participating threads.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ bool elect_one_sync() {
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\t"
        "elect.sync rx|px, %1;\n\t"
        "selp.b32 %0, 1, 0, px;\n\t}"
        : "=r"(pred)
        : "r"(0xffffffffu));
    return pred != 0;
}

}  // namespace conv2d_gb300
