// Winograd minimal filtering F(2x2, 3x3) in fp32 on the CUDA cores, for 3x3
// stride-1 layers: the method of "OpenCNN: a Winograd minimal filtering
// algorithm implementation in CUDA" (Sec. 2, Eqs. (2)-(5); Sec. 3: a separate
// filter-transform kernel, then one kernel that transforms input tiles,
// multiplies in the transformed domain as 16 batched GEMMs and transforms the
// sums back), and of "im2col Expansion, FFT Convolution, and Winograd
// Transforms", Winograd section.
//
// Per 2x2 output tile Y of one output channel, with d the 4x4 input tile
// (zero outside the image) of each input channel and g that channel's 3x3
// filter:
//     Y = A^T [ sum_ci (G g G^T) (*) (B^T d B) ] A          (* elementwise)
// with interpolation points 0, 1, -1 and infinity:
//     B^T d : rows (d0 - d2, d1 + d2, d2 - d1, d1 - d3)
//     G g   : rows (g0, (g0 + g1 + g2)/2, (g0 - g1 + g2)/2, g2)
//     A^T m : rows (m0 + m1 + m2, m1 - m2 - m3)
// (each applied along both axes).  16 multiplications per tile and channel
// pair instead of 36.  The sum over input channels runs in the transformed
// domain, so accumulation error grows with the transforms' coefficients; the
// parity tests hold it to the fp32 contract against the direct sum.
#include "internal.h"
#include "ptx.cuh"

namespace conv2d_gb300 {

constexpr int kWgTiles = 32;      // output tiles per block: 4 rows x 8 columns of 2x2 (8 x 16 outputs)
constexpr int kWgCo = 64;         // output channels per block
constexpr int kWgCb = 8;          // input channels per pipeline stage
constexpr int kWgThreads = 256;

// ---------------------------------------------------------------- filter transform
// U[kb][ci][e][k] = (G g G^T)[e] of filter (co = 64 kb + k, ci), e = 4a + b,
// zero for co >= Co or ci >= Ci (ci runs to Ci rounded up to kWgCb).  One
// thread per (co, ci) pair.  A stage's slice (8 channels x 16 x 64) is then
// one contiguous 32 KB block.
__global__ void __launch_bounds__(256) winograd_filter_kernel(const float* __restrict__ w, float* __restrict__ u,
                                                              int Co, int Ci, int Ci8) {
    pdl_wait();                 // first kernel of a call: see pack_filter_tc_kernel
    pdl_launch_dependents();
    const int kb_n = (Co + kWgCo - 1) / kWgCo;
    const long long total = (long long)kb_n * kWgCo * Ci8;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int k = (int)(i % kWgCo);
        const long long r = i / kWgCo;
        const int ci = (int)(r % Ci8);
        const int kb = (int)(r / Ci8);
        const int co = kb * kWgCo + k;
        float g[9];
#pragma unroll
        for (int j = 0; j < 9; ++j) g[j] = (co < Co && ci < Ci) ? __ldg(w + ((long long)co * Ci + ci) * 9 + j) : 0.f;
        // G g (columns), then (G g) G^T (rows): t[a][c], then U[a][b].
        float t[4][3];
#pragma unroll
        for (int c = 0; c < 3; ++c) {
            const float g0 = g[c], g1 = g[3 + c], g2 = g[6 + c];
            t[0][c] = g0;
            t[1][c] = 0.5f * (g0 + g1 + g2);
            t[2][c] = 0.5f * (g0 - g1 + g2);
            t[3][c] = g2;
        }
        float* dst = u + ((((long long)kb * Ci8 + ci) * 16) * kWgCo) + k;
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const float h0 = t[a][0], h1 = t[a][1], h2 = t[a][2];
            dst[(4 * a + 0) * kWgCo] = h0;
            dst[(4 * a + 1) * kWgCo] = 0.5f * (h0 + h1 + h2);
            dst[(4 * a + 2) * kWgCo] = 0.5f * (h0 - h1 + h2);
            dst[(4 * a + 3) * kWgCo] = h2;
        }
    }
}

// ---------------------------------------------------------------- main kernel
struct WgParams {
    const float* x;     // NCHW input
    const float* u;     // transformed filter (winograd_filter_kernel)
    float* y;           // NCHW output
    const float* bias;  // Co values or null
    int N, Ci, Ci8, H, W, Co, Ho, Wo, p;
    int n_bx, n_by, kb_n;   // blocks along output columns (16 wide) and rows (8 high); channel blocks
};

constexpr int kWgVFloats = kWgCb * 16 * kWgTiles;          // V stage: [c][e][t]
constexpr int kWgUFloats = kWgCb * 16 * kWgCo;             // U stage: [c][e][k]
constexpr int kWgStageFloats = kWgVFloats + kWgUFloats;
constexpr int kWgExchFloats = 16 * kWgCo * kWgTiles;       // sums before the output transform: [e][k][t]
constexpr int kWgSmemFloats = (2 * kWgStageFloats > kWgExchFloats) ? 2 * kWgStageFloats : kWgExchFloats;
constexpr int kWgSmemBytes = kWgSmemFloats * 4 + 128;

// One block: 32 output tiles (2x2 each, 8 rows x 16 columns of outputs) of one
// image for 64 output channels, over all input channels in stages of 8.
// Thread (c, t) = (tid / 32, tid % 32) transforms the 4x4 input tile t of
// channel c of a stage (B^T d B) into V[c][e][t].  Warp w then accumulates
// transform points e = 2w, 2w+1; lane (ti, ki) = (lane / 8, lane % 8) holds
// tiles 8ti..8ti+7 x channels 8ki..8ki+7 of both: per (channel, e) one 8x8
// outer product from two float4 reads of V and two of U (shared-memory reads
// broadcast within the warp).  The next stage's filter slice arrives by bulk
// copy and its input tiles are loaded into registers while this stage runs.
// At the end the sums go through shared memory as [e][k][t] so that each
// thread holds all 16 points of its (tile, channel) pairs for A^T m A.
__global__ void __launch_bounds__(kWgThreads, 1) winograd_f2x3_kernel(const WgParams prm) {
    extern __shared__ uint8_t wg_smem_raw[];
    float* smem = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(wg_smem_raw) + 127) & ~uintptr_t(127));
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    long long b = blockIdx.x;
    const int kb = (int)(b % prm.kb_n); b /= prm.kb_n;
    const int bx = (int)(b % prm.n_bx); b /= prm.n_bx;
    const int by = (int)(b % prm.n_by);
    const int n = (int)(b / prm.n_by);
    const int n_chunks = prm.Ci8 / kWgCb;

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(smem_addr(&bars[0]), 1);
        mbar_init(smem_addr(&bars[1]), 1);
        mbar_fence_init();
    }
    __syncthreads();
    pdl_wait();   // the transformed filter comes from the kernel launched just before

    // This thread's input tile: channel c of the stage, tile t = (ty, tx).
    const int c_in = tid >> 5, t_in = tid & 31;
    const int gy = by * 4 + (t_in >> 3), gx = bx * 8 + (t_in & 7);
    const int iy0 = 2 * gy - prm.p, ix0 = 2 * gx - prm.p;
    auto load_tile = [&](int chunk, float (&d)[16]) {
        const int ci = chunk * kWgCb + c_in;
        const float* plane = prm.x + ((long long)n * prm.Ci + ci) * prm.H * prm.W;
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int iy = iy0 + r, ix = ix0 + q;
                d[4 * r + q] = (ci < prm.Ci && iy >= 0 && iy < prm.H && ix >= 0 && ix < prm.W)
                                   ? __ldg(plane + (long long)iy * prm.W + ix)
                                   : 0.f;
            }
    };
    // B^T d B into V[c][e][t] of a stage.
    auto store_tile = [&](int stage, const float (&d)[16]) {
        float t[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {      // columns: B^T along rows
            const float d0 = d[q], d1 = d[4 + q], d2 = d[8 + q], d3 = d[12 + q];
            t[q] = d0 - d2;
            t[4 + q] = d1 + d2;
            t[8 + q] = d2 - d1;
            t[12 + q] = d1 - d3;
        }
        float* v = smem + stage * kWgStageFloats + c_in * 16 * kWgTiles + t_in;
#pragma unroll
        for (int a = 0; a < 4; ++a) {      // rows: B along columns
            const float h0 = t[4 * a], h1 = t[4 * a + 1], h2 = t[4 * a + 2], h3 = t[4 * a + 3];
            v[(4 * a + 0) * kWgTiles] = h0 - h2;
            v[(4 * a + 1) * kWgTiles] = h1 + h2;
            v[(4 * a + 2) * kWgTiles] = h2 - h1;
            v[(4 * a + 3) * kWgTiles] = h1 - h3;
        }
    };
    auto issue_u = [&](int chunk, int stage) {     // one thread: the stage's 32 KB filter slice
        const float* src = prm.u + ((long long)kb * prm.Ci8 + (long long)chunk * kWgCb) * 16 * kWgCo;
        const uint32_t bar = smem_addr(&bars[stage]);
        fence_proxy_async_smem();        // the previous reads of this stage come before the copy's writes
        mbar_arrive_expect_tx(bar, kWgUFloats * 4);
        bulk_load(smem_addr(smem + stage * kWgStageFloats + kWgVFloats), src, kWgUFloats * 4, bar);
    };

    float acc[2][8][8];
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[e][i][j] = 0.f;

    {
        float d[16];
        if (tid == 0) issue_u(0, 0);
        load_tile(0, d);
        store_tile(0, d);
    }
    __syncthreads();
    const int ti = lane >> 3, ki = lane & 7;
    bool ok = true;
    for (int k = 0; k < n_chunks; ++k) {
        const int s = k & 1;
        float d[16];
        const bool more = k + 1 < n_chunks;
        if (more) {
            if (tid == 0) issue_u(k + 1, s ^ 1);   // stage s^1 is free: its last reader finished before the barrier
            load_tile(k + 1, d);
        }
        if (mbar_wait(smem_addr(&bars[s]), (uint32_t)((k >> 1) & 1), &abort_flag)) {
            const float* vs = smem + s * kWgStageFloats;
            const float* us = vs + kWgVFloats;
#pragma unroll 2
            for (int c = 0; c < kWgCb; ++c) {
#pragma unroll
                for (int ee = 0; ee < 2; ++ee) {
                    const int e = 2 * warp + ee;
                    const float4 va = *reinterpret_cast<const float4*>(vs + (c * 16 + e) * kWgTiles + 8 * ti);
                    const float4 vb = *reinterpret_cast<const float4*>(vs + (c * 16 + e) * kWgTiles + 8 * ti + 4);
                    const float4 ua = *reinterpret_cast<const float4*>(us + (c * 16 + e) * kWgCo + 8 * ki);
                    const float4 ub = *reinterpret_cast<const float4*>(us + (c * 16 + e) * kWgCo + 8 * ki + 4);
                    const float vv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
                    const float uu[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i)
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[ee][i][j] = fmaf(vv[i], uu[j], acc[ee][i][j]);
                }
            }
        }
        if (more) store_tile(s ^ 1, d);
        __syncthreads();
        if (*reinterpret_cast<volatile int*>(&abort_flag)) {
            // Let the filter copies issued for this stage and the next land before exiting.
            if (tid == 0) {
                mbar_drain_wait(smem_addr(&bars[s]), (uint32_t)((k >> 1) & 1));
                if (more) mbar_drain_wait(smem_addr(&bars[s ^ 1]), (uint32_t)(((k + 1) >> 1) & 1));
            }
            ok = false;
            break;
        }
    }
    if (!ok) return;

    // Sums of the 16 transform points, [e][k][t], then A^T m A per (tile, channel).
#pragma unroll
    for (int ee = 0; ee < 2; ++ee) {
        const int e = 2 * warp + ee;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float* dst = smem + (e * kWgCo + 8 * ki + j) * kWgTiles + 8 * ti;
            reinterpret_cast<float4*>(dst)[0] = make_float4(acc[ee][0][j], acc[ee][1][j], acc[ee][2][j], acc[ee][3][j]);
            reinterpret_cast<float4*>(dst)[1] = make_float4(acc[ee][4][j], acc[ee][5][j], acc[ee][6][j], acc[ee][7][j]);
        }
    }
    __syncthreads();
    const int t = tid & 31;
    const int oy = 2 * (by * 4 + (t >> 3)), ox = 2 * (bx * 8 + (t & 7));
#pragma unroll 1
    for (int kk = tid >> 5; kk < kWgCo; kk += kWgThreads / 32) {
        const int co = kb * kWgCo + kk;
        if (co >= prm.Co) break;
        float m[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) m[e] = smem[(e * kWgCo + kk) * kWgTiles + t];
        float r0[4], r1[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {      // A^T along rows
            r0[q] = m[q] + m[4 + q] + m[8 + q];
            r1[q] = m[4 + q] - m[8 + q] - m[12 + q];
        }
        const float bv = prm.bias ? __ldg(prm.bias + co) : 0.f;
        const float out[2][2] = {{r0[0] + r0[1] + r0[2] + bv, r0[1] - r0[2] - r0[3] + bv},
                                 {r1[0] + r1[1] + r1[2] + bv, r1[1] - r1[2] - r1[3] + bv}};
        float* yp = prm.y + ((long long)n * prm.Co + co) * prm.Ho * prm.Wo;
#pragma unroll
        for (int dy = 0; dy < 2; ++dy)
#pragma unroll
            for (int dx = 0; dx < 2; ++dx)
                if (oy + dy < prm.Ho && ox + dx < prm.Wo) yp[(long long)(oy + dy) * prm.Wo + ox + dx] = out[dy][dx];
    }
}

// ---------------------------------------------------------------- host side
size_t winograd_filter_bytes(const conv2d_desc& d) {
    const long long kb_n = (d.Co + kWgCo - 1) / kWgCo, ci8 = (d.Ci + kWgCb - 1) / kWgCb * kWgCb;
    return (size_t)(kb_n * kWgCo * ci8 * 16) * 4;
}

cudaError_t launch_winograd_filter(const conv2d_desc& d, const float* w, float* u, cudaStream_t st) {
    const int ci8 = (d.Ci + kWgCb - 1) / kWgCb * kWgCb;
    const int kb_n = (d.Co + kWgCo - 1) / kWgCo;
    const long long fthreads = (long long)kb_n * kWgCo * ci8;
    long long fblocks = (fthreads + 255) / 256;
    const long long cap = (long long)device_sm_count() * 8;
    if (fblocks > cap) fblocks = cap;
    return launch_after(winograd_filter_kernel, dim3((unsigned)fblocks), dim3(256), 0, st, w, u, d.Co, d.Ci, ci8);
}

// The main kernel waits (griddepcontrol) before reading anything, so it may
// also be the first kernel of a call.
conv2d_status launch_winograd_main(const conv2d_desc& d, const float* x, const float* u, float* y,
                                   cudaStream_t st) {
    const int ci8 = (d.Ci + kWgCb - 1) / kWgCb * kWgCb;
    const int kb_n = (d.Co + kWgCo - 1) / kWgCo;
    cudaError_t e;
    WgParams prm{};
    prm.x = x; prm.u = u; prm.y = y; prm.bias = static_cast<const float*>(d.bias);
    prm.N = d.N; prm.Ci = d.Ci; prm.Ci8 = ci8; prm.H = d.H; prm.W = d.W; prm.Co = d.Co;
    prm.Ho = d.Ho; prm.Wo = d.Wo; prm.p = d.p;
    const int th = (d.Ho + 1) / 2, tw = (d.Wo + 1) / 2;
    prm.n_by = (th + 3) / 4;
    prm.n_bx = (tw + 7) / 8;
    prm.kb_n = kb_n;
    const long long blocks = (long long)d.N * prm.n_by * prm.n_bx * kb_n;
    if (blocks > 0x7fffffffLL) return CONV2D_ERR_UNSUPPORTED;
    e = cudaFuncSetAttribute(winograd_f2x3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kWgSmemBytes);
    if (e == cudaSuccess)
        e = launch_after(winograd_f2x3_kernel, dim3((unsigned)blocks), dim3(kWgThreads), kWgSmemBytes, st, prm);
    return e == cudaSuccess ? CONV2D_OK : CONV2D_ERR_CUDA;
}

cudaError_t status_read_clear_wg(cudaStream_t st, uint32_t* out) { return status_read_clear(st, out); }
cudaError_t wait_limit_set_wg(cudaStream_t st, uint64_t ns) { return wait_limit_set(st, ns); }

}  // namespace conv2d_gb300
