// fp32 convolution on CUDA cores (FFMA only; no TF32 anywhere).
//
// Work split: a block computes one output row (n, ho), 64 consecutive output
// columns and 32*warps output channels.  A lane owns an 8 x 8 register tile:
// 8 consecutive output columns (lane % 8 picks which 8) x 8 output channels
// (lane / 8 and the warp pick which 8).  Narrow maps (im2win mode, Wo <= 32)
// give a block `rows` output rows instead: the 8 column groups of a lane row
// split into rows x G, G = ceil(Wo / 8) groups per output row, so that up to
// 8 rows of a 5-wide map share a block rather than 3 of its 64 columns.  Per (input channel, filter row,
// filter column) a lane does 64 FMAs for two 16-byte filter loads, which the
// 8 lanes of a channel group share as a broadcast.
//
// K loop: input channels in chunks staged in shared memory, double-buffered,
// by the asynchronous copy engine (completion on an mbarrier):
//   im2win mode  one 1-D bulk copy per channel of the Eq. (2) strip range the
//                block's windows touch ("Enabling Memory-efficient Im2win
//                Convolution ...", Sec. III-B/C: a window is a contiguous run
//                of the strip, Kh elements per input column);
//   direct mode  one 3-D tensor-map copy of the Kh input rows of the chunk,
//                zero-filled outside the image (padding), x origin aligned
//                down to 16 bytes.
// plus one bulk copy of the chunk's repacked filter ([ci][kh][kw][32*warps]).
//
// Reuse across output columns: for each (channel, filter row) a lane loads
// only its own 8*s window columns and takes the Kw - s columns its windows
// share with the next lanes of its group by warp shuffle.
#include <cuda.h>

#include "internal.h"
#include "ptx.cuh"

namespace conv2d_gb300 {

struct Fp32Params {
    const float* src;   // im2win strips [N][Ci][Ho][Lp] or X [N][Ci][H][W]
    const float* wq;    // packed filter
    float* y;
    int N, Ci, H, W, Co, Kh, Kw, s, p, Ho, Wo, Lp;
    int BCO, n_cb, n_wb, chunk, n_chunks;
    int pitch;          // floats per channel of staged input (im2win), or Kh*boxw (direct)
    int rows, G;        // output rows per block; column groups (of 8) per row: 1 and 8 unless im2win and Wo <= 32
    int rpitch;         // im2win: staged floats per output row (pitch = rows * rpitch)
    int n_hb;           // row blocks per image (ceil(Ho / rows))
    int boxw;           // direct mode: staged row width (multiple of 4)
    int xs_floats;      // staged-input floats per stage (including read slack)
    int ws_floats;      // filter floats per stage
    const float* bias;  // Co bias values, or null
    int nst;            // stages in the ring: 2 (copies of chunk k+1 overlap the FMAs of chunk k) or 1
};

constexpr int kCcCols = 64;    // output columns per block (8 lanes x 8)

template <int KW, int S, bool IM2WIN, bool ROWS>
__global__ void __launch_bounds__(128) conv_fp32_kernel(const Fp32Params prm,
                                                        const __grid_constant__ CUtensorMap xmap) {
    extern __shared__ uint8_t smem_raw[];
    // Tensor-map copies need 128-byte aligned destinations.
    float* smem = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    long long b = blockIdx.x;
    const int cb = (int)(b % prm.n_cb); b /= prm.n_cb;
    const int wb = (int)(b % prm.n_wb); b /= prm.n_wb;
    const int ho0 = (int)(b % prm.n_hb) * (ROWS ? prm.rows : 1);   // first output row of the block
    const int n = (int)(b / prm.n_hb);
    const int rows_v = ROWS ? min(prm.rows, prm.Ho - ho0) : 1;     // rows of the block that exist
    const int Kh = prm.Kh;
    const int kw_n = KW > 0 ? KW : prm.Kw;
    const int sd = S > 0 ? S : prm.s;
    const int wo0 = wb * kCcCols;
    const int wb_valid = min(kCcCols, prm.Wo - wo0);
    const int KK = Kh * kw_n;
    const int stage_floats = prm.xs_floats + prm.ws_floats;

    // First staged strip element (im2win) / first staged column (direct).
    const int e0 = IM2WIN ? ((wo0 * sd * Kh) & ~3) : 0;
    int e1 = 0;
    if (IM2WIN) {
        e1 = ((wo0 + wb_valid - 1) * sd + kw_n) * Kh;
        e1 = (e1 + 3) & ~3;
        if (e1 > prm.Lp) e1 = prm.Lp;
    }
    const int xbase = IM2WIN ? 0 : ((wo0 * sd - prm.p) >= 0 ? ((wo0 * sd - prm.p) & ~3)
                                                             : -(((prm.p - wo0 * sd) + 3) & ~3));

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(smem_addr(&bars[0]), 1);
        mbar_init(smem_addr(&bars[1]), 1);
        mbar_fence_init();
        if (!IM2WIN) tma_prefetch_desc(&xmap);
    }
    __syncthreads();
    pdl_wait();   // the repacked filter / strips come from the kernels launched just before

    // Stage and barrier parity of chunk k.
    auto stage_of = [&](int k) { return prm.nst == 2 ? (k & 1) : 0; };
    auto parity_of = [&](int k) { return (uint32_t)(prm.nst == 2 ? (k >> 1) & 1 : k & 1); };
    auto issue = [&](int k) {
        const int st = stage_of(k);
        float* xs = smem + st * stage_floats;
        float* ws = xs + prm.xs_floats;
        const uint32_t bar = smem_addr(&bars[st]);
        const int ci0 = k * prm.chunk;
        const int nci = min(prm.chunk, prm.Ci - ci0);
        const uint32_t wbytes = (uint32_t)(nci * KK * prm.BCO * 4);
        if (IM2WIN) {
            const uint32_t xbytes = (uint32_t)((e1 - e0) * 4);
            mbar_arrive_expect_tx(bar, wbytes + xbytes * nci * rows_v);
            for (int c = 0; c < nci; ++c)
                for (int r = 0; r < rows_v; ++r) {
                    const float* src =
                        prm.src + (((long long)n * prm.Ci + ci0 + c) * prm.Ho + ho0 + r) * prm.Lp + e0;
                    bulk_load(smem_addr(xs + c * prm.pitch + r * prm.rpitch), src, xbytes, bar);
                }
        } else {
            const uint32_t xbytes = (uint32_t)(prm.boxw * Kh * prm.chunk * 4);
            mbar_arrive_expect_tx(bar, wbytes + xbytes);
            tma_load_3d(smem_addr(xs), &xmap, bar, xbase, ho0 * sd - prm.p, n * prm.Ci + ci0);
        }
        bulk_load(smem_addr(ws), prm.wq + ((long long)cb * prm.Ci + ci0) * KK * prm.BCO, wbytes, bar);
    };

    const int lw = lane & 7, lc = lane >> 3;
    // This lane's output row within the block (spare lanes, when rows * G < 8,
    // work on the last row and store nothing) and column group within it.
    const int G = ROWS ? prm.G : 8;
    const int lrow = ROWS ? lw / G : 0, lg = lw - lrow * G;
    const int lr = lrow < prm.rows ? lrow : prm.rows - 1;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

    // Padded column of this lane's first window.
    const int cl = (wo0 + 8 * lg) * sd;
    constexpr int C = 8 * (S > 0 ? S : 1);
    constexpr int WIN = KW > 0 ? 7 * S + KW : 1;

    if (tid == 0) issue(0);
    bool ok = true;
    for (int k = 0; k < prm.n_chunks; ++k) {
        if (prm.nst == 2 && tid == 0 && k + 1 < prm.n_chunks) issue(k + 1);
        // A thread whose wait gives up (or sees another's abort) skips the
        // chunk but still meets the barrier at the end of the iteration; the
        // abort flag, set before that barrier, is then read by all threads
        // alike, so the block leaves the loop together.
        if (mbar_wait(smem_addr(&bars[stage_of(k)]), parity_of(k), &abort_flag)) {
        const float* xs = smem + stage_of(k) * stage_floats;
        const float* ws = xs + prm.xs_floats;
        const int nci = min(prm.chunk, prm.Ci - k * prm.chunk);
        for (int c = 0; c < nci; ++c) {
            for (int kh = 0; kh < Kh; ++kh) {
                // row[col * xstr] = padded input value at column col of this filter row.
                const float* row;
                int xstr;
                if (IM2WIN) { row = xs + c * prm.pitch + (ROWS ? lr * prm.rpitch : 0) + kh - e0; xstr = Kh; }
                else        { row = xs + (c * Kh + kh) * prm.boxw - prm.p - xbase; xstr = 1; }
                const float* wr = ws + ((c * Kh + kh) * kw_n) * prm.BCO + warp * 32 + lc * 8;
                if constexpr (KW > 0) {
                    float v[WIN];
#pragma unroll
                    for (int j = 0; j < C; ++j) v[j] = row[(cl + j) * xstr];
#pragma unroll
                    for (int j = C; j < WIN; ++j) {
                        float t = __shfl_down_sync(0xffffffffu, v[j % C], j / C);
                        if (lg + j / C >= G) t = row[(cl + j) * xstr];   // the neighbour is in another row
                        v[j] = t;
                    }
#pragma unroll
                    for (int kw = 0; kw < KW; ++kw) {
                        const float4 wa = *reinterpret_cast<const float4*>(wr + kw * prm.BCO);
                        const float4 wb4 = *reinterpret_cast<const float4*>(wr + kw * prm.BCO + 4);
                        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb4.x, wb4.y, wb4.z, wb4.w};
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float xv = v[i * S + kw];
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv, wv[j], acc[i][j]);
                        }
                    }
                } else {
                    for (int kw = 0; kw < kw_n; ++kw) {
                        const float4 wa = *reinterpret_cast<const float4*>(wr + kw * prm.BCO);
                        const float4 wb4 = *reinterpret_cast<const float4*>(wr + kw * prm.BCO + 4);
                        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb4.x, wb4.y, wb4.z, wb4.w};
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float xv = row[(cl + i * sd + kw) * xstr];
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(xv, wv[j], acc[i][j]);
                        }
                    }
                }
            }
        }
        }   // chunk k staged
        __syncthreads();
        if (*reinterpret_cast<volatile int*>(&abort_flag)) {
            // Let the copies of this chunk and of the next one (issued before
            // this chunk's wait) land before the CTA exits.
            if (tid == 0) {
                mbar_drain_wait(smem_addr(&bars[stage_of(k)]), parity_of(k));
                if (prm.nst == 2 && k + 1 < prm.n_chunks)
                    mbar_drain_wait(smem_addr(&bars[stage_of(k + 1)]), parity_of(k + 1));
            }
            ok = false;
            break;
        }
        // One stage: the next chunk's copies start once every warp is done with this one.
        if (prm.nst == 1 && tid == 0 && k + 1 < prm.n_chunks) issue(k + 1);
    }
    if (!ok) return;

    // Store: each channel row gets 8 consecutive columns (two 16-byte stores
    // when the row is 16-byte aligned and all 8 columns are outputs).
    const int co_base = cb * prm.BCO + warp * 32 + lc * 8;
    if (ROWS && lrow >= rows_v) return;                       // a spare lane or a row past Ho
    const int ho = ho0 + lrow;
    const int wt = wo0 + 8 * lg;
    const bool vec = (prm.Wo % 4) == 0 && wt + 8 <= prm.Wo;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int co = co_base + j;
        if (co >= prm.Co) continue;
        if (prm.bias) {
            const float bj = __ldg(prm.bias + co);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i][j] += bj;
        }
        float* out = prm.y + (((long long)n * prm.Co + co) * prm.Ho + ho) * prm.Wo + wt;
        if (vec) {
            reinterpret_cast<float4*>(out)[0] = make_float4(acc[0][j], acc[1][j], acc[2][j], acc[3][j]);
            reinterpret_cast<float4*>(out)[1] = make_float4(acc[4][j], acc[5][j], acc[6][j], acc[7][j]);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (wt + i < prm.Wo) out[i] = acc[i][j];
        }
    }
}

// ---------------------------------------------------------------- host side
cudaError_t status_read_clear_fp32(cudaStream_t st, uint32_t* out) { return status_read_clear(st, out); }
cudaError_t wait_limit_set_fp32(cudaStream_t st, uint64_t ns) { return wait_limit_set(st, ns); }

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
void* driver_entry(const char* name);   // conv_tc.cu

template <int KW, int S, bool IM2WIN, bool ROWS = false>
static cudaError_t launch_fp32_inst(const Fp32Params& prm, const CUtensorMap& map, int threads, size_t smem,
                                    long long blocks, cudaStream_t st) {
    auto kern = conv_fp32_kernel<KW, S, IM2WIN, ROWS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_after(kern, dim3((unsigned)blocks), dim3(threads), smem, st, prm, map);
}

template <bool IM2WIN>
static cudaError_t launch_fp32_shape(const conv2d_desc& d, const Fp32Params& prm, const CUtensorMap& map,
                                     int threads, size_t smem, long long blocks, cudaStream_t st) {
    if constexpr (IM2WIN) {
        if (prm.rows > 1) {   // narrow maps: several output rows per block
            if (d.Kw == 3 && d.s == 1) return launch_fp32_inst<3, 1, true, true>(prm, map, threads, smem, blocks, st);
            if (d.Kw == 5 && d.s == 1) return launch_fp32_inst<5, 1, true, true>(prm, map, threads, smem, blocks, st);
            if (d.Kw == 3 && d.s == 2) return launch_fp32_inst<3, 2, true, true>(prm, map, threads, smem, blocks, st);
            return launch_fp32_inst<0, 0, true, true>(prm, map, threads, smem, blocks, st);
        }
    }
#define CONV2D_FP32_CASE(KW_, S_) \
    if (d.Kw == KW_ && d.s == S_) return launch_fp32_inst<KW_, S_, IM2WIN>(prm, map, threads, smem, blocks, st);
    CONV2D_FP32_CASE(1, 1)
    CONV2D_FP32_CASE(3, 1)
    CONV2D_FP32_CASE(5, 1)
    CONV2D_FP32_CASE(7, 1)
    CONV2D_FP32_CASE(9, 1)
    CONV2D_FP32_CASE(11, 1)
    CONV2D_FP32_CASE(3, 2)
    CONV2D_FP32_CASE(7, 2)
#undef CONV2D_FP32_CASE
    return launch_fp32_inst<0, 0, IM2WIN>(prm, map, threads, smem, blocks, st);
}

conv2d_status launch_conv_fp32(const conv2d_desc& d, const float* src, const float* wq, float* y, bool im2win,
                               cudaStream_t st) {
    Fp32Params prm{};
    prm.src = src; prm.wq = wq; prm.y = y; prm.bias = static_cast<const float*>(d.bias);
    prm.nst = d.tune_stages == 1 ? 1 : 2;
    prm.N = d.N; prm.Ci = d.Ci; prm.H = d.H; prm.W = d.W; prm.Co = d.Co; prm.Kh = d.Kh; prm.Kw = d.Kw;
    prm.s = d.s; prm.p = d.p; prm.Ho = d.Ho; prm.Wo = d.Wo; prm.Lp = d.Lp;
    prm.BCO = 32 * d.cc_warps;
    prm.n_cb = (d.Co + prm.BCO - 1) / prm.BCO;
    prm.n_wb = (d.Wo + kCcCols - 1) / kCcCols;
    prm.rows = 1;
    prm.G = 8;
    if (im2win && d.Wo <= 32) {
        prm.G = (d.Wo + 7) / 8;
        prm.rows = 8 / prm.G;
    }
    prm.n_hb = (d.Ho + prm.rows - 1) / prm.rows;
    // Staged input per channel, with slack so that lanes past Wo read inside the buffer.
    const int span = (kCcCols - 1) * d.s + d.Kw;          // padded columns 64 windows touch
    const int slack = kCcCols * d.s + d.Kw + 8;
    int per_ci_x;
    if (im2win) {
        // Staged range [e0, e1) is rounded out to 16 bytes on both ends (+6 at most).
        prm.pitch = ((span * d.Kh + 8) + 3) & ~3;
        prm.rpitch = prm.pitch;
        if (prm.rows > 1) {
            // A lane group reads at most ((8G-1)*s + Kw)*Kh floats from its row's start.
            prm.rpitch = ((((8 * prm.G - 1) * d.s + d.Kw) * d.Kh + 8) + 3) & ~3;
            prm.pitch = prm.rows * prm.rpitch;
        }
        per_ci_x = prm.pitch;
        prm.boxw = 0;
    } else {
        prm.boxw = ((span + 3) + 3) & ~3;
        if (prm.boxw > 256) return CONV2D_ERR_UNSUPPORTED;   // tensor-map box limit
        prm.pitch = d.Kh * prm.boxw;
        per_ci_x = prm.pitch;
    }
    const int per_ci_w = d.Kh * d.Kw * prm.BCO;
    const int budget = 12 * 1024 / 4;    // floats per stage: two stages ~24 KB, several blocks per SM
    int chunk = budget / (per_ci_x + per_ci_w);
    if (chunk < 1) chunk = 1;
    if (chunk > d.Ci) chunk = d.Ci;
    if (chunk > 32) chunk = 32;
    if (!im2win && chunk * d.Kh > 256) chunk = 256 / d.Kh;
    if (chunk < 1) return CONV2D_ERR_UNSUPPORTED;
    prm.chunk = chunk;
    prm.n_chunks = (d.Ci + chunk - 1) / chunk;
    prm.xs_floats = ((chunk * per_ci_x + slack) + 31) & ~31;
    prm.ws_floats = (chunk * per_ci_w + 31) & ~31;
    const size_t smem = (size_t)2 * (prm.xs_floats + prm.ws_floats) * 4 + 128;
    if (smem > 220 * 1024) return CONV2D_ERR_UNSUPPORTED;

    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    if (!im2win) {
        auto enc = reinterpret_cast<PFN_encodeTiled>(driver_entry("cuTensorMapEncodeTiled"));
        if (!enc) return CONV2D_ERR_CUDA;
        cuuint64_t dims[3] = {(cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)d.N * d.Ci};
        cuuint64_t strides[2] = {(cuuint64_t)d.W * 4, (cuuint64_t)d.W * d.H * 4};
        cuuint32_t box[3] = {(cuuint32_t)prm.boxw, (cuuint32_t)d.Kh, (cuuint32_t)chunk};
        cuuint32_t estr[3] = {1, 1, 1};
        if ((d.W * 4) % 16 != 0) return CONV2D_ERR_UNSUPPORTED;   // row pitch must be 16-byte aligned
        CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(src), dims, strides, box,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
    }
    const long long blocks = (long long)d.N * prm.n_hb * prm.n_wb * prm.n_cb;
    if (blocks > 0x7fffffffLL) return CONV2D_ERR_UNSUPPORTED;
    const int threads = 32 * d.cc_warps;
    cudaError_t e = im2win ? launch_fp32_shape<true>(d, prm, map, threads, smem, blocks, st)
                           : launch_fp32_shape<false>(d, prm, map, threads, smem, blocks, st);
    return e == cudaSuccess ? CONV2D_OK : CONV2D_ERR_CUDA;
}

}  // namespace conv2d_gb300
