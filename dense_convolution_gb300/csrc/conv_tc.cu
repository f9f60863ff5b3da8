// fp16/bf16-in, fp32-accumulate convolution on the 5th-generation tensor
// cores (tcgen05 MMA, accumulators in tensor memory), operands fed by TMA.
//
// GEMM view ("Enabling Memory-efficient Im2win Convolution ...", Sec. III-D,
// Algorithm 1 line 1, with the roles of M and N swapped so that the MMA's
// 128-row side runs over output pixels):
//   M = N*Ho*Wo output pixels (row-major over n, ho, wo = NCHW plane order),
//   N = Co output channels,
//   K = taps x channel chunks, 64 16-bit elements per pipeline stage.
//
// A tile (128 pixels x 64 K) comes from one TMA load, in one of two forms:
//   implicit  (kernel MODE 0) an im2col-mode load of X in NHWC [N][H][W][Ci8]:
//             the copy engine walks 128 consecutive output pixels (across
//             row and image boundaries) and reads 64 channels at each
//             pixel's window origin plus the tap offset (kw, kh); the map's
//             bounding box shifts by -p and the walk strides by s, so padding
//             is the copy engine's zero fill.  Tap t = (kh, kw).
//   grid      (kernel MODE 1) a tiled load of 128 consecutive rows of a
//             "virtual pixel grid" [N][Hv][Wq]: row q is one output position,
//             rows past Wo in an image row (or past Ho) are junk that the
//             epilogue drops.  Two sources use it:
//     padded  the zero-padded NHWC copy [N][H+2p][Wq][Ci8], stride 1: virtual
//             row q reads pixel q + kh*Wq + kw for tap (kh, kw); kpb
//             neighbouring taps share one halo box of 128 + kpb - 1 rows.
//     im2win  the window tensor [N][Ho][Wq*s][Ck] (Eq. (2)/(3) of the im2win
//             paper, channels-last): the whole window of output (ho, wo) is
//             the Kw*Ck contiguous elements from column wo*s on, so the map's
//             rows are s*Ck elements apart and overlap; one tap, K = Kw*Ck.
// B tile (BN channels x 64 K) is a tiled TMA load of the repacked filter.
//
// Warp roles (192 threads; one CTA per SM, two for tiles up to 128 channels wide; persistent over tiles):
//   warp 0     TMA producer (one elected lane), STAGES-deep shared-memory ring
//   warp 1     TMEM allocation + MMA issue (one lane): 4 x (128xBNx16) per stage
//   warps 2-5  epilogue: tcgen05.ld of their 32-lane TMEM quarter, round to the
//              output type, store NCHW (32 consecutive pixels per store)
// Two TMEM accumulators let the epilogue of tile i overlap the MMAs of i+1
// (with 256-wide tiles and two CTAs per SM, one each: the other CTA's MMAs
// fill the gap).
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains what it issued,
// frees its TMEM and exits with the device status word set.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace conv2d_gb300 {

struct TcParams {
    int M, HoWo, Ho, Wo, Co;
    int n_n_tiles, n_tiles;
    int n_cchunks, n_kchunks, CP, Kw, s, p;
    int amode;          // A source: 0 implicit, 1 im2win, 2 padded (1 and 2 run kernel MODE 1)
    int N, Wq, HpWq;    // grid modes: batch, row pitch and image pitch of the virtual pixel grid
    int vec_store;      // MODE 0: Ho*Wo % 8 == 0 (16-byte stores); MODE 1: Wo % 4 == 0 (8-byte stores)
    int kpb;            // MMA chunks per pipeline stage (one A copy + one B copy per stage)
    int stages;         // depth of the shared-memory ring (<= kMaxStages)
    int stage_bytes;    // A region + kpb B chunks
    int a_bytes;        // A region of a stage: one 128-row chunk, or a halo of 128 + kpb - 1 rows
    int halo;           // padded mode: a stage holds kpb neighbouring taps kw0..kw0+kpb-1 of one
                        // filter row, all read from one halo A tile at row offsets 0..kpb-1
    int n_sp;           // pipeline stages per output tile
    int n_acc;          // TMEM accumulators (BN columns each): 2 lets the epilogue of one tile
                        // overlap the MMAs of the next; 1 when two CTAs share an SM's TMEM
    void* y;
};

constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448;                               // 227 KB per block
constexpr int kSmemPerSm = 233472;                               // 228 KB per SM, 1 KB of it reserved per block

template <int BN>
struct TcConfig {
    static constexpr int kABytes = kTcBlockM * kTcBlockK * 2;   // one 128 x 64 A chunk: 16 KB
    static constexpr int kBBytes = BN * kTcBlockK * 2;          // one BN x 64 B chunk
    static constexpr int kChunkBytes = kABytes + kBBytes;
    static constexpr int kEpiBytes = 32 * kTcBlockM * 2;        // epilogue staging: 32 channels x 128 pixels
    static constexpr int kTailBytes = kEpiBytes + 256 + 1024;   // staging + barriers + alignment slack
};
// Shared memory layout for a ring of `stages` stages of `stage_bytes`:
//   [stage 0 .. stage S-1][epilogue staging][barriers]; a stage is
//   [kpb A chunks][kpb B chunks], each chunk 1024-byte aligned (128-byte swizzle).

// MODE is the A addressing (0 im2col walk, 1 virtual-grid rows); each compiles
// to its own kernel so the producer and MMA loops carry no run-time mode tests.
template <int BN, bool BF16, int MODE>
__global__ void __launch_bounds__(192, 2) conv_tc_kernel(const __grid_constant__ CUtensorMap amap,
                                                         const __grid_constant__ CUtensorMap bmap,
                                                         const TcParams prm) {
    using Cfg = TcConfig<BN>;
    const int S = prm.stages;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzled operand tiles need 1024-byte alignment.
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int epi_off = S * prm.stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + epi_off + Cfg::kEpiBytes);
    // bars[0..S) full, [S..2S) empty, [2S..2S+2) accumulator full, [2S+2..2S+4) accumulator empty, [2S+4] drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full_bar = [&](int i) { return smem_addr(&bars[i]); };
    auto empty_bar = [&](int i) { return smem_addr(&bars[S + i]); };
    auto accf_bar = [&](int i) { return smem_addr(&bars[2 * S + i]); };
    auto acce_bar = [&](int i) { return smem_addr(&bars[2 * S + 2 + i]); };
    const uint32_t drain_bar = smem_addr(&bars[2 * S + 4]);

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < S; ++i) { mbar_init(full_bar(i), 1); mbar_init(empty_bar(i), 1); }
        for (int i = 0; i < 2; ++i) { mbar_init(accf_bar(i), 1); mbar_init(acce_bar(i), 4); }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&amap);
        tma_prefetch_desc(&bmap);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), prm.n_acc * BN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Operands (window / NHWC tensor, repacked filter) come from the kernels
    // launched just before this one; the set-up above overlapped their tail.
    pdl_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < prm.n_tiles && ok; tile += gridDim.x) {
                const int m0 = (tile / prm.n_n_tiles) * kTcBlockM;
                const int n0 = (tile % prm.n_n_tiles) * BN;
                int img = 0, ho = 0, wo = 0;
                if constexpr (MODE == 0) {
                    img = m0 / prm.HoWo;
                    const int r = m0 - img * prm.HoWo;
                    ho = r / prm.Wo;
                    wo = r - ho * prm.Wo;
                }
                for (int sp = 0; sp < prm.n_sp; ++sp) {
                    // Stage sp covers taps t..t+kpb-1 (halo) or chunk sp, channel block cb.
                    int t, cb;
                    if constexpr (MODE == 1) {
                        cb = sp % prm.n_cchunks;
                        const int rest = sp / prm.n_cchunks, ngw = prm.Kw / prm.kpb;
                        t = (rest / ngw) * prm.Kw + (rest % ngw) * prm.kpb;
                    } else {
                        t = sp / prm.n_cchunks;
                        cb = sp - t * prm.n_cchunks;
                    }
                    const int c0 = cb * kTcBlockK;
                    if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
                    mbar_arrive_expect_tx(full_bar(stage), prm.stage_bytes);
                    const uint32_t a_dst = smem_addr(smem + stage * prm.stage_bytes);
                    const uint32_t b_dst = a_dst + prm.a_bytes;
                    if constexpr (MODE == 1) {
                        // Virtual pixel q reads padded pixel q + kh*Wq + kw.  In halo mode
                        // the box has 128 + kpb - 1 rows: taps kw..kw+kpb-1 are the same
                        // rows shifted by one pixel each, so they share one copy.  (im2win:
                        // one tap, t = 0.)
                        const int kh = t / prm.Kw, kw = t - kh * prm.Kw;
                        tma_load_2d(a_dst, &amap, full_bar(stage), c0, m0 + kh * prm.Wq + kw);
                    } else {
                        const int kh = t / prm.Kw, kw = t - kh * prm.Kw;
                        tma_load_im2col_4d(a_dst, &amap, full_bar(stage), c0, wo * prm.s - prm.p,
                                           ho * prm.s - prm.p, img, (uint16_t)kw, (uint16_t)kh);
                    }
                    // Filter chunks of taps t..t+kpb-1, channel block cb: one copy (a 3-D
                    // box in halo mode; higher-rank maps cost the copy engine more, so
                    // the other modes keep a 2-D map).
                    if constexpr (MODE == 1) tma_load_3d(b_dst, &bmap, full_bar(stage), c0, n0, t);
                    else                     tma_load_2d(b_dst, &bmap, full_bar(stage), t * prm.CP + c0, n0);
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // Let every copy already issued land before the CTA can exit.
                int dummy = 0;
                int st = stage;
                uint32_t ph = phase;
                for (int i = 0; i < S && i < issued; ++i) {
                    if (--st < 0) { st = S - 1; ph ^= 1; }
                    mbar_wait(full_bar(st), ph, &dummy);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_f16(BF16, kTcBlockM, BN);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, issued_any = false;
            for (int tile = blockIdx.x; tile < prm.n_tiles && ok; tile += gridDim.x) {
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int sp = 0; sp < prm.n_sp; ++sp) {
                    if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = smem_addr(smem + stage * prm.stage_bytes);
                    const uint32_t b_base = a_base + prm.a_bytes;
                    const int kpb = MODE == 1 ? prm.kpb : 1;
                    for (int i = 0; i < kpb; ++i) {
                        // Halo: tap kw0+i reads the A tile from row i (128 bytes per row).
                        const uint32_t a_sub = a_base + i * 128u, b_sub = b_base + i * Cfg::kBBytes;
#pragma unroll
                        for (int k = 0; k < kTcBlockK / 16; ++k) {
                            umma_f16(d_tmem, sw128_kmajor_desc(a_sub + 32 * k), sw128_kmajor_desc(b_sub + 32 * k),
                                     idesc, (sp > 0 || i > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    issued_any = true;
                    umma_commit(empty_bar(stage));
                    if (++stage == S) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                umma_commit(accf_bar(acc));
                if (++acc == prm.n_acc) { acc = 0; acc_phase ^= 1; }
            }
            if (!ok && issued_any) {
                int dummy = 0;
                umma_commit(drain_bar);
                mbar_wait(drain_bar, 0, &dummy);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // Each 32-column chunk of the accumulator (32 output channels x 128
        // pixels) is rounded, staged in shared memory as [channel][pixel] and
        // written as whole 256-byte channel rows with 16-byte stores.  The
        // four epilogue warps synchronise on named barrier 1; the per-tile
        // barrier also ANDs the wait results so all four leave together.
        const int quarter = warp & 3;
        const int et = threadIdx.x - 64;                 // 0..127
        uint16_t* stage_out = reinterpret_cast<uint16_t*>(smem + epi_off);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < prm.n_tiles; tile += gridDim.x) {
            const bool got = mbar_wait(accf_bar(acc), acc_phase, abort_flag);
            if (!named_bar_and(1, 128, got)) break;
            tc_fence_after();
            const int m0 = (tile / prm.n_n_tiles) * kTcBlockM;
            const int n0 = (tile % prm.n_n_tiles) * BN;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
            if constexpr (MODE == 1) {
                // Rows are virtual pixels of the grid [N][Hv][Wq]; only
                // those with y < Ho and x < Wo are outputs.  With Wo % 4 == 0 a
                // 4-pixel group is all-valid or all-junk: 8-byte stores.
                const int g = et & 31;
                const int qg = m0 + 4 * g;
                const int ng = qg / prm.HpWq, rg = qg - ng * prm.HpWq;
                const int yg = rg / prm.Wq, xg = rg - yg * prm.Wq;
                const bool g_ok = ng < prm.N && yg < prm.Ho && xg < prm.Wo;
                uint16_t* gbase = static_cast<uint16_t*>(prm.y) + (long long)ng * prm.Co * prm.HoWo + yg * prm.Wo + xg;
                const int qp = m0 + et;                      // scalar fallback: one pixel per thread
                const int np = qp / prm.HpWq, rp = qp - np * prm.HpWq;
                const int yp = rp / prm.Wq, xp = rp - yp * prm.Wq;
                const bool p_ok = np < prm.N && yp < prm.Ho && xp < prm.Wo;
                uint16_t* pbase = static_cast<uint16_t*>(prm.y) + (long long)np * prm.Co * prm.HoWo + yp * prm.Wo + xp;
#pragma unroll 1
                for (int cc = 0; cc < BN / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_row + cc * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float f = __uint_as_float(v[j]);
                        uint16_t h;
                        if (BF16) h = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                        else      h = __half_as_ushort(__float2half_rn(f));
                        stage_out[j * kTcBlockM + quarter * 32 + lane] = h;
                    }
                    named_bar_sync(1, 128);
                    if (prm.vec_store) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int row = (et >> 5) + 4 * i;
                            const int co = n0 + cc * 32 + row;
                            if (g_ok && co < prm.Co)
                                *reinterpret_cast<uint2*>(gbase + (long long)co * prm.HoWo) =
                                    *reinterpret_cast<const uint2*>(stage_out + row * kTcBlockM + 4 * g);
                        }
                    } else if (p_ok) {
#pragma unroll 4
                        for (int row = 0; row < 32; ++row) {
                            const int co = n0 + cc * 32 + row;
                            if (co < prm.Co) pbase[(long long)co * prm.HoWo] = stage_out[row * kTcBlockM + et];
                        }
                    }
                    named_bar_sync(1, 128);
                }
            } else if (prm.vec_store) {
                const int grp = et & 15;                    // this thread's 8-pixel group
                const int mg = m0 + 8 * grp;
                const bool g_ok = mg < prm.M;
                const int img = g_ok ? mg / prm.HoWo : 0;
                const int r = g_ok ? mg - img * prm.HoWo : 0;
                uint16_t* gbase = static_cast<uint16_t*>(prm.y) + ((long long)img * prm.Co) * prm.HoWo + r;
#pragma unroll 1
                for (int cc = 0; cc < BN / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_row + cc * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float f = __uint_as_float(v[j]);
                        uint16_t h;
                        if (BF16) h = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                        else      h = __half_as_ushort(__float2half_rn(f));
                        stage_out[j * kTcBlockM + quarter * 32 + lane] = h;
                    }
                    named_bar_sync(1, 128);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int row = (et >> 4) + 8 * i;
                        const int co = n0 + cc * 32 + row;
                        if (g_ok && co < prm.Co) {
                            const uint4 val = *reinterpret_cast<const uint4*>(stage_out + row * kTcBlockM + 8 * grp);
                            *reinterpret_cast<uint4*>(gbase + (long long)co * prm.HoWo) = val;
                        }
                    }
                    named_bar_sync(1, 128);
                }
            } else {
                const int m = m0 + quarter * 32 + lane;
                const bool m_ok = m < prm.M;
                const int img = m_ok ? m / prm.HoWo : 0;
                const int r = m_ok ? m - img * prm.HoWo : 0;
                uint16_t* out = static_cast<uint16_t*>(prm.y) + ((long long)img * prm.Co) * prm.HoWo + r;
#pragma unroll 1
                for (int cc = 0; cc < BN / 32; ++cc) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(t_row + cc * 32, v);
                    tmem_ld_wait();
                    const int cob = n0 + cc * 32;
                    if (m_ok) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const int co = cob + j;
                            if (co < prm.Co) {
                                const float f = __uint_as_float(v[j]);
                                uint16_t h;
                                if (BF16) h = __bfloat16_as_ushort(__float2bfloat16_rn(f));
                                else      h = __half_as_ushort(__float2half_rn(f));
                                out[(long long)co * prm.HoWo] = h;
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(acc));
            if (++acc == prm.n_acc) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, prm.n_acc * BN);
    }
}

// ---------------------------------------------------------------- host side
void* driver_entry(const char* name) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return fn;
}

cudaError_t status_read_clear_tc(cudaStream_t st, uint32_t* out) { return status_read_clear(st, out); }

int device_sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev];
    int v = 148;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (dev >= 0 && dev < 64) cached[dev] = v;
    return v;
}

typedef CUresult (*PFN_encodeTiled_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                      const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                      CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);
typedef CUresult (*PFN_encodeIm2col_t)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                       const cuuint64_t*, const int*, const int*, cuuint32_t, cuuint32_t,
                                       const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                       CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

template <int BN, bool BF16, int MODE>
static cudaError_t launch_tc_inst(const CUtensorMap& a, const CUtensorMap& b, const TcParams& prm, int grid,
                                  cudaStream_t st) {
    auto kern = conv_tc_kernel<BN, BF16, MODE>;
    const int smem = prm.stages * prm.stage_bytes + TcConfig<BN>::kTailBytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_after(kern, dim3(grid), dim3(192), smem, st, a, b, prm);
}

template <bool BF16, int MODE>
static cudaError_t launch_tc_bn(int BN, const CUtensorMap& a, const CUtensorMap& b, const TcParams& prm, int grid,
                                cudaStream_t st) {
    switch (BN) {
        case 64:  return launch_tc_inst<64, BF16, MODE>(a, b, prm, grid, st);
        case 128: return launch_tc_inst<128, BF16, MODE>(a, b, prm, grid, st);
        default:  return launch_tc_inst<256, BF16, MODE>(a, b, prm, grid, st);
    }
}

template <bool BF16>
static cudaError_t launch_tc_mode(int BN, int amode, const CUtensorMap& a, const CUtensorMap& b, const TcParams& prm,
                                  int grid, cudaStream_t st) {
    return amode == 0 ? launch_tc_bn<BF16, 0>(BN, a, b, prm, grid, st) : launch_tc_bn<BF16, 1>(BN, a, b, prm, grid, st);
}

conv2d_status launch_conv_tc(const conv2d_desc& d, const void* src, const void* wq, void* y, int amode,
                             cudaStream_t st) {
    const bool im2win = amode == 1;
    auto enc_tiled = reinterpret_cast<PFN_encodeTiled_t>(driver_entry("cuTensorMapEncodeTiled"));
    auto enc_im2col = reinterpret_cast<PFN_encodeIm2col_t>(driver_entry("cuTensorMapEncodeIm2col"));
    if (!enc_tiled || !enc_im2col) return CONV2D_ERR_CUDA;
    const CUtensorMapDataType dt =
        d.dtype == CONV2D_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;

    CUtensorMap amap, bmap;
    // Ring layout.  Padded mode groups kpb neighbouring taps of one filter row
    // per stage around one halo A tile (128 + kpb - 1 pixel rows): each stage
    // costs the producer and MMA threads a fixed run of waits, copies and a
    // commit, so fewer stages with more MMAs each feed the tensor core better.
    const int n_cchunks = d.CP / kTcBlockK;
    const int b_chunk = d.BN * kTcBlockK * 2;
    const int tail = 32 * kTcBlockM * 2 + 256 + 1024;
    const bool halo = amode == 2;
    const bool grid_rows = amode != 0;
    // Last virtual row that is an output, plus one (grid modes).
    const int m_end = grid_rows ? (d.N - 1) * d.Hp * d.Wq + (d.Ho - 1) * d.Wq + d.Wo : 0;
    // Ring plan for a shared-memory budget: halo width kpb (largest divisor of
    // Kw leaving at least min_halo stages), stage size and depth.
    auto plan = [&](int budget, int min_halo, int& kpb_o, int& rows_o, int& stages_o) {
        kpb_o = 1; rows_o = kTcBlockM;
        if (halo) {
            for (int c = d.Kw; c >= 2; --c) {
                if (d.Kw % c) continue;
                const int rows = (kTcBlockM + c - 1 + 7) / 8 * 8;
                if ((budget - tail) / (rows * 128 + c * b_chunk) >= min_halo) { kpb_o = c; rows_o = rows; break; }
            }
        }
        stages_o = (budget - tail) / (rows_o * 128 + kpb_o * b_chunk);
        if (stages_o > kMaxStages) stages_o = kMaxStages;
    };
    // Two CTAs per SM where both fit in half the SM's shared memory (TMEM: two
    // BN-column accumulators each, or one for 256-wide tiles): a CTA's TMA
    // producer and MMA issuer are single threads whose per-instruction
    // latency, not the copy engine or the tensor core, bounds narrow tiles,
    // and a second CTA doubles the issue rate (measured on GB300: about 81
    // cycles per tcgen05.mma in one thread, while a 128x64x16 MMA executes in
    // 32; 100-140 cycles per TMA copy, wait or commit).  Each CTA keeps at
    // least 3 stages, or 2 when a stage holds several taps' MMAs (halo) or
    // 256-wide ones.
    int kpb, a_rows, stages, ctas_per_sm = 1, n_acc = 2;
    plan(kSmemPerSm / 2 - 1024, 2, kpb, a_rows, stages);
    if (stages >= (kpb > 1 || d.BN == 256 ? 2 : 3)) {
        ctas_per_sm = 2;
        if (d.BN == 256) n_acc = 1;
    } else {
        plan(kSmemLimit, 3, kpb, a_rows, stages);
    }
    if (stages < 2) return CONV2D_ERR_UNSUPPORTED;
    const int stage_bytes = a_rows * 128 + kpb * b_chunk;

    CUresult r;
    if (im2win) {
        // Window tensor rows of Ck elements, Wq*s per image row: virtual row q
        // starts s*Ck elements after row q-1 and spans Kw*Ck elements.  Rows
        // at or past m_end read as zero, so no copy runs off the tensor's end.
        cuuint64_t wdims[2] = {(cuuint64_t)d.Kw * d.Ck, (cuuint64_t)m_end};
        cuuint64_t wstr[1] = {(cuuint64_t)d.s * d.Ck * 2};
        cuuint32_t wbox[2] = {(cuuint32_t)kTcBlockK, (cuuint32_t)kTcBlockM};
        cuuint32_t westr[2] = {1, 1};
        r = enc_tiled(&amap, dt, 2, const_cast<void*>(src), wdims, wstr, wbox, westr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (amode == 2) {
        // Padded channels-last copy viewed as [N*Hp*Wq pixel rows][Ci8 channels];
        // box 64 channels x a_rows pixels (rows past the end read as zero).
        cuuint64_t pdims[2] = {(cuuint64_t)d.Ci8, (cuuint64_t)d.N * d.Hp * d.Wq};
        cuuint64_t pstr[1] = {(cuuint64_t)d.Ci8 * 2};
        cuuint32_t pbox[2] = {(cuuint32_t)kTcBlockK, (cuuint32_t)a_rows};
        cuuint32_t pestr[2] = {1, 1};
        r = enc_tiled(&amap, dt, 2, const_cast<void*>(src), pdims, pstr, pbox, pestr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // im2col view of X in NHWC, dims (Ci8, W, H, N).
        cuuint64_t adims[4] = {(cuuint64_t)d.Ci8, (cuuint64_t)d.W, (cuuint64_t)d.H, (cuuint64_t)d.N};
        cuuint64_t astr[3] = {adims[0] * 2, adims[0] * 2 * adims[1], adims[0] * 2 * adims[1] * adims[2]};
        int lower[2] = {-d.p, -d.p}, upper[2] = {d.p - (d.Kw - 1), d.p - (d.Kh - 1)};
        cuuint32_t estr[4] = {1, (cuuint32_t)d.s, (cuuint32_t)d.s, 1};
        r = enc_im2col(&amap, dt, 4, const_cast<void*>(src), adims, astr, lower, upper, kTcBlockK, kTcBlockM, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return CONV2D_ERR_CUDA;

    // B: repacked filter [Co][taps][CP].  Grid modes: (CP, Co, tap) with box
    // 64 x BN x kpb = the chunks of kpb consecutive taps for one channel block;
    // otherwise 2-D (taps*CP, Co) with box 64 x BN.
    if (grid_rows) {
        cuuint64_t bdims[3] = {(cuuint64_t)d.CP, (cuuint64_t)d.Co, (cuuint64_t)d.taps};
        cuuint64_t bstr[2] = {(cuuint64_t)d.taps * d.CP * 2, (cuuint64_t)d.CP * 2};
        cuuint32_t bbox[3] = {(cuuint32_t)kTcBlockK, (cuuint32_t)d.BN, (cuuint32_t)kpb};
        cuuint32_t bestr[3] = {1, 1, 1};
        r = enc_tiled(&bmap, dt, 3, const_cast<void*>(wq), bdims, bstr, bbox, bestr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t bdims[2] = {(cuuint64_t)d.taps * d.CP, (cuuint64_t)d.Co};
        cuuint64_t bstr[1] = {(cuuint64_t)d.taps * d.CP * 2};
        cuuint32_t bbox[2] = {(cuuint32_t)kTcBlockK, (cuuint32_t)d.BN};
        cuuint32_t bestr[2] = {1, 1};
        r = enc_tiled(&bmap, dt, 2, const_cast<void*>(wq), bdims, bstr, bbox, bestr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) return CONV2D_ERR_CUDA;

    TcParams prm{};
    // M runs over output pixels, or over the virtual grid up to the last output (grid modes).
    prm.M = grid_rows ? m_end : d.N * d.Ho * d.Wo;
    prm.N = d.N;
    prm.Wq = d.Wq;
    prm.HpWq = d.Hp * d.Wq;
    prm.HoWo = d.Ho * d.Wo; prm.Ho = d.Ho; prm.Wo = d.Wo; prm.Co = d.Co;
    prm.n_n_tiles = (d.Co + d.BN - 1) / d.BN;
    const int n_m_tiles = (prm.M + kTcBlockM - 1) / kTcBlockM;
    prm.n_tiles = n_m_tiles * prm.n_n_tiles;
    prm.n_cchunks = d.CP / kTcBlockK;
    prm.n_kchunks = d.taps * prm.n_cchunks;
    prm.CP = d.CP; prm.Kw = d.Kw; prm.s = d.s; prm.p = d.p;
    prm.amode = amode;
    prm.kpb = kpb;
    prm.stages = stages;
    prm.stage_bytes = stage_bytes;
    prm.a_bytes = a_rows * 128;
    prm.halo = halo ? 1 : 0;
    prm.n_sp = halo ? d.Kh * (d.Kw / kpb) * n_cchunks : d.taps * n_cchunks;
    prm.n_acc = n_acc;
    prm.y = y;
    if (grid_rows)
        prm.vec_store = ((d.Wo % 4) == 0 && (d.Wq % 4) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) ? 1 : 0;
    else
        prm.vec_store = ((prm.HoWo % 8) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) ? 1 : 0;
    int grid = device_sm_count() * ctas_per_sm;
    if (grid > prm.n_tiles) grid = prm.n_tiles;

    const bool bf = d.dtype == CONV2D_BF16;
    cudaError_t e = bf ? launch_tc_mode<true>(d.BN, amode, amap, bmap, prm, grid, st)
                       : launch_tc_mode<false>(d.BN, amode, amap, bmap, prm, grid, st);
    return e == cudaSuccess ? CONV2D_OK : CONV2D_ERR_CUDA;
}

}  // namespace conv2d_gb300
