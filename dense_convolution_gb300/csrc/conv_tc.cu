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
// B tile (BN channels x 64 K) is a tiled TMA load of the repacked filter;
// BN is 64, 128, 176 or 256 (the host picks the width with the fewest waves
// of tile groups; a 176-wide accumulator sits on a 256-column TMEM boundary).
//
// 1x1 layers (stride 1, no padding; kernel MODE 3) need no transform at all:
// per image Y[co][p] = sum_ci W[co][ci] X[ci][p] is a plain GEMM on the NCHW
// tensors.  The MMA runs with M = 128 output channels (W, K-major, straight
// from the caller's filter) and N = 128 pixels (X, read as [ci][p] rows:
// the "MN-major" operand layout, two 64-pixel boxes per chunk), so each
// accumulator lane is one output channel and its columns are consecutive
// pixels: the epilogue rounds them into a swizzled shared-memory box that one
// TMA store writes to Y.
//
// Warp roles (352 threads, or 480 with a third epilogue group or the MODE 4
// halo builders; one persistent CTA per SM):
//   warp 0      TMA producer (one lane), STAGES-deep shared-memory ring
//   warps 1-2   MMA issue (one lane each; warp 1 also allocates TMEM): tile i
//               of a pair of tiles into its own TMEM accumulators
//   warps 3-10  two epilogue groups of four warps, group e draining issuer e
//               (warps 3-14, three groups, optional: group e drains both tiles
//               of every third item): tcgen05.ld of their 32-lane TMEM
//               quarter, round to the output type, transpose through shared
//               memory, store NCHW
// Two TMEM accumulators per issuer (three with three groups; when TMEM holds
// them) let the epilogue of one tile overlap the MMAs of the next.
// Every wait is bounded (ptx.cuh); on a timeout the CTA drains what it issued,
// frees its TMEM and exits with the device status word set.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <chrono>

#include "internal.h"
#include "ptx.cuh"

namespace conv2d_gb300 {

// Division of a non-negative 31-bit integer by a divisor fixed per launch,
// as a multiply-high, an add and a shift (Granlund and Montgomery, "Division
// by invariant integers using multiplication", 1994): with s = ceil(log2 d)
// and m = floor(2^32 (2^s - d) / d) + 1, x / d = (umulhi(x, m) + x) >> s.
struct FastDiv {
    uint32_t m, s;
};
inline FastDiv make_fastdiv(uint32_t d) {
    uint32_t s = 0;
    while ((1ull << s) < d) ++s;
    return FastDiv{(uint32_t)(((1ull << 32) * ((1ull << s) - d)) / d + 1), s};
}
__device__ __forceinline__ int fdiv(const FastDiv& f, int x) {
    return (int)((__umulhi((uint32_t)x, f.m) + (uint32_t)x) >> f.s);
}

struct TcParams {
    int M, HoWo, Ho, Wo, Co;
    int n_n_tiles;      // output-channel tiles (BN wide)
    int group;          // tiles per group (1 or kIssuers): consecutive 128-pixel tiles of one channel tile
    int n_groups;       // tile groups
    int n_m_tiles;      // 128-pixel tiles (groups past the end are padded with empty tiles)
    int n_cchunks, CP, Kw, s, p;
    int amode;          // A source: 0 implicit, 1 im2win, 2 padded (1 and 2 run kernel MODE 1), 3 1x1 GEMM
    int N, Wq, HpWq;    // grid modes: batch, row pitch and image pitch of the virtual pixel grid
    FastDiv fd_wq, fd_hpwq, fd_howo, fd_nnt;   // division by Wq, HpWq, Ho*Wo and n_n_tiles
    int vec_store;      // MODE 0: Ho*Wo % 8 == 0 (16-byte stores); MODE 1: Wo % 4 == 0 (8-byte stores); MODE 3 unused
    int kpb;            // taps per pipeline stage (halo mode), else 1
    int stages;         // depth of the shared-memory ring (<= kMaxStages)
    int stage_bytes;    // `group` A regions (+ the stage's B chunks unless B is resident)
    int a_bytes;        // one A region: a 128-row chunk, or a halo of 128 + kpb - 1 rows
    int n_sp;           // pipeline stages per tile group
    int n_acc;          // TMEM accumulators per issuer (BN columns each)
    int n_egroups;      // epilogue groups of four warps: 2 (group e drains issuer e), or 3 with n_acc == 3
                        // (group e drains both tiles of the items idx with idx % 3 == e)
    int epi_bytes;      // epilogue staging: 4 * n_egroups warps
    int taps;           // filter taps of the repacked filter
    int b_res;          // 1: the whole filter slice of the (single) channel tile stays in shared memory
    int b_res_off;      // byte offsets in the aligned dynamic shared memory
    int epi_off;
    int n_pt;           // MODE 3: 128-pixel tiles per image
    void* y;
    const void* bias;   // Co bias values of the input type, or null
    int out32;          // 1: Y is fp32 (no rounding to the input type)
    // MODE 4 (halo tiles built from NCHW X in shared memory): the A ring
    // holds a_stages stages of `group` halo regions of halo_rows rows each,
    // one stage per (channel chunk, group of khg filter rows); B streams
    // through the ring above (stages, stage_bytes) unless resident.
    const void* x;      // NCHW input
    int Ci, H, W;
    int khg, n_khg;     // filter rows per A stage; A stages per channel chunk
    int halo_rows;      // rows (pixels) of one halo region, a multiple of 8
    int a_stages, a_stage_bytes, a_ring_off;
    int vecw;           // pixels per vector load (W % vecw == 0, Wq % vecw == 0)
    int staged;         // 1: X arrives by TMA boxes of kSeg pixels x 64 channels into per-warp
                        //    staging slots (H*W % 8 == 0); 0: builder lanes load X themselves
    int n_slots;        // staging slots per builder warp
    int stg_off;        // staging region (slots, then a 128-byte discard row per warp)
    // Ablation knobs (conv2d_desc_set_tuning).
    int raster;         // tile-group visit order: 0 channel tile fastest, 1 pixel group fastest,
                        // 2 zig-zag (channel tiles in alternating direction on successive pixel groups)
    int sync_copies;    // 1: the producer waits for each stage's copies before issuing the next stage
    int n_mg;           // pixel groups (ceil(n_m_tiles / group))
    // Split tail (MODE 0/1): groups [0, g_dp) are taken whole, one per CTA per
    // wave; the k-stages of the remaining groups (t_stages in all) are divided
    // evenly over the CTAs.  A group's first contributor owns it: the others
    // store fp32 partial accumulators in `part` and publish `epoch` in `flags`;
    // the owner adds them before its epilogue.
    // A contributor CTA c stores its partial in block (c - 1)*group + tile
    // (each such c is a share boundary inside a group, so grid - 1 blocks
    // per tile suffice) and its flag at the same index.
    int split, g_dp;
    long long t_stages;
    float* part;
    unsigned long long* flags;
    unsigned long long epoch;
};

// One unit of a CTA's work: stages [k0, k1) of tile group g.
struct TcItem {
    int g, k0, k1;
    int owner;          // 1: this CTA stores the group's output (it holds the group's first stage)
    int n_contrib;      // CTAs that share the group
    int c_first;        // the owner CTA (split groups)
    int tg;             // tail group index (split groups), else -1
};

// First stage of CTA c's share of the tail.
__device__ __forceinline__ long long tail_begin(const TcParams& prm, int c) {
    return (long long)c * prm.t_stages / gridDim.x;
}
// The CTA whose share holds tail stage x.
__device__ __forceinline__ int tail_cta(const TcParams& prm, long long x) {
    int c = (int)(x * gridDim.x / prm.t_stages);
    while (c + 1 < (int)gridDim.x && tail_begin(prm, c + 1) <= x) ++c;
    while (c > 0 && tail_begin(prm, c) > x) --c;
    return c;
}

// Item `idx` of this CTA (false when there is none): first its whole groups,
// g = blockIdx.x + i*gridDim.x below g_dp, then (SPLIT kernels) the group
// pieces of its share of the tail in stage order.  Every role of the CTA
// walks the same items.
template <bool SPLIT>
__device__ __forceinline__ bool tc_item(const TcParams& prm, int idx, TcItem& it) {
    const int n_dp = prm.g_dp > (int)blockIdx.x ? (prm.g_dp - (int)blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    if (idx < n_dp) {
        it.g = blockIdx.x + idx * gridDim.x;
        it.k0 = 0; it.k1 = prm.n_sp; it.owner = 1; it.n_contrib = 1; it.c_first = blockIdx.x; it.tg = -1;
        return true;
    }
    if constexpr (!SPLIT) {
        return false;
    } else {
    if (!prm.split) return false;
    const long long b0 = tail_begin(prm, blockIdx.x), b1 = tail_begin(prm, blockIdx.x + 1);
    const long long tg = b0 / prm.n_sp + (idx - n_dp);
    const long long gs = tg * prm.n_sp, ge = gs + prm.n_sp;
    if (b0 >= b1 || gs >= b1) return false;
    it.tg = (int)tg;
    it.g = prm.g_dp + (int)tg;
    it.k0 = (int)((b0 > gs ? b0 : gs) - gs);
    it.k1 = (int)((b1 < ge ? b1 : ge) - gs);
    const int c_first = tail_cta(prm, gs), c_last = tail_cta(prm, ge - 1);
    it.owner = (int)blockIdx.x == c_first;
    it.n_contrib = c_last - c_first + 1;
    it.c_first = c_first;
    return true;
    }
}

// Tile group g -> (channel tile nt, pixel group mg) in the chosen raster order.
// Every role walks g = blockIdx.x, +gridDim.x, ... and maps it the same way.
__device__ __forceinline__ void tile_of(const TcParams& prm, int g, int& nt, int& mg) {
    if (prm.raster == 1) {
        nt = g / prm.n_mg;
        mg = g - nt * prm.n_mg;
    } else {
        mg = fdiv(prm.fd_nnt, g);
        nt = g - mg * prm.n_n_tiles;
        if (prm.raster == 2 && (mg & 1)) nt = prm.n_n_tiles - 1 - nt;
    }
}

// Bias of output channel co, widened to fp32.
template <bool BF16>
__device__ __forceinline__ float load_bias(const void* bias, int co) {
    const unsigned short u = __ldg(static_cast<const unsigned short*>(bias) + co);
    if (BF16) return __bfloat162float(__ushort_as_bfloat16(u));
    return __half2float(__ushort_as_half(u));
}

constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448;                               // 227 KB per block
constexpr int kIssuers = 2;                                      // MMA-issuing threads (one tile each)
constexpr int kEpiWarpBytes = 32 * 32 * 2;                       // epilogue staging per warp: 32 ch x 32 px
constexpr int kEpiBytes = 2 * 4 * kEpiWarpBytes;                 // two epilogue groups of four warps
constexpr int kEpi1x1WarpBytes = 32 * 64 * 2;                      // MODE 3: one 32 ch x 64 px store box per warp
constexpr int kEpi1x1Bytes = 2 * 4 * kEpi1x1WarpBytes;
constexpr int kBarBytes = 512;
constexpr int kTcThreads = 32 * (1 + kIssuers + 8);              // producer, issuers, 8 epilogue warps
constexpr int kTransposerWarps = 4;                              // MODE 4: halo builders
constexpr int kMaxAStages = 4;
template <int MODE>
__host__ __device__ constexpr int tc_threads() { return kTcThreads + (MODE == 4 ? 32 * kTransposerWarps : 0); }
// Launch bound: modes 0 and 1 (without the split protocol) may run a third
// epilogue group of four warps.
template <int MODE, bool SPLIT>
__host__ __device__ constexpr int tc_max_threads() {
    return ((MODE == 0 || MODE == 1) && !SPLIT) ? kTcThreads + 32 * 4 : tc_threads<MODE>();
}

// TMEM columns between accumulators: BN rounded up to a power of two (a
// 176-wide accumulator starts on a 256-column boundary).
__host__ __device__ constexpr int acc_stride(int bn) { return bn <= 64 ? 64 : (bn <= 128 ? 128 : 256); }

template <int BN>
struct TcConfig {
    static constexpr int kBBytes = BN * kTcBlockK * 2;          // one BN x 64 B chunk
};
// Dynamic shared memory (1024-byte aligned): [stage 0 .. stage S-1][resident
// filter][epilogue staging][barriers].  A stage is [A region of issuer 0]
// [A region of issuer 1][kpb B chunks, unless the filter is resident]; every
// region is a multiple of 1024 bytes (128-byte swizzle atoms).

// ---------------------------------------------------------------- MODE 4 halo builders
// V consecutive pixels of one channel from global memory (16-bit elements;
// the address is aligned to 2*V bytes), as V halves in d[0..].
template <int V>
__device__ __forceinline__ void load_pixels(const uint16_t* src, uint32_t (&d)[4]) {
    if constexpr (V == 8) {
        const uint4 t = __ldg(reinterpret_cast<const uint4*>(src));
        d[0] = t.x; d[1] = t.y; d[2] = t.z; d[3] = t.w;
    } else if constexpr (V == 4) {
        const uint2 t = __ldg(reinterpret_cast<const uint2*>(src));
        d[0] = t.x; d[1] = t.y;
    } else if constexpr (V == 2) {
        d[0] = __ldg(reinterpret_cast<const unsigned int*>(src));
    } else {
        d[0] = __ldg(src);
    }
}

constexpr int kBuildBatch = 8;   // vector groups whose loads a builder lane keeps in flight
constexpr int kSeg = 56;         // staged pixels per TMA box (112-byte rows: conflict-free ldmatrix rows)
constexpr int kSegBytes = kSeg * kTcBlockK * 2;
constexpr int kMaxSlots = 2;

// Build this warp's share of one A stage from TMA-staged X (H*W % 8 == 0).
// The stage needs the padded pixels [Pa, Pb) of the virtual grid; their image
// rows are read as runs of whole input rows, flat along the image (n, ci, HW),
// in boxes of kSeg pixels x 64 channels (copy-engine zero fill past HW and Ci).
// Segment k of the stage goes to builder warp k % 4, through this warp's
// staging slots (copies of later segments in flight while one is transposed).
// A box is transposed 8 pixels x 32 channels at a time (ldmatrix .trans) and
// stored as 16-byte channel chunks of the halo rows of every tile that holds
// the pixel (stmatrix; a lane whose pixel no tile needs writes a discard row).
// Rows of padding, pitch junk and images past N are written as zeros.
__device__ __forceinline__ void build_halo_stage_staged(const TcParams& prm, const CUtensorMap* xmap, int tw,
                                                        int lane, uint32_t stage_base, uint32_t slot_base,
                                                        uint32_t slot_bar0, uint32_t& slot_phases, uint32_t discard,
                                                        int mt0, int n_val, int cb, int kg) {
    const int R = prm.halo_rows, Wq = prm.Wq, Hp = prm.HpWq / prm.Wq, HW = prm.H * prm.W;
    const int off = kg * prm.khg * Wq;
    const int Pa = mt0 * kTcBlockM + off, Pb = (mt0 + n_val - 1) * kTcBlockM + off + R;
    const int Y_lo = Pa / Wq, Y_hi = (Pb - 1) / Wq;         // padded rows n*Hp + yy of the stage
    const int n_lo = Y_lo / Hp, n_hi = min(Y_hi / Hp, prm.N - 1);
    // Segments per image: input rows iy_lo..iy_hi, flat [iy_lo*W, (iy_hi+1)*W) from a multiple of 8.
    auto image_rows = [&](int n, int& f0, int& f1) {
        const int ylo = max(Y_lo - n * Hp, 0) - prm.p, yhi = min(Y_hi - n * Hp, Hp - 1) - prm.p;
        const int ia = max(ylo, 0), ib = min(yhi, prm.H - 1);
        if (ia > ib) { f0 = f1 = 0; return 0; }
        f0 = (ia * prm.W) & ~7;
        f1 = (ib + 1) * prm.W;
        return (f1 - f0 + kSeg - 1) / kSeg;
    };
    int total = 0;
    for (int n = n_lo; n <= n_hi; ++n) { int a, b; total += image_rows(n, a, b); }
    auto seg_at = [&](int k, int& n_out, int& x_out) {
        for (int n = n_lo; n <= n_hi; ++n) {
            int f0, f1;
            const int c = image_rows(n, f0, f1);
            if (k < c) { n_out = n; x_out = f0 + k * kSeg; return; }
            k -= c;
        }
        n_out = 0; x_out = 0;
    };
    const int n_slots = prm.n_slots;
    auto issue = [&](int k, int slot) {
        int n, x;
        seg_at(k, n, x);
        if (lane == 0) {
            const uint32_t bar = slot_bar0 + 8u * (uint32_t)slot;
            fence_proxy_async_smem();                    // earlier ldmatrix reads of the slot come first
            mbar_arrive_expect_tx(bar, (uint32_t)kSegBytes);
            tma_load_3d(slot_base + (uint32_t)(slot * kSegBytes), xmap, bar, x, cb * kTcBlockK, n);
        }
    };
    int k_issue = tw;
    for (int sl = 0; sl < n_slots && k_issue < total; ++sl, k_issue += kTransposerWarps) issue(k_issue, sl);

    // Zero rows while the copies are in flight: padded rows Y_lo + tw, + 4, ...
    for (int Y = Y_lo + tw; Y <= Y_hi; Y += kTransposerWarps) {
        const int n = Y / Hp, yy = Y - n * Hp;
        const bool blank = n >= prm.N || yy < prm.p || yy >= prm.p + prm.H;
        for (int run = 0; run < 2; ++run) {
            const int c0 = blank ? (run ? Wq : 0) : (run ? prm.p + prm.W : 0);
            const int c1 = blank ? Wq : (run ? Wq : prm.p);
            if (c0 >= c1) continue;
            for (int i = 0; i < n_val; ++i) {
                const int base = (mt0 + i) * kTcBlockM + off;
                const int r0 = max(Y * Wq + c0 - base, 0), r1 = min(Y * Wq + c1 - base, R);
                const uint32_t tile = stage_base + (uint32_t)(i * prm.a_bytes);
                for (int t = lane; t < (r1 - r0) * 8; t += 32)
                    st_shared_v4(tile + (uint32_t)(r0 + (t >> 3)) * 128u + (uint32_t)(t & 7) * 16u, 0u, 0u, 0u, 0u);
            }
        }
    }

    int slot = 0;
    for (int k = tw; k < total; k += kTransposerWarps) {
        int n, x;
        seg_at(k, n, x);
        const uint32_t bar = slot_bar0 + 8u * (uint32_t)slot;
        mbar_drain_wait(bar, (slot_phases >> slot) & 1u);   // this warp's own copy: it always lands
        slot_phases ^= 1u << slot;
        const uint32_t sbase = slot_base + (uint32_t)(slot * kSegBytes);
        const int j = lane & 7;
        for (int b = 0; b < kSeg / 8; ++b) {
            const int f = x + 8 * b + j;
            int r[kIssuers];
            bool any = false;
            const int iy = f / prm.W, ix = f - iy * prm.W;
            const int P = n * prm.HpWq + (iy + prm.p) * Wq + ix + prm.p;
#pragma unroll
            for (int i = 0; i < kIssuers; ++i) {
                r[i] = P - ((mt0 + i) * kTcBlockM + off);
                const bool in = i < n_val && f < HW && r[i] >= 0 && r[i] < R;
                if (!in) r[i] = -1;
                any |= in;
            }
            if (!__any_sync(0xffffffffu, any)) continue;
            uint32_t q[2][4];
            ldsm_x4_trans(sbase + (uint32_t)lane * (kSeg * 2) + 16u * b, q[0]);
            ldsm_x4_trans(sbase + (uint32_t)(lane + 32) * (kSeg * 2) + 16u * b, q[1]);
            const uint32_t mm = (uint32_t)(lane >> 3);
#pragma unroll
            for (int i = 0; i < kIssuers; ++i) {
                if (i >= n_val) break;
                const uint32_t tile = stage_base + (uint32_t)(i * prm.a_bytes);
                const uint32_t row = tile + (uint32_t)r[i] * 128u;
                const uint32_t ph = (uint32_t)(r[i] & 7);
                stsm_x4(r[i] >= 0 ? row + ((mm ^ ph) << 4) : discard, q[0]);
                stsm_x4(r[i] >= 0 ? row + (((mm + 4u) ^ ph) << 4) : discard, q[1]);
            }
        }
        __syncwarp();
        if (k_issue < total) { issue(k_issue, slot); k_issue += kTransposerWarps; }
        if (++slot == n_slots) slot = 0;
    }
}


// Build this warp's share of one A stage: for each valid tile i of the group,
// halo_rows rows of 64 channels (chunk cb) in the 128-byte-swizzled K-major
// layout, row r = padded pixel P = (mt0 + i)*128 + kg*khg*Wq + r of the
// virtual grid [N][H+2p][Wq]:  X[n][c][yy-p][xx-p], zero outside the image,
// past Ci, in the pitch's junk columns and past the last image.  Rows are
// taken in groups of V pixels that start at padded column = p (mod V), so a
// group lies in one image row and is either all inside the image (one V-wide
// load per channel) or all padding.  Lane l carries channels 2l and 2l+1 and
// writes them as one 32-bit word, so a warp store fills one 128-byte row.
template <int V>
__device__ __forceinline__ void build_halo_stage(const TcParams& prm, int tw, int lane, uint32_t stage_base,
                                                 int mt0, int n_val, int cb, int kg) {
    const uint16_t* __restrict__ xg = static_cast<const uint16_t*>(prm.x);
    const long long plane = (long long)prm.H * prm.W;
    const int R = prm.halo_rows;
    const int g0 = prm.p % V ? prm.p % V - V : 0;           // first group's first row (<= 0)
    const int n_vg = (R - g0 + V - 1) / V;                   // groups per halo region
    const int ch = cb * kTcBlockK + 2 * lane;                // this lane's channel pair
    const int total = n_val * n_vg;
    for (int j0 = tw; j0 < total; j0 += kTransposerWarps * kBuildBatch) {
        uint32_t d0[kBuildBatch][4], d1[kBuildBatch][4];
        int ti[kBuildBatch], tr[kBuildBatch];               // tile (-1: no group) and first row
#pragma unroll
        for (int u = 0; u < kBuildBatch; ++u) {
            const int j = j0 + u * kTransposerWarps;
#pragma unroll
            for (int e = 0; e < 4; ++e) d0[u][e] = d1[u][e] = 0u;
            ti[u] = -1;
            tr[u] = 0;
            if (j >= total) continue;
            const int i = j / n_vg, jg = j - i * n_vg;
            const int r0 = g0 + jg * V;
            ti[u] = i;
            tr[u] = r0;
            const int P = (mt0 + i) * kTcBlockM + kg * prm.khg * prm.Wq + r0;
            if (P < 0) continue;
            const int n = P / prm.HpWq;
            const int rem = P - n * prm.HpWq;
            const int yy = rem / prm.Wq, xx = rem - yy * prm.Wq;
            const int iy = yy - prm.p, ix = xx - prm.p;
            if (n >= prm.N || iy < 0 || iy >= prm.H || ix < 0 || ix >= prm.W) continue;
            const uint16_t* src = xg + ((long long)n * prm.Ci + ch) * plane + (long long)iy * prm.W + ix;
            if (ch < prm.Ci) load_pixels<V>(src, d0[u]);
            if (ch + 1 < prm.Ci) load_pixels<V>(src + plane, d1[u]);
        }
#pragma unroll
        for (int u = 0; u < kBuildBatch; ++u) {
            if (ti[u] < 0) continue;                          // warp-uniform
            const int r0 = tr[u];
            const uint32_t tile = stage_base + (uint32_t)(ti[u] * prm.a_bytes);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const int r = r0 + e;
                if (r < 0 || r >= R) continue;
                const uint32_t lo = (d0[u][e >> 1] >> (16 * (e & 1))) & 0xffffu;
                const uint32_t hi = (d1[u][e >> 1] >> (16 * (e & 1))) & 0xffffu;
                const uint32_t addr =
                    tile + (uint32_t)r * 128u + ((((uint32_t)(lane >> 2) ^ (uint32_t)(r & 7)) << 4) | ((lane & 3) << 2));
                st_shared_b32(addr, lo | (hi << 16));
            }
        }
    }
}

// MODE is the A addressing (0 im2col walk, 1 virtual-grid rows, 3 1x1 GEMM
// on NCHW); each compiles to its own kernel so the producer and MMA loops
// carry no run-time mode tests.
//
// Tiles are taken in groups of kIssuers consecutive 128-pixel tiles of one
// channel tile (single tiles when there are fewer than two tiles per SM).  A stage holds the A chunks of every tile in the group and
// one B chunk they share, so B is read once per group; issuer i runs the MMAs
// of tile i of the group into its own TMEM accumulators.  One thread issuing
// tcgen05.mma takes about 81 cycles per instruction (measured on GB300), while
// a 128x64x16 MMA executes in 32: two issuers keep narrow tiles fed.  When the
// whole filter slice fits (one channel tile), it is loaded once per CTA and
// stays resident, and stages carry A only.
template <int BN, bool BF16, int MODE, bool SPLIT>
__global__ void __launch_bounds__(tc_max_threads<MODE, SPLIT>(), 1) conv_tc_kernel(const __grid_constant__ CUtensorMap amap,
                                                                const __grid_constant__ CUtensorMap bmap,
                                                                const __grid_constant__ CUtensorMap ymap,
                                                                const TcParams prm) {
    using Cfg = TcConfig<BN>;
    const int S = prm.stages;
    extern __shared__ uint8_t smem_raw[];
    // 128-byte swizzled operand tiles need 1024-byte alignment.  (Offsetting
    // the shared array itself keeps pointers in the shared address space.)
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + prm.epi_off + prm.epi_bytes);
    // bars: [0, S) full, [S, 2S) empty, then per issuer i: accf[i][0..n_acc),
    // acce[i][0..n_acc), then the resident-filter barrier and kIssuers drain barriers.
    const int nacc = prm.n_acc;
    // MODE 4 A ring: afull[0..kMaxAStages), aempty[0..kMaxAStages) after the drain barriers.
    uint64_t* abars = bars + 2 * S + 2 * kIssuers * nacc + 1 + kIssuers;
    // MODE 4 staging: one barrier per (builder warp, slot) after those.
    uint64_t* sbars = abars + 2 * kMaxAStages;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sbars + kTransposerWarps * kMaxSlots);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    auto full_bar = [&](int i) { return smem_addr(&bars[i]); };
    auto empty_bar = [&](int i) { return smem_addr(&bars[S + i]); };
    auto accf_bar = [&](int is, int a) { return smem_addr(&bars[2 * S + is * 2 * nacc + a]); };
    auto acce_bar = [&](int is, int a) { return smem_addr(&bars[2 * S + is * 2 * nacc + nacc + a]); };
    const uint32_t bres_bar = smem_addr(&bars[2 * S + 2 * kIssuers * nacc]);
    auto drain_bar = [&](int is) { return smem_addr(&bars[2 * S + 2 * kIssuers * nacc + 1 + is]); };
    // Accumulators: (issuer, buffer) at column (is * nacc + a) * BN; the
    // allocation is a power of two of at least 32 columns.
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)(prm.group * nacc * acc_stride(BN))) tmem_cols <<= 1;

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < S; ++i) { mbar_init(full_bar(i), 1); mbar_init(empty_bar(i), prm.group); }
        for (int is = 0; is < kIssuers; ++is)
            for (int a = 0; a < nacc; ++a) { mbar_init(accf_bar(is, a), 1); mbar_init(acce_bar(is, a), 4); }
        mbar_init(bres_bar, 1);
        for (int is = 0; is < kIssuers; ++is) mbar_init(drain_bar(is), 1);
        if constexpr (MODE == 4) {
            for (int i = 0; i < prm.a_stages; ++i) {
                mbar_init(smem_addr(&abars[i]), kTransposerWarps);          // one arrive per builder warp
                mbar_init(smem_addr(&abars[kMaxAStages + i]), prm.group);    // one commit per issuer
            }
            for (int i = 0; i < kTransposerWarps * kMaxSlots; ++i) mbar_init(smem_addr(&sbars[i]), 1);
        }
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&amap);
        tma_prefetch_desc(&bmap);
        if constexpr (MODE == 3) tma_prefetch_desc(&ymap);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Operands (window / NHWC tensor, repacked filter) come from the kernels
    // launched just before this one; the set-up above overlapped their tail.
    pdl_wait();
    // A kernel launched after this one as a programmatic dependent may now be
    // scheduled: its CTAs take SMs as ours leave and run their set-up there,
    // and its own wait still holds it until this grid has completed.
    pdl_launch_dependents();

    const int kpb = MODE == 1 ? prm.kpb : 1;
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            bool ok = true;
            if (prm.b_res) {
                // The filter slice of channel tile 0: chunk (cb, t) at ((cb*taps + t) * kBBytes).
                const uint32_t bdst = smem_addr(smem + prm.b_res_off);
                mbar_arrive_expect_tx(bres_bar, (uint32_t)(prm.n_cchunks * prm.taps * Cfg::kBBytes));
                for (int cb = 0; cb < prm.n_cchunks; ++cb)
                    for (int t = 0; t < prm.taps; t += kpb) {
                        const uint32_t dst = bdst + (uint32_t)((cb * prm.taps + t) * Cfg::kBBytes);
                        if constexpr (MODE == 1) tma_load_3d(dst, &bmap, bres_bar, cb * kTcBlockK, 0, t);
                        else                     tma_load_2d(dst, &bmap, bres_bar, t * prm.CP + cb * kTcBlockK, 0);
                    }
            }
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            bool free_now = false;
            TcItem it;
            for (int idx = 0; ok && tc_item<SPLIT>(prm, idx, it); ++idx) {
                const int g = it.g;
                if constexpr (MODE == 4) {
                    // A is built by the halo builders; only filter chunks stream
                    // here, one per (channel chunk, tap), in the issuers' order.
                    if (prm.b_res) break;
                    int nt_, mg_;
                    tile_of(prm, g, nt_, mg_);
                    const int nb0 = nt_ * BN;
                    const int Kh = prm.taps / prm.Kw;
                    for (int cb = 0; cb < prm.n_cchunks && ok; ++cb)
                        for (int kg = 0; kg < prm.n_khg && ok; ++kg) {
                            const int kh1 = min(Kh, (kg + 1) * prm.khg);
                            for (int kh = kg * prm.khg; kh < kh1 && ok; ++kh)
                                for (int kw = 0; kw < prm.Kw; ++kw) {
                                    if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
                                    mbar_arrive_expect_tx(full_bar(stage), (uint32_t)Cfg::kBBytes);
                                    tma_load_2d(smem_addr(smem + stage * prm.stage_bytes), &bmap, full_bar(stage),
                                                (kh * prm.Kw + kw) * prm.CP + cb * kTcBlockK, nb0);
                                    const bool landed =
                                        !prm.sync_copies || mbar_wait(full_bar(stage), phase, abort_flag);
                                    ++issued;
                                    if (++stage == S) { stage = 0; phase ^= 1; }
                                    if (!landed) { ok = false; break; }
                                }
                        }
                    continue;
                }
                int nt_, mg_;
                tile_of(prm, g, nt_, mg_);
                const int n0 = nt_ * BN;
                const int mt0 = mg_ * prm.group;
                int m0[kIssuers], img[kIssuers], ho[kIssuers], wo[kIssuers];
                bool val[kIssuers];
                int n_val = 0;
#pragma unroll
                for (int i = 0; i < kIssuers; ++i) {
                    m0[i] = (mt0 + i) * kTcBlockM;
                    val[i] = i < prm.group && mt0 + i < prm.n_m_tiles;
                    n_val += val[i] ? 1 : 0;
                    img[i] = ho[i] = wo[i] = 0;
                    if constexpr (MODE == 0) {
                        if (val[i]) {
                            img[i] = m0[i] / prm.HoWo;
                            const int r = m0[i] - img[i] * prm.HoWo;
                            ho[i] = r / prm.Wo;
                            wo[i] = r - ho[i] * prm.Wo;
                        }
                    } else if constexpr (MODE == 3) {
                        if (val[i]) {                      // image and first pixel of the tile
                            img[i] = (mt0 + i) / prm.n_pt;
                            wo[i] = ((mt0 + i) - img[i] * prm.n_pt) * kTcBlockM;
                        }
                    }
                }
                const uint32_t tx = (uint32_t)(n_val * prm.a_bytes + (prm.b_res ? 0 : kpb * Cfg::kBBytes));
                // Stage coordinates advance incrementally (no divisions in the loop):
                // channel block cb, first tap t = kh*Kw + kw of the stage's kpb taps.
                // Stage coordinates of stage k0: channel block cb, first tap t = kh*Kw + kw.
                int cb = it.k0 % prm.n_cchunks, t = (it.k0 / prm.n_cchunks) * kpb, kw = t % prm.Kw, kh = t / prm.Kw;
                for (int sp = it.k0; sp < it.k1; ++sp) {
                    if (!free_now && !mbar_wait(empty_bar(stage), phase ^ 1, abort_flag)) { ok = false; break; }
                    // Probe the next slot now; the answer is used one stage later, so
                    // the probe's latency hides behind this stage's copies.
                    const int nstage = stage + 1 == S ? 0 : stage + 1;
                    const uint32_t nphase = stage + 1 == S ? phase ^ 1 : phase;
                    const bool free_next = mbar_test_wait(empty_bar(nstage), nphase ^ 1);
                    const int c0 = cb * kTcBlockK;
                    mbar_arrive_expect_tx(full_bar(stage), tx);
                    const uint32_t a_dst = smem_addr(smem + stage * prm.stage_bytes);
#pragma unroll
                    for (int i = 0; i < kIssuers; ++i) {
                        if (!val[i]) continue;     // empty tile of a short last group: no copy
                        const uint32_t dst = a_dst + (uint32_t)(i * prm.a_bytes);
                        if constexpr (MODE == 1) {
                            // Virtual pixel q reads padded pixel q + kh*Wq + kw.  In halo
                            // mode the box has 128 + kpb - 1 rows: taps kw..kw+kpb-1 are the
                            // same rows shifted by one pixel each, so they share one copy.
                            // (im2win: one tap, t = 0.)
                            tma_load_2d(dst, &amap, full_bar(stage), c0, m0[i] + kh * prm.Wq + kw);
                        } else if constexpr (MODE == 3) {
                            // X[img][c0..c0+63][p0..p0+127] as two 64-pixel boxes.
                            tma_load_3d(dst, &amap, full_bar(stage), wo[i], c0, img[i]);
                            tma_load_3d(dst + 8192u, &amap, full_bar(stage), wo[i] + 64, c0, img[i]);
                        } else {
                            tma_load_im2col_4d(dst, &amap, full_bar(stage), c0, wo[i] * prm.s - prm.p,
                                               ho[i] * prm.s - prm.p, img[i], (uint16_t)kw, (uint16_t)kh);
                        }
                    }
                    if (!prm.b_res) {
                        // Filter chunks of taps t..t+kpb-1, channel block cb: one copy (a 3-D
                        // box in the grid modes; the implicit mode keeps a 2-D map).
                        const uint32_t b_dst = a_dst + (uint32_t)(prm.group * prm.a_bytes);
                        if constexpr (MODE == 1) tma_load_3d(b_dst, &bmap, full_bar(stage), c0, n0, t);
                        else                     tma_load_2d(b_dst, &bmap, full_bar(stage), t * prm.CP + c0, n0);
                    }
                    const bool landed = !prm.sync_copies || mbar_wait(full_bar(stage), phase, abort_flag);
                    ++issued;
                    stage = nstage; phase = nphase; free_now = free_next;
                    if (!landed) { ok = false; break; }   // (the drain below waits for this stage too)
                    if (++cb == prm.n_cchunks) {
                        cb = 0; t += kpb; kw += kpb;
                        if (kw == prm.Kw) { kw = 0; ++kh; }
                    }
                }
            }
            if (!ok) {
                // Let every copy already issued land before the CTA can exit.
                int st = stage;
                uint32_t ph = phase;
                for (int i = 0; i < S && i < issued; ++i) {
                    if (--st < 0) { st = S - 1; ph ^= 1; }
                    mbar_drain_wait(full_bar(st), ph);
                }
            }
            if (prm.b_res) mbar_drain_wait(bres_bar, 0);
        }
    } else if (warp <= kIssuers) {
        // ------------------------------------------------------------ MMA issuers
        const int is = warp - 1;
        if (lane == 0 && is < prm.group) {
            // MODE 3: the pixel operand is MN-major (instruction descriptor bit 16).
            constexpr uint32_t idesc = umma_idesc_f16(BF16, kTcBlockM, BN) | (MODE == 3 ? (1u << 16) : 0u);
            int stage = 0, acc = 0, a_stage = 0;
            uint32_t phase = 0, acc_phase = 0, a_phase = 0;
            bool ok = true, issued_any = false, ready_now = false;
            if (prm.b_res && !mbar_wait(bres_bar, 0, abort_flag)) ok = false;
            const uint32_t bres_base = smem_addr(smem + prm.b_res_off);
            TcItem it;
            for (int idx = 0; ok && tc_item<SPLIT>(prm, idx, it); ++idx) {
                const int g = it.g;
                (void)g;
                if (!mbar_wait(acce_bar(is, acc), acc_phase ^ 1, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)((is * nacc + acc) * acc_stride(BN));
                if constexpr (MODE == 4) {
                    // One A stage = this tile's halo for (channel chunk cb, filter rows
                    // kg*khg ..): tap (kh, kw) reads it from row (kh - kg*khg)*Wq + kw
                    // (128 bytes per row; descriptor addresses in 16-byte units).
                    const int Kh = prm.taps / prm.Kw;
                    bool first = true;
                    for (int cb = 0; cb < prm.n_cchunks && ok; ++cb)
                        for (int kg = 0; kg < prm.n_khg && ok; ++kg) {
                            const uint32_t afull = smem_addr(&abars[a_stage]);
                            if (!mbar_wait(afull, a_phase, abort_flag)) { ok = false; break; }
                            tc_fence_after();
                            const uint64_t a_desc = sw128_kmajor_desc(smem_addr(
                                smem + prm.a_ring_off + a_stage * prm.a_stage_bytes + is * prm.a_bytes));
                            const int kh1 = min(Kh, (kg + 1) * prm.khg);
                            for (int kh = kg * prm.khg; kh < kh1 && ok; ++kh)
                                for (int kw = 0; kw < prm.Kw; ++kw) {
                                    const int t = kh * prm.Kw + kw;
                                    uint32_t b_addr;
                                    if (prm.b_res) {
                                        b_addr = bres_base + (uint32_t)((cb * prm.taps + t) * Cfg::kBBytes);
                                    } else {
                                        if (!mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
                                        tc_fence_after();
                                        b_addr = smem_addr(smem + stage * prm.stage_bytes);
                                    }
                                    const uint64_t b_desc = sw128_kmajor_desc(b_addr);
                                    const uint64_t a_off = (uint64_t)(((kh - kg * prm.khg) * prm.Wq + kw) * 8);
#pragma unroll
                                    for (int k = 0; k < kTcBlockK / 16; ++k)
                                        umma_f16(d_tmem, a_desc + a_off + (uint64_t)(2 * k), b_desc + (uint64_t)(2 * k),
                                                 idesc, (!first || k > 0) ? 1u : 0u);
                                    first = false;
                                    issued_any = true;
                                    if (!prm.b_res) {
                                        umma_commit(empty_bar(stage));
                                        if (++stage == S) { stage = 0; phase ^= 1; }
                                    }
                                }
                            if (!ok) break;
                            umma_commit(smem_addr(&abars[kMaxAStages + a_stage]));
                            if (++a_stage == prm.a_stages) { a_stage = 0; a_phase ^= 1; }
                        }
                    if (!ok) break;
                    umma_commit(accf_bar(is, acc));
                    if (++acc == nacc) { acc = 0; acc_phase ^= 1; }
                    continue;
                }
                int cb = it.k0 % prm.n_cchunks, t = (it.k0 / prm.n_cchunks) * kpb;
                for (int sp = it.k0; sp < it.k1; ++sp) {
                    if (!ready_now && !mbar_wait(full_bar(stage), phase, abort_flag)) { ok = false; break; }
                    // Probe the next slot before issuing this stage's MMAs (its answer
                    // is used one stage later).
                    const int nstage = stage + 1 == S ? 0 : stage + 1;
                    const uint32_t nphase = stage + 1 == S ? phase ^ 1 : phase;
                    const bool ready_next = mbar_test_wait(full_bar(nstage), nphase);
                    tc_fence_after();
                    const uint32_t st_base = smem_addr(smem + stage * prm.stage_bytes);
                    const uint64_t a_desc = sw128_kmajor_desc(st_base + (uint32_t)(is * prm.a_bytes));
                    const uint64_t b_desc = sw128_kmajor_desc(
                        prm.b_res ? bres_base + (uint32_t)((cb * prm.taps + t) * Cfg::kBBytes)
                                  : st_base + (uint32_t)(prm.group * prm.a_bytes));
                    if constexpr (MODE == 3) {
                        // M = output channels (the filter chunk, K-major), N = pixels
                        // (this tile's X chunk, MN-major: 16 K rows = 2 KB per step).
                        const uint64_t x_desc = sw128_mnmajor_desc(st_base + (uint32_t)(is * prm.a_bytes), 8192u);
#pragma unroll
                        for (int k = 0; k < kTcBlockK / 16; ++k)
                            umma_f16(d_tmem, b_desc + (uint64_t)(2 * k), x_desc + (uint64_t)(128 * k), idesc,
                                     (sp > it.k0 || k > 0) ? 1u : 0u);
                    } else {
                        for (int i = 0; i < kpb; ++i) {
                            // Halo: tap kw0+i reads the A tile from row i (128 bytes per row).
                            // Descriptor start addresses are in 16-byte units.
#pragma unroll
                            for (int k = 0; k < kTcBlockK / 16; ++k) {
                                umma_f16(d_tmem, a_desc + (uint64_t)(i * 8 + 2 * k),
                                         b_desc + (uint64_t)(i * (Cfg::kBBytes >> 4) + 2 * k), idesc,
                                         (sp > it.k0 || i > 0 || k > 0) ? 1u : 0u);
                            }
                        }
                    }
                    issued_any = true;
                    umma_commit(empty_bar(stage));
                    stage = nstage; phase = nphase; ready_now = ready_next;
                    if (++cb == prm.n_cchunks) { cb = 0; t += kpb; }
                }
                if (!ok) break;
                umma_commit(accf_bar(is, acc));
                if (++acc == nacc) { acc = 0; acc_phase ^= 1; }
            }
            if (!ok && issued_any) {
                umma_commit(drain_bar(is));
                mbar_drain_wait(drain_bar(is), 0);
            }
        }
    } else if (warp < 1 + kIssuers + 4 * prm.n_egroups) {
        // ------------------------------------------------------------ epilogue
        // Groups of four warps (which tiles a group drains: below).  Warp q
        // of a group owns TMEM lanes 32q..32q+31, i.e. pixels
        // 32q..32q+31 of the tile, and works on its own: each 32-column chunk
        // (32 channels x its 32 pixels) is rounded, transposed through the
        // warp's 2 KB of shared memory as [channel][pixel] and written as
        // 64-byte runs of one channel (16-byte stores; 8-byte stores over the
        // virtual grid, where a 4-pixel group is all-valid or all-junk when
        // Wo % 4 == 0).  Two chunks are loaded from TMEM per wait.  The
        // per-tile barrier only ANDs the wait results so that a group's four
        // warps leave together.
        const int ew = warp - 1 - kIssuers;             // 0 .. 4 * n_egroups - 1
        const int eg = ew >> 2;                         // epilogue group
        const int quarter = warp & 3;                   // TMEM lane quarter this warp may access
        uint16_t* wst = reinterpret_cast<uint16_t*>(smem + prm.epi_off + ew * kEpiWarpBytes);
        // Every accumulator buffer (issuer is, buffer acc) is drained by one
        // group only, so its uses are waited for in order: with two groups,
        // group e takes issuer e's tiles of every item; with three (n_acc = 3),
        // group e takes both tiles of the items idx = e, e + 3, ..., whose
        // buffer is acc = idx % 3 = e.  Use j = idx / n_acc of a buffer
        // completes its barriers' phase j.
        const bool by_item = prm.n_egroups == 3;
        const int istep = by_item ? 3 : 1;
        const int is_lo = by_item ? 0 : eg, is_hi = by_item ? prm.group : eg + 1;
        TcItem it;
        bool go = by_item || eg < prm.group;
        for (int idx = by_item ? eg : 0; go && tc_item<SPLIT>(prm, idx, it); idx += istep) {
          const int acc = idx % nacc;
          const uint32_t acc_phase = (uint32_t)(idx / nacc) & 1u;
          for (int is = is_lo; is < is_hi; ++is) {
            const int g = it.g;
            const bool got = mbar_wait(accf_bar(is, acc), acc_phase, abort_flag);
            if (!named_bar_and(1 + eg, 128, got)) { go = false; break; }
            tc_fence_after();
            int nt_, mg_;
            tile_of(prm, g, nt_, mg_);
            const int n0 = nt_ * BN;
            const int m0 = (mg_ * prm.group + is) * kTcBlockM;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                   (uint32_t)((is * nacc + acc) * acc_stride(BN));
            if constexpr (MODE == 3) {
                // Lane = output channel co0 + lane; columns = the tile's pixels p0..
                // of one image.  Each 64-pixel half goes through the warp's 4 KB
                // box in shared memory (128-byte rows, 128-byte swizzle, so the
                // 16-byte writes of 8 lanes cover all banks) and leaves as one TMA
                // store of 32 channels x 64 pixels; the store clips the pixel and
                // channel tails.
                const int mt = m0 / kTcBlockM;
                const int img = mt / prm.n_pt, p0 = (mt - img * prm.n_pt) * kTcBlockM;
                const int co0 = n0 + quarter * 32;
                const bool live = img < prm.N && co0 < prm.Co;
                const uint32_t wbuf = smem_addr(smem + prm.epi_off + ew * kEpi1x1WarpBytes);
                const float bl = (prm.bias && co0 + lane < prm.Co) ? load_bias<BF16>(prm.bias, co0 + lane) : 0.f;
#pragma unroll 1
                for (int h = 0; h < BN / 64; ++h) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(t_row + h * 64, v0);
                    tmem_ld_32x32b_x32(t_row + h * 64 + 32, v1);
                    tmem_ld_wait();
                    if (!live || p0 + h * 64 >= prm.HoWo) continue;   // warp-uniform
                    if (prm.bias) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            v0[j] = __float_as_uint(__uint_as_float(v0[j]) + bl);
                            v1[j] = __float_as_uint(__uint_as_float(v1[j]) + bl);
                        }
                    }
                    const uint32_t row = wbuf + (uint32_t)lane * 128u;
                    if (prm.out32) {
                        // fp32 output: two stores of 32 channels x 32 pixels (128-byte rows).
#pragma unroll
                        for (int sub = 0; sub < 2; ++sub) {
                            const uint32_t(&v)[32] = sub == 0 ? v0 : v1;
                            if (p0 + h * 64 + sub * 32 >= prm.HoWo) break;   // warp-uniform
                            if (lane == 0) bulk_wait_read_all();
                            __syncwarp();
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                st_shared_v4(row + (uint32_t)((c ^ (lane & 7)) * 16), v[4 * c], v[4 * c + 1],
                                             v[4 * c + 2], v[4 * c + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_3d(&ymap, wbuf, p0 + h * 64 + sub * 32, co0, img);
                                bulk_commit_group();
                            }
                        }
                        continue;
                    }
                    if (lane == 0) bulk_wait_read_all();              // the box is free again
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t(&v)[32] = c < 4 ? v0 : v1;
                        uint32_t h4[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float lo = __uint_as_float(v[(c & 3) * 8 + 2 * j]);
                            const float hi = __uint_as_float(v[(c & 3) * 8 + 2 * j + 1]);
                            if (BF16) {
                                const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
                                h4[j] = *reinterpret_cast<const uint32_t*>(&b2);
                            } else {
                                const __half2 f2 = __floats2half2_rn(lo, hi);
                                h4[j] = *reinterpret_cast<const uint32_t*>(&f2);
                            }
                        }
                        st_shared_v4(row + (uint32_t)((c ^ (lane & 7)) * 16), h4[0], h4[1], h4[2], h4[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&ymap, wbuf, p0 + h * 64, co0, img);
                        bulk_commit_group();
                    }
                }
            } else {
            const int mw = m0 + quarter * 32;
            // Channels this tile stores: a 176-wide tile's last 32-column chunk
            // reaches 16 columns past it.
            const int co_end = min(prm.Co, n0 + BN);
            // Store geometry: this lane's piece of the warp's 32 pixels (vector
            // paths) or its own pixel (scalar path), as element offsets into Y.
            bool v_ok, p_ok;
            long long voff, poff;
            int vpc, vrow0;
            if constexpr (MODE == 1 || MODE == 4) {
                vpc = lane & 7; vrow0 = lane >> 3;
                const int qg = mw + 4 * vpc;
                const int ng = fdiv(prm.fd_hpwq, qg), rg = qg - ng * prm.HpWq;
                const int yg = fdiv(prm.fd_wq, rg), xg = rg - yg * prm.Wq;
                v_ok = ng < prm.N && yg < prm.Ho && xg < prm.Wo;
                voff = (long long)ng * prm.Co * prm.HoWo + yg * prm.Wo + xg;
                const int qp = mw + lane;
                const int np = fdiv(prm.fd_hpwq, qp), rp = qp - np * prm.HpWq;
                const int yp = fdiv(prm.fd_wq, rp), xp = rp - yp * prm.Wq;
                p_ok = np < prm.N && yp < prm.Ho && xp < prm.Wo;
                poff = (long long)np * prm.Co * prm.HoWo + yp * prm.Wo + xp;
            } else {
                vpc = lane & 3; vrow0 = lane >> 2;
                const int mg = mw + 8 * vpc;
                v_ok = mg < prm.M;
                const int img = v_ok ? fdiv(prm.fd_howo, mg) : 0;
                const int r = v_ok ? mg - img * prm.HoWo : 0;
                voff = ((long long)img * prm.Co) * prm.HoWo + r;
                const int m = mw + lane;
                p_ok = m < prm.M;
                const int imgp = p_ok ? fdiv(prm.fd_howo, m) : 0;
                const int rp = p_ok ? m - imgp * prm.HoWo : 0;
                poff = ((long long)imgp * prm.Co) * prm.HoWo + rp;
            }
            auto cvt = [](float f) -> uint16_t {
                if (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(f));
                return __half_as_ushort(__float2half_rn(f));
            };
            // Register j of a chunk is channel cob + j of this lane's pixel.
            // fp32 output: 16 channels x 32 pixels (2 KB) per pass.
            auto emit32 = [&](const uint32_t (&v)[32], int cob) {
                float* const y32 = static_cast<float*>(prm.y);
                float* const wf = reinterpret_cast<float*>(wst);
#pragma unroll
                for (int hlf = 0; hlf < 2; ++hlf) {
                    const int c16 = cob + hlf * 16;
                    if (prm.vec_store) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) wf[j * 32 + lane] = __uint_as_float(v[hlf * 16 + j]);
                        __syncwarp();
                        if constexpr (MODE == 1 || MODE == 4) {
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const int row = vrow0 + 4 * i;
                                if (v_ok && c16 + row < co_end)
                                    *reinterpret_cast<float4*>(y32 + voff + (long long)(c16 + row) * prm.HoWo) =
                                        *reinterpret_cast<const float4*>(wf + row * 32 + 4 * vpc);
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < 2; ++i) {
                                const int row = vrow0 + 8 * i;
                                if (v_ok && c16 + row < co_end) {
                                    float4* dst = reinterpret_cast<float4*>(y32 + voff + (long long)(c16 + row) * prm.HoWo);
                                    const float4* src = reinterpret_cast<const float4*>(wf + row * 32 + 8 * vpc);
                                    dst[0] = src[0];
                                    dst[1] = src[1];
                                }
                            }
                        }
                        __syncwarp();
                    } else if (p_ok) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c16 + j < co_end) y32[poff + (long long)(c16 + j) * prm.HoWo] = __uint_as_float(v[hlf * 16 + j]);
                    }
                }
            };
            auto emit = [&](uint32_t (&v)[32], int cc) {
                const int cob = n0 + cc * 32;
                if (prm.bias) {
                    // The bias of channel cob + lane is loaded by lane `lane` and broadcast.
                    const float bl = cob + lane < prm.Co ? load_bias<BF16>(prm.bias, cob + lane) : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        v[j] = __float_as_uint(__uint_as_float(v[j]) + __shfl_sync(0xffffffffu, bl, j));
                }
                if (prm.out32) {
                    emit32(v, cob);
                    return;
                }
                uint16_t* const yout = static_cast<uint16_t*>(prm.y);
                if (prm.vec_store) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) wst[j * 32 + lane] = cvt(__uint_as_float(v[j]));
                    __syncwarp();
                    if constexpr (MODE == 1 || MODE == 4) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int row = vrow0 + 4 * i;
                            if (v_ok && cob + row < co_end)
                                *reinterpret_cast<uint2*>(yout + voff + (long long)(cob + row) * prm.HoWo) =
                                    *reinterpret_cast<const uint2*>(wst + row * 32 + 4 * vpc);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const int row = vrow0 + 8 * i;
                            if (v_ok && cob + row < co_end)
                                *reinterpret_cast<uint4*>(yout + voff + (long long)(cob + row) * prm.HoWo) =
                                    *reinterpret_cast<const uint4*>(wst + row * 32 + 8 * vpc);
                        }
                    }
                    __syncwarp();
                } else if (p_ok) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (cob + j < co_end) yout[poff + (long long)(cob + j) * prm.HoWo] = cvt(__uint_as_float(v[j]));
                }
            };
            // Split tail: contributor CTA c's partial accumulators are block
            // (c - 1)*group + eg of prm.part, laid out [channel chunk of 32]
            // [4-channel column q][pixel 0..127][4] fp32, so that a warp (32
            // consecutive pixels) reads and writes 512 contiguous bytes per access.
            const int pix = quarter * 32 + lane;
            auto pidx = [&](int chunk, int q) { return ((long long)(chunk * 8 + q) * kTcBlockM + pix) * 4; };
            auto part_block = [&](int c) { return prm.part + ((long long)(c - 1) * prm.group + is) * ((long long)kTcBlockM * BN); };
            auto flag_of = [&](int c) { return prm.flags + (long long)(c - 1) * prm.group + is; };
            bool emit_y = true, add_parts = false;
            if (SPLIT && it.tg >= 0 && !it.owner) {
                // Contributor: store the partial sums, then publish this call's epoch.
                float* dst = part_block(blockIdx.x);
#pragma unroll 1
                for (int cc = 0; cc < BN / 32; cc += 2) {
                    uint32_t v0[32], v1[32];
                    tmem_ld_32x32b_x32(t_row + cc * 32, v0);
                    tmem_ld_32x32b_x32(t_row + (cc + 1) * 32, v1);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        *reinterpret_cast<uint4*>(dst + pidx(cc, q)) =
                            make_uint4(v0[4 * q], v0[4 * q + 1], v0[4 * q + 2], v0[4 * q + 3]);
                        *reinterpret_cast<uint4*>(dst + pidx(cc + 1, q)) =
                            make_uint4(v1[4 * q], v1[4 * q + 1], v1[4 * q + 2], v1[4 * q + 3]);
                    }
                }
                __threadfence();                              // this row before the flag
                named_bar_sync(1 + eg, 128);                  // the group's 128 rows are written
                if ((ew & 3) == 0 && lane == 0) {
                    __threadfence();
                    *reinterpret_cast<volatile unsigned long long*>(flag_of(blockIdx.x)) = prm.epoch;
                }
                emit_y = false;
            } else if (SPLIT && it.tg >= 0 && it.n_contrib > 1) {
                // Owner: wait (bounded) until every other contributor has published.
                bool okf = true;
                if ((ew & 3) == 0 && lane == 0)
                    for (int c = it.c_first + 1; c < it.c_first + it.n_contrib && okf; ++c)
                        if (tail_begin(prm, c) < tail_begin(prm, c + 1))   // CTAs with an empty share add nothing
                            okf = flag_wait(flag_of(c), prm.epoch, abort_flag);
                if (!named_bar_and(1 + eg, 128, okf)) { go = false; break; }
                __threadfence();
                add_parts = true;
            }
            if (emit_y) {
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; cc += 2) {
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(t_row + cc * 32, v0);
                tmem_ld_32x32b_x32(t_row + (cc + 1) * 32, v1);
                tmem_ld_wait();
                if (SPLIT && add_parts) {
                    // One 32-channel chunk at a time keeps 8 loads (32 registers) in flight.
                    for (int c = it.c_first + 1; c < it.c_first + it.n_contrib; ++c) {
                        if (tail_begin(prm, c) == tail_begin(prm, c + 1)) continue;
                        const float* src = part_block(c);
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            uint32_t(&v)[32] = h == 0 ? v0 : v1;
                            float4 pa[8];
#pragma unroll
                            for (int q = 0; q < 8; ++q) pa[q] = __ldcg(reinterpret_cast<const float4*>(src + pidx(cc + h, q)));
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                v[4 * q] = __float_as_uint(__uint_as_float(v[4 * q]) + pa[q].x);
                                v[4 * q + 1] = __float_as_uint(__uint_as_float(v[4 * q + 1]) + pa[q].y);
                                v[4 * q + 2] = __float_as_uint(__uint_as_float(v[4 * q + 2]) + pa[q].z);
                                v[4 * q + 3] = __float_as_uint(__uint_as_float(v[4 * q + 3]) + pa[q].w);
                            }
                        }
                    }
                }
                emit(v0, cc);
                emit(v1, cc + 1);
            }
            }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(is, acc));
          }
        }
        // MODE 3: the TMA stores of this warp complete before the CTA exits.
        if constexpr (MODE == 3) {
            if (lane == 0) bulk_wait_all();
        }
    } else {
        // ------------------------------------------------------------ halo builders (MODE 4)
        // Each A stage: wait until both issuers have released the slot, build
        // this warp's share of the group's halo regions, make the generic-proxy
        // stores visible to the tensor core (async proxy), arrive.
        if constexpr (MODE == 4) {
            const int tw = warp - kTcThreads / 32;     // (two epilogue groups in this mode)
            int a_stage = 0;
            uint32_t a_phase = 0, slot_phases = 0;
            bool ok = true;
            const uint32_t slot_base = smem_addr(smem + prm.stg_off + tw * prm.n_slots * kSegBytes);
            const uint32_t discard =
                smem_addr(smem + prm.stg_off + kTransposerWarps * prm.n_slots * kSegBytes + tw * 128);
            const uint32_t slot_bar0 = smem_addr(&sbars[tw * kMaxSlots]);
            TcItem it;
            for (int idx = 0; ok && tc_item<SPLIT>(prm, idx, it); ++idx) {
                const int g = it.g;
                int nt_, mg_;
                tile_of(prm, g, nt_, mg_);
                const int mt0 = mg_ * prm.group;
                int n_val = 0;
                for (int i = 0; i < prm.group; ++i) n_val += (mt0 + i < prm.n_m_tiles) ? 1 : 0;
                for (int cb = 0; cb < prm.n_cchunks && ok; ++cb)
                    for (int kg = 0; kg < prm.n_khg; ++kg) {
                        if (!mbar_wait(smem_addr(&abars[kMaxAStages + a_stage]), a_phase ^ 1, abort_flag)) {
                            ok = false;
                            break;
                        }
                        const uint32_t base = smem_addr(smem + prm.a_ring_off + a_stage * prm.a_stage_bytes);
                        if (prm.staged) {
                            build_halo_stage_staged(prm, &amap, tw, lane, base, slot_base, slot_bar0, slot_phases,
                                                    discard, mt0, n_val, cb, kg);
                        } else switch (prm.vecw) {
                            case 8: build_halo_stage<8>(prm, tw, lane, base, mt0, n_val, cb, kg); break;
                            case 4: build_halo_stage<4>(prm, tw, lane, base, mt0, n_val, cb, kg); break;
                            case 2: build_halo_stage<2>(prm, tw, lane, base, mt0, n_val, cb, kg); break;
                            default: build_halo_stage<1>(prm, tw, lane, base, mt0, n_val, cb, kg); break;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_addr(&abars[a_stage]));
                        if (++a_stage == prm.a_stages) { a_stage = 0; a_phase ^= 1; }
                    }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
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
cudaError_t wait_limit_set_tc(cudaStream_t st, uint64_t ns) { return wait_limit_set(st, ns); }

// Whether the MODE 4 rings fit for this shape with tile pairs (the larger
// case): two A stages of the smallest halo (one filter row) and three
// streamed filter chunks.
bool halo_plan_fits(const conv2d_desc& d) {
    const int rows = (kTcBlockM + d.Kw - 1 + 7) / 8 * 8;
    const int budget = kSmemLimit - 1024 - kEpiBytes - kBarBytes;
    const int stg = ((long long)d.H * d.W) % 8 == 0 ? kTransposerWarps * (kSegBytes + 128) : 0;
    return 2 * (kIssuers * rows * 128) + 3 * d.BN * kTcBlockK * 2 + stg <= budget;
}

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
static cudaError_t launch_tc_inst(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y,
                                  const TcParams& prm, int grid, int smem, cudaStream_t st) {
    // The split-tail protocol is compiled only into the kernels that run it
    // (modes 0 and 1), so the others carry none of its code or registers.
    auto kern = conv_tc_kernel<BN, BF16, MODE, false>;
    if constexpr ((MODE == 0 || MODE == 1) && BN % 64 == 0) {
        if (prm.split) kern = conv_tc_kernel<BN, BF16, MODE, true>;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int threads = 32 * (1 + kIssuers + 4 * prm.n_egroups) + (MODE == 4 ? 32 * kTransposerWarps : 0);
    return launch_after(kern, dim3(grid), dim3(threads), smem, st, a, b, y, prm);
}

template <bool BF16, int MODE>
static cudaError_t launch_tc_bn(int BN, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y,
                                const TcParams& prm, int grid, int smem, cudaStream_t st) {
    if constexpr (MODE == 3) {                 // 128 output channels x 128 pixels only
        return BN == 128 ? launch_tc_inst<128, BF16, 3>(a, b, y, prm, grid, smem, st) : cudaErrorInvalidValue;
    } else {
        switch (BN) {
            case 64:  return launch_tc_inst<64, BF16, MODE>(a, b, y, prm, grid, smem, st);
            case 128: return launch_tc_inst<128, BF16, MODE>(a, b, y, prm, grid, smem, st);
            case 176:
                if constexpr (MODE == 0 || MODE == 1) return launch_tc_inst<176, BF16, MODE>(a, b, y, prm, grid, smem, st);
                return cudaErrorInvalidValue;
            default:  return launch_tc_inst<256, BF16, MODE>(a, b, y, prm, grid, smem, st);
        }
    }
}

template <bool BF16>
static cudaError_t launch_tc_mode(int BN, int amode, const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& y,
                                  const TcParams& prm, int grid, int smem, cudaStream_t st) {
    switch (amode) {
        case 0:  return launch_tc_bn<BF16, 0>(BN, a, b, y, prm, grid, smem, st);
        case 3:  return launch_tc_bn<BF16, 3>(BN, a, b, y, prm, grid, smem, st);
        case 4:  return launch_tc_bn<BF16, 4>(BN, a, b, y, prm, grid, smem, st);
        default: return launch_tc_bn<BF16, 1>(BN, a, b, y, prm, grid, smem, st);
    }
}

// Split-tail workspace: fp32 partial sums (128 pixels x BN channels) and one
// 64-bit flag per tile of each of the grid - 1 share boundaries.
size_t tc_split_bytes(int grid, int group, int BN) {
    if (grid < 2) return 0;
    const size_t blocks = (size_t)(grid - 1) * group;
    return align_up(blocks * kTcBlockM * BN * 4, 256) + blocks * 8;
}

// Bytes of split-tail workspace a launch of this descriptor on `n_sm` SMs
// uses (0 when its tile groups divide evenly enough): the same tile geometry
// as launch_conv_tc.
size_t tc_split_need(const conv2d_desc& d, int n_sm) {
    const bool grid_rows = d.algo == CONV2D_ALGO_PADDED_TC || d.algo == CONV2D_ALGO_IM2WIN_TC;
    const long long m = grid_rows ? (long long)(d.N - 1) * d.Hp * d.Wq + (long long)(d.Ho - 1) * d.Wq + d.Wo
                                  : (long long)d.N * d.Ho * d.Wo;
    const long long m_tiles = (m + kTcBlockM - 1) / kTcBlockM, n_tiles = (d.Co + d.BN - 1) / d.BN;
    const int group = m_tiles * n_tiles >= 2LL * n_sm ? kIssuers : 1;
    const long long n_groups = (m_tiles + group - 1) / group * n_tiles;
    const long long grid = n_sm < n_groups ? n_sm : n_groups;
    if (n_groups <= grid || n_groups % grid == 0) return 0;
    const long long waves = (n_groups + grid - 1) / grid;
    if ((double)n_groups / grid / waves >= 0.95) return 0;
    return tc_split_bytes((int)grid, group, d.BN);
}

// A value no flag of an earlier call (this process or another) is likely to
// hold: the call count, offset by the time the library first ran.
static unsigned long long next_epoch() {
    static std::atomic<unsigned long long> counter{0};
    static const unsigned long long base =
        (unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() * 1000003ull;
    return base + 2 * counter.fetch_add(1) + 1;
}

conv2d_status launch_conv_tc(const conv2d_desc& d, const void* src, const void* wq, void* y, int amode,
                             cudaStream_t st, void* split_ws, size_t split_bytes) {
    const bool im2win = amode == 1;
    auto enc_tiled = reinterpret_cast<PFN_encodeTiled_t>(driver_entry("cuTensorMapEncodeTiled"));
    auto enc_im2col = reinterpret_cast<PFN_encodeIm2col_t>(driver_entry("cuTensorMapEncodeIm2col"));
    if (!enc_tiled || !enc_im2col) return CONV2D_ERR_CUDA;
    const CUtensorMapDataType dt =
        d.dtype == CONV2D_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;

    CUtensorMap amap, bmap, ymap;
    // Ring layout.  A stage holds the A chunks of the tiles of a group and,
    // unless the filter is resident, the B chunks they share.
    // Padded mode puts kpb neighbouring taps of one filter row in a stage,
    // around one halo A tile (128 + kpb - 1 pixel rows) per tile: each stage
    // costs the producer and MMA threads a fixed run of waits, copies and a
    // commit, so fewer stages with more MMAs each feed the tensor core better.
    const int n_cchunks = d.CP / kTcBlockK;
    const int b_chunk = d.BN * kTcBlockK * 2;
    const bool halo = amode == 2;
    const bool halo4 = amode == 4;                 // halo tiles built from NCHW X in the kernel
    const bool grid_rows = amode == 1 || amode == 2 || halo4;
    const bool gemm1x1 = amode == 3;
    const int n_pt = (d.H * d.W + kTcBlockM - 1) / kTcBlockM;   // 1x1 GEMM: pixel tiles per image
    const int n_n_tiles = (d.Co + d.BN - 1) / d.BN;
    const int n_sm = device_sm_count();
    // Last virtual row that is an output, plus one (grid modes).
    const int m_end = grid_rows ? (d.N - 1) * d.Hp * d.Wq + (d.Ho - 1) * d.Wq + d.Wo : 0;
    const int n_m_tiles =
        gemm1x1 ? d.N * n_pt : ((grid_rows ? m_end : d.N * d.Ho * d.Wo) + kTcBlockM - 1) / kTcBlockM;
    // Pairs of tiles share B and keep two MMA issuers busy; with fewer than
    // two tiles per SM, single tiles keep every SM busy instead.
    int group = (long long)n_m_tiles * n_n_tiles >= 2LL * n_sm ? kIssuers : 1;
    // Epilogue groups: three (a third buffer of BN columns per issuer in
    // TMEM: 2 x 3 x 64 columns with tile pairs, 1 x 3 x 128 with single tiles)
    // where storing the output, not the MMAs, bounds the kernel.
    int n_eg = 2;
    if (!halo4 && !gemm1x1 && !d.tune_split && d.tune_epi_groups == 3) {
        if (d.BN == 64 && group == kIssuers) n_eg = 3;
        else if (d.BN <= 128) { n_eg = 3; group = 1; }
    }
    const int epi_region = gemm1x1 ? kEpi1x1Bytes : n_eg * 4 * kEpiWarpBytes;
    const int budget = kSmemLimit - 1024 - epi_region - kBarBytes;
    // Ring plan for a budget: halo width kpb (largest divisor of Kw leaving at
    // least 2 stages: a halo stage holds kpb taps' MMAs, so two of them keep
    // the pipe busier than three narrow ones; measured on the K=3 layer with
    // 128 output channels), stage size and depth.
    auto plan = [&](int bud, bool bres, int& kpb_o, int& rows_o, int& stages_o) {
        kpb_o = 1; rows_o = kTcBlockM;
        auto stage_of = [&](int rows, int c) { return group * rows * 128 + (bres ? 0 : c * b_chunk); };
        if (halo) {
            for (int c = d.Kw; c >= 2; --c) {
                if (d.Kw % c) continue;
                const int rows = (kTcBlockM + c - 1 + 7) / 8 * 8;
                if (bud / stage_of(rows, c) >= 2) { kpb_o = c; rows_o = rows; break; }
            }
        }
        stages_o = bud / stage_of(rows_o, kpb_o);
        if (stages_o > kMaxStages) stages_o = kMaxStages;
    };
    // The filter slice stays resident when there is one channel tile and the
    // ring keeps at least 3 stages beside it.
    const int bres_bytes = n_cchunks * d.taps * b_chunk;
    int kpb = 1, a_rows = kTcBlockM, stages = 0;
    bool b_res = false;
    if (n_n_tiles == 1 && bres_bytes < budget && !d.tune_no_resident) {
        plan(budget - bres_bytes, true, kpb, a_rows, stages);
        b_res = stages >= 3;
    }
    if (!b_res) plan(budget, false, kpb, a_rows, stages);
    int stage_bytes = group * a_rows * 128 + (b_res ? 0 : kpb * b_chunk);
    // MODE 4: A ring of halo regions (two stages), B streamed (>= 3 stages)
    // or resident; the largest filter-row group whose halo fits.
    int khg = 0, halo_rows = 0, a_stage_bytes = 0, n_slots = 0, stg_bytes = 0;
    const int a_stages4 = d.tune_stages == 1 ? 1 : 2;
    const bool staged = halo4 && ((long long)d.H * d.W) % 8 == 0;   // flat TMA boxes need a 16-byte plane pitch
    if (halo4) {
        b_res = false;
        stages = 0;
        // Largest filter-row group first; two staging slots per builder warp
        // before one; a resident filter before a streamed one.
        for (int g = d.Kh; g >= 1 && !khg; --g) {
            const int rows = (kTcBlockM + (g - 1) * d.Wq + d.Kw - 1 + 7) / 8 * 8;
            const int ast = group * rows * 128;
            for (int ns = staged ? kMaxSlots : 0; ns >= (staged ? 1 : 0) && !khg; --ns) {
                const int stg = staged ? (kTransposerWarps * (ns * kSegBytes + 128) + 1023) / 1024 * 1024 : 0;
                if (n_n_tiles == 1 && !d.tune_no_resident && a_stages4 * ast + bres_bytes + stg <= budget) {
                    b_res = true;
                    stages = 1;
                } else if (a_stages4 * ast + 3 * b_chunk + stg <= budget) {
                    stages = (budget - a_stages4 * ast - stg) / b_chunk;
                    if (stages > kMaxStages) stages = kMaxStages;
                } else {
                    continue;
                }
                khg = g; halo_rows = rows; a_stage_bytes = ast; n_slots = ns; stg_bytes = stg;
            }
        }
        if (!khg) return CONV2D_ERR_UNSUPPORTED;
        stage_bytes = b_chunk;
        kpb = 1;
    }
    if (stages < (halo4 ? 1 : 2)) return CONV2D_ERR_UNSUPPORTED;
    if (d.tune_stages > 0 && stages > d.tune_stages) {   // ablation: a shallower ring
        stages = d.tune_stages;
        if (!halo4) stage_bytes = group * a_rows * 128 + (b_res ? 0 : kpb * b_chunk);
    }
    const int n_acc = n_eg == 3 ? 3 : (2 * kIssuers * acc_stride(d.BN) <= 512 ? 2 : 1);

    CUresult r;
    if (halo4) {
        // A is built in the kernel.  Staged builders read X as [N][Ci][H*W] in
        // boxes of kSeg pixels x 64 channels (zero past H*W and Ci, no swizzle).
        r = CUDA_SUCCESS;
        if (staged) {
            const cuuint64_t P = (cuuint64_t)d.H * d.W;
            cuuint64_t xdims[3] = {P, (cuuint64_t)d.Ci, (cuuint64_t)d.N};
            cuuint64_t xstr[2] = {P * 2, P * 2 * (cuuint64_t)d.Ci};
            cuuint32_t xbox[3] = {(cuuint32_t)kSeg, (cuuint32_t)kTcBlockK, 1};
            cuuint32_t xestr[3] = {1, 1, 1};
            r = enc_tiled(&amap, dt, 3, const_cast<void*>(src), xdims, xstr, xbox, xestr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        }
    } else if (im2win) {
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
    } else if (gemm1x1) {
        // X as [N][Ci][P]: boxes of 64 pixels x 64 channels (rows past P or Ci read as zero).
        const cuuint64_t P = (cuuint64_t)d.H * d.W;
        cuuint64_t xdims[3] = {P, (cuuint64_t)d.Ci, (cuuint64_t)d.N};
        cuuint64_t xstr[2] = {P * 2, P * 2 * (cuuint64_t)d.Ci};
        cuuint32_t xbox[3] = {64, (cuuint32_t)kTcBlockK, 1};
        cuuint32_t xestr[3] = {1, 1, 1};
        r = enc_tiled(&amap, dt, 3, const_cast<void*>(src), xdims, xstr, xbox, xestr, CU_TENSOR_MAP_INTERLEAVE_NONE,
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
    if (gemm1x1) {
        // The caller's filter [Co][Ci] as is (no repack): boxes of 64 channels x 128 output channels.
        cuuint64_t bdims[2] = {(cuuint64_t)d.Ci, (cuuint64_t)d.Co};
        cuuint64_t bstr[1] = {(cuuint64_t)d.Ci * 2};
        cuuint32_t bbox[2] = {(cuuint32_t)kTcBlockK, (cuuint32_t)d.BN};
        cuuint32_t bestr[2] = {1, 1};
        r = enc_tiled(&bmap, dt, 2, const_cast<void*>(wq), bdims, bstr, bbox, bestr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (grid_rows && !halo4) {
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
    if (gemm1x1) {
        // Y as [N][Co][P]: store boxes of 64 pixels x 32 channels (one epilogue warp's lanes).
        const cuuint64_t P = (cuuint64_t)d.H * d.W;
        // fp32 Y: boxes of 32 pixels x 32 channels (128-byte rows as well).
        const bool o32 = d.out_dtype == CONV2D_F32;
        const cuuint64_t ye = o32 ? 4 : 2;
        cuuint64_t ydims[3] = {P, (cuuint64_t)d.Co, (cuuint64_t)d.N};
        cuuint64_t ystr[2] = {P * ye, P * ye * (cuuint64_t)d.Co};
        cuuint32_t ybox[3] = {o32 ? 32u : 64u, 32, 1};
        cuuint32_t yestr[3] = {1, 1, 1};
        r = enc_tiled(&ymap, o32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : dt, 3, y, ydims, ystr, ybox, yestr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
    } else {
        if (halo4 && !staged) amap = bmap;   // unused
        ymap = amap;   // unused by the other modes
    }

    TcParams prm{};
    // M runs over output pixels, or over the virtual grid up to the last output (grid modes).
    prm.M = grid_rows ? m_end : d.N * d.Ho * d.Wo;
    prm.N = d.N;
    prm.Wq = d.Wq;
    prm.HpWq = d.Hp * d.Wq;
    prm.HoWo = d.Ho * d.Wo; prm.Ho = d.Ho; prm.Wo = d.Wo; prm.Co = d.Co;
    prm.n_n_tiles = n_n_tiles;
    prm.fd_wq = make_fastdiv(prm.Wq > 0 ? prm.Wq : 1);
    prm.fd_hpwq = make_fastdiv(prm.HpWq > 0 ? prm.HpWq : 1);
    prm.fd_howo = make_fastdiv(prm.HoWo > 0 ? prm.HoWo : 1);
    prm.fd_nnt = make_fastdiv(n_n_tiles > 0 ? n_n_tiles : 1);
    prm.n_m_tiles = n_m_tiles;
    prm.group = group;
    prm.n_groups = (n_m_tiles + group - 1) / group * n_n_tiles;
    prm.n_cchunks = n_cchunks;
    prm.CP = d.CP; prm.Kw = d.Kw; prm.s = d.s; prm.p = d.p;
    prm.amode = amode;
    prm.kpb = kpb;
    prm.stages = stages;
    prm.stage_bytes = stage_bytes;
    prm.a_bytes = a_rows * 128;
    prm.n_sp = halo ? d.Kh * (d.Kw / kpb) * n_cchunks : d.taps * n_cchunks;
    prm.n_acc = n_acc;
    prm.n_egroups = n_eg;
    prm.epi_bytes = epi_region;
    prm.taps = d.taps;
    prm.b_res = b_res ? 1 : 0;
    prm.b_res_off = stages * stage_bytes;
    if (halo4) {
        // [B ring][A ring][resident filter][epilogue][barriers]
        prm.a_ring_off = (int)align_up((size_t)(b_res ? 0 : stages * stage_bytes), 1024);
        prm.a_stages = a_stages4;
        prm.a_stage_bytes = a_stage_bytes;
        prm.a_bytes = halo_rows * 128;
        prm.halo_rows = halo_rows;
        prm.khg = khg;
        prm.n_khg = (d.Kh + khg - 1) / khg;
        prm.stg_off = prm.a_ring_off + a_stages4 * a_stage_bytes;
        prm.staged = staged ? 1 : 0;
        prm.n_slots = n_slots;
        prm.b_res_off = prm.stg_off + stg_bytes;
        prm.x = src;
        prm.Ci = d.Ci; prm.H = d.H; prm.W = d.W;
        prm.vecw = d.halo_v;
    }
    prm.epi_off = prm.b_res_off + (b_res ? bres_bytes : 0);
    prm.n_pt = n_pt;
    prm.raster = d.tune_raster;
    prm.sync_copies = d.tune_sync_copies;
    prm.n_mg = (n_m_tiles + group - 1) / group;
    prm.y = y;
    prm.bias = d.bias;
    prm.out32 = d.out_dtype == CONV2D_F32 ? 1 : 0;
    if (grid_rows)
        prm.vec_store = ((d.Wo % 4) == 0 && (d.Wq % 4) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) ? 1 : 0;
    else
        prm.vec_store = ((prm.HoWo % 8) == 0 && (reinterpret_cast<uintptr_t>(y) & 15) == 0) ? 1 : 0;
    // At least half the SM's shared memory, so that one CTA runs per SM (it
    // may take all of TMEM).
    int smem = prm.epi_off + epi_region + kBarBytes + 1024;
    if (smem > kSmemLimit) return CONV2D_ERR_UNSUPPORTED;
    if (smem < kSmemLimit / 2 + 4096) smem = kSmemLimit / 2 + 4096;
    int grid = n_sm;
    if (grid > prm.n_groups) grid = prm.n_groups;
    // Split tail (opt-in): when the groups do not divide evenly over the CTAs
    // (the last wave leaves some SMs idle for a whole group) and that costs
    // more than 5 %, the stages of the last partial wave are spread over all
    // CTAs.
    prm.split = 0;
    prm.g_dp = prm.n_groups;
    prm.t_stages = 0;
    if ((amode == 0 || amode == 1 || amode == 2) && d.tune_split && d.BN % 64 == 0 && prm.n_groups > grid &&
        prm.n_groups % grid != 0) {
        const int waves = (prm.n_groups + grid - 1) / grid;
        const double balance = (double)prm.n_groups / grid / waves;
        const size_t need = tc_split_bytes(grid, group, d.BN);
        if (balance < 0.95 && split_ws && need <= split_bytes) {
            prm.split = 1;
            prm.g_dp = prm.n_groups / grid * grid;
            prm.t_stages = (long long)(prm.n_groups - prm.g_dp) * prm.n_sp;
            prm.part = static_cast<float*>(split_ws);
            prm.flags = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(split_ws) +
                                                              align_up((size_t)(grid - 1) * group * kTcBlockM * d.BN * 4, 256));
            prm.epoch = next_epoch();
        }
    }

    const bool bf = d.dtype == CONV2D_BF16;
    cudaError_t e = bf ? launch_tc_mode<true>(d.BN, amode, amap, bmap, ymap, prm, grid, smem, st)
                       : launch_tc_mode<false>(d.BN, amode, amap, bmap, ymap, prm, grid, smem, st);
    return e == cudaSuccess ? CONV2D_OK : CONV2D_ERR_CUDA;
}

}  // namespace conv2d_gb300
