// Data transforms that feed the convolution kernels.
//
//  - im2win strips, fp32 ("Enabling Memory-efficient Im2win Convolution with
//    Multi-precision Support on GPU CUDA and Tensor Cores", Sec. III-B,
//    Eq. (2), 0-based, with zero padding): for every (n, ci, ho) a strip whose
//    element kx*Kh + u is Xpad[n][ci][ho*s + u][kx], kx in [0, W+2p).
//  - channels-innermost window tensor, 16-bit (the NHWC arrangement the same
//    paper uses on tensor cores, Sec. III-D): out[n][r][kx][u][c] =
//    Xpad[n][c][r*s + u][kx], channels padded with zeros to a multiple of 8.
//    With Kh = 1, s = 1, p = 0 it is a plain NCHW -> NHWC copy.
//  - filter repacks into the K order each convolution kernel consumes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace conv2d_gb300 {

// ---------------------------------------------------------------- fp32 strips
// A block makes the strips of `rows` (up to kStripRows) consecutive output rows of one
// (n, ci) plane.  It first stages the input rows those strips read —
// (rows - 1)*s + Kh rows of W floats, zero rows for the padding above and
// below — with 16-byte loads where the rows allow (W % 4 == 0), then writes
// each strip as 16-byte vectors, consecutive threads on consecutive vectors:
// strip element e = kx*Kh + u is staged row (r*s + u) at column kx - p (zero
// outside [0, W)).
constexpr int kStripRows = 32;
constexpr long long kStripSmemTarget = 48 * 1024;   // several blocks per SM

__global__ void __launch_bounds__(256) im2win_strips_f32_kernel(const float* __restrict__ x,
                                                                float4* __restrict__ xw, int Ci, int H, int W,
                                                                int Ho, int Kh, int s, int p, int Wp, int Lp,
                                                                int rows, int n_rb, int vec_ok) {
    extern __shared__ __align__(16) float srows[];            // [n_y][W]
    pdl_launch_dependents();
    const int rb = blockIdx.x % n_rb;
    const long long nc = blockIdx.x / n_rb;                   // n*Ci + ci
    const int r0 = rb * rows, nrows = min(rows, Ho - r0);
    const int n_y = (nrows - 1) * s + Kh;
    const int y_lo = r0 * s - p;
    const float* plane = x + nc * (long long)H * W;
    if (vec_ok) {
        const int wv = W >> 2;
        for (int i = threadIdx.x; i < n_y * wv; i += blockDim.x) {
            const int yi = i / wv, v = i - yi * wv;
            const int y = y_lo + yi;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (y >= 0 && y < H) val = __ldg(reinterpret_cast<const float4*>(plane + (long long)y * W) + v);
            reinterpret_cast<float4*>(srows + yi * W)[v] = val;
        }
    } else {
        for (int i = threadIdx.x; i < n_y * W; i += blockDim.x) {
            const int yi = i / W, xx = i - yi * W;
            const int y = y_lo + yi;
            srows[i] = (y >= 0 && y < H) ? __ldg(plane + (long long)y * W + xx) : 0.f;
        }
    }
    __syncthreads();
    const int Lv = Lp >> 2;
    float4* out = xw + (nc * Ho + r0) * (long long)Lv;
    for (int q = threadIdx.x; q < nrows * Lv; q += blockDim.x) {
        const int r = q / Lv, e0 = (q - r * Lv) * 4;
        int kx = e0 / Kh, u = e0 - kx * Kh;
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int xx = kx - p;
            v[j] = (kx < Wp && xx >= 0 && xx < W) ? srows[(r * s + u) * W + xx] : 0.f;
            if (++u == Kh) { u = 0; ++kx; }
        }
        out[q] = make_float4(v[0], v[1], v[2], v[3]);
    }
    pdl_wait();   // complete only after the filter repack launched before us
}

cudaError_t launch_im2win_strips_f32(const float* x, float* xw, const conv2d_desc& d, cudaStream_t st, bool pdl) {
    const long long total_vec = (long long)d.N * d.Ci * d.Ho * (d.Lp / 4);
    if (total_vec > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    int rows = kStripRows;
    while (rows > 1 && (long long)((rows - 1) * d.s + d.Kh) * d.W * 4 > kStripSmemTarget) --rows;
    const int n_rb = (d.Ho + rows - 1) / rows;
    const long long blocks = (long long)d.N * d.Ci * n_rb;
    const long long smem = (long long)((rows - 1) * d.s + d.Kh) * d.W * 4;
    if (blocks > 0x7fffffffLL || smem > kStripSmemMax) return cudaErrorInvalidConfiguration;
    cudaError_t e = cudaFuncSetAttribute(im2win_strips_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    const int vec_ok = (d.W % 4 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) ? 1 : 0;
    return launch_chain(pdl, im2win_strips_f32_kernel, dim3((unsigned)blocks), dim3(256), (size_t)smem, st, x,
                        reinterpret_cast<float4*>(xw), d.Ci, d.H, d.W, d.Ho, d.Kh, d.s, d.p, d.Wp, d.Lp, rows,
                        n_rb, vec_ok);
}

// ---------------------------------------------------------------- 16-bit NCHW -> NHWC (channels padded to 8)
// Batched transpose of [C][P] planes (P = H*W) into [P][C8]: a block moves a
// 64-channel x 64-pixel tile, reading 16-byte vectors along pixels and
// writing 16-byte vectors along channels (a warp writes 4 x 128 contiguous
// bytes).  The shared tile pitch of 66 halves keeps the column reads at two
// ways of bank conflict.
constexpr int kNhwcTile = 64;
constexpr int kNhwcPitch = 66;

__global__ void __launch_bounds__(256) nchw_to_nhwc16_kernel(const uint16_t* __restrict__ x,
                                                             uint4* __restrict__ out, int C, int C8, int P,
                                                             int vec_ok) {
    __shared__ uint32_t tile[kNhwcTile * kNhwcPitch / 2];
    uint16_t* t16 = reinterpret_cast<uint16_t*>(tile);
    pdl_launch_dependents();
    const int p0 = blockIdx.x * kNhwcTile, c0 = blockIdx.y * kNhwcTile;
    const long long n = blockIdx.z;
    const uint16_t* xn = x + n * (long long)C * P;
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int c = tid / 8 + 32 * i, pv = (tid % 8) * 8;
        const int cc = c0 + c, pp = p0 + pv;
        uint32_t w[4] = {0, 0, 0, 0};
        if (cc < C) {
            const uint16_t* src = xn + (long long)cc * P + pp;
            if (vec_ok && pp + 8 <= P) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (pp + j < P) w[j >> 1] |= (uint32_t)src[j] << (16 * (j & 1));
            }
        }
        uint32_t* dst = tile + (c * kNhwcPitch + pv) / 2;
        dst[0] = w[0]; dst[1] = w[1]; dst[2] = w[2]; dst[3] = w[3];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int pl = tid / 8 + 32 * i, cg = tid % 8;
        const int pp = p0 + pl, cc = c0 + cg * 8;
        if (pp < P && cc < C8) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                w[j] = (uint32_t)t16[(cg * 8 + 2 * j) * kNhwcPitch + pl] |
                       ((uint32_t)t16[(cg * 8 + 2 * j + 1) * kNhwcPitch + pl] << 16);
            out[((n * P + pp) * C8 + cc) >> 3] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
    pdl_wait();   // complete only after the filter repack launched before us
}

static cudaError_t launch_padded_reg(const void* x, void* out, int N, int C, int C8, int H, int W, int Hp, int Wq,
                                     int p, cudaStream_t st, bool pdl);

cudaError_t launch_nchw_to_nhwc16(const void* x, void* out, int N, int C, int H, int W, int C8, cudaStream_t st,
                                  bool pdl) {
    const int P = H * W;
    // The image plane as one row of P columns, no padding.
    const cudaError_t r = launch_padded_reg(x, out, N, C, C8, 1, P, 1, P, 0, st, pdl);
    if (r != cudaErrorNotSupported) return r;
    const int vec_ok = (P % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) ? 1 : 0;
    dim3 grid((P + kNhwcTile - 1) / kNhwcTile, (C8 + kNhwcTile - 1) / kNhwcTile, N);
    if (grid.z > 65535 || grid.y > 65535) return cudaErrorInvalidConfiguration;
    return launch_chain(pdl, nchw_to_nhwc16_kernel, grid, dim3(256), 0, st, static_cast<const uint16_t*>(x),
                        static_cast<uint4*>(out), C, C8, P, vec_ok);
}

// ---------------------------------------------------------------- 16-bit NCHW -> zero-padded NHWC
// out[n][yy][xx][c] = X[n][c][yy-p][xx-p] (zero outside the image and for
// c >= C), yy in [0, Hp), xx in [0, Wq): every output pixel of the padded
// grid is written, borders included.  A block covers one padded row, 64
// channels and kRowTileX output columns.  It reads the 64 channel rows of the
// image row as 16-byte vectors (8 pixels; when W % 8 == 0) and scatters them
// into a pixel-major shared tile [pixel][64 channels], then writes each
// pixel's channels as 16-byte vectors, consecutive threads on consecutive
// vectors.  The tile's 16-byte channel chunks are XOR-swizzled by the pixel's
// 8-pixel group so that both phases run free of bank conflicts.
constexpr int kRowTileX = 128;
constexpr int kRowTileRows = kRowTileX + 8;   // staged pixels: the tile plus the 8-alignment slack

__device__ __forceinline__ int row_tile_index(int x, int c) {
    return x * 64 + ((((c >> 3) ^ (x >> 3)) & 7) << 3) + (c & 7);
}

__global__ void __launch_bounds__(256) nchw_to_padded_nhwc16_kernel(const uint16_t* __restrict__ x,
                                                                    uint4* __restrict__ out, int C, int C8, int H,
                                                                    int W, int Hp, int Wq, int p, int n_xt,
                                                                    int vec_ok) {
    __shared__ __align__(16) uint16_t tile[kRowTileRows * 64];
    pdl_launch_dependents();
    const int xt = blockIdx.x % n_xt, yy = blockIdx.x / n_xt;
    const int c0 = blockIdx.y * 64;
    const long long n = blockIdx.z;
    const int xq0 = xt * kRowTileX;                          // first output column of the tile
    const int xq_n = min(kRowTileX, Wq - xq0);
    const int cg_n = min(64, C8 - c0) / 8;                   // channel vectors per pixel in this block
    const int y = yy - p;
    const bool row_in = y >= 0 && y < H;
    // Image columns [xa, xhi) cover the tile's interior pixels; xa is xlo
    // rounded down to 8 so that vector loads stay 16-byte aligned.
    const int xlo = max(xq0 - p, 0), xhi = min(xq0 + xq_n - p, W);
    const int xa = xlo & ~7;
    if (row_in && xhi > xlo) {
        const uint16_t* src = x + ((n * C + c0) * H + y) * (long long)W + xa;
        if (vec_ok) {
            const int nv = (xhi - xa + 7) >> 3;              // W % 8 == 0: never past the row end
            for (int i = threadIdx.x; i < 64 * nv; i += blockDim.x) {
                const int c = i / nv, v = i - c * nv;
                uint4 val = make_uint4(0, 0, 0, 0);
                if (c0 + c < C) val = __ldg(reinterpret_cast<const uint4*>(src + (long long)c * H * W) + v);
                const uint32_t w[4] = {val.x, val.y, val.z, val.w};
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    tile[row_tile_index(8 * v + k, c)] = (uint16_t)(w[k >> 1] >> (16 * (k & 1)));
            }
        } else {
            const int span = xhi - xa;
            for (int i = threadIdx.x; i < 64 * span; i += blockDim.x) {
                const int c = i / span, v = i - c * span;
                tile[row_tile_index(v, c)] = (c0 + c < C && xa + v >= xlo) ? src[(long long)c * H * W + v] : 0;
            }
        }
    }
    __syncthreads();
    uint4* dst = out + (((n * Hp + yy) * Wq + xq0) * C8 + c0) / 8;
    for (int i = threadIdx.x; i < xq_n * cg_n; i += blockDim.x) {
        const int xl = i / cg_n, g = i - xl * cg_n;
        const int xw = xq0 + xl - p;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row_in && xw >= 0 && xw < W) v = *reinterpret_cast<const uint4*>(tile + row_tile_index(xw - xa, 8 * g));
        dst[(long long)xl * (C8 / 8) + g] = v;
    }
    pdl_wait();   // complete only after the filter repack launched before us
}

// Register-transposing variant for W % V == 0 (V = 8 or 4 image columns per
// load; X aligned to 2V bytes).  A block makes one segment of one padded row
// (n, yy) for one 64-channel chunk: lane l of warp w takes channel group
// cg = l & 7 (8 channels) and column group 4w + (l >> 3) of the segment.  It
// loads V columns of each of its 8 channel rows (a warp's loads of one
// channel are 4 contiguous pieces), transposes the 8 x V block in registers
// (byte permutes merge the two channels of a pair, pixel by pixel), and
// stores V pixels x 8 channels as 16-byte vectors: the 8 lanes of a column
// group write each pixel's 128 contiguous bytes.  No shared memory.  Border
// and junk columns, padding rows and channels past C are written as zeros
// (a padding row's columns split over its segments; the border columns of an
// image row by its first segment).  With H = 1, Hp = 1, p = 0 and W = H*W of
// the image it is the plain NCHW -> NHWC copy.
template <int V>
__global__ void __launch_bounds__(128) nchw_to_padded_nhwc16_reg_kernel(const uint16_t* __restrict__ x,
                                                                        uint4* __restrict__ out, int C, int C8,
                                                                        int H, int W, int Hp, int Wq, int p,
                                                                        int n_seg) {
    pdl_launch_dependents();
    const int nw = blockDim.x >> 5;
    const int seg = blockIdx.x % n_seg, yy = blockIdx.x / n_seg;
    const long long n = blockIdx.y;
    const int y = yy - p;
    const int cgn = C8 / 8;                                   // 16-byte channel vectors per pixel
    const int g0 = blockIdx.z * 8, ng = min(8, cgn - g0);     // this chunk's vectors
    const int seg_cols = 4 * nw * V;                          // image columns per segment
    uint4* const orow = out + (n * Hp + yy) * (long long)Wq * cgn + g0;
    const uint4 z = make_uint4(0, 0, 0, 0);
    if (y < 0 || y >= H) {
        const int xa = seg * seg_cols, xb = seg == n_seg - 1 ? Wq : min(Wq, xa + seg_cols);
        for (int i = threadIdx.x; i < (xb - xa) * ng; i += blockDim.x)
            orow[(long long)(xa + i / ng) * cgn + i % ng] = z;
        pdl_wait();
        return;
    }
    if (seg == 0) {
        // Columns [0, p) and [W + p, Wq): zc < p is column zc, the others W + zc.
        for (int i = threadIdx.x; i < (Wq - W) * ng; i += blockDim.x) {
            const int zc = i / ng;
            orow[(long long)(zc < p ? zc : W + zc) * cgn + i % ng] = z;
        }
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int cg = lane & 7;
    const int pg = seg * 4 * nw + 4 * w + (lane >> 3);
    if (cg < ng && pg < W / V) {
        const int c = 8 * (g0 + cg), x0 = pg * V;
        const long long plane = (long long)H * W;
        const uint16_t* const src0 = x + (n * C + c) * plane + (long long)y * W + x0;
        uint32_t r[8][V / 2];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (c + k < C) {
                if constexpr (V == 8) {
                    const uint4 t = __ldg(reinterpret_cast<const uint4*>(src0 + k * plane));
                    r[k][0] = t.x; r[k][1] = t.y; r[k][2] = t.z; r[k][3] = t.w;
                } else {
                    const uint2 t = __ldg(reinterpret_cast<const uint2*>(src0 + k * plane));
                    r[k][0] = t.x; r[k][1] = t.y;
                }
            } else {
#pragma unroll
                for (int j = 0; j < V / 2; ++j) r[k][j] = 0;
            }
        }
        // Word j of channel row k holds pixels 2j (low half) and 2j + 1.
        uint4* dst = orow + (long long)(x0 + p) * cgn + cg;
#pragma unroll
        for (int j = 0; j < V / 2; ++j) {
            uint32_t lo[4], hi[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                lo[kk] = __byte_perm(r[2 * kk][j], r[2 * kk + 1][j], 0x5410);   // pixel 2j: channels 2kk, 2kk+1
                hi[kk] = __byte_perm(r[2 * kk][j], r[2 * kk + 1][j], 0x7632);   // pixel 2j + 1
            }
            dst[(long long)(2 * j) * cgn] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            dst[(long long)(2 * j + 1) * cgn] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        }
    }
    pdl_wait();   // complete only after the filter repack launched before us
}

// Launch of the register-transposing copy, or cudaErrorNotSupported when the
// shape or the alignment does not allow it.
static cudaError_t launch_padded_reg(const void* x, void* out, int N, int C, int C8, int H, int W, int Hp, int Wq,
                                     int p, cudaStream_t st, bool pdl) {
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x);
    const int v = (W % 8 == 0 && (xa & 15) == 0) ? 8 : ((W % 4 == 0 && (xa & 7) == 0) ? 4 : 0);
    if (!v || N > 65535 || C8 % 8 != 0 || (C8 + 63) / 64 > 65535) return cudaErrorNotSupported;
    const int n_pg = W / v;
    const int nw = n_pg <= 4 ? 1 : (n_pg <= 8 ? 2 : 4);       // warps per block: 4 column groups each
    const int n_seg = (n_pg + 4 * nw - 1) / (4 * nw);
    const long long gx = (long long)Hp * n_seg;
    if (gx > 0x7fffffffLL) return cudaErrorNotSupported;
    const dim3 grid((unsigned)gx, (unsigned)N, (unsigned)((C8 + 63) / 64));
    auto kern = v == 8 ? nchw_to_padded_nhwc16_reg_kernel<8> : nchw_to_padded_nhwc16_reg_kernel<4>;
    return launch_chain(pdl, kern, grid, dim3(32 * nw), 0, st, static_cast<const uint16_t*>(x),
                        static_cast<uint4*>(out), C, C8, H, W, Hp, Wq, p, n_seg);
}

cudaError_t launch_nchw_to_padded_nhwc16(const void* x, void* out, const conv2d_desc& d, cudaStream_t st, bool pdl) {
    const cudaError_t r = launch_padded_reg(x, out, d.N, d.Ci, d.Ci8, d.H, d.W, d.Hp, d.Wq, d.p, st, pdl);
    if (r != cudaErrorNotSupported) return r;
    const int n_xt = (d.Wq + kRowTileX - 1) / kRowTileX;
    const long long gx = (long long)n_xt * d.Hp;
    const int vec_ok = (d.W % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) ? 1 : 0;
    dim3 grid((unsigned)gx, (d.Ci8 + 63) / 64, d.N);
    if (gx > 0x7fffffffLL || grid.z > 65535 || grid.y > 65535) return cudaErrorInvalidConfiguration;
    return launch_chain(pdl, nchw_to_padded_nhwc16_kernel, grid, dim3(256), 0, st, static_cast<const uint16_t*>(x),
                        static_cast<uint4*>(out), d.Ci, d.Ci8, d.H, d.W, d.Hp, d.Wq, d.p, n_xt, vec_ok);
}

// ---------------------------------------------------------------- 16-bit channels-innermost window
// Tiled version (Ci8 > 16): a block makes the window-tensor run of one image
// row r and XT consecutive padded columns kx0.., i.e. out[n][r][kx][u][c] for
// all (u, c): one contiguous run of XT*Kh*Ci8 elements.  It stages the Kh
// input rows r*s + u - p, all Ci8 channels (zero past Ci and outside the
// image), columns [xa, xa + XTs) with xa = kx0 - p rounded down to 8, as
// [u][c][col] with 16-byte loads where the rows allow (W % 8 == 0; 8-byte
// loads when W % 4 == 0); then
// transposes 8 channels x 8 columns at a time (ldmatrix .trans) into a second
// buffer laid out like the output run (stmatrix: one 16-byte row per
// (column, u, 8 channels); columns outside the tile go to a discard row); then
// copies that buffer to the output with 16-byte stores, consecutive threads
// on consecutive vectors.
__global__ void __launch_bounds__(256) window_cl16_tiled_kernel(const uint16_t* __restrict__ x,
                                                                uint4* __restrict__ out, int Ci, int H, int W,
                                                                int Ci8, int R, int Wq, int Kh, int s, int p,
                                                                int XT, int XTs, int n_xt, int vec_ok) {
    extern __shared__ __align__(16) uint16_t wsm[];
    uint16_t* in = wsm;                                   // [Kh][Ci8][XTs]
    uint16_t* ob = wsm + (size_t)Kh * Ci8 * XTs;          // [XT][Kh][Ci8], then a 16-byte discard row
    pdl_launch_dependents();
    const int xt = blockIdx.x % n_xt;
    const long long nr = blockIdx.x / n_xt;               // n*R + r
    const int r = (int)(nr % R);
    const long long n = nr / R;
    const int kx0 = xt * XT;
    const int xt_n = min(XT, Wq - kx0);
    int xa = kx0 - p;
    xa = xa >= 0 ? (xa & ~7) : -((-xa + 7) & ~7);        // floor to a multiple of 8
    const int nv = XTs / 8;
    for (int i = threadIdx.x; i < Kh * Ci8 * nv; i += 256) {
        const int v = i % nv, uc = i / nv;
        const int c = uc % Ci8, u = uc / Ci8;
        const int y = r * s + u - p, x0 = xa + 8 * v;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (c < Ci && y >= 0 && y < H) {
            const uint16_t* src = x + ((n * Ci + c) * H + y) * (long long)W;
            if (vec_ok == 2 && x0 >= 0 && x0 + 8 <= W) {
                val = __ldg(reinterpret_cast<const uint4*>(src + x0));
            } else if (vec_ok == 1 && x0 >= 0 && x0 + 8 <= W) {       // rows 8-byte aligned (W % 4 == 0)
                const uint2 lo = __ldg(reinterpret_cast<const uint2*>(src + x0));
                const uint2 hi = __ldg(reinterpret_cast<const uint2*>(src + x0 + 4));
                val = make_uint4(lo.x, lo.y, hi.x, hi.y);
            } else {
                uint32_t w4[4] = {0, 0, 0, 0};
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (x0 + e >= 0 && x0 + e < W) w4[e >> 1] |= (uint32_t)__ldg(src + x0 + e) << (16 * (e & 1));
                val = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
        *reinterpret_cast<uint4*>(in + (size_t)uc * XTs + 8 * v) = val;
    }
    __syncthreads();
    // Transpose: x4 item = (u, 32 channels, 8 columns); lane 8i + j addresses
    // row j (channel) of matrix i for the load and row j (column) for the store.
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c32 = (Ci8 + 31) / 32, items = Kh * c32 * nv;
    const uint32_t discard = smem_addr(ob + (size_t)XT * Kh * Ci8);
    for (int it = warp; it < items; it += 8) {
        const int v = it % nv, rest = it / nv;
        const int cq = rest % c32, u = rest / c32;
        const int mi = lane >> 3, j = lane & 7;
        int c = cq * 32 + mi * 8 + j;
        if (c >= Ci8) c = Ci8 - 1;                        // a matrix past Ci8: load any row, store nowhere
        uint32_t q[4];
        ldsm_x4_trans(smem_addr(in + ((size_t)u * Ci8 + c) * XTs + 8 * v), q);
        const int col = xa + 8 * v + j + p - kx0;         // tile column of this lane's row
        const int cg = cq * 32 + mi * 8;
        const bool ok = col >= 0 && col < xt_n && cg < Ci8;
        stsm_x4(ok ? smem_addr(ob + ((size_t)col * Kh + u) * Ci8 + cg) : discard, q);
    }
    __syncthreads();
    const long long run = (long long)xt_n * Kh * Ci8 / 8;  // 16-byte vectors
    uint4* dst = out + ((nr * Wq + kx0) * (long long)Kh * Ci8) / 8;
    for (long long i = threadIdx.x; i < run; i += 256) dst[i] = reinterpret_cast<const uint4*>(ob)[i];
    pdl_wait();   // complete only after the filter repack launched before us
}

// Small-channel version (Ci8 <= 16): the Kh*Ci (row, channel) pairs of a
// padded column are packed densely, c = u*Ci + ci, and rounded up to Ck (a
// multiple of 8); one thread builds one 8-element vector, consecutive
// threads write consecutive vectors.  With Ci a multiple of 8 this is the
// same layout as the tiled version.
__global__ void __launch_bounds__(256) window_cl16_small_kernel(const uint16_t* __restrict__ x,
                                                                uint4* __restrict__ out, int Ci, int H, int W,
                                                                int Ck, int R, int Wq, int Kh, int s, int p,
                                                                long long total_vec) {
    pdl_launch_dependents();
    const int cgs = Ck / 8;
    const int KC = Kh * Ci;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total_vec;
         q += (long long)gridDim.x * blockDim.x) {
        long long t = q;
        const int cg = (int)(t % cgs); t /= cgs;
        const int kx = (int)(t % Wq);  t /= Wq;
        const int r = (int)(t % R);
        const long long n = t / R;
        const int xx = kx - p;
        uint32_t w[4] = {0, 0, 0, 0};
        if (xx >= 0 && xx < W) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = cg * 8 + j;
                const int u = c / Ci, ci = c - u * Ci;
                const int y = r * s + u - p;
                uint32_t v = 0;
                if (c < KC && y >= 0 && y < H) v = x[((n * Ci + ci) * H + y) * (long long)W + xx];
                w[j >> 1] |= v << (16 * (j & 1));
            }
        }
        out[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    pdl_wait();   // complete only after the filter repack launched before us
}

// Small-channel version staged through shared memory: a block covers
// kWinRowsPerBlock consecutive window rows r0.. of one image and kWinRowX
// output columns.  It loads the input rows those window rows need once (they
// overlap: (rows - 1)*s + Kh rows per channel; staged row yi*Ci + ci holds
// X[n][ci][r0*s - p + yi][.], zero outside the image), as 16-byte vectors
// where aligned, then builds each 8-element vector of packed (row, channel)
// pairs from shared memory: pair c = u*Ci + ci of window row r is staged row
// (r - r0)*s*Ci + c.  The row pitch kWinRowPitch (not a multiple of 8 halves)
// spreads rows 8 apart over different banks.
constexpr long long kWindowSmemTarget = 64 * 1024;   // tiled window: both buffers of a block
constexpr int kWinRowX = 128;                 // output columns per block
constexpr int kWinRowCols = kWinRowX + 8;     // staged input columns (the 8-alignment slack)
constexpr int kWinRowPitch = kWinRowCols + 2;
constexpr int kWinRowsPerBlock = 4;

__global__ void __launch_bounds__(256) window_cl16_rows_kernel(const uint16_t* __restrict__ x,
                                                               uint4* __restrict__ out, int Ci, int H, int W, int Ck,
                                                               int R, int Wq, int Kh, int s, int p, int n_xt,
                                                               int n_rb, int vec_ok) {
    extern __shared__ __align__(16) uint16_t rows[];         // [n_y*Ci][kWinRowPitch]
    pdl_launch_dependents();
    const int tid = threadIdx.x;
    const int xt = blockIdx.x % n_xt;
    const int rb = (blockIdx.x / n_xt) % n_rb;
    const int n = blockIdx.x / (n_xt * n_rb);
    const int r0 = rb * kWinRowsPerBlock, nrows = min(kWinRowsPerBlock, R - r0);
    const int kx0 = xt * kWinRowX, kx_n = min(kWinRowX, Wq - kx0);
    const int KC = Kh * Ci;
    const int n_y = (nrows - 1) * s + Kh;                    // staged input rows per channel
    const int y_lo = r0 * s - p;
    int xa = kx0 - p;
    xa = (xa >= 0) ? (xa & ~7) : -((-xa + 7) & ~7);          // floor to a multiple of 8
    constexpr int nv = kWinRowCols / 8;
    const long long plane = (long long)H * W;
    for (int i = tid; i < n_y * Ci * nv; i += 256) {
        const int row = i / nv, v = i - row * nv;
        const int yi = row / Ci, ci = row - yi * Ci;
        const int y = y_lo + yi, x0 = xa + 8 * v;
        uint32_t w[4] = {0, 0, 0, 0};
        if (y >= 0 && y < H) {
            const uint16_t* src = x + ((long long)n * Ci + ci) * plane + (long long)y * W;
            if (vec_ok && x0 >= 0 && x0 + 8 <= W) {
                const uint4 val = __ldg(reinterpret_cast<const uint4*>(src + x0));
                w[0] = val.x; w[1] = val.y; w[2] = val.z; w[3] = val.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (x0 + e >= 0 && x0 + e < W) w[e >> 1] |= (uint32_t)__ldg(src + x0 + e) << (16 * (e & 1));
            }
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(rows + row * kWinRowPitch + 8 * v);
        dst[0] = w[0]; dst[1] = w[1]; dst[2] = w[2]; dst[3] = w[3];
    }
    __syncthreads();
    const int cgs = Ck / 8;
    const int per_row = kx_n * cgs;
    for (int i = tid; i < nrows * per_row; i += 256) {
        const int rr = i / per_row, j = i - rr * per_row;
        const int kxl = j / cgs, cg = j - kxl * cgs;
        const int col = kx0 + kxl - p - xa;                  // in [0, kWinRowCols)
        const uint16_t* base = rows + (rr * s * Ci) * kWinRowPitch + col;
        uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int c = cg * 8 + e;
            if (c < KC) w[e >> 1] |= (uint32_t)base[c * kWinRowPitch] << (16 * (e & 1));
        }
        out[(((long long)n * R + r0 + rr) * Wq + kx0 + kxl) * cgs + cg] = make_uint4(w[0], w[1], w[2], w[3]);
    }
    pdl_wait();   // complete only after the filter repack launched before us
}

cudaError_t launch_window_cl16(const void* x, void* out, int N, int Ci, int H, int W, int Ci8, int Ck, int R,
                               int Wq, int Kh, int s, int p, cudaStream_t st, bool pdl) {
    const uint16_t* xi = static_cast<const uint16_t*>(x);
    uint4* o = static_cast<uint4*>(out);
    const long long row_smem = (long long)((kWinRowsPerBlock - 1) * s + Kh) * Ci * kWinRowPitch * 2;
    const int n_xr = (Wq + kWinRowX - 1) / kWinRowX;
    const int n_rb = (R + kWinRowsPerBlock - 1) / kWinRowsPerBlock;
    const long long blocks = (long long)N * n_rb * n_xr;
    if (Ci8 <= 16 && row_smem <= 96 * 1024 && blocks <= 0x7fffffffLL) {
        cudaError_t e = cudaFuncSetAttribute(window_cl16_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)row_smem);
        if (e != cudaSuccess) return e;
        const int vec_ok = (W % 8 == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) ? 1 : 0;
        return launch_chain(pdl, window_cl16_rows_kernel, dim3((unsigned)blocks), dim3(256), (size_t)row_smem, st, xi, o,
                            Ci, H, W, Ck, R, Wq, Kh, s, p, n_xr, n_rb, vec_ok);
    }
    if (Ci8 <= 16) {
        long long total_vec = (long long)N * R * Wq * (Ck / 8);
        long long blocks = (total_vec + 255) / 256, cap = (long long)device_sm_count() * 16;
        int grid = (int)(blocks < cap ? blocks : cap);
        return launch_chain(pdl, window_cl16_small_kernel, dim3(grid < 1 ? 1 : grid), dim3(256), 0, st, xi, o, Ci, H, W,
                            Ck, R, Wq, Kh, s, p, total_vec);
    } else {
        // Columns per block: as many as keep both buffers within the budget (at least 1).
        const long long per_col = (long long)Kh * Ci8 * 2 * 2;   // staged input + output bytes per column
        int XT = (int)((kWindowSmemTarget - (long long)Kh * Ci8 * 2 * 8 - 16) / per_col);
        if (XT > 64) XT = 64;
        if (XT > Wq) XT = Wq;
        if (XT < 1) XT = 1;
        const int XTs = (XT + 7 + 7) / 8 * 8;
        const long long smem = (long long)Kh * Ci8 * XTs * 2 + (long long)XT * Kh * Ci8 * 2 + 16;
        if (smem > 200 * 1024) return cudaErrorInvalidConfiguration;
        const int n_xt = (Wq + XT - 1) / XT;
        const long long blocks = (long long)n_xt * N * R;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        cudaError_t e = cudaFuncSetAttribute(window_cl16_tiled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        const bool a16 = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
        const int vec_ok = (W % 8 == 0 && a16) ? 2 : ((W % 4 == 0 && a16) ? 1 : 0);
        return launch_chain(pdl, window_cl16_tiled_kernel, dim3((unsigned)blocks), dim3(256), (size_t)smem, st, xi, o,
                            Ci, H, W, Ci8, R, Wq, Kh, s, p, XT, XTs, n_xt, vec_ok);
    }
}

// ---------------------------------------------------------------- filter repacks
// Tensor-core filter: wq[co][t][c], c in [0, CP).
//   im2win   one tap; c = kw*Ck + u*cdiv + ci, the order of a window in the
//            window tensor (cdiv = Ci when its (u, ci) pairs are packed
//            densely, Ci8 otherwise)
//   implicit t = kh*Kw + kw, c = ci
// Entries outside the real filter are zero.  One block per output channel:
// the channel's Ci*Kh*Kw filter (contiguous) is staged in shared memory, then
// the repacked row is written contiguously.
constexpr int kPackSmemElems = 16384;   // 32 KB of 16-bit filter per output channel

__global__ void __launch_bounds__(256) pack_filter_tc_kernel(const uint16_t* __restrict__ w,
                                                             uint16_t* __restrict__ wq, int Ci, int Kh, int Kw,
                                                             int cdiv, int ck, int taps, int CP, int im2win) {
    __shared__ __align__(16) uint16_t fw[kPackSmemElems];
    // First kernel of a call, launched as a programmatic dependent of whatever
    // ran before on the stream: wait for it before touching memory, and only
    // then let the transform behind this kernel start (it reads X at once).
    pdl_wait();
    pdl_launch_dependents();
    const int co = blockIdx.x;
    const int KK = Kh * Kw, n = Ci * KK;
    const uint16_t* src = w + (long long)co * n;
    if ((n & 7) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
        for (int i = threadIdx.x; i < (n >> 3); i += blockDim.x) reinterpret_cast<uint4*>(fw)[i] = __ldg(s4 + i);
    } else {
        for (int i = threadIdx.x; i < n; i += blockDim.x) fw[i] = src[i];
    }
    __syncthreads();
    // One 16-byte vector = 8 consecutive packed channels of one tap.
    uint4* dst = reinterpret_cast<uint4*>(wq + (long long)co * taps * CP);
    const int cpv = CP >> 3, total = taps * cpv;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int t = i / cpv, c0 = (i - t * cpv) * 8;
        uint32_t v[4] = {0, 0, 0, 0};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = c0 + j;
            int ci, kh, kw;
            if (im2win) {
                kw = c / ck;
                const int cc = c - kw * ck;
                kh = cc / cdiv; ci = cc - kh * cdiv;
            } else {
                kh = t / Kw; kw = t - kh * Kw; ci = c;
            }
            const uint32_t h = (ci < Ci && kh < Kh && kw < Kw) ? fw[ci * KK + kh * Kw + kw] : 0u;
            v[j >> 1] |= h << (16 * (j & 1));
        }
        dst[i] = make_uint4(v[0], v[1], v[2], v[3]);
    }
}

cudaError_t launch_pack_filter_tc(const void* w, void* wq, const conv2d_desc& d, bool im2win, cudaStream_t st) {
    if ((long long)d.Ci * d.Kh * d.Kw > kPackSmemElems) return cudaErrorInvalidValue;
    const int cdiv = d.Ci8 <= 16 ? d.Ci : d.Ci8;
    return launch_after(pack_filter_tc_kernel, dim3(d.Co), dim3(256), 0, st, static_cast<const uint16_t*>(w),
                        static_cast<uint16_t*>(wq), d.Ci, d.Kh, d.Kw, cdiv, d.Ck, d.taps, d.CP, im2win ? 1 : 0);
}

// CUDA-core filter: wq[cb][ci][k][j] = w[cb*BCO + j][ci][k] (k = kh*Kw + kw),
// BCO = 32 * warps output channels per block, zero past Co, so that a block's
// slice for a run of input channels is one contiguous range.  One block per
// (cb, ci): reads BCO runs of Kh*Kw floats, writes Kh*Kw*BCO floats in order.
__global__ void __launch_bounds__(256) pack_filter_f32_kernel(const float* __restrict__ w, float* __restrict__ wq,
                                                              int Co, int Ci, int KK, int BCO) {
    pdl_wait();                 // first kernel of a call: see pack_filter_tc_kernel
    pdl_launch_dependents();
    const int ci = blockIdx.x, cb = blockIdx.y;
    float* dst = wq + ((long long)cb * Ci + ci) * KK * BCO;
    const int total = KK * BCO;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int k = i / BCO, j = i - k * BCO;
        const int co = cb * BCO + j;
        dst[i] = co < Co ? __ldg(w + ((long long)co * Ci + ci) * KK + k) : 0.f;
    }
}

cudaError_t launch_pack_filter_f32(const float* w, float* wq, const conv2d_desc& d, cudaStream_t st) {
    const int BCO = 32 * d.cc_warps;
    const int ncb = (d.Co + BCO - 1) / BCO;
    if (ncb > 65535) return cudaErrorInvalidConfiguration;
    return launch_after(pack_filter_f32_kernel, dim3(d.Ci, ncb), dim3(256), 0, st, w, wq, d.Co, d.Ci, d.Kh * d.Kw,
                        BCO);
}

}  // namespace conv2d_gb300
