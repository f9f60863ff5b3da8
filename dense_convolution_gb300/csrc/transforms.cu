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

namespace conv2d_gb300 {

// ---------------------------------------------------------------- fp32 strips
// One thread writes one 16-byte vector (4 consecutive strip elements); a warp
// writes 512 contiguous bytes.  Reads walk Kh neighbouring rows and are served
// by L1/L2.
__global__ void __launch_bounds__(256) im2win_strips_f32_kernel(const float* __restrict__ x,
                                                                float4* __restrict__ xw, int Ci, int H, int W,
                                                                int Ho, int Kh, int s, int p, int Wp, int Lp,
                                                                long long total_vec) {
    const int Lv = Lp >> 2;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total_vec;
         q += (long long)gridDim.x * blockDim.x) {
        long long strip = q / Lv;
        int e = (int)(q - strip * Lv) * 4;
        int ho = (int)(strip % Ho);
        long long nc = strip / Ho;                      // n*Ci + ci
        const float* plane = x + nc * (long long)H * W;
        int kx = e / Kh, u = e - kx * Kh;
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            int y = ho * s + u - p, xx = kx - p;
            float val = 0.f;
            if (kx < Wp && y >= 0 && y < H && xx >= 0 && xx < W) val = __ldg(plane + (long long)y * W + xx);
            v[j] = val;
            if (++u == Kh) { u = 0; ++kx; }
        }
        xw[q] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

cudaError_t launch_im2win_strips_f32(const float* x, float* xw, const conv2d_desc& d, cudaStream_t st) {
    long long total_vec = (long long)d.N * d.Ci * d.Ho * (d.Lp / 4);
    long long blocks = (total_vec + 255) / 256;
    long long cap = (long long)device_sm_count() * 16;
    int grid = (int)(blocks < cap ? blocks : cap);
    if (grid < 1) grid = 1;
    im2win_strips_f32_kernel<<<grid, 256, 0, st>>>(x, reinterpret_cast<float4*>(xw), d.Ci, d.H, d.W, d.Ho, d.Kh,
                                                     d.s, d.p, d.Wp, d.Lp, total_vec);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- 16-bit channels-innermost window
// Tiled version: a block transposes a 64-channel x 32-column tile of one input
// row (reads coalesced along x) and writes it channel-innermost, one 16-byte
// vector (8 channels) per thread.
constexpr int kWinTileC = 64;
constexpr int kWinTileX = 32;

__global__ void __launch_bounds__(256) window_cl16_tiled_kernel(const uint16_t* __restrict__ x,
                                                                uint4* __restrict__ out, int Ci, int H, int W,
                                                                int Ci8, int R, int Wq, int Kh, int s, int p,
                                                                int n_xt, int n_ct) {
    __shared__ uint16_t tile[kWinTileC][kWinTileX + 2];
    long long b = blockIdx.x;
    const int xt = (int)(b % n_xt); b /= n_xt;
    const int ct = (int)(b % n_ct); b /= n_ct;
    const int u = (int)(b % Kh);    b /= Kh;
    const long long nr = b;                              // n*R + r
    const int r = (int)(nr % R);
    const long long n = nr / R;
    const int y = r * s + u - p;
    const int kx0 = xt * kWinTileX, c0 = ct * kWinTileC;
    const bool row_ok = (y >= 0 && y < H);
#pragma unroll
    for (int i = 0; i < (kWinTileC * kWinTileX) / 256; ++i) {
        int e = threadIdx.x + 256 * i;
        int c = e / kWinTileX, k = e % kWinTileX;
        int xx = kx0 + k - p, cc = c0 + c;
        uint16_t v = 0;
        if (row_ok && cc < Ci && xx >= 0 && xx < W) v = x[((n * Ci + cc) * H + y) * (long long)W + xx];
        tile[c][k] = v;
    }
    __syncthreads();
    const int k = threadIdx.x / 8, cg = threadIdx.x % 8;
    const int kx = kx0 + k, cc = c0 + cg * 8;
    if (kx < Wq && cc < Ci8) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = (uint32_t)tile[cg * 8 + 2 * j][k] | ((uint32_t)tile[cg * 8 + 2 * j + 1][k] << 16);
        long long o = ((nr * Wq + kx) * Kh + u) * (long long)Ci8 + cc;
        out[o >> 3] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Small-channel version (Ci8 <= 16): one thread builds one 8-channel vector;
// consecutive threads write consecutive vectors.
__global__ void __launch_bounds__(256) window_cl16_small_kernel(const uint16_t* __restrict__ x,
                                                                uint4* __restrict__ out, int Ci, int H, int W,
                                                                int Ci8, int R, int Wq, int Kh, int s, int p,
                                                                long long total_vec) {
    const int cgs = Ci8 / 8;
    for (long long q = blockIdx.x * (long long)blockDim.x + threadIdx.x; q < total_vec;
         q += (long long)gridDim.x * blockDim.x) {
        long long t = q;
        const int cg = (int)(t % cgs); t /= cgs;
        const int u = (int)(t % Kh);   t /= Kh;
        const int kx = (int)(t % Wq);  t /= Wq;
        const int r = (int)(t % R);
        const long long n = t / R;
        const int y = r * s + u - p, xx = kx - p;
        uint32_t w[4] = {0, 0, 0, 0};
        if (y >= 0 && y < H && xx >= 0 && xx < W) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                int c = cg * 8 + j;
                uint32_t v = c < Ci ? x[((n * Ci + c) * H + y) * (long long)W + xx] : 0u;
                w[j >> 1] |= v << (16 * (j & 1));
            }
        }
        out[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_window_cl16(const void* x, void* out, int N, int Ci, int H, int W, int Ci8, int R, int Wq,
                               int Kh, int s, int p, cudaStream_t st) {
    const uint16_t* xi = static_cast<const uint16_t*>(x);
    uint4* o = static_cast<uint4*>(out);
    if (Ci8 <= 16) {
        long long total_vec = (long long)N * R * Wq * Kh * (Ci8 / 8);
        long long blocks = (total_vec + 255) / 256, cap = (long long)device_sm_count() * 16;
        int grid = (int)(blocks < cap ? blocks : cap);
        window_cl16_small_kernel<<<grid < 1 ? 1 : grid, 256, 0, st>>>(xi, o, Ci, H, W, Ci8, R, Wq, Kh, s, p,
                                                                       total_vec);
    } else {
        int n_xt = (Wq + kWinTileX - 1) / kWinTileX, n_ct = (Ci8 + kWinTileC - 1) / kWinTileC;
        long long blocks = (long long)n_xt * n_ct * Kh * N * R;
        if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        window_cl16_tiled_kernel<<<(unsigned)blocks, 256, 0, st>>>(xi, o, Ci, H, W, Ci8, R, Wq, Kh, s, p, n_xt,
                                                                    n_ct);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------- filter repacks
// Tensor-core filter: wq[co][t][c], c in [0, CP).
//   im2win   t = kw, c = u*Ci8 + ci  (the window tensor's (u, ci) column order)
//   implicit t = kh*Kw + kw, c = ci
// Entries outside the real filter are zero.
__global__ void pack_filter_tc_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ wq, int Co, int Ci,
                                      int Kh, int Kw, int Ci8, int taps, int CP, int im2win, long long total) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(i % CP);
        const int t = (int)((i / CP) % taps);
        const int co = (int)(i / ((long long)CP * taps));
        int ci, kh, kw;
        if (im2win) { kw = t; kh = c / Ci8; ci = c - kh * Ci8; }
        else        { kh = t / Kw; kw = t - kh * Kw; ci = c; }
        uint16_t v = 0;
        if (ci < Ci && kh < Kh) v = w[(((long long)co * Ci + ci) * Kh + kh) * Kw + kw];
        wq[i] = v;
    }
}

cudaError_t launch_pack_filter_tc(const void* w, void* wq, const conv2d_desc& d, bool im2win, cudaStream_t st) {
    long long total = (long long)d.Co * d.taps * d.CP;
    long long blocks = (total + 255) / 256, cap = (long long)device_sm_count() * 8;
    int grid = (int)(blocks < cap ? blocks : cap);
    pack_filter_tc_kernel<<<grid < 1 ? 1 : grid, 256, 0, st>>>(static_cast<const uint16_t*>(w),
                                                                static_cast<uint16_t*>(wq), d.Co, d.Ci, d.Kh,
                                                                d.Kw, d.Ci8, d.taps, d.CP, im2win ? 1 : 0, total);
    return cudaGetLastError();
}

// CUDA-core filter: wq[cb][ci][kh][kw][j] = w[cb*BCO + j][ci][kh][kw], BCO = 16 * warps
// output channels per block, zero past Co.  A block's slice for a run of
// input channels is then one contiguous range.
__global__ void pack_filter_f32_kernel(const float* __restrict__ w, float* __restrict__ wq, int Co, int Ci,
                                       int KK, int BCO, long long total) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(i % BCO);
        long long r = i / BCO;
        const int k = (int)(r % KK); r /= KK;
        const int ci = (int)(r % Ci);
        const int cb = (int)(r / Ci);
        const int co = cb * BCO + j;
        wq[i] = co < Co ? w[((long long)co * Ci + ci) * KK + k] : 0.f;
    }
}

cudaError_t launch_pack_filter_f32(const float* w, float* wq, const conv2d_desc& d, cudaStream_t st) {
    const int BCO = 16 * d.cc_warps;
    const int ncb = (d.Co + BCO - 1) / BCO;
    long long total = (long long)ncb * d.Ci * d.Kh * d.Kw * BCO;
    long long blocks = (total + 255) / 256, cap = (long long)device_sm_count() * 8;
    int grid = (int)(blocks < cap ? blocks : cap);
    pack_filter_f32_kernel<<<grid < 1 ? 1 : grid, 256, 0, st>>>(w, wq, d.Co, d.Ci, d.Kh * d.Kw, BCO, total);
    return cudaGetLastError();
}

}  // namespace conv2d_gb300
