// C ABI: descriptor creation and validation, per-shape algorithm choice,
// workspace layout and the launch sequence of conv2d_fwd.  Host code only;
// the kernels live in transforms.cu, conv_fp32.cu and conv_tc.cu.
#include <new>
#include <stdint.h>
#include <string.h>

#include "internal.h"

#define CONV2D_API extern "C" __attribute__((visibility("default")))

using namespace conv2d_gb300;

namespace {

constexpr long long kMaxElems = 0x7fffffffLL;   // kernels index tensors with 32-bit element counts

bool is_tc(conv2d_algo a) {
    return a == CONV2D_ALGO_IM2WIN_TC || a == CONV2D_ALGO_IMPLICIT_TC || a == CONV2D_ALGO_PADDED_TC ||
           a == CONV2D_ALGO_IMPLICIT_NCHW_TC;
}

// Padded algorithm geometry: row pitch W+2p, rounded up to 4 when Wo % 4 == 0
// so that 4-pixel output groups never straddle a row (8-byte stores).
// Output-channel tile width of the tensor-core kernel: 64 for Co <= 64, 128
// for Co <= 128; wider layers take the one of 256, 176 and 128 that needs
// the fewest waves of tile groups on this GPU, each wave weighted by the
// group's MMA time (tiles per group x width).  A group is a pair of
// 128-pixel tiles when there are at least two tiles per SM; ties keep the
// wider tile.  176 = 512 / 3 rounded up to 16: three tiles of a 512-channel
// layer instead of two (not with the split tail, whose partial blocks are
// laid out in 64-wide pairs of chunks).
int choose_bn(const conv2d_desc& d, int n_sm) {
    if (d.Co <= 64) return 64;
    if (d.Co <= 128) return 128;
    const long long m_tiles = ((long long)d.N * d.Ho * d.Wo + kTcBlockM - 1) / kTcBlockM;
    int best = 256;
    long long best_t = -1;
    for (int bn : {256, 176, 128}) {
        if (bn == 176 && d.tune_split) continue;
        const long long n_tiles = (d.Co + bn - 1) / bn;
        const int group = m_tiles * n_tiles >= 2LL * n_sm ? 2 : 1;
        const long long groups = (m_tiles + group - 1) / group * n_tiles;
        const long long t = (groups + n_sm - 1) / n_sm * group * bn;
        if (best_t < 0 || t < best_t) { best_t = t; best = bn; }
    }
    return best;
}

int padded_pitch(const conv2d_desc& d) { return d.Wo % 4 == 0 ? (d.Wp + 3) / 4 * 4 : d.Wp; }

// Fraction of the padded grid's virtual pixels that are junk (not outputs).
double padded_waste(const conv2d_desc& d) {
    const double grid = (double)(d.H + 2 * d.p) * padded_pitch(d);
    return 1.0 - (double)d.Ho * d.Wo / grid;
}

// im2win window tensor: channels per padded column (row, channel pairs).
long long window_ck(const conv2d_desc& d) {
    const long long ci8 = (d.Ci + 7) / 8 * 8;
    return ci8 <= 16 ? ((long long)d.Kh * d.Ci + 7) / 8 * 8 : (long long)d.Kh * ci8;
}

// Fraction of the tensor-core K extent that holds real filter taps, for the
// two operand sources (the rest is zero fill up to the 64-element chunk):
// implicit runs Kh*Kw taps of Ci8 channels, im2win one window of Kw*Ck.
double tc_k_efficiency(const conv2d_desc& d, bool im2win) {
    auto up64 = [](long long v) { return (v + kTcBlockK - 1) / kTcBlockK * kTcBlockK; };
    if (im2win) return (double)d.Kh * d.Kw * d.Ci / (double)up64(d.Kw * window_ck(d));
    return (double)d.Ci / (double)up64((d.Ci + 7) / 8 * 8);
}

// im2win virtual grid: Wq output slots per image row, Wq*s window columns per
// row (at least W+2p), rounded up to 4 when Wo % 4 == 0 (8-byte stores).
int window_grid_pitch(const conv2d_desc& d) {
    int wq = (d.Wp + d.s - 1) / d.s;
    if (wq < d.Wo) wq = d.Wo;
    if (d.Wo % 4 == 0) wq = (wq + 3) / 4 * 4;
    return wq;
}

// Shape limits of the tensor-core kernels (im2col-mode TMA corners are 8-bit
// signed for a 4-D map; channel pitch must be a 16-byte multiple).
bool tc_shape_ok(const conv2d_desc& d, bool im2win) {
    if (!im2win) {
        if (d.p > 128 || d.p - (d.Kw - 1) < -128 || d.p - (d.Kh - 1) < -128) return false;
        if (d.p - (d.Kw - 1) > 127 || d.p - (d.Kh - 1) > 127) return false;
        if (d.layout == CONV2D_LAYOUT_NHWC && d.Ci % 8 != 0) return false;
    }
    if (d.Kh > 0xffff || d.Kw > 0xffff) return false;
    return true;
}

// Recorded per-shape choice.  fp32: the im2win strips (the method of the
// im2win paper).  16-bit: the padded path where its halo reuse pays (below);
// otherwise the window tensor only for small channel counts (Ci8 <= 16),
// where its dense (row, channel) packing fills the 64-wide K chunk that a
// 3-channel tap would leave nearly empty, and the channels-last copy for the
// rest: the window tensor is about Kh/s times X, and its transform costs more
// than the copy saves in K fill (measured on GB300, the im2win paper's cv5,
// 96 channels, 5x5: 198.8 us per call on the window path, 113.5 us on the
// channels-last one).
conv2d_algo resolve_auto(const conv2d_desc& d) {
    if (d.dtype == CONV2D_F32) return CONV2D_ALGO_IM2WIN_FP32_CC;
    if (d.layout == CONV2D_LAYOUT_NHWC) return CONV2D_ALGO_IMPLICIT_TC;
    // Stride 1 with two or three taps per filter row: the padded path shares
    // one halo operand tile among neighbouring taps, which wins unless the
    // padded grid adds too many junk rows (measured on GB300: ResNet stage 1
    // and the K=3 sweep layer gain 2-4 %; 1x1 layers, VGG and 5-wide filters,
    // whose halo stages grow to five taps' filter chunks, do not: the K=5
    // sweep layer runs 7 % faster implicit).
    if (d.s == 1 && d.Kw >= 2 && d.Kw <= 3 && padded_waste(d) <= 0.15 && (d.Ci + 7) / 8 * 8 >= 64)
        return CONV2D_ALGO_PADDED_TC;
    const bool imp_ok = tc_shape_ok(d, false), win_ok = tc_shape_ok(d, true);
    const bool small_ci = (d.Ci + 7) / 8 * 8 <= 16;
    if (imp_ok && (!win_ok || !small_ci || tc_k_efficiency(d, false) >= tc_k_efficiency(d, true)))
        return CONV2D_ALGO_IMPLICIT_TC;
    return CONV2D_ALGO_IM2WIN_TC;
}

conv2d_status finalize(conv2d_desc& d) {
    d.algo = d.requested == CONV2D_ALGO_AUTO ? resolve_auto(d) : d.requested;
    const bool tc = is_tc(d.algo);
    if (tc != (d.dtype != CONV2D_F32)) return CONV2D_ERR_BAD_PARAM;
    if (d.layout == CONV2D_LAYOUT_NHWC && d.algo != CONV2D_ALGO_IMPLICIT_TC) return CONV2D_ERR_UNSUPPORTED;
    d.ws_weights = d.ws_input = d.ws_input_off = d.ws_total = 0;
    d.gemm1x1 = false;
    if (d.algo == CONV2D_ALGO_WINOGRAD_FP32_CC) {
        // F(2x2, 3x3): 3x3 filters, stride 1, NCHW input; workspace = the transformed filter.
        if (d.Kh != 3 || d.Kw != 3 || d.s != 1) return CONV2D_ERR_UNSUPPORTED;
        d.ws_weights = winograd_filter_bytes(d);
        d.ws_total = d.prepacked ? 0 : d.ws_weights;
        return CONV2D_OK;
    }
    if (!tc) {
        d.Lp = (d.Wp * d.Kh + 3) & ~3;
        // 32 output channels per warp, 1, 2 or 4 warps; fewer warps when one
        // channel's filter slice for the block would not stay small.
        int warps = d.Co > 64 ? 4 : (d.Co > 32 ? 2 : 1);
        while (warps > 1 && (long long)d.Kh * d.Kw * 32 * warps * 4 > 24 * 1024) warps /= 2;
        d.cc_warps = warps;
        if ((long long)d.Kh * d.Kw * 32 * 4 > 96 * 1024) return CONV2D_ERR_UNSUPPORTED;
        const long long bco = 32LL * warps, ncb = (d.Co + bco - 1) / bco;
        d.ws_weights = (size_t)(ncb * bco * d.Ci * d.Kh * d.Kw * 4);
        if (d.algo == CONV2D_ALGO_IM2WIN_FP32_CC) {
            const long long strips = (long long)d.N * d.Ci * d.Ho * d.Lp;
            if (strips / 4 > kMaxElems) return CONV2D_ERR_UNSUPPORTED;   // 32-bit vector index
            if ((long long)d.Kh * d.W * 4 > kStripSmemMax) return CONV2D_ERR_UNSUPPORTED;   // staged rows
            d.ws_input = (size_t)strips * 4;
        } else {
            if (d.W % 4 != 0) return CONV2D_ERR_UNSUPPORTED;    // 16-byte row pitch for the row copies
            if (d.Kh > 256) return CONV2D_ERR_UNSUPPORTED;
            if (63 * d.s + d.Kw + 6 > 256) return CONV2D_ERR_UNSUPPORTED;   // staged rows fit one box
        }
    } else {
        const bool im2win = d.algo == CONV2D_ALGO_IM2WIN_TC;
        const bool padded = d.algo == CONV2D_ALGO_PADDED_TC;
        if (d.algo == CONV2D_ALGO_IMPLICIT_NCHW_TC && (d.s != 1 || d.layout != CONV2D_LAYOUT_NCHW))
            return CONV2D_ERR_UNSUPPORTED;
        if (padded) {
            if (d.s != 1 || d.layout != CONV2D_LAYOUT_NCHW) return CONV2D_ERR_UNSUPPORTED;
        } else if (!tc_shape_ok(d, im2win)) {
            return CONV2D_ERR_UNSUPPORTED;
        }
        d.Ci8 = (d.Ci + 7) / 8 * 8;
        if (window_ck(d) * d.Kw > kMaxElems) return CONV2D_ERR_UNSUPPORTED;
        d.Ck = (int)window_ck(d);
        d.taps = im2win ? 1 : d.Kh * d.Kw;
        const long long chunk = im2win ? (long long)d.Kw * d.Ck : d.Ci8;
        d.CP = (int)((chunk + kTcBlockK - 1) / kTcBlockK * kTcBlockK);
        d.BN = d.tune_tile_n ? d.tune_tile_n : choose_bn(d, device_sm_count());
        // A 1x1 layer is a GEMM on the NCHW tensors themselves: the TMA maps
        // read X as [N][Ci][H*W] and the filter as [Co][Ci] (16-byte strides).
        d.gemm1x1 = d.algo == CONV2D_ALGO_IMPLICIT_TC && d.layout == CONV2D_LAYOUT_NCHW && d.Kh == 1 &&
                    d.Kw == 1 && d.s == 1 && d.p == 0 && d.Ci % 8 == 0 && ((long long)d.H * d.W) % 8 == 0;
        if (d.gemm1x1) d.BN = 128;   // 128 output channels x 128 pixels per MMA tile
        if (d.BN == 176 && d.tune_split) return CONV2D_ERR_UNSUPPORTED;   // the split's partial layout
        // Implicit GEMM on NCHW input at stride 1: operand tiles are built from X
        // inside the contraction kernel (zero-padded halo over a virtual grid of
        // pitch Wq), so no copy of X is made.  Vector width: the widest that
        // divides W; the pitch is W + 2p rounded up to it (and to 4 when Wo % 4
        // == 0 for the 8-byte stores); the narrowest pitch wins.
        d.nchw_halo = false;
        if (d.algo == CONV2D_ALGO_IMPLICIT_NCHW_TC) {
            if (d.tune_tile_n == 176) return CONV2D_ERR_UNSUPPORTED;   // the in-kernel builders: 64, 128, 256
            d.BN = d.tune_tile_n ? d.tune_tile_n : (d.Co <= 64 ? 64 : (d.Co <= 128 ? 128 : 256));
            int best_v = 0, best_wq = 0;
            for (int v = 8; v >= 1; v /= 2) {
                if (d.W % v) continue;
                const int a = v > (d.Wo % 4 == 0 ? 4 : 1) ? v : (d.Wo % 4 == 0 ? 4 : 1);
                const int wq = (d.Wp + a - 1) / a * a;
                if (!best_v || wq < best_wq) { best_v = v; best_wq = wq; }
            }
            d.halo_v = best_v;
            d.Wq = best_wq;
            d.Hp = d.H + 2 * d.p;
            const long long rows = (long long)d.N * d.Hp * d.Wq;
            d.nchw_halo = rows + (long long)d.Kh * d.Wq + d.Kw + kTcBlockM <= kMaxElems && halo_plan_fits(d);
            if (!d.nchw_halo) return CONV2D_ERR_UNSUPPORTED;
        }
        if ((long long)d.Ci * d.Kh * d.Kw > 16384) return CONV2D_ERR_UNSUPPORTED;   // per-channel filter staging
        if (d.N > 65535) return CONV2D_ERR_UNSUPPORTED;
        const long long wq = (long long)d.Co * d.taps * d.CP;
        if (wq > kMaxElems) return CONV2D_ERR_UNSUPPORTED;
        d.ws_weights = d.gemm1x1 ? 0 : (size_t)wq * 2;
        if (d.gemm1x1) {
            // No workspace: X and the filter are read in place.
        } else if (padded) {
            d.Hp = d.H + 2 * d.p;
            d.Wq = padded_pitch(d);
            const long long rows = (long long)d.N * d.Hp * d.Wq;
            if (rows + (long long)d.Kh * d.Wq + d.Kw + kTcBlockM > kMaxElems) return CONV2D_ERR_UNSUPPORTED;
            if (rows * d.Ci8 > kMaxElems * 4) return CONV2D_ERR_UNSUPPORTED;
            d.ws_input = (size_t)(rows * d.Ci8) * 2;
        } else if (im2win) {
            // Window transform for Ci8 > 16: Kh rows x Ci8 channels of at least 16 staged columns
            // plus one output column per block in shared memory.
            if (d.Ci8 > 16 && (long long)d.Kh * d.Ci8 * (16 * 2 + 2) + 16 > 200 * 1024) return CONV2D_ERR_UNSUPPORTED;
            d.Hp = d.Ho;
            d.Wq = window_grid_pitch(d);
            const long long rows = (long long)d.N * d.Ho * d.Wq;
            if (rows + kTcBlockM > kMaxElems) return CONV2D_ERR_UNSUPPORTED;
            const long long win = rows * d.s * d.Ck;
            if (win > kMaxElems * 4) return CONV2D_ERR_UNSUPPORTED;
            d.ws_input = (size_t)win * 2;
        } else if (d.layout == CONV2D_LAYOUT_NCHW && !d.nchw_halo) {
            d.ws_input = (size_t)((long long)d.N * d.H * d.W * d.Ci8) * 2;
        }
    }
    if (d.prepacked) {   // the filter lives in the caller's packed buffer
        d.ws_input_off = 0;
        d.ws_total = d.ws_input;
    } else {
        d.ws_input_off = d.ws_input ? align_up(d.ws_weights, 1024) : 0;
        d.ws_total = d.ws_input ? d.ws_input_off + d.ws_input : d.ws_weights;
    }
    // Split tail (opt-in; tensor-core modes that take the im2col, padded or
    // window source): room for the partial sums of grid - 1 share boundaries on the
    // current device (a 148-SM one when there is none), when the tile groups
    // leave the last wave short and the total stays within the im2win tensor
    // N*Ci*Ho*(W+2p)*Kh of the im2win paper's Eq. (2).
    d.ws_split_off = d.ws_split = 0;
    const bool splittable = (d.algo == CONV2D_ALGO_IMPLICIT_TC && !d.gemm1x1) || d.algo == CONV2D_ALGO_PADDED_TC ||
                            d.algo == CONV2D_ALGO_IM2WIN_TC;
    if (splittable && d.tune_split && d.BN % 64 == 0) {
        const size_t need = tc_split_need(d, device_sm_count());
        const double cap = 2.0 * d.N * d.Ci * d.Ho * (double)(d.W + 2 * d.p) * d.Kh;
        const size_t off = align_up(d.ws_total, 256);
        if (need && (double)(off + need) <= cap) {
            d.ws_split = need;
            d.ws_split_off = off;
            d.ws_total = off + need;
        }
    }
    return CONV2D_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

CONV2D_API conv2d_status conv2d_desc_create(conv2d_desc_t* out, int N, int Cin, int H, int W, int Cout, int Kh,
                                            int Kw, int stride, int pad, conv2d_dtype dtype, conv2d_algo algo) {
    if (!out) return CONV2D_ERR_NULL_PTR;
    *out = nullptr;
    if (N < 1 || Cin < 1 || H < 1 || W < 1 || Cout < 1 || Kh < 1 || Kw < 1 || stride < 1 || pad < 0)
        return CONV2D_ERR_BAD_PARAM;
    if (dtype != CONV2D_F32 && dtype != CONV2D_F16 && dtype != CONV2D_BF16) return CONV2D_ERR_BAD_PARAM;
    if (algo < CONV2D_ALGO_AUTO || algo > CONV2D_ALGO_WINOGRAD_FP32_CC) return CONV2D_ERR_BAD_PARAM;
    const long long Hp = (long long)H + 2LL * pad, Wp = (long long)W + 2LL * pad;
    if (Hp < Kh || Wp < Kw || Wp > 0x7fffffffLL) return CONV2D_ERR_BAD_PARAM;
    const long long Ho = (Hp - Kh) / stride + 1, Wo = (Wp - Kw) / stride + 1;
    if ((long long)N * Cin * H * W > kMaxElems || (long long)N * Cout * Ho * Wo > kMaxElems ||
        (long long)Cout * Cin * Kh * Kw > kMaxElems)
        return CONV2D_ERR_BAD_PARAM;
    conv2d_desc d{};
    d.N = N; d.Ci = Cin; d.H = H; d.W = W; d.Co = Cout; d.Kh = Kh; d.Kw = Kw; d.s = stride; d.p = pad;
    d.dtype = dtype;
    d.requested = algo;
    d.layout = CONV2D_LAYOUT_NCHW;
    d.out_dtype = dtype;
    d.bias = nullptr;
    d.Ho = (int)Ho; d.Wo = (int)Wo; d.Wp = (int)Wp;
    conv2d_status st = finalize(d);
    if (st != CONV2D_OK) return st;
    conv2d_desc* h = new (std::nothrow) conv2d_desc(d);
    if (!h) return CONV2D_ERR_BAD_PARAM;
    *out = h;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_desc_set_input_layout(conv2d_desc_t d, conv2d_layout layout) {
    if (!d) return CONV2D_ERR_NULL_PTR;
    if (layout != CONV2D_LAYOUT_NCHW && layout != CONV2D_LAYOUT_NHWC) return CONV2D_ERR_BAD_PARAM;
    conv2d_desc t = *d;
    t.layout = layout;
    conv2d_status st = finalize(t);
    if (st != CONV2D_OK) return st;
    *d = t;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_desc_set_output_dtype(conv2d_desc_t d, conv2d_dtype out) {
    if (!d) return CONV2D_ERR_NULL_PTR;
    if (out != d->dtype && !(out == CONV2D_F32 && d->dtype != CONV2D_F32)) return CONV2D_ERR_BAD_PARAM;
    d->out_dtype = out;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_desc_set_bias(conv2d_desc_t d, const void* bias) {
    if (!d) return CONV2D_ERR_NULL_PTR;
    const size_t align = d->dtype == CONV2D_F32 ? 4 : 2;
    if (reinterpret_cast<uintptr_t>(bias) % align) return CONV2D_ERR_MISALIGNED;
    d->bias = bias;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_desc_set_tuning(conv2d_desc_t d, conv2d_tuning knob, int value) {
    if (!d) return CONV2D_ERR_NULL_PTR;
    switch (knob) {
        case CONV2D_TUNE_STAGES:
            if (value < 0 || value > 8) return CONV2D_ERR_BAD_PARAM;
            d->tune_stages = value;
            return CONV2D_OK;
        case CONV2D_TUNE_SYNC_COPIES:
            if (value < 0 || value > 1) return CONV2D_ERR_BAD_PARAM;
            d->tune_sync_copies = value;
            return CONV2D_OK;
        case CONV2D_TUNE_RASTER:
            if (value < 0 || value > 2) return CONV2D_ERR_BAD_PARAM;
            d->tune_raster = value;
            return CONV2D_OK;
        case CONV2D_TUNE_NO_RESIDENT:
            if (value < 0 || value > 1) return CONV2D_ERR_BAD_PARAM;
            d->tune_no_resident = value;
            return CONV2D_OK;
        case CONV2D_TUNE_EPI_GROUPS:
            if (value != 0 && value != 2 && value != 3) return CONV2D_ERR_BAD_PARAM;
            d->tune_epi_groups = value;
            return CONV2D_OK;
        case CONV2D_TUNE_TILE_N: {
            if (value != 0 && value != 64 && value != 128 && value != 176 && value != 256) return CONV2D_ERR_BAD_PARAM;
            conv2d_desc t = *d;
            t.tune_tile_n = value;
            const conv2d_status st = finalize(t);
            if (st != CONV2D_OK) return st;
            *d = t;
            return CONV2D_OK;
        }
        case CONV2D_TUNE_SPLIT: {
            if (value < 0 || value > 1) return CONV2D_ERR_BAD_PARAM;
            conv2d_desc t = *d;
            t.tune_split = value;
            const conv2d_status st = finalize(t);   // the split's workspace comes or goes
            if (st != CONV2D_OK) return st;
            *d = t;
            return CONV2D_OK;
        }
    }
    return CONV2D_ERR_BAD_PARAM;
}

CONV2D_API conv2d_status conv2d_packed_filter_bytes(conv2d_desc_t d, size_t* bytes) {
    if (!d || !bytes) return CONV2D_ERR_NULL_PTR;
    *bytes = d->gemm1x1 ? (size_t)d->Co * d->Ci * 2 : d->ws_weights;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_desc_set_filter_prepacked(conv2d_desc_t d, int prepacked) {
    if (!d) return CONV2D_ERR_NULL_PTR;
    if (prepacked != 0 && prepacked != 1) return CONV2D_ERR_BAD_PARAM;
    conv2d_desc t = *d;
    t.prepacked = prepacked != 0;
    conv2d_status st = finalize(t);
    if (st != CONV2D_OK) return st;
    *d = t;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_pack_filter(conv2d_desc_t dp, const void* w, void* w_packed, void* stream) {
    if (!dp || !w || !w_packed) return CONV2D_ERR_NULL_PTR;
    if (!aligned16(w) || !aligned16(w_packed)) return CONV2D_ERR_MISALIGNED;
    const conv2d_desc& d = *dp;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    switch (d.algo) {
        case CONV2D_ALGO_IM2WIN_FP32_CC:
        case CONV2D_ALGO_IMPLICIT_FP32_CC:
            e = launch_pack_filter_f32(static_cast<const float*>(w), static_cast<float*>(w_packed), d, st);
            break;
        case CONV2D_ALGO_WINOGRAD_FP32_CC:
            e = launch_winograd_filter(d, static_cast<const float*>(w), static_cast<float*>(w_packed), st);
            break;
        case CONV2D_ALGO_IM2WIN_TC:
            e = launch_pack_filter_tc(w, w_packed, d, true, st);
            break;
        default:
            if (d.gemm1x1)   // the 1x1 GEMM reads the filter as given
                e = cudaMemcpyAsync(w_packed, w, (size_t)d.Co * d.Ci * 2, cudaMemcpyDeviceToDevice, st);
            else
                e = launch_pack_filter_tc(w, w_packed, d, false, st);
    }
    return e == cudaSuccess ? CONV2D_OK : CONV2D_ERR_CUDA;
}

CONV2D_API conv2d_status conv2d_desc_destroy(conv2d_desc_t d) {
    delete d;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_out_dims(conv2d_desc_t d, int* Ho, int* Wo) {
    if (!d || !Ho || !Wo) return CONV2D_ERR_NULL_PTR;
    *Ho = d->Ho;
    *Wo = d->Wo;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_workspace_size(conv2d_desc_t d, size_t* bytes) {
    if (!d || !bytes) return CONV2D_ERR_NULL_PTR;
    *bytes = d->ws_total;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_get_algo(conv2d_desc_t d, conv2d_algo* chosen) {
    if (!d || !chosen) return CONV2D_ERR_NULL_PTR;
    *chosen = d->algo;
    return CONV2D_OK;
}

namespace {

// Records an optional event on the stream; false when the record fails.
bool record(void* ev, cudaStream_t st) {
    return !ev || cudaEventRecord(static_cast<cudaEvent_t>(ev), st) == cudaSuccess;
}

conv2d_status fwd_impl(conv2d_desc_t dp, const void* x, const void* w, void* y, void* workspace,
                       size_t workspace_bytes, void* stream, void* ev0, void* ev1) {
    if (!dp || !x || !w || !y) return CONV2D_ERR_NULL_PTR;
    const conv2d_desc& d = *dp;
    if (d.ws_total > 0 && !workspace) return CONV2D_ERR_NULL_PTR;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (workspace && !aligned16(workspace)))
        return CONV2D_ERR_MISALIGNED;
    if (workspace_bytes < d.ws_total) return CONV2D_ERR_WORKSPACE_TOO_SMALL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    // Pre-packed filter: w is already in the kernel's order (conv2d_pack_filter)
    // and the workspace holds only the input-side tensor; the first kernel of
    // the call is then a transform or the contraction itself.
    const bool pre = d.prepacked;
    void* wq = pre ? const_cast<void*>(w) : ws;
    void* win = ws ? ws + d.ws_input_off : nullptr;
    cudaError_t e = cudaSuccess;
    conv2d_status s = CONV2D_OK;
    switch (d.algo) {
        case CONV2D_ALGO_IM2WIN_FP32_CC:
            if (!pre) e = launch_pack_filter_f32(static_cast<const float*>(w), static_cast<float*>(wq), d, st);
            if (e == cudaSuccess)
                e = launch_im2win_strips_f32(static_cast<const float*>(x), static_cast<float*>(win), d, st, !pre);
            if (e == cudaSuccess && !record(ev0, st)) return CONV2D_ERR_CUDA;
            if (e == cudaSuccess)
                s = launch_conv_fp32(d, static_cast<const float*>(win), static_cast<const float*>(wq),
                                     static_cast<float*>(y), true, st);
            break;
        case CONV2D_ALGO_IMPLICIT_FP32_CC:
            if (!pre) e = launch_pack_filter_f32(static_cast<const float*>(w), static_cast<float*>(wq), d, st);
            if (e == cudaSuccess && !record(ev0, st)) return CONV2D_ERR_CUDA;
            if (e == cudaSuccess)
                s = launch_conv_fp32(d, static_cast<const float*>(x), static_cast<const float*>(wq),
                                     static_cast<float*>(y), false, st);
            break;
        case CONV2D_ALGO_WINOGRAD_FP32_CC:
            if (!record(ev0, st)) return CONV2D_ERR_CUDA;   // brackets both kernels (filter transform + main)
            if (!pre) e = launch_winograd_filter(d, static_cast<const float*>(w), static_cast<float*>(wq), st);
            if (e == cudaSuccess)
                s = launch_winograd_main(d, static_cast<const float*>(x), static_cast<const float*>(wq),
                                         static_cast<float*>(y), st);
            break;
        case CONV2D_ALGO_IM2WIN_TC:
            if (!pre) e = launch_pack_filter_tc(w, wq, d, true, st);
            if (e == cudaSuccess)
                e = launch_window_cl16(x, win, d.N, d.Ci, d.H, d.W, d.Ci8, d.Ck, d.Ho, d.Wq * d.s, d.Kh, d.s, d.p,
                                       st, !pre);
            if (e == cudaSuccess && !record(ev0, st)) return CONV2D_ERR_CUDA;
            if (e == cudaSuccess) s = launch_conv_tc(d, win, wq, y, 1, st, ws + d.ws_split_off, d.ws_split);
            break;
        case CONV2D_ALGO_IMPLICIT_TC: {
            if (d.gemm1x1) {   // no repack, no copy: one launch on the caller's tensors
                if (!record(ev0, st)) return CONV2D_ERR_CUDA;
                s = launch_conv_tc(d, x, w, y, 3, st);
                break;
            }
            if (!pre) e = launch_pack_filter_tc(w, wq, d, false, st);
            const void* src = x;
            if (e == cudaSuccess && d.layout == CONV2D_LAYOUT_NCHW) {
                e = launch_nchw_to_nhwc16(x, win, d.N, d.Ci, d.H, d.W, d.Ci8, st, !pre);
                src = win;
            }
            if (e == cudaSuccess && !record(ev0, st)) return CONV2D_ERR_CUDA;
            if (e == cudaSuccess) s = launch_conv_tc(d, src, wq, y, 0, st, ws + d.ws_split_off, d.ws_split);
            break;
        }
        case CONV2D_ALGO_IMPLICIT_NCHW_TC:   // the contraction kernel reads NCHW X itself
            if (!pre) e = launch_pack_filter_tc(w, wq, d, false, st);
            if (e == cudaSuccess && !record(ev0, st)) return CONV2D_ERR_CUDA;
            if (e == cudaSuccess) s = launch_conv_tc(d, x, wq, y, 4, st);
            break;
        case CONV2D_ALGO_PADDED_TC:
            if (!pre) e = launch_pack_filter_tc(w, wq, d, false, st);
            if (e == cudaSuccess) e = launch_nchw_to_padded_nhwc16(x, win, d, st, !pre);
            if (e == cudaSuccess && !record(ev0, st)) return CONV2D_ERR_CUDA;
            if (e == cudaSuccess) s = launch_conv_tc(d, win, wq, y, 2, st, ws + d.ws_split_off, d.ws_split);
            break;
        default:
            return CONV2D_ERR_BAD_PARAM;
    }
    if (e != cudaSuccess) return CONV2D_ERR_CUDA;
    if (s == CONV2D_OK && !record(ev1, st)) return CONV2D_ERR_CUDA;
    return s;
}

}  // namespace

CONV2D_API conv2d_status conv2d_fwd(conv2d_desc_t d, const void* x, const void* w, void* y, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    return fwd_impl(d, x, w, y, workspace, workspace_bytes, stream, nullptr, nullptr);
}

CONV2D_API conv2d_status conv2d_fwd_profiled(conv2d_desc_t d, const void* x, const void* w, void* y,
                                             void* workspace, size_t workspace_bytes, void* stream, void* ev_start,
                                             void* ev_end) {
    return fwd_impl(d, x, w, y, workspace, workspace_bytes, stream, ev_start, ev_end);
}

CONV2D_API conv2d_status conv2d_fwd_host(conv2d_desc_t dp, const void* x_host, const void* w_host, void* y_host,
                                         void* x_dev, void* w_dev, void* y_dev, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    if (!dp || !x_host || !w_host || !y_host || !x_dev || !w_dev || !y_dev) return CONV2D_ERR_NULL_PTR;
    const conv2d_desc& d = *dp;
    // The device-side checks of conv2d_fwd, before any copy is issued.
    if (d.ws_total > 0 && !workspace) return CONV2D_ERR_NULL_PTR;
    if (!aligned16(x_dev) || !aligned16(w_dev) || !aligned16(y_dev) || (workspace && !aligned16(workspace)))
        return CONV2D_ERR_MISALIGNED;
    if (workspace_bytes < d.ws_total) return CONV2D_ERR_WORKSPACE_TOO_SMALL;
    const size_t elem = d.dtype == CONV2D_F32 ? 4 : 2;
    const size_t x_bytes = (size_t)d.N * d.Ci * d.H * d.W * elem;
    const size_t w_bytes = d.prepacked ? (d.gemm1x1 ? (size_t)d.Co * d.Ci * elem : d.ws_weights)
                                       : (size_t)d.Co * d.Ci * d.Kh * d.Kw * elem;
    const size_t y_bytes = (size_t)d.N * d.Co * d.Ho * d.Wo * (d.out_dtype == CONV2D_F32 ? 4 : 2);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(x_dev, x_host, x_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (cudaMemcpyAsync(w_dev, w_host, w_bytes, cudaMemcpyHostToDevice, st) != cudaSuccess) return CONV2D_ERR_CUDA;
    const conv2d_status s = fwd_impl(dp, x_dev, w_dev, y_dev, workspace, workspace_bytes, stream, nullptr, nullptr);
    if (s != CONV2D_OK) return s;
    if (cudaMemcpyAsync(y_host, y_dev, y_bytes, cudaMemcpyDeviceToHost, st) != cudaSuccess) return CONV2D_ERR_CUDA;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_launches_per_call(conv2d_desc_t d, int* launches) {
    if (!d || !launches) return CONV2D_ERR_NULL_PTR;
    if (d->gemm1x1) {   // the contraction alone
        *launches = 1;
        return CONV2D_OK;
    }
    int n = d->prepacked ? 1 : 2;   // filter repack (unless pre-packed) + contraction
    if (d->algo == CONV2D_ALGO_IM2WIN_FP32_CC || d->algo == CONV2D_ALGO_IM2WIN_TC || d->algo == CONV2D_ALGO_PADDED_TC ||
        (d->algo == CONV2D_ALGO_IMPLICIT_TC && d->layout == CONV2D_LAYOUT_NCHW && !d->nchw_halo))
        ++n;
    *launches = n;
    return CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_device_status(void* stream, uint32_t* code_out) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t a = 0, b = 0, c = 0;
    if (status_read_clear_tc(st, &a) != cudaSuccess || status_read_clear_fp32(st, &b) != cudaSuccess ||
        status_read_clear_wg(st, &c) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    if (code_out) *code_out = a | b | c;
    return (a | b | c) ? CONV2D_ERR_DEVICE_TIMEOUT : CONV2D_OK;
}

CONV2D_API conv2d_status conv2d_set_wait_limit(uint64_t ns, void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (wait_limit_set_tc(st, ns) != cudaSuccess || wait_limit_set_fp32(st, ns) != cudaSuccess ||
        wait_limit_set_wg(st, ns) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    return CONV2D_OK;
}

CONV2D_API const char* conv2d_status_string(conv2d_status s) {
    switch (s) {
        case CONV2D_OK: return "ok";
        case CONV2D_ERR_BAD_PARAM: return "bad parameter";
        case CONV2D_ERR_UNSUPPORTED: return "unsupported shape or option";
        case CONV2D_ERR_NULL_PTR: return "null pointer";
        case CONV2D_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case CONV2D_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case CONV2D_ERR_CUDA: return "CUDA error";
        case CONV2D_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}
