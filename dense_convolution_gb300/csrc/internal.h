// Host-side plan shared by the translation units of the library (not public).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/conv2d.h"

struct conv2d_desc {
    // Problem, as given to conv2d_desc_create.
    int N, Ci, H, W, Co, Kh, Kw, s, p;
    conv2d_dtype dtype;
    conv2d_algo requested;
    conv2d_layout layout;
    conv2d_dtype out_dtype;   // element type of Y: dtype, or F32 for 16-bit inputs
    const void* bias;         // Co bias values of the input type (device), or null
    // Ablation knobs (conv2d_desc_set_tuning); 0 = automatic.
    int tune_stages;          // cap on the shared-memory ring depth
    int tune_sync_copies;     // 1: each stage's copies land before the next stage's are issued
    int tune_raster;          // tile visit order (0 channel tile fastest, 1 pixel group fastest, 2 zig-zag)
    int tune_no_resident;     // 1: never keep the whole filter slice resident in shared memory
    int tune_split;           // 1: split the last partial wave of tiles over all SMs (opt-in)
    int tune_epi_groups;      // epilogue groups of four warps: 2, 3, or 0 = automatic
    int tune_tile_n;          // tensor-core channel tile width: 64, 128, 176, 256, or 0 = automatic
    bool prepacked;           // conv2d_fwd's w is the filter conv2d_pack_filter wrote (no repack per call)
    // Derived geometry.
    int Ho, Wo, Wp;       // output size; padded input width W + 2p
    conv2d_algo algo;     // resolved (never AUTO)
    // fp32 CUDA-core paths.
    int Lp;               // im2win strip pitch in floats: Wp*Kh rounded up to 4
    int cc_warps;         // warps per block (32 output channels each)
    // Tensor-core paths.
    int Ci8;              // Ci rounded up to 8 (16-byte channel vectors)
    int Ck;               // im2win window: channels per padded column.  Ci8 <= 16: the Kh*Ci
                          // (row, channel) pairs packed densely, c = u*Ci + ci, rounded up to 8;
                          // otherwise Kh*Ci8 with c = u*Ci8 + ci
    int taps;             // filter taps per K-chunk group: Kw (im2win) or Kh*Kw (implicit)
    int CP;               // channel extent per tap, padded to the 64-element K chunk
    int BN;               // output channels per MMA tile (64, 128 or 256)
    bool gemm1x1;         // implicit path on a 1x1, stride-1, unpadded NCHW layer with Ci and H*W multiples
                          // of 8: one GEMM per image straight on the caller's X and filter (no copies)
    bool nchw_halo;       // implicit path on NCHW input, stride 1: the contraction kernel builds its operand
                          // tiles from X itself (no input copy; workspace = the repacked filter)
    int halo_v;           // pixels per vector load of X in that kernel (W % halo_v == 0, Wq % halo_v == 0)
    int Hp, Wq;           // virtual pixel grid [N][Hp][Wq] of the grid-row tensor-core paths.  Padded:
                          // H+2p rows of pitch W+2p (rounded up to 4 when Wo % 4 == 0).  im2win: Ho rows
                          // of Wq output slots (window tensor rows hold Wq*s columns)
    // Workspace layout (bytes): packed filter at 0, input-side tensor after it.
    size_t ws_weights, ws_input_off, ws_input, ws_total;
    size_t ws_split_off, ws_split;   // split-tail partial sums and flags (tensor-core modes 0-2), at the end
};

namespace conv2d_gb300 {

constexpr int kTcBlockM = 128;   // output pixels per MMA tile
constexpr int kTcBlockK = 64;    // K elements per pipeline stage (128 bytes of 16-bit)
constexpr long long kStripSmemMax = 200 * 1024;   // fp32 im2win transform: staged input rows per block

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Launch that may overlap the previous kernel of the stream (programmatic
// dependent launch): the kernel can start while its predecessor finishes, and
// must execute griddepcontrol.wait (pdl_wait) before touching that
// predecessor's results.  Used for every kernel of a conv2d_fwd call; the
// first one waits before touching any memory (its predecessor may be any
// kernel of the caller's) and signals its dependents only after that wait.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// A launch that is either a programmatic dependent of the previous kernel of
// the stream (pdl) or an ordinary stream-ordered launch, for kernels that are
// the first of a call when the filter repack is skipped (they read X at once
// and must not start before the stream's previous work has finished).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_chain(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t st, Args... args) {
    if (pdl) return launch_after(kernel, grid, block, smem, st, args...);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// transforms.cu (pdl = false: the first kernel of a call, see launch_chain)
cudaError_t launch_im2win_strips_f32(const float* x, float* xw, const conv2d_desc& d, cudaStream_t st,
                                     bool pdl = true);
cudaError_t launch_window_cl16(const void* x, void* out, int N, int Ci, int H, int W, int Ci8, int Ck, int R,
                               int Wq, int Kh, int s, int p, cudaStream_t st, bool pdl = true);
cudaError_t launch_nchw_to_nhwc16(const void* x, void* out, int N, int C, int H, int W, int C8, cudaStream_t st,
                                  bool pdl = true);
cudaError_t launch_nchw_to_padded_nhwc16(const void* x, void* out, const conv2d_desc& d, cudaStream_t st,
                                         bool pdl = true);
cudaError_t launch_pack_filter_tc(const void* w, void* wq, const conv2d_desc& d, bool im2win, cudaStream_t st);
cudaError_t launch_pack_filter_f32(const float* w, float* wq, const conv2d_desc& d, cudaStream_t st);

// conv_fp32.cu
conv2d_status launch_conv_fp32(const conv2d_desc& d, const float* src, const float* wq, float* y,
                               bool im2win, cudaStream_t st);

// winograd.cu
size_t winograd_filter_bytes(const conv2d_desc& d);
cudaError_t launch_winograd_filter(const conv2d_desc& d, const float* w, float* u, cudaStream_t st);
conv2d_status launch_winograd_main(const conv2d_desc& d, const float* x, const float* u, float* y,
                                   cudaStream_t st);
cudaError_t status_read_clear_wg(cudaStream_t st, uint32_t* out);
cudaError_t wait_limit_set_wg(cudaStream_t st, uint64_t ns);

// conv_tc.cu
conv2d_status launch_conv_tc(const conv2d_desc& d, const void* src, const void* wq, void* y, int amode,
                             cudaStream_t st, void* split_ws = nullptr, size_t split_bytes = 0);
size_t tc_split_bytes(int grid, int group, int BN);
size_t tc_split_need(const conv2d_desc& d, int n_sm);
int device_sm_count();
bool halo_plan_fits(const conv2d_desc& d);
void* driver_entry(const char* name);
cudaError_t status_read_clear_tc(cudaStream_t st, uint32_t* out);
cudaError_t status_read_clear_fp32(cudaStream_t st, uint32_t* out);
cudaError_t wait_limit_set_tc(cudaStream_t st, uint64_t ns);
cudaError_t wait_limit_set_fp32(cudaStream_t st, uint64_t ns);

}  // namespace conv2d_gb300
