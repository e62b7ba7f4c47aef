// gs_internal.h -- host-side interface between the C ABI (gs_api.cu) and the
// per-dtype kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace gs {

// Host-side per-device setup (a kernel's shared-memory attribute, a symbol's
// device address) runs on the first call that needs it on each device.  The
// flags are atomics, so first calls from several host threads at once do not
// race on them; the setup steps are idempotent, so two such calls may both run
// a step and both get the same result.
constexpr int kMaxDevices = 64;

struct DeviceFlags {
    std::atomic<bool> set[kMaxDevices];
};

// Runs setup() unless it already succeeded on the current device; returns its
// error (cudaSuccess once done).
template <typename F>
cudaError_t once_per_device(DeviceFlags &flags, F &&setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const bool cached = dev >= 0 && dev < kMaxDevices;
    if (cached && flags.set[dev].load(std::memory_order_acquire)) return cudaSuccess;
    e = setup();
    if (e == cudaSuccess && cached) flags.set[dev].store(true, std::memory_order_release);
    return e;
}

constexpr int kSampleThreads = 256;

struct Axis;   // gs_common.cuh

// Arguments of the sampling kernels (GridSample and the fused affine path).
// Largest spatial rank GridSample takes (ranks 4 and up run on one
// rank-general kernel; the fused and channel-last paths take ranks 2 and 3).
constexpr int kMaxRankND = 6;

struct SampleArgs {
    int N, C;
    int in[kMaxRankND];  // input spatial extents, outermost first (1 when unused)
    int out[kMaxRankND]; // output spatial extents, outermost first
    int64_t in_plane;    // product of in[]
    int64_t out_plane;   // product of out[]
    int tiles;           // blocks per image: ceil(out_plane / kSampleThreads)
    int pad, ac;
    float a;             // Keys coefficient
    unsigned *err;       // device error word (bounded waits record timeouts here)
};

// Arguments of the standalone AffineGrid kernel.
struct AffineGridArgs {
    int N;
    int out[3];
    int64_t out_plane;
    int ac;
};

// Arguments of DeformConv.
struct DeformArgs {
    int N, C, H, W, oC, oH, oW;
    int kH, kW, pad_t, pad_l, sH, sW, dH, dW, group, offset_group;
    int has_bias, has_mask;
    unsigned *err;       // device error word (bounded waits record timeouts here)
};

// Resize (Resize - 18): coordinate maps and nearest rounding.
enum { RS_HALF_PIXEL = 0, RS_PYTORCH_HALF_PIXEL = 1, RS_ALIGN_CORNERS = 2, RS_ASYMMETRIC = 3,
       RS_TF_CROP_AND_RESIZE = 4 };
enum { RS_ROUND_PREFER_FLOOR = 0, RS_ROUND_PREFER_CEIL = 1, RS_FLOOR = 2, RS_CEIL = 3 };

// One resized axis.  taps: taps per output index (1 nearest, 2 linear,
// 4 cubic, more when antialiasing a downscale); k0: offset of the first tap
// from floor(x) (the last is 1 - k0); aa_scale: the scale the filter is
// stretched by (1 unless antialiasing a downscale).
struct ResizeAxis {
    int n_in, n_out;
    double scale, length_resized, roi_start, roi_end, aa_scale;
    int k0, taps;
};

constexpr int kRsMaxTapsHost = 64;   // taps per output index the Resize kernel holds

// Arguments of the Resize kernel: r trailing resized axes in ax[3-r..2]
// (ax[0..2-r] are unit axes), B slices made of the leading axes.
struct ResizeArgs {
    ResizeAxis ax[3];
    int64_t B;
    int r;
    int mode, coord, nearest_mode;
    double a;
    int exclude_outside;
    float extrapolation_value;
    unsigned *err;   // device error word (bounded waits record timeouts here)
};

// Per-dtype launchers; T is float, __half or __nv_bfloat16.  Each enqueues on
// `s` and returns the launch error (cudaSuccess when fine).
// `ws`, `ws_bytes`: optional device workspace for the channel-last GridSample
// path (NULL, or fewer bytes than one image: the NCHW gather runs instead).
template <typename T>
cudaError_t launch_sample(const void *X, const void *src, void *Y, const SampleArgs &args, int r,
                          int mode, bool affine, void *ws, size_t ws_bytes, cudaStream_t s);
// Workspace bytes the channel-last path asks for (0: this call never takes it),
// and the least it runs with (one image slot).
template <typename T>
size_t sample_workspace_bytes(const SampleArgs &args, int r, bool affine);
template <typename T>
size_t sample_min_workspace_bytes(const SampleArgs &args);
template <typename T>
cudaError_t launch_affine_grid(const void *theta, void *grid, const AffineGridArgs &args, int r,
                               cudaStream_t s);
template <typename T>
cudaError_t launch_deform(const void *X, const void *W, const void *offset, const void *B,
                          const void *mask, void *Y, const DeformArgs &args, cudaStream_t s);
// DeformConv with an optional workspace for the channel-last tensor-core path
// (too small or NULL: launch_deform), and the workspace bytes that path asks
// for (0: it never takes the shape).
template <typename T>
cudaError_t launch_deform_ws(const void *X, const void *W, const void *offset, const void *B,
                             const void *mask, void *Y, const DeformArgs &args, void *ws,
                             size_t ws_bytes, cudaStream_t s);
template <typename T>
size_t deform_ws_bytes(const DeformArgs &args);
// DeformConv (fp16 / bf16) on the staged persistent tensor-core kernel
// (gs_deform_st.cuh) when it takes the shape and pointers; *used reports
// whether it ran.  deform_staged_takes answers the same question.
template <typename T>
cudaError_t launch_deform_staged(const void *X, const void *W, const void *offset, const void *B,
                                 const void *mask, void *Y, const DeformArgs &args, cudaStream_t s,
                                 bool *used);
bool deform_staged_takes(const DeformArgs &args, const void *X, const void *W, const void *offset,
                         const void *mask);
// DeformConv (fp32) on the windowed register-tiled kernel (gs_deform_f32.cu)
// when it takes the shape and X pointer; *used reports whether it ran.
cudaError_t launch_deform_f32(const void *X, const void *W, const void *offset, const void *B,
                              const void *mask, void *Y, const DeformArgs &args, cudaStream_t s,
                              bool *used);
bool deform_f32_takes(const DeformArgs &args, const void *X);
template <typename T>
cudaError_t launch_resize(const void *X, void *Y, const ResizeArgs &args, cudaStream_t s);
// GridSample with integer X (TX: uint8_t, int8_t, uint16_t, int16_t) and a float
// grid of gs_dtype code `grid_dt`.
template <typename TX>
cudaError_t launch_sample_int(const void *X, const void *grid, int grid_dt, void *Y,
                              const SampleArgs &args, int r, int mode, cudaStream_t s);

}  // namespace gs
