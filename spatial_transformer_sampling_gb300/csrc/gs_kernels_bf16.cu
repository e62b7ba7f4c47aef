// gs_kernels_bf16.cu -- __nv_bfloat16 instantiations of the libgs kernels (one
// translation unit per dtype so the build compiles them in parallel).
#include "gs_deform.cuh"
#include "gs_resize.cuh"
#include "gs_sample.cuh"

namespace gs {
template cudaError_t launch_sample<__nv_bfloat16>(const void *, const void *, void *, const SampleArgs &,
                                          int, int, bool, void *, size_t, cudaStream_t);
template size_t sample_workspace_bytes<__nv_bfloat16>(const SampleArgs &, int, bool);
template size_t sample_min_workspace_bytes<__nv_bfloat16>(const SampleArgs &);
template cudaError_t launch_affine_grid<__nv_bfloat16>(const void *, void *, const AffineGridArgs &, int,
                                               cudaStream_t);
template cudaError_t launch_deform<__nv_bfloat16>(const void *, const void *, const void *, const void *,
                                          const void *, void *, const DeformArgs &, cudaStream_t);
template cudaError_t launch_deform_ws<__nv_bfloat16>(const void *, const void *, const void *, const void *,
                                             const void *, void *, const DeformArgs &, void *,
                                             size_t, cudaStream_t);
template size_t deform_ws_bytes<__nv_bfloat16>(const DeformArgs &);
template cudaError_t launch_resize<__nv_bfloat16>(const void *, void *, const ResizeArgs &, cudaStream_t);
}  // namespace gs
