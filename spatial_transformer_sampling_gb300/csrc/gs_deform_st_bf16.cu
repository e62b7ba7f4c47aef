// gs_deform_st_bf16.cu -- __nv_bfloat16 instantiation of the staged DeformConv kernel
// (its own translation unit so the build compiles it in parallel).
#include "gs_deform_st.cuh"

namespace gs {
template cudaError_t launch_deform_staged<__nv_bfloat16>(const void *, const void *, const void *,
                                               const void *, const void *, void *,
                                               const DeformArgs &, cudaStream_t, bool *);

bool deform_staged_takes(const DeformArgs &args, const void *X, const void *W, const void *offset,
                         const void *mask) {
    DeformStParams q;
    return deform_st_params(args, X, W, offset, mask, &q);
}
}  // namespace gs
