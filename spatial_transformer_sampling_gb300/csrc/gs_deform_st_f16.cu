// gs_deform_st_f16.cu -- __half instantiation of the staged DeformConv kernel
// (its own translation unit so the build compiles it in parallel).
#include "gs_deform_st.cuh"

namespace gs {
template cudaError_t launch_deform_staged<__half>(const void *, const void *, const void *,
                                               const void *, const void *, void *,
                                               const DeformArgs &, cudaStream_t, bool *);
}  // namespace gs
