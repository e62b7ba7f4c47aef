// gs_kernels_int.cu -- GridSample with integer-typed X (uint8, int8, uint16,
// int16) and a floating-point grid.
//
// GridSample - version 20, Outputs: for integer input types the intermediate
// values are computed as floating point and cast to the integer type at the
// end.  Here the taps and weights are those of sample_kernel (exact
// fixed-point coordinates, the same padding), the values are widened to fp32
// (exact for 8- and 16-bit integers) and accumulated in fp32, and the result
// is truncated toward zero and saturated at the type's range (IO<int type>).
// One thread per output position loops over the channels.
#include <stdint.h>

#include "gs_sample.cuh"

namespace gs {

template <typename TX, int R, int MODE>
__global__ void __launch_bounds__(kSampleThreads)
sample_int_kernel(const TX *__restrict__ X, const void *__restrict__ grid, int grid_dt,
                  TX *__restrict__ Y, const SampleParams P) {
    const SampleArgs &a = P.a;
    const int n = blockIdx.x / a.tiles;
    const int tile = blockIdx.x - n * a.tiles;
    const int64_t o = (int64_t)tile * kSampleThreads + threadIdx.x;
    if (o >= a.out_plane) return;
    // the location vector lists the innermost axis first
    AxisTaps<MODE> tp[R];
    const int64_t g0 = ((int64_t)n * a.out_plane + o) * R;
#pragma unroll
    for (int d = 0; d < R; ++d)
        make_taps<MODE>(grid_to_q(grid_value(grid, grid_dt, g0 + (R - 1 - d)), P.ax[d], a.pad),
                        P.ax[d], a.pad, a.ac, a.a, tp[d]);
    int off_hi[R == 3 ? 16 : 4];
    outer_offsets<R, MODE>(tp, a, off_hi);
    const TX *Xc = X + (int64_t)n * a.C * a.in_plane;
    TX *Yc = Y + (int64_t)n * a.C * a.out_plane + o;
#pragma unroll 4
    for (int c = 0; c < a.C; ++c) {
        *Yc = IO<TX>::st(interp<TX, R, MODE>(Xc, tp, off_hi));
        Xc += a.in_plane;
        Yc += a.out_plane;
    }
}

template <typename TX, int R>
static cudaError_t launch_int_r(const void *X, const void *grid, int grid_dt, void *Y,
                                const SampleParams &P, int mode, cudaStream_t s) {
    const unsigned blocks = (unsigned)((int64_t)P.a.N * P.a.tiles);
    switch (mode) {
        case MODE_LINEAR:
            sample_int_kernel<TX, R, MODE_LINEAR><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, P);
            break;
        case MODE_NEAREST:
            sample_int_kernel<TX, R, MODE_NEAREST><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, P);
            break;
        default:
            sample_int_kernel<TX, R, MODE_CUBIC><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, P);
            break;
    }
    return cudaGetLastError();
}

template <typename TX>
cudaError_t launch_sample_int(const void *X, const void *grid, int grid_dt, void *Y,
                              const SampleArgs &args, int r, int mode, cudaStream_t s) {
    if (r > 3) return launch_sample_nd<TX>(X, grid, grid_dt, Y, args, r, mode, s);
    const SampleParams P = make_params<float>(args, r);
    if (r == 1) return launch_int_r<TX, 1>(X, grid, grid_dt, Y, P, mode, s);
    if (r == 2) return launch_int_r<TX, 2>(X, grid, grid_dt, Y, P, mode, s);
    return launch_int_r<TX, 3>(X, grid, grid_dt, Y, P, mode, s);
}

template cudaError_t launch_sample_int<uint8_t>(const void *, const void *, int, void *,
                                                const SampleArgs &, int, int, cudaStream_t);
template cudaError_t launch_sample_int<int8_t>(const void *, const void *, int, void *,
                                               const SampleArgs &, int, int, cudaStream_t);
template cudaError_t launch_sample_int<uint16_t>(const void *, const void *, int, void *,
                                                 const SampleArgs &, int, int, cudaStream_t);
template cudaError_t launch_sample_int<int16_t>(const void *, const void *, int, void *,
                                                const SampleArgs &, int, int, cudaStream_t);

}  // namespace gs
