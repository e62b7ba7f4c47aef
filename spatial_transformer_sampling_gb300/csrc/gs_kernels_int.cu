// gs_kernels_int.cu -- GridSample with integer-typed X (uint8, int8, uint16,
// int16) and a floating-point grid.
//
// GridSample - version 20, Outputs: for integer input types the intermediate
// values are computed as floating point and cast to the integer type at the
// end.  The cast (truncation toward zero, saturated at the type's range)
// turns the last bit of the interpolated value into a whole unit when the
// value sits next to an integer, so this path evaluates each output in fp64
// with every product and sum rounded on its own (no fused multiply-add):
//  - x = unnormalised grid value (GridSample - version 20, Attributes,
//    align_corners), padded for linear and nearest (border: clip;
//    reflection: mirror at the borders with fmod, then clip);
//  - nearest: the nearest index, ties to even; linear: floor(x), floor(x)+1
//    with weights 1-t, t; cubic: floor(x)-1 .. floor(x)+2, each index padded
//    (border: clamp; reflection: mirror, then clip), Keys weights at
//    distances t+1, t, 1-t, 2-t with cubic_coeff_a (Resize - 18, Attributes);
//  - the value is the sum, over the tensor product of the axes' taps (the
//    innermost axis fastest), of (1 * w_outermost * ... * w_innermost) * X,
//    a tap outside X (zeros padding) adding nothing.
// Each output's integer is then the truncation of that double, saturated.
// One thread per output position; ranks 1 to 6.
#include <math.h>
#include <stdint.h>

#include "gs_sample.cuh"

namespace gs {

__device__ __forceinline__ double d_add(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ double d_sub(double a, double b) { return __dsub_rn(a, b); }
__device__ __forceinline__ double d_mul(double a, double b) { return __dmul_rn(a, b); }

__device__ __forceinline__ double i64_unnormalize(double g, int n, int ac) {
    if (ac) return d_mul(d_mul(d_add(g, 1.0), 0.5), (double)(n - 1));   // (g+1)/2*(n-1)
    return d_mul(d_sub(d_mul(d_add(g, 1.0), (double)n), 1.0), 0.5);     // ((g+1)n-1)/2
}

// mirror into [lo, hi] (period 2*(hi-lo), fmod is exact); a zero-width range maps to lo
__device__ __forceinline__ double i64_reflect(double x, double lo, double hi) {
    const double span = d_sub(hi, lo);
    if (span <= 0.0) return lo;
    const double period = d_mul(2.0, span);
    double m = fmod(d_sub(x, lo), period);
    if (m < 0.0) m = d_add(m, period);
    if (m > span) m = d_sub(period, m);
    return d_add(lo, m);
}

__device__ __forceinline__ double i64_clip(double x, double lo, double hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

__device__ __forceinline__ double i64_reflect_axis(double x, int n, int ac) {
    if (ac) return i64_reflect(x, 0.0, (double)(n - 1));
    return i64_reflect(x, -0.5, d_sub((double)n, 0.5));
}

// Keys' cubic convolution kernel, each polynomial evaluated left to right
__device__ __forceinline__ double i64_keys(double s, double a) {
    s = fabs(s);
    if (s <= 1.0) {
        const double t1 = d_mul(d_mul(d_mul(d_add(a, 2.0), s), s), s);
        const double t2 = d_mul(d_mul(d_add(a, 3.0), s), s);
        return d_add(d_sub(t1, t2), 1.0);
    }
    if (s < 2.0) {
        const double t1 = d_mul(d_mul(d_mul(a, s), s), s);
        const double t2 = d_mul(d_mul(d_mul(5.0, a), s), s);
        const double t3 = d_mul(d_mul(8.0, a), s);
        const double t4 = d_mul(4.0, a);
        return d_sub(d_add(d_sub(t1, t2), t3), t4);
    }
    return 0.0;
}

// a coordinate beyond every extent only needs to stay on its side
__device__ __forceinline__ int64_t i64_index(double f) {
    if (!(f > -1.0e15)) f = -1.0e15;
    if (f > 1.0e15) f = 1.0e15;
    return (int64_t)f;
}

// taps of one axis from the grid value g: indices (maybe outside [0, n)) and weights
template <int MODE>
__device__ __forceinline__ int i64_axis_taps(double g, int n, int pad, int ac, double a,
                                             int64_t (&idx)[4], double (&w)[4]) {
    double x = i64_unnormalize(g, n, ac);
    if constexpr (MODE == MODE_NEAREST || MODE == MODE_LINEAR) {
        if (pad == PAD_BORDER) x = i64_clip(x, 0.0, (double)(n - 1));
        else if (pad == PAD_REFLECTION) x = i64_clip(i64_reflect_axis(x, n, ac), 0.0, (double)(n - 1));
    }
    if constexpr (MODE == MODE_NEAREST) {
        idx[0] = i64_index(rint(x));   // half to even
        w[0] = 1.0;
        return 1;
    }
    const double f = floor(x);
    const double t = d_sub(x, f);
    const int64_t i0 = i64_index(f);
    if constexpr (MODE == MODE_LINEAR) {
        idx[0] = i0;
        w[0] = d_sub(1.0, t);
        idx[1] = i0 + 1;
        w[1] = t;
        return 2;
    }
    if constexpr (MODE == MODE_CUBIC) {
        for (int k = 0; k < 4; ++k) {
            int64_t j = i0 - 1 + k;
            if (pad == PAD_BORDER) {
                j = j < 0 ? 0 : (j > n - 1 ? n - 1 : j);
            } else if (pad == PAD_REFLECTION) {
                j = (int64_t)i64_clip(i64_reflect_axis((double)j, n, ac), 0.0, (double)(n - 1));
            }
            idx[k] = j;
            w[k] = i64_keys(d_sub(d_add(t, 1.0), (double)k), a);
        }
    }
    return 4;
}

// the cast at the end: truncation toward zero, saturated; NaN reads 0
template <typename TX> struct IntRange;
template <> struct IntRange<uint8_t> { static constexpr double lo = 0, hi = 255; };
template <> struct IntRange<int8_t> { static constexpr double lo = -128, hi = 127; };
template <> struct IntRange<uint16_t> { static constexpr double lo = 0, hi = 65535; };
template <> struct IntRange<int16_t> { static constexpr double lo = -32768, hi = 32767; };

template <typename TX>
__device__ __forceinline__ TX i64_cast(double v) {
    if (v != v) return (TX)0;
    v = v < IntRange<TX>::lo ? IntRange<TX>::lo : (v > IntRange<TX>::hi ? IntRange<TX>::hi : v);
    return (TX)(int)trunc(v);
}

template <typename TX, int MODE>
__global__ void __launch_bounds__(kSampleThreads)
sample_int_kernel(const TX *__restrict__ X, const void *__restrict__ grid, int grid_dt,
                  TX *__restrict__ Y, const SampleArgs a, int r) {
    const int n = blockIdx.x / a.tiles;
    const int tile = blockIdx.x - n * a.tiles;
    const int64_t o = (int64_t)tile * kSampleThreads + threadIdx.x;
    if (o >= a.out_plane) return;
    int64_t idx[kMaxRankND][4];
    double w[kMaxRankND][4];
    int nt[kMaxRankND];
    int64_t total = 1;
    const int64_t g0 = ((int64_t)n * a.out_plane + o) * r;
    for (int d = 0; d < r; ++d) {
        // the location vector lists the innermost axis first
        const double g = (double)grid_value(grid, grid_dt, g0 + (r - 1 - d));
        nt[d] = i64_axis_taps<MODE>(g, a.in[d], a.pad, a.ac, (double)a.a, idx[d], w[d]);
        total *= nt[d];
    }
    const TX *Xc = X + (int64_t)n * a.C * a.in_plane;
    TX *Yc = Y + (int64_t)n * a.C * a.out_plane + o;
    for (int c = 0; c < a.C; ++c) {
        double acc = 0.0;
        for (int64_t tt = 0; tt < total; ++tt) {
            // tap tt of the tensor product, the innermost axis fastest
            int64_t rem = tt, off = 0;
            double weight = 1.0;
            bool inside = true;
            int k[kMaxRankND];
            for (int d = r - 1; d >= 0; --d) {
                k[d] = (int)(rem % nt[d]);
                rem /= nt[d];
            }
            for (int d = 0; d < r; ++d) {
                const int64_t j = idx[d][k[d]];
                inside = inside && j >= 0 && j < a.in[d];
                weight = d_mul(weight, w[d][k[d]]);
                off = off * a.in[d] + j;
            }
            if (inside) acc = d_add(acc, d_mul(weight, (double)Xc[off]));
        }
        *Yc = i64_cast<TX>(acc);
        Xc += a.in_plane;
        Yc += a.out_plane;
    }
}

template <typename TX>
cudaError_t launch_sample_int(const void *X, const void *grid, int grid_dt, void *Y,
                              const SampleArgs &args, int r, int mode, cudaStream_t s) {
    SampleArgs a = args;
    a.tiles = (int)((a.out_plane + kSampleThreads - 1) / kSampleThreads);
    const unsigned blocks = (unsigned)((int64_t)a.N * a.tiles);
    switch (mode) {
        case MODE_LINEAR:
            sample_int_kernel<TX, MODE_LINEAR><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, a, r);
            break;
        case MODE_NEAREST:
            sample_int_kernel<TX, MODE_NEAREST><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, a, r);
            break;
        default:
            sample_int_kernel<TX, MODE_CUBIC><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, a, r);
            break;
    }
    return cudaGetLastError();
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
