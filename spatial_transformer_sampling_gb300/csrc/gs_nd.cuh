// gs_nd.cuh -- GridSample for spatial ranks 4 to kMaxRankND (tensor grid, any
// element type of X).
//
// GridSample - version 20 (description, Inputs) defines the operator for an X
// of rank r+2 and any r: X (N, C, D1..Dr), grid (N, D1_out..Dr_out, r) whose
// location vector lists the innermost axis first, Y (N, C, D1_out..Dr_out).
// Ranks 1-3 have their own kernels; this one takes the rank at run time.
//
// One thread per output position.  Each axis's taps (the same 32.32
// fixed-point coordinate, padding and weights as every other path, from
// make_taps) are computed once and serve all C channels.  The tensor product
// of the taps is summed in separable order, innermost axis first: the K taps
// of the innermost axis form a partial sum, which enters the next axis's
// partial sum with that axis's weight, and so on outwards -- the order the
// rank-2 and rank-3 kernels use, so that a rank-r sum is r nested K-term sums
// rather than one K^r-term sum.  Taps out of range (zeros padding) read 0;
// their indices are clamped into range, so every address stays inside X.
#pragma once

#include <type_traits>

#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

struct NDParams {
    SampleArgs a;                 // in[] / out[] hold all r extents
    int r;
    Axis ax[kMaxRankND];
    int64_t stride[kMaxRankND];   // elements between neighbours along input axis d
};

// Per-axis taps of one output position: element offsets (index * stride),
// 1-D weights, validity bits.
template <int MODE> struct NDTaps {
    static constexpr int K = TapCount<MODE>::K;
    int64_t off[kMaxRankND][K];
    float w[kMaxRankND][K];
    unsigned ok[kMaxRankND];
};

// One output value of one (n, c) slab.
template <typename TX, int MODE>
__device__ __forceinline__ float nd_value(const TX *__restrict__ Xc, int r, const NDTaps<MODE> &t) {
    constexpr int K = TapCount<MODE>::K;
    int k[kMaxRankND];          // current tap of each outer axis
    float part[kMaxRankND];     // partial sum of each outer axis
#pragma unroll
    for (int d = 0; d < kMaxRankND; ++d) {
        k[d] = 0;
        part[d] = 0.0f;
    }
    const int last = r - 1;     // the innermost axis
    for (;;) {
        int64_t base = 0;
        bool in = true;
        for (int d = 0; d < last; ++d) {
            base += t.off[d][k[d]];
            in = in && ((t.ok[d] >> k[d]) & 1u);
        }
        float s = 0.0f;
        if (in) {
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const float v = ((t.ok[last] >> kx) & 1u) ? IO<TX>::ld(Xc + base + t.off[last][kx])
                                                          : 0.0f;
                s = fmaf(t.w[last][kx], v, s);
            }
        }
        // fold s outwards: into the next axis's partial sum, and on, as each
        // axis runs through its K taps
        int d = last - 1;
        for (; d >= 0; --d) {
            part[d] = fmaf(t.w[d][k[d]], s, part[d]);
            if (++k[d] < K) break;
            k[d] = 0;
            s = part[d];
            part[d] = 0.0f;
        }
        if (d < 0) return s;
    }
}

template <typename TX, int MODE>
__global__ void __launch_bounds__(kSampleThreads)
sample_nd_kernel(const TX *__restrict__ X, const void *__restrict__ grid, int grid_dt,
                 TX *__restrict__ Y, const NDParams P) {
    constexpr int K = TapCount<MODE>::K;
    const SampleArgs &a = P.a;
    const int r = P.r;
    const int n = blockIdx.x / a.tiles;
    const int tile = blockIdx.x - n * a.tiles;
    const int64_t o = (int64_t)tile * kSampleThreads + threadIdx.x;
    if (o >= a.out_plane) return;

    NDTaps<MODE> t;
    const int64_t g0 = ((int64_t)n * a.out_plane + o) * r;
#pragma unroll
    for (int d = 0; d < kMaxRankND; ++d) {
        if (d < r) {
            AxisTaps<MODE> at;
            // the location vector lists the innermost axis first
            make_taps<MODE>(grid_to_q(grid_value(grid, grid_dt, g0 + (r - 1 - d)), P.ax[d], a.pad),
                            P.ax[d], a.pad, a.ac, a.a, at);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                t.off[d][k] = (int64_t)at.idx[k] * P.stride[d];
                t.w[d][k] = at.w[k];
            }
            t.ok[d] = at.ok;
        }
    }
    const TX *Xc = X + (int64_t)n * a.C * a.in_plane;
    TX *Yc = Y + (int64_t)n * a.C * a.out_plane + o;
    for (int c = 0; c < a.C; ++c) {
        *Yc = IO<TX>::st(nd_value<TX, MODE>(Xc, r, t));
        Xc += a.in_plane;
        Yc += a.out_plane;
    }
}

// Grid type code of a float X type (a float X's grid has X's type).
template <typename T> constexpr int grid_dt_of() {
    return std::is_same<T, float>::value ? 0 : (std::is_same<T, __half>::value ? 1 : 2);
}

// GridSample of rank r (4 .. kMaxRankND) with a grid of float type grid_dt
// (0 fp32, 1 fp16, 2 bf16).  args holds the validated shapes; make_axis
// (gs_sample.cuh, which includes this file after it) gives each axis.
template <typename TX>
cudaError_t launch_sample_nd(const void *X, const void *grid, int grid_dt, void *Y,
                             const SampleArgs &args, int r, int mode, cudaStream_t s) {
    NDParams P;
    P.a = args;
    P.r = r;
    int64_t stride = 1;
    for (int d = kMaxRankND - 1; d >= 0; --d) {
        P.ax[d] = make_axis(d < r ? args.in[d] : 1, args.ac);
        P.stride[d] = d < r ? stride : 0;
        if (d < r) stride *= args.in[d];
    }
    P.a.tiles = (int)((P.a.out_plane + kSampleThreads - 1) / kSampleThreads);
    const unsigned blocks = (unsigned)((int64_t)P.a.N * P.a.tiles);
    switch (mode) {
        case MODE_LINEAR:
            sample_nd_kernel<TX, MODE_LINEAR><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, P);
            break;
        case MODE_NEAREST:
            sample_nd_kernel<TX, MODE_NEAREST><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, P);
            break;
        default:
            sample_nd_kernel<TX, MODE_CUBIC><<<blocks, kSampleThreads, 0, s>>>(
                (const TX *)X, grid, grid_dt, (TX *)Y, P);
            break;
    }
    return cudaGetLastError();
}

}  // namespace gs
