// gs_sample.cuh -- GridSample and fused AffineGrid+GridSample kernels, and the
// standalone AffineGrid kernel (templates; instantiated once per dtype).
//
// Work split: one thread per output position (n, d, h, w), looping over all C
// channels.  The coordinate, padding and tap weights are computed once per
// position in registers and reused by every channel (GridSample - version 20:
// the grid vector is shared by all channels of Y[n, :, ...]).  Consecutive
// threads take consecutive positions, so each channel's Y store is one
// coalesced 128-byte line per warp, and for smooth (e.g. affine) grids the
// gathers of a warp fall on a few neighbouring lines of X.
#pragma once

#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

struct SampleParams {
    SampleArgs a;
    Axis ax[kMaxRank];
};

// Per-image affine map from output index to input position, 24.40 fixed
// point, built once per block by one thread.  AffineGrid (description): the
// base position of output index i on an axis of m is (2i+1)/m - 1
// (align_corners=0) or -1 + 2i/(m-1) (align_corners=1, m = 1 -> 0), both
// affine in i; theta is affine; GridSample's unnormalisation is affine.  So
// the input position on axis d is sum_j coef[d][j]*i_j + cst[d].
struct AffineMap {
    int64_t coef_q[kMaxRank][kMaxRank];
    int64_t cst_q[kMaxRank];
    double coef[kMaxRank][kMaxRank];
    double cst[kMaxRank];
    int wide;   // positions may exceed 2^22 px: evaluate them in fp64 instead
};

template <typename T, int R>
__device__ void build_affine_map(const T *__restrict__ theta, const SampleArgs &a, AffineMap &m) {
    m.wide = 0;
    for (int d = 0; d < R; ++d) {
        const int row = R - 1 - d;   // theta row giving the coordinate of input axis d
        const int n = a.in[d];
        const double alpha = a.ac ? 0.5 * (double)(n - 1) : 0.5 * (double)n;
        const double beta = 0.5 * (double)(n - 1);
        double cst = IO<T>::to_double(theta[row * (R + 1) + R]);
        double bound = 0.0;
        for (int j = 0; j < R; ++j) {
            const int mo = a.out[j];
            const int col = R - 1 - j;   // theta column multiplying output axis j
            const double th = IO<T>::to_double(theta[row * (R + 1) + col]);
            double slope, off;
            if (a.ac) {
                slope = mo > 1 ? 2.0 / (double)(mo - 1) : 0.0;
                off = mo > 1 ? -1.0 : 0.0;
            } else {
                slope = 2.0 / (double)mo;
                off = 1.0 / (double)mo - 1.0;
            }
            m.coef[d][j] = alpha * th * slope;
            cst += th * off;
            bound += fabs(m.coef[d][j]) * (double)(mo - 1);
        }
        m.cst[d] = alpha * cst + beta;
        bound += fabs(m.cst[d]);
        if (!(bound < (double)kFarOut)) m.wide = 1;   // also NaN / inf
    }
    if (!m.wide) {
        for (int d = 0; d < R; ++d) {
            for (int j = 0; j < R; ++j) m.coef_q[d][j] = __double2ll_rn(m.coef[d][j] * 1099511627776.0);
            m.cst_q[d] = __double2ll_rn(m.cst[d] * 1099511627776.0);   // * 2^40
        }
    }
}

template <typename T, int R, int MODE, bool AFFINE>
__global__ void __launch_bounds__(kSampleThreads)
sample_kernel(const T *__restrict__ X, const T *__restrict__ src, T *__restrict__ Y,
              const SampleParams P) {
    const SampleArgs &a = P.a;
    const int n = blockIdx.x / a.tiles;
    const int tile = blockIdx.x - n * a.tiles;
    const int64_t o = (int64_t)tile * kSampleThreads + threadIdx.x;

    __shared__ AffineMap s_map;
    if constexpr (AFFINE) {
        if (threadIdx.x == 0) build_affine_map<T, R>(src + (int64_t)n * R * (R + 1), a, s_map);
        __syncthreads();
    }
    if (o >= a.out_plane) return;

    // output spatial index, outermost first
    int opos[R];
    {
        int64_t rem = o;
#pragma unroll
        for (int j = R - 1; j >= 0; --j) {
            opos[j] = (int)(rem % a.out[j]);
            rem /= a.out[j];
        }
    }

    // input position of every axis, 32.32 fixed point
    int64_t xq[R];
    if constexpr (AFFINE) {
        if (!s_map.wide) {
#pragma unroll
            for (int d = 0; d < R; ++d) {
                int64_t acc = s_map.cst_q[d];
#pragma unroll
                for (int j = 0; j < R; ++j) acc += s_map.coef_q[d][j] * (int64_t)opos[j];
                xq[d] = acc >> 8;   // 24.40 -> 32.32 (floor)
            }
        } else {
#pragma unroll
            for (int d = 0; d < R; ++d) {
                double x = s_map.cst[d];
#pragma unroll
                for (int j = 0; j < R; ++j) x += s_map.coef[d][j] * (double)opos[j];
                xq[d] = pos_to_q(x, P.ax[d], a.pad);
            }
        }
    } else {
        // GridSample grid: the location vector lists the innermost axis first
        const T *g = src + ((int64_t)n * a.out_plane + o) * R;
#pragma unroll
        for (int d = 0; d < R; ++d) xq[d] = grid_to_q(IO<T>::ld(g + (R - 1 - d)), P.ax[d], a.pad);
    }

    AxisTaps<MODE> tp[R];
#pragma unroll
    for (int d = 0; d < R; ++d) make_taps<MODE>(xq[d], P.ax[d], a.pad, a.ac, a.a, tp[d]);

    constexpr int K = TapCount<MODE>::K;
    const T *__restrict__ Xn = X + (int64_t)n * a.C * a.in_plane;
    T *__restrict__ Yn = Y + (int64_t)n * a.C * a.out_plane + o;

    if constexpr (R == 1) {
#pragma unroll 4
        for (int c = 0; c < a.C; ++c) {
            const T *Xc = Xn + (int64_t)c * a.in_plane;
            float acc = 0.0f;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const float v = ((tp[0].ok >> k) & 1u) ? IO<T>::ld(Xc + tp[0].idx[k]) : 0.0f;
                acc = fmaf(tp[0].w[k], v, acc);
            }
            Yn[(int64_t)c * a.out_plane] = IO<T>::st(acc);
        }
    } else if constexpr (R == 2) {
        int rowoff[K];
#pragma unroll
        for (int k = 0; k < K; ++k) rowoff[k] = tp[0].idx[k] * a.in[1];
#pragma unroll 4
        for (int c = 0; c < a.C; ++c) {
            const T *Xc = Xn + (int64_t)c * a.in_plane;
            float acc = 0.0f;
#pragma unroll
            for (int ky = 0; ky < K; ++ky) {
                float s = 0.0f;
#pragma unroll
                for (int kx = 0; kx < K; ++kx) {
                    const bool ok = ((tp[0].ok >> ky) & (tp[1].ok >> kx) & 1u) != 0;
                    const float v = ok ? IO<T>::ld(Xc + rowoff[ky] + tp[1].idx[kx]) : 0.0f;
                    s = fmaf(tp[1].w[kx], v, s);
                }
                acc = fmaf(tp[0].w[ky], s, acc);
            }
            Yn[(int64_t)c * a.out_plane] = IO<T>::st(acc);
        }
    } else {
        int zoff[K], yoff[K];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            zoff[k] = tp[0].idx[k] * a.in[1] * a.in[2];
            yoff[k] = tp[1].idx[k] * a.in[2];
        }
#pragma unroll 2
        for (int c = 0; c < a.C; ++c) {
            const T *Xc = Xn + (int64_t)c * a.in_plane;
            float acc = 0.0f;
#pragma unroll
            for (int kz = 0; kz < K; ++kz) {
                float sz = 0.0f;
#pragma unroll
                for (int ky = 0; ky < K; ++ky) {
                    float s = 0.0f;
#pragma unroll
                    for (int kx = 0; kx < K; ++kx) {
                        const bool ok =
                            ((tp[0].ok >> kz) & (tp[1].ok >> ky) & (tp[2].ok >> kx) & 1u) != 0;
                        const float v =
                            ok ? IO<T>::ld(Xc + zoff[kz] + yoff[ky] + tp[2].idx[kx]) : 0.0f;
                        s = fmaf(tp[2].w[kx], v, s);
                    }
                    sz = fmaf(tp[1].w[ky], s, sz);
                }
                acc = fmaf(tp[0].w[kz], sz, acc);
            }
            Yn[(int64_t)c * a.out_plane] = IO<T>::st(acc);
        }
    }
}

inline Axis make_axis(int n, int ac) {
    Axis A;
    A.n = n;
    A.h = ac ? 0.5f * (float)(n - 1) : 0.5f * (float)n;
    const int64_t span2 = ac ? 2 * (int64_t)(n - 1) : 2 * (int64_t)n;   // in half pixels... period
    A.period_f = (float)span2;
    A.pad_ = 0;
    A.c_q = (int64_t)(n - 1) * kHalfQ;                  // (n-1)/2
    A.lo_q = ac ? 0 : -kHalfQ;
    A.span_q = ac ? (int64_t)(n - 1) * kOneQ : (int64_t)n * kOneQ;
    A.hi_q = (int64_t)(n - 1) * kOneQ;
    return A;
}

template <typename T, int R, int MODE, bool AFFINE>
static cudaError_t launch_sample_t(const void *X, const void *src, void *Y, const SampleParams &P,
                                   cudaStream_t s) {
    const unsigned blocks = (unsigned)((int64_t)P.a.N * P.a.tiles);
    sample_kernel<T, R, MODE, AFFINE><<<blocks, kSampleThreads, 0, s>>>(
        (const T *)X, (const T *)src, (T *)Y, P);
    return cudaGetLastError();
}

template <typename T, int R, bool AFFINE>
static cudaError_t launch_sample_mode(const void *X, const void *src, void *Y,
                                     const SampleParams &P, int mode, cudaStream_t s) {
    switch (mode) {
        case MODE_LINEAR: return launch_sample_t<T, R, MODE_LINEAR, AFFINE>(X, src, Y, P, s);
        case MODE_NEAREST: return launch_sample_t<T, R, MODE_NEAREST, AFFINE>(X, src, Y, P, s);
        default: return launch_sample_t<T, R, MODE_CUBIC, AFFINE>(X, src, Y, P, s);
    }
}

template <typename T>
cudaError_t launch_sample(const void *X, const void *src, void *Y, const SampleArgs &args, int r,
                          int mode, bool affine, cudaStream_t s) {
    SampleParams P;
    P.a = args;
    for (int d = 0; d < kMaxRank; ++d) P.ax[d] = make_axis(d < r ? args.in[d] : 1, args.ac);
    if (affine) {
        if (r == 2) return launch_sample_mode<T, 2, true>(X, src, Y, P, mode, s);
        return launch_sample_mode<T, 3, true>(X, src, Y, P, mode, s);
    }
    if (r == 1) return launch_sample_mode<T, 1, false>(X, src, Y, P, mode, s);
    if (r == 2) return launch_sample_mode<T, 2, false>(X, src, Y, P, mode, s);
    return launch_sample_mode<T, 3, false>(X, src, Y, P, mode, s);
}

// ------------------------------------------------------------ AffineGrid

// AffineGrid (description): grid[n, pos, :] = theta[n] . [x, y, (z,) 1] with
// the base positions of the align_corners rule; evaluated in fp64 and
// rounded once to T.  One thread per output position.
template <typename T, int R>
__global__ void __launch_bounds__(256)
affine_grid_kernel(const T *__restrict__ theta, T *__restrict__ grid, const AffineGridArgs a) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)a.N * a.out_plane) return;
    const int64_t n = idx / a.out_plane;
    int64_t rem = idx - n * a.out_plane;
    double b[R];   // b[0] = x (innermost output axis), b[1] = y, b[2] = z
#pragma unroll
    for (int k = 0; k < R; ++k) {
        const int m = a.out[R - 1 - k];
        const int i = (int)(rem % m);
        rem /= m;
        if (a.ac) {
            b[k] = m > 1 ? -1.0 + 2.0 * (double)i / (double)(m - 1) : 0.0;
        } else {
            b[k] = (2.0 * (double)i + 1.0) / (double)m - 1.0;
        }
    }
    const T *th = theta + n * R * (R + 1);
    T *out = grid + idx * R;
#pragma unroll
    for (int row = 0; row < R; ++row) {
        double s = IO<T>::to_double(th[row * (R + 1) + R]);
#pragma unroll
        for (int k = 0; k < R; ++k) s = fma(IO<T>::to_double(th[row * (R + 1) + k]), b[k], s);
        out[row] = IO<T>::st(__double2float_rn(s));
    }
}

template <typename T>
cudaError_t launch_affine_grid(const void *theta, void *grid, const AffineGridArgs &args, int r,
                               cudaStream_t s) {
    const int64_t total = (int64_t)args.N * args.out_plane;
    const unsigned blocks = (unsigned)((total + 255) / 256);
    if (r == 2) {
        affine_grid_kernel<T, 2><<<blocks, 256, 0, s>>>((const T *)theta, (T *)grid, args);
    } else {
        affine_grid_kernel<T, 3><<<blocks, 256, 0, s>>>((const T *)theta, (T *)grid, args);
    }
    return cudaGetLastError();
}

}  // namespace gs
