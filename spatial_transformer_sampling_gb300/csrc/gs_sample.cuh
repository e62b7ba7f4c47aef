// gs_sample.cuh -- GridSample and fused AffineGrid+GridSample kernels, and the
// standalone AffineGrid kernel (templates; instantiated once per dtype).
//
// sample_kernel (ranks 1-3, tensor grid or fused affine; gs_band.cuh streams
// the fused 2-D case through shared memory instead, gs_vol.cuh the fused 3-D
// trilinear and nearest cases, gs_nd.cuh takes ranks 4 and up): one thread per output
// position, looping over all C channels.  Coordinates, padding and tap
// weights are computed once per position in registers and reused by every
// channel (GridSample - version 20: the grid vector is shared by all channels
// of Y[n, :, ...]).  Consecutive threads take consecutive positions, so each
// channel's store is a whole line per warp and, for smooth grids, the gathers
// of a warp fall on a few neighbouring lines.
#pragma once

#include "gs_common.cuh"
#include "gs_internal.h"

namespace gs {

struct SampleParams {
    SampleArgs a;
    Axis ax[kMaxRank];
    // fused path: base position of output index i on output axis j is
    // slope[j]*i + off[j]; input axis d maps a grid value g to alpha[d]*g + beta[d]
    double slope[kMaxRank], off[kMaxRank], alpha[kMaxRank], beta[kMaxRank];
};

// Per-image affine map from output index to input position, 24.40 fixed
// point.  AffineGrid (description): base positions are affine in the output
// index; theta is affine; GridSample's unnormalisation is affine.  So the
// position on input axis d is sum_j coef[d][j]*i_j + cst[d].
struct AffineMap {
    int64_t coef_q[kMaxRank][kMaxRank];
    int64_t cst_q[kMaxRank];
    double coef[kMaxRank][kMaxRank];
    double cst[kMaxRank];
    int wide;   // positions may reach 2^22 px: evaluate them in fp64 instead
};

// Built by the first warp, one map entry per lane (no fp64 division: the
// slopes and offsets come from the host).
template <typename T, int R>
__device__ void build_affine_map_warp(const T *__restrict__ theta, const SampleParams &P,
                                      AffineMap &m) {
    constexpr int E = R * (R + 1);   // entry (d, j): j < R coefficient, j == R constant
    const int lane = threadIdx.x & 31;
    double val = 0.0;
    bool far = false;
    if (lane < E) {
        const int d = lane / (R + 1), j = lane - (lane / (R + 1)) * (R + 1);
        const int row = R - 1 - d;   // theta row giving the coordinate of input axis d
        const T *th = theta + row * (R + 1);
        if (j < R) {
            // theta column R-1-j multiplies the base position of output axis j
            val = P.alpha[d] * IO<T>::to_double(th[R - 1 - j]) * P.slope[j];
            far = !(fabs(val) * (double)(P.a.out[j] - 1) < (double)kFarOut / (R + 1));
        } else {
            double s = IO<T>::to_double(th[R]);
            for (int jj = 0; jj < R; ++jj) s += IO<T>::to_double(th[R - 1 - jj]) * P.off[jj];
            val = P.alpha[d] * s + P.beta[d];
            far = !(fabs(val) < (double)kFarOut / (R + 1));
        }
    }
    const bool wide = __any_sync(0xffffffffu, far);
    if (lane < E) {
        const int d = lane / (R + 1), j = lane - (lane / (R + 1)) * (R + 1);
        const int64_t q = wide ? 0 : __double2ll_rn(val * 1099511627776.0);   // * 2^40
        if (j < R) {
            m.coef[d][j] = val;
            m.coef_q[d][j] = q;
        } else {
            m.cst[d] = val;
            m.cst_q[d] = q;
        }
    }
    if (lane == 0) m.wide = wide;
}

// ------------------------------------------------------------ interpolation

// One output value of one channel slab from precomputed taps (separable sum,
// innermost axis first).  off_hi holds the combined offsets of the outer axes.
template <typename T, int R, int MODE>
__device__ __forceinline__ float interp(const T *__restrict__ Xc, const AxisTaps<MODE> (&tp)[R],
                                        const int (&off_hi)[R == 3 ? 16 : 4]) {
    constexpr int K = TapCount<MODE>::K;
    if constexpr (R == 1) {
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const float v = ((tp[0].ok >> k) & 1u) ? IO<T>::ld(Xc + tp[0].idx[k]) : 0.0f;
            s = fmaf(tp[0].w[k], v, s);
        }
        return s;
    } else if constexpr (R == 2) {
        float acc = 0.0f;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
            float s = 0.0f;
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const bool ok = ((tp[0].ok >> ky) & (tp[1].ok >> kx) & 1u) != 0;
                const float v = ok ? IO<T>::ld(Xc + off_hi[ky] + tp[1].idx[kx]) : 0.0f;
                s = fmaf(tp[1].w[kx], v, s);
            }
            acc = fmaf(tp[0].w[ky], s, acc);
        }
        return acc;
    } else {
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
                    const float v = ok ? IO<T>::ld(Xc + off_hi[kz * K + ky] + tp[2].idx[kx]) : 0.0f;
                    s = fmaf(tp[2].w[kx], v, s);
                }
                sz = fmaf(tp[1].w[ky], s, sz);
            }
            acc = fmaf(tp[0].w[kz], sz, acc);
        }
        return acc;
    }
}

// ------------------------------------------------------------ the kernel

// Output-position taps from a 32.32 position per axis.
template <typename T, int R, int MODE, bool AFFINE>
__device__ __forceinline__ void position_taps(const T *__restrict__ src, const SampleParams &P,
                                              const AffineMap &m, int n, int64_t o,
                                              AxisTaps<MODE> (&tp)[R]) {
    const SampleArgs &a = P.a;
    int opos[R];   // output spatial index, outermost first
    int64_t rem = o;
#pragma unroll
    for (int j = R - 1; j >= 0; --j) {
        opos[j] = (int)(rem % a.out[j]);
        rem /= a.out[j];
    }
    if constexpr (AFFINE) {
#pragma unroll
        for (int d = 0; d < R; ++d) {
            int64_t xq;
            if (!m.wide) {
                int64_t acc = m.cst_q[d];
#pragma unroll
                for (int j = 0; j < R; ++j) acc += m.coef_q[d][j] * (int64_t)opos[j];
                xq = acc >> 8;   // 24.40 -> 32.32 (floor)
            } else {
                double x = m.cst[d];
#pragma unroll
                for (int j = 0; j < R; ++j) x += m.coef[d][j] * (double)opos[j];
                xq = pos_to_q(x, P.ax[d], a.pad);
            }
            make_taps<MODE>(xq, P.ax[d], a.pad, a.ac, a.a, tp[d]);
        }
    } else {
        // GridSample grid: the location vector lists the innermost axis first
        const T *g = src + ((int64_t)n * a.out_plane + o) * R;
#pragma unroll
        for (int d = 0; d < R; ++d)
            make_taps<MODE>(grid_to_q(IO<T>::ld(g + (R - 1 - d)), P.ax[d], a.pad), P.ax[d], a.pad,
                            a.ac, a.a, tp[d]);
    }
}

// Combined offsets of the outer axes (rows, or depth*rows) for interp().
template <int R, int MODE>
__device__ __forceinline__ void outer_offsets(const AxisTaps<MODE> (&tp)[R], const SampleArgs &a,
                                              int (&off_hi)[R == 3 ? 16 : 4]) {
    constexpr int K = TapCount<MODE>::K;
    if constexpr (R == 2) {
#pragma unroll
        for (int k = 0; k < K; ++k) off_hi[k] = tp[0].idx[k] * a.in[1];
    } else if constexpr (R == 3) {
#pragma unroll
        for (int kz = 0; kz < K; ++kz)
#pragma unroll
            for (int ky = 0; ky < K; ++ky)
                off_hi[kz * K + ky] = (tp[0].idx[kz] * a.in[1] + tp[1].idx[ky]) * a.in[2];
    }
}

// Flattened taps of one output position: byte offsets inside a channel slab
// (always in range) and combined weights (product of the per-axis weights).
template <int R, int MODE> struct FlatTaps {
    static constexpr int K = TapCount<MODE>::K;
    static constexpr int NT = R == 1 ? K : (R == 2 ? K * K : K * K * K);
    uint32_t off[NT];
    float w[NT];
    uint32_t ok;    // bit t: tap t reads X (clear: it reads 0)
};

template <typename T, int R, int MODE>
__device__ __forceinline__ void flatten_taps(const AxisTaps<MODE> (&tp)[R], const SampleArgs &a,
                                             FlatTaps<R, MODE> &f) {
    constexpr int K = TapCount<MODE>::K;
    f.ok = 0;
    int t = 0;
    if constexpr (R == 1) {
#pragma unroll
        for (int k = 0; k < K; ++k, ++t) {
            f.off[t] = (uint32_t)tp[0].idx[k] * sizeof(T);
            f.w[t] = tp[0].w[k];
            f.ok |= ((tp[0].ok >> k) & 1u) << t;
        }
    } else if constexpr (R == 2) {
#pragma unroll
        for (int ky = 0; ky < K; ++ky)
#pragma unroll
            for (int kx = 0; kx < K; ++kx, ++t) {
                f.off[t] = (uint32_t)(tp[0].idx[ky] * a.in[1] + tp[1].idx[kx]) * sizeof(T);
                f.w[t] = tp[0].w[ky] * tp[1].w[kx];
                f.ok |= ((tp[0].ok >> ky) & (tp[1].ok >> kx) & 1u) << t;
            }
    } else {
#pragma unroll
        for (int kz = 0; kz < K; ++kz)
#pragma unroll
            for (int ky = 0; ky < K; ++ky)
#pragma unroll
                for (int kx = 0; kx < K; ++kx, ++t) {
                    f.off[t] = (uint32_t)((tp[0].idx[kz] * a.in[1] + tp[1].idx[ky]) * a.in[2] +
                                          tp[2].idx[kx]) * sizeof(T);
                    f.w[t] = tp[0].w[kz] * tp[1].w[ky] * tp[2].w[kx];
                    f.ok |= ((tp[0].ok >> kz) & (tp[1].ok >> ky) & (tp[2].ok >> kx) & 1u) << t;
                }
    }
}

template <typename T>
__device__ __forceinline__ float ld_at(const char *base, uint32_t byte_off) {
    return IO<T>::ld(reinterpret_cast<const T *>(base + byte_off));
}

// Channel loop over flattened taps.  `Xb` and `Yb` are warp-uniform channel
// base pointers (block-uniform image, loop-uniform channel), so each load is
// a uniform base plus a per-thread 32-bit offset.  MASKED=false is taken only
// when every tap of the position is in range.
template <typename T, int NT, bool MASKED>
__device__ __forceinline__ void channel_loop(const char *__restrict__ Xb, char *__restrict__ Yb,
                                             int C, int64_t in_bytes, int64_t out_bytes,
                                             const uint32_t (&off)[NT], const float (&w)[NT],
                                             uint32_t ok) {
#pragma unroll 4
    for (int c = 0; c < C; ++c) {
        float acc = 0.0f;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const float v = (!MASKED || ((ok >> t) & 1u)) ? ld_at<T>(Xb, off[t]) : 0.0f;
            acc = fmaf(w[t], v, acc);
        }
        *reinterpret_cast<T *>(Yb) = IO<T>::st(acc);
        Xb += in_bytes;
        Yb += out_bytes;
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
        if (threadIdx.x < 32) build_affine_map_warp<T, R>(src + (int64_t)n * R * (R + 1), P, s_map);
        __syncthreads();
    }
    if (o >= a.out_plane) return;

    AxisTaps<MODE> tp[R];
    position_taps<T, R, MODE, AFFINE>(src, P, s_map, n, o, tp);

    const char *Xb = reinterpret_cast<const char *>(X + (int64_t)n * a.C * a.in_plane);
    char *Yb = reinterpret_cast<char *>(Y + (int64_t)n * a.C * a.out_plane + o);
    const int64_t in_bytes = a.in_plane * (int64_t)sizeof(T);
    const int64_t out_bytes = a.out_plane * (int64_t)sizeof(T);

    if constexpr (R == 3) {
        // rank 3 keeps the separable form: fewer live registers than 8 (or 64)
        // flattened taps, which measures faster here
        int off_hi[16];
        outer_offsets<R, MODE>(tp, a, off_hi);
        const T *Xc = reinterpret_cast<const T *>(Xb);
        T *Yc = reinterpret_cast<T *>(Yb);
#pragma unroll 4
        for (int c = 0; c < a.C; ++c) {
            *Yc = IO<T>::st(interp<T, R, MODE>(Xc, tp, off_hi));
            Xc += a.in_plane;
            Yc += a.out_plane;
        }
    } else {
        FlatTaps<R, MODE> f;
        flatten_taps<T, R, MODE>(tp, a, f);
        constexpr int NT = FlatTaps<R, MODE>::NT;
        if (f.ok == (NT == 32 ? 0xffffffffu : ((1u << NT) - 1u)))
            channel_loop<T, NT, false>(Xb, Yb, a.C, in_bytes, out_bytes, f.off, f.w, f.ok);
        else
            channel_loop<T, NT, true>(Xb, Yb, a.C, in_bytes, out_bytes, f.off, f.w, f.ok);
    }
}

inline Axis make_axis(int n, int ac) {
    Axis A;
    A.n = n;
    A.h = ac ? 0.5f * (float)(n - 1) : 0.5f * (float)n;
    A.period_f = ac ? 2.0f * (float)(n - 1) : 2.0f * (float)n;   // twice the reflection span
    A.pad_ = 0;
    A.c_q = (int64_t)(n - 1) * kHalfQ;                              // (n-1)/2
    A.lo_q = ac ? 0 : -kHalfQ;
    A.span_q = ac ? (int64_t)(n - 1) * kOneQ : (int64_t)n * kOneQ;
    A.hi_q = (int64_t)(n - 1) * kOneQ;
    return A;
}

}  // namespace gs

#include "gs_band.cuh"
#include "gs_nd.cuh"
#include "gs_nhwc.cuh"
#include "gs_vol.cuh"
#include "gs_vol_tma.cuh"

namespace gs {

template <typename T, int R, int MODE, bool AFFINE>
static cudaError_t launch_sample_t(const void *X, const void *src, void *Y, SampleParams P,
                                   cudaStream_t s) {
    if constexpr (AFFINE && R == 2) {
        bool used = false;
        const cudaError_t e = launch_band<T, MODE>(X, src, Y, P, s, &used);
        if (used || e != cudaSuccess) return e;
    }
    if constexpr (AFFINE && R == 3 && MODE != MODE_CUBIC) {
        bool used = false;
        cudaError_t e = launch_vol_tma<T, MODE>(X, src, Y, P, s, &used);
        if (used || e != cudaSuccess) return e;
        e = launch_vol<T, MODE>(X, src, Y, P, s, &used);
        if (used || e != cudaSuccess) return e;
    }

    P.a.tiles = (int)((P.a.out_plane + kSampleThreads - 1) / kSampleThreads);
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
static SampleParams make_params(const SampleArgs &args, int r) {
    SampleParams P;
    P.a = args;
    for (int d = 0; d < kMaxRank; ++d) {
        const int n = d < r ? args.in[d] : 1;
        const int m = d < r ? args.out[d] : 1;
        P.ax[d] = make_axis(n, args.ac);
        // AffineGrid base positions: (2i+1)/m - 1 (align_corners=0) or
        // -1 + 2i/(m-1) (align_corners=1; a single position sits at 0)
        if (args.ac) {
            P.slope[d] = m > 1 ? 2.0 / (double)(m - 1) : 0.0;
            P.off[d] = m > 1 ? -1.0 : 0.0;
        } else {
            P.slope[d] = 2.0 / (double)m;
            P.off[d] = 1.0 / (double)m - 1.0;
        }
        // GridSample unnormalisation x = alpha*g + beta
        P.alpha[d] = args.ac ? 0.5 * (double)(n - 1) : 0.5 * (double)n;
        P.beta[d] = 0.5 * (double)(n - 1);
    }
    return P;
}

template <typename T>
size_t sample_workspace_bytes(const SampleArgs &args, int r, bool affine) {
    return nhwc_workspace_bytes<T>(args, r, affine);
}

template <typename T>
size_t sample_min_workspace_bytes(const SampleArgs &args) {
    return nhwc_min_workspace_bytes<T>(args);
}

template <typename T>
cudaError_t launch_sample(const void *X, const void *src, void *Y, const SampleArgs &args, int r,
                          int mode, bool affine, void *ws, size_t ws_bytes, cudaStream_t s) {
    const SampleParams P = make_params<T>(args, r);
    if (affine) {
        if (r == 2) return launch_sample_mode<T, 2, true>(X, src, Y, P, mode, s);
        return launch_sample_mode<T, 3, true>(X, src, Y, P, mode, s);
    }
    if (r > 3) return launch_sample_nd<T>(X, src, grid_dt_of<T>(), Y, args, r, mode, s);
    if (ws && nhwc_workspace_bytes<T>(args, r, affine) > 0 &&
        ws_bytes >= nhwc_min_workspace_bytes<T>(args))
        return launch_nhwc<T>(X, src, Y, P, mode, ws, ws_bytes, s);
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
