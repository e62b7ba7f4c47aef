// gs_resize.cuh -- Resize (Resize - 18) on the separable sampler.
//
// Resize maps every output axis on its own: output index o -> source
// coordinate x (coordinate_transformation_mode), then taps and 1-D weights
// (nearest with nearest_mode, linear, Keys cubic with cubic_coeff_a; with
// antialias the linear / cubic filter is stretched by 1/scale when
// downscaling and renormalised; exclude_outside drops taps outside the axis
// and renormalises; other taps outside the axis read the edge value).  The
// value is the sum over the tensor product of the taps of the product of
// the weights times X.  tf_crop_and_resize puts extrapolation_value wherever a
// coordinate leaves the input on any axis.
//
// The host folds every axis whose map is the identity into a batch axis of B
// slices, leaving r = 1, 2 or 3 trailing resized axes.  A block owns a tile
// of at most 256 output positions (tz x ty x tx) and a range of slices.  It
// first tabulates the taps of its tile's indices along each axis in shared
// memory (source coordinates in fp64, the precision the operator's
// definition is written in, so the tap choice of nearest and the crop test
// are exact), then each thread takes one position and sweeps the slices,
// holding its taps in registers when every axis has a fixed tap count (1, 2
// or 4) and reading them from shared memory otherwise (antialias).
#pragma once

#include <algorithm>

#include "gs_common.cuh"
#include "gs_internal.h"
#include "gs_ptx.cuh"

namespace gs {

constexpr int kRsThreads = 256;
constexpr int kRsMaxTaps = kRsMaxTapsHost;   // per axis (antialias at scale >= ~1/16 cubic, ~1/32 linear)

// Output tile of a block.
struct ResizeTile {
    int t[3];        // tile extents, outermost axis first (1 for unused axes)
    int tiles[3];    // tiles along each axis
};

__host__ __device__ inline double rs_keys(double s, double a) {
    s = fabs(s);
    if (s <= 1.0) return ((a + 2.0) * s - (a + 3.0)) * s * s + 1.0;
    if (s < 2.0) return ((a * s - 5.0 * a) * s + 8.0 * a) * s - 4.0 * a;
    return 0.0;
}

// Products and sums that decide a tap index or the crop test are rounded one
// by one (no fused multiply-add), on the host and the device alike.
__host__ __device__ inline double rs_mul(double a, double b) {
#ifdef __CUDA_ARCH__
    return __dmul_rn(a, b);
#else
    return a * b;
#endif
}
__host__ __device__ inline double rs_add(double a, double b) {
#ifdef __CUDA_ARCH__
    return __dadd_rn(a, b);
#else
    return a + b;
#endif
}

// Taps of output index o on axis A: indices clamped to the axis (edge values),
// weights; returns the count, or -1 when the element takes
// extrapolation_value.  The count depends only on the axis (the host sets it
// with A.k0 and A.taps), so every entry of a table has the same length.  Runs
// on the host (tables passed to resize_rows_kernel) and on the device (tables
// built per block by resize_kernel).
__host__ __device__ inline int rs_axis_taps(int o, const ResizeAxis &A, const ResizeArgs &p,
                                            int *idx, float *w) {
    const double xr = (double)o;
    double x;
    switch (p.coord) {
        case RS_PYTORCH_HALF_PIXEL:
            x = A.n_out > 1 ? (xr + 0.5) / A.scale - 0.5 : 0.0;
            break;
        case RS_ALIGN_CORNERS:
            x = A.length_resized > 1.0 ? rs_mul(xr, (double)(A.n_in - 1)) / (A.length_resized - 1.0)
                                       : 0.0;
            break;
        case RS_ASYMMETRIC:
            x = xr / A.scale;
            break;
        case RS_TF_CROP_AND_RESIZE:
            x = A.n_out > 1
                    ? rs_add(rs_mul(A.roi_start, (double)(A.n_in - 1)),
                             rs_mul(rs_mul(xr, A.roi_end - A.roi_start), (double)(A.n_in - 1)) /
                                 (double)(A.n_out - 1))
                    : rs_mul(rs_mul(0.5, A.roi_start + A.roi_end), (double)(A.n_in - 1));
            break;
        default:   // half_pixel
            x = (xr + 0.5) / A.scale - 0.5;
            break;
    }
    if (p.coord == RS_TF_CROP_AND_RESIZE && (x < 0.0 || x > (double)(A.n_in - 1))) return -1;
    // keep the integer conversions defined for coordinates far outside
    x = fmin(fmax(x, -1.0e9), 1.0e9);
    const int n = A.n_in;
    int cnt;
    double wd[kRsMaxTaps];
    if (p.mode == MODE_NEAREST) {
        double r;
        switch (p.nearest_mode) {
            case RS_ROUND_PREFER_CEIL: r = floor(x + 0.5); break;
            case RS_FLOOR: r = floor(x); break;
            case RS_CEIL: r = ceil(x); break;
            default: r = ceil(x - 0.5); break;   // round_prefer_floor
        }
        idx[0] = (int)r;
        wd[0] = 1.0;
        cnt = 1;
    } else {
        const double f = floor(x), t = x - f;
        const int i0 = (int)f;
        const double s = A.aa_scale;   // scale when antialiasing a downscale, else 1
        const int k0 = A.k0;           // first tap offset from floor(x); the last is 1 - k0
        cnt = 1 - 2 * k0 + 1;
        double sum = 0.0;
        for (int k = 0; k < cnt; ++k) {
            const double d = ((double)(k0 + k) - t) * s;
            const double wk = p.mode == MODE_LINEAR ? fmax(0.0, 1.0 - fabs(d)) : rs_keys(d, p.a);
            idx[k] = i0 + k0 + k;
            wd[k] = wk;
            sum += wk;
        }
        if (s < 1.0)
            for (int k = 0; k < cnt; ++k) wd[k] /= sum;
    }
    if (p.exclude_outside) {
        double sum = 0.0;
        for (int k = 0; k < cnt; ++k) {
            if (idx[k] < 0 || idx[k] > n - 1) wd[k] = 0.0;
            sum += wd[k];
        }
        if (sum != 0.0)
            for (int k = 0; k < cnt; ++k) wd[k] /= sum;
    }
    for (int k = 0; k < cnt; ++k) {
        idx[k] = idx[k] < 0 ? 0 : (idx[k] > n - 1 ? n - 1 : idx[k]);
        w[k] = (float)wd[k];
    }
    return cnt;
}

// One output value of one slice from per-axis taps (separable sum, innermost
// axis first).  K: taps per axis when fixed (1, 2, 4), 0 when read from the
// shared tables with counts cnt[].
template <typename T, int R, int K>
__device__ __forceinline__ float rs_value(const T *__restrict__ Xs, const ResizeArgs &p,
                                          const int (*ti)[K > 0 ? K : 1],
                                          const float (*tw)[K > 0 ? K : 1],
                                          const int *const *si, const float *const *sw,
                                          const int *cnt) {
    const int W = p.ax[2].n_in, H = p.ax[1].n_in;
    auto row_sum = [&](const T *row) {
        float s = 0.0f;
        if constexpr (K > 0) {
#pragma unroll
            for (int kx = 0; kx < K; ++kx) s = fmaf(tw[2][kx], IO<T>::ld(row + ti[2][kx]), s);
        } else {
            for (int kx = 0; kx < cnt[2]; ++kx) s = fmaf(sw[2][kx], IO<T>::ld(row + si[2][kx]), s);
        }
        return s;
    };
    auto plane_sum = [&](const T *plane) {
        if constexpr (R == 1) {
            return row_sum(plane);
        } else {
            float s = 0.0f;
            if constexpr (K > 0) {
#pragma unroll
                for (int ky = 0; ky < K; ++ky)
                    s = fmaf(tw[1][ky], row_sum(plane + (int64_t)ti[1][ky] * W), s);
            } else {
                for (int ky = 0; ky < cnt[1]; ++ky)
                    s = fmaf(sw[1][ky], row_sum(plane + (int64_t)si[1][ky] * W), s);
            }
            return s;
        }
    };
    if constexpr (R <= 2) {
        return plane_sum(Xs);
    } else {
        float s = 0.0f;
        const int64_t HW = (int64_t)H * W;
        if constexpr (K > 0) {
#pragma unroll
            for (int kz = 0; kz < K; ++kz) s = fmaf(tw[0][kz], plane_sum(Xs + ti[0][kz] * HW), s);
        } else {
            for (int kz = 0; kz < cnt[0]; ++kz) s = fmaf(sw[0][kz], plane_sum(Xs + si[0][kz] * HW), s);
        }
        return s;
    }
}

// Grid: blockIdx.x = tile, blockIdx.y = slice chunk.  Axes are stored in
// p.ax[0..2] outermost first; for R < 3 the leading entries are unit axes.
template <typename T, int R, int K>
__global__ void __launch_bounds__(kRsThreads)
resize_kernel(const T *__restrict__ X, T *__restrict__ Y, const ResizeArgs p, const ResizeTile tl,
              int slices_per_block) {
    extern __shared__ __align__(128) unsigned char rs_smem[];
    const int tid = threadIdx.x;
    int tile = blockIdx.x;
    int tc[3];
    for (int d = 2; d >= 0; --d) {
        tc[d] = tile % tl.tiles[d];
        tile /= tl.tiles[d];
    }
    int o0[3], ext[3];
    for (int d = 0; d < 3; ++d) {
        o0[d] = tc[d] * tl.t[d];
        ext[d] = min(tl.t[d], p.ax[d].n_out - o0[d]);
    }
    // shared tables: per axis, tile entries x taps (index, weight), plus a flag
    int *s_idx[3];
    float *s_w[3];
    int *s_flag[3];
    {
        unsigned char *q = rs_smem;
        for (int d = 0; d < 3; ++d) {
            const int entries = tl.t[d] * p.ax[d].taps;
            s_idx[d] = reinterpret_cast<int *>(q);
            q += (size_t)entries * 4;
            s_w[d] = reinterpret_cast<float *>(q);
            q += (size_t)entries * 4;
            s_flag[d] = reinterpret_cast<int *>(q);
            q += (size_t)tl.t[d] * 4;
        }
    }
    for (int d = 0; d < 3; ++d) {
        for (int e = tid; e < ext[d]; e += kRsThreads) {
            const int taps = p.ax[d].taps;
            if (d < 3 - R) {   // a unit axis: index 0, weight 1
                s_idx[d][e] = 0;
                s_w[d][e] = 1.0f;
                s_flag[d][e] = 0;
                continue;
            }
            int ib[kRsMaxTaps];
            float wb[kRsMaxTaps];
            const int c = rs_axis_taps(o0[d] + e, p.ax[d], p, ib, wb);
            s_flag[d][e] = c < 0 ? 1 : 0;
            for (int k = 0; k < taps; ++k) {
                s_idx[d][e * taps + k] = c < 0 ? 0 : ib[k];
                s_w[d][e * taps + k] = c < 0 ? 0.0f : wb[k];
            }
        }
    }
    __syncthreads();

    // this thread's position in the tile
    const int tx = tl.t[2], ty = tl.t[1];
    const int pz = tid / (tx * ty), py = (tid / tx) % ty, px = tid % tx;
    const int pe[3] = {pz, py, px};
    if (pz >= tl.t[0] || pz >= ext[0] || py >= ext[1] || px >= ext[2]) return;
    const bool extrap = s_flag[0][pz] | s_flag[1][py] | s_flag[2][px];

    constexpr int KK = K > 0 ? K : 1;
    int ti[3][KK];
    float tw[3][KK];
    const int *si[3];
    const float *sw[3];
    int cnt[3];
#pragma unroll
    for (int d = 0; d < 3; ++d) {
        cnt[d] = p.ax[d].taps;
        si[d] = s_idx[d] + pe[d] * cnt[d];
        sw[d] = s_w[d] + pe[d] * cnt[d];
        if constexpr (K > 0) {
            if (d >= 3 - R) {   // resized axes hold K taps each
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    ti[d][k] = si[d][k];
                    tw[d][k] = sw[d][k];
                }
            }
        }
    }

    const int64_t in_slice = (int64_t)p.ax[0].n_in * p.ax[1].n_in * p.ax[2].n_in;
    const int64_t out_slice = (int64_t)p.ax[0].n_out * p.ax[1].n_out * p.ax[2].n_out;
    const int64_t oidx = ((int64_t)(o0[0] + pz) * p.ax[1].n_out + (o0[1] + py)) * p.ax[2].n_out +
                         (o0[2] + px);
    const int64_t b0 = (int64_t)blockIdx.y * slices_per_block;
    const int64_t b1 = min((int64_t)p.B, b0 + slices_per_block);
    const T *Xs = X + b0 * in_slice;
    T *Yp = Y + b0 * out_slice + oidx;
    if (extrap) {
        const T v = IO<T>::st(p.extrapolation_value);
        for (int64_t b = b0; b < b1; ++b, Yp += out_slice) *Yp = v;
        return;
    }
    constexpr int KR = K == 0 ? 0 : (R == 1 ? K : (R == 2 ? K * K : K * K * K));
    if constexpr (K > 0 && KR <= 16) {
        // the tap tuple flattened: offsets inside a slice and weight products,
        // row-major over the axes (the order of the operator's sum)
        int off[KR];
        float wt[KR];
#pragma unroll
        for (int t = 0; t < KR; ++t) {
            int rem = t;
            const int kx = rem % K;
            rem /= K;
            const int ky = R >= 2 ? rem % K : 0;
            const int kz = R >= 3 ? rem / K : 0;
            const int iz = R >= 3 ? ti[0][kz] : 0, iy = R >= 2 ? ti[1][ky] : 0;
            off[t] = (iz * p.ax[1].n_in + iy) * p.ax[2].n_in + ti[2][kx];
            wt[t] = (R >= 3 ? tw[0][kz] : 1.0f) * (R >= 2 ? tw[1][ky] : 1.0f) * tw[2][kx];
        }
        // four independent slices per step: all their loads are in flight together
        int64_t b = b0;
        for (; b + 4 <= b1; b += 4) {
            float acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc[u] = 0.0f;
#pragma unroll
                for (int t = 0; t < KR; ++t)
                    acc[u] = fmaf(wt[t], IO<T>::ld(Xs + u * in_slice + off[t]), acc[u]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) Yp[u * out_slice] = IO<T>::st(acc[u]);
            Xs += 4 * in_slice;
            Yp += 4 * out_slice;
        }
        for (; b < b1; ++b) {
            float acc = 0.0f;
#pragma unroll
            for (int t = 0; t < KR; ++t) acc = fmaf(wt[t], IO<T>::ld(Xs + off[t]), acc);
            *Yp = IO<T>::st(acc);
            Xs += in_slice;
            Yp += out_slice;
        }
    } else {
        for (int64_t b = b0; b < b1; ++b) {
            *Yp = IO<T>::st(rs_value<T, R, K>(Xs, p, ti, tw, si, sw, cnt));
            Xs += in_slice;
            Yp += out_slice;
        }
    }
}

// ------------------------------------------------------------------
// Row kernel (resizes of one or two trailing axes): per-axis tap tables built
// once on the host, in the same fp64 arithmetic, and passed as a kernel
// parameter.  A block owns a band of output rows, full width, for a range of
// slices; a thread owns output columns x = tid, tid + 256, ... (at most four)
// and keeps their taps in registers.  Warps read whole input rows.

constexpr int kRsTableBytes = 30 * 1024;   // kernel parameters hold up to 32 KB
constexpr int kRsRowsMaxCols = 4;           // output columns per thread

struct ResizeTables {
    int nx, ny, kx, ky;   // output extents (rows axis, columns axis) and taps per index
    // x idx[nx*kx] (int), x w[nx*kx] (float), y idx[ny*ky], y w[ny*ky],
    // x flags[nx], y flags[ny] (1: extrapolation_value)
    unsigned char data[kRsTableBytes];
};

inline size_t rs_table_bytes(int nx, int kx, int ny, int ky) {
    return ((size_t)nx * kx + (size_t)ny * ky) * 8 + (size_t)nx + (size_t)ny;
}

template <typename T, int KY, int KX>
__global__ void __launch_bounds__(kRsThreads)
resize_rows_kernel(const T *__restrict__ X, T *__restrict__ Y, const __grid_constant__ ResizeTables tb,
                   int64_t B, int H, int W, int rows_per_block, int slices_per_block,
                   float extrapolation_value) {
    const int nx = tb.nx, ny = tb.ny;
    const int *xi = reinterpret_cast<const int *>(tb.data);
    const float *xw = reinterpret_cast<const float *>(tb.data + (size_t)nx * KX * 4);
    const int *yi = reinterpret_cast<const int *>(tb.data + (size_t)nx * KX * 8);
    const float *yw = reinterpret_cast<const float *>(tb.data + (size_t)nx * KX * 8 + (size_t)ny * KY * 4);
    const unsigned char *xf = tb.data + ((size_t)nx * KX + (size_t)ny * KY) * 8;
    const unsigned char *yf = xf + nx;

    const int y0 = blockIdx.x * rows_per_block;
    const int y1 = min(ny, y0 + rows_per_block);
    const int64_t b0 = (int64_t)blockIdx.y * slices_per_block;
    const int64_t b1 = min(B, b0 + slices_per_block);
    const int tid = threadIdx.x;

    // this thread's columns and their taps
    int cx[kRsRowsMaxCols][KX];
    float cw[kRsRowsMaxCols][KX];
    bool cf[kRsRowsMaxCols];
    int ncols = 0;
#pragma unroll
    for (int j = 0; j < kRsRowsMaxCols; ++j) {
        const int x = tid + j * kRsThreads;
        const bool in = x < nx;
        if (in) ncols = j + 1;
#pragma unroll
        for (int k = 0; k < KX; ++k) {
            cx[j][k] = in ? xi[x * KX + k] : 0;
            cw[j][k] = in ? xw[x * KX + k] : 0.0f;
        }
        cf[j] = in && xf[x];
    }
    const int64_t in_slice = (int64_t)H * W, out_slice = (int64_t)ny * nx;
    // rows outer (their taps read once), slices inner, four slices per step so
    // their loads are in flight together
    for (int y = y0; y < y1; ++y) {
        int ry[KY];
        float wy[KY];
#pragma unroll
        for (int k = 0; k < KY; ++k) {
            ry[k] = yi[y * KY + k];
            wy[k] = yw[y * KY + k];
        }
        const bool fy = yf[y] != 0;
#pragma unroll
        for (int j = 0; j < kRsRowsMaxCols; ++j) {
            if (j >= ncols) break;
            const int x = tid + j * kRsThreads;
            const T *rows[KY];
#pragma unroll
            for (int k = 0; k < KY; ++k) rows[k] = X + b0 * in_slice + (int64_t)ry[k] * W;
            T *yp = Y + b0 * out_slice + (int64_t)y * nx + x;
            if (fy || cf[j]) {
                const T v = IO<T>::st(extrapolation_value);
                for (int64_t b = b0; b < b1; ++b, yp += out_slice) *yp = v;
                continue;
            }
            int64_t b = b0;
            for (; b + 4 <= b1; b += 4) {
                float acc[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc[u] = 0.0f;
#pragma unroll
                    for (int ky = 0; ky < KY; ++ky) {
                        const T *row = rows[ky] + u * in_slice;
                        float sx = 0.0f;
#pragma unroll
                        for (int kx = 0; kx < KX; ++kx) sx = fmaf(cw[j][kx], IO<T>::ld(row + cx[j][kx]), sx);
                        acc[u] = fmaf(wy[ky], sx, acc[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) yp[u * out_slice] = IO<T>::st(acc[u]);
#pragma unroll
                for (int k = 0; k < KY; ++k) rows[k] += 4 * in_slice;
                yp += 4 * out_slice;
            }
            for (; b < b1; ++b) {
                float acc = 0.0f;
#pragma unroll
                for (int ky = 0; ky < KY; ++ky) {
                    float sx = 0.0f;
#pragma unroll
                    for (int kx = 0; kx < KX; ++kx) sx = fmaf(cw[j][kx], IO<T>::ld(rows[ky] + cx[j][kx]), sx);
                    acc = fmaf(wy[ky], sx, acc);
                }
                *yp = IO<T>::st(acc);
#pragma unroll
                for (int k = 0; k < KY; ++k) rows[k] += in_slice;
                yp += out_slice;
            }
        }
    }
}

// Per-axis tap tables of the row kernels (r <= 2, fixed tap counts): false
// when they do not fit the kernel parameters.
inline bool build_resize_tables(const ResizeArgs &p, ResizeTables &tb) {
    if (p.r > 2) return false;
    const ResizeAxis &AX = p.ax[2], &AY = p.ax[1];
    const int kx = AX.taps, ky = p.r == 2 ? AY.taps : 1;
    const bool ok_taps = (p.r == 2 && kx == ky && (kx == 1 || kx == 2 || kx == 4)) ||
                         (p.r == 1 && (kx == 1 || kx == 2 || kx == 4));
    if (!ok_taps || AX.n_out > kRsThreads * kRsRowsMaxCols) return false;
    const int nx = AX.n_out, ny = p.r == 2 ? AY.n_out : 1;
    if (rs_table_bytes(nx, kx, ny, ky) > (size_t)kRsTableBytes) return false;
    tb.nx = nx;
    tb.ny = ny;
    tb.kx = kx;
    tb.ky = ky;
    int *xi = reinterpret_cast<int *>(tb.data);
    float *xw = reinterpret_cast<float *>(tb.data + (size_t)nx * kx * 4);
    int *yi = reinterpret_cast<int *>(tb.data + (size_t)nx * kx * 8);
    float *yw = reinterpret_cast<float *>(tb.data + (size_t)nx * kx * 8 + (size_t)ny * ky * 4);
    unsigned char *xf = tb.data + ((size_t)nx * kx + (size_t)ny * ky) * 8;
    unsigned char *yf = xf + nx;
    int ib[kRsMaxTaps];
    float wb[kRsMaxTaps];
    for (int o = 0; o < nx; ++o) {
        const int c = rs_axis_taps(o, AX, p, ib, wb);
        xf[o] = c < 0 ? 1 : 0;
        for (int k = 0; k < kx; ++k) {
            xi[o * kx + k] = c < 0 ? 0 : ib[k];
            xw[o * kx + k] = c < 0 ? 0.0f : wb[k];
        }
    }
    for (int o = 0; o < ny; ++o) {
        int c = 1;
        if (p.r == 2) {
            c = rs_axis_taps(o, AY, p, ib, wb);
        } else {
            ib[0] = 0;
            wb[0] = 1.0f;
        }
        yf[o] = c < 0 ? 1 : 0;
        for (int k = 0; k < ky; ++k) {
            yi[o * ky + k] = c < 0 ? 0 : ib[k];
            yw[o * ky + k] = c < 0 ? 0.0f : wb[k];
        }
    }
    return true;
}

template <typename T, int KY, int KX>
static void launch_rows_kernel(const T *X, T *Y, const ResizeTables &tb, const ResizeArgs &p,
                               dim3 grid, int rows, int per, cudaStream_t s) {
    const int H = p.r == 2 ? p.ax[1].n_in : 1, W = p.ax[2].n_in;
    resize_rows_kernel<T, KY, KX><<<grid, kRsThreads, 0, s>>>(X, Y, tb, p.B, H, W, rows, per,
                                                              p.extrapolation_value);
}

// Row kernel for r <= 2 and fixed tap counts when the tables fit the kernel
// parameters; *used reports whether it ran.
template <typename T>
cudaError_t launch_resize_rows(const void *X, void *Y, const ResizeArgs &p, cudaStream_t s,
                               bool *used) {
    *used = false;
    ResizeTables tb;
    if (!build_resize_tables(p, tb)) return cudaSuccess;
    const int ny = tb.ny, kx = tb.kx, ky = tb.ky;
    // enough blocks for several waves: bands of rows x chunks of slices
    int rows = 8;
    int64_t per = 64;
    auto blocks = [&](int r_, int64_t p_) {
        return (int64_t)((ny + r_ - 1) / r_) * ((p.B + p_ - 1) / p_);
    };
    while (per > 1 && blocks(rows, per) < 8 * 152) per >>= 1;
    while (rows > 1 && blocks(rows, per) < 8 * 152) rows >>= 1;
    per = std::max<int64_t>(per, (p.B + 65534) / 65535);
    const dim3 grid((unsigned)((ny + rows - 1) / rows), (unsigned)((p.B + per - 1) / per));
    const T *x = (const T *)X;
    T *y = (T *)Y;
    if (kx == 1 && ky == 1) launch_rows_kernel<T, 1, 1>(x, y, tb, p, grid, rows, (int)per, s);
    else if (ky == 1 && kx == 2) launch_rows_kernel<T, 1, 2>(x, y, tb, p, grid, rows, (int)per, s);
    else if (ky == 1 && kx == 4) launch_rows_kernel<T, 1, 4>(x, y, tb, p, grid, rows, (int)per, s);
    else if (kx == 2) launch_rows_kernel<T, 2, 2>(x, y, tb, p, grid, rows, (int)per, s);
    else launch_rows_kernel<T, 4, 4>(x, y, tb, p, grid, rows, (int)per, s);
    *used = true;
    return cudaGetLastError();
}

// ------------------------------------------------------------------
// Staged row kernel: the row kernel's tables and loop, with a slice's input
// rows copied into shared memory first.  A block owns a band of output rows
// (full width) for a range of slices.  The rows the band's taps read form
// one contiguous range of every slice, so one bulk async copy per slice
// (counted on an mbarrier) fills a stage of a ring; the taps are then
// shared-memory loads instead of cached global gathers.  The arithmetic (and
// so every bit of the result) is the row kernel's.

constexpr int kRsStageRing = 48 * 1024;   // four blocks per SM
constexpr int kRsStageMax = 16;
constexpr int kRsStageRows = 32;          // output rows per band, at most

// Thread 0 of a staged block: the input rows the band's taps read (rows set
// to extrapolation_value read none), the stages of that many rows that fit
// the ring, the stage barriers, and the copies of the first slices, one bulk
// async copy per slice.
template <typename T, int KY>
__device__ __forceinline__ void rs_ring_start(const T *__restrict__ X, const int *yi,
                                              const unsigned char *yf, int y0, int y1, int64_t b0,
                                              int nb, int64_t in_slice, int W, uint32_t row_bytes,
                                              unsigned char *ring, uint64_t *full, int *r0,
                                              int *rows, int *stages_out) {
    int lo = 0x7fffffff, hi = -1;
    for (int y = y0; y < y1; ++y) {
        if (yf[y]) continue;
        for (int k = 0; k < KY; ++k) {
            lo = min(lo, yi[y * KY + k]);
            hi = max(hi, yi[y * KY + k]);
        }
    }
    if (hi < 0) lo = hi = 0;
    const uint32_t stage = (uint32_t)(hi - lo + 1) * row_bytes;
    const int stages = min(kRsStageMax, (int)(kRsStageRing / stage));   // >= 2 (host)
    for (int st = 0; st < kRsStageMax; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
    const T *src = X + b0 * in_slice + (int64_t)lo * W;
    for (int st = 0; st < stages && st < nb; ++st) {
        mbar_arrive_expect_tx(&full[st], stage);
        bulk_copy_g2s(ring + (size_t)st * stage, src + (int64_t)st * in_slice, stage, &full[st]);
    }
    *r0 = lo;
    *rows = hi - lo + 1;
    *stages_out = stages;
}

// All threads of a staged block: the band's row taps in shared memory (byte
// offsets within a stage, weights, extrapolation flags), read once per block
// rather than from the parameter table for every slice.
template <int KY>
__device__ __forceinline__ void rs_band_rows(const int *yi, const float *yw, const unsigned char *yf,
                                             int y0, int y1, int r0, uint32_t row_bytes,
                                             uint32_t *s_ry, float *s_wy, int *s_fy) {
    for (int e = threadIdx.x; e < (y1 - y0) * KY; e += kRsThreads) {
        const int y = y0 + e / KY, k = e - (e / KY) * KY;
        // rows set to extrapolation_value never read their (zero) offsets
        s_ry[e] = yf[y] ? 0u : (uint32_t)(yi[y * KY + k] - r0) * row_bytes;
        s_wy[e] = yw[y * KY + k];
        if (k == 0) s_fy[e / KY] = yf[y];
    }
}

template <typename T, int KY, int KX, int G>
__global__ void __launch_bounds__(kRsThreads, 4)
resize_stage_kernel(const T *__restrict__ X, T *__restrict__ Y,
                    const __grid_constant__ ResizeTables tb, int64_t B, int H, int W,
                    int rows_per_block, int slices_per_block, float extrapolation_value,
                    unsigned *err) {
    extern __shared__ __align__(128) unsigned char rs_smem[];
    __shared__ __align__(8) uint64_t full[kRsStageMax];
    __shared__ int s_r0, s_rows, s_stages, s_abort;
    // the band's row taps: byte offsets within a stage, weights, flags (read
    // once here rather than from the parameter table for every slice)
    __shared__ uint32_t s_ry[kRsStageRows * KY];
    __shared__ float s_wy[kRsStageRows * KY];
    __shared__ int s_fy[kRsStageRows];
    const int nx = tb.nx, ny = tb.ny;
    const int *xi = reinterpret_cast<const int *>(tb.data);
    const float *xw = reinterpret_cast<const float *>(tb.data + (size_t)nx * KX * 4);
    const int *yi = reinterpret_cast<const int *>(tb.data + (size_t)nx * KX * 8);
    const float *yw = reinterpret_cast<const float *>(tb.data + (size_t)nx * KX * 8 + (size_t)ny * KY * 4);
    const unsigned char *xf = tb.data + ((size_t)nx * KX + (size_t)ny * KY) * 8;
    const unsigned char *yf = xf + nx;

    const int y0 = blockIdx.x * rows_per_block;
    const int y1 = min(ny, y0 + rows_per_block);
    const int64_t b0 = (int64_t)blockIdx.y * slices_per_block;
    const int nb = (int)(min(B, b0 + slices_per_block) - b0);
    const int tid = threadIdx.x;
    const int64_t in_slice = (int64_t)H * W, out_slice = (int64_t)ny * nx;
    const uint32_t row_bytes = (uint32_t)W * (uint32_t)sizeof(T);

    if (tid == 0) {
        rs_ring_start<T, KY>(X, yi, yf, y0, y1, b0, nb, in_slice, W, row_bytes, rs_smem, full,
                             &s_r0, &s_rows, &s_stages);
        s_abort = 0;
    }

    // this thread's columns: byte offsets of their taps within a row, weights
    uint32_t cx[kRsRowsMaxCols][KX];
    float cw[kRsRowsMaxCols][KX];
    bool cf[kRsRowsMaxCols];
    int ncols = 0;
#pragma unroll
    for (int j = 0; j < kRsRowsMaxCols; ++j) {
        const int x = tid + j * kRsThreads;
        const bool in = x < nx;
        if (in) ncols = j + 1;
#pragma unroll
        for (int k = 0; k < KX; ++k) {
            cx[j][k] = in ? (uint32_t)xi[x * KX + k] * (uint32_t)sizeof(T) : 0u;
            cw[j][k] = in ? xw[x * KX + k] : 0.0f;
        }
        cf[j] = in && xf[x];
    }
    __syncthreads();
    const int S = s_stages, r0 = s_r0;
    const uint32_t stage_bytes = (uint32_t)s_rows * row_bytes;
    rs_band_rows<KY>(yi, yw, yf, y0, y1, r0, row_bytes, s_ry, s_wy, s_fy);
    __syncthreads();
    const uint32_t ring = smem_u32(rs_smem);
    const T *src = X + b0 * in_slice + (int64_t)r0 * W;
    const T ext = IO<T>::st(extrapolation_value);

    // G slices per pass (their stages land, are read and are refilled
    // together), so each row's taps are read once for all G; the host picks
    // G <= S/2, which keeps the next group's copies in flight meanwhile
    int st = 0;
    uint32_t parity = 0;
    int c = 0;
    while (c < nb) {
        const int gn = min(G, nb - c);
        uint32_t base[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (g >= gn) break;
            const int sg = st + g < S ? st + g : st + g - S;
            const uint32_t pg = st + g < S ? parity : parity ^ 1u;
            if (!mbar_wait_bounded(&full[sg], pg, err)) s_abort = 1;
            base[g] = ring + (uint32_t)sg * stage_bytes;
        }
        __syncthreads();   // every thread has waited (or given up) on the group's stages
        if (s_abort) break;
        T *yslice = Y + (b0 + c) * out_slice;
        for (int y = y0; y < y1; ++y) {
            uint32_t ry[KY];
            float wy[KY];
#pragma unroll
            for (int k = 0; k < KY; ++k) {
                ry[k] = s_ry[(y - y0) * KY + k];
                wy[k] = s_wy[(y - y0) * KY + k];
            }
            const bool fy = s_fy[y - y0] != 0;
            T *yrow = yslice + (int64_t)y * nx + tid;
#pragma unroll
            for (int j = 0; j < kRsRowsMaxCols; ++j) {
                if (j >= ncols) break;
                const int x = tid + j * kRsThreads;
                if (x >= nx) break;
                if (fy || cf[j]) {
                    for (int g = 0; g < gn; ++g) yrow[g * out_slice + j * kRsThreads] = ext;
                    continue;
                }
                float acc[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    acc[g] = 0.0f;
                    if (g >= gn) continue;
#pragma unroll
                    for (int ky = 0; ky < KY; ++ky) {
                        const uint32_t row = base[g] + ry[ky];
                        float sx = 0.0f;
#pragma unroll
                        for (int kx = 0; kx < KX; ++kx) sx = fmaf(cw[j][kx], lds_at<T>(row + cx[j][kx]), sx);
                        acc[g] = fmaf(wy[ky], sx, acc[g]);
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g)
                    if (g < gn) yrow[g * out_slice + j * kRsThreads] = IO<T>::st(acc[g]);
            }
        }
        __syncthreads();   // the group's stages fully read
        if (tid == 0) {
            fence_proxy_async_smem();
            for (int g = 0; g < gn; ++g) {
                if (c + g + S >= nb) break;
                const int sg = st + g < S ? st + g : st + g - S;
                mbar_arrive_expect_tx(&full[sg], stage_bytes);
                bulk_copy_g2s(rs_smem + (size_t)sg * stage_bytes,
                              src + (int64_t)(c + g + S) * in_slice, stage_bytes, &full[sg]);
            }
        }
        c += gn;
        st += gn;
        if (st >= S) {
            st -= S;
            parity ^= 1u;
        }
    }
    if (c < nb && tid == 0) {
        // a wait gave up: let the copies still in flight land before the
        // block's shared memory is released (bounded again)
        for (int cc = c; cc < nb && cc < c + S; ++cc)
            mbar_wait_bounded(&full[cc % S], (uint32_t)(cc / S) & 1u, nullptr);
    }
}

// Two adjacent 16-bit outputs from an fp32 pair, each rounded to nearest even
// as IO<T>::st rounds it, packed into one 32-bit word.
template <typename T> __device__ __forceinline__ uint32_t rs_pack2(float2 v) {
    if constexpr (std::is_same<T, __half>::value) {
        const __half2 h = __floats2half2_rn(v.x, v.y);
        return *reinterpret_cast<const uint32_t *>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
        return *reinterpret_cast<const uint32_t *>(&h);
    }
}

// resize_stage_kernel for 16-bit types with an even output width of at most
// 512: a thread makes two adjacent outputs (x = 2p, 2p + 1) of G slices per
// row, their horizontal taps on packed fp32 FMAs (fma.rn.f32x2, each lane
// rounded as fmaf), one packed conversion and one 4-byte store per pair.
// Widths of at most 256 take two or more rows per pass (256 / (width / 2)).
// Same stage ring, tables and per-output arithmetic as resize_stage_kernel.
template <typename T, int KY, int KX, int G>
__global__ void __launch_bounds__(kRsThreads, 4)
resize_pair_kernel(const T *__restrict__ X, T *__restrict__ Y,
                   const __grid_constant__ ResizeTables tb, int64_t B, int H, int W,
                   int rows_per_block, int slices_per_block, float extrapolation_value,
                   unsigned *err) {
    extern __shared__ __align__(128) unsigned char rs_smem[];
    __shared__ __align__(8) uint64_t full[kRsStageMax];
    __shared__ int s_r0, s_rows, s_stages;
    __shared__ uint32_t s_ry[kRsStageRows * KY];
    __shared__ float s_wy[kRsStageRows * KY];
    __shared__ int s_fy[kRsStageRows];
    const int nx = tb.nx, ny = tb.ny;
    const int *xi = reinterpret_cast<const int *>(tb.data);
    const float *xw = reinterpret_cast<const float *>(tb.data + (size_t)nx * KX * 4);
    const int *yi = reinterpret_cast<const int *>(tb.data + (size_t)nx * KX * 8);
    const float *yw = reinterpret_cast<const float *>(tb.data + (size_t)nx * KX * 8 + (size_t)ny * KY * 4);
    const unsigned char *xf = tb.data + ((size_t)nx * KX + (size_t)ny * KY) * 8;
    const unsigned char *yf = xf + nx;

    const int y0 = blockIdx.x * rows_per_block;
    const int y1 = min(ny, y0 + rows_per_block);
    const int64_t b0 = (int64_t)blockIdx.y * slices_per_block;
    const int nb = (int)(min(B, b0 + slices_per_block) - b0);
    const int tid = threadIdx.x;
    const int64_t in_slice = (int64_t)H * W, out_slice = (int64_t)ny * nx;
    const uint32_t row_bytes = (uint32_t)W * (uint32_t)sizeof(T);

    if (tid == 0)
        rs_ring_start<T, KY>(X, yi, yf, y0, y1, b0, nb, in_slice, W, row_bytes, rs_smem, full,
                             &s_r0, &s_rows, &s_stages);

    // this thread's column pair and first row of each pass
    const int npairs = nx >> 1;
    const int rpp = kRsThreads / npairs;   // rows per pass (>= 1: nx <= 512)
    const int pr = tid / npairs, pc = tid - pr * npairs;
    const bool active = pr < rpp;
    const int x0 = 2 * pc;
    uint32_t c0[KX], c1[KX];
    float2 cw[KX];   // (weight of column x0, of column x0 + 1), tap by tap
    bool f0 = false, f1 = false;
#pragma unroll
    for (int k = 0; k < KX; ++k) {
        c0[k] = 0u;
        c1[k] = 0u;
        cw[k] = make_float2(0.0f, 0.0f);
    }
    if (active) {
        f0 = xf[x0] != 0;
        f1 = xf[x0 + 1] != 0;
#pragma unroll
        for (int k = 0; k < KX; ++k) {
            // an extrapolated column reads offset 0 (in the stage) and stores
            // extrapolation_value instead
            c0[k] = f0 ? 0u : (uint32_t)xi[x0 * KX + k] * (uint32_t)sizeof(T);
            c1[k] = f1 ? 0u : (uint32_t)xi[(x0 + 1) * KX + k] * (uint32_t)sizeof(T);
            cw[k] = make_float2(xw[x0 * KX + k], xw[(x0 + 1) * KX + k]);
        }
    }
    __syncthreads();
    const int S = s_stages, r0 = s_r0;
    const uint32_t stage_bytes = (uint32_t)s_rows * row_bytes;
    rs_band_rows<KY>(yi, yw, yf, y0, y1, r0, row_bytes, s_ry, s_wy, s_fy);
    __syncthreads();
    const uint32_t ring = smem_u32(rs_smem);
    const T *src = X + b0 * in_slice + (int64_t)r0 * W;
    const float ext = extrapolation_value;

    int st = 0;
    uint32_t parity = 0;
    int c = 0;
    while (c < nb) {
        const int gn = min(G, nb - c);
        uint32_t base[G];
        bool bad = false;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            if (g >= gn) break;
            const int sg = st + g < S ? st + g : st + g - S;
            const uint32_t pg = st + g < S ? parity : parity ^ 1u;
            if (!bad && !mbar_wait_bounded(&full[sg], pg, err)) bad = true;
            base[g] = ring + (uint32_t)sg * stage_bytes;
        }
        if (__syncthreads_or(bad)) break;   // every thread has waited (or given up)
        if (active) {
            uint32_t *yslice = reinterpret_cast<uint32_t *>(Y + (b0 + c) * out_slice);
            for (int y = y0 + pr; y < y1; y += rpp) {
                uint32_t ry[KY];
                float2 wy[KY];
#pragma unroll
                for (int k = 0; k < KY; ++k) {
                    ry[k] = s_ry[(y - y0) * KY + k];
                    const float w = s_wy[(y - y0) * KY + k];
                    wy[k] = make_float2(w, w);
                }
                const bool fy = s_fy[y - y0] != 0;
                float2 acc[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    acc[g] = make_float2(0.0f, 0.0f);
                    if (g >= gn) continue;
#pragma unroll
                    for (int ky = 0; ky < KY; ++ky) {
                        const uint32_t row = base[g] + ry[ky];
                        float2 sx = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int kx = 0; kx < KX; ++kx)
                            sx = fma_f32x2(cw[kx], make_float2(lds_at<T>(row + c0[kx]), lds_at<T>(row + c1[kx])), sx);
                        acc[g] = fma_f32x2(wy[ky], sx, acc[g]);
                    }
                }
                // the pair as one 32-bit word: (x0, x0 + 1) at element y * nx + x0
                uint32_t *yp = yslice + (((int64_t)y * nx + x0) >> 1);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (g >= gn) break;
                    float2 v = acc[g];
                    if (fy || f0) v.x = ext;
                    if (fy || f1) v.y = ext;
                    yp[g * (out_slice >> 1)] = rs_pack2<T>(v);
                }
            }
        }
        __syncthreads();   // the group's stages fully read
        if (tid == 0) {
            fence_proxy_async_smem();
            for (int g = 0; g < gn; ++g) {
                if (c + g + S >= nb) break;
                const int sg = st + g < S ? st + g : st + g - S;
                mbar_arrive_expect_tx(&full[sg], stage_bytes);
                bulk_copy_g2s(rs_smem + (size_t)sg * stage_bytes,
                              src + (int64_t)(c + g + S) * in_slice, stage_bytes, &full[sg]);
            }
        }
        c += gn;
        st += gn;
        if (st >= S) {
            st -= S;
            parity ^= 1u;
        }
    }
    if (c < nb && tid == 0) {
        // a wait gave up: let the copies still in flight land before the
        // block's shared memory is released (bounded again)
        for (int cc = c; cc < nb && cc < c + S; ++cc)
            mbar_wait_bounded(&full[cc % S], (uint32_t)(cc / S) & 1u, nullptr);
    }
}

// 16-bit types with an even output width up to 512 and Y aligned to a pair
// run resize_pair_kernel (two outputs per thread on packed FMAs).
template <typename T> inline bool rs_takes_pair(int nx, const void *Y) {
    return sizeof(T) == 2 && nx % 2 == 0 && nx <= 2 * kRsThreads &&
           (uintptr_t)Y % (2 * sizeof(T)) == 0;
}

template <typename T, int KY, int KX, int G>
static cudaError_t launch_stage_g(const T *X, T *Y, const ResizeTables &tb, const ResizeArgs &p,
                                  dim3 grid, int rows, int per, unsigned *err, cudaStream_t s) {
    const int H = p.r == 2 ? p.ax[1].n_in : 1, W = p.ax[2].n_in;
    if (rs_takes_pair<T>(tb.nx, Y)) {
        static DeviceFlags pair_set;
        const cudaError_t e = once_per_device(pair_set, [] {
            return cudaFuncSetAttribute(resize_pair_kernel<T, KY, KX, G>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, kRsStageRing);
        });
        if (e != cudaSuccess) return e;
        resize_pair_kernel<T, KY, KX, G><<<grid, kRsThreads, kRsStageRing, s>>>(
            X, Y, tb, p.B, H, W, rows, per, p.extrapolation_value, err);
        return cudaGetLastError();
    }
    static DeviceFlags attr_set;
    const cudaError_t e = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(resize_stage_kernel<T, KY, KX, G>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kRsStageRing);
    });
    if (e != cudaSuccess) return e;
    resize_stage_kernel<T, KY, KX, G><<<grid, kRsThreads, kRsStageRing, s>>>(
        X, Y, tb, p.B, H, W, rows, per, p.extrapolation_value, err);
    return cudaGetLastError();
}

// G: slices per pass, at most half the stages.  Sixteen taps per output
// (4 x 4) keep G = 1: grouping them spills registers.
template <typename T, int KY, int KX>
static cudaError_t launch_stage_kernel(const T *X, T *Y, const ResizeTables &tb,
                                       const ResizeArgs &p, dim3 grid, int rows, int per,
                                       int stages, unsigned *err, cudaStream_t s) {
    if (KY * KX < 16 && stages >= 8)
        return launch_stage_g<T, KY, KX, (KY * KX < 16 ? 4 : 1)>(X, Y, tb, p, grid, rows, per, err, s);
    if (KY * KX < 16 && stages >= 4)
        return launch_stage_g<T, KY, KX, (KY * KX < 16 ? 2 : 1)>(X, Y, tb, p, grid, rows, per, err, s);
    return launch_stage_g<T, KY, KX, 1>(X, Y, tb, p, grid, rows, per, err, s);
}

// Staged row kernel when the row kernel's tables apply, rows are whole
// 16-byte chunks and every band's input rows fit two stages; *used reports
// whether it ran.
template <typename T>
cudaError_t launch_resize_stage(const void *X, void *Y, const ResizeArgs &p, unsigned *err,
                                cudaStream_t s, bool *used) {
    *used = false;
    const int W = p.ax[2].n_in;
    if (((size_t)W * sizeof(T)) % 16 != 0 || (uintptr_t)X % 16 != 0) return cudaSuccess;
    ResizeTables tb;
    if (!build_resize_tables(p, tb)) return cudaSuccess;
    const int ny = tb.ny, kx = tb.kx, ky = tb.ky;
    // fp32 with at most four taps per output measured faster on the row
    // kernel (2x bilinear upscale of 16x64x128x128: 108 us there, 129 us here)
    if (sizeof(T) == 4 && kx * ky <= 4) return cudaSuccess;
    const int *yi = reinterpret_cast<const int *>(tb.data + (size_t)tb.nx * kx * 8);
    const unsigned char *yf = tb.data + ((size_t)tb.nx * kx + (size_t)ny * ky) * 8 + tb.nx;
    auto max_rows = [&](int th) {
        int m = 1;
        for (int y0 = 0; y0 < ny; y0 += th) {
            int lo = 0x7fffffff, hi = -1;
            for (int y = y0; y < std::min(ny, y0 + th); ++y) {
                if (yf[y]) continue;
                for (int k = 0; k < ky; ++k) {
                    lo = std::min(lo, yi[y * ky + k]);
                    hi = std::max(hi, yi[y * ky + k]);
                }
            }
            if (hi >= 0) m = std::max(m, hi - lo + 1);
        }
        return m;
    };
    // tallest band (up to 32 output rows) whose input rows fit two stages:
    // every slice costs the block two barriers, so taller bands amortise them
    int rows = kRsStageRows;
    while (rows > 1 && (size_t)2 * max_rows(rows) * W * sizeof(T) > (size_t)kRsStageRing) rows >>= 1;
    const size_t stage = (size_t)max_rows(rows) * W * sizeof(T);
    if (2 * stage > (size_t)kRsStageRing) return cudaSuccess;
    const int stages = (int)std::min<size_t>(kRsStageMax, kRsStageRing / stage);
    // Slices per block.  The pair kernel: about six blocks per SM slot-wave;
    // fewer, longer blocks keep each block's copies in flight behind its own
    // work (2x bilinear bf16: 4 slices per block 93.9 us, 8: 83.8 us, 16:
    // 93.2 us; one wave of resident blocks, 14: 85.4 us).  resize_stage_kernel:
    // one wave of resident blocks (four per SM), so each block fills and
    // drains its ring once (antialiased 1/2 fp32: 16 slices per block over
    // 1.7 waves 97.6 us, one wave of 27 slices per block 89.5 us).
    const int64_t nbands = (ny + rows - 1) / rows;
    int64_t per = 64;
    if (rs_takes_pair<T>(tb.nx, Y)) {
        while (per > 1 && nbands * ((p.B + per - 1) / per) < 6 * 152) per >>= 1;
    } else {
        int dev = 0, sms = 0;
        cudaError_t ea = cudaGetDevice(&dev);
        if (ea == cudaSuccess) ea = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (ea != cudaSuccess) return ea;
        const int64_t slots = 4 * (int64_t)std::max(sms, 1);
        per = std::max<int64_t>(1, (nbands * p.B + slots - 1) / slots);
        per = std::min<int64_t>(per, std::min<int64_t>(std::max<int64_t>(p.B, 1), (int64_t)1 << 30));
    }
    per = std::max<int64_t>(per, (p.B + 65534) / 65535);
    const dim3 grid((unsigned)((ny + rows - 1) / rows), (unsigned)((p.B + per - 1) / per));
    const T *x = (const T *)X;
    T *y = (T *)Y;
    cudaError_t e;
    const int pb = (int)per;
    if (kx == 1 && ky == 1) e = launch_stage_kernel<T, 1, 1>(x, y, tb, p, grid, rows, pb, stages, err, s);
    else if (ky == 1 && kx == 2) e = launch_stage_kernel<T, 1, 2>(x, y, tb, p, grid, rows, pb, stages, err, s);
    else if (ky == 1 && kx == 4) e = launch_stage_kernel<T, 1, 4>(x, y, tb, p, grid, rows, pb, stages, err, s);
    else if (kx == 2) e = launch_stage_kernel<T, 2, 2>(x, y, tb, p, grid, rows, pb, stages, err, s);
    else e = launch_stage_kernel<T, 4, 4>(x, y, tb, p, grid, rows, pb, stages, err, s);
    *used = true;
    return e;
}

template <typename T, int R>
static cudaError_t launch_resize_r(const void *X, void *Y, const ResizeArgs &p, cudaStream_t s) {
    // tile: up to 256 positions, innermost axis widest
    ResizeTile tl;
    const int n2 = p.ax[2].n_out, n1 = p.ax[1].n_out, n0 = p.ax[0].n_out;
    tl.t[2] = min(n2, 32);
    tl.t[1] = min(n1, kRsThreads / tl.t[2]);
    tl.t[0] = min(n0, kRsThreads / (tl.t[2] * tl.t[1]));
    for (int d = 0; d < 3; ++d) {
        const int n = p.ax[d].n_out;
        tl.tiles[d] = (n + tl.t[d] - 1) / tl.t[d];
    }
    const int64_t tiles = (int64_t)tl.tiles[0] * tl.tiles[1] * tl.tiles[2];
    // slices per block: enough blocks for several waves, at most 64 slices each
    int64_t per = 64;
    while (per > 1 && tiles * ((p.B + per - 1) / per) < 8 * 152) per >>= 1;
    per = std::max<int64_t>(per, (p.B + 65534) / 65535);   // gridDim.y limit
    const int64_t chunks = (p.B + per - 1) / per;
    if (tiles > 0x7fffffffLL || chunks > 65535) return cudaErrorInvalidConfiguration;
    size_t smem = 0;
    for (int d = 0; d < 3; ++d) smem += (size_t)tl.t[d] * (p.ax[d].taps * 8 + 4);
    const dim3 grid((unsigned)tiles, (unsigned)chunks);
    // one fixed tap count on every resized axis: taps in registers
    const int taps = p.ax[2].taps;
    bool fixed = taps == 1 || taps == 2 || taps == 4;
    for (int d = 3 - R; d < 3; ++d) fixed = fixed && p.ax[d].taps == taps;
    if (fixed && taps == 1) {
        resize_kernel<T, R, 1><<<grid, kRsThreads, smem, s>>>((const T *)X, (T *)Y, p, tl, (int)per);
    } else if (fixed && taps == 2) {
        resize_kernel<T, R, 2><<<grid, kRsThreads, smem, s>>>((const T *)X, (T *)Y, p, tl, (int)per);
    } else if (fixed && taps == 4) {
        resize_kernel<T, R, 4><<<grid, kRsThreads, smem, s>>>((const T *)X, (T *)Y, p, tl, (int)per);
    } else {
        resize_kernel<T, R, 0><<<grid, kRsThreads, smem, s>>>((const T *)X, (T *)Y, p, tl, (int)per);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_resize(const void *X, void *Y, const ResizeArgs &p, cudaStream_t s) {
    bool used = false;
    cudaError_t e = launch_resize_stage<T>(X, Y, p, p.err, s, &used);
    if (used || e != cudaSuccess) return e;
    e = launch_resize_rows<T>(X, Y, p, s, &used);
    if (used || e != cudaSuccess) return e;
    if (p.r == 1) return launch_resize_r<T, 1>(X, Y, p, s);
    if (p.r == 2) return launch_resize_r<T, 2>(X, Y, p, s);
    return launch_resize_r<T, 3>(X, Y, p, s);
}

}  // namespace gs
