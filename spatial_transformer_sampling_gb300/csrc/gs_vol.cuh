// gs_vol.cuh -- fused AffineGrid+GridSample, 3-D, trilinear and nearest: the
// staged box kernel.
//
// A block owns one image and a tile of output positions (tz x ty x tx, up to
// 1024 positions, four per thread).  Under an affine map the tile's positions
// fill a parallelepiped whose extremes sit at the tile's corners, so every tap
// the tile reads lies in one axis-aligned input box.  The block streams that
// box, channel by channel, into a ring of shared-memory stages with 16-byte
// asynchronous copies (cp.async) issued by all threads; the parts of the box
// outside X are written as zeros by the copy itself (source size 0).  Rows of
// the box start every 128 bytes, so the eight tap loads of a warp (32
// consecutive output columns, spread over a few input rows and planes) fall
// in distinct banks.  Each position's first tap index is clamped into the
// box: the clamp moves an index only where both of its taps read zero anyway
// (zeros padding: everything past index -1 or n is zero), so every tap is a
// plain shared-memory load at one of eight fixed offsets from the position's
// base, with no mask and no select.
//
// A block whose box does not fit two stages (strong zoom-out, rotation by a
// large angle, reflection of far-out positions), or whose map needs fp64
// positions, gathers from global memory instead with the taps of
// sample_kernel.
#pragma once

#include "gs_ptx.cuh"

namespace gs {

constexpr int kVolThreads = 256;
constexpr int kVolPPT = 4;                         // output positions per thread
constexpr int kVolTile = kVolThreads * kVolPPT;    // output positions per block
constexpr int kVolMaxStages = 4;
constexpr int kVolRingBytes = 96 * 1024;
constexpr int kVolMaxChunks = 2048;                // 16-byte chunks copied per stage
constexpr int kVolSmemBytes = kVolRingBytes + kVolMaxChunks * 8;   // ring + chunk table

struct VolParams {
    int tz, ty, tx;         // tile extents along output depth, rows, columns (tx: 8, 16 or 32)
    int tiles_y, tiles_x;   // tiles along output rows and columns
    int tiles;              // tiles per image
};

// Index of the first tap (linear) or the tap (nearest) on one axis from a
// 32.32 position, after the coordinate padding, clamped to [-2, n] (linear)
// or [-1, n] (nearest).  Monotone in xq for zeros and border padding, and for
// reflection wherever the fold leaves positions in place.
template <int MODE>
__device__ __forceinline__ int vol_index(int64_t xq, int n) {
    int64_t i;
    if (MODE == MODE_NEAREST) {
        i = (xq + kHalfQ) >> 32;                               // floor(x + 1/2)
        if ((uint32_t)xq == 0x80000000u && (i & 1)) i -= 1;   // exact tie: even index
        return (int)(i < -1 ? -1 : (i > n ? n : i));
    }
    i = xq >> 32;
    return (int)(i < -2 ? -2 : (i > n ? n : i));
}

__device__ __forceinline__ int64_t vol_pad(int64_t xq, const Axis &A, int pad) {
    if (pad == PAD_BORDER) return clamp_q(xq, 0, A.hi_q);
    if (pad == PAD_REFLECTION) return clamp_q(reflect_q(xq, A.lo_q, A.span_q), 0, A.hi_q);
    return xq;
}

// Shared-memory load at a 32-bit shared address plus a constant byte offset.
template <typename T, int OFF> __device__ __forceinline__ float lds_off(uint32_t addr);
template <> __device__ __forceinline__ float lds_off<float, 0>(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
template <> __device__ __forceinline__ float lds_off<float, 4>(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1+4];" : "=f"(v) : "r"(addr));
    return v;
}
template <> __device__ __forceinline__ float lds_off<__half, 0>(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return __half2float(__ushort_as_half(v));
}
template <> __device__ __forceinline__ float lds_off<__half, 2>(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1+2];" : "=h"(v) : "r"(addr));
    return __half2float(__ushort_as_half(v));
}
template <> __device__ __forceinline__ float lds_off<__nv_bfloat16, 0>(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return __uint_as_float((uint32_t)v << 16);
}
template <> __device__ __forceinline__ float lds_off<__nv_bfloat16, 2>(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1+2];" : "=h"(v) : "r"(addr));
    return __uint_as_float((uint32_t)v << 16);
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kVolThreads, 2)
vol_kernel(const T *__restrict__ X, const T *__restrict__ theta, T *__restrict__ Y,
           const SampleParams P, const VolParams V) {
    constexpr int K = MODE == MODE_NEAREST ? 1 : 2;
    constexpr int NT = K * K * K;
    constexpr int EPC = 16 / (int)sizeof(T);   // elements per 16-byte chunk
    extern __shared__ __align__(128) unsigned char vol_smem[];
    __shared__ AffineMap s_map;
    __shared__ int s_lo[3], s_ext[3], s_chunks, s_stages;
    __shared__ uint32_t s_pitch;   // bytes between box rows (a multiple of 128)

    const SampleArgs &a = P.a;
    const int n = blockIdx.x / V.tiles;
    const int tile = blockIdx.x - n * V.tiles;
    const int tzi = tile / (V.tiles_y * V.tiles_x);
    const int trem = tile - tzi * (V.tiles_y * V.tiles_x);
    const int tyi = trem / V.tiles_x;
    const int txi = trem - tyi * V.tiles_x;
    const int oz0 = tzi * V.tz, oy0 = tyi * V.ty, ox0 = txi * V.tx;
    const int tid = threadIdx.x;

    if (tid < 32) build_affine_map_warp<T, 3>(theta + (int64_t)n * 12, P, s_map);
    __syncthreads();
    if (tid < 3) {
        // box of input indices along axis d = tid, from the tile's eight corners
        const int d = tid;
        const int o_hi[3] = {min(oz0 + V.tz, a.out[0]) - 1, min(oy0 + V.ty, a.out[1]) - 1,
                             min(ox0 + V.tx, a.out[2]) - 1};
        const int o_lo[3] = {oz0, oy0, ox0};
        int64_t qmin = INT64_MAX, qmax = INT64_MIN;
        for (int ci = 0; ci < 8; ++ci) {
            int64_t q = s_map.cst_q[d];
            for (int j = 0; j < 3; ++j)
                q += s_map.coef_q[d][j] * (int64_t)(((ci >> j) & 1) ? o_hi[j] : o_lo[j]);
            q >>= 8;
            qmin = q < qmin ? q : qmin;
            qmax = q > qmax ? q : qmax;
        }
        const Axis &A = P.ax[d];
        if (a.pad == PAD_REFLECTION && (qmin < A.lo_q || qmax > A.lo_q + A.span_q)) {
            qmin = 0;   // folded positions can land anywhere on the axis
            qmax = A.hi_q;
        } else {
            qmin = vol_pad(qmin, A, a.pad);
            qmax = vol_pad(qmax, A, a.pad);
        }
        int lo = vol_index<MODE>(qmin, A.n);
        const int hi = vol_index<MODE>(qmax, A.n) + (K - 1);
        int ext = hi - lo + 1;
        if (d == 2) {
            lo &= ~(EPC - 1);              // whole 16-byte chunks
            ext = (hi - lo) / EPC + 1;     // in chunks
        }
        s_lo[d] = lo;
        s_ext[d] = ext;
    }
    __syncthreads();
    if (tid == 0) {
        int stages = 0, chunks = 0;
        const uint32_t pitch = ((uint32_t)s_ext[2] * 16u + 127u) & ~127u;
        if (!s_map.wide) {
            const int64_t nch = (int64_t)s_ext[0] * s_ext[1] * s_ext[2];
            const int64_t bytes = (int64_t)s_ext[0] * s_ext[1] * pitch;
            if (nch <= kVolMaxChunks && bytes * 2 <= kVolRingBytes) {
                chunks = (int)nch;
                stages = min(kVolMaxStages, (int)(kVolRingBytes / bytes));
            }
        }
        s_chunks = chunks;
        s_stages = stages;
        s_pitch = pitch;
    }
    __syncthreads();
    const int S = s_stages;   // 0: gather from global

    const int64_t in_plane = a.in_plane;
    const T *__restrict__ Xn = X + (int64_t)n * a.C * in_plane;
    T *__restrict__ Yc = Y + (int64_t)n * a.C * a.out_plane;
    const int Ho = a.out[1], Wo = a.out[2];
    const int tx_shift = V.tx == 32 ? 5 : (V.tx == 16 ? 4 : 3);

    if (S == 0) {
        // gather from global memory, one position at a time
        for (int j = 0; j < kVolPPT; ++j) {
            const int p = tid + j * kVolThreads;
            const int row = p >> tx_shift;
            const int oz = oz0 + row / V.ty, oy = oy0 + row % V.ty, ox = ox0 + (p & (V.tx - 1));
            if (row >= V.tz * V.ty || oz >= a.out[0] || oy >= Ho || ox >= Wo) continue;
            AxisTaps<MODE> tp[3];
            const int opos[3] = {oz, oy, ox};
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                int64_t xq;
                if (!s_map.wide) {
                    int64_t acc = s_map.cst_q[d];
#pragma unroll
                    for (int jj = 0; jj < 3; ++jj) acc += s_map.coef_q[d][jj] * (int64_t)opos[jj];
                    xq = acc >> 8;
                } else {
                    double x = s_map.cst[d];
#pragma unroll
                    for (int jj = 0; jj < 3; ++jj) x += s_map.coef[d][jj] * (double)opos[jj];
                    xq = pos_to_q(x, P.ax[d], a.pad);
                }
                make_taps<MODE>(xq, P.ax[d], a.pad, a.ac, a.a, tp[d]);
            }
            int off_hi[16];
            outer_offsets<3, MODE>(tp, a, off_hi);
            const int64_t yo = ((int64_t)oz * Ho + oy) * Wo + ox;
            const T *Xc = Xn;
            T *Yp = Yc + yo;
            for (int c = 0; c < a.C; ++c) {
                *Yp = IO<T>::st(interp<T, 3, MODE>(Xc, tp, off_hi));
                Xc += in_plane;
                Yp += a.out_plane;
            }
        }
        return;
    }

    // chunk table: (element offset of the chunk inside a channel volume, or -1
    // where it lies outside X and is zero-filled; byte offset inside a stage)
    int2 *s_tab = reinterpret_cast<int2 *>(vol_smem + kVolRingBytes);
    const int chunks = s_chunks;
    const uint32_t dy_b = s_pitch;
    const uint32_t dz_b = (uint32_t)s_ext[1] * dy_b;
    const uint32_t stage_bytes = (uint32_t)s_ext[0] * dz_b;
    {
        const int ey = s_ext[1], exc = s_ext[2];
        const int bz = s_lo[0], by = s_lo[1], bx = s_lo[2];
        const int Di = a.in[0], Hi = a.in[1], Wi = a.in[2];
        for (int i = tid; i < chunks; i += kVolThreads) {
            const int row = i / exc;
            const int xc = i - row * exc;
            const int z = row / ey;
            const int y = row - z * ey;
            const int gz = bz + z, gy = by + y, gx = bx + xc * EPC;
            const bool in = gz >= 0 && gz < Di && gy >= 0 && gy < Hi && gx >= 0 && gx < Wi;
            s_tab[i] = make_int2(in ? (gz * Hi + gy) * Wi + gx : -1,
                                 (int)((uint32_t)row * dy_b + (uint32_t)xc * 16u));
        }
    }

    // this thread's positions: base byte offset in a stage, weights, Y offset
    uint32_t base[kVolPPT];
    float2 w2[kVolPPT / 2][NT];   // weights of positions (2i, 2i+1), tap by tap
    int yoff[kVolPPT];
    unsigned live = 0;
#pragma unroll
    for (int j = 0; j < kVolPPT; ++j) {
        const int p = tid + j * kVolThreads;
        const int row = p >> tx_shift;
        const int oz = oz0 + row / V.ty, oy = oy0 + row % V.ty, ox = ox0 + (p & (V.tx - 1));
        const bool ok = row < V.tz * V.ty && oz < a.out[0] && oy < Ho && ox < Wo;
        live |= (ok ? 1u : 0u) << j;
        const int opos[3] = {ok ? oz : oz0, ok ? oy : oy0, ok ? ox : ox0};
        int li[3];
        float t[3];
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            int64_t acc = s_map.cst_q[d];
#pragma unroll
            for (int jj = 0; jj < 3; ++jj) acc += s_map.coef_q[d][jj] * (int64_t)opos[jj];
            const int64_t xq = vol_pad(acc >> 8, P.ax[d], a.pad);
            li[d] = vol_index<MODE>(xq, P.ax[d].n) - s_lo[d];
            t[d] = __uint2float_rn((uint32_t)xq) * 2.3283064365386963e-10f;   // * 2^-32
        }
        base[j] = (uint32_t)li[0] * dz_b + (uint32_t)li[1] * dy_b + (uint32_t)li[2] * (uint32_t)sizeof(T);
        if (MODE != MODE_NEAREST) {
#pragma unroll
            for (int kz = 0; kz < 2; ++kz)
#pragma unroll
                for (int ky = 0; ky < 2; ++ky) {
                    const float wzy = (kz ? t[0] : 1.0f - t[0]) * (ky ? t[1] : 1.0f - t[1]);
                    const float w0 = wzy * (1.0f - t[2]), w1 = wzy * t[2];
                    float2 &a0 = w2[j >> 1][kz * 4 + ky * 2 + 0];
                    float2 &a1 = w2[j >> 1][kz * 4 + ky * 2 + 1];
                    if (j & 1) {
                        a0.y = w0;
                        a1.y = w1;
                    } else {
                        a0.x = w0;
                        a1.x = w1;
                    }
                }
        }
        yoff[j] = (opos[0] * Ho + opos[1]) * Wo + opos[2];
    }
    __syncthreads();   // chunk table complete

    const uint32_t ring = smem_u32(vol_smem);
    const int C = a.C;
    const int64_t out_plane = a.out_plane;
    auto issue = [&](int cc, int stg) {
        const T *Xc = Xn + (int64_t)cc * in_plane;
        const uint32_t dst = ring + (uint32_t)stg * stage_bytes;
        for (int i = tid; i < chunks; i += kVolThreads) {
            const int2 e = s_tab[i];
            cp_async16(dst + (uint32_t)e.y, e.x >= 0 ? (const void *)(Xc + e.x) : (const void *)Xc,
                       e.x >= 0 ? 16u : 0u);
        }
    };
    for (int s = 0; s < S - 1; ++s) {
        if (s < C) issue(s, s);
        cp_async_commit();
    }
    // a tile inside the output stores every position: no per-position predicate
    const bool full_tile = oz0 + V.tz <= a.out[0] && oy0 + V.ty <= Ho && ox0 + V.tx <= Wo &&
                           V.tz * V.ty * V.tx == kVolTile;
    int st = 0;
    for (int c = 0; c < C; ++c) {
        cp_async_wait_pending(S - 2);   // this thread's copies of channel c have landed
        __syncthreads();                // everyone's have; stage (c-1) % S is free again
        if (c + S - 1 < C) issue(c + S - 1, st == 0 ? S - 1 : st - 1);
        cp_async_commit();
        const uint32_t sb = ring + (uint32_t)st * stage_bytes;
#pragma unroll
        for (int h = 0; h < kVolPPT / 2; ++h) {
            constexpr int E = (int)sizeof(T);
            const uint32_t qa = sb + base[2 * h], qb = sb + base[2 * h + 1];
            float2 acc;
            if (MODE == MODE_NEAREST) {
                acc = make_float2(lds_off<T, 0>(qa), lds_off<T, 0>(qb));
            } else {
                const uint32_t qa1 = qa + dy_b, qa2 = qa + dz_b, qa3 = qa2 + dy_b;
                const uint32_t qb1 = qb + dy_b, qb2 = qb + dz_b, qb3 = qb2 + dy_b;
                float2 v[NT];
                v[0] = make_float2(lds_off<T, 0>(qa), lds_off<T, 0>(qb));
                v[1] = make_float2(lds_off<T, E>(qa), lds_off<T, E>(qb));
                v[2] = make_float2(lds_off<T, 0>(qa1), lds_off<T, 0>(qb1));
                v[3] = make_float2(lds_off<T, E>(qa1), lds_off<T, E>(qb1));
                v[4] = make_float2(lds_off<T, 0>(qa2), lds_off<T, 0>(qb2));
                v[5] = make_float2(lds_off<T, E>(qa2), lds_off<T, E>(qb2));
                v[6] = make_float2(lds_off<T, 0>(qa3), lds_off<T, 0>(qb3));
                v[7] = make_float2(lds_off<T, E>(qa3), lds_off<T, E>(qb3));
                acc = mul_f32x2(w2[h][0], v[0]);
#pragma unroll
                for (int t = 1; t < NT; ++t) acc = fma_f32x2(w2[h][t], v[t], acc);
            }
            if (full_tile) {
                Yc[yoff[2 * h]] = IO<T>::st(acc.x);
                Yc[yoff[2 * h + 1]] = IO<T>::st(acc.y);
            } else {
                if ((live >> (2 * h)) & 1u) Yc[yoff[2 * h]] = IO<T>::st(acc.x);
                if ((live >> (2 * h + 1)) & 1u) Yc[yoff[2 * h + 1]] = IO<T>::st(acc.y);
            }
        }
        Yc += out_plane;
        if (++st == S) st = 0;
    }
    cp_async_wait_pending(0);   // nothing may be in flight when the block exits
}

// Host side: the staged kernel for trilinear / nearest when rows can be
// copied in 16-byte chunks; *used tells the caller whether it ran.
template <typename T, int MODE>
cudaError_t launch_vol(const void *X, const void *theta, void *Y, const SampleParams &P,
                       cudaStream_t s, bool *used) {
    *used = false;
    if (MODE == MODE_CUBIC) return cudaSuccess;
    const SampleArgs &a = P.a;
    if (((size_t)a.in[2] * sizeof(T)) % 16 != 0 || (uintptr_t)X % 16 != 0) return cudaSuccess;
    const int Do = a.out[0], Ho = a.out[1], Wo = a.out[2];
    VolParams V;
    V.tx = Wo > 16 ? 32 : (Wo > 8 ? 16 : 8);
    const int rows = kVolTile / V.tx;   // (depth, row) pairs per tile
    V.tz = min(Do, V.tx == 32 ? 4 : 8);
    V.ty = min(Ho, rows / V.tz);
    V.tz = min(Do, rows / V.ty);
    V.tiles_y = (Ho + V.ty - 1) / V.ty;
    V.tiles_x = (Wo + V.tx - 1) / V.tx;
    const int64_t tiles = (int64_t)((Do + V.tz - 1) / V.tz) * V.tiles_y * V.tiles_x;
    if (tiles * a.N > 0x7fffffffLL) return cudaSuccess;
    V.tiles = (int)tiles;
    static DeviceFlags attr_set;
    const cudaError_t e = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(vol_kernel<T, MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kVolSmemBytes);
    });
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)(tiles * a.N);
    vol_kernel<T, MODE><<<blocks, kVolThreads, kVolSmemBytes, s>>>(
        (const T *)X, (const T *)theta, (T *)Y, P, V);
    *used = true;
    return cudaGetLastError();
}

}  // namespace gs
