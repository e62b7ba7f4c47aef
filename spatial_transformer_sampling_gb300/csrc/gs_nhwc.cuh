// gs_nhwc.cuh -- GridSample 2-D (tensor grid) from a channel-last copy of X.
//
// GridSample - version 20 (description): every channel of Y[n, :, h, w] is
// sampled at the same grid location.  With an arbitrary grid, neighbouring
// outputs read unrelated pixels, and in the operator's NCHW layout each tap of
// each channel is a separate 32-byte sector for 4 (or 2) useful bytes.  This
// path first copies a chunk of images to NHWC in a caller-provided workspace
// (sized to stay resident in L2), then reads every tap as 16-byte vectors of
// consecutive channels, eight lanes per position: one warp load touches four
// pixels' 128-byte channel runs instead of 32 scattered sectors.
//
// Taps (indices, weights, validity) are computed once per position by one
// thread, kept in shared memory and reused for every channel pass; the weights
// and the order of accumulation are those of the NCHW gather (flattened taps,
// row-major, one fmaf per tap), so both paths give identical results.  Y is
// staged through shared memory and written in the operator's NCHW layout with
// whole-line stores.
#pragma once

#include <algorithm>
#include <cstring>
#include <type_traits>

namespace gs {

constexpr int kTrTile = 32;        // transpose tile (channels x pixels)
constexpr int kNhPos = 128;        // output positions per block
constexpr int kNhThreads = 256;
constexpr int kNhChan = 64;        // channels per pass (8 lanes x 8 channels)
constexpr int kNhLanes = 8;        // lanes per position
constexpr size_t kNhChunkTarget = (size_t)32 << 20;   // channel-last bytes per chunk

// X[n, c, p] -> Xt[n, p, c] for the images of one chunk; 32 x 32 tiles through
// shared memory, coalesced on both sides.  Block (ct, pt, n) = blockIdx.x.
template <typename T>
__global__ void __launch_bounds__(256)
nchw_to_nhwc_kernel(const T *__restrict__ X, T *__restrict__ Xt, int C, int64_t P, int ctiles,
                    int64_t ptiles) {
    __shared__ T tile[kTrTile][kTrTile + 1];
    int64_t b = blockIdx.x;
    const int ct = (int)(b % ctiles);
    b /= ctiles;
    const int64_t pt = b % ptiles;
    const int64_t n = b / ptiles;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
    const int c0 = ct * kTrTile;
    const int64_t p0 = pt * kTrTile;
    const T *src = X + n * C * P;
    T *dst = Xt + n * C * P;
#pragma unroll
    for (int i = 0; i < kTrTile; i += 8) {
        const int c = c0 + ty + i;
        const int64_t p = p0 + tx;
        if (c < C && p < P) tile[ty + i][tx] = src[(int64_t)c * P + p];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTrTile; i += 8) {
        const int64_t p = p0 + ty + i;
        const int c = c0 + tx;
        if (c < C && p < P) dst[p * C + c] = tile[tx][ty + i];
    }
}

// One 16-byte vector of channels, widened to fp32.
template <typename T> struct Vec16 { static constexpr int E = 16 / (int)sizeof(T); };

template <typename T>
__device__ __forceinline__ void load_vec16(const T *p, float (&v)[Vec16<T>::E]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    if constexpr (sizeof(T) == 4) {
        v[0] = __uint_as_float(u.x);
        v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z);
        v[3] = __uint_as_float(u.w);
    } else {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float2 f;
            if constexpr (std::is_same<T, __half>::value) {
                __half2 h;
                memcpy(&h, &w[i], 4);
                f = __half22float2(h);
            } else {
                __nv_bfloat162 h;
                memcpy(&h, &w[i], 4);
                f = __bfloat1622float2(h);
            }
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
    }
}

// Per-position taps in shared memory, [field][position]: row offsets (pixels),
// column indices, the two axes' weights, and the validity bits (y | x << K).
template <int MODE> struct NhTaps {
    static constexpr int K = TapCount<MODE>::K;
    int row[K][kNhPos];
    int col[K][kNhPos];
    float wy[K][kNhPos];
    float wx[K][kNhPos];
    unsigned ok[kNhPos];
};

// Block = kNhPos consecutive output positions of one image of the chunk.
// Warp w, lane (q = lane / 8, j = lane % 8) handles positions w*16 + 4g + q
// (g = 0..3) and, in each pass of kNhChan channels, the 16-byte vectors j and
// j + 8 (fp32) or j (half types) of the pass.
template <typename T, int MODE>
__global__ void __launch_bounds__(kNhThreads, 4)
nhwc_sample_kernel(const T *__restrict__ Xt, const T *__restrict__ grid, T *__restrict__ Y,
                   const SampleParams P, int n_begin) {
    constexpr int K = TapCount<MODE>::K;
    constexpr int E = Vec16<T>::E;            // channels per vector
    constexpr int NV = kNhChan / (E * kNhLanes);   // vectors per lane per pass: 2 or 1
    __shared__ NhTaps<MODE> s_t;
    __shared__ float s_y[kNhChan][kNhPos + 1];

    const SampleArgs &a = P.a;
    const int ni = blockIdx.x / a.tiles;       // image within the chunk
    const int tile = blockIdx.x - ni * a.tiles;
    const int n = n_begin + ni;
    const int64_t o0 = (int64_t)tile * kNhPos;
    const int C = a.C;

    if (threadIdx.x < kNhPos) {
        const int p = threadIdx.x;
        const int64_t o = o0 + p;
        AxisTaps<MODE> ty, tx;
        if (o < a.out_plane) {
            const T *g = grid + ((int64_t)n * a.out_plane + o) * 2;
            make_taps<MODE>(grid_to_q(IO<T>::ld(g + 1), P.ax[0], a.pad), P.ax[0], a.pad, a.ac,
                            a.a, ty);
            make_taps<MODE>(grid_to_q(IO<T>::ld(g + 0), P.ax[1], a.pad), P.ax[1], a.pad, a.ac,
                            a.a, tx);
        } else {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                ty.idx[k] = tx.idx[k] = 0;
                ty.w[k] = tx.w[k] = 0.0f;
            }
            ty.ok = tx.ok = 0;
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            s_t.row[k][p] = ty.idx[k] * a.in[1];
            s_t.col[k][p] = tx.idx[k];
            s_t.wy[k][p] = ty.w[k];
            s_t.wx[k][p] = tx.w[k];
        }
        s_t.ok[p] = ty.ok | (tx.ok << K);
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = lane >> 3, j = lane & 7;
    const T *Xn = Xt + (int64_t)ni * C * a.in_plane;
    T *Yn = Y + (int64_t)n * C * a.out_plane;

    for (int c0 = 0; c0 < C; c0 += kNhChan) {
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            const int p = warp * 16 + g * 4 + q;
            const unsigned okb = s_t.ok[p];
            float acc[NV][E];
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[v][e] = 0.0f;
#pragma unroll
            for (int ky = 0; ky < K; ++ky) {
                const int row = s_t.row[ky][p];
                const float wy = s_t.wy[ky][p];
#pragma unroll
                for (int kx = 0; kx < K; ++kx) {
                    const bool ok = ((okb >> ky) & (okb >> (K + kx)) & 1u) != 0;
                    if (!ok) continue;   // the tap reads 0: fmaf(w, 0, acc) == acc
                    const float w = wy * s_t.wx[kx][p];
                    const T *px = Xn + (int64_t)(row + s_t.col[kx][p]) * C + c0;
#pragma unroll
                    for (int v = 0; v < NV; ++v) {
                        const int cv = (j + v * kNhLanes) * E;
                        if (c0 + cv < C) {
                            float x[E];
                            load_vec16<T>(px + cv, x);
#pragma unroll
                            for (int e = 0; e < E; ++e) acc[v][e] = fmaf(w, x[e], acc[v][e]);
                        }
                    }
                }
            }
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int e = 0; e < E; ++e) s_y[(j + v * kNhLanes) * E + e][p] = acc[v][e];
        }
        __syncthreads();
        const int cn = min(kNhChan, C - c0);
        for (int i = threadIdx.x; i < cn * kNhPos; i += kNhThreads) {
            const int c = i / kNhPos, p = i - c * kNhPos;
            if (o0 + p < a.out_plane)
                Yn[(int64_t)(c0 + c) * a.out_plane + o0 + p] = IO<T>::st(s_y[c][p]);
        }
        __syncthreads();
    }
}

// Whether the channel-last path takes this call, and the workspace bytes it
// asks for: a chunk of whole images (at least one) of about kNhChunkTarget.
template <typename T>
size_t nhwc_workspace_bytes(const SampleArgs &a, int r, bool affine) {
    if (affine || r != 2 || a.N == 0 || a.C == 0 || a.out_plane == 0) return 0;
    if (((int64_t)a.C * sizeof(T)) % 16 != 0) return 0;          // 16-byte vectors per pixel
    if ((int64_t)a.C * a.in_plane >= ((int64_t)1 << 31)) return 0;   // 32-bit pixel offsets
    const size_t img = (size_t)a.C * a.in_plane * sizeof(T);
    const size_t per = std::max<size_t>(1, std::min<size_t>((size_t)a.N, kNhChunkTarget / img));
    return per * img;
}

template <typename T>
cudaError_t launch_nhwc(const void *X, const void *grid, void *Y, const SampleParams &P0,
                        int mode, void *ws, size_t ws_bytes, cudaStream_t s) {
    SampleParams P = P0;
    const SampleArgs &a = P.a;
    const size_t img = (size_t)a.C * a.in_plane * sizeof(T);
    P.a.tiles = (int)((a.out_plane + kNhPos - 1) / kNhPos);
    const int ctiles = (a.C + kTrTile - 1) / kTrTile;
    const int64_t ptiles = (a.in_plane + kTrTile - 1) / kTrTile;
    // as many whole images per chunk as the workspace holds (at least one),
    // within the 2^31 - 1 blocks of a launch
    const int64_t max_blocks = ((int64_t)1 << 31) - 1;
    int64_t per = std::min<int64_t>((int64_t)a.N, std::max<int64_t>(1, (int64_t)(ws_bytes / img)));
    per = std::min<int64_t>(per, std::max<int64_t>(1, max_blocks / (ptiles * ctiles)));
    per = std::min<int64_t>(per, std::max<int64_t>(1, max_blocks / P.a.tiles));
    const int per_chunk = (int)per;
    for (int n0 = 0; n0 < a.N; n0 += per_chunk) {
        const int nc = std::min(per_chunk, a.N - n0);
        const T *Xc = (const T *)X + (int64_t)n0 * a.C * a.in_plane;
        nchw_to_nhwc_kernel<T><<<(unsigned)((int64_t)nc * ptiles * ctiles), 256, 0, s>>>(
            Xc, (T *)ws, a.C, a.in_plane, ctiles, ptiles);
        const unsigned blocks = (unsigned)((int64_t)nc * P.a.tiles);
        switch (mode) {
            case MODE_LINEAR:
                nhwc_sample_kernel<T, MODE_LINEAR><<<blocks, kNhThreads, 0, s>>>(
                    (const T *)ws, (const T *)grid, (T *)Y, P, n0);
                break;
            case MODE_NEAREST:
                nhwc_sample_kernel<T, MODE_NEAREST><<<blocks, kNhThreads, 0, s>>>(
                    (const T *)ws, (const T *)grid, (T *)Y, P, n0);
                break;
            default:
                nhwc_sample_kernel<T, MODE_CUBIC><<<blocks, kNhThreads, 0, s>>>(
                    (const T *)ws, (const T *)grid, (T *)Y, P, n0);
                break;
        }
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gs
