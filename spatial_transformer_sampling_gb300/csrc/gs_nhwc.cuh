// gs_nhwc.cuh -- GridSample 2-D (tensor grid) from a channel-last copy of X.
//
// GridSample - version 20 (description): every channel of Y[n, :, h, w] is
// sampled at the same grid location.  With an arbitrary grid, neighbouring
// outputs read unrelated pixels, and in the operator's NCHW layout each tap of
// each channel is a separate 32-byte sector for 4 (or 2) useful bytes.  This
// path copies X to NHWC in a caller-provided workspace, a chunk of images at
// a time, and reads every tap as 16-byte vectors of consecutive channels,
// eight lanes per position: one warp load moves four pixels' 128-byte channel
// runs instead of 32 scattered sectors.
//
// Taps are computed once per position and flattened into shared memory as
// (element offset, weight) pairs; the weights and the order of accumulation
// are those of the NCHW gather (flattened taps, row-major, one fmaf per tap),
// so both paths give identical results.  A tap that reads 0 points at an
// all-zero pixel stored just before each image, so the loads of a row of taps
// carry no branch and are all in flight together.  Y is staged through shared
// memory and written in the operator's NCHW layout with whole-line stores.
//
// Workspace: image slots of one zero pixel (C elements) followed by the H*W
// pixels, C elements each.  Each chunk of as many images as the workspace
// holds is copied, then sampled; every copy rewrites the zero pixels of its
// slots.  (Overlapping the copy of the next chunk with the sampling of the
// current one, in one launch and a second buffer, measured slower here: the
// copy evicts the chunk being sampled from L2, and smaller chunks leave the
// launches short of a full wave.)
#pragma once

#include <algorithm>
#include <cstring>
#include <type_traits>

#include "gs_copy.cuh"

namespace gs {

constexpr int kNhPos = 128;      // output positions per block
constexpr int kNhThreads = 256;
constexpr int kNhChan = 64;      // channels per pass (8 lanes x 8 channels)
constexpr int kNhLanes = 8;      // lanes per position
constexpr size_t kNhChunkTarget = (size_t)512 << 20;   // workspace bytes asked for, at most

// One 16-byte vector of channels.
template <typename T> struct Vec16 { static constexpr int E = 16 / (int)sizeof(T); };

template <typename T>
__device__ __forceinline__ void unpack_vec16(const uint4 u, float (&v)[Vec16<T>::E]) {
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

// Per-axis taps of the block's positions (scratch of the tap phase).
template <int MODE> struct NhAxisTaps {
    static constexpr int K = TapCount<MODE>::K;
    int idx[2][K][kNhPos];
    float w[2][K][kNhPos];
    unsigned ok[2][kNhPos];
};

// Shared memory reused by the phases of a block: the tap phase's per-axis
// taps, then the output staging [channel][position], whose position is
// XOR-swizzled by the channel's vector index so that the eight lanes of a
// position write eight different banks.
template <int MODE> union NhStage {
    float y[kNhChan][kNhPos];
    NhAxisTaps<MODE> ax;
};

template <typename T>
__device__ __forceinline__ int nh_swz(int c) {
    return ((c / Vec16<T>::E) & 7) << 2;
}

// One pass of kNhChan channels (from c0) for the block's positions.
// FULL: every vector of the pass lies inside C.
template <typename T, int MODE, bool FULL>
__device__ __forceinline__ void nhwc_pass(const T *__restrict__ Xn, const int2 (*s_tap)[kNhPos],
                                          float (*s_y)[kNhPos], int C, int c0, int warp, int q,
                                          int j) {
    constexpr int K = TapCount<MODE>::K;
    constexpr int E = Vec16<T>::E;                 // channels per vector
    constexpr int NV = kNhChan / (E * kNhLanes);   // vectors per lane per pass: 2 or 1
    bool vin[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) vin[v] = FULL || c0 + (j + v * kNhLanes) * E < C;
    const T *Xc = Xn + c0 + j * E;
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
        const int p = warp * 16 + g * 4 + q;
        float acc[NV][E];
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[v][e] = 0.0f;
        // rows in flight: two for fp32 (more spill registers than they hide
        // latency), all for the half types
        constexpr int RU = NV == 2 ? 2 : K;
#pragma unroll RU
        for (int ky = 0; ky < K; ++ky) {
            int2 tw[K];
            uint4 raw[K][NV];
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                tw[kx] = s_tap[ky * K + kx][p];
                const T *src = Xc + tw[kx].x;
#pragma unroll
                for (int v = 0; v < NV; ++v)
                    raw[kx][v] = vin[v] ? __ldg(reinterpret_cast<const uint4 *>(
                                              src + v * kNhLanes * E))
                                        : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const float w = __int_as_float(tw[kx].y);
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    float x[E];
                    unpack_vec16<T>(raw[kx][v], x);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[v][e] = fmaf(w, x[e], acc[v][e]);
                }
            }
        }
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const int c = (j + v * kNhLanes) * E + e;
                s_y[c][p ^ nh_swz<T>(c)] = acc[v][e];
            }
    }
}

// Sampling: block b takes kNhPos consecutive output positions of image
// n_begin + b / tiles of the chunk in `ws`.  Taps: thread t computes axis
// t % 2 (0: height, 1: width) of position t / 2, then taps t % 2, t % 2 + 2,
// ... of the flattened K x K taps of position t / 2.  Passes: warp w, lane
// (q = lane / 8, j = lane % 8) handles positions w*16 + 4g + q (g = 0..3)
// and, in each pass of kNhChan channels, the 16-byte vectors j and j + 8
// (fp32) or j (half types) of the pass.
template <typename T, int MODE>
__global__ void __launch_bounds__(kNhThreads, 4)
nhwc_sample_kernel(const T *__restrict__ ws, const T *__restrict__ grid, T *__restrict__ Y,
                   const SampleParams P, int n_begin) {
    constexpr int K = TapCount<MODE>::K;
    __shared__ int2 s_tap[K * K][kNhPos];   // (element offset from pixel 0, weight bits)
    __shared__ NhStage<MODE> s_u;
    const SampleArgs &a = P.a;
    const int C = a.C;
    const int sb = blockIdx.x;

    const int ni = sb / a.tiles;   // image within the chunk
    const int tile = sb - ni * a.tiles;
    const int n = n_begin + ni;
    const int64_t o0 = (int64_t)tile * kNhPos;
    {
        const int p = threadIdx.x >> 1, axis = threadIdx.x & 1;
        const int64_t o = o0 + p;
        AxisTaps<MODE> tp;
        if (o < a.out_plane) {
            // the grid vector lists width first: axis 0 (height) reads component 1
            const T *g = grid + ((int64_t)n * a.out_plane + o) * 2 + (1 - axis);
            make_taps<MODE>(grid_to_q(IO<T>::ld(g), P.ax[axis], a.pad), P.ax[axis], a.pad, a.ac,
                            a.a, tp);
        } else {
#pragma unroll
            for (int k = 0; k < K; ++k) {
                tp.idx[k] = 0;
                tp.w[k] = 0.0f;
            }
            tp.ok = 0;
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            s_u.ax.idx[axis][k][p] = tp.idx[k];
            s_u.ax.w[axis][k][p] = tp.w[k];
        }
        s_u.ax.ok[axis][p] = tp.ok;
    }
    __syncthreads();
    {
        const int p = threadIdx.x >> 1;
        const unsigned oky = s_u.ax.ok[0][p], okx = s_u.ax.ok[1][p];
#pragma unroll
        for (int t = threadIdx.x & 1; t < K * K; t += 2) {
            const int ky = t / K, kx = t - (t / K) * K;
            const bool ok = ((oky >> ky) & (okx >> kx) & 1u) != 0;
            const int off = ok ? (s_u.ax.idx[0][ky][p] * a.in[1] + s_u.ax.idx[1][kx][p]) * C
                               : -C;   // the zero pixel
            const float w = s_u.ax.w[0][ky][p] * s_u.ax.w[1][kx][p];
            s_tap[t][p] = make_int2(off, __float_as_int(w));
        }
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = lane >> 3, j = lane & 7;
    const T *Xn = ws + (int64_t)ni * C * (a.in_plane + 1) + C;   // pixel 0 of the slot
    T *Yn = Y + (int64_t)n * C * a.out_plane;

    for (int c0 = 0; c0 < C; c0 += kNhChan) {
        if (c0 + kNhChan <= C)
            nhwc_pass<T, MODE, true>(Xn, s_tap, s_u.y, C, c0, warp, q, j);
        else
            nhwc_pass<T, MODE, false>(Xn, s_tap, s_u.y, C, c0, warp, q, j);
        __syncthreads();
        const int cn = min(kNhChan, C - c0);
        for (int i = threadIdx.x; i < cn * kNhPos; i += kNhThreads) {
            const int c = i / kNhPos, p = i - c * kNhPos;
            if (o0 + p < a.out_plane)
                Yn[(int64_t)(c0 + c) * a.out_plane + o0 + p] =
                    IO<T>::st(s_u.y[c][p ^ nh_swz<T>(c)]);
        }
        __syncthreads();
    }
}

// Bytes of one image slot: the zero pixel and H*W pixels, C elements each.
inline size_t nhwc_slot_bytes(const SampleArgs &a, size_t elem) {
    return (size_t)a.C * (size_t)(a.in_plane + 1) * elem;
}

// Whether the channel-last path takes this call (0: never), else the
// workspace bytes it asks for: whole slots for the batch in chunks of at most
// about kNhChunkTarget, balanced (at least one slot).
template <typename T>
size_t nhwc_workspace_bytes(const SampleArgs &a, int r, bool affine) {
    if (affine || r != 2 || a.N == 0 || a.C == 0 || a.out_plane == 0) return 0;
    if (((int64_t)a.C * sizeof(T)) % 16 != 0) return 0;   // 16-byte vectors per pixel
    // 32-bit element offsets within a slot
    if ((int64_t)a.C * (a.in_plane + 1) >= ((int64_t)1 << 31)) return 0;
    const size_t slot = nhwc_slot_bytes(a, sizeof(T));
    const size_t cap = std::max<size_t>(1, kNhChunkTarget / slot);   // slots per chunk
    const size_t chunks = ((size_t)a.N + cap - 1) / cap;
    return (((size_t)a.N + chunks - 1) / chunks) * slot;
}

// Smallest workspace the channel-last path runs with: one slot.
template <typename T>
size_t nhwc_min_workspace_bytes(const SampleArgs &a) {
    return nhwc_slot_bytes(a, sizeof(T));
}

template <typename T, int MODE>
static cudaError_t launch_nhwc_mode(const void *X, const void *grid, void *Y, const SampleParams &P,
                                    void *ws, size_t ws_bytes, cudaStream_t s) {
    using R = RawOf<T>;
    const SampleArgs &a = P.a;
    const size_t slot = nhwc_slot_bytes(a, sizeof(T));
    const int64_t tiles_img = copy_tiles_per_image(a.C, a.in_plane);   // copy blocks per image
    // as many slots per chunk as the workspace holds (at least one), within
    // the 2^31 - 1 blocks of a launch
    const int64_t max_blocks = ((int64_t)1 << 31) - 1;
    int64_t per = std::min<int64_t>((int64_t)a.N, std::max<int64_t>(1, (int64_t)(ws_bytes / slot)));
    per = std::min<int64_t>(per, std::max<int64_t>(1, max_blocks / tiles_img));
    per = std::min<int64_t>(per, std::max<int64_t>(1, max_blocks / a.tiles));
    for (int64_t n0 = 0; n0 < a.N; n0 += per) {
        const int64_t nc = std::min<int64_t>(per, a.N - n0);
        launch_copy_to_slots<R>((const R *)X + n0 * a.C * a.in_plane, (R *)ws, nc, a.C,
                                a.in_plane, s);
        nhwc_sample_kernel<T, MODE><<<(unsigned)(nc * a.tiles), kNhThreads, 0, s>>>(
            (const T *)ws, (const T *)grid, (T *)Y, P, (int)n0);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t launch_nhwc(const void *X, const void *grid, void *Y, const SampleParams &P0,
                        int mode, void *ws, size_t ws_bytes, cudaStream_t s) {
    SampleParams P = P0;
    P.a.tiles = (int)((P.a.out_plane + kNhPos - 1) / kNhPos);
    switch (mode) {
        case MODE_LINEAR: return launch_nhwc_mode<T, MODE_LINEAR>(X, grid, Y, P, ws, ws_bytes, s);
        case MODE_NEAREST: return launch_nhwc_mode<T, MODE_NEAREST>(X, grid, Y, P, ws, ws_bytes, s);
        default: return launch_nhwc_mode<T, MODE_CUBIC>(X, grid, Y, P, ws, ws_bytes, s);
    }
}

}  // namespace gs
