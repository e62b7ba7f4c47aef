// gs_copy.cuh -- copy of X from the operators' channel-first layout
// (N, C, spatial...) to channel-last image slots in a caller-provided
// workspace, shared by the channel-last GridSample and DeformConv paths.
//
// Slot layout: one zero pixel (C elements of 0), then the P spatial
// positions, C elements each; slot n starts at element n * C * (P + 1).  A tap
// that reads 0 points at the zero pixel, so gathers from a slot need no
// branch for out-of-range taps.
#pragma once

#include <cstring>
#include <stdint.h>
#include <type_traits>

#include <cuda_runtime.h>

namespace gs {

// Element bits, moved unchanged by the transpose.
template <typename T> using RawOf = typename std::conditional<sizeof(T) == 4, uint32_t, uint16_t>::type;

// X[n, c, p] -> slot n of the workspace, pixel p, channel c.  One tile of TC
// channels x TP pixels (TC * TP = 4096 elements) per block through shared
// memory: the reads run along pixels and the writes along channels, both in
// 16-byte vectors where the layout allows (every pixel's channel run is a
// whole number of vectors: C * element size is a multiple of 16).  Block
// (ct, pt, n) = blockIdx.x; blocks with pt = 0 also zero their channels of the
// slot's zero pixel.  Elements move as raw bits.
template <typename R, int TC>
__device__ __forceinline__ void nchw_to_nhwc_block(const R *__restrict__ X, R *__restrict__ ws,
                                                   int C, int64_t P, int ctiles, int64_t ptiles,
                                                   int64_t b, R (&tile)[TC][4096 / TC + 1]) {
    constexpr int TP = 4096 / TC;               // pixels per tile
    constexpr int E = 16 / (int)sizeof(R);      // elements per 16-byte vector
    const int ct = (int)(b % ctiles);
    b /= ctiles;
    const int64_t pt = b % ptiles;
    const int64_t n = b / ptiles;
    const int c0 = ct * TC;
    const int64_t p0 = pt * TP;
    const R *src = X + n * C * P;
    R *dst = ws + n * C * (P + 1) + C;   // pixel 0 of slot n
    if (pt == 0) {
        for (int c = threadIdx.x; c < TC && c0 + c < C; c += blockDim.x) dst[c0 + c - C] = 0;
    }
    // reads: E consecutive pixels of one channel per thread and step, all of
    // a thread's loads issued before any is stored
    constexpr int NL = TC * (TP / E) / 256;
    // rows of X start on 16-byte boundaries (X itself need only be element-aligned)
    const bool vec_in = (P % E) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0;
    if (vec_in) {
        uint4 u[NL];
#pragma unroll
        for (int k = 0; k < NL; ++k) {
            const int i = threadIdx.x + k * 256;
            const int c = i / (TP / E), pv = (i - c * (TP / E)) * E;
            const int64_t gp = p0 + pv;
            u[k] = (c0 + c < C && gp < P)   // P % E == 0: a vector is all in or all out
                       ? __ldg(reinterpret_cast<const uint4 *>(src + (int64_t)(c0 + c) * P + gp))
                       : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int k = 0; k < NL; ++k) {
            const int i = threadIdx.x + k * 256;
            const int c = i / (TP / E), pv = (i - c * (TP / E)) * E;
            R v[E];
            memcpy(v, &u[k], 16);
#pragma unroll
            for (int e = 0; e < E; ++e) tile[c][pv + e] = v[e];
        }
    } else {
        for (int i = threadIdx.x; i < TC * TP; i += 256) {
            const int c = i / TP, p = i - c * TP;
            if (c0 + c < C && p0 + p < P) tile[c][p] = src[(int64_t)(c0 + c) * P + p0 + p];
        }
    }
    __syncthreads();
    // writes: E consecutive channels of one pixel per thread and step
    for (int i = threadIdx.x; i < TP * (TC / E); i += 256) {
        const int p = i / (TC / E), cv = (i - p * (TC / E)) * E;
        const int gc = c0 + cv;
        const int64_t gp = p0 + p;
        if (gc >= C || gp >= P) continue;
        R v[E];
#pragma unroll
        for (int k = 0; k < E; ++k) v[k] = tile[cv + k][p];
        uint4 u;
        memcpy(&u, v, 16);
        *reinterpret_cast<uint4 *>(dst + gp * C + gc) = u;
    }
}

template <typename R, int TC>
__global__ void __launch_bounds__(256)
nchw_to_nhwc_kernel(const R *__restrict__ X, R *__restrict__ ws, int C, int64_t P, int ctiles,
                    int64_t ptiles) {
    __shared__ R tile[TC][4096 / TC + 1];
    nchw_to_nhwc_block<R, TC>(X, ws, C, P, ctiles, ptiles, (int64_t)blockIdx.x, tile);
}

// Copy tiles per image for C channels and P positions: TC channels (the
// fewest of 16, 32, 64 that cover C, else 64) by 4096 / TC positions.
inline int copy_tc(int C) { return C <= 16 ? 16 : (C <= 32 ? 32 : 64); }
inline int64_t copy_tiles_per_image(int C, int64_t P) {
    const int TC = copy_tc(C);
    return ((int64_t)(C + TC - 1) / TC) * ((P + 4096 / TC - 1) / (4096 / TC));
}

// Copies images [0, nc) of X (channel-first, C x P each) into slots 0.. of ws.
// nc * copy_tiles_per_image(C, P) must stay below 2^31.
template <typename R>
void launch_copy_to_slots(const R *X, R *ws, int64_t nc, int C, int64_t P, cudaStream_t s) {
    const int TC = copy_tc(C);
    const int ctiles = (C + TC - 1) / TC;
    const int64_t ptiles = (P + 4096 / TC - 1) / (4096 / TC);
    const unsigned blocks = (unsigned)(nc * ctiles * ptiles);
    if (TC == 16)
        nchw_to_nhwc_kernel<R, 16><<<blocks, 256, 0, s>>>(X, ws, C, P, ctiles, ptiles);
    else if (TC == 32)
        nchw_to_nhwc_kernel<R, 32><<<blocks, 256, 0, s>>>(X, ws, C, P, ctiles, ptiles);
    else
        nchw_to_nhwc_kernel<R, 64><<<blocks, 256, 0, s>>>(X, ws, C, P, ctiles, ptiles);
}

}  // namespace gs
