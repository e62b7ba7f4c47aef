// gs_deform.cuh -- DeformConv 2-D with fp32 FMAs (every dtype and attribute):
// the general kernel for the shapes the faster ones do not take (fp16/bf16:
// the tensor-core kernels of gs_deform_st.cuh and gs_deform_tc.cuh; fp32: the
// windowed kernel of gs_deform_f32.cu).
//
// DeformConv (ai.onnx, since version 22), Inputs: the output is an ordinary
// convolution over a column of samples, each a bilinear read of X at the
// kernel tap's position moved by its offset, times its mask.
//
// Work split: a block owns one image, a tile of kTP consecutive output
// positions and up to kOCB output channels of one group.  For every kernel
// position k and chunk of kCC input channels it (1) computes, once per
// position, the four bilinear taps (in-slab offsets, weights with the mask
// folded in) -- shared by all channels of one offset group; (2) samples the
// kCC x kTP column tile into shared memory; (3) stages the matching kOCB x kCC
// slice of W; (4) accumulates the tile product in registers (each thread owns
// one position and kOCB/4 output channels).
#pragma once

#include <type_traits>

#include "gs_common.cuh"
#include "gs_deform_tc.cuh"
#include "gs_internal.h"

namespace gs {

constexpr int kDTP = 64;        // output positions per block
constexpr int kDOCB = 64;       // output channels per block
constexpr int kDCC = 32;        // input channels per chunk
constexpr int kDThreads = 256;  // 64 positions x 4 channel lanes

template <typename T>
__global__ void __launch_bounds__(kDThreads)
deform_simt_kernel(const T *__restrict__ X, const T *__restrict__ Wt, const T *__restrict__ offset,
                   const T *__restrict__ B, const T *__restrict__ mask, T *__restrict__ Y,
                   const DeformArgs a, int pos_tiles, int oc_blocks) {
    __shared__ int s_off[4][kDTP];
    __shared__ float s_w[4][kDTP];
    __shared__ float s_col[kDCC][kDTP];
    __shared__ __align__(16) float s_wk[kDOCB][kDCC + 4];

    const int P = a.oH * a.oW;
    int b = blockIdx.x;
    const int pt = b % pos_tiles;
    b /= pos_tiles;
    const int ob = b % oc_blocks;
    b /= oc_blocks;
    const int g = b % a.group;
    const int n = b / a.group;

    const int Cg = a.C / a.group, oCg = a.oC / a.group, Cog = a.C / a.offset_group;
    const int K = a.kH * a.kW;
    const int oc0 = g * oCg + ob * kDOCB;
    const int noc = min(kDOCB, g * oCg + oCg - oc0);
    const int c_begin = g * Cg;
    const int tid = threadIdx.x;
    const int p_local = tid % kDTP;
    const int lane = tid / kDTP;   // 0..3: output channels lane, lane+4, ...
    const int p0 = pt * kDTP;
    const int64_t HW = (int64_t)a.H * a.W;

    float acc[kDOCB / 4], comp[kDOCB / 4];
#pragma unroll
    for (int j = 0; j < kDOCB / 4; ++j) acc[j] = comp[j] = 0.0f;

    for (int k = 0; k < K; ++k) {
        const int kh = k / a.kW, kw = k - kh * a.kW;
        int c = c_begin;
        int cur_og = -1;
        while (c < c_begin + Cg) {
            const int og = c / Cog;
            const int cc = min(kDCC, min(c_begin + Cg, (og + 1) * Cog) - c);
            if (og != cur_og) {
                __syncthreads();
                if (tid < kDTP) {
                    const int p = p0 + tid;
                    int off4[4] = {-1, -1, -1, -1};
                    float w4[4] = {0.f, 0.f, 0.f, 0.f};
                    if (p < P) {
                        const int oh = p / a.oW, ow = p - (p / a.oW) * a.oW;
                        const int64_t plane = (int64_t)P;
                        const int64_t obase = ((int64_t)n * a.offset_group + og) * 2 * K;
                        const float dy = IO<T>::ld(offset + (obase + 2 * k) * plane + p);
                        const float dx = IO<T>::ld(offset + (obase + 2 * k + 1) * plane + p);
                        const float m = a.has_mask
                            ? IO<T>::ld(mask + (((int64_t)n * a.offset_group + og) * K + k) * plane + p)
                            : 1.0f;
                        // position = integer anchor + offset; floor/fraction of the
                        // offset are exact, so the split loses nothing
                        if (fabsf(dy) < 1.0e8f && fabsf(dx) < 1.0e8f) {
                            const float fy = floorf(dy), fx = floorf(dx);
                            const float ty = dy - fy, tx = dx - fx;
                            const int y0 = oh * a.sH - a.pad_t + kh * a.dH + (int)fy;
                            const int x0 = ow * a.sW - a.pad_l + kw * a.dW + (int)fx;
#pragma unroll
                            for (int t = 0; t < 4; ++t) {
                                const int yy = y0 + (t >> 1), xx = x0 + (t & 1);
                                if (yy >= 0 && yy < a.H && xx >= 0 && xx < a.W) {
                                    off4[t] = yy * a.W + xx;
                                    w4[t] = ((t >> 1) ? ty : 1.0f - ty) * ((t & 1) ? tx : 1.0f - tx) * m;
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        s_off[t][tid] = off4[t];
                        s_w[t][tid] = w4[t];
                    }
                }
                cur_og = og;
            }
            __syncthreads();
            // sample the column tile: s_col[ci][p] for cc channels
            for (int e = tid; e < kDCC * kDTP; e += kDThreads) {
                const int ci = e / kDTP, pp = e - ci * kDTP;
                float v = 0.0f;
                if (ci < cc) {
                    const T *Xc = X + ((int64_t)n * a.C + c + ci) * HW;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int off = s_off[t][pp];
                        if (off >= 0) v = fmaf(s_w[t][pp], IO<T>::ld(Xc + off), v);
                    }
                }
                s_col[ci][pp] = v;
            }
            // stage W[oc0 + ocl, c - c_begin + ci, kh, kw]
            for (int e = tid; e < kDOCB * kDCC; e += kDThreads) {
                const int ocl = e / kDCC, ci = e - ocl * kDCC;
                float wv = 0.0f;
                if (ocl < noc && ci < cc)
                    wv = IO<T>::ld(Wt + ((int64_t)(oc0 + ocl) * Cg + (c - c_begin + ci)) * K + k);
                s_wk[ocl][ci] = wv;
            }
            __syncthreads();
            // The chunk's dot products accumulate from zero and are then added
            // to the running sums with Kahan compensation: the error grows with
            // the chunk length, not with the full C*kH*kW.
            float part[kDOCB / 4];
#pragma unroll
            for (int j = 0; j < kDOCB / 4; ++j) part[j] = 0.0f;
            for (int ci = 0; ci < kDCC; ci += 4) {
                const float v0 = s_col[ci][p_local], v1 = s_col[ci + 1][p_local];
                const float v2 = s_col[ci + 2][p_local], v3 = s_col[ci + 3][p_local];
#pragma unroll
                for (int j = 0; j < kDOCB / 4; ++j) {
                    const float4 w = *reinterpret_cast<const float4 *>(&s_wk[lane + 4 * j][ci]);
                    float s = part[j];
                    s = fmaf(w.x, v0, s);
                    s = fmaf(w.y, v1, s);
                    s = fmaf(w.z, v2, s);
                    s = fmaf(w.w, v3, s);
                    part[j] = s;
                }
            }
#pragma unroll
            for (int j = 0; j < kDOCB / 4; ++j) {
                const float y = part[j] - comp[j];
                const float t = acc[j] + y;
                comp[j] = (t - acc[j]) - y;
                acc[j] = t;
            }
            c += cc;
            __syncthreads();
        }
    }
    const int p = p0 + p_local;
    if (p < P) {
#pragma unroll
        for (int j = 0; j < kDOCB / 4; ++j) {
            const int ocl = lane + 4 * j;
            if (ocl < noc) {
                const int oc = oc0 + ocl;
                const float bias = a.has_bias ? IO<T>::ld(B + oc) : 0.0f;
                Y[((int64_t)n * a.oC + oc) * P + p] = IO<T>::st(acc[j] + bias);
            }
        }
    }
}

template <typename T>
cudaError_t launch_deform(const void *X, const void *W, const void *offset, const void *B,
                          const void *mask, void *Y, const DeformArgs &a, cudaStream_t s) {
    if constexpr (!std::is_same<T, float>::value) {
        // half types: contraction on the tensor cores where the shape allows,
        // on the staged persistent kernel first
        bool used = false;
        cudaError_t e = launch_deform_staged<T>(X, W, offset, B, mask, Y, a, s, &used);
        if (used || e != cudaSuccess) return e;
        e = launch_deform_tc<T>(X, W, offset, B, mask, Y, a, s, &used);
        if (used || e != cudaSuccess) return e;
    } else {
        // fp32: the windowed register-tiled kernel where the shape allows
        bool used = false;
        const cudaError_t e = launch_deform_f32(X, W, offset, B, mask, Y, a, s, &used);
        if (used || e != cudaSuccess) return e;
    }
    const int P = a.oH * a.oW;
    const int pos_tiles = (P + kDTP - 1) / kDTP;
    const int oCg = a.oC / a.group;
    const int oc_blocks = (oCg + kDOCB - 1) / kDOCB;
    const int64_t blocks = (int64_t)pos_tiles * oc_blocks * a.group * a.N;
    deform_simt_kernel<T><<<(unsigned)blocks, kDThreads, 0, s>>>(
        (const T *)X, (const T *)W, (const T *)offset, (const T *)B, (const T *)mask, (T *)Y, a,
        pos_tiles, oc_blocks);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_deform_ws(const void *X, const void *W, const void *offset, const void *B,
                             const void *mask, void *Y, const DeformArgs &a, void *ws,
                             size_t ws_bytes, cudaStream_t s) {
    if constexpr (!std::is_same<T, float>::value) {
        // the staged kernel needs no workspace: it runs whenever it takes the
        // call, as in launch_deform
        if (!deform_staged_takes(a, X, W, offset, mask)) {
            bool used = false;
            const cudaError_t e = launch_deform_tc_ws<T>(X, W, offset, B, mask, Y, a, ws, ws_bytes,
                                                         s, &used);
            if (used || e != cudaSuccess) return e;
        }
    }
    return launch_deform<T>(X, W, offset, B, mask, Y, a, s);
}

// Workspace bytes gs_deform_conv_ws asks for: 0 for shapes the staged kernel
// takes (given 16-byte aligned tensors), else the channel-last path's.
template <typename T>
size_t deform_ws_bytes(const DeformArgs &a) {
    if (std::is_same<T, float>::value) return 0;
    const void *aligned16 = reinterpret_cast<const void *>(uintptr_t(256));
    if (deform_staged_takes(a, aligned16, aligned16, aligned16, a.has_mask ? aligned16 : nullptr))
        return 0;
    return deform_workspace_bytes<T>(a);
}

}  // namespace gs
