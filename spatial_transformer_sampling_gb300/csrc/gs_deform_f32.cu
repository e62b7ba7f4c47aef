// gs_deform_f32.cu -- DeformConv 2-D in fp32 on the CUDA cores for the common
// shapes: per chunk of input channels, a window of X staged in shared memory,
// the column tile gathered from it, and a register-tiled contraction with W.
//
// DeformConv (ai.onnx, since version 22), Inputs and Outputs:
//   Y[n, oc, p] = B[oc] + sum over the group's input channels c and kernel
//                 taps k of W[oc, c, k] * col[c, k, p],
// col[c, k, p] being the bilinear sample of X[n, c] at tap k's position of
// output p moved by its offset, times its mask (zero outside the image).
//
// Work split: a block owns one image, a tile of 128 consecutive output
// positions and up to 64 output channels of one group.  Per chunk of 8 input
// channels it
//   (1) copies the chunk's X window -- the rows and columns the tile's taps
//       reach with offsets of up to `margin` pixels -- into shared memory
//       (one plane per channel) with 16-byte cp.async copies, while the
//       previous chunk is multiplied;
//   (2) copies W[oc, chunk, :] transposed to [(c, k)][oc] with 4-byte cp.async
//       copies, while the column tile is gathered;
//   (3) gathers the column tile A[(c, k)][p] (8 kH kW rows x 128 positions):
//       four window reads and FMAs per value, from tap window offsets and
//       weights computed once per tile (and offset group); taps inside the
//       image but outside the window are read from global memory;
//   (4) multiplies: each thread accumulates 8 positions x 4 output channels
//       with packed FMA pairs, 3 shared-memory vector loads per 32 FMAs.
// A chunk's products are summed from zero and then added to the running sums,
// so rounding grows with the chunk length (8 kH kW), not with C kH kW.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "gs_common.cuh"
#include "gs_internal.h"
#include "gs_ptx.cuh"

namespace gs {
namespace {

constexpr int kFTP = 128;                    // output positions per tile
constexpr int kFOC = 64;                     // output channels per tile
constexpr int kFCC = 8;                      // input channels per chunk
constexpr int kFMaxK = 9;                    // kernel taps (kH kW) at most
constexpr int kFThreads = 256;
constexpr int kFWPitch = kFOC + 4;           // floats per row of the staged W chunk
constexpr int kFMaxMargin = 4;               // offset reach the window allows for
constexpr int kFPlane = 896;                 // floats per staged channel plane
constexpr int kFZero = kFPlane - 4;          // four zero floats at the end of each plane
constexpr size_t kFSmemLimit = 113 * 1024;   // two blocks per SM
constexpr uint32_t kFOutside = 0x8000u;      // tap flag: in the image, outside the window

// Dynamic shared memory of the kernel for K kernel taps: window planes |
// A [8K][128] | W chunk [8K][68] | tap offsets [K][128] (4 x u16) | weights [K][128].
__host__ __device__ constexpr size_t f32_smem(int K) {
    return (size_t)kFCC * kFPlane * 4 + (size_t)kFCC * K * kFTP * 4 +
           (size_t)kFCC * K * kFWPitch * 4 + (size_t)K * kFTP * (8 + 16);
}
static_assert(f32_smem(kFMaxK) <= kFSmemLimit, "two blocks per SM");

struct FWindow {
    int y0, x0, rh, rw;   // origin in the image, rows, columns (a multiple of 4)
};

// The X window of the tile whose first position is p0: the pixels its taps
// reach with offsets in [-margin, margin], clipped to the image.  x0 and the
// width are rounded to whole 16-byte runs (W % 4 == 0 keeps them inside).
__host__ __device__ inline FWindow f32_window(const DeformArgs &a, int p0, int margin) {
    const int P = a.oH * a.oW;
    const int p1 = (p0 + kFTP < P ? p0 + kFTP : P) - 1;
    const int oh0 = p0 / a.oW, oh1 = p1 / a.oW;
    const int ow0 = oh0 == oh1 ? p0 - oh0 * a.oW : 0;
    const int ow1 = oh0 == oh1 ? p1 - oh1 * a.oW : a.oW - 1;
    int ylo = oh0 * a.sH - a.pad_t - margin;
    int yhi = oh1 * a.sH - a.pad_t + (a.kH - 1) * a.dH + 1 + margin;
    int xlo = ow0 * a.sW - a.pad_l - margin;
    int xhi = ow1 * a.sW - a.pad_l + (a.kW - 1) * a.dW + 1 + margin;
    ylo = ylo < 0 ? 0 : ylo;
    yhi = yhi > a.H - 1 ? a.H - 1 : yhi;
    xlo = xlo < 0 ? 0 : (xlo & ~3);
    xhi = xhi > a.W - 1 ? a.W - 1 : xhi;
    FWindow w;
    w.y0 = ylo;
    w.x0 = xlo;
    w.rh = yhi >= ylo ? yhi - ylo + 1 : 0;
    w.rw = xhi >= xlo ? ((xhi + 4) & ~3) - xlo : 0;
    if (w.rh == 0 || w.rw == 0) w.rh = w.rw = 0;
    return w;
}

// Top-left tap of kernel tap k at output p (oh, ow), its bilinear fractions,
// and whether the offset is finite and in range (else the sample is zero).
__device__ __forceinline__ bool f32_tap_origin(const DeformArgs &a, const float *__restrict__ offn,
                                               int k, int p, int oh, int ow, int P, int &y0,
                                               int &x0, float &ty, float &tx) {
    const float dy = __ldg(offn + (int64_t)(2 * k) * P + p);
    const float dx = __ldg(offn + (int64_t)(2 * k + 1) * P + p);
    if (!(fabsf(dy) < 1.0e8f && fabsf(dx) < 1.0e8f)) return false;
    const float fy = floorf(dy), fx = floorf(dx);
    ty = dy - fy;
    tx = dx - fx;
    const int kh = k / a.kW, kw = k - kh * a.kW;
    y0 = oh * a.sH - a.pad_t + kh * a.dH + (int)fy;
    x0 = ow * a.sW - a.pad_l + kw * a.dW + (int)fx;
    return true;
}

template <int K>
__global__ void __launch_bounds__(kFThreads, 2)
deform_f32_kernel(const float *__restrict__ X, const float *__restrict__ Wt,
                  const float *__restrict__ offset, const float *__restrict__ Bias,
                  const float *__restrict__ mask, float *__restrict__ Y, const DeformArgs a,
                  int margin, int pos_tiles, int oc_blocks) {
    constexpr int KC = kFCC * K;   // contraction rows per chunk: (channel, tap), W's order
    extern __shared__ __align__(16) float f_smem[];
    // the window planes come first, so a tap's byte offset is its address
    unsigned char *const smem = reinterpret_cast<unsigned char *>(f_smem);
    float *const win_s = f_smem;
    float *const A_s = f_smem + kFCC * kFPlane;
    float *const W_s = A_s + KC * kFTP;
    uint2 *const off_s = reinterpret_cast<uint2 *>(W_s + KC * kFWPitch);
    float4 *const wt_s = reinterpret_cast<float4 *>(off_s + K * kFTP);

    int b = blockIdx.x;
    const int pt = b % pos_tiles;
    b /= pos_tiles;
    const int ob = b % oc_blocks;
    b /= oc_blocks;
    const int g = b % a.group;
    const int n = b / a.group;

    const int P = a.oH * a.oW, HW = a.H * a.W;
    const int Cg = a.C / a.group, oCg = a.oC / a.group, Cog = a.C / a.offset_group;
    const int oc0 = g * oCg + ob * kFOC;
    const int noc = min(kFOC, oCg - ob * kFOC);
    const int c_begin = g * Cg;
    const int p0 = pt * kFTP;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const FWindow win = f32_window(a, p0, margin);
    const float *Xn = X + (int64_t)n * a.C * HW;

    if (tid < kFCC * 4) win_s[(tid >> 2) * kFPlane + kFZero + (tid & 3)] = 0.0f;

    // this thread's window copy item (at most one: rh rw <= 892): row r,
    // 16-byte run q, the same in every channel plane
    const int nq = win.rw >> 2;
    int src_item = -1, dst_item = 0;
    if (tid < win.rh * nq) {
        const int r = tid / nq, q = tid - r * nq;
        src_item = (win.y0 + r) * a.W + win.x0 + 4 * q;
        dst_item = r * win.rw + 4 * q;
    }
    auto issue_window = [&](int c) {
        if (src_item >= 0) {
#pragma unroll
            for (int cc = 0; cc < kFCC; ++cc)
                cp_async16(smem_u32(win_s + cc * kFPlane + dst_item),
                           Xn + (int64_t)(c + cc) * HW + src_item, 16);
        }
    };
    // W[oc0 + ocl, c_rel .. c_rel + 7, :] -> W_s[e][ocl], e = c * K + k (W's own
    // order).  This thread copies e = 8 m + e_l (m < K) for output channels ocA
    // and ocA + 32; a warp's copies are 4 channels x 32-byte runs in global
    // memory and 32 distinct banks in shared memory.
    const int64_t wrow = (int64_t)Cg * K;
    const int ocA = (warp << 2) | ((lane >> 3) & 3), e_l = lane & 7;
    auto issue_w = [&](int c_rel) {
        const float *Wc = Wt + (int64_t)oc0 * wrow + (int64_t)c_rel * K + e_l;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int ocl = ocA + 32 * h;
            const bool ok = ocl < noc;
            const float *src = ok ? Wc + ocl * wrow : Wt;
            const uint32_t dst = smem_u32(W_s + e_l * kFWPitch + ocl);
#pragma unroll
            for (int m = 0; m < K; ++m)
                cp_async4(dst + (uint32_t)(m * 8 * kFWPitch * 4), ok ? src + 8 * m : Wt, ok ? 4u : 0u);
        }
    };
    // taps of (k, p) for offset group og: byte offsets of the four pixels in a
    // window plane (the zero slot outside the image; flagged when in the image
    // but outside the window) and their weights, mask folded in
    auto setup_taps = [&](int og) {
        const float *offn = offset + ((int64_t)n * a.offset_group + og) * 2 * K * P;
        const float *mskn = a.has_mask ? mask + ((int64_t)n * a.offset_group + og) * K * P : nullptr;
        for (int e = tid; e < K * kFTP; e += kFThreads) {
            const int k = e / kFTP, pl = e - k * kFTP;
            const int p = p0 + pl;
            uint32_t o[4] = {kFZero * 4, kFZero * 4, kFZero * 4, kFZero * 4};
            float w[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            int y0, x0;
            float ty, tx;
            if (p < P) {
                const int oh = p / a.oW, ow = p - oh * a.oW;
                if (f32_tap_origin(a, offn, k, p, oh, ow, P, y0, x0, ty, tx)) {
                    const float m = mskn ? __ldg(mskn + (int64_t)k * P + p) : 1.0f;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int yy = y0 + (t >> 1), xx = x0 + (t & 1);
                        if (yy >= 0 && yy < a.H && xx >= 0 && xx < a.W) {
                            w[t] = ((t >> 1) ? ty : 1.0f - ty) * ((t & 1) ? tx : 1.0f - tx) * m;
                            const uint32_t ry = (uint32_t)(yy - win.y0), rx = (uint32_t)(xx - win.x0);
                            o[t] = ry < (uint32_t)win.rh && rx < (uint32_t)win.rw
                                       ? (ry * (uint32_t)win.rw + rx) * 4
                                       : (kFZero * 4) | kFOutside;
                        }
                    }
                }
            }
            off_s[e] = make_uint2(o[0] | (o[1] << 16), o[2] | (o[3] << 16));
            wt_s[e] = make_float4(w[0], w[1], w[2], w[3]);
        }
    };

    // gather roles: position gp, channels 4 gh .. 4 gh + 3 of the chunk
    const int gp = tid & (kFTP - 1), gh = tid >> 7;
    const unsigned char *const wb = smem + gh * (4 * kFPlane * 4);
    float *const arow = A_s + gh * 4 * K * kFTP + gp;
    auto gather = [&](int c, int og) {
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const uint2 ov = off_s[k * kFTP + gp];
            const float4 w = wt_s[k * kFTP + gp];
            const unsigned char *b0 = wb + (ov.x & 0x7FFFu), *b1 = wb + ((ov.x >> 16) & 0x7FFFu);
            const unsigned char *b2 = wb + (ov.y & 0x7FFFu), *b3 = wb + ((ov.y >> 16) & 0x7FFFu);
            float v[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int pb = cc * kFPlane * 4;
                float s = w.x * *reinterpret_cast<const float *>(b0 + pb);
                s = fmaf(w.y, *reinterpret_cast<const float *>(b1 + pb), s);
                s = fmaf(w.z, *reinterpret_cast<const float *>(b2 + pb), s);
                s = fmaf(w.w, *reinterpret_cast<const float *>(b3 + pb), s);
                v[cc] = s;
            }
            if ((ov.x | ov.y) & 0x80008000u) {
                // pixels outside the window (they read the zero slot above):
                // add them from global memory
                const int p = p0 + gp;
                const int oh = p / a.oW, ow = p - oh * a.oW;
                const float *offn = offset + ((int64_t)n * a.offset_group + og) * 2 * K * P;
                int y0 = 0, x0 = 0;
                float ty, tx;
                f32_tap_origin(a, offn, k, p, oh, ow, P, y0, x0, ty, tx);
                const float wv[4] = {w.x, w.y, w.z, w.w};
                const uint32_t flags[4] = {ov.x & kFOutside, (ov.x >> 16) & kFOutside,
                                           ov.y & kFOutside, (ov.y >> 16) & kFOutside};
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    if (!flags[t]) continue;
                    const int64_t px = (int64_t)(y0 + (t >> 1)) * a.W + x0 + (t & 1);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        v[cc] = fmaf(wv[t], __ldg(Xn + (int64_t)(c + gh * 4 + cc) * HW + px), v[cc]);
                }
            }
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) arow[(cc * K + k) * kFTP] = v[cc];
        }
    };

    // contraction roles: output channels og4 .. og4 + 3, positions pg8 .. pg8 + 7;
    // a warp spans 8 channel groups x 4 position groups, so each of its
    // vector loads is one shared-memory wavefront
    const int og4 = ((lane & 7) | ((warp & 1) << 3)) * 4;
    const int pg8 = ((lane >> 3) | ((warp >> 1) << 2)) * 8;
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    const int nchunks = Cg / kFCC;
    int cur_og = -1;
    issue_window(c_begin);
    cp_async_commit();
    for (int ch = 0; ch < nchunks; ++ch) {
        const int c = c_begin + ch * kFCC;
        issue_w(c - c_begin);
        cp_async_commit();
        const int og = c / Cog;
        if (og != cur_og) {   // block-uniform
            setup_taps(og);
            cur_og = og;
        }
        cp_async_wait_pending(1);   // this chunk's window
        __syncthreads();
        gather(c, og);
        cp_async_wait_pending(0);   // this chunk's W
        __syncthreads();
        if (ch + 1 < nchunks) issue_window(c + kFCC);   // lands during the contraction
        cp_async_commit();

        // packed pairs of FMAs: positions (2i, 2i+1) x output channels
        // (j, j') and (j', j) -- each lane pair an ordinary fmaf
        float2 part[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int q = 0; q < 4; ++q) part[i][q] = make_float2(0.0f, 0.0f);
        const float *ap = A_s + pg8;
        const float *wp = W_s + og4;
#pragma unroll 8
        for (int e = 0; e < KC; ++e) {
            const float4 a0 = *reinterpret_cast<const float4 *>(ap + e * kFTP);
            const float4 a1 = *reinterpret_cast<const float4 *>(ap + e * kFTP + 4);
            const float4 w4 = *reinterpret_cast<const float4 *>(wp + e * kFWPitch);
            const float2 av[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w),
                                  make_float2(a1.x, a1.y), make_float2(a1.z, a1.w)};
            const float2 w01 = make_float2(w4.x, w4.y), w10 = make_float2(w4.y, w4.x);
            const float2 w23 = make_float2(w4.z, w4.w), w32 = make_float2(w4.w, w4.z);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                part[i][0] = fma_f32x2(av[i], w01, part[i][0]);
                part[i][1] = fma_f32x2(av[i], w10, part[i][1]);
                part[i][2] = fma_f32x2(av[i], w23, part[i][2]);
                part[i][3] = fma_f32x2(av[i], w32, part[i][3]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc[2 * i][0] += part[i][0].x;
            acc[2 * i + 1][1] += part[i][0].y;
            acc[2 * i][1] += part[i][1].x;
            acc[2 * i + 1][0] += part[i][1].y;
            acc[2 * i][2] += part[i][2].x;
            acc[2 * i + 1][3] += part[i][2].y;
            acc[2 * i][3] += part[i][3].x;
            acc[2 * i + 1][2] += part[i][3].y;
        }
        __syncthreads();   // A and W are rewritten by the next chunk
    }
    cp_async_wait_pending(0);

    const int pb = p0 + pg8;
    const bool vec = (P % 4 == 0) && ((reinterpret_cast<uintptr_t>(Y) & 15u) == 0) && pb + 8 <= P;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int ocl = og4 + j;
        if (ocl >= noc) continue;
        const int oc = oc0 + ocl;
        const float bias = a.has_bias ? __ldg(Bias + oc) : 0.0f;
        float *yr = Y + ((int64_t)n * a.oC + oc) * P + pb;
        if (vec) {
            reinterpret_cast<float4 *>(yr)[0] =
                make_float4(acc[0][j] + bias, acc[1][j] + bias, acc[2][j] + bias, acc[3][j] + bias);
            reinterpret_cast<float4 *>(yr)[1] =
                make_float4(acc[4][j] + bias, acc[5][j] + bias, acc[6][j] + bias, acc[7][j] + bias);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (pb + i < P) yr[i] = acc[i][j] + bias;
        }
    }
}

// Whether the kernel takes the shape and X pointer, and the window margin.
bool f32_params(const DeformArgs &a, const void *X, int *margin) {
    const int K = a.kH * a.kW;
    if (a.N < 1 || a.C < 1 || a.oC < 1 || a.oH < 1 || a.oW < 1 || a.H < 1 || a.W < 1) return false;
    if (K < 1 || K > kFMaxK || a.group < 1 || a.offset_group < 1) return false;
    const int Cg = a.C / a.group, Cog = a.C / a.offset_group;
    if (Cg % kFCC != 0 || Cog % kFCC != 0) return false;
    if (a.W % 4 != 0 || (reinterpret_cast<uintptr_t>(X) & 15u) != 0) return false;
    if ((int64_t)a.H * a.W > INT32_MAX / 2 || (int64_t)a.oH * a.oW > INT32_MAX / 2) return false;
    const int P = a.oH * a.oW;
    const int tiles = (P + kFTP - 1) / kFTP;
    const int64_t blocks = (int64_t)tiles * ((a.oC / a.group + kFOC - 1) / kFOC) * a.group * a.N;
    if (blocks > INT32_MAX) return false;
    for (int m = kFMaxMargin; m >= 0; --m) {
        int rh = 0, rw = 0;
        for (int t = 0; t < tiles; ++t) {
            const FWindow w = f32_window(a, t * kFTP, m);
            rh = w.rh > rh ? w.rh : rh;
            rw = w.rw > rw ? w.rw : rw;
        }
        if ((int64_t)rh * rw <= kFZero) {
            *margin = m;
            return true;
        }
    }
    return false;
}

template <int K>
cudaError_t launch_f32_k(const float *X, const float *W, const float *offset, const float *B,
                         const float *mask, float *Y, const DeformArgs &a, int margin,
                         cudaStream_t s) {
    static DeviceFlags attr_set;
    const cudaError_t e = once_per_device(attr_set, [] {
        cudaError_t r = cudaFuncSetAttribute(deform_f32_kernel<K>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)f32_smem(K));
        if (r == cudaSuccess)
            r = cudaFuncSetAttribute(deform_f32_kernel<K>,
                                     cudaFuncAttributePreferredSharedMemoryCarveout,
                                     (int)cudaSharedmemCarveoutMaxShared);
        return r;
    });
    if (e != cudaSuccess) return e;
    const int P = a.oH * a.oW;
    const int pos_tiles = (P + kFTP - 1) / kFTP;
    const int oc_blocks = (a.oC / a.group + kFOC - 1) / kFOC;
    const int64_t blocks = (int64_t)pos_tiles * oc_blocks * a.group * a.N;
    deform_f32_kernel<K><<<(unsigned)blocks, kFThreads, f32_smem(K), s>>>(
        X, W, offset, B, mask, Y, a, margin, pos_tiles, oc_blocks);
    return cudaGetLastError();
}

}  // namespace

bool deform_f32_takes(const DeformArgs &args, const void *X) {
    int m;
    return f32_params(args, X, &m);
}

cudaError_t launch_deform_f32(const void *X, const void *W, const void *offset, const void *B,
                              const void *mask, void *Y, const DeformArgs &a, cudaStream_t s,
                              bool *used) {
    *used = false;
    int m = 0;
    if (!f32_params(a, X, &m)) return cudaSuccess;
    const float *x = (const float *)X, *w = (const float *)W, *o = (const float *)offset;
    const float *b = (const float *)B, *mk = (const float *)mask;
    float *y = (float *)Y;
    cudaError_t e = cudaSuccess;
    switch (a.kH * a.kW) {
        case 1: e = launch_f32_k<1>(x, w, o, b, mk, y, a, m, s); break;
        case 2: e = launch_f32_k<2>(x, w, o, b, mk, y, a, m, s); break;
        case 3: e = launch_f32_k<3>(x, w, o, b, mk, y, a, m, s); break;
        case 4: e = launch_f32_k<4>(x, w, o, b, mk, y, a, m, s); break;
        case 5: e = launch_f32_k<5>(x, w, o, b, mk, y, a, m, s); break;
        case 6: e = launch_f32_k<6>(x, w, o, b, mk, y, a, m, s); break;
        case 7: e = launch_f32_k<7>(x, w, o, b, mk, y, a, m, s); break;
        case 8: e = launch_f32_k<8>(x, w, o, b, mk, y, a, m, s); break;
        default: e = launch_f32_k<9>(x, w, o, b, mk, y, a, m, s); break;
    }
    *used = true;
    return e;
}

}  // namespace gs
