// gs_deform_tc.cuh -- DeformConv 2-D with the contraction on the tensor cores
// (tcgen05, fp32 accumulation in tensor memory), for fp16/bf16 I/O.
//
// DeformConv (ai.onnx, since version 22), Inputs: Y[n, oc, p] = B[oc] +
// sum_{c, k} W[oc, c, k] * col[n, (c, k), p], where col is the bilinear sample
// of X[n, c] at output position p's kernel tap k moved by its offset, times
// its mask.  Here the GEMM is M = output positions, N = oC, K = C * kH * kW.
//
// One CTA owns a tile of 128 consecutive output positions of one image and
// all oC output channels (the accumulator: 128 TMEM lanes x oC columns).
//  - W is repacked once per CTA into shared memory as the B operand:
//    K-major, 8-row x 16-byte core matrices, no swizzling.
//  - For each chunk (kernel tap k, up to 64 input channels) all 256 threads
//    sample the column tile straight into an A-operand buffer (each thread
//    writes whole 16-byte core-matrix rows: 8 channels of one position).
//    Two buffers alternate; a buffer is refilled only after the MMAs that read
//    it have completed (tcgen05.commit -> mbarrier, bounded wait).
//  - One thread issues the chunk's MMAs (M=128, N=oC, K=16 each).
//  - Epilogue: tcgen05.ld, + bias, round to T, store Y.
// The column tile is rounded to T before the MMA; accumulation is fp32.
#pragma once

#include <type_traits>

#include "gs_common.cuh"
#include "gs_copy.cuh"
#include "gs_internal.h"
#include "gs_ptx.cuh"

namespace gs {

constexpr int kTcThreads = 256;
constexpr int kTcM = 128;   // output positions per CTA (= TMEM lanes)
constexpr int kTcMaxSmem = 200 * 1024;   // dynamic shared memory: packed W + two A buffers

struct DeformTcParams {
    int kc;            // input channels per chunk (64, 32 or 16)
    int tiles;         // position tiles per image
    uint32_t w_bytes;  // bytes of the packed W (all kernel taps)
    uint32_t tmem_cols;
};

template <typename T> __device__ __forceinline__ uint32_t pack_pair(float a, float b);
template <> __device__ __forceinline__ uint32_t pack_pair<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t pack_pair<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <typename T>
__global__ void __launch_bounds__(kTcThreads, 1)
deform_tc_kernel(const T *__restrict__ X, const T *__restrict__ Wt, const T *__restrict__ offset,
                 const T *__restrict__ Bias, const T *__restrict__ mask, T *__restrict__ Y,
                 const DeformArgs a, const DeformTcParams q) {
    unsigned *err = a.err;
    extern __shared__ __align__(1024) unsigned char tc_smem[];
    __shared__ __align__(8) uint64_t mma_done[2];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int tid = threadIdx.x;
    const int n = blockIdx.x / q.tiles;
    const int tile = blockIdx.x - n * q.tiles;
    const int P = a.oH * a.oW;
    const int p0 = tile * kTcM;
    const int C = a.C, oC = a.oC, K = a.kH * a.kW;
    const int KC = q.kc;
    const int chunks_per_tap = C / KC;
    const int nchunks = K * chunks_per_tap;
    unsigned char *w_s = tc_smem;                      // packed W
    unsigned char *a_s = tc_smem + q.w_bytes;          // two A buffers
    const uint32_t a_buf_bytes = (uint32_t)kTcM * KC * 2;
    const uint32_t sbo_a = (uint32_t)KC * 16;          // 8 rows x KC channels x 2 bytes
    const uint32_t sbo_b = (uint32_t)C * 16;
    const uint32_t slice_b = (uint32_t)oC * C * 2;

    if (tid < 32) tmem_alloc(&s_tmem, q.tmem_cols);
    if (tid == 0) {
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        fence_mbar_init();
        s_abort = 0;
    }
    // repack W[oc, c, k] into core-matrix rows of 8 channels (16 bytes)
    for (int e = tid; e < K * oC * (C / 8); e += kTcThreads) {
        const int c8 = e % (C / 8);
        const int oc = (e / (C / 8)) % oC;
        const int k = e / ((C / 8) * oC);
        const T *src = Wt + ((int64_t)oc * C + c8 * 8) * K + k;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = IO<T>::ld(src + (int64_t)i * K);
        uint4 pk = make_uint4(pack_pair<T>(v[0], v[1]), pack_pair<T>(v[2], v[3]),
                              pack_pair<T>(v[4], v[5]), pack_pair<T>(v[6], v[7]));
        *reinterpret_cast<uint4 *>(w_s + (size_t)k * slice_b + (oc / 8) * sbo_b + c8 * 128 +
                                   (oc % 8) * 16) = pk;
    }
    fence_proxy_async_smem();
    tcgen05_fence_before_sync();
    __syncthreads();
    tcgen05_fence_after_sync();
    const uint32_t tmem_d = s_tmem;

    const int p_local = tid & (kTcM - 1);
    const int half = tid >> 7;   // 0/1: this thread's octets are half, half+2, ...
    const int p = p0 + p_local;
    const bool live = p < P;
    const int oh = live ? p / a.oW : 0, ow = live ? p - (p / a.oW) * a.oW : 0;
    const int64_t HW = (int64_t)a.H * a.W;
    const T *Xn = X + (int64_t)n * C * HW;
    const uint32_t idesc = umma_idesc_f16(std::is_same<T, __nv_bfloat16>::value, kTcM, oC);

    int cur_k = -1;
    int toff[4];
    float tw[4];
    int chunk = 0;
    for (; chunk < nchunks; ++chunk) {
        const int k = chunk / chunks_per_tap;
        const int cb = chunk - k * chunks_per_tap;
        const int buf = chunk & 1;
        if (k != cur_k) {
            // bilinear taps of (p, k), mask folded into the weights
            cur_k = k;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                toff[t] = -1;
                tw[t] = 0.0f;
            }
            if (live) {
                const int kh = k / a.kW, kw = k - (k / a.kW) * a.kW;
                const int64_t plane = P;
                const float dy = IO<T>::ld(offset + ((int64_t)n * 2 * K + 2 * k) * plane + p);
                const float dx = IO<T>::ld(offset + ((int64_t)n * 2 * K + 2 * k + 1) * plane + p);
                const float m = a.has_mask ? IO<T>::ld(mask + ((int64_t)n * K + k) * plane + p) : 1.0f;
                if (fabsf(dy) < 1.0e8f && fabsf(dx) < 1.0e8f) {
                    const float fy = floorf(dy), fx = floorf(dx);
                    const float ty = dy - fy, tx = dx - fx;
                    const int y0 = oh * a.sH - a.pad_t + kh * a.dH + (int)fy;
                    const int x0 = ow * a.sW - a.pad_l + kw * a.dW + (int)fx;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const int yy = y0 + (t >> 1), xx = x0 + (t & 1);
                        if (yy >= 0 && yy < a.H && xx >= 0 && xx < a.W) {
                            toff[t] = yy * a.W + xx;
                            tw[t] = ((t >> 1) ? ty : 1.0f - ty) * ((t & 1) ? tx : 1.0f - tx) * m;
                        }
                    }
                }
            }
        }
        if (chunk >= 2) {
            // the MMAs of chunk-2 read this buffer: wait until they are done
            if (!mbar_wait_bounded(&mma_done[buf], (uint32_t)((chunk - 2) >> 1) & 1u, err))
                s_abort = 1;
            __syncthreads();
            if (s_abort) break;
        }
        unsigned char *abuf = a_s + (size_t)buf * a_buf_bytes;
        for (int oq = half; oq < KC / 8; oq += 2) {
            const int c0 = cb * KC + oq * 8;
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const T *Xc = Xn + (int64_t)(c0 + i) * HW;
                float s = 0.0f;
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    if (toff[t] >= 0) s = fmaf(tw[t], IO<T>::ld(Xc + toff[t]), s);
                v[i] = s;
            }
            *reinterpret_cast<uint4 *>(abuf + (p_local / 8) * sbo_a + oq * 128 + (p_local % 8) * 16) =
                make_uint4(pack_pair<T>(v[0], v[1]), pack_pair<T>(v[2], v[3]),
                           pack_pair<T>(v[4], v[5]), pack_pair<T>(v[6], v[7]));
        }
        fence_proxy_async_smem();   // the tile is read by the tensor cores (async proxy)
        __syncthreads();
        if (tid == 0) {
            tcgen05_fence_after_sync();
            const uint32_t a_addr = smem_u32(abuf);
            const uint32_t b_addr = smem_u32(w_s) + (uint32_t)k * slice_b + (uint32_t)(cb * KC / 8) * 128;
            for (int ks = 0; ks < KC / 16; ++ks) {
                const uint64_t ad = umma_desc_kmajor(a_addr + ks * 256, 128, sbo_a);
                const uint64_t bd = umma_desc_kmajor(b_addr + ks * 256, 128, sbo_b);
                umma_f16(tmem_d, ad, bd, idesc, (chunk > 0 || ks > 0) ? 1u : 0u);
            }
            umma_commit(&mma_done[buf]);
        }
    }

    const bool aborted = chunk < nchunks;
    if (!aborted) {
        // all MMAs are done once the last commit has arrived
        const int last = nchunks - 1;
        if (!mbar_wait_bounded(&mma_done[last & 1], (uint32_t)(last >> 1) & 1u, err)) s_abort = 1;
    }
    __syncthreads();
    if (s_abort) {
        // a wait gave up: give the outstanding MMAs a bounded chance to finish
        // before the accumulator is released
        if (tid == 0) {
            const int last = chunk < nchunks ? chunk - 1 : nchunks - 1;
            if (last >= 0) mbar_wait_bounded(&mma_done[last & 1], (uint32_t)(last >> 1) & 1u, nullptr);
        }
        tcgen05_fence_before_sync();
        __syncthreads();
        if (tid < 32) {
            tcgen05_fence_after_sync();
            tmem_dealloc(tmem_d, q.tmem_cols);
        }
        return;
    }
    tcgen05_fence_after_sync();

    // epilogue: warp w reads TMEM lanes 32*(w%4).. (positions) and half of the
    // columns (output channels)
    const int warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3, ch = warp >> 2;
    const int pe = p0 + lq * 32 + lane;
    const int cols = oC / 2;
    for (int col0 = ch * cols; col0 < (ch + 1) * cols; col0 += 8) {
        float v[8];
        tmem_ld_x8(tmem_d + ((uint32_t)(lq * 32) << 16) + (uint32_t)col0, v);
        if (pe < P) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int oc = col0 + i;
                const float b = a.has_bias ? IO<T>::ld(Bias + oc) : 0.0f;
                Y[((int64_t)n * oC + oc) * P + pe] = IO<T>::st(v[i] + b);
            }
        }
    }
    tcgen05_fence_before_sync();
    __syncthreads();
    if (tid < 32) {
        tcgen05_fence_after_sync();
        tmem_dealloc(tmem_d, q.tmem_cols);
    }
}

// Host side: the tensor-core path handles group == offset_group == 1,
// C % 16 == 0, oC % 16 == 0 with 16 <= oC <= 256, and a packed W that fits
// next to the two column buffers in shared memory; *used reports whether it
// ran.
template <typename T>
cudaError_t launch_deform_tc(const void *X, const void *W, const void *offset, const void *B,
                             const void *mask, void *Y, const DeformArgs &a, cudaStream_t s,
                             bool *used) {
    *used = false;
    if (a.group != 1 || a.offset_group != 1) return cudaSuccess;
    if (a.C % 16 != 0 || a.oC % 16 != 0 || a.oC < 16 || a.oC > 256) return cudaSuccess;
    DeformTcParams q;
    q.kc = a.C % 64 == 0 ? 64 : (a.C % 32 == 0 ? 32 : 16);
    const int P = a.oH * a.oW;
    q.tiles = (P + kTcM - 1) / kTcM;
    q.w_bytes = (uint32_t)a.kH * a.kW * a.oC * a.C * 2;
    const size_t smem = (size_t)q.w_bytes + 2 * (size_t)kTcM * q.kc * 2;
    if (smem > 200 * 1024) return cudaSuccess;
    uint32_t cols = 32;
    while (cols < (uint32_t)a.oC) cols <<= 1;
    q.tmem_cols = cols;
    const cudaError_t e = cudaFuncSetAttribute(deform_tc_kernel<T>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (int64_t)a.N * q.tiles;
    deform_tc_kernel<T><<<(unsigned)blocks, kTcThreads, smem, s>>>(
        (const T *)X, (const T *)W, (const T *)offset, (const T *)B, (const T *)mask, (T *)Y, a, q);
    *used = true;
    return cudaGetLastError();
}

// ------------------------------------------------------------------
// Channel-last variant (gs_deform_conv_ws): X is first copied to channel-last
// slots in the workspace (gs_copy.cuh) and W packed there once in the B
// operand's layout.  Each CTA copies the packed W with 16-byte loads, and
// samples the column tile eight channels per lane: a bilinear tap of one
// position is one 16-byte load from that pixel's channel run, the KC / 8
// lanes of a position together reading whole pixel lines.  A tap outside X
// reads the slot's zero pixel.  Weights, mask folding and the order of the
// four fmaf per column value are those of deform_tc_kernel, so both give the
// same values.

// W[oc, c, k] -> workspace, K-major core-matrix rows of 8 channels (16 bytes)
// per (k, oc): byte k * oC*C*2 + (oc / 8) * C*16 + (c / 8) * 128 + (oc % 8) * 16.
// Element e of the pack (one 16-byte row); e < K * oC * (C / 8).
template <typename T>
__device__ __forceinline__ void deform_pack_w_row(const T *__restrict__ Wt, uint16_t *__restrict__ wp,
                                                  int oC, int C, int K, int e) {
    const int c8 = e % (C / 8);
    const int oc = (e / (C / 8)) % oC;
    const int k = e / ((C / 8) * oC);
    const uint16_t *src = reinterpret_cast<const uint16_t *>(Wt) + ((int64_t)oc * C + c8 * 8) * K + k;
    uint16_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = src[(int64_t)i * K];
    uint4 u;
    memcpy(&u, v, 16);
    *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(wp) + (size_t)k * oC * C * 2 +
                               (size_t)(oc / 8) * C * 16 + c8 * 128 + (oc % 8) * 16) = u;
}

// One launch for the channel-last path's preparation: blocks below
// copy_blocks copy X to the slots (nchw_to_nhwc_block), the rest pack W.
template <typename T, int TC>
__global__ void __launch_bounds__(256)
deform_prep_kernel(const uint16_t *__restrict__ X, uint16_t *__restrict__ slots, int C, int64_t P,
                   int ctiles, int64_t ptiles, int64_t copy_blocks, const T *__restrict__ Wt,
                   uint16_t *__restrict__ wp, int oC, int K) {
    __shared__ uint16_t tile[TC][4096 / TC + 1];
    const int64_t b = blockIdx.x;
    if (b < copy_blocks) {
        nchw_to_nhwc_block<uint16_t, TC>(X, slots, C, P, ctiles, ptiles, b, tile);
        return;
    }
    const int e = (int)(b - copy_blocks) * blockDim.x + threadIdx.x;
    if (e < K * oC * (C / 8)) deform_pack_w_row<T>(Wt, wp, oC, C, K, e);
}

// Offsets and mask of position p's kernel tap k (plane = P positions).
template <typename T>
__device__ __forceinline__ void deform_tap_inputs(const T *__restrict__ offset,
                                                  const T *__restrict__ mask, const DeformArgs &a,
                                                  int n, int k, int p, int P, float &dy, float &dx,
                                                  float &m) {
    const int K = a.kH * a.kW;
    dy = IO<T>::ld(offset + ((int64_t)n * 2 * K + 2 * k) * P + p);
    dx = IO<T>::ld(offset + ((int64_t)n * 2 * K + 2 * k + 1) * P + p);
    m = a.has_mask ? IO<T>::ld(mask + ((int64_t)n * K + k) * P + p) : 1.0f;
}

// KC input channels per chunk (64, 32 or 16); a position's KC / 8 lanes each
// take one 16-byte octet, and each thread takes KC / 16 positions per chunk.
template <typename T, int KC>
__global__ void __launch_bounds__(kTcThreads, 1)
deform_tc_nhwc_kernel(const T *__restrict__ Xs, const uint4 *__restrict__ wpk,
                      const T *__restrict__ offset, const T *__restrict__ Bias,
                      const T *__restrict__ mask, T *__restrict__ Y, const DeformArgs a,
                      const DeformTcParams q, int n_begin) {
    constexpr int LPP = KC / 8;                 // lanes per position
    constexpr int PPP = kTcThreads / LPP;       // positions per pass
    constexpr int NP = kTcM / PPP;              // positions per thread
    unsigned *err = a.err;
    extern __shared__ __align__(1024) unsigned char tc_smem[];
    __shared__ __align__(8) uint64_t mma_done[2];
    __shared__ __align__(8) uint64_t w_ready;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ int s_toff[4][kTcM];     // element offsets of the taps from pixel 0 (-C: zero pixel)
    __shared__ float s_tw[4][kTcM];     // bilinear weight x mask

    const int tid = threadIdx.x;
    const int ni = blockIdx.x / q.tiles;   // image within the chunk
    const int tile = blockIdx.x - ni * q.tiles;
    const int n = n_begin + ni;
    const int P = a.oH * a.oW;
    const int p0 = tile * kTcM;
    const int C = a.C, oC = a.oC, K = a.kH * a.kW;
    const int chunks_per_tap = C / KC;
    const int nchunks = K * chunks_per_tap;
    // 64-channel chunks use the 128-byte-swizzled A layout: the eight lanes that
    // store one position's eight channel octets then hit eight different bank
    // groups (unswizzled, the octets sit 128 bytes apart and collide).
    constexpr bool kSwz = KC == 64;
    unsigned char *w_s = tc_smem;                      // packed W
    // two A buffers, 1024-byte aligned (the swizzle atom); the launch asks for
    // 1 KB of slack
    const uint32_t a_pad = (1024u - ((smem_u32(tc_smem) + q.w_bytes) & 1023u)) & 1023u;
    unsigned char *a_s = tc_smem + q.w_bytes + a_pad;
    constexpr uint32_t a_buf_bytes = (uint32_t)kTcM * KC * 2;
    constexpr uint32_t sbo_a = (uint32_t)KC * 16;      // 8 rows x KC channels x 2 bytes
    const uint32_t sbo_b = (uint32_t)C * 16;
    const uint32_t slice_b = (uint32_t)oC * C * 2;

    if (tid < 32) tmem_alloc(&s_tmem, q.tmem_cols);
    if (tid == 0) {
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        mbar_init(&w_ready, 1);
        fence_mbar_init();
        s_abort = 0;
        // the packed W arrives by bulk copies while the first chunk is sampled
        mbar_arrive_expect_tx(&w_ready, q.w_bytes);
        for (uint32_t off = 0; off < q.w_bytes; off += 32768u)
            bulk_copy_g2s(w_s + off, reinterpret_cast<const unsigned char *>(wpk) + off,
                          min(32768u, q.w_bytes - off), &w_ready);
    }
    tcgen05_fence_before_sync();
    __syncthreads();
    tcgen05_fence_after_sync();
    const uint32_t tmem_d = s_tmem;

    const int64_t HW = (int64_t)a.H * a.W;
    const T *Xn = Xs + (int64_t)ni * C * (HW + 1) + C;   // pixel 0 of the slot
    const uint32_t idesc = umma_idesc_f16(std::is_same<T, __nv_bfloat16>::value, kTcM, oC);
    const int j = tid % LPP, q0 = tid / LPP;

    // threads 0..kTcM-1 own one position each for the tap setup; the next
    // kernel tap's offsets and mask are loaded one chunk ahead
    const int pt = p0 + tid;
    const bool tap_owner = tid < kTcM && pt < P;
    float ndy = 0.0f, ndx = 0.0f, nm = 0.0f;
    if (tap_owner) deform_tap_inputs<T>(offset, mask, a, n, 0, pt, P, ndy, ndx, nm);

    int cur_k = -1;
    bool w_waited = false;
    int chunk = 0;
    for (; chunk < nchunks; ++chunk) {
        const int k = chunk / chunks_per_tap;
        const int cb = chunk - k * chunks_per_tap;
        const int buf = chunk & 1;
        if (k != cur_k) {
            // bilinear taps of (position, k), mask folded into the weights; every
            // thread has passed the previous chunk's barrier, so no one still
            // reads the old taps
            cur_k = k;
            if (tid < kTcM) {
                int toff[4] = {-C, -C, -C, -C};
                float tw[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (tap_owner) {
                    const float dy = ndy, dx = ndx, m = nm;
                    if (k + 1 < K) deform_tap_inputs<T>(offset, mask, a, n, k + 1, pt, P, ndy, ndx, nm);
                    const int oh = pt / a.oW, ow = pt - (pt / a.oW) * a.oW;
                    const int kh = k / a.kW, kw = k - (k / a.kW) * a.kW;
                    if (fabsf(dy) < 1.0e8f && fabsf(dx) < 1.0e8f) {
                        const float fy = floorf(dy), fx = floorf(dx);
                        const float ty = dy - fy, tx = dx - fx;
                        const int y0 = oh * a.sH - a.pad_t + kh * a.dH + (int)fy;
                        const int x0 = ow * a.sW - a.pad_l + kw * a.dW + (int)fx;
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int yy = y0 + (t >> 1), xx = x0 + (t & 1);
                            if (yy >= 0 && yy < a.H && xx >= 0 && xx < a.W) {
                                toff[t] = (yy * a.W + xx) * C;
                                tw[t] = ((t >> 1) ? ty : 1.0f - ty) * ((t & 1) ? tx : 1.0f - tx) * m;
                            }
                        }
                    }
                }
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    s_toff[t][tid] = toff[t];
                    s_tw[t][tid] = tw[t];
                }
            }
        }
        if (chunk >= 2) {
            // the MMAs of chunk-2 read this buffer: wait until they are done
            if (!mbar_wait_bounded(&mma_done[buf], (uint32_t)((chunk - 2) >> 1) & 1u, err))
                s_abort = 1;
        }
        __syncthreads();
        if (s_abort) break;
        unsigned char *abuf = a_s + (size_t)buf * a_buf_bytes;
        const T *Xc = Xn + cb * KC + j * 8;
        uint4 raw[NP][4];
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int pl = q0 + i * PPP;
#pragma unroll
            for (int t = 0; t < 4; ++t)
                raw[i][t] = __ldg(reinterpret_cast<const uint4 *>(Xc + s_toff[t][pl]));
        }
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int pl = q0 + i * PPP;
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.0f;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float w = s_tw[t][pl];
                const T *h = reinterpret_cast<const T *>(&raw[i][t]);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = fmaf(w, IO<T>::to_float(h[e]), v[e]);
            }
            const uint32_t a_off = kSwz ? (uint32_t)((pl / 8) * 1024 + (pl % 8) * 128 +
                                                     ((j ^ (pl % 8)) << 4))
                                        : (uint32_t)((pl / 8) * sbo_a + j * 128 + (pl % 8) * 16);
            *reinterpret_cast<uint4 *>(abuf + a_off) =
                make_uint4(pack_pair<T>(v[0], v[1]), pack_pair<T>(v[2], v[3]),
                           pack_pair<T>(v[4], v[5]), pack_pair<T>(v[6], v[7]));
        }
        fence_proxy_async_smem();   // the tile is read by the tensor cores (async proxy)
        __syncthreads();
        if (tid == 0) {
            bool go = true;
            if (!w_waited) {
                go = mbar_wait_bounded(&w_ready, 0, err);
                w_waited = go;
            }
            if (go) {
                tcgen05_fence_after_sync();
                const uint32_t a_addr = smem_u32(abuf);
                const uint32_t b_addr =
                    smem_u32(w_s) + (uint32_t)k * slice_b + (uint32_t)(cb * KC / 8) * 128;
#pragma unroll
                for (int ks = 0; ks < KC / 16; ++ks) {
                    const uint64_t ad = kSwz ? umma_desc_kmajor_sw128(a_addr + ks * 32, 1024)
                                             : umma_desc_kmajor(a_addr + ks * 256, 128, sbo_a);
                    const uint64_t bd = umma_desc_kmajor(b_addr + ks * 256, 128, sbo_b);
                    umma_f16(tmem_d, ad, bd, idesc, (chunk > 0 || ks > 0) ? 1u : 0u);
                }
                umma_commit(&mma_done[buf]);
            } else {
                s_abort = 1;   // seen by all at the next chunk's barrier
            }
        }
    }

    const bool aborted = chunk < nchunks || s_abort;
    if (!aborted) {
        // all MMAs are done once the last commit has arrived
        const int last = nchunks - 1;
        if (!mbar_wait_bounded(&mma_done[last & 1], (uint32_t)(last >> 1) & 1u, err)) s_abort = 1;
    }
    __syncthreads();
    if (s_abort) {
        // a wait gave up: give the outstanding copy and MMAs a bounded chance to
        // finish before shared memory and the accumulator are released
        if (tid == 0) {
            if (!w_waited) mbar_wait_bounded(&w_ready, 0, nullptr);
            const int last = chunk < nchunks ? chunk - 1 : nchunks - 1;
            if (last >= 0 && w_waited)
                mbar_wait_bounded(&mma_done[last & 1], (uint32_t)(last >> 1) & 1u, nullptr);
        }
        tcgen05_fence_before_sync();
        __syncthreads();
        if (tid < 32) {
            tcgen05_fence_after_sync();
            tmem_dealloc(tmem_d, q.tmem_cols);
        }
        return;
    }
    tcgen05_fence_after_sync();

    const int warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3, ch = warp >> 2;
    const int pe = p0 + lq * 32 + lane;
    const int cols = oC / 2;
    for (int col0 = ch * cols; col0 < (ch + 1) * cols; col0 += 8) {
        float v[8];
        tmem_ld_x8(tmem_d + ((uint32_t)(lq * 32) << 16) + (uint32_t)col0, v);
        if (pe < P) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int oc = col0 + i;
                const float b = a.has_bias ? IO<T>::ld(Bias + oc) : 0.0f;
                Y[((int64_t)n * oC + oc) * P + pe] = IO<T>::st(v[i] + b);
            }
        }
    }
    tcgen05_fence_before_sync();
    __syncthreads();
    if (tid < 32) {
        tcgen05_fence_after_sync();
        tmem_dealloc(tmem_d, q.tmem_cols);
    }
}

// Tensor-core parameters for a shape, false when the tensor-core path does
// not take it (see launch_deform_tc).
inline bool deform_tc_params(const DeformArgs &a, DeformTcParams *q, size_t *smem) {
    if (a.group != 1 || a.offset_group != 1) return false;
    if (a.C % 16 != 0 || a.oC % 16 != 0 || a.oC < 16 || a.oC > 256) return false;
    q->kc = a.C % 64 == 0 ? 64 : (a.C % 32 == 0 ? 32 : 16);
    const int P = a.oH * a.oW;
    q->tiles = (P + kTcM - 1) / kTcM;
    q->w_bytes = (uint32_t)a.kH * a.kW * a.oC * a.C * 2;
    *smem = (size_t)q->w_bytes + 2 * (size_t)kTcM * q->kc * 2 + 1024;   // + alignment slack
    if (*smem > (size_t)kTcMaxSmem) return false;
    uint32_t cols = 32;
    while (cols < (uint32_t)a.oC) cols <<= 1;
    q->tmem_cols = cols;
    return true;
}

// Workspace of the channel-last DeformConv: the packed W (rounded up to 256
// bytes), then image slots of (H*W + 1) * C elements.
inline size_t deform_w_region(const DeformTcParams &q) { return ((size_t)q.w_bytes + 255) / 256 * 256; }
inline size_t deform_slot_bytes(const DeformArgs &a) {
    return (size_t)a.C * ((size_t)a.H * a.W + 1) * 2;
}

// Workspace bytes the channel-last path asks for (0: it never takes the shape):
// W and a slot for every image.
template <typename T>
size_t deform_workspace_bytes(const DeformArgs &a) {
    if (std::is_same<T, float>::value) return 0;
    DeformTcParams q;
    size_t smem;
    if (!deform_tc_params(a, &q, &smem)) return 0;
    if ((int64_t)a.C * ((int64_t)a.H * a.W + 1) >= ((int64_t)1 << 31)) return 0;
    return deform_w_region(q) + (size_t)a.N * deform_slot_bytes(a);
}

// Runs the channel-last path when the workspace holds W and at least one
// slot; *used reports whether it ran.
template <typename T>
cudaError_t launch_deform_tc_ws(const void *X, const void *W, const void *offset, const void *B,
                                const void *mask, void *Y, const DeformArgs &a, void *ws,
                                size_t ws_bytes, cudaStream_t s, bool *used) {
    *used = false;
    if (!ws || deform_workspace_bytes<T>(a) == 0) return cudaSuccess;
    DeformTcParams q;
    size_t smem;
    deform_tc_params(a, &q, &smem);
    const size_t wreg = deform_w_region(q), slot = deform_slot_bytes(a);
    if (ws_bytes < wreg + slot) return cudaSuccess;
    // the largest dynamic shared memory this path uses (deform_tc_params), set
    // once per device
    static DeviceFlags attr_set;
    const cudaError_t ae = once_per_device(attr_set, [] {
        for (const void *f : {(const void *)deform_tc_nhwc_kernel<T, 64>,
                              (const void *)deform_tc_nhwc_kernel<T, 32>,
                              (const void *)deform_tc_nhwc_kernel<T, 16>}) {
            const cudaError_t e =
                cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcMaxSmem);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    });
    if (ae != cudaSuccess) return ae;
    const int K = a.kH * a.kW;
    const int packs = K * a.oC * (a.C / 8);
    uint16_t *slots = (uint16_t *)((unsigned char *)ws + wreg);
    const int64_t HW = (int64_t)a.H * a.W;
    const int64_t max_blocks = ((int64_t)1 << 31) - 1;
    int64_t per = std::min<int64_t>((int64_t)a.N, (int64_t)((ws_bytes - wreg) / slot));
    per = std::min<int64_t>(per, std::max<int64_t>(1, max_blocks / copy_tiles_per_image(a.C, HW)));
    per = std::min<int64_t>(per, std::max<int64_t>(1, max_blocks / q.tiles));
    for (int64_t n0 = 0; n0 < a.N; n0 += per) {
        const int64_t nc = std::min<int64_t>(per, a.N - n0);
        if (n0 == 0) {
            // the first chunk's copy and the W pack share one launch
            const int TC = copy_tc(a.C);
            const int ctiles = (a.C + TC - 1) / TC;
            const int64_t ptiles = (HW + 4096 / TC - 1) / (4096 / TC);
            const int64_t copy_blocks = nc * ctiles * ptiles;
            const unsigned blocks = (unsigned)(copy_blocks + (packs + 255) / 256);
            const uint16_t *Xc = (const uint16_t *)X;
            if (TC == 16)
                deform_prep_kernel<T, 16><<<blocks, 256, 0, s>>>(Xc, slots, a.C, HW, ctiles, ptiles,
                                                                copy_blocks, (const T *)W,
                                                                (uint16_t *)ws, a.oC, K);
            else if (TC == 32)
                deform_prep_kernel<T, 32><<<blocks, 256, 0, s>>>(Xc, slots, a.C, HW, ctiles, ptiles,
                                                                copy_blocks, (const T *)W,
                                                                (uint16_t *)ws, a.oC, K);
            else
                deform_prep_kernel<T, 64><<<blocks, 256, 0, s>>>(Xc, slots, a.C, HW, ctiles, ptiles,
                                                                copy_blocks, (const T *)W,
                                                                (uint16_t *)ws, a.oC, K);
        } else {
            launch_copy_to_slots<uint16_t>((const uint16_t *)X + n0 * a.C * HW, slots, nc, a.C, HW,
                                           s);
        }
        const unsigned blocks = (unsigned)(nc * q.tiles);
        const T *Xs = (const T *)slots;
        if (q.kc == 64)
            deform_tc_nhwc_kernel<T, 64><<<blocks, kTcThreads, smem, s>>>(
                Xs, (const uint4 *)ws, (const T *)offset, (const T *)B, (const T *)mask, (T *)Y, a,
                q, (int)n0);
        else if (q.kc == 32)
            deform_tc_nhwc_kernel<T, 32><<<blocks, kTcThreads, smem, s>>>(
                Xs, (const uint4 *)ws, (const T *)offset, (const T *)B, (const T *)mask, (T *)Y, a,
                q, (int)n0);
        else
            deform_tc_nhwc_kernel<T, 16><<<blocks, kTcThreads, smem, s>>>(
                Xs, (const uint4 *)ws, (const T *)offset, (const T *)B, (const T *)mask, (T *)Y, a,
                q, (int)n0);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    *used = true;
    return cudaSuccess;
}

}  // namespace gs
