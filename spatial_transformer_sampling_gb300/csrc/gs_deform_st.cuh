// gs_deform_st.cuh -- DeformConv 2-D for fp16/bf16 on the tensor cores, with X
// staged in shared memory: persistent CTAs, one per SM.
//
// DeformConv (ai.onnx, since version 22), Inputs X, W, offset, B, mask:
//   Y[n, oc, p] = B[oc] + sum_{c, k} W[oc, c, k] * col[n, c, k, p],
//   col[n, c, k, p] = mask[n, k, p] * bilinear(X[n, c], p0(p) + k*dil + d(n, k, p)).
// As a GEMM: M = output positions (128 per tile), N = oC, and the K index runs
// over (k, c), kernel tap outer, channel inner, so that one 16-byte operand
// row holds 8 channels of one kernel tap: one bilinear sample of a channel-last
// pixel run.
//
// Per CTA (256 * G threads, G tap groups):
//  - W is copied once, with coalesced 16-byte loads from its (oc, c, k) order
//    into 8-row x 16-byte core matrices in (k, c) order (K-major, no
//    swizzle), and stays resident for all tiles.
//  - Tiles of 128 consecutive positions of one image are taken round robin;
//    a tile's offsets and mask arrive by cp.async one tile ahead.
//  - Thread (tap group grp, position pl, channel octet j) owns K / G kernel
//    taps of its position: it computes their bilinear taps once per tile (mask
//    folded into the weights) and keeps them in registers.
//  - Input channels are taken 16 at a time (a chunk).  For each chunk the X
//    window that the tile's taps can reach is staged in shared memory in
//    channel-last order (32 bytes per pixel), two stages deep: the loads for
//    the next chunk (or the next tile's first chunk) are issued before this
//    chunk's gather and stored after it.  A tap outside the window reads X
//    from global memory (rare: the window has margins of several pixels);
//    a tap outside the image reads a zero pixel.
//  - Per chunk and owned kernel tap, a thread reads four 16-byte runs, forms
//    eight column values and stores them as one A-operand row of one of two
//    A buffers; one thread then issues K MMAs (M = 128, N = oC, K = 16 each)
//    into the TMEM accumulator and commits them to that buffer's mbarrier, so
//    the next chunk's gather overlaps them.
//  - Epilogue per tile: tcgen05.ld, + B, round to T, store Y.
// Each column value is w0*x0 + w1*x1 + w2*x2 + w3*x3 in tap order (fmul, then
// fma, fma, fma; an out-of-image tap adds w * 0), rounded to T once;
// accumulation is fp32.
#pragma once

#include <type_traits>

#include "gs_common.cuh"
#include "gs_internal.h"
#include "gs_ptx.cuh"
#include "gs_tma.cuh"

namespace gs {

constexpr int kStM = 128;                 // positions per tile (TMEM lanes)
constexpr int kStKC = 16;                 // input channels per chunk
constexpr int kStWinPx = 1024;            // pixels of an X window (32 bytes each)
constexpr uint32_t kStStageBytes = (kStWinPx + 1) * 32;   // + one zero pixel
constexpr uint32_t kStZeroOff = kStWinPx * 32;            // the zero pixel's offset
constexpr int kStSmemLimit = 226 * 1024;  // dynamic; the static barriers take the rest

// Tap groups for K kernel taps (256 threads each): group grp owns kernel taps
// grp*TG .. min(K, (grp+1)*TG) - 1, TG = ceil(K / G).
__host__ __device__ constexpr int st_groups(int K) { return K == 9 ? 2 : (K % 3 == 0 ? 3 : (K % 2 == 0 ? 2 : 1)); }

struct DeformStParams {
    int tiles;          // tiles per image
    int total;          // N * tiles
    int rh, rw;         // window rows, columns (rw a multiple of 8, rh * rw <= kStWinPx)
    int my, mx;         // window margins around a tile's nominal footprint
    uint32_t w_bytes;   // oC * C * K * 2
    uint32_t a_bytes;   // one A buffer: 128 * 16 * K * 2
    uint32_t tap_bytes; // one tile's offsets (and mask): planes x 128 x 2
    uint32_t raw_bytes; // the TMA box of one chunk: 16 x rh x rw x 2, rounded up to 128
    uint32_t tmem_cols;
};

// Shared-memory slot of window pixel q: the low two bits are XORed with bits
// 3-4, so the four 8-pixel groups a warp stores at once use different banks.
__device__ __forceinline__ uint32_t st_slot(uint32_t q) { return q ^ ((q >> 3) & 3u); }

struct StWindow {
    int y0, x0;   // origin; the extent (rows, cols) is the same for every tile
};

// The X window of the tile starting at position p0: the tile's nominal
// footprint (all taps at zero offset, plus one row and column for the
// bilinear neighbour), widened by the margins, shifted into the image, x0
// rounded down to a multiple of 8 (16-byte loads).
__device__ __forceinline__ StWindow st_window(const DeformArgs &a, const DeformStParams &q, int p0) {
    const int P = a.oH * a.oW;
    const int pl = min(p0 + kStM - 1, P - 1);
    const int oha = p0 / a.oW, ohb = pl / a.oW;
    const int owa = oha == ohb ? p0 - oha * a.oW : 0;
    StWindow w;
    w.y0 = min(max(oha * a.sH - a.pad_t - q.my, 0), max(a.H - q.rh, 0));
    w.x0 = min(max(owa * a.sW - a.pad_l - q.mx, 0), max(a.W - q.rw, 0)) & ~7;
    return w;
}

// Window layout in shared memory: pixel q = row * rw + column holds 16
// channels in a 32-byte slot; slot(q) XORs the low two bits of q with bits
// 3-4, and the slot's two 16-byte halves (channels 0-7, 8-15) swap when bit 5
// of q is set.  Eight pixels that lie 8 apart in one row then cover all 32
// banks with one half each, and random pixels spread evenly.
__device__ __forceinline__ uint32_t st_half(uint32_t q, uint32_t half) {
    return st_slot(q) * 32 + ((half ^ ((q >> 5) & 1u)) << 4);
}

// 16 channels of the window: the raw stage that the TMA box fills,
// channel-first ([16][rh][rw] elements), -> the channel-last window.  Item i of
// a thread is one 8-column group of one row for a channel pair: two 16-byte
// loads (consecutive lanes take consecutive column groups of one plane, so a
// warp reads whole 128-byte lines) and eight 32-bit stores.  The window's
// extent is the same for every tile, so each item's offsets are computed once
// per CTA.
template <int NT, int ITEMS>
struct StTranspose {
    uint32_t src[ITEMS];   // byte offset of (channel 2cp, row, column 8g) in the raw stage; ~0: none
    uint32_t dst[ITEMS];   // pixel index q0 of the item's first column | channel pair << 24
    uint32_t plane;        // bytes of one channel plane of the raw stage

    // Thread t of the nthreads transposing threads (t < 0: none) takes items
    // t, t + nthreads, ...
    __device__ __forceinline__ void setup(int rows, int rw, int t, int nthreads) {
        const int gpr = rw >> 3;   // 8-column groups per row
        const int items = t < 0 ? 0 : rows * gpr * 8;
        plane = (uint32_t)(rows * rw * 2);
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            const int it = t + i * nthreads;
            const int g = it % gpr, rest = it / gpr;
            const int cp = rest & 7, r = rest >> 3;
            src[i] = t >= 0 && it < items ? (uint32_t)(2 * cp) * plane + (uint32_t)(r * rw + 8 * g) * 2
                                           : ~0u;
            dst[i] = (uint32_t)(r * rw + 8 * g) | ((uint32_t)cp << 24);
        }
    }

    __device__ __forceinline__ void run(const unsigned char *raw, unsigned char *stage) const {
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) {
            if (src[i] != ~0u) {
                const uint4 lo = *reinterpret_cast<const uint4 *>(raw + src[i]);
                const uint4 hi = *reinterpret_cast<const uint4 *>(raw + src[i] + plane);
                const uint32_t q0 = dst[i] & 0xFFFFFFu, cp = dst[i] >> 24;
                const uint32_t a4[4] = {lo.x, lo.y, lo.z, lo.w};
                const uint32_t b4[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const uint32_t word = __byte_perm(a4[e >> 1], b4[e >> 1], (e & 1) ? 0x7632 : 0x5410);
                    *reinterpret_cast<uint32_t *>(stage + st_half(q0 + e, cp >> 2) + (cp & 3) * 4) = word;
                }
            }
        }
    }
};

// Eight consecutive 16-bit values -> four fp32 pairs.
template <typename T> __device__ __forceinline__ void unpack8(const uint4 v, float2 (&x)[4]);
template <> __device__ __forceinline__ void unpack8<__nv_bfloat16>(const uint4 v, float2 (&x)[4]) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h)
        x[h] = make_float2(__uint_as_float(u[h] << 16), __uint_as_float(u[h] & 0xFFFF0000u));
}
template <> __device__ __forceinline__ void unpack8<__half>(const uint4 v, float2 (&x)[4]) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) x[h] = __half22float2(*reinterpret_cast<const __half2 *>(&u[h]));
}

template <typename T> __device__ __forceinline__ uint32_t st_pack2(float a, float b);
template <> __device__ __forceinline__ uint32_t st_pack2<__nv_bfloat16>(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <> __device__ __forceinline__ uint32_t st_pack2<__half>(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// The four bilinear taps of position (oh, ow) and kernel tap (kh, kw):
// image pixels and weights (mask folded in); tap t is (y0 + t/2, x0 + t%2).
// in[t] is false for a tap outside the image (weight 0).  Offsets of 1e8 or
// more (or NaN) give four zero taps.
__device__ __forceinline__ void st_taps(const DeformArgs &a, int oh, int ow, int kh, int kw,
                                        float dy, float dx, float m, int (&yy)[4], int (&xx)[4],
                                        float (&w)[4], bool (&in)[4]) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        yy[t] = 0;
        xx[t] = 0;
        w[t] = 0.0f;
        in[t] = false;
    }
    if (!(fabsf(dy) < 1.0e8f && fabsf(dx) < 1.0e8f)) return;
    const float fy = floorf(dy), fx = floorf(dx);
    const float ty = dy - fy, tx = dx - fx;
    const int y0 = oh * a.sH - a.pad_t + kh * a.dH + (int)fy;
    const int x0 = ow * a.sW - a.pad_l + kw * a.dW + (int)fx;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        yy[t] = y0 + (t >> 1);
        xx[t] = x0 + (t & 1);
        if (yy[t] >= 0 && yy[t] < a.H && xx[t] >= 0 && xx[t] < a.W) {
            in[t] = true;
            w[t] = ((t >> 1) ? ty : 1.0f - ty) * ((t & 1) ? tx : 1.0f - tx) * m;
        }
    }
}

// Eight channels of one pixel from global memory (NCHW), packed as in the
// shared-memory window: for taps that leave the window.
template <typename T>
__device__ __forceinline__ uint4 st_fetch8(const T *__restrict__ px, int HW) {
    uint16_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __ldg(reinterpret_cast<const uint16_t *>(px + (int64_t)e * HW));
    return make_uint4(v[0] | ((uint32_t)v[1] << 16), v[2] | ((uint32_t)v[3] << 16),
                      v[4] | ((uint32_t)v[5] << 16), v[6] | ((uint32_t)v[7] << 16));
}

// The four 16-byte runs of one owned kernel tap (packed window offsets).
__device__ __forceinline__ void st_load4(uint4 (&raw)[4], const unsigned char *xs,
                                         const uint32_t (&off)[2]) {
    raw[0] = *reinterpret_cast<const uint4 *>(xs + (off[0] & 0xFFFFu));
    raw[1] = *reinterpret_cast<const uint4 *>(xs + (off[0] >> 16));
    raw[2] = *reinterpret_cast<const uint4 *>(xs + (off[1] & 0xFFFFu));
    raw[3] = *reinterpret_cast<const uint4 *>(xs + (off[1] >> 16));
}

// One A row: eight column values w0*x0 + w1*x1 + w2*x2 + w3*x3 (fmul, then
// fma in tap order), rounded to T and stored as 16 bytes.
template <typename T>
__device__ __forceinline__ void st_row(unsigned char *dst, const uint4 (&raw)[4], const float (&w)[4]) {
    float2 acc[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        float2 x[4];
        unpack8<T>(raw[t], x);
        const float2 w2 = make_float2(w[t], w[t]);
#pragma unroll
        for (int h = 0; h < 4; ++h) acc[h] = t == 0 ? mul_f32x2(w2, x[h]) : fma_f32x2(w2, x[h], acc[h]);
    }
    *reinterpret_cast<uint4 *>(dst) =
        make_uint4(st_pack2<T>(acc[0].x, acc[0].y), st_pack2<T>(acc[1].x, acc[1].y),
                   st_pack2<T>(acc[2].x, acc[2].y), st_pack2<T>(acc[3].x, acc[3].y));
}

template <typename T, int K>
__global__ void __launch_bounds__(256 * st_groups(K), 1)
deform_st_kernel(const T *__restrict__ X, const T *__restrict__ Wt, const T *__restrict__ offset,
                 const T *__restrict__ Bias, const T *__restrict__ mask, T *__restrict__ Y,
                 const DeformArgs a, const DeformStParams q,
                 const __grid_constant__ CUtensorMap xmap) {
    constexpr int G = st_groups(K);
    constexpr int TG = (K + G - 1) / G;             // kernel taps per thread (at most)
    constexpr int NT = 256 * G;                     // threads
    // the window transpose runs on warps 1.., so that thread 0's MMA issue for
    // the previous chunk overlaps the other warps' share
    constexpr int ITEMS = (kStWinPx + NT - 33) / (NT - 32); // window transpose items per thread
    extern __shared__ __align__(128) unsigned char st_smem[];
    __shared__ __align__(8) uint64_t mma_done[2];
    __shared__ __align__(8) uint64_t raw_full;
    __shared__ uint32_t s_tmem;

    const int tid = threadIdx.x;
    const int C = a.C, oC = a.oC;
    const int P = a.oH * a.oW;
    const int HW = a.H * a.W;
    const int nch = C / kStKC;                       // chunks per tile
    const int planes = a.has_mask ? 3 * K : 2 * K;   // offset (2K) and mask (K) planes
    const int rows = q.rh, cols = q.rw;              // the window (inside the image)
    unsigned *err = a.err;

    // shared memory, from a 128-byte boundary (the launch adds 128 bytes of
    // slack): W | two A buffers | raw stage (TMA box) | window | taps | bias
    unsigned char *w_s = st_smem + ((128u - (smem_u32(st_smem) & 127u)) & 127u);
    unsigned char *a_s = w_s + q.w_bytes;
    unsigned char *raw_s = a_s + 2 * q.a_bytes;
    unsigned char *x_s = raw_s + q.raw_bytes;
    T *tap_s = reinterpret_cast<T *>(x_s + kStStageBytes);
    float *bias_s = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(tap_s) + q.tap_bytes);
    const uint32_t lbo_a = (kStM / 8) * 128;         // K-adjacent core matrices of A
    const uint32_t lbo_b = (uint32_t)oC * 16;        // K-adjacent core matrices of B
    const uint32_t raw_tx = (uint32_t)kStKC * rows * cols * 2;

    // the chunk of a tile: window origin and channel block, as TMA coordinates
    auto issue_raw = [&](int tile, int cb) {
        const int n = tile / q.tiles, p0 = (tile - n * q.tiles) * kStM;
        const StWindow w = st_window(a, q, p0);
        mbar_arrive_expect_tx(&raw_full, raw_tx);
        tma_load_4d(raw_s, &xmap, w.x0, w.y0, cb * kStKC, n, &raw_full);
    };
    // offsets and mask of a tile: planes x 128 positions, 16 bytes per cp.async
    // (spread over the threads; one committed group per tile)
    auto fetch_taps = [&](int tile) {
        const int n = tile / q.tiles, p0 = (tile - n * q.tiles) * kStM;
        for (int e = tid; e < planes * 16; e += NT) {
            const int pl = e >> 4, part = e & 15;
            const T *src = pl < 2 * K ? offset + ((int64_t)n * 2 * K + pl) * P
                                      : mask + ((int64_t)n * K + (pl - 2 * K)) * P;
            const int pbeg = p0 + part * 8;
            const int valid = min(max(P - pbeg, 0), 8);
            cp_async16(smem_u32(tap_s + pl * kStM + part * 8), src + (valid > 0 ? pbeg : 0),
                       (uint32_t)valid * 2);
        }
        cp_async_commit();
    };

    // start-up: the first chunk's window and the first tile's offsets are in
    // flight while W is repacked
    int tile_id = blockIdx.x;
    if (tid == 0) tma_prefetch_map(&xmap);
    if (tid == 0) {
        mbar_init(&mma_done[0], 1);
        mbar_init(&mma_done[1], 1);
        mbar_init(&raw_full, 1);
        fence_mbar_init();
    }
    __syncthreads();   // no thread waits on a barrier before it is initialised
    if (tid == 0 && tile_id < q.total) issue_raw(tile_id, 0);
    if (tile_id < q.total) fetch_taps(tile_id);
    // the last warp allocates the accumulator, off warp 0's start-up path
    if (tid >= NT - 32) {
        tmem_alloc(&s_tmem, q.tmem_cols);
        tcgen05_fence_before_sync();   // the address is read by others after a barrier
    }
    // W -> B operand in (k, c) order.  Item (oc, c8): W[oc, 8*c8 .. 8*c8+7, 0..K-1]
    // is 8K contiguous elements (16-byte aligned: C % 16 == 0) and holds, for
    // each kernel tap k, the 16-byte B row of K index k*C + 8*c8 .. +7 for oc,
    // stored at (k*C/8 + c8) * lbo_b + (oc / 8) * 128 + (oc % 8) * 16.  A warp's
    // 32 items share c8 and store 512 contiguous bytes per tap.
    for (int e = tid; e < oC * (C / 8); e += NT) {
        const int oc = e % oC, c8 = e / oC;
        const uint4 *src = reinterpret_cast<const uint4 *>(Wt + ((int64_t)oc * C + 8 * c8) * K);
        uint32_t u[4 * K];   // 8K elements, two per word
#pragma unroll
        for (int v = 0; v < K; ++v) {
            const uint4 x = __ldg(src + v);
            u[4 * v] = x.x;
            u[4 * v + 1] = x.y;
            u[4 * v + 2] = x.z;
            u[4 * v + 3] = x.w;
        }
        unsigned char *dst = w_s + (uint32_t)c8 * lbo_b + (oc >> 3) * 128 + (oc & 7) * 16;
#pragma unroll
        for (int k = 0; k < K; ++k) {
            uint32_t r[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                // channels 2h, 2h+1 of tap k: elements (2h)*K + k and (2h+1)*K + k
                const int e0 = 2 * h * K + k, e1 = e0 + K;
                const uint32_t lo = (e0 & 1) ? u[e0 >> 1] >> 16 : u[e0 >> 1] & 0xFFFFu;
                const uint32_t hi = (e1 & 1) ? u[e1 >> 1] & 0xFFFF0000u : u[e1 >> 1] << 16;
                r[h] = lo | hi;
            }
            *reinterpret_cast<uint4 *>(dst + (uint32_t)(k * C / 8) * lbo_b) =
                make_uint4(r[0], r[1], r[2], r[3]);
        }
    }
    if (tid < oC) bias_s[tid] = a.has_bias ? IO<T>::ld(Bias + tid) : 0.0f;
    if (tid < 2)   // the zero pixel
        *reinterpret_cast<uint4 *>(x_s + kStZeroOff + tid * 16) = make_uint4(0, 0, 0, 0);

    const int grp = tid >> 8, pl = (tid & 255) >> 1, j = tid & 1;
    const int k0 = grp * TG;                         // this thread's first kernel tap
    const int ntap = min(TG, K - k0);                // and how many it owns (warp-uniform)
    const uint32_t idesc = umma_idesc_f16(std::is_same<T, __nv_bfloat16>::value, kStM, oC);
    StTranspose<NT, ITEMS> tr;
    tr.setup(rows, cols, tid - 32, NT - 32);

    uint32_t g = 0;          // chunks done by this CTA (A buffer = g % 2, raw phase = g % 2)
    bool aborted = false;    // a bounded wait gave up (agreed on at a barrier)
    int prev_n = -1, prev_p0 = 0;   // the tile whose epilogue is still due
    uint32_t raw_issued = tile_id < q.total ? 1 : 0;   // TMA boxes thread 0 has issued

    // epilogue of tile (n, p0), once its last commit has arrived: warp w reads
    // TMEM lanes 32 * (w % 4) (positions) and half the columns, + B, rounds,
    // stores Y.  False if the wait gave up.
    auto epilogue = [&](int n, int p0) -> bool {
        const uint32_t last = g - 1;
        const bool bad = tid == 0 && !mbar_wait_bounded(&mma_done[last & 1], (last >> 1) & 1u, err);
        if (__syncthreads_or(bad)) return false;
        tcgen05_fence_after_sync();
        const int warp = tid >> 5, lane = tid & 31;
        if (warp < 8) {
            const int lq = warp & 3, half = warp >> 2;
            const int pe = p0 + lq * 32 + lane;
            const int ncol = oC / 2;
            for (int col0 = half * ncol; col0 < (half + 1) * ncol; col0 += 8) {
                float v[8];
                tmem_ld_x8(s_tmem + ((uint32_t)(lq * 32) << 16) + (uint32_t)col0, v);
                if (pe < P) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        Y[((int64_t)n * oC + col0 + i) * P + pe] = IO<T>::st(v[i] + bias_s[col0 + i]);
                }
            }
        }
        tcgen05_fence_before_sync();
        return true;
    };

    for (; tile_id < q.total; tile_id += gridDim.x) {
        const int n = tile_id / q.tiles, p0 = (tile_id - n * q.tiles) * kStM;
        const StWindow win = st_window(a, q, p0);
        cp_async_wait_pending(0);     // this tile's offsets and mask
        fence_proxy_async_smem();     // W (first tile) is read by the tensor cores
        __syncthreads();
        // taps of (pl, k) for this thread's kernel taps: window byte offsets of
        // this thread's channel half, and weights.  The window lies inside the
        // image, so a tap in it is in the image.
        const int p = p0 + pl;
        const bool live = p < P;
        const int oh = live ? p / a.oW : 0, ow = live ? p - (p / a.oW) * a.oW : 0;
        uint32_t off[TG][2];   // byte offsets of taps 2h, 2h+1: low, high half
        float wt[TG][4];
        uint32_t fb = 0;       // bit 4i+t: tap t of owned kernel tap i leaves the window
        // The two threads of a position (channel octets j = 0, 1; adjacent
        // lanes) need the same taps: each computes every other owned kernel
        // tap, for the slot's first half, and they swap results; the second
        // octet's offsets are the first's with the half bit flipped.
        constexpr int TP = (TG + 1) / 2;   // owned kernel taps computed per thread
#pragma unroll
        for (int s2 = 0; s2 < TP; ++s2) {
            const int i_mine = 2 * s2 + j;
            const int k = min(k0 + i_mine, K - 1);   // a tap past the group's end is never used
            const int kh = k / a.kW, kw = k - kh * a.kW;
            const float dy = IO<T>::to_float(tap_s[(2 * k) * kStM + pl]);
            const float dx = IO<T>::to_float(tap_s[(2 * k + 1) * kStM + pl]);
            const float m = a.has_mask ? IO<T>::to_float(tap_s[(2 * K + k) * kStM + pl]) : 1.0f;
            int yy[4], xx[4];
            float w[4];
            bool in[4];
            st_taps(a, oh, ow, kh, kw, dy, dx, m, yy, xx, w, in);
            uint32_t o[4];
            float wm[4];
            uint32_t bits = 0;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const bool ok = live && in[t];
                wm[t] = ok ? w[t] : 0.0f;
                const uint32_t ry = (uint32_t)(yy[t] - win.y0), rx = (uint32_t)(xx[t] - win.x0);
                if (ok && ry < (uint32_t)rows && rx < (uint32_t)cols) {
                    o[t] = st_half(ry * (uint32_t)cols + rx, 0u);
                } else {
                    o[t] = kStZeroOff;   // outside the image, or read again below
                    if (ok) bits |= 1u << t;
                }
            }
            const uint32_t m0 = o[0] | (o[1] << 16), m1 = o[2] | (o[3] << 16);
            // the partner's tap (index 2 s2 + 1 - j)
            const uint32_t p0 = __shfl_xor_sync(0xFFFFFFFFu, m0, 1);
            const uint32_t p1 = __shfl_xor_sync(0xFFFFFFFFu, m1, 1);
            const uint32_t pb = __shfl_xor_sync(0xFFFFFFFFu, bits, 1);
            float pw[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) pw[t] = __shfl_xor_sync(0xFFFFFFFFu, wm[t], 1);
            const int ia = 2 * s2, ib = 2 * s2 + 1;   // even and odd owned tap
            off[ia][0] = j ? p0 : m0;
            off[ia][1] = j ? p1 : m1;
            fb |= (j ? pb : bits) << (4 * ia);
#pragma unroll
            for (int t = 0; t < 4; ++t) wt[ia][t] = j ? pw[t] : wm[t];
            if (ib < TG) {
                off[ib][0] = j ? m0 : p0;
                off[ib][1] = j ? m1 : p1;
                fb |= (j ? bits : pb) << (4 * ib);
#pragma unroll
                for (int t = 0; t < 4; ++t) wt[ib][t] = j ? wm[t] : pw[t];
            }
        }
        // this thread's octet: the slot's second half for j = 1 (the zero
        // pixel's two halves are both zero)
        const uint32_t hmask = j ? 0x00100010u : 0u;
#pragma unroll
        for (int i = 0; i < TG; ++i) {
            off[i][0] ^= hmask;
            off[i][1] ^= hmask;
        }
        __syncthreads();   // every thread has read this tile's offsets
        const int next = tile_id + gridDim.x;
        if (next < q.total) fetch_taps(next);
        // owned kernel taps with a window-leaving tap anywhere in the warp
        uint32_t wfb = 0;
#pragma unroll
        for (int i = 0; i < TG; ++i)
            wfb |= __any_sync(0xFFFFFFFFu, ((fb >> (4 * i)) & 15u) != 0) ? 1u << i : 0u;
        // the previous tile's epilogue: its last MMAs ran during the tap setup
        if (prev_n >= 0 && !epilogue(prev_n, prev_p0)) {
            aborted = true;
            break;
        }
        prev_n = n;
        prev_p0 = p0;
        const T *Xn = X + (int64_t)n * C * HW;

        for (int cb = 0; cb < nch; ++cb, ++g) {
            const uint32_t buf = g & 1;
            // this chunk's raw stage -> window (the previous chunk's gather
            // finished at the last barrier)
            bool bad = !mbar_wait_bounded(&raw_full, g & 1u, err);
            if (!bad) tr.run(raw_s, x_s);
            if (__syncthreads_or(bad)) {
                aborted = true;
                break;
            }
            // the raw stage is free: the next chunk's box lands during this gather
            if (tid == 0) {
                if (cb + 1 < nch) {
                    issue_raw(tile_id, cb + 1);
                    ++raw_issued;
                } else if (next < q.total) {
                    issue_raw(next, 0);
                    ++raw_issued;
                }
            }
            unsigned char *arow = a_s + buf * q.a_bytes + (uint32_t)j * lbo_a + (pl >> 3) * 128 +
                                  (pl & 7) * 16;
            const unsigned char *xs = x_s;
            // main pass: taps that leave the window read the zero pixel here;
            // the next owned kernel tap's runs are loaded before this one's math
            uint4 raw[4];
            st_load4(raw, xs, off[0]);
#pragma unroll
            for (int i = 0; i < TG; ++i) {
                if (i >= ntap) break;
                uint4 nxt[4];
                if (i + 1 < TG && i + 1 < ntap) st_load4(nxt, xs, off[i + 1 < TG ? i + 1 : i]);
                st_row<T>(arow + (uint32_t)(2 * (k0 + i)) * lbo_a, raw, wt[i]);
                if (i + 1 < TG) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) raw[t] = nxt[t];
                }
            }
            // rows with taps outside the window, again with those taps read
            // from global memory (rare; warp-uniform branch)
            if (wfb) {
#pragma unroll
                for (int i = 0; i < TG; ++i) {
                    const uint32_t bits = (fb >> (4 * i)) & 15u;
                    if (i >= ntap || !((wfb >> i) & 1u) || !bits) continue;
                    uint4 r4[4];
                    st_load4(r4, xs, off[i]);
                    // the taps' top-left pixel, as st_taps finds it (the offsets
                    // are finite: the tap lies in the image)
                    const int k = k0 + i;
                    const float dy = IO<T>::ld(offset + ((int64_t)n * 2 * K + 2 * k) * P + p);
                    const float dx = IO<T>::ld(offset + ((int64_t)n * 2 * K + 2 * k + 1) * P + p);
                    const int y0 = oh * a.sH - a.pad_t + (k / a.kW) * a.dH + (int)floorf(dy);
                    const int x0 = ow * a.sW - a.pad_l + (k % a.kW) * a.dW + (int)floorf(dx);
                    const T *Xc = Xn + (int64_t)(cb * kStKC + j * 8) * HW;
#pragma unroll 1
                    for (int t = 0; t < 4; ++t) {
                        if ((bits >> t) & 1u) {
                            const uint4 v =
                                st_fetch8(Xc + (int64_t)(y0 + (t >> 1)) * a.W + x0 + (t & 1), HW);
                            r4[0] = t == 0 ? v : r4[0];
                            r4[1] = t == 1 ? v : r4[1];
                            r4[2] = t == 2 ? v : r4[2];
                            r4[3] = t == 3 ? v : r4[3];
                        }
                    }
                    st_row<T>(arow + (uint32_t)(2 * k) * lbo_a, r4, wt[i]);
                }
            }
            fence_proxy_async_smem();   // the column tile is read by the tensor cores
            // the next chunk writes the other A buffer, which the MMAs of chunk
            // g-1 read: one thread waits for them, the rest at the barrier
            bad = tid == 0 && g >= 1 && !mbar_wait_bounded(&mma_done[buf ^ 1u], ((g - 1) >> 1) & 1u, err);
            if (__syncthreads_or(bad)) {
                aborted = true;
                break;
            }
            if (tid == 0) {
                tcgen05_fence_after_sync();
                const uint32_t a_addr = smem_u32(a_s + buf * q.a_bytes);
                const uint32_t b_addr = smem_u32(w_s) + (uint32_t)(cb * 2) * lbo_b;
#pragma unroll
                for (int k = 0; k < K; ++k) {
                    // K step k: kernel tap k, the chunk's 16 channels
                    const uint64_t ad = umma_desc_kmajor(a_addr + 2 * k * lbo_a, lbo_a, 128);
                    const uint64_t bd =
                        umma_desc_kmajor(b_addr + (uint32_t)(k * C / 8) * lbo_b, lbo_b, 128);
                    umma_f16(s_tmem, ad, bd, idesc, (cb > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(&mma_done[buf]);
            }
        }
        if (aborted) break;
    }
    if (!aborted && prev_n >= 0 && !epilogue(prev_n, prev_p0)) aborted = true;
    cp_async_wait_pending(0);
    if (aborted && tid == 0) {
        // a wait gave up: give the copies and MMAs in flight a bounded chance
        // to finish before shared memory and the accumulator are released
        if (raw_issued > 0) mbar_wait_bounded(&raw_full, (raw_issued - 1) & 1u, nullptr);
        if (g > 0) mbar_wait_bounded(&mma_done[(g - 1) & 1], ((g - 1) >> 1) & 1u, nullptr);
    }
    tcgen05_fence_before_sync();
    __syncthreads();
    if (tid >= NT - 32) {   // the allocating warp releases it
        tcgen05_fence_after_sync();
        tmem_dealloc(s_tmem, q.tmem_cols);
    }
}

// Dynamic shared memory of the staged kernel: W, two A buffers, the raw TMA
// stage, the window, one tile's offsets and mask, B.
inline size_t deform_st_smem(const DeformArgs &a, const DeformStParams &q) {
    return (size_t)q.w_bytes + 2 * q.a_bytes + q.raw_bytes + kStStageBytes + q.tap_bytes +
           (size_t)a.oC * 4 + 128;
}

// Host: the parameters of the staged kernel for a shape, or false when it does
// not take the shape (then the other DeformConv kernels run).  It takes
// group = offset_group = 1, C % 16 == 0, 16 <= oC <= 256 with oC % 16 == 0,
// kH * kW in {1, 2, 3, 4, 6, 9}, W % 8 == 0, oH * oW % 8 == 0, 16-byte aligned
// X, W, offset and mask, shared memory within the limit, and a tile footprint
// that fits the X window with a margin of at least one pixel.
inline bool deform_st_params(const DeformArgs &a, const void *X, const void *W,
                             const void *offset, const void *mask, DeformStParams *q) {
    const int K = a.kH * a.kW;
    if (a.group != 1 || a.offset_group != 1) return false;
    if (a.C % kStKC != 0 || a.oC % 16 != 0 || a.oC < 16 || a.oC > 256) return false;
    if (!(K == 1 || K == 2 || K == 3 || K == 4 || K == 6 || K == 9)) return false;
    const int64_t P = (int64_t)a.oH * a.oW;
    if (a.W % 8 != 0 || P % 8 != 0) return false;
    for (const void *ptr : {X, W, offset, mask})
        if (ptr && ((uintptr_t)ptr & 15u)) return false;
    if ((int64_t)a.C * a.H * a.W >= ((int64_t)1 << 31)) return false;
    q->tiles = (int)((P + kStM - 1) / kStM);
    if ((int64_t)q->tiles * a.N >= ((int64_t)1 << 31)) return false;
    q->total = q->tiles * a.N;
    q->w_bytes = (uint32_t)a.oC * a.C * K * 2;
    q->a_bytes = (uint32_t)kStM * kStKC * K * 2;
    q->tap_bytes = (uint32_t)(a.has_mask ? 3 : 2) * K * kStM * 2;
    // nominal footprint of a tile (offsets 0): output rows and columns it spans
    const int64_t span_rows = (kStM % a.oW == 0) ? std::min<int64_t>(kStM / a.oW, a.oH)
                                                 : std::min<int64_t>((kStM - 1) / a.oW + 2, a.oH);
    const int64_t span_cols = span_rows > 1 ? a.oW : std::min<int64_t>(kStM, a.oW);
    const int64_t nr = (span_rows - 1) * a.sH + (int64_t)(a.kH - 1) * a.dH + 2;
    const int64_t nc = (span_cols - 1) * a.sW + (int64_t)(a.kW - 1) * a.dW + 2;
    for (int m = 8; m >= 1; --m) {
        const int64_t rh = std::min<int64_t>(a.H, nr + 2 * m);
        int64_t rw = (nc + 2 * m + 7 + 7) / 8 * 8;   // + up to 7 columns lost to the alignment
        if (span_rows > 1 || rw >= a.W) rw = a.W;
        if (rh * rw <= kStWinPx && rw <= 256 && rh <= 256) {
            q->rh = (int)rh;
            q->rw = (int)rw;
            q->raw_bytes = (uint32_t)((kStKC * rh * rw * 2 + 127) / 128 * 128);
            if (deform_st_smem(a, *q) > (size_t)kStSmemLimit) return false;
            q->my = m;
            q->mx = rw == a.W ? 0 : m;
            uint32_t cols = 32;
            while (cols < (uint32_t)a.oC) cols <<= 1;
            q->tmem_cols = cols;
            return true;
        }
    }
    return false;
}


template <typename T, int K>
cudaError_t launch_deform_st_k(const void *X, const void *W, const void *offset, const void *B,
                               const void *mask, void *Y, const DeformArgs &a,
                               const DeformStParams &q, const CUtensorMap &xmap, cudaStream_t s) {
    static DeviceFlags attr_set;
    cudaError_t e = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(deform_st_kernel<T, K>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kStSmemLimit);
    });
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = std::min(q.total, std::max(sms, 1));
    deform_st_kernel<T, K><<<grid, 256 * st_groups(K), deform_st_smem(a, q), s>>>(
        (const T *)X, (const T *)W, (const T *)offset, (const T *)B, (const T *)mask, (T *)Y, a, q,
        xmap);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_deform_staged(const void *X, const void *W, const void *offset, const void *B,
                                 const void *mask, void *Y, const DeformArgs &a, cudaStream_t s,
                                 bool *used) {
    *used = false;
    DeformStParams q;
    if (!deform_st_params(a, X, W, offset, mask, &q)) return cudaSuccess;
    // X as a 4-D tensor (W, H, C, N), innermost first; one box is a chunk's
    // window: rw columns x rh rows x 16 channels of one image
    CUtensorMap xmap;
    const uint64_t dims[4] = {(uint64_t)a.W, (uint64_t)a.H, (uint64_t)a.C, (uint64_t)a.N};
    const uint64_t strides[3] = {(uint64_t)a.W * 2, (uint64_t)a.H * a.W * 2,
                                 (uint64_t)a.C * a.H * a.W * 2};
    const uint32_t box[4] = {(uint32_t)q.rw, (uint32_t)q.rh, (uint32_t)kStKC, 1};
    if (!tmap_encode(&xmap, 2, std::is_same<T, __nv_bfloat16>::value, 4, X, dims, strides, box))
        return cudaSuccess;
    *used = true;
    switch (a.kH * a.kW) {
        case 1: return launch_deform_st_k<T, 1>(X, W, offset, B, mask, Y, a, q, xmap, s);
        case 2: return launch_deform_st_k<T, 2>(X, W, offset, B, mask, Y, a, q, xmap, s);
        case 3: return launch_deform_st_k<T, 3>(X, W, offset, B, mask, Y, a, q, xmap, s);
        case 4: return launch_deform_st_k<T, 4>(X, W, offset, B, mask, Y, a, q, xmap, s);
        case 6: return launch_deform_st_k<T, 6>(X, W, offset, B, mask, Y, a, q, xmap, s);
        default: return launch_deform_st_k<T, 9>(X, W, offset, B, mask, Y, a, q, xmap, s);
    }
}

}  // namespace gs
