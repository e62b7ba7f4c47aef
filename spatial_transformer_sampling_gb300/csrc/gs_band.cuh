// gs_band.cuh -- fused AffineGrid+GridSample, 2-D: the streamed band kernel.
//
// A block owns one image and a band of `th` consecutive output rows (full
// width).  Under an affine map the input rows a band reads form one
// contiguous range [r0, r0+rows) of every channel plane: the row position is
// affine in the output index, so its extremes over the band sit at the
// band's corners.  One elected thread streams that range channel by channel
// into a ring of shared-memory stages with bulk async copies (one contiguous
// cp.async.bulk per channel, completion counted on an mbarrier), and every
// thread interpolates its positions from shared memory.  DRAM sees long
// contiguous reads instead of short gathers, and the taps are plain
// shared-memory loads instead of multi-sector L1 requests.
//
// Taps are flattened once per position into byte offsets inside a stage plus
// combined weights.  Each stage ends with a 16-byte zero pad: a tap outside X
// (zeros padding) points at it, so it reads exactly 0 with no branch or
// select.  The ring is split into as many stages as the band's row range
// allows (up to 16).  A band whose rows do not fit two stages (strong
// zoom-out, large rotation, reflection of far-out positions) or whose map
// needs fp64 gathers from global memory instead, with the same taps.
//
// Warp 0 builds the map, finds the row range and issues the first stages
// before the block sets up its taps, so those reads overlap the setup.  A
// thread's outputs are paired on packed fp32 FMAs (see PAIRS below).
#pragma once

#include "gs_ptx.cuh"

namespace gs {

constexpr int kBandThreads = 256;
constexpr int kBandPPT = 4;          // output positions per thread: th * Wo <= 1024
constexpr int kBandMaxStages = 16;
constexpr int kBandMinStages = 2;
constexpr int kBandZeroPad = 16;     // bytes of zeros after each stage's rows

// Blocks per SM and shared-memory ring per block.  Linear and nearest on
// 16-bit types: 4 blocks of 48 KB (a 64-register budget, which their taps
// fit).  On fp32 a stage is twice as large, so the same ring holds half as
// many channels in flight; 3 blocks of 72 KB keep more of them in flight and
// measure faster (stn2d fp32: 53.9 -> 52.1 us), while 16-bit types lose more
// to the lower occupancy than they gain.  Cubic's 16 taps per position need
// more registers: one block per SM.
template <typename T, int MODE> struct BandCfg {
    static constexpr int min_blocks = sizeof(T) == 4 ? 3 : 4;
    static constexpr int ring = sizeof(T) == 4 ? 72 * 1024 : 48 * 1024;
};
template <typename T> struct BandCfg<T, MODE_CUBIC> {
    static constexpr int min_blocks = 1;
    static constexpr int ring = 48 * 1024;
};

struct BandParams {
    int th;            // output rows per band
    int bands;         // bands per image
    int ring_bytes;    // shared-memory ring, split into stages per band
};

// Two adjacent outputs from an fp32 pair, each rounded to nearest even as
// IO<T>::st rounds it, in one store (p is aligned to two elements).
template <typename T> __device__ __forceinline__ void st_pair(T *p, float2 v);
template <> __device__ __forceinline__ void st_pair<float>(float *p, float2 v) {
    *reinterpret_cast<float2 *>(p) = v;
}
template <> __device__ __forceinline__ void st_pair<__half>(__half *p, float2 v) {
    *reinterpret_cast<__half2 *>(p) = __floats2half2_rn(v.x, v.y);
}
template <> __device__ __forceinline__ void st_pair<__nv_bfloat16>(__nv_bfloat16 *p, float2 v) {
    *reinterpret_cast<__nv_bfloat162 *>(p) = __floats2bfloat162_rn(v.x, v.y);
}

// PAIRS: how a thread's outputs share packed fp32 FMAs (fma.rn.f32x2; each
// lane rounds exactly as fmaf does).
//   kPairNone     outputs t, t+256, t+512, t+768, one FMA per tap each;
//   kPairAdjacent outputs 2t, 2t+1, 2t+512, 2t+513: a pair shares one FMA per
//                 tap, one conversion and one store (16-bit types; needs an
//                 even output width and Y aligned to two elements; for fp32
//                 the lanes' 8-byte-apart loads would conflict in the banks);
//   kPairStrided  outputs t, t+256, ...: t and t+256 share one FMA per tap,
//                 stored apart (fp32).
enum { kPairNone = 0, kPairAdjacent = 1, kPairStrided = 2 };

template <typename T, int MODE, int PAIRS>
__global__ void __launch_bounds__(kBandThreads, BandCfg<T, MODE>::min_blocks)
band_kernel(const T *__restrict__ X, const T *__restrict__ theta, T *__restrict__ Y,
            const SampleParams P, const BandParams B) {
    constexpr int K = TapCount<MODE>::K;
    constexpr int NT = K * K;
    extern __shared__ __align__(128) unsigned char band_smem[];
    __shared__ __align__(8) uint64_t full[kBandMaxStages];
    __shared__ AffineMap s_map;
    __shared__ int s_r0, s_rows, s_stages, s_abort;

    const SampleArgs &a = P.a;
    const int n = blockIdx.x / B.bands;
    const int band = blockIdx.x - n * B.bands;
    const int Ho = a.out[0], Wo = a.out[1], Hi = a.in[0], Wi = a.in[1];
    const int h0 = band * B.th;
    const int hn = min(B.th, Ho - h0);
    const int npos = hn * Wo;
    const int tid = threadIdx.x;

    const T *Xn = X + (int64_t)n * a.C * a.in_plane;
    if (tid < 32) {
        // warp 0: the affine map, the band's input row range, the ring's
        // split, and the first copies -- issued before the taps are set up,
        // so the reads overlap that work
        build_affine_map_warp<T, 2>(theta + (int64_t)n * 6, P, s_map);
        __syncwarp();
        const bool wide = s_map.wide;
        // input row of the band's four corners, one lane each
        int64_t y = 0;
        if (tid < 4 && !wide) {
            const int h = (tid & 1) ? h0 + hn - 1 : h0;
            const int w = (tid & 2) ? Wo - 1 : 0;
            y = (s_map.cst_q[0] + s_map.coef_q[0][0] * h + s_map.coef_q[0][1] * w) >> 8;
        }
        int64_t ymin = tid < 4 ? y : INT64_MAX, ymax = tid < 4 ? y : INT64_MIN;
#pragma unroll
        for (int o = 1; o < 4; o <<= 1) {
            const int64_t a0 = __shfl_xor_sync(0xffffffffu, ymin, o);
            const int64_t a1 = __shfl_xor_sync(0xffffffffu, ymax, o);
            ymin = a0 < ymin ? a0 : ymin;
            ymax = a1 > ymax ? a1 : ymax;
        }
        if (tid == 0) {
            for (int s = 0; s < kBandMaxStages; ++s) mbar_init(&full[s], 1);
            fence_mbar_init();
            int stages = 0, lo = 0, hi = 0;
            if (!wide) {
                if (MODE != MODE_CUBIC && a.pad == PAD_BORDER) {
                    // linear/nearest clamp the coordinate before taking taps: a
                    // clamped position keeps its (zero-weight) second tap
                    ymin = clamp_q(ymin, 0, P.ax[0].hi_q);
                    ymax = clamp_q(ymax, 0, P.ax[0].hi_q);
                }
                lo = (int)(ymin >> 32) - (MODE == MODE_CUBIC ? 1 : 0);
                hi = (int)(ymax >> 32) + (MODE == MODE_CUBIC ? 2 : 1);
                if (a.pad == PAD_REFLECTION && (lo < 0 || hi > Hi - 1)) {
                    lo = 0;   // folded positions can land anywhere: take the plane
                    hi = Hi - 1;
                }
                // Border padding moves taps onto rows 0 and Hi-1, zeros padding
                // masks taps outside; either way clamping both ends into range
                // keeps every row a tap reads.
                lo = min(max(lo, 0), Hi - 1);
                hi = min(max(hi, 0), Hi - 1);
                const int64_t stage =
                    (int64_t)(hi - lo + 1) * Wi * (int64_t)sizeof(T) + kBandZeroPad;
                stages = (int)min((int64_t)kBandMaxStages, (int64_t)B.ring_bytes / stage);
                if (stages < kBandMinStages) stages = 0;
            }
            s_r0 = lo;
            s_rows = hi - lo + 1;
            s_stages = stages;
            s_abort = 0;
            if (stages) {
                const uint32_t bytes = (uint32_t)(hi - lo + 1) * (uint32_t)Wi * (uint32_t)sizeof(T);
                const T *Xr = Xn + (int64_t)lo * Wi;
                for (int st = 0; st < stages && st < a.C; ++st) {
                    mbar_arrive_expect_tx(&full[st], bytes);
                    bulk_copy_g2s(band_smem + (size_t)st * (bytes + kBandZeroPad),
                                  Xr + (int64_t)st * a.in_plane, bytes, &full[st]);
                }
            }
        }
    }
    __syncthreads();
    const int S = s_stages;   // 0: gather from global
    const int r0 = s_r0, rows = s_rows;
    const uint32_t data_bytes = (uint32_t)rows * (uint32_t)Wi * (uint32_t)sizeof(T);
    const uint32_t stage_bytes = data_bytes + kBandZeroPad;
    if (S) {
        // zero pads (generic writes; the copies never touch them), made
        // visible by the barrier after the taps
        for (int e = tid; e < S * (kBandZeroPad / 4); e += kBandThreads) {
            const int st = e / (kBandZeroPad / 4), k = e - st * (kBandZeroPad / 4);
            *reinterpret_cast<uint32_t *>(band_smem + (size_t)st * stage_bytes + data_bytes + 4 * k) =
                0u;
        }
    }

    // flattened taps of this thread's positions (each channel's stores are
    // whole lines per warp).  Consecutive positions of a thread are a fixed
    // distance apart (kBandThreads; for adjacent pairs alternately 1 and
    // 2*kBandThreads-1): the output index advances by (dh, dw) with a carry
    // into the row, and the 24.40 coordinates by the matching constants.
    uint32_t off[kBandPPT][NT];
    float wt[kBandPPT][NT];
    uint32_t okm[kBandPPT];
    // position of this thread's j-th output within the band
    constexpr bool kAdj = PAIRS == kPairAdjacent;
    auto pos_of = [&](int j) {
        return kAdj ? 2 * tid + (j & 1) + (j >> 1) * (2 * kBandThreads) : tid + j * kBandThreads;
    };
    constexpr int kStepA = kAdj ? 1 : kBandThreads;                      // after even j
    constexpr int kStepB = kAdj ? 2 * kBandThreads - 1 : kBandThreads;   // after odd j
    const int dhA = kStepA / Wo, dwA = kStepA - (kStepA / Wo) * Wo;
    const int dhB = kStepB / Wo, dwB = kStepB - (kStepB / Wo) * Wo;
    const int p0 = pos_of(0);
    int h = h0 + p0 / Wo, w = p0 - (p0 / Wo) * Wo;
    const bool wide = s_map.wide;
    int64_t yacc = 0, xacc = 0, ystepA = 0, xstepA = 0, ystepB = 0, xstepB = 0, ywrap = 0,
            xwrap = 0;
    if (!wide) {
        yacc = s_map.cst_q[0] + s_map.coef_q[0][0] * h + s_map.coef_q[0][1] * w;
        xacc = s_map.cst_q[1] + s_map.coef_q[1][0] * h + s_map.coef_q[1][1] * w;
        ystepA = s_map.coef_q[0][0] * dhA + s_map.coef_q[0][1] * dwA;
        xstepA = s_map.coef_q[1][0] * dhA + s_map.coef_q[1][1] * dwA;
        ystepB = s_map.coef_q[0][0] * dhB + s_map.coef_q[0][1] * dwB;
        xstepB = s_map.coef_q[1][0] * dhB + s_map.coef_q[1][1] * dwB;
        ywrap = s_map.coef_q[0][0] - s_map.coef_q[0][1] * Wo;
        xwrap = s_map.coef_q[1][0] - s_map.coef_q[1][1] * Wo;
    }
#pragma unroll
    for (int j = 0; j < kBandPPT; ++j) {
        const int p = pos_of(j);
        int64_t yq, xq;
        if (!wide) {
            yq = yacc >> 8;   // 24.40 -> 32.32 (floor)
            xq = xacc >> 8;
        } else {
            const int hh = p < npos ? h : h0, ww = p < npos ? w : 0;
            yq = pos_to_q(s_map.cst[0] + s_map.coef[0][0] * hh + s_map.coef[0][1] * ww, P.ax[0], a.pad);
            xq = pos_to_q(s_map.cst[1] + s_map.coef[1][0] * hh + s_map.coef[1][1] * ww, P.ax[1], a.pad);
        }
        // next position
        const bool stepA = (j & 1) == 0;
        h += stepA ? dhA : dhB;
        w += stepA ? dwA : dwB;
        yacc += stepA ? ystepA : ystepB;
        xacc += stepA ? xstepA : xstepB;
        if (w >= Wo) {
            w -= Wo;
            h += 1;
            yacc += ywrap;
            xacc += xwrap;
        }
        AxisTaps<MODE> ty, tx;
        make_taps<MODE>(yq, P.ax[0], a.pad, a.ac, a.a, ty);
        make_taps<MODE>(xq, P.ax[1], a.pad, a.ac, a.a, tx);
        okm[j] = 0;
#pragma unroll
        for (int ky = 0; ky < K; ++ky) {
#pragma unroll
            for (int kx = 0; kx < K; ++kx) {
                const int t = ky * K + kx;
                const bool ok = ((ty.ok >> ky) & (tx.ok >> kx) & 1u) != 0;
                wt[j][t] = ty.w[ky] * tx.w[kx];
                okm[j] |= (ok ? 1u : 0u) << t;
                if (S) {
                    // slab rows are clamped into the loaded range, so a read
                    // can never leave the stage
                    const int row = min(max(ty.idx[ky] - r0, 0), rows - 1);
                    off[j][t] = ok ? (uint32_t)(row * Wi + tx.idx[kx]) * (uint32_t)sizeof(T)
                                   : data_bytes;   // the zero pad
                } else {
                    off[j][t] = (uint32_t)(ty.idx[ky] * Wi + tx.idx[kx]) * (uint32_t)sizeof(T);
                }
            }
        }
    }

    T *__restrict__ Yn = Y + (int64_t)n * a.C * a.out_plane + (int64_t)h0 * Wo;
    if (S == 0) {
        const unsigned char *Xb = reinterpret_cast<const unsigned char *>(Xn);
        const int64_t in_bytes = a.in_plane * (int64_t)sizeof(T);
        for (int c = 0; c < a.C; ++c) {
#pragma unroll
            for (int j = 0; j < kBandPPT; ++j) {
                const int p = pos_of(j);
                if (p >= npos) continue;
                float acc = 0.0f;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    const float v = ((okm[j] >> t) & 1u)
                        ? IO<T>::ld(reinterpret_cast<const T *>(Xb + off[j][t])) : 0.0f;
                    acc = fmaf(wt[j][t], v, acc);
                }
                Yn[p] = IO<T>::st(acc);
            }
            Xb += in_bytes;
            Yn += a.out_plane;
        }
        return;
    }

    // One channel from the stage at `base`: every position of this thread
    // (full: the band is whole, no bounds checks).
    auto channel_out = [&](uint32_t base, T *__restrict__ Yc, bool full) {
        if constexpr (PAIRS != kPairNone) {
#pragma unroll
            for (int jp = 0; jp < kBandPPT / 2; ++jp) {
                const int j0 = 2 * jp, j1 = 2 * jp + 1;
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int t = 0; t < NT; ++t)
                    acc = fma_f32x2(make_float2(wt[j0][t], wt[j1][t]),
                                    make_float2(lds_at<T>(base + off[j0][t]),
                                                lds_at<T>(base + off[j1][t])),
                                    acc);
                if constexpr (kAdj) {
                    if (full || pos_of(j0) < npos) st_pair<T>(Yc + pos_of(j0), acc);
                } else {
                    if (full || pos_of(j0) < npos) Yc[pos_of(j0)] = IO<T>::st(acc.x);
                    if (full || pos_of(j1) < npos) Yc[pos_of(j1)] = IO<T>::st(acc.y);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < kBandPPT; ++j) {
                float acc = 0.0f;
#pragma unroll
                for (int t = 0; t < NT; ++t) acc = fmaf(wt[j][t], lds_at<T>(base + off[j][t]), acc);
                if (full || pos_of(j) < npos) Yc[pos_of(j)] = IO<T>::st(acc);
            }
        }
    };

    __syncthreads();   // zero pads written
    const T *Xr = Xn + (int64_t)r0 * Wi;
    const uint32_t ring = smem_u32(band_smem);
    int c = 0;
    int s = 0;
    uint32_t parity = 0;
    if (npos == kBandThreads * kBandPPT && S >= 4) {
        // Full band, deep ring: two channels per pair of barriers, and no
        // per-position bounds checks.
        for (; c + 1 < a.C; c += 2) {
            int s2 = s + 1;
            uint32_t p2 = parity;
            if (s2 == S) {
                s2 = 0;
                p2 ^= 1u;
            }
            if (!mbar_wait_bounded(&full[s], parity, a.err)) s_abort = 1;
            if (!mbar_wait_bounded(&full[s2], p2, a.err)) s_abort = 1;
            __syncthreads();   // every thread has waited (or given up) on both stages
            if (s_abort) break;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint32_t base = ring + (uint32_t)(k ? s2 : s) * stage_bytes;
                channel_out(base, Yn, true);
                Yn += a.out_plane;
            }
            __syncthreads();   // both stages fully read
            if (tid == 0) {
                fence_proxy_async_smem();
                if (c + S < a.C) {
                    mbar_arrive_expect_tx(&full[s], data_bytes);
                    bulk_copy_g2s(band_smem + (size_t)s * stage_bytes,
                                  Xr + (int64_t)(c + S) * a.in_plane, data_bytes, &full[s]);
                }
                if (c + 1 + S < a.C) {
                    mbar_arrive_expect_tx(&full[s2], data_bytes);
                    bulk_copy_g2s(band_smem + (size_t)s2 * stage_bytes,
                                  Xr + (int64_t)(c + 1 + S) * a.in_plane, data_bytes, &full[s2]);
                }
            }
            s = s2 + 1;
            parity = p2;
            if (s == S) {
                s = 0;
                parity ^= 1u;
            }
        }
    }
    for (; c < a.C && !s_abort; ++c) {
        if (!mbar_wait_bounded(&full[s], parity, a.err)) s_abort = 1;
        __syncthreads();   // every thread has waited (or given up) on stage s
        if (s_abort) break;
        const uint32_t base = ring + (uint32_t)s * stage_bytes;
        channel_out(base, Yn, false);
        Yn += a.out_plane;
        __syncthreads();   // stage s fully read
        if (tid == 0 && c + S < a.C) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&full[s], data_bytes);
            bulk_copy_g2s(band_smem + (size_t)s * stage_bytes, Xr + (int64_t)(c + S) * a.in_plane,
                          data_bytes, &full[s]);
        }
        if (++s == S) {
            s = 0;
            parity ^= 1u;
        }
    }
    if (c < a.C && tid == 0) {
        // a wait gave up: let the copies still in flight land before the
        // block's shared memory is released (bounded again)
        for (int cc = c; cc < a.C && cc < c + S; ++cc)
            mbar_wait_bounded(&full[cc % S], (uint32_t)(cc / S) & 1u, nullptr);
    }
}

// Host side: use the band kernel when rows can be bulk-copied (16-byte
// multiples and alignment) and a band of whole output rows fits 1024
// positions; *used tells the caller whether it ran.
template <typename T, int MODE>
cudaError_t launch_band(const void *X, const void *theta, void *Y, const SampleParams &P,
                        cudaStream_t s, bool *used) {
    *used = false;
    const SampleArgs &a = P.a;
    const int Wi = a.in[1], Wo = a.out[1];
    const size_t row_bytes = (size_t)Wi * sizeof(T);
    if (row_bytes % 16 != 0 || (uintptr_t)X % 16 != 0) return cudaSuccess;
    if (Wo > kBandThreads * kBandPPT) return cudaSuccess;
    constexpr int kRingBytes = BandCfg<T, MODE>::ring;
    if ((size_t)kRingBytes < (size_t)kBandMinStages * (4 * row_bytes + kBandZeroPad))
        return cudaSuccess;                 // rows too wide to stage usefully
    BandParams B;
    B.th = min(a.out[0], (kBandThreads * kBandPPT) / Wo);
    B.bands = (a.out[0] + B.th - 1) / B.th;
    B.ring_bytes = kRingBytes;
    // packed FMAs for linear and nearest: fp32 pairs outputs t and t+256;
    // 16-bit types pair adjacent outputs when the width is even and Y is
    // aligned to a pair
    constexpr int kPairs = MODE == MODE_CUBIC ? kPairNone
                           : (sizeof(T) == 4 ? kPairStrided : kPairAdjacent);
    const bool pairs = kPairs == kPairStrided ||
                       (kPairs == kPairAdjacent && Wo % 2 == 0 &&
                        (uintptr_t)Y % (2 * sizeof(T)) == 0);
    auto kern = pairs ? band_kernel<T, MODE, kPairs> : band_kernel<T, MODE, kPairNone>;
    static DeviceFlags attr_set[2];
    const cudaError_t e = once_per_device(attr_set[pairs], [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    });
    if (e != cudaSuccess) return e;
    const unsigned blocks = (unsigned)((int64_t)a.N * B.bands);
    kern<<<blocks, kBandThreads, kRingBytes, s>>>((const T *)X, (const T *)theta, (T *)Y, P, B);
    *used = true;
    return cudaGetLastError();
}

}  // namespace gs
