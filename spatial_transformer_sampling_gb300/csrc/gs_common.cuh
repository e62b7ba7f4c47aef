// gs_common.cuh -- device helpers shared by the libgs kernels: typed I/O, the
// exact fixed-point coordinate pipeline, padding, and per-axis taps/weights.
//
// Coordinates.  GridSample's unnormalised position is x = g*h + c with
// h = n/2 (align_corners=0) or (n-1)/2 (align_corners=1) and c = (n-1)/2
// (GridSample - version 20, Attributes, align_corners).  Forming x in fp32
// would round it at the ulp of ~n (1.5e-5 px at n = 256), which alone breaks a
// 1e-6 tolerance on N(0,1) data.  Instead the product g*h is split exactly
// into p + e (fp32 product plus its FMA-computed rounding error), and p, e and
// c are summed in signed 32.32 fixed point.  Every padding rule then runs on
// integers, exactly, and only the final fraction t in [0,1) is rounded to fp32.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gs {

enum { MODE_LINEAR = 0, MODE_NEAREST = 1, MODE_CUBIC = 2 };
enum { PAD_ZEROS = 0, PAD_BORDER = 1, PAD_REFLECTION = 2 };

constexpr int kMaxRank = 3;
constexpr int64_t kOneQ = int64_t(1) << 32;    // 1.0 in 32.32
constexpr int64_t kHalfQ = int64_t(1) << 31;   // 0.5 in 32.32
constexpr float kFarOut = 4194304.0f;          // 2^22 px: beyond every valid extent

// ---------------------------------------------------------------- typed I/O

template <typename T> struct IO;
template <> struct IO<float> {
    static __device__ __forceinline__ float ld(const float *p) { return __ldg(p); }
    static __device__ __forceinline__ float st(float v) { return v; }
    static __host__ __device__ __forceinline__ double to_double(float v) { return v; }
    static __device__ __forceinline__ float to_f(float v) { return v; }
};
template <> struct IO<__half> {
    static __device__ __forceinline__ float ld(const __half *p) { return __half2float(__ldg(p)); }
    static __device__ __forceinline__ __half st(float v) { return __float2half_rn(v); }
    static __device__ __forceinline__ double to_double(__half v) { return __half2float(v); }
    static __device__ __forceinline__ float to_float(__half v) { return __half2float(v); }
    static __device__ __forceinline__ float to_f(__half v) { return __half2float(v); }
};
template <> struct IO<__nv_bfloat16> {
    static __device__ __forceinline__ float ld(const __nv_bfloat16 *p) {
        return __bfloat162float(__ldg(p));
    }
    static __device__ __forceinline__ __nv_bfloat16 st(float v) { return __float2bfloat16_rn(v); }
    static __device__ __forceinline__ double to_double(__nv_bfloat16 v) {
        return __bfloat162float(v);
    }
    static __device__ __forceinline__ float to_float(__nv_bfloat16 v) { return __bfloat162float(v); }
    static __device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
};

// Integer X (GridSample - version 20, Outputs: for integer input types the
// intermediate values are floating point, cast to the integer type at the
// end).  The cast truncates toward zero and saturates at the type's range
// (cubic weights can overshoot it); NaN reads as 0.
template <typename I, int LO, int HI> struct IntIO {
    static __device__ __forceinline__ float ld(const I *p) { return (float)__ldg(p); }
    static __device__ __forceinline__ I st(float v) {
        v = fminf(fmaxf(v, (float)LO), (float)HI);   // fmaxf(NaN, LO) is LO
        return (I)(int)v;                             // truncation toward zero
    }
};
template <> struct IO<uint8_t> : IntIO<uint8_t, 0, 255> {};
template <> struct IO<int8_t> : IntIO<int8_t, -128, 127> {};
template <> struct IO<uint16_t> : IntIO<uint16_t, 0, 65535> {};
template <> struct IO<int16_t> : IntIO<int16_t, -32768, 32767> {};

// Shared-memory load at a 32-bit shared address (volatile: never moved across
// the stage waits and barriers).
template <typename T> __device__ __forceinline__ float lds_at(uint32_t addr);
template <> __device__ __forceinline__ float lds_at<float>(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
template <> __device__ __forceinline__ float lds_at<__half>(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return __half2float(__ushort_as_half(v));
}
template <> __device__ __forceinline__ float lds_at<__nv_bfloat16>(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return __uint_as_float((uint32_t)v << 16);
}

// ------------------------------------------------------------- axis params

// One input spatial axis, precomputed on the host.
struct Axis {
    int n;            // input extent along the axis
    float h;          // grid scale: n/2 (align_corners=0) or (n-1)/2 (align_corners=1)
    float period_f;   // reflection period 2*span (exact in fp32); 0 when span == 0
    int pad_;         // keeps the int64 fields 8-byte aligned
    int64_t c_q;      // (n-1)/2 in 32.32
    int64_t lo_q;     // reflection border: -0.5 (align_corners=0) or 0 (1), 32.32
    int64_t span_q;   // distance between the reflection borders: n or n-1, 32.32
    int64_t hi_q;     // n-1 in 32.32, the clip bound
};

// Grid value -> 32.32 position.  Exact except when |g*h| < 2^-9, where the
// last bits fall below 2^-32 px.  Values so far out that no tap can land in
// range are pinned at +-2^22 px (zeros, border); under reflection they are
// first reduced by the fold's period, which leaves the folded result as is.
__device__ __forceinline__ int64_t grid_to_q(float g, const Axis &A, int pad) {
    float p = g * A.h;
    float e = fmaf(g, A.h, -p);   // g*h == p + e exactly
    if (!(fabsf(p) < kFarOut)) {  // also NaN
        if (pad == PAD_REFLECTION && A.period_f > 0.0f && isfinite(p)) {
            p = fmodf(p, A.period_f);   // fmodf is exact
            e = fmodf(e, A.period_f);
        } else {
            p = (p > 0.0f) ? kFarOut : -kFarOut;
            e = 0.0f;
        }
    }
    return __float2ll_rn(p * 4294967296.0f) + __float2ll_rn(e * 4294967296.0f) + A.c_q;
}

// fp64 position -> 32.32 (used only for affine maps too wide for the integer
// path, i.e. with positions beyond 2^22 px).
__device__ __forceinline__ int64_t pos_to_q(double x, const Axis &A, int pad) {
    if (!(fabs(x) < (double)kFarOut)) {
        if (pad == PAD_REFLECTION && A.period_f > 0.0f && isfinite(x)) {
            double lo = (double)A.lo_q * (1.0 / 4294967296.0);
            x = lo + fmod(x - lo, (double)A.period_f);
        } else {
            x = (x > 0.0) ? (double)kFarOut : -(double)kFarOut;
        }
    }
    return __double2ll_rn(x * 4294967296.0);
}

// Element i of a grid of float type dt (0 fp32, 1 fp16, 2 bf16), widened to fp32.
__device__ __forceinline__ float grid_value(const void *grid, int dt, int64_t i) {
    if (dt == 0) return __ldg(reinterpret_cast<const float *>(grid) + i);
    if (dt == 1) return __half2float(__ldg(reinterpret_cast<const __half *>(grid) + i));
    return __bfloat162float(__ldg(reinterpret_cast<const __nv_bfloat16 *>(grid) + i));
}

__device__ __forceinline__ int64_t clamp_q(int64_t x, int64_t lo, int64_t hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

// Reflection of a 32.32 position: mirror at lo and lo+span until inside
// (GridSample padding_mode=reflection).  The fold is periodic with period
// 2*span, so one remainder finds the position inside the period.
__device__ __forceinline__ int64_t reflect_q(int64_t x, int64_t lo, int64_t span) {
    if (span == 0) return lo;
    const int64_t period = 2 * span;
    int64_t d = x - lo;
    if (d < 0 || d >= period) {
        d %= period;
        if (d < 0) d += period;
    }
    if (d > span) d = period - d;
    return lo + d;
}

// Reflection of an integer tap index.  align_corners=1 mirrors at the centres
// of pixels 0 and n-1 (index -1 reads index 1); align_corners=0 mirrors at the
// outer edges (index -1 reads index 0, index n reads n-1).
__device__ __forceinline__ int reflect_index(int j, int n, int ac) {
    if (ac) {
        if (n == 1) return 0;
        const int period = 2 * (n - 1);
        int m = j % period;
        if (m < 0) m += period;
        return m <= n - 1 ? m : period - m;
    }
    const int period = 2 * n;
    int m = j % period;
    if (m < 0) m += period;
    return m < n ? m : period - 1 - m;
}

// ------------------------------------------------------------------- taps

template <int MODE> struct TapCount { static constexpr int K = 2; };
template <> struct TapCount<MODE_NEAREST> { static constexpr int K = 1; };
template <> struct TapCount<MODE_CUBIC> { static constexpr int K = 4; };

// Taps of one axis: indices (clamped into range whenever `ok` is clear, so an
// address formed from them is always inside X), 1-D weights, validity bits.
template <int MODE> struct AxisTaps {
    static constexpr int K = TapCount<MODE>::K;
    int idx[K];
    float w[K];
    unsigned ok;   // bit k set: tap k reads X; clear: tap k reads 0
};

// Keys' cubic convolution weights for the four taps floor(x)-1 .. floor(x)+2
// at fraction t (distances t+1, t, 1-t, 2-t).  On 1 <= s <= 2 the kernel
// a*s^3 - 5a*s^2 + 8a*s - 4a factors as a*(s-1)*(s-2)^2, which at s = 1+t and
// s = 2-t gives the short, well-conditioned forms below.
__device__ __forceinline__ void keys_weights(float t, float a, float w[4]) {
    const float u = 1.0f - t;
    w[0] = a * t * u * u;
    w[1] = ((a + 2.0f) * t - (a + 3.0f)) * t * t + 1.0f;
    w[2] = ((a + 2.0f) * u - (a + 3.0f)) * u * u + 1.0f;
    w[3] = a * u * t * t;
}

// GridSample mode/padding_mode on one axis, from its 32.32 position.
// Linear and nearest pad the coordinate; cubic pads each tap index.
template <int MODE>
__device__ __forceinline__ void make_taps(int64_t xq, const Axis &A, int pad, int ac, float a,
                                          AxisTaps<MODE> &T) {
    const int n = A.n;
    if (MODE != MODE_CUBIC) {
        if (pad == PAD_BORDER) {
            xq = clamp_q(xq, 0, A.hi_q);
        } else if (pad == PAD_REFLECTION) {
            xq = clamp_q(reflect_q(xq, A.lo_q, A.span_q), 0, A.hi_q);
        }
    }
    T.ok = 0;
    if (MODE == MODE_NEAREST) {
        int64_t r = (xq + kHalfQ) >> 32;                       // floor(x + 1/2)
        if ((uint32_t)xq == 0x80000000u && (r & 1)) r -= 1;   // exact tie: even index
        const bool in = r >= 0 && r < n;
        T.idx[0] = in ? (int)r : 0;
        T.w[0] = 1.0f;
        T.ok = in ? 1u : 0u;
        return;
    }
    const int i0 = (int)(xq >> 32);
    const float t = __uint2float_rn((uint32_t)xq) * 2.3283064365386963e-10f;   // * 2^-32
    if (MODE == MODE_LINEAR) {
        T.w[0] = 1.0f - t;
        T.w[1] = t;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int j = i0 + k;
            const bool in = j >= 0 && j < n;
            T.idx[k] = in ? j : 0;
            T.ok |= (in ? 1u : 0u) << k;
        }
        return;
    }
    keys_weights(t, a, T.w);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        int j = i0 - 1 + k;
        bool in;
        if (pad == PAD_BORDER) {
            j = j < 0 ? 0 : (j > n - 1 ? n - 1 : j);
            in = true;
        } else if (pad == PAD_REFLECTION) {
            j = reflect_index(j, n, ac);
            in = true;
        } else {
            in = j >= 0 && j < n;
            j = in ? j : 0;
        }
        T.idx[k] = j;
        T.ok |= (in ? 1u : 0u) << k;
    }
}

}  // namespace gs
