// gs_api.cu -- the C ABI of libgs (declared in include/gs.h): host-side
// argument checks, then dispatch to the per-dtype launchers.  Nothing here
// allocates, synchronises (except gs_device_status) or throws.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include "../../include/gs.h"
#include "gs_internal.h"
#include "gs_ptx.cuh"

// Device error word: kernels whose bounded waits give up record it here;
// gs_device_status reads and clears it.
__device__ unsigned g_gs_error_word = 0;

// Scratch of gs_grid_sample_static: GS_STATIC_WORKSPACE_BYTES per device in
// the module's static device memory, so the call allocates nothing.  Nothing
// in it needs to start at zero: each call's copy kernel writes every byte the
// sampler then reads, the zero pixels included.
static __device__ __align__(256) unsigned char g_gs_static_ws[GS_STATIC_WORKSPACE_BYTES];

// Test hook behind gs_test_bounded_wait_expires: one thread arms an mbarrier
// for 16 bytes of transfer that no copy will ever deliver (none is issued), so
// the phase cannot complete, and waits on it with the pipelines' bounded wait.
// The wait gives up after limit_ns, sets the timeout bit in the error word and
// the kernel returns; nothing is in flight, so leaving is safe.
__global__ void bounded_wait_probe_kernel(unsigned *err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    gs::mbar_init(&bar, 1);
    gs::fence_mbar_init();
    gs::mbar_arrive_expect_tx(&bar, 16);
    gs::mbar_wait_bounded(&bar, 0, err, limit_ns);
    gs::mbar_inval(&bar);
}

namespace {

// Device address of a __device__ symbol on the current device, looked up once
// per device (a host-side symbol is not a device address; nullptr if the
// lookup fails).  The per-device caches are atomics: first calls from several
// host threads may both look the address up, and both store the same value.
template <typename S>
void *symbol_address(std::atomic<void *> (&cache)[gs::kMaxDevices], const S &symbol) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= gs::kMaxDevices) return nullptr;
    void *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(&p, symbol) != cudaSuccess) return nullptr;
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

// Device address of g_gs_error_word.
unsigned *error_word() {
    static std::atomic<void *> cache[gs::kMaxDevices];
    return (unsigned *)symbol_address(cache, g_gs_error_word);
}

// Device address of g_gs_static_ws.
void *static_workspace() {
    static std::atomic<void *> cache[gs::kMaxDevices];
    return symbol_address(cache, g_gs_static_ws);
}

constexpr int64_t kMaxExtent = int64_t(1) << 20;
constexpr int64_t kMaxSlab = (int64_t(1) << 31) - 1;

size_t elem_size(gs_dtype dt) { return dt == GS_F32 ? 4 : 2; }
bool dtype_ok(int dt) { return dt == GS_F32 || dt == GS_F16 || dt == GS_BF16; }
bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

template <typename F>
gs_status dispatch(gs_dtype dt, F &&f) {
    cudaError_t e;
    switch (dt) {
        case GS_F32: e = f(float()); break;
        case GS_F16: e = f(__half()); break;
        default: e = f(__nv_bfloat16()); break;
    }
    return e == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}

// Spatial extents: all >= 0, each <= 2^20, product (returned) < 2^31.
gs_status check_spatial(const int64_t *ext, int r, int64_t *prod, bool *empty) {
    int64_t p = 1;
    *empty = false;
    for (int d = 0; d < r; ++d) {
        if (ext[d] < 0 || ext[d] > kMaxExtent) return GS_ERR_SHAPE;
        if (ext[d] == 0) *empty = true;
        p *= ext[d];
        if (p > kMaxSlab) return GS_ERR_SHAPE;
    }
    *prod = p;
    return GS_OK;
}

bool nc_ok(int64_t N, int64_t C) { return N >= 0 && C >= 0 && N <= kMaxSlab && C <= kMaxSlab; }

// Shape and attribute checks shared by the sampling entry points (no pointers).
gs_status check_sample_shape(const int64_t *x_shape, int r, const int64_t *out_sp, gs_dtype dt,
                             gs_mode mode, gs_pad pad, int ac, float a, gs::SampleArgs *args,
                             bool *skip) {
    if (!x_shape || !out_sp) return GS_ERR_NULL;
    if (!dtype_ok(dt)) return GS_ERR_DTYPE;
    if ((int)mode < GS_LINEAR || (int)mode > GS_CUBIC) return GS_ERR_ATTR;
    if ((int)pad < GS_PAD_ZEROS || (int)pad > GS_PAD_REFLECTION) return GS_ERR_ATTR;
    if (ac != 0 && ac != 1) return GS_ERR_ATTR;
    if (mode == GS_CUBIC && !isfinite(a)) return GS_ERR_ATTR;
    const int64_t N = x_shape[0], C = x_shape[1];
    if (!nc_ok(N, C)) return GS_ERR_SHAPE;
    int64_t in_plane, out_plane;
    bool in_empty, out_empty;
    gs_status st = check_spatial(x_shape + 2, r, &in_plane, &in_empty);
    if (st != GS_OK) return st;
    st = check_spatial(out_sp, r, &out_plane, &out_empty);
    if (st != GS_OK) return st;
    *skip = out_empty || N == 0 || C == 0;
    if (*skip) return GS_OK;
    if (in_empty) return GS_ERR_SHAPE;   // nothing to sample from
    const int64_t tiles = (out_plane + gs::kSampleThreads - 1) / gs::kSampleThreads;
    if (N * tiles > kMaxSlab) return GS_ERR_SHAPE;
    args->N = (int)N;
    args->C = (int)C;
    for (int d = 0; d < gs::kMaxRankND; ++d) {
        args->in[d] = d < r ? (int)x_shape[2 + d] : 1;
        args->out[d] = d < r ? (int)out_sp[d] : 1;
    }
    args->in_plane = in_plane;
    args->out_plane = out_plane;
    args->tiles = (int)tiles;
    args->pad = (int)pad;
    args->ac = ac;
    args->a = a;
    args->err = nullptr;
    return GS_OK;
}

// All checks of gs_grid_sample and gs_affine_sample except the grid / theta.
gs_status check_sample(const void *X, const int64_t *x_shape, int r, const int64_t *out_sp,
                       gs_dtype dt, gs_mode mode, gs_pad pad, int ac, float a, const void *Y,
                       gs::SampleArgs *args, bool *skip) {
    const gs_status st = check_sample_shape(x_shape, r, out_sp, dt, mode, pad, ac, a, args, skip);
    if (st != GS_OK || *skip) return st;
    if (!X || !Y) return GS_ERR_NULL;
    if (!aligned(X, elem_size(dt)) || !aligned(Y, elem_size(dt))) return GS_ERR_ALIGN;
    return GS_OK;
}

}  // namespace

namespace {

// Checks of gs_deform_conv; fills *a (err unset) or sets *skip for an empty output.
gs_status check_deform(const void *X, const int64_t *x_shape, const void *W, int64_t oC,
                       const void *offset, const void *B, const void *mask,
                       const gs_deform_attrs *at, gs_dtype dt, const void *Y, bool shapes_only,
                       gs::DeformArgs *a, bool *skip) {
    *skip = false;
    if (!x_shape || !at) return GS_ERR_NULL;
    if (!dtype_ok(dt)) return GS_ERR_DTYPE;
    const int64_t N = x_shape[0], C = x_shape[1], H = x_shape[2], Wd = x_shape[3];
    if (!nc_ok(N, C) || oC < 0 || oC > kMaxSlab) return GS_ERR_SHAPE;
    if (H < 0 || Wd < 0 || H > kMaxExtent || Wd > kMaxExtent || H * Wd > kMaxSlab)
        return GS_ERR_SHAPE;
    for (int i = 0; i < 2; ++i) {
        if (at->kernel[i] < 1 || at->kernel[i] > 64) return GS_ERR_ATTR;
        if (at->strides[i] < 1 || at->dilations[i] < 1) return GS_ERR_ATTR;
        if (at->strides[i] > kMaxExtent || at->dilations[i] > kMaxExtent) return GS_ERR_ATTR;
    }
    for (int i = 0; i < 4; ++i)
        if (at->pads[i] < 0 || at->pads[i] > kMaxExtent) return GS_ERR_ATTR;
    if (at->group < 1 || at->offset_group < 1) return GS_ERR_ATTR;
    if (C % at->group || oC % at->group || C % at->offset_group) return GS_ERR_ATTR;
    const int64_t kH = at->kernel[0], kW = at->kernel[1];
    const int64_t oH = (H + at->pads[0] + at->pads[2] - at->dilations[0] * (kH - 1) - 1) / at->strides[0] + 1;
    const int64_t oW = (Wd + at->pads[1] + at->pads[3] - at->dilations[1] * (kW - 1) - 1) / at->strides[1] + 1;
    if (H + at->pads[0] + at->pads[2] - at->dilations[0] * (kH - 1) - 1 < 0 ||
        Wd + at->pads[1] + at->pads[3] - at->dilations[1] * (kW - 1) - 1 < 0)
        return GS_ERR_SHAPE;
    if (oH * oW > kMaxSlab) return GS_ERR_SHAPE;
    if (N == 0 || oC == 0 || oH == 0 || oW == 0) {
        *skip = true;
        return GS_OK;
    }
    if (C == 0 || H == 0 || Wd == 0) return GS_ERR_SHAPE;
    a->N = (int)N; a->C = (int)C; a->H = (int)H; a->W = (int)Wd; a->oC = (int)oC;
    a->oH = (int)oH; a->oW = (int)oW; a->kH = (int)kH; a->kW = (int)kW;
    a->pad_t = (int)at->pads[0]; a->pad_l = (int)at->pads[1];
    a->sH = (int)at->strides[0]; a->sW = (int)at->strides[1];
    a->dH = (int)at->dilations[0]; a->dW = (int)at->dilations[1];
    a->group = (int)at->group; a->offset_group = (int)at->offset_group;
    a->has_bias = B != nullptr; a->has_mask = mask != nullptr;
    a->err = nullptr;
    if (shapes_only) return GS_OK;
    if (!X || !W || !offset || !Y) return GS_ERR_NULL;
    const size_t es = elem_size(dt);
    if (!aligned(X, es) || !aligned(W, es) || !aligned(offset, es) || !aligned(Y, es) ||
        (B && !aligned(B, es)) || (mask && !aligned(mask, es)))
        return GS_ERR_ALIGN;
    return GS_OK;
}

}  // namespace

namespace {

// Resize - 18: output extents and per-axis coordinate parameters.
constexpr int kRsMaxRank = 8;
constexpr int64_t kRsMaxExtent = int64_t(1) << 24;

struct ResizePlan {
    int rank;
    int64_t in[kRsMaxRank], out[kRsMaxRank];
    double scale[kRsMaxRank], lres[kRsMaxRank], r0[kRsMaxRank], r1[kRsMaxRank];
};

gs_status resize_plan(int rank, const int64_t *x_shape, const int64_t *axes, int naxes,
                      const float *scales, const int64_t *sizes, const float *roi,
                      const gs_resize_attrs *at, ResizePlan *P) {
    if (!x_shape || !at) return GS_ERR_NULL;
    if (rank < 1 || rank > kRsMaxRank) return GS_ERR_RANK;
    if ((scales == nullptr) == (sizes == nullptr)) return GS_ERR_ATTR;
    if ((int)at->mode < GS_LINEAR || (int)at->mode > GS_CUBIC) return GS_ERR_ATTR;
    if ((int)at->coord < GS_RS_HALF_PIXEL || (int)at->coord > GS_RS_TF_CROP_AND_RESIZE)
        return GS_ERR_ATTR;
    if ((int)at->nearest_mode < GS_RS_ROUND_PREFER_FLOOR || (int)at->nearest_mode > GS_RS_CEIL)
        return GS_ERR_ATTR;
    if ((int)at->keep_aspect_ratio_policy < GS_RS_STRETCH ||
        (int)at->keep_aspect_ratio_policy > GS_RS_NOT_SMALLER)
        return GS_ERR_ATTR;
    if ((at->exclude_outside != 0 && at->exclude_outside != 1) ||
        (at->antialias != 0 && at->antialias != 1) || !isfinite(at->cubic_coeff_a))
        return GS_ERR_ATTR;
    if (naxes < 0 || naxes > rank || (naxes > 0 && !axes)) return GS_ERR_SHAPE;
    const int na = naxes > 0 ? naxes : rank;
    int ax[kRsMaxRank];
    bool seen[kRsMaxRank] = {};
    for (int i = 0; i < na; ++i) {
        int64_t d = naxes > 0 ? axes[i] : i;
        if (d < 0) d += rank;
        if (d < 0 || d >= rank || seen[d]) return GS_ERR_SHAPE;
        seen[d] = true;
        ax[i] = (int)d;
    }
    P->rank = rank;
    for (int d = 0; d < rank; ++d) {
        if (x_shape[d] < 0 || x_shape[d] > kRsMaxExtent) return GS_ERR_SHAPE;
        P->in[d] = P->out[d] = x_shape[d];
        P->scale[d] = 1.0;
        P->lres[d] = (double)x_shape[d];
        P->r0[d] = 0.0;
        P->r1[d] = 1.0;
    }
    if (roi && at->coord == GS_RS_TF_CROP_AND_RESIZE) {
        for (int i = 0; i < na; ++i) {
            if (!isfinite(roi[i]) || !isfinite(roi[na + i])) return GS_ERR_ATTR;
            P->r0[ax[i]] = roi[i];
            P->r1[ax[i]] = roi[na + i];
        }
    }
    if (scales) {
        for (int i = 0; i < na; ++i) {
            const int d = ax[i];
            const double sc = scales[i];
            if (!(sc > 0.0) || !isfinite(sc)) return GS_ERR_ATTR;
            const double len = (double)P->in[d] * (P->r1[d] - P->r0[d]) * sc;
            if (!(len >= 0.0) || len >= (double)(kRsMaxExtent + 1)) return GS_ERR_SHAPE;
            P->out[d] = (int64_t)floor(len);
            P->scale[d] = sc;
            P->lres[d] = len;
        }
        return GS_OK;
    }
    double common = 0.0;
    if (at->keep_aspect_ratio_policy != GS_RS_STRETCH) {
        for (int i = 0; i < na; ++i) {
            if (P->in[ax[i]] == 0) return GS_ERR_SHAPE;
            const double q = (double)sizes[i] / (double)P->in[ax[i]];
            if (i == 0 || (at->keep_aspect_ratio_policy == GS_RS_NOT_LARGER ? q < common : q > common))
                common = q;
        }
    }
    for (int i = 0; i < na; ++i) {
        const int d = ax[i];
        if (sizes[i] < 0 || sizes[i] > kRsMaxExtent) return GS_ERR_SHAPE;
        const double o = at->keep_aspect_ratio_policy == GS_RS_STRETCH
                             ? (double)sizes[i]
                             : floor(common * (double)P->in[d] + 0.5);
        if (!(o >= 0.0) || o > (double)kRsMaxExtent) return GS_ERR_SHAPE;
        P->out[d] = (int64_t)o;
        P->scale[d] = P->in[d] > 0 ? o / (double)P->in[d] : 1.0;
        P->lres[d] = o;
    }
    return GS_OK;
}

// Taps per output index on one axis: 1 (nearest), else the offsets k0 .. 1-k0
// from floor(x) where the filter, stretched by 1/aa when antialiasing a
// downscale, can be nonzero (linear reaches 1, cubic 2).
void resize_taps_per_axis(const gs_resize_attrs *at, double scale, gs::ResizeAxis *A) {
    A->aa_scale = (at->antialias && at->mode != GS_NEAREST && scale < 1.0) ? scale : 1.0;
    if (at->mode == GS_NEAREST) {
        A->k0 = 0;
        A->taps = 1;
        return;
    }
    const double reach = at->mode == GS_LINEAR ? 1.0 : 2.0;
    const double k0 = floor(-reach / A->aa_scale) + 1.0;
    A->k0 = k0 < -1.0e6 ? -1000000 : (int)k0;
    A->taps = 2 - 2 * A->k0;
}

}  // namespace

extern "C" {

gs_status gs_resize_output_shape(int rank, const int64_t *x_shape, const int64_t *axes, int naxes,
                                 const float *scales, const int64_t *sizes, const float *roi,
                                 const gs_resize_attrs *attrs, int64_t *y_shape) {
    if (!y_shape) return GS_ERR_NULL;
    ResizePlan P;
    const gs_status st = resize_plan(rank, x_shape, axes, naxes, scales, sizes, roi, attrs, &P);
    if (st != GS_OK) return st;
    for (int d = 0; d < rank; ++d) y_shape[d] = P.out[d];
    return GS_OK;
}

gs_status gs_resize(const void *X, int rank, const int64_t *x_shape, const int64_t *axes,
                    int naxes, const float *scales, const int64_t *sizes, const float *roi,
                    const gs_resize_attrs *attrs, gs_dtype dt, void *Y, cudaStream_t stream) {
    ResizePlan P;
    gs_status st = resize_plan(rank, x_shape, axes, naxes, scales, sizes, roi, attrs, &P);
    if (st != GS_OK) return st;
    if (!dtype_ok(dt)) return GS_ERR_DTYPE;
    bool empty_out = false, empty_in = false;
    for (int d = 0; d < rank; ++d) {
        empty_out = empty_out || P.out[d] == 0;
        empty_in = empty_in || P.in[d] == 0;
    }
    if (empty_out) return GS_OK;
    if (empty_in) return GS_ERR_SHAPE;   // nothing to sample from
    if (!X || !Y) return GS_ERR_NULL;
    if (!aligned(X, elem_size(dt)) || !aligned(Y, elem_size(dt))) return GS_ERR_ALIGN;
    // identity axes (same extent, scale 1, whole roi) in front of the first
    // resized one become slices
    auto identity = [&](int d) {
        return P.out[d] == P.in[d] && P.scale[d] == 1.0 && P.r0[d] == 0.0 && P.r1[d] == 1.0;
    };
    int f = 0;
    while (f < rank - 1 && identity(f)) ++f;
    const int R = rank - f;
    if (R > 3) return GS_ERR_UNSUPPORTED;
    gs::ResizeArgs a;
    a.r = R;
    a.B = 1;
    for (int d = 0; d < f; ++d) a.B *= P.in[d];
    a.mode = (int)attrs->mode;
    a.coord = (int)attrs->coord;
    a.nearest_mode = (int)attrs->nearest_mode;
    a.a = attrs->cubic_coeff_a;
    a.exclude_outside = attrs->exclude_outside;
    a.extrapolation_value = attrs->extrapolation_value;
    for (int i = 0; i < 3; ++i) {
        gs::ResizeAxis &A = a.ax[i];
        const int d = f + i - (3 - R);
        if (i < 3 - R) {   // unit axis
            A.n_in = A.n_out = 1;
            A.scale = A.length_resized = A.roi_end = A.aa_scale = 1.0;
            A.roi_start = 0.0;
            A.k0 = 0;
            A.taps = 1;
            continue;
        }
        A.n_in = (int)P.in[d];
        A.n_out = (int)P.out[d];
        A.scale = P.scale[d];
        A.length_resized = P.lres[d];
        A.roi_start = P.r0[d];
        A.roi_end = P.r1[d];
        resize_taps_per_axis(attrs, P.scale[d], &A);
        if (A.taps > gs::kRsMaxTapsHost) return GS_ERR_UNSUPPORTED;
    }
    a.err = error_word();
    return dispatch(dt, [&](auto tag) {
        return gs::launch_resize<decltype(tag)>(X, Y, a, stream);
    });
}

gs_status gs_affine_grid(const void *theta, gs_dtype dt, int r, const int64_t *size,
                         int align_corners, void *grid, cudaStream_t stream) {
    if (!size) return GS_ERR_NULL;
    if (!dtype_ok(dt)) return GS_ERR_DTYPE;
    if (r != 2 && r != 3) return GS_ERR_RANK;
    if (align_corners != 0 && align_corners != 1) return GS_ERR_ATTR;
    const int64_t N = size[0];
    if (!nc_ok(N, size[1])) return GS_ERR_SHAPE;
    int64_t plane;
    bool empty;
    gs_status st = check_spatial(size + 2, r, &plane, &empty);
    if (st != GS_OK) return st;
    if (empty || N == 0) return GS_OK;
    if (!theta || !grid) return GS_ERR_NULL;
    if (!aligned(theta, elem_size(dt)) || !aligned(grid, elem_size(dt))) return GS_ERR_ALIGN;
    if ((N * plane + 255) / 256 > kMaxSlab) return GS_ERR_SHAPE;
    gs::AffineGridArgs a;
    a.N = (int)N;
    for (int d = 0; d < 3; ++d) a.out[d] = d < r ? (int)size[2 + d] : 1;
    a.out_plane = plane;
    a.ac = align_corners;
    return dispatch(dt, [&](auto tag) {
        return gs::launch_affine_grid<decltype(tag)>(theta, grid, a, r, stream);
    });
}

gs_status gs_grid_sample(const void *X, const int64_t *x_shape, int r, const void *grid,
                         const int64_t *out_spatial, gs_dtype dt, gs_mode mode, gs_pad pad,
                         int align_corners, float cubic_coeff_a, void *Y, cudaStream_t stream) {
    if (r < 1 || r > gs::kMaxRankND) return GS_ERR_RANK;
    gs::SampleArgs args;
    bool skip = false;
    gs_status st = check_sample(X, x_shape, r, out_spatial, dt, mode, pad, align_corners,
                                cubic_coeff_a, Y, &args, &skip);
    if (st != GS_OK || skip) return st;
    if (!grid) return GS_ERR_NULL;
    if (!aligned(grid, elem_size(dt))) return GS_ERR_ALIGN;
    args.err = error_word();
    return dispatch(dt, [&](auto tag) {
        return gs::launch_sample<decltype(tag)>(X, grid, Y, args, r, (int)mode, false, nullptr, 0,
                                                stream);
    });
}

gs_status gs_grid_sample_int(const void *X, gs_itype xt, const int64_t *x_shape, int r,
                             const void *grid, gs_dtype grid_dt, const int64_t *out_spatial,
                             gs_mode mode, gs_pad pad, int align_corners, float cubic_coeff_a,
                             void *Y, cudaStream_t stream) {
    if (r < 1 || r > gs::kMaxRankND) return GS_ERR_RANK;
    if (xt != GS_U8 && xt != GS_I8 && xt != GS_U16 && xt != GS_I16) return GS_ERR_DTYPE;
    gs::SampleArgs args;
    bool skip = false;
    // shape and attribute checks as gs_grid_sample, with the grid's float type
    gs_status st = check_sample_shape(x_shape, r, out_spatial, grid_dt, mode, pad, align_corners,
                                      cubic_coeff_a, &args, &skip);
    if (st != GS_OK || skip) return st;
    const size_t xs = (xt == GS_U8 || xt == GS_I8) ? 1 : 2;
    if (!X || !Y || !grid) return GS_ERR_NULL;
    if (!aligned(X, xs) || !aligned(Y, xs) || !aligned(grid, elem_size(grid_dt))) return GS_ERR_ALIGN;
    cudaError_t e;
    switch (xt) {
        case GS_U8:
            e = gs::launch_sample_int<uint8_t>(X, grid, (int)grid_dt, Y, args, r, (int)mode, stream);
            break;
        case GS_I8:
            e = gs::launch_sample_int<int8_t>(X, grid, (int)grid_dt, Y, args, r, (int)mode, stream);
            break;
        case GS_U16:
            e = gs::launch_sample_int<uint16_t>(X, grid, (int)grid_dt, Y, args, r, (int)mode, stream);
            break;
        default:
            e = gs::launch_sample_int<int16_t>(X, grid, (int)grid_dt, Y, args, r, (int)mode, stream);
            break;
    }
    return e == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}

gs_status gs_grid_sample_workspace_size(const int64_t *x_shape, int r, const int64_t *out_spatial,
                                        gs_dtype dt, size_t *bytes) {
    if (!bytes) return GS_ERR_NULL;
    *bytes = 0;
    if (r < 1 || r > gs::kMaxRankND) return GS_ERR_RANK;
    gs::SampleArgs args;
    bool skip = false;
    // mode and padding do not change the size: check the shapes only
    const gs_status st = check_sample_shape(x_shape, r, out_spatial, dt, GS_LINEAR, GS_PAD_ZEROS,
                                            0, -0.75f, &args, &skip);
    if (st != GS_OK || skip) return st;
    switch (dt) {
        case GS_F32: *bytes = gs::sample_workspace_bytes<float>(args, r, false); break;
        case GS_F16: *bytes = gs::sample_workspace_bytes<__half>(args, r, false); break;
        default: *bytes = gs::sample_workspace_bytes<__nv_bfloat16>(args, r, false); break;
    }
    return GS_OK;
}

gs_status gs_grid_sample_ws(const void *X, const int64_t *x_shape, int r, const void *grid,
                            const int64_t *out_spatial, gs_dtype dt, gs_mode mode, gs_pad pad,
                            int align_corners, float cubic_coeff_a, void *workspace,
                            size_t workspace_bytes, void *Y, cudaStream_t stream) {
    if (r < 1 || r > gs::kMaxRankND) return GS_ERR_RANK;
    gs::SampleArgs args;
    bool skip = false;
    gs_status st = check_sample(X, x_shape, r, out_spatial, dt, mode, pad, align_corners,
                                cubic_coeff_a, Y, &args, &skip);
    if (st != GS_OK || skip) return st;
    if (!grid) return GS_ERR_NULL;
    if (!aligned(grid, elem_size(dt))) return GS_ERR_ALIGN;
    if (workspace && !aligned(workspace, 16)) return GS_ERR_ALIGN;
    if (workspace_bytes && !workspace) return GS_ERR_NULL;
    args.err = error_word();
    return dispatch(dt, [&](auto tag) {
        return gs::launch_sample<decltype(tag)>(X, grid, Y, args, r, (int)mode, false, workspace,
                                                workspace_bytes, stream);
    });
}

gs_status gs_grid_sample_static(const void *X, const int64_t *x_shape, int r, const void *grid,
                                const int64_t *out_spatial, gs_dtype dt, gs_mode mode, gs_pad pad,
                                int align_corners, float cubic_coeff_a, void *Y,
                                cudaStream_t stream) {
    if (r < 1 || r > gs::kMaxRankND) return GS_ERR_RANK;
    gs::SampleArgs args;
    bool skip = false;
    gs_status st = check_sample(X, x_shape, r, out_spatial, dt, mode, pad, align_corners,
                                cubic_coeff_a, Y, &args, &skip);
    if (st != GS_OK || skip) return st;
    if (!grid) return GS_ERR_NULL;
    if (!aligned(grid, elem_size(dt))) return GS_ERR_ALIGN;
    size_t need = 0, slot = 0;   // asked-for size; one image slot (the least it runs with)
    switch (dt) {
        case GS_F32:
            need = gs::sample_workspace_bytes<float>(args, r, false);
            slot = gs::sample_min_workspace_bytes<float>(args);
            break;
        case GS_F16:
            need = gs::sample_workspace_bytes<__half>(args, r, false);
            slot = gs::sample_min_workspace_bytes<__half>(args);
            break;
        default:
            need = gs::sample_workspace_bytes<__nv_bfloat16>(args, r, false);
            slot = gs::sample_min_workspace_bytes<__nv_bfloat16>(args);
            break;
    }
    void *ws = nullptr;
    size_t ws_bytes = 0;
    if (need > 0) {   // the channel-last path takes this call
        if (slot > (size_t)GS_STATIC_WORKSPACE_BYTES) return GS_ERR_SHAPE;
        ws = static_workspace();
        if (!ws) return GS_ERR_CUDA;
        ws_bytes = (size_t)GS_STATIC_WORKSPACE_BYTES;
    }
    args.err = error_word();
    return dispatch(dt, [&](auto tag) {
        return gs::launch_sample<decltype(tag)>(X, grid, Y, args, r, (int)mode, false, ws, ws_bytes,
                                                stream);
    });
}

gs_status gs_affine_sample(const void *theta, const int64_t *size, int r, const void *X,
                           const int64_t *x_shape, gs_dtype dt, gs_mode mode, gs_pad pad,
                           int align_corners, float cubic_coeff_a, void *Y,
                           cudaStream_t stream) {
    if (r != 2 && r != 3) return GS_ERR_RANK;
    if (!size || !x_shape) return GS_ERR_NULL;
    if (size[0] != x_shape[0] || size[1] != x_shape[1]) return GS_ERR_SHAPE;
    gs::SampleArgs args;
    bool skip = false;
    gs_status st = check_sample(X, x_shape, r, size + 2, dt, mode, pad, align_corners,
                                cubic_coeff_a, Y, &args, &skip);
    if (st != GS_OK || skip) return st;
    if (!theta) return GS_ERR_NULL;
    if (!aligned(theta, elem_size(dt))) return GS_ERR_ALIGN;
    args.err = error_word();
    return dispatch(dt, [&](auto tag) {
        return gs::launch_sample<decltype(tag)>(X, theta, Y, args, r, (int)mode, true, nullptr, 0,
                                                stream);
    });
}

gs_status gs_affine_sample_from_host(const void *theta_h, const int64_t *size, int r,
                                     const void *X_h, const int64_t *x_shape, gs_dtype dt,
                                     gs_mode mode, gs_pad pad, int align_corners,
                                     float cubic_coeff_a, void *Y_h, void *theta_d, void *X_d,
                                     void *Y_d, int chunks, const cudaStream_t *streams) {
    if (r != 2 && r != 3) return GS_ERR_RANK;
    if (!size || !x_shape) return GS_ERR_NULL;
    if (size[0] != x_shape[0] || size[1] != x_shape[1]) return GS_ERR_SHAPE;
    gs::SampleArgs args;
    bool skip = false;
    gs_status st = check_sample(X_d, x_shape, r, size + 2, dt, mode, pad, align_corners,
                                cubic_coeff_a, Y_d, &args, &skip);
    if (st != GS_OK || skip) return st;
    if (!theta_d || !theta_h || !X_h || !Y_h || !streams) return GS_ERR_NULL;
    if (!aligned(theta_d, elem_size(dt))) return GS_ERR_ALIGN;
    args.err = error_word();
    const int64_t N = args.N;
    const int64_t runs = chunks < 1 ? 1 : (chunks > N ? N : chunks);
    const int64_t step = (N + runs - 1) / runs;
    const size_t es = elem_size(dt);
    const size_t th_img = (size_t)r * (r + 1) * es;
    const size_t x_img = (size_t)args.C * (size_t)args.in_plane * es;
    const size_t y_img = (size_t)args.C * (size_t)args.out_plane * es;
    cudaEvent_t ev_in = nullptr, ev_run = nullptr;
    if (cudaEventCreateWithFlags(&ev_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ev_run, cudaEventDisableTiming) != cudaSuccess) {
        if (ev_in) cudaEventDestroy(ev_in);
        return GS_ERR_CUDA;
    }
    const cudaStream_t s_in = streams[0], s_run = streams[1], s_out = streams[2];
    gs_status res = GS_OK;
    for (int64_t n0 = 0; n0 < N && res == GS_OK; n0 += step) {
        const int64_t n = N - n0 < step ? N - n0 : step;
        const char *th_src = static_cast<const char *>(theta_h) + n0 * th_img;
        const char *x_src = static_cast<const char *>(X_h) + n0 * x_img;
        char *th_dst = static_cast<char *>(theta_d) + n0 * th_img;
        char *x_dst = static_cast<char *>(X_d) + n0 * x_img;
        char *y_dev = static_cast<char *>(Y_d) + n0 * y_img;
        char *y_dst = static_cast<char *>(Y_h) + n0 * y_img;
        // the event calls order the streams: a wait enqueued here refers to the
        // record just before it, so both events are reused run after run
        if (cudaMemcpyAsync(th_dst, th_src, n * th_img, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
            cudaMemcpyAsync(x_dst, x_src, n * x_img, cudaMemcpyHostToDevice, s_in) != cudaSuccess ||
            cudaEventRecord(ev_in, s_in) != cudaSuccess ||
            cudaStreamWaitEvent(s_run, ev_in, 0) != cudaSuccess) {
            res = GS_ERR_CUDA;
            break;
        }
        gs::SampleArgs a = args;
        a.N = (int)n;
        const gs_status ls = dispatch(dt, [&](auto tag) {
            return gs::launch_sample<decltype(tag)>(x_dst, th_dst, y_dev, a, r, (int)mode, true,
                                                    nullptr, 0, s_run);
        });
        if (ls != GS_OK || cudaEventRecord(ev_run, s_run) != cudaSuccess ||
            cudaStreamWaitEvent(s_out, ev_run, 0) != cudaSuccess ||
            cudaMemcpyAsync(y_dst, y_dev, n * y_img, cudaMemcpyDeviceToHost, s_out) != cudaSuccess)
            res = GS_ERR_CUDA;
    }
    // events may be destroyed with work still pending on them
    cudaEventDestroy(ev_in);
    cudaEventDestroy(ev_run);
    return res;
}

gs_status gs_deform_conv(const void *X, const int64_t *x_shape, const void *W, int64_t oC,
                         const void *offset, const void *B, const void *mask,
                         const gs_deform_attrs *at, gs_dtype dt, void *Y, cudaStream_t stream) {
    gs::DeformArgs a;
    bool skip = false;
    const gs_status st = check_deform(X, x_shape, W, oC, offset, B, mask, at, dt, Y, false, &a, &skip);
    if (st != GS_OK || skip) return st;
    a.err = error_word();
    return dispatch(dt, [&](auto tag) {
        return gs::launch_deform<decltype(tag)>(X, W, offset, B, mask, Y, a, stream);
    });
}

gs_status gs_deform_conv_workspace_size(const int64_t *x_shape, int64_t oC,
                                        const gs_deform_attrs *attrs, gs_dtype dt, size_t *bytes) {
    if (!bytes) return GS_ERR_NULL;
    *bytes = 0;
    gs::DeformArgs a;
    bool skip = false;
    const gs_status st = check_deform(nullptr, x_shape, nullptr, oC, nullptr, nullptr, nullptr,
                                      attrs, dt, nullptr, true, &a, &skip);
    if (st != GS_OK || skip) return st;
    a.has_bias = 1;
    a.has_mask = 1;
    switch (dt) {
        case GS_F32: *bytes = gs::deform_ws_bytes<float>(a); break;
        case GS_F16: *bytes = gs::deform_ws_bytes<__half>(a); break;
        default: *bytes = gs::deform_ws_bytes<__nv_bfloat16>(a); break;
    }
    return GS_OK;
}

gs_status gs_deform_conv_ws(const void *X, const int64_t *x_shape, const void *W, int64_t oC,
                            const void *offset, const void *B, const void *mask,
                            const gs_deform_attrs *at, gs_dtype dt, void *workspace,
                            size_t workspace_bytes, void *Y, cudaStream_t stream) {
    gs::DeformArgs a;
    bool skip = false;
    const gs_status st = check_deform(X, x_shape, W, oC, offset, B, mask, at, dt, Y, false, &a, &skip);
    if (st != GS_OK || skip) return st;
    if (workspace && !aligned(workspace, 256)) return GS_ERR_ALIGN;
    if (workspace_bytes && !workspace) return GS_ERR_NULL;
    a.err = error_word();
    return dispatch(dt, [&](auto tag) {
        return gs::launch_deform_ws<decltype(tag)>(X, W, offset, B, mask, Y, a, workspace,
                                                   workspace_bytes, stream);
    });
}

const char *gs_status_str(gs_status s) {
    switch (s) {
        case GS_OK: return "ok";
        case GS_ERR_NULL: return "null pointer";
        case GS_ERR_RANK: return "unsupported spatial rank";
        case GS_ERR_SHAPE: return "bad shape";
        case GS_ERR_DTYPE: return "bad dtype";
        case GS_ERR_ATTR: return "bad attribute";
        case GS_ERR_ALIGN: return "misaligned pointer";
        case GS_ERR_CUDA: return "CUDA error";
        case GS_ERR_TIMEOUT: return "device-side wait timed out";
        case GS_ERR_UNSUPPORTED: return "unsupported";
    }
    return "unknown status";
}

gs_status gs_device_status(cudaStream_t stream) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GS_ERR_CUDA;
    unsigned word = 0;
    if (cudaMemcpyFromSymbol(&word, g_gs_error_word, sizeof(word)) != cudaSuccess) return GS_ERR_CUDA;
    if (word) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_gs_error_word, &zero, sizeof(zero)) != cudaSuccess) return GS_ERR_CUDA;
        return GS_ERR_TIMEOUT;
    }
    return GS_OK;
}

gs_status gs_test_bounded_wait_expires(uint64_t limit_ns, cudaStream_t stream) {
    if (limit_ns == 0 || limit_ns > 1000000000ull) return GS_ERR_ATTR;
    unsigned *err = error_word();
    if (!err) return GS_ERR_CUDA;
    bounded_wait_probe_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
    return cudaGetLastError() == cudaSuccess ? GS_OK : GS_ERR_CUDA;
}

const char *gs_version(void) { return "0.2.0"; }

}  // extern "C"
