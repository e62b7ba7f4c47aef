/*
 * gs.h -- C ABI of libgs, GB300 (sm_103a) kernels for spatial-transformer
 * sampling: AffineGrid, GridSample, the two fused, and DeformConv.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are caller-owned, dense, row-major (C-contiguous) DEVICE buffers
 *    in the operators' layouts.  Shapes and attributes are HOST values.
 *  - One dtype per call: theta, X, grid, W, offset, B, mask and Y all use
 *    `dt`.  Arithmetic is fp32 (coordinates in exact fixed point, see
 *    gs_grid_sample); half types are widened on load and rounded to nearest
 *    even on store.
 *  - The library allocates no memory, keeps no state between calls and never
 *    synchronises: every call only enqueues kernels on `stream` (0 = the
 *    legacy default stream) and returns.  Scratch space, where a path uses
 *    some, is a workspace the caller passes in, or (gs_grid_sample_static) a
 *    fixed array in the library's static device memory.  Output buffers must
 *    not overlap inputs.
 *  - Arguments are checked on the host before anything is enqueued; a bad
 *    argument returns its gs_status and leaves the outputs untouched.  A
 *    failed launch returns GS_ERR_CUDA.  A tensor with a zero extent is valid
 *    and returns GS_OK without a launch.  Nothing throws across the ABI.
 *  - Pointers must be aligned to their element size (GS_ERR_ALIGN).
 *  - Limits (GS_ERR_SHAPE beyond them): each spatial extent <= 2^20; each
 *    (n, c) slab of X or Y < 2^31 elements; batch and channel counts < 2^31.
 *  - Host threads may call the library at the same time.  The only host-side
 *    state is per-device setup done on the first call that needs it (a
 *    kernel's shared-memory limit, a symbol's device address); it is kept in
 *    atomics, and two threads that both run it get the same result.  Calls
 *    whose outputs overlap race on the device, as any two kernels would, and
 *    so do overlapping gs_grid_sample_static calls (one scratch).
 */
#ifndef GS_H
#define GS_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GS_OK = 0,
    GS_ERR_NULL = 1,        /* a required pointer is NULL                          */
    GS_ERR_RANK = 2,        /* spatial rank r not supported by this entry point    */
    GS_ERR_SHAPE = 3,       /* extents inconsistent, negative or beyond the limits */
    GS_ERR_DTYPE = 4,       /* unknown gs_dtype                                    */
    GS_ERR_ATTR = 5,        /* unknown mode / padding, bad kernel/stride/group ... */
    GS_ERR_ALIGN = 6,       /* a pointer is not aligned to its element size        */
    GS_ERR_CUDA = 7,        /* the CUDA runtime reported an error at launch        */
    GS_ERR_TIMEOUT = 8,     /* a bounded device-side wait gave up (see gs_device_status) */
    GS_ERR_UNSUPPORTED = 9  /* valid by the operator spec, not implemented here    */
} gs_status;

typedef enum { GS_F32 = 0, GS_F16 = 1, GS_BF16 = 2 } gs_dtype;

/* GridSample - version 20, Attributes, mode.  The version-16 names "bilinear"
 * and "bicubic" are the same modes (the Python binding maps them). */
typedef enum { GS_LINEAR = 0, GS_NEAREST = 1, GS_CUBIC = 2 } gs_mode;

/* GridSample - version 20, Attributes, padding_mode. */
typedef enum { GS_PAD_ZEROS = 0, GS_PAD_BORDER = 1, GS_PAD_REFLECTION = 2 } gs_pad;

/*
 * gs_affine_grid -- AffineGrid (ai.onnx, since version 20): description and
 * Inputs/Outputs.
 *
 *   theta  device, (N, r, r+1): the affine matrices without their implicit
 *          last row [0 .. 0 1].
 *   r      2 or 3.
 *   size   host, r+2 int64: (N, C, H, W) or (N, C, D, H, W); C is unused.
 *   align_corners  0: -1 and 1 are the outer edges of the corner pixels, the
 *          base positions are (2i+1)/n - 1; 1: they are the corner pixel
 *          centres, -1 + 2i/(n-1) (an axis of length 1 sits at 0).
 *   grid   device output, (N, H, W, 2) or (N, D, H, W, 3); each vector lists
 *          the width coordinate first.  Computed in fp64, rounded once.
 */
gs_status gs_affine_grid(const void *theta, gs_dtype dt, int r, const int64_t *size,
                         int align_corners, void *grid, cudaStream_t stream);

/*
 * gs_grid_sample -- GridSample - version 20 (and version 22): description,
 * Inputs, Outputs and Attributes.
 *
 *   X        device, (N, C, D1..Dr): values at pixel centres.
 *   x_shape  host, r+2 int64.
 *   r        1 to 6 spatial dimensions (GS_ERR_RANK otherwise).
 *   grid     device, (N, D1_out..Dr_out, r); the location vector lists the
 *            innermost axis first (x -> width, y -> height, z -> depth).
 *   out_spatial  host, r int64: D1_out..Dr_out.
 *   mode     linear (N-linear), nearest (ties to the even index), cubic
 *            (N-cubic, Keys kernel with coefficient cubic_coeff_a).
 *   pad      zeros: out-of-range taps read 0; border: clamp; reflection:
 *            mirror at the borders until in range, then clamp.  For linear
 *            and nearest the coordinate is padded; for cubic each tap index is.
 *   align_corners  as in gs_affine_grid: x = (g+1)/2*(n-1) for 1,
 *            x = ((g+1)*n - 1)/2 for 0.
 *   cubic_coeff_a  Keys' a (the operator uses -0.75); ignored unless cubic.
 *   Y        device output, (N, C, D1_out..Dr_out).
 *
 * The unnormalised coordinate is formed without rounding error (an exact
 * product split, then 32.32 fixed point), so nearest picks the same index as
 * exact arithmetic, ties included.  Ranks 4 to 6 run on one rank-general
 * kernel (the tap product summed axis by axis, innermost first); the
 * operator's description defines any rank r, and 6 is this library's limit.
 *
 * Speed: this call reads X in its own NCHW layout, one 2- or 4-byte load per
 * tap and channel.  Grids with spatial locality (smooth warps) are served well
 * from L2; random-access 2-D grids are not, since every tap of every channel
 * then touches its own 32-byte sector.  For those, gs_grid_sample_ws (or
 * gs_grid_sample_static) copies X to channel-last order first and reads each
 * tap as 16-byte runs of channels; on a 16 x 64 x 256^2 fp32 image batch with
 * a uniformly random cubic grid it is about five times faster, copy included.
 */
gs_status gs_grid_sample(const void *X, const int64_t *x_shape, int r, const void *grid,
                         const int64_t *out_spatial, gs_dtype dt, gs_mode mode, gs_pad pad,
                         int align_corners, float cubic_coeff_a, void *Y, cudaStream_t stream);

/*
 * gs_grid_sample_workspace_size -- device workspace that gs_grid_sample_ws
 * asks for with these shapes: whole image slots, a slot being (H*W + 1) * C
 * elements of `dt`, enough for the batch in equal chunks of at most about
 * 512 MB (at least one slot).  0 means the call never uses a workspace (rank
 * other than 2, C * element size not a multiple of 16 bytes,
 * (H*W + 1) * C >= 2^31, or an empty tensor).  Arguments as gs_grid_sample;
 * `bytes` is a host output.  Shape errors are reported as by gs_grid_sample.
 */
gs_status gs_grid_sample_workspace_size(const int64_t *x_shape, int r, const int64_t *out_spatial,
                                        gs_dtype dt, size_t *bytes);

/*
 * gs_grid_sample_ws -- gs_grid_sample with a caller-owned device workspace
 * (GridSample - version 20, as above; the same results, value for value).
 *
 *   workspace        device, 16-byte aligned (GS_ERR_ALIGN), or NULL.
 *   workspace_bytes  its size.  With room for one image slot ((H*W + 1) * C
 *                    elements of `dt`: a zero pixel, then the image), 2-D
 *                    calls copy X to channel-last order there, as many whole
 *                    images at a time as it holds, then read every tap as
 *                    16-byte runs of channels: for grids without spatial
 *                    locality this cuts the bytes read per output several
 *                    fold.  Each chunk costs a copy launch and a sampling
 *                    launch, so fewer, larger chunks are faster.  With less
 *                    than one slot, or NULL, it is gs_grid_sample.
 *
 * The workspace's contents on entry do not matter and are garbage on return.
 * Calls on different streams must not share a workspace while in flight.
 */
gs_status gs_grid_sample_ws(const void *X, const int64_t *x_shape, int r, const void *grid,
                            const int64_t *out_spatial, gs_dtype dt, gs_mode mode, gs_pad pad,
                            int align_corners, float cubic_coeff_a, void *workspace,
                            size_t workspace_bytes, void *Y, cudaStream_t stream);

/* Integer element types of X for gs_grid_sample_int. */
typedef enum { GS_U8 = 16, GS_I8 = 17, GS_U16 = 18, GS_I16 = 19 } gs_itype;

/*
 * gs_grid_sample_int -- GridSample - version 20 with an integer-typed X
 * (Type Constraints, T1; Outputs: "for integer input types, intermediate
 * values are computed as floating point and cast to integer at the end").
 *
 *   X, Y     device, integer type `xt` (uint8, int8, uint16, int16), the
 *            layouts of gs_grid_sample.
 *   grid     device, floating type `grid_dt` (T2: float, float16; bfloat16
 *            as in version 22).
 *   Other arguments, and the taps and weights, as gs_grid_sample.
 *
 * X is widened to fp32 (exact for these types), interpolated in fp32, then
 * truncated toward zero and saturated at the range of `xt` (cubic weights can
 * overshoot it).  Errors as gs_grid_sample; GS_ERR_DTYPE for another `xt` or
 * `grid_dt`.
 */
gs_status gs_grid_sample_int(const void *X, gs_itype xt, const int64_t *x_shape, int r,
                             const void *grid, gs_dtype grid_dt, const int64_t *out_spatial,
                             gs_mode mode, gs_pad pad, int align_corners, float cubic_coeff_a,
                             void *Y, cudaStream_t stream);

/* Size of the scratch gs_grid_sample_static uses: 64 MiB per device. */
#define GS_STATIC_WORKSPACE_BYTES (64u << 20)

/*
 * gs_grid_sample_static -- gs_grid_sample_ws whose workspace is a fixed
 * GS_STATIC_WORKSPACE_BYTES array in the library's static device memory, so
 * the call allocates nothing (no cudaMalloc, no allocating library call) and
 * needs no caller buffer.  It is meant for callers that cannot allocate
 * device memory at the point of the call: a plugin inside a host framework
 * that owns all device memory through its own pool and hands out only
 * inputs and outputs; a real-time loop that must not block, since
 * cudaMalloc and cudaFree can synchronise the device; or code whose memory
 * budget is fixed at start-up, where an allocation failing mid-run has no
 * way to recover.  The operator pages have no counterpart to this call; it
 * wraps the same kernels as gs_grid_sample_ws.
 *
 *   Arguments, results and errors as gs_grid_sample.  A call the channel-
 *   last path takes (see gs_grid_sample_workspace_size) whose image slot,
 *   (H*W + 1) * C elements of `dt`, exceeds GS_STATIC_WORKSPACE_BYTES
 *   returns GS_ERR_SHAPE before anything is enqueued; other calls run the
 *   NCHW gather and touch no scratch.
 *
 * The scratch needs no clearing: each call writes every byte it reads.  The
 * first call on each device looks up the scratch's address (and the error
 * word's) once with cudaGetSymbolAddress, GS_ERR_CUDA if that fails: make it
 * before any stream capture.  There is one scratch per device and process:
 * calls in flight at the same time on different streams, or from different
 * host threads, race on it and corrupt each other's results.
 */
gs_status gs_grid_sample_static(const void *X, const int64_t *x_shape, int r, const void *grid,
                                const int64_t *out_spatial, gs_dtype dt, gs_mode mode, gs_pad pad,
                                int align_corners, float cubic_coeff_a, void *Y,
                                cudaStream_t stream);

/*
 * gs_affine_sample -- GridSample(X, AffineGrid(theta, size)) in one kernel
 * (AffineGrid, ai.onnx since version 20: description, Inputs and Outputs;
 * GridSample - version 20: description, Inputs and Attributes): the grid is
 * generated per output position in registers and never touches memory (the
 * spatial transformer's grid generator and sampler).
 *
 *   theta    device, (N, r, r+1).
 *   size     host, r+2 int64: (N, C, out...), AffineGrid's size input; N and
 *            C must equal X's.
 *   X, x_shape, mode, pad, align_corners, cubic_coeff_a, Y: as gs_grid_sample,
 *            with Y (N, C, out...).  align_corners applies to both operators.
 *
 * The grid is not rounded to `dt` between the two operators.  Positions are
 * affine in the output index; the kernel evaluates that map in 64-bit fixed
 * point (coefficients from fp64), so an identity theta reproduces X exactly.
 */
gs_status gs_affine_sample(const void *theta, const int64_t *size, int r, const void *X,
                           const int64_t *x_shape, gs_dtype dt, gs_mode mode, gs_pad pad,
                           int align_corners, float cubic_coeff_a, void *Y,
                           cudaStream_t stream);

/*
 * gs_affine_sample_from_host -- gs_affine_sample with theta, X and Y in host
 * memory: the batch is cut into `chunks` runs of whole images, and for each
 * run the upload of theta and X (streams[0]), the kernel (streams[1]) and the
 * download of Y (streams[2]) are enqueued with cudaMemcpyAsync and ordered by
 * events, so the copies of neighbouring runs overlap the kernels.  The
 * operator is independent per image, so the result equals gs_affine_sample's
 * bit for bit.
 *
 *   theta_h, X_h, Y_h     host; page-locked (cudaHostAlloc / cudaHostRegister)
 *                         for the copies to overlap, pageable works but
 *                         serialises them.  Y_h is written.
 *   theta_d, X_d, Y_d     device buffers of the full sizes (caller-owned; the
 *                         library allocates nothing), aligned as gs_affine_sample
 *                         wants X, theta and Y.
 *   chunks                runs to cut the batch into (clamped to [1, N]).
 *   streams               host, three caller-owned streams: upload, kernel,
 *                         download.  Nothing orders them against other work:
 *                         make streams[0] wait for whatever produced theta_h
 *                         and X_h, and wait on streams[2] before reading Y_h.
 *   Other arguments as gs_affine_sample.
 *
 * Errors as gs_affine_sample; GS_ERR_NULL for a missing host or device buffer
 * or stream array; GS_ERR_CUDA if a copy, event or launch fails to enqueue
 * (runs already enqueued stay enqueued).
 */
gs_status gs_affine_sample_from_host(const void *theta_h, const int64_t *size, int r,
                                     const void *X_h, const int64_t *x_shape, gs_dtype dt,
                                     gs_mode mode, gs_pad pad, int align_corners,
                                     float cubic_coeff_a, void *Y_h, void *theta_d, void *X_d,
                                     void *Y_d, int chunks, const cudaStream_t *streams);

/*
 * DeformConv attributes.  The DeformConv page lists no Attributes section; its
 * examples use kernel_shape, pads and offset_group.  The rest follow ONNX Conv:
 *   kernel     (kH, kW); 0 means "take it from W".
 *   pads       (top, left, bottom, right).
 *   strides    (sH, sW), >= 1.     dilations (dH, dW), >= 1.
 *   group      C and oC divisible by it.
 *   offset_group  C divisible by it.
 * Output extents: oH = (H + top + bottom - dH*(kH-1) - 1) / sH + 1, same for W.
 */
typedef struct {
    int64_t kernel[2], pads[4], strides[2], dilations[2], group, offset_group;
} gs_deform_attrs;

/*
 * gs_deform_conv -- DeformConv (ai.onnx, since version 22), 2-D: Inputs and
 * Outputs.
 *
 *   X       device, (N, C, H, W).        x_shape host, 4 int64.
 *   W       device, (oC, C/group, kH, kW).
 *   oC      output channels.
 *   offset  device, (N, offset_group*kH*kW*2, oH, oW): for offset group o and
 *           kernel position k = kh*kW + kw, channel o*2K + 2k is the row (y)
 *           offset and o*2K + 2k + 1 the column (x) offset, K = kH*kW.
 *   B       device, (oC), or NULL for zeros.
 *   mask    device, (N, offset_group*kH*kW, oH, oW), or NULL for ones.
 *   Y       device output, (N, oC, oH, oW).
 *
 * Each sample is bilinear in X at (oh*sH - top + kh*dH + dy,
 * ow*sW - left + kw*dW + dx); taps outside X read 0.  fp32 contracts with
 * fp32 FMAs; bf16 and fp16 contract the sampled column tile on the tensor
 * cores where the shape allows (fp32 accumulation), else with fp32 FMAs.
 */
gs_status gs_deform_conv(const void *X, const int64_t *x_shape, const void *W, int64_t oC,
                         const void *offset, const void *B, const void *mask,
                         const gs_deform_attrs *attrs, gs_dtype dt, void *Y,
                         cudaStream_t stream);

/*
 * gs_deform_conv_workspace_size -- device workspace gs_deform_conv_ws asks
 * for: the packed W (rounded up to 256 bytes) and one channel-last slot of
 * (H*W + 1) * C elements per image.  0 means the call never uses a
 * workspace: fp32, or a shape outside the tensor-core path (group or
 * offset_group > 1, C or oC not a multiple of 16, oC > 256, or W too large
 * for shared memory).  Arguments as gs_deform_conv (no tensors needed);
 * `bytes` is a host output.
 */
gs_status gs_deform_conv_workspace_size(const int64_t *x_shape, int64_t oC,
                                        const gs_deform_attrs *attrs, gs_dtype dt, size_t *bytes);

/*
 * gs_deform_conv_ws -- gs_deform_conv with a caller-owned device workspace
 * (DeformConv, as above; the same values).
 *
 *   workspace        device, 256-byte aligned (GS_ERR_ALIGN), or NULL.
 *   workspace_bytes  its size.  With room for the packed W and at least one
 *                    image slot, fp16/bf16 calls on the tensor-core path pack
 *                    W once, copy X to channel-last order (as many images at a
 *                    time as it holds) and read each bilinear tap as 16-byte
 *                    runs of channels.  Otherwise it is gs_deform_conv.
 *
 * The workspace's contents on entry do not matter and are garbage on return.
 * Calls on different streams must not share a workspace while in flight.
 */
gs_status gs_deform_conv_ws(const void *X, const int64_t *x_shape, const void *W, int64_t oC,
                            const void *offset, const void *B, const void *mask,
                            const gs_deform_attrs *attrs, gs_dtype dt, void *workspace,
                            size_t workspace_bytes, void *Y, cudaStream_t stream);

/*
 * Resize -- Resize - 18 (Summary, Attributes, Inputs) on the same separable
 * sampler.  Attribute values follow the operator's names.
 */
typedef enum {
    GS_RS_HALF_PIXEL = 0, GS_RS_PYTORCH_HALF_PIXEL = 1, GS_RS_ALIGN_CORNERS = 2,
    GS_RS_ASYMMETRIC = 3, GS_RS_TF_CROP_AND_RESIZE = 4
} gs_resize_coord;
typedef enum {
    GS_RS_ROUND_PREFER_FLOOR = 0, GS_RS_ROUND_PREFER_CEIL = 1, GS_RS_FLOOR = 2, GS_RS_CEIL = 3
} gs_resize_nearest;
typedef enum { GS_RS_STRETCH = 0, GS_RS_NOT_LARGER = 1, GS_RS_NOT_SMALLER = 2 } gs_resize_keep;

typedef struct {
    gs_mode mode;                  /* nearest (the operator's default), linear, cubic      */
    gs_resize_coord coord;         /* coordinate_transformation_mode, default half_pixel   */
    gs_resize_nearest nearest_mode;/* default round_prefer_floor                           */
    float cubic_coeff_a;           /* default -0.75                                        */
    int exclude_outside;           /* 0 or 1                                               */
    float extrapolation_value;     /* tf_crop_and_resize outside the input                 */
    int antialias;                 /* 0 or 1: stretch linear / cubic by 1/scale downscaling */
    gs_resize_keep keep_aspect_ratio_policy;   /* applies to sizes                         */
} gs_resize_attrs;

/*
 * gs_resize_output_shape -- output extents of Resize (host only).
 *
 *   rank, x_shape  host: X's rank (1..8) and extents.
 *   axes, naxes    host: the axes scales / sizes / roi refer to (negative
 *                  counts from the back), or NULL / 0 for all axes in order.
 *   scales         host float[naxes or rank], > 0, or NULL.  Output extent
 *                  floor(in * (roi_end - roi_start) * scale).
 *   sizes          host int64[naxes or rank], >= 0, or NULL.  Exactly one of
 *                  scales and sizes.  keep_aspect_ratio_policy not_larger /
 *                  not_smaller take one common scale, min / max of
 *                  sizes[i] / in[axes[i]], and round scale * in halfway up.
 *   roi            host float[2 * (naxes or rank)]: starts then ends,
 *                  normalised; used only with tf_crop_and_resize (NULL: 0..1).
 *   y_shape        host output, rank int64.
 * Errors: GS_ERR_NULL, GS_ERR_RANK, GS_ERR_SHAPE (bad extents, repeated axis),
 * GS_ERR_ATTR (bad attribute, scale <= 0, both or neither of scales/sizes).
 */
gs_status gs_resize_output_shape(int rank, const int64_t *x_shape, const int64_t *axes, int naxes,
                                 const float *scales, const int64_t *sizes, const float *roi,
                                 const gs_resize_attrs *attrs, int64_t *y_shape);

/*
 * gs_resize -- Resize - 18 of X into Y (device buffers, `dt` for both).
 * Arguments as gs_resize_output_shape; Y must have that shape.
 *
 * Each axis maps output index o to x_original by the coordinate
 * transformation (with "scales" the given scale is used and the resized
 * length is n * scale, unfloored; with "sizes" scale = out / in), then takes
 * its taps: nearest (nearest_mode), linear (floor(x), floor(x) + 1), cubic
 * (floor(x) - 1 .. floor(x) + 2, Keys with cubic_coeff_a); antialias stretches
 * the linear / cubic filter by 1/scale when downscaling and rescales the
 * weights to sum 1; taps outside the axis read the edge value, or get weight
 * 0 with the rest rescaled when exclude_outside = 1.  The output is the sum
 * over the tensor product of the taps of the weights' product times X;
 * tf_crop_and_resize writes extrapolation_value wherever x_original leaves
 * [0, n - 1] on any axis.  Coordinates are formed in fp64; values accumulate
 * in fp32.
 *
 * Axes whose map is the identity (same extent, scale 1, whole roi) are
 * batched; the resized ones must be the last three or fewer
 * (GS_ERR_UNSUPPORTED otherwise), with at most 64 taps per output index
 * (antialias down to scale ~1/16 cubic, ~1/32 linear).
 */
gs_status gs_resize(const void *X, int rank, const int64_t *x_shape, const int64_t *axes,
                    int naxes, const float *scales, const int64_t *sizes, const float *roi,
                    const gs_resize_attrs *attrs, gs_dtype dt, void *Y, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
const char *gs_status_str(gs_status s);

/*
 * gs_device_status -- synchronises `stream`, then reports (and clears) the
 * library's device-side error word: GS_ERR_TIMEOUT if a bounded wait inside a
 * kernel gave up since the last call, GS_ERR_CUDA if the stream holds a CUDA
 * error, else GS_OK.  Kernels that give up a wait stop early and leave their
 * output incomplete; they never trap.
 */
gs_status gs_device_status(cudaStream_t stream);

/*
 * gs_test_bounded_wait_expires -- a test hook, not an operator (no page
 * defines it).  Enqueues one kernel on `stream` in which a single thread arms
 * an mbarrier for 16 bytes of transfer that no copy will ever deliver, then
 * waits on it with the same bounded wait the pipelined kernels use, with a
 * limit of `limit_ns` nanoseconds of the GPU's global timer.  The wait runs
 * out, records GS_ERR_TIMEOUT in the device error word and the kernel
 * returns, so a test can check that path without breaking a pipeline: the
 * next gs_device_status reports GS_ERR_TIMEOUT (and clears it).  Nothing is in
 * flight when the kernel leaves, so the context stays usable.  `limit_ns`
 * must lie in [1, 1e9] (GS_ERR_ATTR otherwise); nothing is allocated.
 */
gs_status gs_test_bounded_wait_expires(uint64_t limit_ns, cudaStream_t stream);

/* Library version, "major.minor.patch" (static storage). */
const char *gs_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GS_H */
