/*
 * oracle.c -- plain double-precision CPU definition of the spatial-transformer
 * sampling path: AffineGrid, GridSample, the two fused, DeformConv, and
 * Resize.
 *
 * TEST INFRASTRUCTURE ONLY.  This is the independent checker for the CUDA
 * library.  Only the tests, the smoke check and the bench's CPU-baseline leg
 * load it; the library never does.  It shares no code, header, table or
 * constant with the CUDA sources.
 *
 * Every value is computed in double precision with scalar loops, one output
 * element at a time, in the order the operator pages state the method.
 * Nothing is blocked, fused or reordered.  The only parallelism is an
 * optional OpenMP split of the independent output elements.
 *
 * Sources (the operator pages):
 *   [AG]  AffineGrid (ai.onnx, since version 20): description, the
 *         align_corners illustration, Inputs/Outputs.
 *   [GS]  GridSample - version 20 (and GridSample, version 22, same text):
 *         description, Inputs (grid coordinate order), Attributes
 *         (align_corners, mode, padding_mode).
 *   [DC]  DeformConv (ai.onnx, since version 22): Inputs (X, W, offset, B,
 *         mask) and Examples (kernel_shape, pads, offset_group).
 *   [RS]  Resize - 18: attribute cubic_coeff_a (names the cubic convolution
 *         kernel of Keys, "Equation (4)", with coefficient a); Summary,
 *         Attributes and Inputs for the Resize operator itself.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_LINEAR = 0, OR_NEAREST = 1, OR_CUBIC = 2 };
enum { OR_ZEROS = 0, OR_BORDER = 1, OR_REFLECTION = 2 };
#define OR_MAX_RANK 6

void or_set_num_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}

int or_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* The host's processors as OpenMP sees them (unaffected by OMP_NUM_THREADS,
   which launchers such as torchrun set to 1 for each rank). */
int or_num_procs(void) {
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* AffineGrid                                                                */
/* ------------------------------------------------------------------------ */

/* [AG] description: the positions are evenly spaced from -1 to 1 along each
 * axis.  align_corners=1: -1 and 1 are the centres of the corner pixels, so
 * pixel i of n sits at -1 + 2i/(n-1).  align_corners=0: -1 and 1 are the outer
 * edges of the corner pixels, so the n pixel centres sit at (2i+1)/n - 1.
 * Reading: an axis of length 1 has its single centre at 0 (the align_corners=1
 * formula is 0/0 there; 0 is also what the align_corners=0 formula gives). */
static double base_coord(int64_t i, int64_t n, int align_corners) {
    if (align_corners) {
        if (n == 1) return 0.0;
        return -1.0 + 2.0 * (double)i / (double)(n - 1);
    }
    return (2.0 * (double)i + 1.0) / (double)n - 1.0;
}

/* [AG] theta (N,2,3) or (N,3,4) applied to the homogeneous position
 * [x, y, (z,) 1]; the implicit last row [0 ... 0 1] is not stored.  The output
 * vector lists x' (width axis) first.  out_pos holds the r output spatial
 * indices outermost first: (h, w) or (d, h, w).  g receives r values. */
static void affine_point(const double *theta_n, int r, const int64_t *out_size,
                         const int64_t *out_pos, int align_corners, double *g) {
    double p[OR_MAX_RANK + 1];
    /* p[0] = x (innermost axis), p[1] = y, p[2] = z, p[r] = 1 */
    for (int k = 0; k < r; ++k) {
        int axis = r - 1 - k; /* spatial axis holding coordinate k */
        p[k] = base_coord(out_pos[axis], out_size[axis], align_corners);
    }
    p[r] = 1.0;
    for (int row = 0; row < r; ++row) {
        double s = 0.0;
        for (int k = 0; k <= r; ++k) s += theta_n[row * (r + 1) + k] * p[k];
        g[row] = s;
    }
}

/* [AG] Output grid (N, D_out..., r).  size = (N, C, spatial...) of length r+2. */
int or_affine_grid(const double *theta, int r, const int64_t *size, int align_corners,
                   double *grid) {
    if (r < 1 || r > OR_MAX_RANK) return -1;
    int64_t N = size[0], P = 1;
    for (int d = 0; d < r; ++d) P *= size[2 + d];
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t o = 0; o < P; ++o) {
            int64_t pos[OR_MAX_RANK], rem = o;
            for (int d = r - 1; d >= 0; --d) { pos[d] = rem % size[2 + d]; rem /= size[2 + d]; }
            affine_point(theta + n * r * (r + 1), r, size + 2, pos, align_corners,
                         grid + (n * P + o) * r);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* GridSample                                                                */
/* ------------------------------------------------------------------------ */

/* [GS] align_corners: with 1 the extrema -1 and 1 are the centres of the
 * corner pixels (0 and n-1); with 0 they are the outer corners of the corner
 * pixels (-0.5 and n-0.5).  The map is affine in the normalised value. */
static double unnormalize(double g, int64_t n, int align_corners) {
    if (align_corners) return (g + 1.0) / 2.0 * (double)(n - 1);
    return ((g + 1.0) * (double)n - 1.0) / 2.0;
}

/* [GS] padding_mode=reflection: a location outside [lo, hi] is mirrored at
 * the border it crossed, and "keeps being reflected until becoming in bound".
 * Repeated mirroring at lo and hi is periodic with period 2*(hi-lo); the
 * position inside one period is computed with fmod (exact in IEEE arithmetic),
 * and the second half of the period is the mirrored half.  A zero-width range
 * maps everything to lo. */
static double reflect(double x, double lo, double hi) {
    double span = hi - lo;
    if (span <= 0.0) return lo;
    double m = fmod(x - lo, 2.0 * span);
    if (m < 0.0) m += 2.0 * span;
    if (m > span) m = 2.0 * span - m;
    return lo + m;
}

static double clip(double x, double lo, double hi) {
    return x < lo ? lo : (x > hi ? hi : x);
}

/* The reflection borders: align_corners=1 mirrors at the centres of the
 * corner pixels (index -1 reads index 1, as the page's example says);
 * align_corners=0 mirrors at their outer edges, -0.5 and n-0.5. */
static double reflect_axis(double x, int64_t n, int align_corners) {
    if (align_corners) return reflect(x, 0.0, (double)(n - 1));
    return reflect(x, -0.5, (double)n - 0.5);
}

/* [RS] cubic_coeff_a names Keys' cubic convolution kernel with coefficient a:
 *   W(s) = (a+2)|s|^3 - (a+3)|s|^2 + 1            for |s| <= 1
 *   W(s) = a|s|^3 - 5a|s|^2 + 8a|s| - 4a           for 1 < |s| < 2
 *   W(s) = 0                                       otherwise.
 * [GS] mode=cubic uses it with a = -0.75 (the worked bicubic examples). */
static double keys(double s, double a) {
    s = fabs(s);
    if (s <= 1.0) return (a + 2.0) * s * s * s - (a + 3.0) * s * s + 1.0;
    if (s < 2.0) return a * s * s * s - 5.0 * a * s * s + 8.0 * a * s - 4.0 * a;
    return 0.0;
}

/* Bound for converting a coordinate to an integer index.  Anything beyond it
 * is so far outside the image that every tap is out of range (zeros) or sits
 * on the border; the bound only keeps the conversion defined (it also sends
 * NaN to the low side). */
#define OR_COORD_LIMIT 1.0e15

static int64_t to_index(double f) {
    if (!(f > -OR_COORD_LIMIT)) f = -OR_COORD_LIMIT;
    if (f > OR_COORD_LIMIT) f = OR_COORD_LIMIT;
    return (int64_t)f;
}

/* Taps of one spatial axis: indices (possibly out of range) and 1-D weights.
 *
 * [GS] mode: nearest takes the nearest index, ties to the even index; linear
 * takes floor(x) and floor(x)+1 with weights 1-t and t (t = x - floor(x));
 * cubic takes floor(x)-1 .. floor(x)+2 with Keys weights at distances t+1,
 * t, 1-t, 2-t.
 * [GS] padding_mode: for linear and nearest the coordinate itself is padded
 * first (border: clip to [0, n-1]; reflection: mirror into range, then clip).
 * For cubic the coordinate is left as it is and each of the four tap indices
 * is padded instead (border: clamp; reflection: mirror, then clip) -- the
 * reading the pages' Resize cubic examples support, since their printed
 * border values need edge-replicated taps at an unclamped position.
 * Under zeros padding nothing is moved; a tap outside [0, n-1] reads 0, which
 * the caller applies. */
static int axis_taps(double g, int64_t n, int mode, int pad, int align_corners, double a,
                     int64_t idx[4], double w[4]) {
    double x = unnormalize(g, n, align_corners);
    if (mode != OR_CUBIC) {
        if (pad == OR_BORDER) {
            x = clip(x, 0.0, (double)(n - 1));
        } else if (pad == OR_REFLECTION) {
            x = clip(reflect_axis(x, n, align_corners), 0.0, (double)(n - 1));
        }
    }
    if (mode == OR_NEAREST) {
        /* nearbyint rounds half to even under the default rounding mode */
        idx[0] = to_index(nearbyint(x));
        w[0] = 1.0;
        return 1;
    }
    double f = floor(x);
    double t = x - f;
    int64_t i0 = to_index(f);
    if (mode == OR_LINEAR) {
        idx[0] = i0;     w[0] = 1.0 - t;
        idx[1] = i0 + 1; w[1] = t;
        return 2;
    }
    for (int k = 0; k < 4; ++k) {
        int64_t j = i0 - 1 + k;
        if (pad == OR_BORDER) {
            j = j < 0 ? 0 : (j > n - 1 ? n - 1 : j);
        } else if (pad == OR_REFLECTION) {
            j = (int64_t)clip(reflect_axis((double)j, n, align_corners), 0.0, (double)(n - 1));
        }
        idx[k] = j;
        w[k] = keys(t + 1.0 - (double)k, a);
    }
    return 4;
}

/* [GS] one output value: the sum over the tensor product of the per-axis
 * taps of (product of 1-D weights) * X[n, c, tap], a tap outside X reading 0.
 * X_nc points at the (n, c) slab; in_size holds the r input extents,
 * outermost first; g holds the grid vector, innermost axis first. */
static double sample_point(const double *X_nc, int r, const int64_t *in_size, const double *g,
                           int mode, int pad, int align_corners, double a) {
    int64_t idx[OR_MAX_RANK][4];
    double w[OR_MAX_RANK][4];
    int nt[OR_MAX_RANK];
    for (int d = 0; d < r; ++d) {
        /* [GS] grid: the location vector lists the innermost axis first */
        nt[d] = axis_taps(g[r - 1 - d], in_size[d], mode, pad, align_corners, a, idx[d], w[d]);
    }
    int k[OR_MAX_RANK] = {0};
    double acc = 0.0;
    for (;;) {
        double weight = 1.0;
        int64_t off = 0;
        int inside = 1;
        for (int d = 0; d < r; ++d) {
            int64_t j = idx[d][k[d]];
            if (j < 0 || j >= in_size[d]) inside = 0;
            weight *= w[d][k[d]];
            off = off * in_size[d] + j;
        }
        if (inside) acc += weight * X_nc[off];
        int d = r - 1;
        while (d >= 0 && ++k[d] == nt[d]) k[d--] = 0;
        if (d < 0) break;
    }
    return acc;
}

/* Shape helpers: x_shape = (N, C, in...), grid (N, out..., r), Y (N, C, out...). */
static int64_t prod(const int64_t *v, int r) {
    int64_t p = 1;
    for (int d = 0; d < r; ++d) p *= v[d];
    return p;
}

/* One Y element by flat index into (N, C, out...), with the grid as a tensor. */
static double grid_sample_elem(const double *X, const int64_t *x_shape, int r, const double *grid,
                               const int64_t *out_spatial, int mode, int pad, int ac, double a,
                               int64_t flat) {
    int64_t C = x_shape[1];
    int64_t P_out = prod(out_spatial, r), P_in = prod(x_shape + 2, r);
    int64_t o = flat % P_out;
    int64_t nc = flat / P_out;
    int64_t n = nc / C;
    return sample_point(X + nc * P_in, r, x_shape + 2, grid + (n * P_out + o) * r, mode, pad, ac, a);
}

int or_grid_sample(const double *X, const int64_t *x_shape, int r, const double *grid,
                   const int64_t *out_spatial, int mode, int pad, int align_corners,
                   double cubic_a, double *Y) {
    if (r < 1 || r > OR_MAX_RANK) return -1;
    int64_t total = x_shape[0] * x_shape[1] * prod(out_spatial, r);
#pragma omp parallel for schedule(static)
    for (int64_t f = 0; f < total; ++f)
        Y[f] = grid_sample_elem(X, x_shape, r, grid, out_spatial, mode, pad, align_corners,
                                cubic_a, f);
    return 0;
}

/* The same, at the listed flat indices of Y only (for spot checks of large outputs). */
int or_grid_sample_at(const double *X, const int64_t *x_shape, int r, const double *grid,
                      const int64_t *out_spatial, int mode, int pad, int align_corners,
                      double cubic_a, const int64_t *flat_idx, int64_t count, double *out) {
    if (r < 1 || r > OR_MAX_RANK) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        out[i] = grid_sample_elem(X, x_shape, r, grid, out_spatial, mode, pad, align_corners,
                                  cubic_a, flat_idx[i]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* AffineGrid feeding GridSample (the spatial transformer)                   */
/* ------------------------------------------------------------------------ */

/* GridSample(X, AffineGrid(theta, size)) with the grid kept in double
 * precision between the two: the fused operation never rounds the grid to
 * the I/O type.  size = (N, C, out...) is AffineGrid's size input; its
 * spatial part is the output extent.  One Y element by flat index. */
static double affine_sample_elem(const double *theta, const int64_t *size, int r, const double *X,
                                 const int64_t *x_shape, int mode, int pad, int ac, double a,
                                 int64_t flat) {
    int64_t C = x_shape[1];
    const int64_t *out_sz = size + 2;
    int64_t P_out = prod(out_sz, r), P_in = prod(x_shape + 2, r);
    int64_t o = flat % P_out;
    int64_t nc = flat / P_out;
    int64_t n = nc / C;
    int64_t pos[OR_MAX_RANK], rem = o;
    for (int d = r - 1; d >= 0; --d) { pos[d] = rem % out_sz[d]; rem /= out_sz[d]; }
    double g[OR_MAX_RANK];
    affine_point(theta + n * r * (r + 1), r, out_sz, pos, ac, g);
    return sample_point(X + nc * P_in, r, x_shape + 2, g, mode, pad, ac, a);
}

int or_affine_sample(const double *theta, const int64_t *size, int r, const double *X,
                     const int64_t *x_shape, int mode, int pad, int align_corners, double cubic_a,
                     double *Y) {
    if (r < 1 || r > OR_MAX_RANK) return -1;
    int64_t total = x_shape[0] * x_shape[1] * prod(size + 2, r);
#pragma omp parallel for schedule(static)
    for (int64_t f = 0; f < total; ++f)
        Y[f] = affine_sample_elem(theta, size, r, X, x_shape, mode, pad, align_corners, cubic_a, f);
    return 0;
}

int or_affine_sample_at(const double *theta, const int64_t *size, int r, const double *X,
                        const int64_t *x_shape, int mode, int pad, int align_corners,
                        double cubic_a, const int64_t *flat_idx, int64_t count, double *out) {
    if (r < 1 || r > OR_MAX_RANK) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        out[i] = affine_sample_elem(theta, size, r, X, x_shape, mode, pad, align_corners, cubic_a,
                                    flat_idx[i]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* DeformConv (2-D)                                                          */
/* ------------------------------------------------------------------------ */

/* [DC] offset: "use linear interpolation for fractional offset values;
 * sampling locations outside of the padded input tensor give zero."  The
 * pads only move the kernel's anchor; X itself is the unpadded input, and a
 * bilinear tap that falls outside it reads 0 (the padded border holds zeros
 * too).  y is the row position, x the column position, in pixels. */
static double bilinear_zero(const double *X_nc, int64_t H, int64_t W, double y, double x) {
    double fy = floor(y), fx = floor(x);
    double ty = y - fy, tx = x - fx;
    int64_t y0 = to_index(fy), x0 = to_index(fx);
    double acc = 0.0;
    for (int dy = 0; dy < 2; ++dy) {
        for (int dx = 0; dx < 2; ++dx) {
            int64_t yy = y0 + dy, xx = x0 + dx;
            if (yy < 0 || yy >= H || xx < 0 || xx >= W) continue;
            double wgt = (dy ? ty : 1.0 - ty) * (dx ? tx : 1.0 - tx);
            acc += wgt * X_nc[yy * W + xx];
        }
    }
    return acc;
}

/* Attributes: kernel (kH, kW), pads (top, left, bottom, right), strides
 * (sH, sW), dilations (dH, dW), group, offset_group.  The page's Attributes
 * section is missing; the reading follows ONNX Conv: stride 1, dilation 1,
 * group 1 by default, pads listed begins then ends, and
 *   oH = floor((H + pad_top + pad_bottom - dH*(kH-1) - 1) / sH) + 1.
 * [DC] W is (oC, C/group, kH, kW); offset is (N, offset_group*kH*kW*2, oH, oW)
 * with, for offset group o and kernel position k = kh*kW + kw (row-major),
 * channel o*2K + 2k holding the row offset and o*2K + 2k + 1 the column
 * offset (the order the worked examples fix); mask is
 * (N, offset_group*kH*kW, oH, oW) and multiplies the sampled value; B is
 * (oC).  B and mask may be NULL (zeros and ones). */
typedef struct {
    int64_t kernel[2], pads[4], strides[2], dilations[2], group, offset_group;
} or_deform_attrs;

int64_t or_deform_out_extent(int64_t in, int64_t k, int64_t pad_begin, int64_t pad_end,
                             int64_t stride, int64_t dil) {
    return (in + pad_begin + pad_end - dil * (k - 1) - 1) / stride + 1;
}

static double deform_elem(const double *X, const int64_t *x_shape, const double *Wt, int64_t oC,
                          const double *offset, const double *B, const double *mask,
                          const or_deform_attrs *at, int64_t flat) {
    int64_t N = x_shape[0], C = x_shape[1], H = x_shape[2], Wd = x_shape[3];
    (void)N;
    int64_t kH = at->kernel[0], kW = at->kernel[1], K = kH * kW;
    int64_t oH = or_deform_out_extent(H, kH, at->pads[0], at->pads[2], at->strides[0],
                                      at->dilations[0]);
    int64_t oW = or_deform_out_extent(Wd, kW, at->pads[1], at->pads[3], at->strides[1],
                                      at->dilations[1]);
    int64_t ow = flat % oW;
    int64_t oh = (flat / oW) % oH;
    int64_t oc = (flat / (oW * oH)) % oC;
    int64_t n = flat / (oW * oH * oC);
    int64_t Cg = C / at->group;            /* input channels per group */
    int64_t oCg = oC / at->group;          /* output channels per group */
    int64_t Cog = C / at->offset_group;    /* input channels per offset group */
    int64_t g = oc / oCg;
    double acc = B ? B[oc] : 0.0;
    for (int64_t ci = 0; ci < Cg; ++ci) {
        int64_t c = g * Cg + ci;
        int64_t og = c / Cog;
        const double *X_nc = X + (n * C + c) * H * Wd;
        for (int64_t kh = 0; kh < kH; ++kh) {
            for (int64_t kw = 0; kw < kW; ++kw) {
                int64_t k = kh * kW + kw;
                int64_t plane = oH * oW, pix = oh * oW + ow;
                double dy = offset[((n * at->offset_group + og) * 2 * K + 2 * k) * plane + pix];
                double dx = offset[((n * at->offset_group + og) * 2 * K + 2 * k + 1) * plane + pix];
                double m = mask ? mask[((n * at->offset_group + og) * K + k) * plane + pix] : 1.0;
                double y = (double)(oh * at->strides[0] - at->pads[0] + kh * at->dilations[0]) + dy;
                double x = (double)(ow * at->strides[1] - at->pads[1] + kw * at->dilations[1]) + dx;
                double v = bilinear_zero(X_nc, H, Wd, y, x) * m;
                acc += Wt[((oc * Cg + ci) * kH + kh) * kW + kw] * v;
            }
        }
    }
    return acc;
}

int or_deform_conv(const double *X, const int64_t *x_shape, const double *Wt, int64_t oC,
                   const double *offset, const double *B, const double *mask,
                   const or_deform_attrs *at, double *Y) {
    int64_t oH = or_deform_out_extent(x_shape[2], at->kernel[0], at->pads[0], at->pads[2],
                                      at->strides[0], at->dilations[0]);
    int64_t oW = or_deform_out_extent(x_shape[3], at->kernel[1], at->pads[1], at->pads[3],
                                      at->strides[1], at->dilations[1]);
    int64_t total = x_shape[0] * oC * oH * oW;
#pragma omp parallel for schedule(static)
    for (int64_t f = 0; f < total; ++f)
        Y[f] = deform_elem(X, x_shape, Wt, oC, offset, B, mask, at, f);
    return 0;
}

int or_deform_conv_at(const double *X, const int64_t *x_shape, const double *Wt, int64_t oC,
                      const double *offset, const double *B, const double *mask,
                      const or_deform_attrs *at, const int64_t *flat_idx, int64_t count,
                      double *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        out[i] = deform_elem(X, x_shape, Wt, oC, offset, B, mask, at, flat_idx[i]);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Resize                                                                    */
/* ------------------------------------------------------------------------ */

/* [RS] Resize - 18 (Summary, Attributes, Inputs).  Every axis is mapped on its
 * own; the output value is the sum, over the tensor product of the per-axis
 * taps, of the product of the 1-D weights times X at the tap.  Readings (the
 * helper functions the page's examples call are not printed, so these are
 * taken from the attribute text and checked against the printed outputs):
 *  - a tap index outside [0, n-1] reads the edge value (index clamped), except
 *    that exclude_outside=1 gives such taps weight 0 and rescales the rest to
 *    sum 1;
 *  - linear: taps floor(x), floor(x)+1, weights 1-t, t;  cubic: taps
 *    floor(x)-1 .. floor(x)+2, Keys weights at distances t+1, t, 1-t, 2-t;
 *  - antialias with scale < 1 stretches the filter by 1/scale: the taps are
 *    the integer offsets k from floor(x) where the stretched filter can be
 *    nonzero (linear: k = s .. 1-s with s = floor(-1/scale)+1; cubic:
 *    k = s .. 1-s with s = floor(-2/scale)+1), weight filter((k-t)*scale),
 *    rescaled to sum 1;
 *  - with "scales" given the coordinate maps use that scale, and
 *    length_resized = n_in * scale, unfloored; with "sizes" given,
 *    scale = length_resized / length_original with length_resized the size;
 *  - tf_crop_and_resize: a coordinate outside [0, n-1] on any axis makes the
 *    whole output element extrapolation_value. */
enum { RS_HALF_PIXEL = 0, RS_PYTORCH_HALF_PIXEL = 1, RS_ALIGN_CORNERS = 2, RS_ASYMMETRIC = 3,
       RS_TF_CROP_AND_RESIZE = 4 };
enum { RS_ROUND_PREFER_FLOOR = 0, RS_ROUND_PREFER_CEIL = 1, RS_FLOOR = 2, RS_CEIL = 3 };
enum { RS_STRETCH = 0, RS_NOT_LARGER = 1, RS_NOT_SMALLER = 2 };
#define RS_MAX_TAPS 4096

/* [RS] coordinate_transformation_mode: x_original of output index x_resized. */
static double rs_source_coord(double xr, int64_t n_in, int64_t n_out, double scale,
                              double length_resized, double start, double end, int coord) {
    switch (coord) {
        case RS_PYTORCH_HALF_PIXEL:
            return n_out > 1 ? (xr + 0.5) / scale - 0.5 : 0.0;
        case RS_ALIGN_CORNERS:
            /* a single output position has no second corner: it sits at 0 */
            return length_resized > 1.0 ? xr * (double)(n_in - 1) / (length_resized - 1.0) : 0.0;
        case RS_ASYMMETRIC:
            return xr / scale;
        case RS_TF_CROP_AND_RESIZE:
            if (n_out > 1)
                return start * (double)(n_in - 1) +
                       xr * (end - start) * (double)(n_in - 1) / (double)(n_out - 1);
            return 0.5 * (start + end) * (double)(n_in - 1);
        default: /* half_pixel */
            return (xr + 0.5) / scale - 0.5;
    }
}

/* [RS] nearest_mode: the nearest pixel of x_original. */
static double rs_nearest(double x, int nearest_mode) {
    switch (nearest_mode) {
        case RS_ROUND_PREFER_CEIL: return floor(x + 0.5);   /* halfway rounds up */
        case RS_FLOOR: return floor(x);
        case RS_CEIL: return ceil(x);
        default: return ceil(x - 0.5);                     /* halfway rounds down */
    }
}

/* Taps of one axis for output index o; returns the tap count, or -1 when the
 * element takes extrapolation_value (tf_crop_and_resize outside the input). */
static int rs_axis_taps(int64_t o, int64_t n_in, int64_t n_out, double scale,
                        double length_resized, double start, double end, int coord, int mode,
                        int nearest_mode, double a, int exclude_outside, int antialias,
                        int64_t *idx, double *w) {
    const double x = rs_source_coord((double)o, n_in, n_out, scale, length_resized, start, end,
                                     coord);
    if (coord == RS_TF_CROP_AND_RESIZE && (x < 0.0 || x > (double)(n_in - 1))) return -1;
    int cnt;
    if (mode == OR_NEAREST) {
        idx[0] = to_index(rs_nearest(x, nearest_mode));
        w[0] = 1.0;
        cnt = 1;
    } else {
        const double f = floor(x), t = x - f;
        const int64_t i0 = to_index(f);
        const double s = (antialias && scale < 1.0) ? scale : 1.0;
        /* first offset from floor(x) at which the (stretched) filter can be nonzero */
        const double reach = mode == OR_LINEAR ? 1.0 : 2.0;
        const int64_t k0 = (int64_t)floor(-reach / s) + 1;
        const int64_t k1 = 1 - k0;   /* last offset, the mirror image of k0 */
        if (k1 - k0 + 1 > RS_MAX_TAPS) return -2;
        cnt = 0;
        double sum = 0.0;
        for (int64_t k = k0; k <= k1; ++k) {
            const double d = ((double)k - t) * s;
            const double wk = mode == OR_LINEAR ? fmax(0.0, 1.0 - fabs(d)) : keys(d, a);
            idx[cnt] = i0 + k;
            w[cnt] = wk;
            sum += wk;
            ++cnt;
        }
        if (s < 1.0) {
            for (int k = 0; k < cnt; ++k) w[k] /= sum;
        }
    }
    if (exclude_outside) {
        double sum = 0.0;
        for (int k = 0; k < cnt; ++k) {
            if (idx[k] < 0 || idx[k] > n_in - 1) w[k] = 0.0;
            sum += w[k];
        }
        if (sum != 0.0)
            for (int k = 0; k < cnt; ++k) w[k] /= sum;
    }
    for (int k = 0; k < cnt; ++k) idx[k] = idx[k] < 0 ? 0 : (idx[k] > n_in - 1 ? n_in - 1 : idx[k]);
    return cnt;
}

/* [RS] output extents and per-axis coordinate parameters from scales or sizes
 * (one of them, for the axes listed in `axes`, or for all axes when naxes is
 * 0).  keep_aspect_ratio_policy applies to sizes: not_larger / not_smaller
 * take one common scale, the smallest / largest of sizes[i] / in[axes[i]],
 * and round scale * in to the nearest integer, halfway up.  Writes out_shape,
 * scale and length_resized per axis (rank entries); returns 0, or -1 on a bad
 * argument. */
int or_resize_shape(int rank, const int64_t *in_shape, const int64_t *axes, int naxes,
                    const double *scales, const int64_t *sizes, const double *roi, int coord,
                    int keep_policy, int64_t *out_shape, double *scale, double *length_resized,
                    double *roi_start, double *roi_end) {
    if (rank < 1 || rank > OR_MAX_RANK || (!scales && !sizes) || (scales && sizes)) return -1;
    int ax[OR_MAX_RANK];
    const int na = naxes > 0 ? naxes : rank;
    for (int i = 0; i < na; ++i) {
        int d = naxes > 0 ? (int)axes[i] : i;
        if (d < 0) d += rank;
        if (d < 0 || d >= rank) return -1;
        ax[i] = d;
    }
    for (int d = 0; d < rank; ++d) {
        out_shape[d] = in_shape[d];
        scale[d] = 1.0;
        length_resized[d] = (double)in_shape[d];
        roi_start[d] = 0.0;
        roi_end[d] = 1.0;
    }
    if (roi && coord == RS_TF_CROP_AND_RESIZE) {
        for (int i = 0; i < na; ++i) {
            roi_start[ax[i]] = roi[i];
            roi_end[ax[i]] = roi[na + i];
        }
    }
    if (scales) {
        for (int i = 0; i < na; ++i) {
            const int d = ax[i];
            if (!(scales[i] > 0.0)) return -1;
            const double len = (double)in_shape[d] * (roi_end[d] - roi_start[d]) * scales[i];
            out_shape[d] = (int64_t)floor(len);
            scale[d] = scales[i];
            length_resized[d] = len;
        }
        return 0;
    }
    double common = 0.0;
    if (keep_policy != RS_STRETCH) {
        for (int i = 0; i < na; ++i) {
            const double r = (double)sizes[i] / (double)in_shape[ax[i]];
            if (i == 0 || (keep_policy == RS_NOT_LARGER ? r < common : r > common)) common = r;
        }
    }
    for (int i = 0; i < na; ++i) {
        const int d = ax[i];
        const int64_t o = keep_policy == RS_STRETCH
                              ? sizes[i]
                              : (int64_t)floor(common * (double)in_shape[d] + 0.5);
        if (o < 0) return -1;
        out_shape[d] = o;
        scale[d] = in_shape[d] > 0 ? (double)o / (double)in_shape[d] : 1.0;
        length_resized[d] = (double)o;
    }
    return 0;
}

/* [RS] Y = Resize(X): direct summation over the tensor product of the taps. */
int or_resize(const double *X, int rank, const int64_t *in_shape, const int64_t *out_shape,
              const double *scale, const double *length_resized, const double *roi_start,
              const double *roi_end, int mode, int coord, int nearest_mode, double a,
              int exclude_outside, double extrapolation_value, int antialias, double *Y) {
    if (rank < 1 || rank > OR_MAX_RANK) return -1;
    const int64_t total = prod(out_shape, rank);
    int bad = 0;
#pragma omp parallel reduction(| : bad)
    {
        /* per-thread tap buffers */
        int64_t *idx_buf = (int64_t *)malloc(sizeof(int64_t) * RS_MAX_TAPS * OR_MAX_RANK);
        double *w_buf = (double *)malloc(sizeof(double) * RS_MAX_TAPS * OR_MAX_RANK);
        if (!idx_buf || !w_buf) bad = 1;
#pragma omp for schedule(dynamic, 64)
        for (int64_t e = 0; e < total; ++e) {
            if (!idx_buf || !w_buf) continue;
            int64_t o[OR_MAX_RANK];
            int64_t rem = e;
            for (int d = rank - 1; d >= 0; --d) {
                o[d] = rem % out_shape[d];
                rem /= out_shape[d];
            }
            int cnt[OR_MAX_RANK];
            int extrap = 0, err = 0;
            for (int d = 0; d < rank && !extrap && !err; ++d) {
                cnt[d] = rs_axis_taps(o[d], in_shape[d], out_shape[d], scale[d], length_resized[d],
                                      roi_start[d], roi_end[d], coord, mode, nearest_mode, a,
                                      exclude_outside, antialias, idx_buf + d * RS_MAX_TAPS,
                                      w_buf + d * RS_MAX_TAPS);
                if (cnt[d] == -1) extrap = 1;
                if (cnt[d] < -1) err = 1;
            }
            double acc = 0.0;
            if (extrap) {
                acc = extrapolation_value;
            } else if (!err) {
                int k[OR_MAX_RANK] = {0};
                for (;;) {
                    double wt = 1.0;
                    int64_t off = 0;
                    for (int d = 0; d < rank; ++d) {
                        wt *= w_buf[d * RS_MAX_TAPS + k[d]];
                        off = off * in_shape[d] + idx_buf[d * RS_MAX_TAPS + k[d]];
                    }
                    acc += wt * X[off];
                    int d = rank - 1;
                    while (d >= 0 && ++k[d] == cnt[d]) k[d--] = 0;
                    if (d < 0) break;
                }
            }
            bad |= err;
            Y[e] = acc;
        }
        free(idx_buf);
        free(w_buf);
    }
    return bad ? -1 : 0;
}
