// gs_vol_tma.cuh -- fused AffineGrid+GridSample, 3-D, trilinear and nearest,
// with each channel's input box brought in by the tensor memory accelerator.
//
// AffineGrid (description) makes every output position an affine function of
// its index, and GridSample - version 20 (description; Attributes mode,
// padding_mode, align_corners) samples X there.  So the taps of a tile of
// output positions lie in one axis-aligned input box, found from the tile's
// eight corners.  Persistent blocks (two per SM) take tiles round robin:
//  - per tile, warp 0 builds the image's affine map (24.40 fixed point) and
//    three threads find the box; the tile then picks the smallest of a
//    family of tensor maps over X whose box covers it (the maps differ in
//    their box's rows and planes), and the ring holds as many stages of that
//    box as fit;
//  - thread 0 issues one cp.async.bulk.tensor.3d per channel (zeros outside
//    X come from the copy), completing on that stage's "full" mbarrier;
//  - every thread interpolates its four positions from the stage (eight
//    shared-memory loads at fixed offsets per position, packed FMAs), then
//    its warp arrives on the stage's "empty" mbarrier; thread 0 refills the
//    stage with channel c + S once all eight warps have arrived.
// A tile that no map covers, or a map that needs fp64 positions, gathers
// from global memory with sample_kernel's taps.
#pragma once

#include "gs_ptx.cuh"
#include "gs_tma.cuh"
#include "gs_vol.cuh"

namespace gs {

constexpr int kVtThreads = 256;
constexpr int kVtWarps = kVtThreads / 32;
constexpr int kVtPPT = 4;                          // output positions per thread
constexpr int kVtTile = kVtThreads * kVtPPT;       // output positions per tile
constexpr int kVtMaps = 9;                         // tensor maps (box sizes) per launch
constexpr int kVtMaxStages = 8;
constexpr int kVtRingBytes = 96 * 1024;            // two blocks per SM

struct VolTmaParams {
    int tz, ty, tx;          // tile extents along output depth, rows, columns (tx: 8, 16 or 32)
    int tiles_y, tiles_x;    // tiles along output rows and columns
    int tiles;               // tiles per image
    int total;               // N * tiles
    int nmaps;               // maps in use, ordered by box bytes
    int box[kVtMaps][3];     // box extents of map k: planes, rows, columns (elements)
};

struct VolTmaMaps {
    CUtensorMap m[kVtMaps];   // X as (W, H, D, N*C), innermost first
};

template <typename T, int MODE>
__global__ void __launch_bounds__(kVtThreads, 2)
vol_tma_kernel(const T *__restrict__ X, const T *__restrict__ theta, T *__restrict__ Y,
               const SampleParams P, const VolTmaParams V, const __grid_constant__ VolTmaMaps maps) {
    constexpr int K = MODE == MODE_NEAREST ? 1 : 2;
    constexpr int NT = K * K * K;
    constexpr int E = (int)sizeof(T);
    constexpr int EPC = 16 / E;   // elements per 16 bytes (the box's x origin is a multiple)
    extern __shared__ __align__(128) unsigned char vt_smem[];
    __shared__ AffineMap s_map;
    __shared__ int s_lo[3], s_k, s_stages;
    __shared__ __align__(8) uint64_t full[kVtMaxStages], empty[kVtMaxStages];

    const SampleArgs &a = P.a;
    const int tid = threadIdx.x, lane = tid & 31;
    unsigned *err = a.err;
    // the ring starts on a 128-byte boundary (the launch adds 128 bytes of slack)
    unsigned char *ring = vt_smem + ((128u - (smem_u32(vt_smem) & 127u)) & 127u);
    if (tid == 0) {
        for (int s = 0; s < kVtMaxStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kVtWarps);
        }
        fence_mbar_init();
        for (int k = 0; k < V.nmaps; ++k) tma_prefetch_map(&maps.m[k]);
    }
    __syncthreads();

    // Use u of a stage completes its full phase u (the copy landed) and its
    // empty phase u (every warp read it).  Bit s of upar is the parity of the
    // uses of stage s so far (the same in every thread); thread 0 keeps the
    // parity of the copies it issued per stage in ipar, and in iany which
    // stages have had one.
    uint32_t upar = 0, ipar = 0, iany = 0;
    bool bad = false;   // a bounded wait gave up
    int map_n = -1;     // the image whose affine map s_map holds
    const int Ho = a.out[1], Wo = a.out[2];
    const int tx_shift = V.tx == 32 ? 5 : (V.tx == 16 ? 4 : 3);
    const int64_t in_plane = a.in_plane, out_plane = a.out_plane;

    for (int tile_id = blockIdx.x; tile_id < V.total; tile_id += gridDim.x) {
        const int n = tile_id / V.tiles;
        const int tile = tile_id - n * V.tiles;
        const int tzi = tile / (V.tiles_y * V.tiles_x);
        const int trem = tile - tzi * (V.tiles_y * V.tiles_x);
        const int tyi = trem / V.tiles_x;
        const int txi = trem - tyi * V.tiles_x;
        const int oz0 = tzi * V.tz, oy0 = tyi * V.ty, ox0 = txi * V.tx;
        // the previous tile's readers of the map, the box and the stages are done
        if (__syncthreads_or(bad)) break;
        if (n != map_n) {   // consecutive tiles of a block are mostly of one image
            if (tid < 32) build_affine_map_warp<T, 3>(theta + (int64_t)n * 12, P, s_map);
            map_n = n;
            __syncthreads();
        }
        if (tid < 32) {
            // box of input indices: lane 8d + ci takes corner ci of the tile
            // on axis d (lanes 24..31 repeat axis 2); min and max over the
            // eight corners by shuffles within each group of eight lanes
            const int d = min(lane >> 3, 2), ci = lane & 7;
            const int o_hi[3] = {min(oz0 + V.tz, a.out[0]) - 1, min(oy0 + V.ty, Ho) - 1,
                                 min(ox0 + V.tx, Wo) - 1};
            const int o_lo[3] = {oz0, oy0, ox0};
            int64_t qq = s_map.cst_q[d];
#pragma unroll
            for (int jj = 0; jj < 3; ++jj)
                qq += s_map.coef_q[d][jj] * (int64_t)(((ci >> jj) & 1) ? o_hi[jj] : o_lo[jj]);
            qq >>= 8;
            int64_t qmin = qq, qmax = qq;
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                const int64_t a0 = __shfl_xor_sync(0xffffffffu, qmin, o);
                const int64_t a1 = __shfl_xor_sync(0xffffffffu, qmax, o);
                qmin = a0 < qmin ? a0 : qmin;
                qmax = a1 > qmax ? a1 : qmax;
            }
            const Axis &A = P.ax[d];
            if (a.pad == PAD_REFLECTION && (qmin < A.lo_q || qmax > A.lo_q + A.span_q)) {
                qmin = 0;   // folded positions can land anywhere on the axis
                qmax = A.hi_q;
            } else {
                qmin = vol_pad(qmin, A, a.pad);
                qmax = vol_pad(qmax, A, a.pad);
            }
            int lo = vol_index<MODE>(qmin, A.n);
            const int hi = vol_index<MODE>(qmax, A.n) + (K - 1);
            if (d == 2) lo = (lo >= 0 ? lo : lo - (EPC - 1)) / EPC * EPC;   // 16-byte origin
            int blo[3], ext[3];
#pragma unroll
            for (int dd = 0; dd < 3; ++dd) {
                blo[dd] = __shfl_sync(0xffffffffu, lo, 8 * dd);
                ext[dd] = __shfl_sync(0xffffffffu, hi - lo + 1, 8 * dd);
            }
            if (lane == 0) {
                // the smallest box that covers the tile, and the stages that fit
                int k = -1, stages = 0;
                if (!s_map.wide) {
                    for (int m = 0; m < V.nmaps && k < 0; ++m)
                        if (V.box[m][0] >= ext[0] && V.box[m][1] >= ext[1] && V.box[m][2] >= ext[2])
                            k = m;
                    if (k >= 0) {
                        const int bytes = (V.box[k][0] * V.box[k][1] * V.box[k][2] * E + 127) & ~127;
                        stages = min(kVtMaxStages, kVtRingBytes / bytes);
                        if (stages < 2) stages = 0;
                    }
                }
#pragma unroll
                for (int dd = 0; dd < 3; ++dd) s_lo[dd] = blo[dd];
                s_k = k;
                s_stages = stages;
            }
        }
        __syncthreads();
        const int S = s_stages;
        const T *__restrict__ Xn = X + (int64_t)n * a.C * in_plane;
        T *__restrict__ Yc = Y + (int64_t)n * a.C * out_plane;

        if (S == 0) {
            // gather from global memory, one position at a time
            for (int j = 0; j < kVtPPT; ++j) {
                const int p = tid + j * kVtThreads;
                const int row = p >> tx_shift;
                const int oz = oz0 + row / V.ty, oy = oy0 + row % V.ty, ox = ox0 + (p & (V.tx - 1));
                if (row >= V.tz * V.ty || oz >= a.out[0] || oy >= Ho || ox >= Wo) continue;
                AxisTaps<MODE> tp[3];
                const int opos[3] = {oz, oy, ox};
#pragma unroll
                for (int d = 0; d < 3; ++d) {
                    int64_t xq;
                    if (!s_map.wide) {
                        int64_t acc = s_map.cst_q[d];
#pragma unroll
                        for (int jj = 0; jj < 3; ++jj) acc += s_map.coef_q[d][jj] * (int64_t)opos[jj];
                        xq = acc >> 8;
                    } else {
                        double x = s_map.cst[d];
#pragma unroll
                        for (int jj = 0; jj < 3; ++jj) x += s_map.coef[d][jj] * (double)opos[jj];
                        xq = pos_to_q(x, P.ax[d], a.pad);
                    }
                    make_taps<MODE>(xq, P.ax[d], a.pad, a.ac, a.a, tp[d]);
                }
                int off_hi[16];
                outer_offsets<3, MODE>(tp, a, off_hi);
                const int64_t yo = ((int64_t)oz * Ho + oy) * Wo + ox;
                const T *Xc = Xn;
                T *Yp = Yc + yo;
                for (int c = 0; c < a.C; ++c) {
                    *Yp = IO<T>::st(interp<T, 3, MODE>(Xc, tp, off_hi));
                    Xc += in_plane;
                    Yp += out_plane;
                }
            }
            continue;
        }

        const int k = s_k;
        const int bz = V.box[k][0], by = V.box[k][1], bx = V.box[k][2];
        const uint32_t dy_b = (uint32_t)bx * E, dz_b = (uint32_t)by * dy_b;
        const uint32_t box_bytes = (uint32_t)bz * dz_b;               // one copy
        const uint32_t stage_bytes = (box_bytes + 127u) & ~127u;      // stage stride
        const int lo_z = s_lo[0], lo_y = s_lo[1], lo_x = s_lo[2];
        const int C = a.C;
        const uint32_t ring_u32 = smem_u32(ring);
        // channel c of this image into stage s (thread 0)
        auto issue = [&](int c, int s) {
            mbar_arrive_expect_tx(&full[s], box_bytes);
            tma_load_4d(ring + (size_t)s * stage_bytes, &maps.m[k], lo_x, lo_y, lo_z, n * C + c,
                        &full[s]);
            ipar ^= 1u << s;
            iany |= 1u << s;
        };
        // the first stages are in flight while the taps are set up
        if (tid == 0)
            for (int c = 0; c < S && c < C; ++c) issue(c, c);

        // this thread's positions: base byte offset in a stage, weights, Y offset
        uint32_t base[kVtPPT];
        float2 w2[kVtPPT / 2][NT];   // weights of positions (2i, 2i+1), tap by tap
        int yoff[kVtPPT];
        unsigned live = 0;
#pragma unroll
        for (int j = 0; j < kVtPPT; ++j) {
            const int p = tid + j * kVtThreads;
            const int row = p >> tx_shift;
            const int oz = oz0 + row / V.ty, oy = oy0 + row % V.ty, ox = ox0 + (p & (V.tx - 1));
            const bool ok = row < V.tz * V.ty && oz < a.out[0] && oy < Ho && ox < Wo;
            live |= (ok ? 1u : 0u) << j;
            const int opos[3] = {ok ? oz : oz0, ok ? oy : oy0, ok ? ox : ox0};
            int li[3];
            float t[3];
            const int lo[3] = {lo_z, lo_y, lo_x};
#pragma unroll
            for (int d = 0; d < 3; ++d) {
                int64_t acc = s_map.cst_q[d];
#pragma unroll
                for (int jj = 0; jj < 3; ++jj) acc += s_map.coef_q[d][jj] * (int64_t)opos[jj];
                const int64_t xq = vol_pad(acc >> 8, P.ax[d], a.pad);
                li[d] = vol_index<MODE>(xq, P.ax[d].n) - lo[d];
                t[d] = __uint2float_rn((uint32_t)xq) * 2.3283064365386963e-10f;   // * 2^-32
            }
            base[j] = (uint32_t)li[0] * dz_b + (uint32_t)li[1] * dy_b + (uint32_t)li[2] * (uint32_t)E;
            if (MODE != MODE_NEAREST) {
#pragma unroll
                for (int kz = 0; kz < 2; ++kz)
#pragma unroll
                    for (int ky = 0; ky < 2; ++ky) {
                        const float wzy = (kz ? t[0] : 1.0f - t[0]) * (ky ? t[1] : 1.0f - t[1]);
                        const float w0 = wzy * (1.0f - t[2]), w1 = wzy * t[2];
                        float2 &a0 = w2[j >> 1][kz * 4 + ky * 2 + 0];
                        float2 &a1 = w2[j >> 1][kz * 4 + ky * 2 + 1];
                        if (j & 1) {
                            a0.y = w0;
                            a1.y = w1;
                        } else {
                            a0.x = w0;
                            a1.x = w1;
                        }
                    }
            }
            yoff[j] = (opos[0] * Ho + opos[1]) * Wo + opos[2];
        }

        // a tile inside the output stores every position: no per-position predicate
        const bool full_tile = oz0 + V.tz <= a.out[0] && oy0 + V.ty <= Ho && ox0 + V.tx <= Wo &&
                               V.tz * V.ty * V.tx == kVtTile;
        int st = 0;
        for (int c = 0; c < C; ++c) {
            const uint32_t u = (upar >> st) & 1u;   // parity of this use
            if (!bad) bad = !mbar_wait_bounded(&full[st], u, err);
            if (!bad) {
                const uint32_t sb = ring_u32 + (uint32_t)st * stage_bytes;
#pragma unroll
                for (int h = 0; h < kVtPPT / 2; ++h) {
                    const uint32_t qa = sb + base[2 * h], qb = sb + base[2 * h + 1];
                    float2 acc;
                    if (MODE == MODE_NEAREST) {
                        acc = make_float2(lds_off<T, 0>(qa), lds_off<T, 0>(qb));
                    } else {
                        const uint32_t qa1 = qa + dy_b, qa2 = qa + dz_b, qa3 = qa2 + dy_b;
                        const uint32_t qb1 = qb + dy_b, qb2 = qb + dz_b, qb3 = qb2 + dy_b;
                        float2 v[NT];
                        v[0] = make_float2(lds_off<T, 0>(qa), lds_off<T, 0>(qb));
                        v[1] = make_float2(lds_off<T, E>(qa), lds_off<T, E>(qb));
                        v[2] = make_float2(lds_off<T, 0>(qa1), lds_off<T, 0>(qb1));
                        v[3] = make_float2(lds_off<T, E>(qa1), lds_off<T, E>(qb1));
                        v[4] = make_float2(lds_off<T, 0>(qa2), lds_off<T, 0>(qb2));
                        v[5] = make_float2(lds_off<T, E>(qa2), lds_off<T, E>(qb2));
                        v[6] = make_float2(lds_off<T, 0>(qa3), lds_off<T, 0>(qb3));
                        v[7] = make_float2(lds_off<T, E>(qa3), lds_off<T, E>(qb3));
                        acc = mul_f32x2(w2[h][0], v[0]);
#pragma unroll
                        for (int tt = 1; tt < NT; ++tt) acc = fma_f32x2(w2[h][tt], v[tt], acc);
                    }
                    if (full_tile) {
                        Yc[yoff[2 * h]] = IO<T>::st(acc.x);
                        Yc[yoff[2 * h + 1]] = IO<T>::st(acc.y);
                    } else {
                        if ((live >> (2 * h)) & 1u) Yc[yoff[2 * h]] = IO<T>::st(acc.x);
                        if ((live >> (2 * h + 1)) & 1u) Yc[yoff[2 * h + 1]] = IO<T>::st(acc.y);
                    }
                }
            }
            // this warp is done with the stage
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            upar ^= 1u << st;
            if (tid == 0 && c + S < C && !bad) {
                // refill once every warp has read this use of the stage
                bad = !mbar_wait_bounded(&empty[st], u, err);
                if (!bad) issue(c + S, st);
            }
            Yc += out_plane;
            if (++st == S) st = 0;
        }
    }
    if (tid == 0) {
        // copies still in flight after a wait gave up must land before the
        // block's shared memory is released
        for (int s = 0; s < kVtMaxStages; ++s)
            if ((iany >> s) & 1u) mbar_wait_bounded(&full[s], ((ipar >> s) & 1u) ^ 1u, nullptr);
    }
    __syncthreads();
}

// Host side: tile shape as launch_vol; the map family is every combination of
// a small and a large margin on each axis around the tile's nominal box (its
// extent under the identity map plus the interpolation neighbour and the
// 16-byte alignment of x), keeping boxes of at most half the ring, ordered by
// size.  *used tells the caller whether the kernel ran.
template <typename T, int MODE>
cudaError_t launch_vol_tma(const void *X, const void *theta, void *Y, const SampleParams &P,
                           cudaStream_t s, bool *used) {
    *used = false;
    if (MODE == MODE_CUBIC) return cudaSuccess;
    constexpr int E = (int)sizeof(T), EPC = 16 / E, K = MODE == MODE_NEAREST ? 1 : 2;
    const SampleArgs &a = P.a;
    const int Di = a.in[0], Hi = a.in[1], Wi = a.in[2];
    if (((size_t)Wi * E) % 16 != 0 || (uintptr_t)X % 16 != 0) return cudaSuccess;
    if ((int64_t)a.N * a.C >= ((int64_t)1 << 31)) return cudaSuccess;
    const int Do = a.out[0], Ho = a.out[1], Wo = a.out[2];
    VolTmaParams V;
    // near-cubic tiles: an affine map's box around a tile grows with the
    // tile's longest side, so 8 x 8 x 16 reads less than 4 x 8 x 32
    V.tx = Wo >= 16 ? 16 : 8;
    const int rows = kVtTile / V.tx;
    V.tz = min(Do, 8);
    V.ty = min(Ho, rows / V.tz);
    V.tz = min(Do, rows / V.ty);
    V.tiles_y = (Ho + V.ty - 1) / V.ty;
    V.tiles_x = (Wo + V.tx - 1) / V.tx;
    const int64_t tiles = (int64_t)((Do + V.tz - 1) / V.tz) * V.tiles_y * V.tiles_x;
    if (tiles * a.N > 0x7fffffffLL) return cudaSuccess;
    V.tiles = (int)tiles;
    V.total = (int)(tiles * a.N);
    // nominal extents: the tile scaled by in/out, + the neighbour tap (x in
    // whole 16-byte runs)
    const int t[3] = {V.tz, V.ty, V.tx};
    const int nin[3] = {Di, Hi, Wi}, nout[3] = {Do, Ho, Wo};
    int nom[3];
    for (int d = 0; d < 3; ++d) {
        nom[d] = (int)ceil((double)t[d] * nin[d] / nout[d]) + K;
        if (d == 2) nom[d] = (nom[d] + EPC - 1) / EPC * EPC;
    }
    // the family: margins of 1 or 3 on planes and rows, 0 or one 16-byte run
    // on x, for near-identity maps; and one box with wide margins (7, 7, three
    // runs) for stronger rotations and zooms.  Wider tiles gather.
    struct Box { int b[3]; int bytes; };
    Box cand[kVtMaps];
    int nc = 0;
    for (int m = 0; m < kVtMaps; ++m) {
        Box bx;
        for (int d = 0; d < 3; ++d) {
            const int bit = (m >> d) & 1;
            int v = m == 8 ? nom[d] + (d == 2 ? 3 * EPC : 7)
                           : nom[d] + (d == 2 ? bit * EPC : (bit ? 3 : 1));
            bx.b[d] = min(v, 256);
        }
        bx.bytes = (bx.b[0] * bx.b[1] * bx.b[2] * E + 127) & ~127;
        if (2 * bx.bytes <= kVtRingBytes) cand[nc++] = bx;
    }
    if (nc == 0) return cudaSuccess;
    std::sort(cand, cand + nc, [](const Box &p, const Box &q) { return p.bytes < q.bytes; });
    VolTmaMaps maps;
    const uint64_t dims[4] = {(uint64_t)Wi, (uint64_t)Hi, (uint64_t)Di, (uint64_t)a.N * a.C};
    const uint64_t strides[3] = {(uint64_t)Wi * E, (uint64_t)Hi * Wi * E, (uint64_t)Di * Hi * Wi * E};
    V.nmaps = 0;
    for (int i = 0; i < nc; ++i) {
        const uint32_t box[4] = {(uint32_t)cand[i].b[2], (uint32_t)cand[i].b[1], (uint32_t)cand[i].b[0], 1};
        if (!tmap_encode(&maps.m[V.nmaps], E, std::is_same<T, __nv_bfloat16>::value, 4, X, dims,
                         strides, box))
            continue;
        for (int d = 0; d < 3; ++d) V.box[V.nmaps][d] = cand[i].b[d];
        ++V.nmaps;
    }
    if (V.nmaps == 0) return cudaSuccess;
    static DeviceFlags attr_set;
    cudaError_t e = once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(vol_tma_kernel<T, MODE>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kVtRingBytes + 128);
    });
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = (int)std::min<int64_t>(V.total, 2 * (int64_t)std::max(sms, 1));
    vol_tma_kernel<T, MODE><<<grid, kVtThreads, kVtRingBytes + 128, s>>>(
        (const T *)X, (const T *)theta, (T *)Y, P, V, maps);
    *used = true;
    return cudaGetLastError();
}

}  // namespace gs
