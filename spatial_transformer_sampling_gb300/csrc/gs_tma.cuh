// gs_tma.cuh -- tensor-memory-accelerator (TMA) tile copies: host-side
// encoding of tiled tensor maps over this GPU's own memory, and the
// cp.async.bulk.tensor loads that fill shared memory from them, completing on
// an mbarrier.  No multicast: every CTA loads its own tiles.
#pragma once

#include <cuda.h>   // CUtensorMap and its enums (the encoder comes from the runtime)
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "gs_ptx.cuh"

namespace gs {

using TmapEncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                       const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                       const cuuint32_t *, CUtensorMapInterleave,
                                       CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point, looked up
// once per process (nullptr if the driver does not provide it).
inline TmapEncodeTiledFn tmap_encoder() {
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load(std::memory_order_acquire);
    if (!f) {
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !f)
            return nullptr;
        fn.store(f, std::memory_order_release);
    }
    return reinterpret_cast<TmapEncodeTiledFn>(f);
}

// A tiled map over a dense tensor of `rank` dimensions (dims[0] innermost,
// elements of `elem_bytes` = 2 or 4 bytes), a box of box[] elements per
// dimension, no swizzle, zeros outside the tensor.  strides[i] is the byte
// distance between consecutive indices of dimension i+1.  Returns false when
// the encoder is missing or rejects the arguments (the caller then takes
// another path); it checks the base's 16-byte alignment, the strides'
// multiples of 16 and each box extent against 256 itself.
inline bool tmap_encode(CUtensorMap *map, int elem_bytes, bool bf16, int rank, const void *base,
                        const uint64_t *dims, const uint64_t *strides, const uint32_t *box) {
    TmapEncodeTiledFn enc = tmap_encoder();
    if (!enc || rank < 1 || rank > 5 || ((uintptr_t)base & 15u)) return false;
    cuuint64_t gd[5], gs[4];
    cuuint32_t bx[5], es[5];
    for (int i = 0; i < rank; ++i) {
        if (dims[i] == 0 || box[i] == 0 || box[i] > 256) return false;
        gd[i] = dims[i];
        bx[i] = box[i];
        es[i] = 1;
        if (i + 1 < rank) {
            if (strides[i] % 16 != 0) return false;
            gs[i] = strides[i];
        }
    }
    if ((box[0] * (uint32_t)elem_bytes) % 16 != 0) return false;
    const CUtensorMapDataType dt = elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : bf16          ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(map, dt, (cuuint32_t)rank, const_cast<void *>(base), gd, gs, bx, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Starts fetching a tensor map's descriptor (kernel-parameter space) so the
// first copy that uses it does not wait for it.
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Loads the box at coordinates (c0 innermost .. c3) of a 4-D map into shared
// memory at dst (128-byte aligned); the bytes complete on `bar`, which the
// issuing thread armed with mbar_arrive_expect_tx for the box's size.  c0
// times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar))
        : "memory");
}

// Same for a 3-D map.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace gs
