// tensor_copy.cuh -- inline-PTX wrappers for tiled tensor copies (TMA through
// a tensor map) between global and shared memory, and host-side encoding of
// the tensor maps.  Used where the shared-memory layout must be swizzled,
// which the plain bulk copies of bulk.cuh cannot do.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bulk.cuh"

namespace ss {

// Tiled 2-D tensor copy global -> shared.  The box, the swizzle and the
// bounds come from the map; x and y are element coordinates (x times the
// element size a multiple of 16 bytes).  Completion is signalled on `bar`
// as transaction bytes.
__device__ __forceinline__ void tensor_load_2d(void* dst_smem, const CUtensorMap* map, int32_t x, int32_t y,
                                               uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Tiled 2-D tensor copy shared -> global in this thread's bulk async-group.
// Every thread that wrote the source must have run fence_async_shared, and
// a barrier must order those writes before this call.
__device__ __forceinline__ void tensor_store_2d(const CUtensorMap* map, int32_t x, int32_t y, const void* src_smem) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(src_smem))
                 : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// This thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_group_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// This thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Byte offset of 16-byte chunk `chunk` of 128-byte row `row` in a
// 1024-byte-aligned shared-memory area written or read by a copy with
// 128-byte swizzle: the chunk index is XORed with the row index modulo 8.
__device__ __forceinline__ uint32_t swizzle128_offset(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Host: a 2-D map over `rows` rows of 16 doubles (128 bytes each, packed)
// at `base` (16-byte aligned), boxes of `box_rows` rows, 128-byte swizzle.
// cudaErrorNotSupported if the driver has no tensor-map encoder,
// cudaErrorInvalidValue if it rejects the arguments.
inline cudaError_t encode_rows128_f64(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
    static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            fn = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {16, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {16, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 2, const_cast<void*>(base), dims, strides, box,
                              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Host: the same for rows of 32 four-byte elements (128 bytes each).
inline cudaError_t encode_rows128_b32(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows) {
    static const PFN_cuTensorMapEncodeTiled_v12000 encode = [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            fn = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {32, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {32, box_rows};
    const cuuint32_t elem_strides[2] = {1, 1};
    const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box,
                              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace ss
