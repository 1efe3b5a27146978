// TMA tensor maps over the weight records and 2-D tiled bulk loads, shared
// by the tensor-core expert paths (many-position and small-batch).
#pragma once
#include <cudaTypedefs.h>
#include "colimoe_internal.cuh"

namespace colimoe {

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)) : "memory");
}

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// A byte matrix of `rows` x `row_bytes` (row pitch row_bytes), loaded in
// boxes of box_rows x box_bytes.  With swizzle128 the box is 128 bytes wide
// and lands with its 16-byte chunks XOR-permuted by (row % 8) inside each
// 1024-byte atom (the destination must be 1024-byte aligned).
inline bool encode_rows(CUtensorMap* m, const void* base, size_t row_bytes, size_t rows, uint32_t box_bytes,
                        uint32_t box_rows, bool swizzle128 = false) {
  auto fn = encode_fn();
  if (!fn || rows == 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same with an explicit swizzle mode: with 64-byte rows and
// CU_TENSOR_MAP_SWIZZLE_64B, the 16-byte chunk c of row r lands at chunk
// c ^ ((r >> 1) & 3) (the destination must be 512-byte aligned); with 128-byte
// rows and CU_TENSOR_MAP_SWIZZLE_128B at c ^ (r & 7) (1024-byte aligned).
inline bool encode_rows_sw(CUtensorMap* m, const void* base, size_t row_bytes, size_t rows, uint32_t box_bytes,
                           uint32_t box_rows, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn || rows == 0) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  const cuuint32_t box[2] = {box_bytes, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace colimoe
