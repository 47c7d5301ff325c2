// Tensor maps for the TMA copies (sm_103a): bf16 views of q and of the
// block pools, 128-byte swizzled, encoded through the driver entry point.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace pka {

inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// A rank-`rank` bf16 tensor map with the 128-byte swizzle (boxes are 64
// columns = 128 bytes wide), out-of-range elements read as zero.
inline bool tmap_bf16(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                      const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  auto fn = tmap_encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
            strides_bytes, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A pool viewed as a 3-D tensor (64 columns, num_blocks * Hkv * 16 rows,
// D / 64 column chunks) with strides (2, 2 D, 128) bytes, read in boxes of
// (64, 16, D / 64): one copy brings a (block, head) 16 x D tile as D / 64
// consecutive 16-row x 64-column boxes.  Fewer, larger copies keep the TMA
// unit's per-copy cost off the critical path.
inline bool tmap_pool_tiles(CUtensorMap* m, const void* base, int D, long long rows) {
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(D / 64)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(D) * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBlockSize),
                             static_cast<cuuint32_t>(D / 64)};
  return tmap_bf16(m, base, 3, dims, str, box);
}

// The same view read in boxes of (64, 16, nchunks): nchunks of the D / 64
// column chunks of a (block, head) tile per copy.
inline bool tmap_pool_tiles_chunks(CUtensorMap* m, const void* base, int D, long long rows,
                                   int nchunks) {
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(D / 64)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(D) * 2, 128};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBlockSize),
                             static_cast<cuuint32_t>(nchunks)};
  return tmap_bf16(m, base, 3, dims, str, box);
}

// q [total_q][Hq][D] as a 3-D tensor (D, Hq, total_q) read in boxes of
// (64 columns, the G heads of one KV group, TQ tokens): one box per 64-column
// chunk of a 128-row query tile.
inline bool tmap_query_tiles(CUtensorMap* m, const void* q, int D, int Hq, long long total_q,
                             int G, int TQ) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                              static_cast<cuuint64_t>(total_q)};
  const cuuint64_t str[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(TQ)};
  return tmap_bf16(m, q, 3, dims, str, box);
}

// A pool as a 2-D tensor (D columns, num_blocks * Hkv * 16 rows) read in
// 16-row x 64-column boxes.
inline bool tmap_pool_rows(CUtensorMap* m, const void* base, int D, long long rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t str[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kBlockSize)};
  return tmap_bf16(m, base, 2, dims, str, box);
}

}  // namespace pka
