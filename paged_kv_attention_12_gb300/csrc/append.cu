// Append of new tokens' K and V rows into a block-paged pool (sm_103a).
//
// The step that precedes attention on every engine tick: the new tokens'
// keys and values are written into the cache blocks the scheduler gave them
// ("Block-paged per-layer KV with refcounted blocks, lazy allocation, and SDPA
// gather -- vLLM/PagedAttention layout", github README, "What's inside",
// Paged KV cache row).  Token t goes to slot s = slot_mapping[t], i.e. block
// s / bs, offset s % bs, of every KV head; s < 0 means "no slot" (padding).
//
// A pure copy: each thread moves one 16-byte chunk of one (token, head) row
// of K or V, consecutive threads covering consecutive chunks, so both the
// reads of the new rows and the writes into the pool are coalesced 16-byte
// accesses.  Bound by HBM (bytes read + written), and for a decode tick's few
// tokens by launch latency.
#include "common.cuh"
#include "kernels.h"

namespace pka {

namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
  const int cpr = a.head_dim / 8;  // 16-byte chunks per (token, head) row
  const long long per_tensor = static_cast<long long>(a.T) * a.Hkv * cpr;
  const long long total = 2 * per_tensor;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const bool is_v = i >= per_tensor;
    const long long r = is_v ? i - per_tensor : i;
    const int c = static_cast<int>(r % cpr);
    const long long th = r / cpr;  // token * Hkv + head
    const int h = static_cast<int>(th % a.Hkv);
    const int t = static_cast<int>(th / a.Hkv);
    const int s = a.slot_mapping[t];
    if (s < 0) continue;
    const int blk = s / a.block_size, off = s % a.block_size;
    if (blk >= a.num_blocks) {
      if (c == 0 && h == 0 && !is_v) report(a.err, PKA_DEVERR_BAD_TABLE);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(is_v ? a.v_new : a.k_new) + th * cpr + c;
    uint4* dst = reinterpret_cast<uint4*>(is_v ? a.v_pool : a.k_pool) +
                 ((static_cast<long long>(blk) * a.Hkv + h) * a.block_size + off) * cpr + c;
    *dst = __ldg(src);
  }
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, int sm_count, cudaStream_t stream) {
  const long long total = 2LL * a.T * a.Hkv * (a.head_dim / 8);
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  kv_append_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pka
