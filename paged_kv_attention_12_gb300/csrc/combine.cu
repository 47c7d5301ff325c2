// Split-K combine and the checked-mode table validator (sm_103a).
//
// The combine is the log-sum-exp merge a split-K softmax needs ("split-K
// decode variant", inference-server README, engine feature list): with
// M = max_s LSE_s and w_s = exp(LSE_s - M), out = sum_s w_s O_s / sum_s w_s
// and LSE = M + ln sum_s w_s.  One warp per (request, query head); lanes
// split the head dimension, so every partial row is read with coalesced
// 16-byte loads.
#include "common.cuh"
#include "kernels.h"

namespace pka {

namespace {

template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const CombineArgs a) {
  constexpr int EPL = D / 32;  // fp32 columns per lane (4 or 8)
  const int row = blockIdx.x * 4 + threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (row >= a.rows) return;
  const int S = a.num_splits;
  const float* lse = a.partial_lse + static_cast<size_t>(row) * S;
  const float* po = a.partial_o + static_cast<size_t>(row) * S * D;

  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float Ms = (M == -INFINITY) ? 0.f : M;

  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float den = 0.f;
  for (int s = 0; s < S; ++s) {
    const float w = fast_exp2((lse[s] - Ms) * kLog2e);  // exp(-inf) = 0 for empty splits
    if (w == 0.f) continue;                             // uniform across the warp
    den += w;
    const float4* src = reinterpret_cast<const float4*>(po + static_cast<size_t>(s) * D + lane * EPL);
#pragma unroll
    for (int e = 0; e < EPL / 4; ++e) {
      const float4 x = src[e];
      acc[4 * e + 0] = fmaf(w, x.x, acc[4 * e + 0]);
      acc[4 * e + 1] = fmaf(w, x.y, acc[4 * e + 1]);
      acc[4 * e + 2] = fmaf(w, x.z, acc[4 * e + 2]);
      acc[4 * e + 3] = fmaf(w, x.w, acc[4 * e + 3]);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint16_t* dst = a.out + static_cast<size_t>(row) * D + lane * EPL;
  uint32_t packed[EPL / 2];
#pragma unroll
  for (int e = 0; e < EPL / 2; ++e) packed[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
  if constexpr (EPL == 8) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  } else {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  }
  if (a.lse_out != nullptr && lane == 0)
    a.lse_out[row] = den > 0.f ? M + logf(den) : -INFINITY;
}

__global__ void check_tables_kernel(const CheckArgs a) {
  const int b = blockIdx.x;
  int L = a.seq_lens[b];
  if (threadIdx.x == 0 && (L < 0 || L > a.max_blocks * a.block_size))
    atomicOr(a.err, PKA_DEVERR_SEQ_LEN);
  L = max(0, min(L, a.max_blocks * a.block_size));
  const int nb = (L + a.block_size - 1) / a.block_size;
  const int32_t* row = a.tables + static_cast<size_t>(b) * a.max_blocks;
  int bad = 0;
  for (int j = threadIdx.x; j < nb; j += blockDim.x)
    bad |= static_cast<unsigned>(row[j]) >= static_cast<unsigned>(a.num_blocks);
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(a.err, PKA_DEVERR_BAD_TABLE);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  const int grid = (a.rows + 3) / 4;
  if (a.head_dim == 128)
    combine_kernel<128><<<grid, 128, 0, stream>>>(a);
  else if (a.head_dim == 256)
    combine_kernel<256><<<grid, 128, 0, stream>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_check_tables(const CheckArgs& a, cudaStream_t stream) {
  check_tables_kernel<<<a.batch, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pka
