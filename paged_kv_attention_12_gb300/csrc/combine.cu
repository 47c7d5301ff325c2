// Split-K combine and the checked-mode table validator (sm_103a).
//
// The combine is the log-sum-exp merge a split-K softmax needs ("split-K
// decode variant", inference-server README, engine feature list): with
// M = max_s LSE_s and w_s = exp(LSE_s - M), out = sum_s w_s O_s / sum_s w_s
// and LSE = M + ln sum_s w_s.  Every partial row is read with coalesced
// 16-byte loads.
#include "common.cuh"
#include "kernels.h"

namespace pka {

namespace {

// One warp per (row, 128-column segment): each lane owns one float4 of the
// output.  The row's LSE values are read 32 at a time (one split per lane);
// the partial rows of eight splits are loaded together (splits with
// LSE = -inf, which no CTA wrote, are not touched) and merged four at a time
// with a running maximum, in the same groups as the decode kernel's fused
// combine.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(const CombineArgs a) {
  constexpr int SEGS = D / 128;
  const int wid = blockIdx.x * 4 + threadIdx.x / 32;
  const int row = wid / SEGS;
  const int seg = wid % SEGS;
  const int lane = threadIdx.x % 32;
  if (row >= a.rows) return;
  const int S = a.num_splits;
  const float* lse = a.partial_lse + static_cast<size_t>(row) * S;
  const float* po = a.partial_o + static_cast<size_t>(row) * S * D + seg * 128 + lane * 4;

  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < S; base += 32) {
    const float lreg = (base + lane < S) ? lse[base + lane] : -INFINITY;
    // all of the (up to) 32 pieces' loads in flight before the first merge
    float lv[32];
    float4 x[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      lv[u] = __shfl_sync(0xffffffffu, lreg, u);  // -inf past the row's end
      x[u] = (lv[u] != -INFINITY)
                 ? *reinterpret_cast<const float4*>(po + static_cast<size_t>(base + u) * D)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 32; u += 4) lse_merge4(M, den, acc, lv + u, x + u);
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint16_t* dst = a.out + static_cast<size_t>(row) * D + seg * 128 + lane * 4;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
  if (a.lse_out != nullptr && lane == 0 && seg == 0)
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

// H2O key mass: mass[b][kvh][t] += sum over the G heads h of the group of
// p_h(t) = exp(s_h(t) - LSE_h), for the keys t the decode query of request b
// sees.  The logits are the split-K kernel's log2-domain values, so
// p = 2^(x - LSE * log2 e).  One thread per (request, KV head, key):
// consecutive threads read consecutive keys of each head and update
// consecutive mass entries.
__global__ void __launch_bounds__(256) key_mass_kernel(const float* logits, const float* lse,
                                                       const int32_t* seq_lens, int32_t B,
                                                       int32_t Hq, int32_t Hkv, int32_t max_keys,
                                                       int32_t window, float* mass) {
  const int G = Hq / Hkv;
  const long long total = static_cast<long long>(B) * Hkv * max_keys;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i % max_keys);
    const long long bk = i / max_keys;
    const int kvh = static_cast<int>(bk % Hkv);
    const int b = static_cast<int>(bk / Hkv);
    const int L = min(max(seq_lens[b], 0), max_keys);
    const int pos = L - 1;
    const int t_lo = (window > 0) ? max(0, pos - window + 1) : 0;
    if (t > pos || t < t_lo) continue;
    float acc = 0.f;
    for (int g = 0; g < G; ++g) {
      const int h = kvh * G + g;
      const float ls = lse[static_cast<size_t>(b) * Hq + h];
      if (ls == -INFINITY) continue;
      acc += fast_exp2(logits[(static_cast<size_t>(b) * Hq + h) * max_keys + t] - ls * kLog2e);
    }
    mass[i] += acc;
  }
}

}  // namespace

cudaError_t launch_key_mass(const float* logits, const float* lse, const int32_t* seq_lens,
                            int32_t B, int32_t Hq, int32_t Hkv, int32_t max_keys, int32_t window,
                            float* key_mass, cudaStream_t stream) {
  const long long total = static_cast<long long>(B) * Hkv * max_keys;
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const int grid = static_cast<int>(want < 8 * 152 ? want : 8 * 152);
  key_mass_kernel<<<grid, 256, 0, stream>>>(logits, lse, seq_lens, B, Hq, Hkv, max_keys, window,
                                            key_mass);
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  const int warps = a.rows * (a.head_dim / 128);
  const int grid = (warps + 3) / 4;
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
