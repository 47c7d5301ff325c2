// Mixed batch -- decode rows and chunked-prefill chunks -- in one launch
// (sm_103a).  Decode tokens and prefill chunks of the same engine tick go
// through one attention call ("mixed-batch chunked prefill", architecture
// page, "Phase status"), and the two kinds of rows want different machines:
// a prefill chunk is a dense contraction for the tcgen05 pipeline, while a
// decode row (one token, G query heads) would fill 4 of the 128 rows of a
// tensor-core tile and is bound by streaming its keys.
//
// So the launch has two kinds of CTAs, 256 threads each:
//  * CTAs [0, n_decode): two decode pipelines each (decode_body.cuh: a
//    producer warp and three consumer warps over half the shared memory),
//    which split the decode rows' keys in the balanced split-K partition and
//    merge the pieces in the launch (fused LSE combine: the last piece of a
//    segment to finish merges it, counted in the workspace);
//  * the CTAs after them: the tcgen05 prefill pipeline (prefill_body.cuh),
//    one (request, KV head, query tile) item each, heaviest first; requests
//    with one query token are left out.
// The hardware starts CTAs in index order: the decode pipelines start at
// once on n_decode SMs and the prefill items take the others.  The host
// sizes n_decode from the number of prefill tokens.
#include "decode_body.cuh"
#include "prefill2_body.cuh"
#include "tmaps.cuh"

namespace pka {

namespace {

// Decode pipelines of the mixed launch: two per CTA of the prefill's 256
// threads, each a producer warp and three consumer warps, each ring in half
// of the prefill's shared memory.
template <int D, int G>
struct MixedDecodeTuning {
  static constexpr int NW = 3;
  static constexpr int NSLOT = (D == 256) ? ((G == 8) ? 3 : 6) : 12;
  static constexpr int kPipeThreads = (NW + 1) * 32;
  static constexpr int kPipeBytes = DecodeShape<D, G, NW, NSLOT>::kSmemBytes;
  static_assert(2 * kPipeThreads == PrefillShape<D, G>::kThreads, "two pipelines per CTA");
  static constexpr int kSmemBytes = (2 * kPipeBytes > PrefillShape<D, G>::kSmemBytes)
                                        ? 2 * kPipeBytes
                                        : PrefillShape<D, G>::kSmemBytes;
};

}  // namespace

// The decode CTAs' part of both mixed kernels: two pipelines per CTA.
template <int D, int G>
__device__ __forceinline__ void mixed_decode_part(const DecodeArgs& da, int n_decode,
                                                  const CUtensorMap* tm_k_tiles,
                                                  const CUtensorMap* tm_v_tiles,
                                                  uint8_t* smem_raw) {
  using T = MixedDecodeTuning<D, G>;
  const int pipe = static_cast<int>(threadIdx.x) / T::kPipeThreads;  // 0 or 1
  // named barriers 1, 2, 5 (pipeline 0) and 3, 4, 6 (pipeline 1)
  const DecodeCtx cx{static_cast<int>(blockIdx.x) * 2 + pipe, n_decode * 2,
                     static_cast<int>(threadIdx.x) % T::kPipeThreads, 1 + 2 * pipe, 2 + 2 * pipe,
                     5 + pipe};
  decode_body<D, G, T::NW, T::NSLOT>(da, tm_k_tiles, tm_v_tiles,
                                     smem_raw + pipe * T::kPipeBytes, cx);
}

template <int D, int G>
__global__ void __launch_bounds__(PrefillShape<D, G>::kThreads, 1)
    paged_mixed_kernel(const __grid_constant__ PrefillArgs pa,
                       const __grid_constant__ DecodeArgs da, const int n_decode,
                       const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k_rows,
                       const __grid_constant__ CUtensorMap tm_k_tiles,
                       const __grid_constant__ CUtensorMap tm_v_tiles,
                       const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ uint8_t smem_raw[];
  if (static_cast<int>(blockIdx.x) >= n_decode) {
    prefill_body<D, G, true>(pa, &tm_q, &tm_k_rows, &tm_v_tiles, &tm_out, smem_raw,
                       static_cast<int>(blockIdx.x) - n_decode);
    return;
  }
  mixed_decode_part<D, G>(da, n_decode, &tm_k_tiles, &tm_v_tiles, smem_raw);
}

// D = 256: the chunks' query tiles run on CTA pairs (prefill2_body.cuh: two
// query tiles per cluster of two SMs, one MMA of M = 256), the decode CTAs
// as above.  n_decode is even, so that every cluster is either two decode
// CTAs or one pair.  kSplit: the pair items may be cut along keys (the
// merge code is compiled in only then; it costs the softmax registers).
template <int G, bool kSplit>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Prefill2Shape<G>::kThreads, 1)
    paged_mixed_pair_kernel(const __grid_constant__ PrefillArgs pa,
                            const __grid_constant__ DecodeArgs da, const int n_decode,
                            const __grid_constant__ CUtensorMap tm_q,
                            const __grid_constant__ CUtensorMap tm_k_rows,
                            const __grid_constant__ CUtensorMap tm_k_tiles,
                            const __grid_constant__ CUtensorMap tm_v_tiles,
                            const __grid_constant__ CUtensorMap tm_v_half,
                            const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ uint8_t smem_raw[];
  if (static_cast<int>(blockIdx.x) >= n_decode) {
    prefill2_body<G, kSplit>(pa, &tm_q, &tm_k_rows, &tm_v_half, &tm_out, smem_raw, n_decode);
    return;
  }
  mixed_decode_part<256, G>(da, n_decode, &tm_k_tiles, &tm_v_tiles, smem_raw);
}

namespace {

template <int D, int G>
cudaError_t launch_mixed_t(const PrefillArgs& pa, const DecodeArgs& da, int decode_ctas,
                           cudaStream_t stream) {
  using S = PrefillShape<D, G>;
  using T = MixedDecodeTuning<D, G>;
  CUtensorMap tq, tkr, tkt, tvt, to;
  const long long rows = static_cast<long long>(pa.num_blocks) * pa.Hkv * kBlockSize;
  if (!tmap_query_tiles(&tq, pa.q, D, pa.Hq, pa.total_q, G, S::TQ) ||
      !tmap_pool_rows(&tkr, pa.k, D, rows) || !tmap_pool_tiles(&tkt, pa.k, D, rows) ||
      !tmap_pool_tiles(&tvt, pa.v, D, rows) ||
      !tmap_query_tiles(&to, pa.out, D, pa.Hq, pa.total_q, G, S::TQ))
    return cudaErrorInvalidValue;
  auto kern = paged_mixed_kernel<D, G>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), T::kSmemBytes);
  if (e != cudaSuccess) return e;
  long long pre = prefill_ranks(pa, S::TQ);
  // with pieces along keys, up to one wave of units
  if (pa.split_o != nullptr && pa.one_wave > pre) pre = min(pa.one_wave, pa.split_slots);
  const long long ctas = static_cast<long long>(decode_ctas) + pre;
  if (ctas > 0x7fffffffLL || decode_ctas <= 0) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(ctas), S::kThreads, T::kSmemBytes, stream>>>(
      pa, da, decode_ctas, tq, tkr, tkt, tvt, to);
  return cudaGetLastError();
}

template <int G>
cudaError_t launch_mixed_pair_t(const PrefillArgs& pa, const DecodeArgs& da, int decode_ctas,
                                bool pieces, cudaStream_t stream) {
  using S = Prefill2Shape<G>;
  using T = MixedDecodeTuning<256, G>;
  static_assert(2 * T::kPipeThreads == S::kThreads, "two pipelines per CTA");
  constexpr int kSmem = (2 * T::kPipeBytes > S::kSmemBytes) ? 2 * T::kPipeBytes : S::kSmemBytes;
  CUtensorMap tq, tkr, tkt, tvt, tvh, to;
  const long long rows = static_cast<long long>(pa.num_blocks) * pa.Hkv * kBlockSize;
  if (!tmap_query_tiles(&tq, pa.q, 256, pa.Hq, pa.total_q, G, S::TQ) ||
      !tmap_pool_rows(&tkr, pa.k, 256, rows) || !tmap_pool_tiles(&tkt, pa.k, 256, rows) ||
      !tmap_pool_tiles(&tvt, pa.v, 256, rows) ||
      !tmap_pool_tiles_chunks(&tvh, pa.v, 256, rows, S::DC / 2) ||
      !tmap_query_tiles(&to, pa.out, 256, pa.Hq, pa.total_q, G, S::TQ))
    return cudaErrorInvalidValue;
  auto kern = pieces ? paged_mixed_pair_kernel<G, true> : paged_mixed_pair_kernel<G, false>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), kSmem);
  if (e != cudaSuccess) return e;
  if (decode_ctas <= 0 || (decode_ctas & 1) != 0) return cudaErrorInvalidValue;
  long long clusters = prefill_ranks(pa, 2 * S::TQ);
  // with pieces along keys, up to one wave of units (pair slots, two
  // workspace slots each)
  if (pieces && pa.split_o != nullptr && pa.one_wave / 2 > clusters)
    clusters = min(pa.one_wave / 2, pa.split_slots / 2);
  const long long ctas = static_cast<long long>(decode_ctas) + 2 * clusters;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(ctas), S::kThreads, kSmem, stream>>>(pa, da, decode_ctas, tq, tkr,
                                                                    tkt, tvt, tvh, to);
  return cudaGetLastError();
}

}  // namespace

int mixed_query_tile(int head_dim, int group) {
  if (head_dim == 128) {
    switch (group) {
      case 1: return PrefillShape<128, 1>::TQ;
      case 2: return PrefillShape<128, 2>::TQ;
      case 4: return PrefillShape<128, 4>::TQ;
      case 8: return PrefillShape<128, 8>::TQ;
    }
  } else if (head_dim == 256) {
    switch (group) {
      case 1: return PrefillShape<256, 1>::TQ;
      case 2: return PrefillShape<256, 2>::TQ;
      case 4: return PrefillShape<256, 4>::TQ;
      case 8: return PrefillShape<256, 8>::TQ;
    }
  }
  return 0;
}

cudaError_t launch_mixed(const PrefillArgs& pa, const DecodeArgs& da, int head_dim, int group,
                         int decode_ctas, bool pairs, bool pair_pieces, cudaStream_t stream) {
  if (pairs && head_dim == 256) {
    switch (group) {
      case 1: return launch_mixed_pair_t<1>(pa, da, decode_ctas, pair_pieces, stream);
      case 2: return launch_mixed_pair_t<2>(pa, da, decode_ctas, pair_pieces, stream);
      case 4: return launch_mixed_pair_t<4>(pa, da, decode_ctas, pair_pieces, stream);
      case 8: return launch_mixed_pair_t<8>(pa, da, decode_ctas, pair_pieces, stream);
    }
    return cudaErrorInvalidValue;
  }
#define PKA_MIX(D_, G_) \
  if (head_dim == D_ && group == G_) return launch_mixed_t<D_, G_>(pa, da, decode_ctas, stream);
  PKA_MIX(128, 1)
  PKA_MIX(128, 2)
  PKA_MIX(128, 4)
  PKA_MIX(128, 8)
  PKA_MIX(256, 1)
  PKA_MIX(256, 2)
  PKA_MIX(256, 4)
  PKA_MIX(256, 8)
#undef PKA_MIX
  return cudaErrorInvalidValue;
}

}  // namespace pka

#ifdef PKA_TIMELINE
// Instrumented builds only: the stamps of the mixed launch's decode
// pipelines and prefill CTAs.
PKA_TIMELINE_EXPORT(_mixed, pka::pka_timeline)
PKA_TIMELINE_EXPORT(_mixed_prefill, pka::pka_timeline_prefill)
#endif
