// Paged prefill / mixed-batch attention launch (sm_103a): one work item
// (request, KV head, query tile) per CTA.  The tcgen05 pipeline is in
// prefill_body.cuh.
#include "prefill2_body.cuh"
#include "tmaps.cuh"

namespace pka {

template <int D, int G>
__global__ void __launch_bounds__(PrefillShape<D, G>::kThreads, 1)
    paged_prefill_kernel(const __grid_constant__ PrefillArgs a,
                         const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ uint8_t smem_raw[];
  prefill_body<D, G, false>(a, &tm_q, &tm_k, &tm_v, &tm_out, smem_raw, static_cast<int>(blockIdx.x));
}

// D = 256 on CTA pairs: cluster i of two CTAs takes pair item i.
template <int G>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Prefill2Shape<G>::kThreads, 1)
    paged_prefill2_kernel(const __grid_constant__ PrefillArgs a,
                          const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_out) {
  extern __shared__ uint8_t smem_raw[];
  prefill2_body<G, false>(a, &tm_q, &tm_k, &tm_v, &tm_out, smem_raw, 0);
}

// ------------------------------------------------------------- launchers
namespace {

template <int G>
cudaError_t launch_prefill2_t(const PrefillArgs& a, cudaStream_t stream) {
  using S = Prefill2Shape<G>;
  CUtensorMap tq, tk, tv, to;
  const long long rows = static_cast<long long>(a.num_blocks) * a.Hkv * kBlockSize;
  if (!tmap_query_tiles(&tq, a.q, S::D, a.Hq, a.total_q, G, S::TQ) ||
      !tmap_pool_rows(&tk, a.k, S::D, rows) ||
      !tmap_pool_tiles_chunks(&tv, a.v, S::D, rows, S::DC / 2) ||
      !tmap_query_tiles(&to, a.out, S::D, a.Hq, a.total_q, G, S::TQ))
    return cudaErrorInvalidValue;
  auto kern = paged_prefill2_kernel<G>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), S::kSmemBytes);
  if (e != cudaSuccess) return e;
  // one cluster per (request, pair of query tiles, KV head)
  const long long clusters = prefill_ranks(a, 2 * S::TQ);
  if (2 * clusters > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(2 * clusters));
  kern<<<grid, S::kThreads, S::kSmemBytes, stream>>>(a, tq, tk, tv, to);
  return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_prefill_t(const PrefillArgs& a, cudaStream_t stream) {
  using S = PrefillShape<D, G>;
  CUtensorMap tq, tk, tv, to;
  const long long rows = static_cast<long long>(a.num_blocks) * a.Hkv * kBlockSize;
  if (!tmap_query_tiles(&tq, a.q, D, a.Hq, a.total_q, G, S::TQ) ||
      !tmap_pool_rows(&tk, a.k, D, rows) || !tmap_pool_tiles(&tv, a.v, D, rows) ||
      !tmap_query_tiles(&to, a.out, D, a.Hq, a.total_q, G, S::TQ))
    return cudaErrorInvalidValue;
  auto kern = paged_prefill_kernel<D, G>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), S::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long long ctas = prefill_ranks(a, S::TQ);
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
  dim3 grid(static_cast<unsigned>(ctas));
  kern<<<grid, S::kThreads, S::kSmemBytes, stream>>>(a, tq, tk, tv, to);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim, int group, int /*sm_count*/,
                           cudaStream_t stream) {

#define PKA_PRE(D_, G_) \
  if (head_dim == D_ && group == G_) return launch_prefill_t<D_, G_>(a, stream);
#define PKA_PRE2(G_) \
  if (head_dim == 256 && group == G_) return launch_prefill2_t<G_>(a, stream);
  PKA_PRE(128, 1)
  PKA_PRE(128, 2)
  PKA_PRE(128, 4)
  PKA_PRE(128, 8)
  PKA_PRE2(1)
  PKA_PRE2(2)
  PKA_PRE2(4)
  PKA_PRE2(8)
#undef PKA_PRE2
#undef PKA_PRE
  return cudaErrorInvalidValue;
}

}  // namespace pka

#ifdef PKA_TIMELINE
// Instrumented builds only: the stamps of the prefill CTAs.
PKA_TIMELINE_EXPORT(_prefill, pka::pka_timeline_prefill)
#endif
