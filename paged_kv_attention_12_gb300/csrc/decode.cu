// Paged decode attention launch (sm_103a): one decode pipeline per CTA,
// two persistent CTAs per SM.  The pipeline itself (work partition, TMA ring,
// warp-level MMA, online softmax, split-K epilogue and fused combine) is in
// decode_body.cuh.
#include "decode_body.cuh"
#include "tmaps.cuh"

namespace pka {

template <int D, int G, int NW, int NSLOT>
__global__ void __launch_bounds__((NW + 1) * 32, 2)
    paged_decode_kernel(const __grid_constant__ DecodeArgs a,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ uint8_t smem_raw[];
  const DecodeCtx cx{static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                     static_cast<int>(threadIdx.x), 0, 1, 2};
  decode_body<D, G, NW, NSLOT>(a, &tm_k, &tm_v, smem_raw, cx);
}

// ------------------------------------------------------------- launchers
namespace {

template <int D, int G>
struct DecodeTuning {
  // Two persistent CTAs per SM, each with one producer warp: one thread's
  // wait -> expect -> issue loop limits a CTA's copy rate, and two CTAs per
  // SM read about 1.5x the bytes per second of one with the same ring bytes
  // in total (6.1 vs 4.0 TB/s on a 2 GiB stream of random 8 KB tiles).
  // Each CTA has NW consumer warps and a ring of 64-96 KB (SPW slots per
  // consumer warp, each slot owned by one warp).  At D = 256, three consumer
  // warps (two at G = 8, whose merge area is twice as large) share the few
  // tiles a CTA gets from a short segment.
  static constexpr int kCtasPerSm = 2;
  static constexpr int NW = (D == 256) ? ((G == 8) ? 2 : 3) : 4;
  static constexpr int SPW = (D == 256) ? 2 : ((G == 8) ? 2 : 3);
  static constexpr int NSLOT = NW * SPW;
};

template <int D, int G>
cudaError_t launch_decode_t(const DecodeArgs& a, int grid, cudaStream_t stream) {
  constexpr int NW = DecodeTuning<D, G>::NW;
  constexpr int NSLOT = DecodeTuning<D, G>::NSLOT;
  using S = DecodeShape<D, G, NW, NSLOT>;
  CUtensorMap tk, tv;
  const long long rows = static_cast<long long>(a.num_blocks) * a.Hkv * kBlockSize;
  if (!tmap_pool_tiles(&tk, a.k, D, rows) || !tmap_pool_tiles(&tv, a.v, D, rows))
    return cudaErrorInvalidValue;
  auto kern = paged_decode_kernel<D, G, NW, NSLOT>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), S::kSmemBytes);
  if (e != cudaSuccess) return e;
  // grid is given per SM count; the kernel is persistent with two CTAs per SM
  const long long g2 = static_cast<long long>(grid) * DecodeTuning<D, G>::kCtasPerSm;
  kern<<<static_cast<unsigned>(g2), (NW + 1) * 32, S::kSmemBytes, stream>>>(a, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int head_dim, int group, int grid,
                          cudaStream_t stream) {
#define PKA_DEC(D_, G_) \
  if (head_dim == D_ && group == G_) return launch_decode_t<D_, G_>(a, grid, stream);
  PKA_DEC(128, 1)
  PKA_DEC(128, 2)
  PKA_DEC(128, 4)
  PKA_DEC(128, 8)
  PKA_DEC(256, 1)
  PKA_DEC(256, 2)
  PKA_DEC(256, 4)
  PKA_DEC(256, 8)
#undef PKA_DEC
  return cudaErrorInvalidValue;
}

}  // namespace pka

#ifdef PKA_TIMELINE
// Instrumented builds only: copy the decode timeline (device to device, into
// dst, 2 * 1024 * 8 uint64) or zero it on the stream.
PKA_TIMELINE_EXPORT(, pka::pka_timeline)
#endif
