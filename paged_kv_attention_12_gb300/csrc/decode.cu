// Paged decode attention, direct and split-K (sm_103a, CUDA cores + TMA bulk).
//
// One query token per request attends over its visible keys, read block by
// block through the request's block table ("Triton paged decode ... kernels
// reading K/V through block tables; split-K decode variant", inference-server
// README, engine feature list).  Decode is bound by HBM: every K/V byte is
// read once, so the design is about keeping enough bytes in flight and doing
// the arithmetic on CUDA cores underneath the copies.
//
// Work items are (request, KV head, split).  The kernel is persistent: each
// CTA takes items blockIdx.x, blockIdx.x + gridDim.x, ...  Inside a CTA:
//
//  * one producer warp walks the items' block tables (32 ids per coalesced
//    load) and issues, per block, two 1-D bulk copies (the (block, head) K
//    and V tiles, each one contiguous bs*D*2-byte run of the pool) into a
//    ring of shared-memory slots, completion counted on a "full" mbarrier;
//  * NW consumer warps take the ring's tiles round robin.  A warp handles a
//    tile with its lanes spread over D (8 bf16 = 16 bytes per lane, so a key
//    row is read conflict-free in one instruction), all G query heads of the
//    KV group at once (each K/V byte feeds G heads), partial dot products
//    transposed-and-reduced across lanes (reduce-scatter with shuffles),
//    online softmax in the exp2 domain, P broadcast through shared memory
//    and P.V accumulated in fp32 registers;
//  * at the end of an item the consumer warps merge their (max, sum, acc)
//    states through shared memory and write the bf16 output (direct) or the
//    fp32 partial output + natural-log LSE (split-K), while the producer is
//    already streaming the next item's tiles.
//
// Tiles with keys outside [first visible, query position] (window start,
// ragged tail) take a masked path that never lets a masked key's K or V --
// which may be stale or NaN -- reach the arithmetic.
#include "common.cuh"
#include "kernels.h"

namespace pka {

namespace {

// Reduce-scatter of N per-lane partial sums across the LPK lanes that share
// a key: stage with xor offset O keeps the upper half of the values on lanes
// with that bit set.  Afterwards lane dl holds the full sums of indices
// (dl / DUP) * NVL + j, j < NVL (NVL = max(N / LPK, 1), DUP = max(LPK / N, 1)).
template <int N, int O>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (O == 0) {
      return;
    } else if constexpr (N >= 2) {
      constexpr int H = N / 2;
      const bool upper = (lane & O) != 0;
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const float send = upper ? v[k] : v[k + H];
        const float keep = upper ? v[k + H] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, O);
      }
      ReduceScatter<H, O / 2>::run(v, lane);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
      ReduceScatter<1, O / 2>::run(v, lane);
    }
  }
};

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Named barrier over the consumer warps only (the producer keeps streaming).
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

struct ItemRange {
  int b, kvh, split;
  int j0, nblk;   // first logical block, number of blocks
  int t_lo, pos;  // visible key positions [t_lo, pos]
  int qrow;       // query row of the request
};

__device__ __forceinline__ ItemRange item_range(const DecodeArgs& a, int item, bool report_err) {
  ItemRange r;
  const int S = a.num_splits;
  r.split = item % S;
  r.kvh = (item / S) % a.Hkv;
  r.b = item / (S * a.Hkv);
  int L = a.seq_lens[r.b];
  const int cap = a.max_blocks * kBlockSize;
  if (L > cap) {
    if (report_err) report(a.err, PKA_DEVERR_SEQ_LEN);
    L = cap;
  }
  if (L < 0) L = 0;
  r.qrow = r.b;
  if (a.query_start_loc != nullptr) {
    // varlen decode rows: the request's last query row attends at L - 1
    r.qrow = a.query_start_loc[r.b + 1] - 1;
  }
  r.pos = L - 1;
  r.t_lo = (a.window > 0) ? max(0, r.pos - a.window + 1) : 0;
  const int jlo = r.t_lo / kBlockSize;
  const int jhi = (L + kBlockSize - 1) / kBlockSize;
  if (L <= 0) {
    r.j0 = 0;
    r.nblk = 0;
    return r;
  }
  if (a.split_blocks > 0) {
    const int j0 = jlo + r.split * a.split_blocks;
    const int j1 = min(jhi, j0 + a.split_blocks);
    if (report_err && r.split == S - 1 && j1 < jhi) report(a.err, PKA_DEVERR_SEQ_LEN);
    r.j0 = j0;
    r.nblk = max(0, j1 - j0);
  } else {
    r.j0 = jlo;
    r.nblk = jhi - jlo;
  }
  return r;
}

}  // namespace

template <int D, int G, int NW, int NSLOT>
struct DecodeShape {
  static constexpr int kTileElems = kBlockSize * D;
  static constexpr int kTileBytes = kTileElems * 2;
  static constexpr int LPK = D / 8;       // lanes per key row (16 bytes per lane)
  static constexpr int KPW = 32 / LPK;    // keys per warp step
  static constexpr int KC = (kBlockSize * G / KPW > 64) ? 8 : 16;  // keys per chunk
  static constexpr int KS = KC / KPW;     // warp steps per chunk
  static constexpr int NV = KS * G;       // partial dots per lane per chunk
  static constexpr int NVL = NV >= LPK ? NV / LPK : 1;
  static constexpr int DUP = NV >= LPK ? 1 : LPK / NV;
  static constexpr int kRingBytes = NSLOT * 2 * kTileBytes;
  static constexpr int kBarBytes = 2 * NSLOT * 8;
  static constexpr int kPBytes = NW * KPW * NV * 4;
  static constexpr int kMergeBytes = NW * G * (D + 2) * 4;
  static constexpr int kSmemBytes = kRingBytes + kBarBytes + kPBytes + kMergeBytes;
  static_assert(D % 8 == 0 && LPK <= 32 && 32 % LPK == 0, "head_dim");
  static_assert(KC % KPW == 0, "chunk");
};

// Processes one KV tile (kBlockSize keys) for one consumer warp.
template <int D, int G, int NW, int NSLOT, bool EDGE>
__device__ __forceinline__ void decode_tile(const uint16_t* __restrict__ Kt,
                                            const uint16_t* __restrict__ Vt,
                                            const float (&qf)[G][8], float (&acc)[G][8],
                                            float (&m)[G],
                                            float (&ls)[DecodeShape<D, G, NW, NSLOT>::NVL],
                                            float* psm, int lane, int tok0, int t_lo, int pos,
                                            float softcap, float inv_cap) {
  using S = DecodeShape<D, G, NW, NSLOT>;
  constexpr int LPK = S::LPK, KPW = S::KPW, KC = S::KC, KS = S::KS, NV = S::NV;
  constexpr int NVL = S::NVL, DUP = S::DUP;
  const int kl = lane / LPK;
  const int dl = lane % LPK;
  float* pw = psm + kl * NV;

#pragma unroll
  for (int c = 0; c < kBlockSize / KC; ++c) {
    // ---- partial q.k over this lane's 8 elements, every key step, every head
    float part[NV];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const int key = c * KC + s * KPW + kl;
      const uint4 u = *reinterpret_cast<const uint4*>(Kt + key * D + dl * 8);
      float kf[8];
      unpack8(u, kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float d0 = qf[g][0] * kf[0];
        float d1 = qf[g][1] * kf[1];
#pragma unroll
        for (int e = 2; e < 8; e += 2) {
          d0 = fmaf(qf[g][e], kf[e], d0);
          d1 = fmaf(qf[g][e + 1], kf[e + 1], d1);
        }
        part[s * G + g] = d0 + d1;
      }
    }
    ReduceScatter<NV, LPK / 2>::run(part, lane);

    // ---- logits (log2 domain), mask, chunk max per head
    float mloc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) mloc[g] = -INFINITY;
    int gj[NVL];
#pragma unroll
    for (int j = 0; j < NVL; ++j) {
      const int i = (dl / DUP) * NVL + j;
      gj[j] = i % G;
      float x = part[j];
      if (softcap > 0.f) x = softcap * tanhf(x * inv_cap) * kLog2e;
      if (EDGE) {
        const int t = tok0 + c * KC + (i / G) * KPW + kl;
        if (t < t_lo || t > pos) x = -INFINITY;
      }
      part[j] = x;
#pragma unroll
      for (int g = 0; g < G; ++g) mloc[g] = (gj[j] == g) ? fmaxf(mloc[g], x) : mloc[g];
    }
    float alpha[G], mref[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mn = fmaxf(m[g], warp_max(mloc[g]));
      mref[g] = (mn == -INFINITY) ? 0.f : mn;
      alpha[g] = fast_exp2(m[g] - mref[g]);
      m[g] = mn;
    }
    // ---- probabilities, lane-local sums, broadcast through shared memory
#pragma unroll
    for (int j = 0; j < NVL; ++j) {
      float a = alpha[0], r = mref[0];
#pragma unroll
      for (int g = 1; g < G; ++g) {
        a = (gj[j] == g) ? alpha[g] : a;
        r = (gj[j] == g) ? mref[g] : r;
      }
      const float p = fast_exp2(part[j] - r);
      ls[j] = ls[j] * a + p;
      pw[(dl / DUP) * NVL + j] = p;
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[g][e] *= alpha[g];
    __syncwarp();

    // ---- P.V over this lane's 8 columns
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const int key = c * KC + s * KPW + kl;
      if (EDGE) {
        const int t = tok0 + key;
        if (t < t_lo || t > pos) continue;  // masked V row may hold NaN
      }
      const uint4 u = *reinterpret_cast<const uint4*>(Vt + key * D + dl * 8);
      float vf[8];
      unpack8(u, vf);
      float pg[G];
#pragma unroll
      for (int g = 0; g < G; ++g) pg[g] = pw[s * G + g];
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pg[g], vf[e], acc[g][e]);
    }
    __syncwarp();
  }
}

template <int D, int G, int NW, int NSLOT>
__global__ void __launch_bounds__((NW + 1) * 32, 1) paged_decode_kernel(const DecodeArgs a) {
  using S = DecodeShape<D, G, NW, NSLOT>;
  constexpr int TE = S::kTileElems;
  constexpr int NVL = S::NVL, LPK = S::LPK;

  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* ring = reinterpret_cast<uint16_t*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kRingBytes);
  uint64_t* empty = full + NSLOT;
  float* psm_all = reinterpret_cast<float*>(smem + S::kRingBytes + S::kBarBytes);
  float* merge = reinterpret_cast<float*>(smem + S::kRingBytes + S::kBarBytes + S::kPBytes);
  float* mrg_m = merge;                  // [NW][G]
  float* mrg_l = merge + NW * G;         // [NW][G]
  float* mrg_acc = merge + 2 * NW * G;   // [NW][G][D]

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int num_items = a.batch * a.Hkv * a.num_splits;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ============================ producer warp ============================
    const uint64_t pol = policy_evict_first();
    long long issued = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < num_items && ok; item += gridDim.x) {
      const ItemRange r = item_range(a, item, lane == 0);
      const int32_t* trow = a.tables + static_cast<size_t>(r.b) * a.max_blocks + r.j0;
      for (int base = 0; base < r.nblk && ok; base += 32) {
        int id = 0;
        if (base + lane < r.nblk) {
          id = trow[base + lane];
          if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.num_blocks)) {
            report(a.err, PKA_DEVERR_BAD_TABLE);
            id = 0;
          }
        }
        const int cnt = min(32, r.nblk - base);
        for (int k = 0; k < cnt; ++k) {
          const int phys = __shfl_sync(0xffffffffu, id, k);
          const int slot = static_cast<int>(issued % NSLOT);
          const long long round = issued / NSLOT;
          int good = 1;
          if (lane == 0) {
            if (round > 0) good = mbar_wait(&empty[slot], static_cast<uint32_t>((round - 1) & 1), a.err);
            if (good) {
              mbar_arrive_expect_tx(&full[slot], 2 * S::kTileBytes);
              const size_t off = (static_cast<size_t>(phys) * a.Hkv + r.kvh) * TE;
              uint16_t* dst = ring + static_cast<size_t>(slot) * 2 * TE;
              bulk_g2s_stream(dst, a.k + off, S::kTileBytes, &full[slot], pol);
              bulk_g2s_stream(dst + TE, a.v + off, S::kTileBytes, &full[slot], pol);
            }
          }
          good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) {
            ok = false;
            break;
          }
          ++issued;
        }
      }
    }
    // Every issued copy must have landed before the CTA may exit.
    if (lane == 0) {
      const long long first = issued > NSLOT ? issued - NSLOT : 0;
      for (long long i = first; i < issued; ++i)
        mbar_wait(&full[i % NSLOT], static_cast<uint32_t>((i / NSLOT) & 1), a.err);
    }
    return;
  }

  // ============================ consumer warps ============================
  const int kl = lane / LPK;
  const int dl = lane % LPK;
  float* psm = psm_all + warp * (S::kPBytes / 4 / NW);
  const float inv_cap = a.softcap > 0.f ? 1.f / a.softcap : 0.f;
  const float qscale = a.scale * (a.softcap > 0.f ? 1.f : kLog2e);
  long long tile_base = 0;
  bool ok = true;

  for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
    const ItemRange r = item_range(a, item, false);
    float qf[G][8], acc[G][8], m[G], ls[NVL];
    {
      const uint16_t* qp = a.q + (static_cast<size_t>(r.qrow) * a.Hq + r.kvh * G) * D + dl * 8;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint4 u = *reinterpret_cast<const uint4*>(qp + g * D);
        unpack8(u, qf[g]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          qf[g][e] *= qscale;
          acc[g][e] = 0.f;
        }
        m[g] = -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < NVL; ++j) ls[j] = 0.f;
    }

    for (int i = warp; i < r.nblk && ok; i += NW) {
      const long long T = tile_base + i;
      const int slot = static_cast<int>(T % NSLOT);
      const bool got = mbar_wait(&full[slot], static_cast<uint32_t>((T / NSLOT) & 1), a.err);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      const uint16_t* Kt = ring + static_cast<size_t>(slot) * 2 * TE;
      const uint16_t* Vt = Kt + TE;
      const int tok0 = (r.j0 + i) * kBlockSize;
      if (tok0 < r.t_lo || tok0 + kBlockSize - 1 > r.pos)
        decode_tile<D, G, NW, NSLOT, true>(Kt, Vt, qf, acc, m, ls, psm, lane, tok0, r.t_lo,
                                           r.pos, a.softcap, inv_cap);
      else
        decode_tile<D, G, NW, NSLOT, false>(Kt, Vt, qf, acc, m, ls, psm, lane, tok0, r.t_lo,
                                            r.pos, a.softcap, inv_cap);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    tile_base += r.nblk;

    // ---- per-warp totals: sums per head, accumulators across key lanes
    float lt[G];
#pragma unroll
    for (int g = 0; g < G; ++g) lt[g] = 0.f;
#pragma unroll
    for (int j = 0; j < NVL; ++j) {
      const int gj = ((dl / S::DUP) * NVL + j) % G;
#pragma unroll
      for (int g = 0; g < G; ++g) lt[g] += (gj == g) ? ls[j] : 0.f;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) lt[g] = warp_sum(lt[g]) * (1.f / S::DUP);
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1)
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);

    if (lane == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        mrg_m[warp * G + g] = m[g];
        mrg_l[warp * G + g] = lt[g];
      }
    }
    if (kl == 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float4* dst = reinterpret_cast<float4*>(mrg_acc + (warp * G + g) * D + dl * 8);
        dst[0] = make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
        dst[1] = make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
      }
    }
    consumer_sync(NW * 32);

    // ---- merge the warps' states and write this item's result
    for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
      const int g = idx / D;
      const int d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg_m[w * G + g]);
      const float Ms = (M == -INFINITY) ? 0.f : M;
      float den = 0.f, num = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float sc = fast_exp2(mrg_m[w * G + g] - Ms);
        den = fmaf(sc, mrg_l[w * G + g], den);
        num = fmaf(sc, mrg_acc[(w * G + g) * D + d], num);
      }
      const float o = (den > 0.f) ? num / den : 0.f;
      const int h = r.kvh * G + g;
      if (a.split_blocks > 0) {
        const size_t ph = (static_cast<size_t>(r.b) * a.Hq + h) * a.num_splits + r.split;
        a.partial_o[ph * D + d] = o;
        if (d == 0) a.partial_lse[ph] = (den > 0.f) ? (M + log2f(den)) * kLn2 : -INFINITY;
      } else {
        reinterpret_cast<uint16_t*>(a.out)[(static_cast<size_t>(r.qrow) * a.Hq + h) * D + d] =
            f32_to_bf16_rn(o);
      }
    }
    consumer_sync(NW * 32);
  }
}

// ------------------------------------------------------------- launchers
namespace {

template <int D, int G>
struct DecodeTuning {
  // 8 consumer warps + 1 producer warp, one CTA per SM; the ring takes what
  // the merge area leaves of the shared memory.
  static constexpr int NW = 8;
  static constexpr int NSLOT = (D == 256) ? 10 : 20;
};

template <int D, int G>
cudaError_t launch_decode_t(const DecodeArgs& a, int grid, cudaStream_t stream) {
  constexpr int NW = DecodeTuning<D, G>::NW;
  constexpr int NSLOT = DecodeTuning<D, G>::NSLOT;
  using S = DecodeShape<D, G, NW, NSLOT>;
  auto kern = paged_decode_kernel<D, G, NW, NSLOT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       S::kSmemBytes);
  if (e != cudaSuccess) return e;
  kern<<<grid, (NW + 1) * 32, S::kSmemBytes, stream>>>(a);
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
