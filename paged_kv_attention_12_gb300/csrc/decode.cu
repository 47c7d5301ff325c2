// Paged decode attention, direct and split-K (sm_103a, CUDA cores + TMA bulk).
//
// One query token per request attends over its visible keys, read block by
// block through the request's block table ("Triton paged decode ... kernels
// reading K/V through block tables; split-K decode variant", inference-server
// README, engine feature list).  Decode is bound by HBM: every K/V byte is
// read once, so the design is about keeping enough bytes in flight, spreading
// them evenly over the SMs, and doing the arithmetic on CUDA cores underneath
// the copies.
//
// Work.  A segment is one (request, KV head): its visible blocks, each a
// 16-key "tile".  The kernel is persistent (one CTA per SM).
//  * split-K: the segments' tiles, laid end to end, are cut into equal
//    contiguous chunks of q = max(min_chunk, ceil(total / grid)) tiles, one
//    chunk per CTA.  Each piece of a segment inside a chunk gives one partial
//    (normalised output, LSE) in slot (CTA index - CTA index of the
//    segment's first tile); the CTA holding a segment's first tile also
//    writes LSE = -inf into the slots the segment does not use, so the LSE
//    combine needs nothing but the partials.  Every CTA streams the same
//    number of tiles whatever the mix of lengths.
//  * direct: CTA c takes whole segments c, c + grid, ... and writes bf16.
//
// Inside a CTA:
//  * one producer warp walks the pieces' block tables (32 ids per coalesced
//    load) and issues, per tile, two 1-D bulk copies (the (block, head) K and
//    V tiles, each one contiguous bs*D*2-byte run of the pool) into a ring of
//    shared-memory slots, completion counted on a "full" mbarrier;
//  * NW consumer warps take the ring's tiles round robin; every slot has
//    one owner warp, so each slot's mbarrier phases are consumed in order.
//    Lanes are spread
//    over D (8 bf16 = 16 bytes per lane, so a key row is read conflict-free
//    in one instruction); all G query heads of the KV group are handled at
//    once (each K/V byte feeds G heads); partial dot products are reduced
//    across lanes with a shuffle reduce-scatter; online softmax runs in the
//    exp2 domain; P is broadcast through shared memory; P.V accumulates in
//    fp32 registers with packed two-wide FMAs;
//  * at the end of a piece the consumer warps merge their (max, sum, acc)
//    states through shared memory and write the piece's result, while the
//    producer already streams the next piece's tiles.
//
// Tiles with keys outside [first visible, query position] (window start,
// ragged tail) take a masked path that never lets a masked key's K or V --
// which may be stale or NaN -- reach the arithmetic.
#include "common.cuh"
#include "kernels.h"

namespace pka {

namespace {

// ---------------------------------------------------------- packed fp32 x2
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Select kept opaque to the compiler: a chain of these over a small array
// must stay a chain of selects (left visible, the compiler turns it into a
// runtime-indexed array in local memory).
__device__ __forceinline__ float opaque_sel(bool c, float a, float b) {
  float r;
  asm("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\tselp.f32 %0, %2, %3, p;\n\t}"
      : "=f"(r)
      : "r"(static_cast<int>(c)), "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ void unpack8x2(const uint4& u, float2 (&f)[4]) {
  bf16x2_to_f32(u.x, f[0].x, f[0].y);
  bf16x2_to_f32(u.y, f[1].x, f[1].y);
  bf16x2_to_f32(u.z, f[2].x, f[2].y);
  bf16x2_to_f32(u.w, f[3].x, f[3].y);
}

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

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Named barrier over the consumer warps only (the producer keeps streaming).
__device__ __forceinline__ void consumer_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Visible keys of request b's decode query: positions [t_lo, pos], blocks
// [jlo, jlo + nb).
struct ReqGeo {
  int jlo, nb, t_lo, pos;
};

__device__ __forceinline__ ReqGeo req_geo(const DecodeArgs& a, int b) {
  ReqGeo g;
  int L = a.seq_lens[b];
  if (L > a.max_blocks * kBlockSize || L < 0) {
    report(a.err, PKA_DEVERR_SEQ_LEN);  // error path only: tables cannot hold it
    L = max(0, min(L, a.max_blocks * kBlockSize));
  }
  g.pos = L - 1;
  g.t_lo = (a.window > 0) ? max(0, g.pos - a.window + 1) : 0;
  g.jlo = g.t_lo / kBlockSize;
  g.nb = (L > 0) ? (L + kBlockSize - 1) / kBlockSize - g.jlo : 0;
  return g;
}

// One piece of work: tiles [first, first + ntiles) of segment (b, kvh).
struct Piece {
  int b, kvh;
  int j0;        // logical block of the first tile
  int ntiles;
  int t_lo, pos;
  int qrow;      // query row of the request
  int slot;      // split-K partial slot (direct mode: unused)
  int fill_from; // >= 0: also write LSE=-inf into slots [fill_from, num_splits)
};

// Enumerates the pieces of one CTA.  Every lane of a warp runs it in
// lockstep (it uses warp scans), and every warp of the CTA sees the same
// sequence.
struct PieceIter {
  const DecodeArgs* a;
  bool direct;
  // direct mode
  int item;
  // split mode
  long long lo, hi, q;
  bool last;
  int b, kvh;
  long long prefix;  // sum of nb over requests before b
  ReqGeo geo;
  bool done;

  __device__ void init(const DecodeArgs& args, int lane) {
    a = &args;
    direct = args.split_blocks <= 0;
    done = false;
    if (direct) {
      item = blockIdx.x;
      return;
    }
    // total tiles T = Hkv * sum_b nb_b (the first 32 requests' counts stay in
    // a register, so batches of up to 32 requests read seq_lens once)
    long long T = 0;
    const int nb0 = (lane < args.batch) ? req_geo(args, lane).nb : 0;
    for (int base = 0; base < args.batch; base += 32) {
      const int bb = base + lane;
      const int nb = (base == 0) ? nb0 : ((bb < args.batch) ? req_geo(args, bb).nb : 0);
      T += __shfl_sync(0xffffffffu, warp_incl_scan(nb, lane), 31);
    }
    T *= args.Hkv;
    const long long grid = gridDim.x;
    q = max(static_cast<long long>(args.split_blocks), (T + grid - 1) / grid);
    const long long weff = T > 0 ? (T + q - 1) / q : 1;
    const long long c = blockIdx.x;
    if (c >= weff) {
      done = true;
      return;
    }
    lo = c * q;
    hi = min(T, lo + q);
    last = (c == weff - 1);
    // first request holding a segment this CTA touches: the first b with
    // Hkv*(prefix_b + nb_b) + (nb_b == 0) > lo
    long long run = 0;
    b = args.batch;
    prefix = run;
    for (int base = 0; base < args.batch; base += 32) {
      const int bb = base + lane;
      const int nb = (base == 0) ? nb0 : ((bb < args.batch) ? req_geo(args, bb).nb : 0);
      const int incl = warp_incl_scan(nb, lane);
      const long long pre = run + incl - nb;
      const bool hit = (bb < args.batch) &&
                       (static_cast<long long>(args.Hkv) * (pre + nb) + (nb == 0 ? 1 : 0) > lo);
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m) {
        const int first = __ffs(m) - 1;
        b = base + first;
        prefix = __shfl_sync(0xffffffffu, pre, first);
        break;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    kvh = 0;
    if (b < args.batch) geo = req_geo(args, b);
  }

  __device__ bool next(Piece& p) {
    if (done) return false;
    const DecodeArgs& A = *a;
    if (direct) {
      const int nseg = A.batch * A.Hkv;
      if (item >= nseg) {
        done = true;
        return false;
      }
      p.b = item / A.Hkv;
      p.kvh = item % A.Hkv;
      const ReqGeo g = req_geo(A, p.b);
      p.j0 = g.jlo;
      p.ntiles = g.nb;
      p.t_lo = g.t_lo;
      p.pos = g.pos;
      p.slot = 0;
      p.fill_from = -1;
      item += gridDim.x;
    } else {
      while (true) {
        if (b >= A.batch) {
          done = true;
          return false;
        }
        const long long seg = static_cast<long long>(A.Hkv) * prefix +
                              static_cast<long long>(kvh) * geo.nb;  // segment start
        const int n = geo.nb;
        const bool before = seg + (n > 0 ? n : 1) <= lo;  // wholly before this chunk
        const bool after = !last && seg >= hi;
        if (after) {
          done = true;
          return false;
        }
        const int cur_b = b, cur_kvh = kvh;
        const ReqGeo g = geo;
        // advance to the next segment
        if (++kvh == A.Hkv) {
          kvh = 0;
          prefix += geo.nb;
          ++b;
          if (b < A.batch) geo = req_geo(A, b);
        }
        if (before) continue;
        const long long t0 = max(seg, lo);
        const long long t1 = min(seg + n, hi);
        p.b = cur_b;
        p.kvh = cur_kvh;
        p.j0 = g.jlo + static_cast<int>(t0 - seg);
        p.ntiles = static_cast<int>(max(0LL, t1 - t0));
        p.t_lo = g.t_lo;
        p.pos = g.pos;
        const long long cfirst = seg / q;
        p.slot = static_cast<int>(static_cast<long long>(blockIdx.x) - cfirst);
        p.fill_from = -1;
        if (n == 0) {
          p.fill_from = 0;
        } else if (p.slot == 0) {
          p.fill_from = static_cast<int>((seg + n - 1) / q - cfirst + 1);
        }
        if (p.ntiles == 0 && p.fill_from < 0) continue;
        break;
      }
    }
    p.qrow = p.b;
    if (A.query_start_loc != nullptr) p.qrow = A.query_start_loc[p.b + 1] - 1;
    return true;
  }
};

}  // namespace

template <int D, int G, int NW, int NSLOT>
struct DecodeShape {
  // A ring slot holds TK keys of one (block, head) tile: a whole block for
  // D=128, half a block for D=256 (8 KB of K + V either way), so that many
  // consumer warps fit next to a deep ring.
  static constexpr int TK = (D == 256) ? 8 : 16;
  static constexpr int SUB = kBlockSize / TK;  // slots per pool block
  static constexpr int kTileElems = TK * D;
  static constexpr int kTileBytes = kTileElems * 2;
  static constexpr int LPK = D / 8;       // lanes per key row (16 bytes per lane)
  static constexpr int KPW = 32 / LPK;    // keys per warp step
  static constexpr int KC = (TK * G / KPW > 64) ? 8 : TK;  // keys per chunk
  static constexpr int KS = KC / KPW;     // warp steps per chunk
  static constexpr int NV = KS * G;       // partial dots per lane per chunk
  static constexpr int NVL = NV >= LPK ? NV / LPK : 1;
  static constexpr int DUP = NV >= LPK ? 1 : LPK / NV;
  static constexpr int kRingBytes = NSLOT * 2 * kTileBytes;
  static constexpr int kBarBytes = (2 * NSLOT * 8 + 15) / 16 * 16;
  static constexpr int kPBytes = (NW * KPW * NV * 4 + 15) / 16 * 16;
  // merge area: m and l of every (warp, head), padded to 16 bytes, then the
  // [NW][G][D] fp32 accumulators (written with 16-byte stores)
  static constexpr int kMergeMLFloats = (2 * NW * G + 3) / 4 * 4;
  static constexpr int kMergeBytes = (kMergeMLFloats + NW * G * D) * 4;
  static constexpr int kSmemBytes = kRingBytes + kBarBytes + kPBytes + kMergeBytes;
  static_assert(D % 8 == 0 && LPK <= 32 && 32 % LPK == 0, "head_dim");
  static_assert(KC % KPW == 0, "chunk");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(NSLOT % NW == 0, "each ring slot must have exactly one owner warp");
  static_assert(kTileBytes % 16 == 0 && kRingBytes % 16 == 0, "bulk-copy destinations 16-byte aligned");
  static_assert((kRingBytes + kBarBytes) % 16 == 0, "P area 16-byte aligned");
  static_assert((kRingBytes + kBarBytes + kPBytes) % 16 == 0, "merge area 16-byte aligned");
  static_assert((KPW * NV * 4) % 16 == 0 || G % 4 != 0, "per-warp P rows 16-byte aligned");
};

// Processes one ring slot (TK keys) for one consumer warp.  EDGE (warp
// uniform) selects the masked path for slots with keys outside the visible
// range.
template <int D, int G, int NW, int NSLOT>
__device__ __forceinline__ void decode_tile(const bool EDGE, const uint16_t* __restrict__ Kt,
                                            const uint16_t* __restrict__ Vt,
                                            const float2 (&qf)[G][4], float2 (&acc)[G][4],
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
  for (int c = 0; c < S::TK / KC; ++c) {
    // ---- partial q.k over this lane's 8 elements, every key step, every head
    float part[NV];
#pragma unroll
    for (int s = 0; s < KS; ++s) {
      const int key = c * KC + s * KPW + kl;
      const uint4 u = *reinterpret_cast<const uint4*>(Kt + key * D + dl * 8);
      float2 kf[4];
      unpack8x2(u, kf);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float2 d = fmul2(qf[g][0], kf[0]);
        d = ffma2(qf[g][1], kf[1], d);
        d = ffma2(qf[g][2], kf[2], d);
        d = ffma2(qf[g][3], kf[3], d);
        part[s * G + g] = d.x + d.y;
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
      for (int g = 0; g < G; ++g) mloc[g] = opaque_sel(gj[j] == g, fmaxf(mloc[g], x), mloc[g]);
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
        a = opaque_sel(gj[j] == g, alpha[g], a);
        r = opaque_sel(gj[j] == g, mref[g], r);
      }
      const float p = fast_exp2(part[j] - r);
      ls[j] = ls[j] * a + p;
      pw[(dl / DUP) * NVL + j] = p;
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float2 a2 = make_float2(alpha[g], alpha[g]);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[g][e] = fmul2(acc[g][e], a2);
    }
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
      float2 vf[4];
      unpack8x2(u, vf);
      float pg[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int g = 0; g < G; g += 4) {
          const float4 t4 = *reinterpret_cast<const float4*>(pw + s * G + g);
          pg[g] = t4.x;
          pg[g + 1] = t4.y;
          pg[g + 2] = t4.z;
          pg[g + 3] = t4.w;
        }
      } else {
#pragma unroll
        for (int g = 0; g < G; ++g) pg[g] = pw[s * G + g];
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float2 p2 = make_float2(pg[g], pg[g]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][e] = ffma2(p2, vf[e], acc[g][e]);
      }
    }
    __syncwarp();
  }
}

template <int D, int G, int NW, int NSLOT>
__global__ void __launch_bounds__((NW + 1) * 32, 1)
    paged_decode_kernel(const __grid_constant__ DecodeArgs a) {
  using S = DecodeShape<D, G, NW, NSLOT>;
  constexpr int TE = S::kTileElems;
  constexpr int NVL = S::NVL, LPK = S::LPK;

  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* ring = reinterpret_cast<uint16_t*>(smem);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kRingBytes);
  uint64_t* empty = full + NSLOT;
  float* psm_all = reinterpret_cast<float*>(smem + S::kRingBytes + S::kBarBytes);
  float* merge = reinterpret_cast<float*>(smem + S::kRingBytes + S::kBarBytes + S::kPBytes);
  float* mrg_m = merge;                       // [NW][G]
  float* mrg_l = merge + NW * G;              // [NW][G]
  float* mrg_acc = merge + S::kMergeMLFloats;  // [NW][G][D], 16-byte aligned

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_fence_init();
  }
  __syncthreads();

  PieceIter iter;
  iter.init(a, lane);
  Piece pc;

  if (warp == NW) {
    // ============================ producer warp ============================
    const uint64_t pol = policy_evict_first();
    long long issued = 0;
    bool ok = true;
    while (ok && iter.next(pc)) {
      const int32_t* trow = a.tables + static_cast<size_t>(pc.b) * a.max_blocks + pc.j0;
      for (int base = 0; base < pc.ntiles && ok; base += 32) {
        int id = 0;
        if (base + lane < pc.ntiles) {
          id = trow[base + lane];
          if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.num_blocks)) {
            report(a.err, PKA_DEVERR_BAD_TABLE);
            id = 0;
          }
        }
        const int cnt = min(32, pc.ntiles - base);
        for (int k = 0; k < cnt * S::SUB; ++k) {
          const int phys = __shfl_sync(0xffffffffu, id, k / S::SUB);
          const int slot = static_cast<int>(issued % NSLOT);
          const long long round = issued / NSLOT;
          int good = 1;
          if (lane == 0) {
            if (round > 0)
              good = mbar_wait(&empty[slot], static_cast<uint32_t>((round - 1) & 1), a.err);
            if (good) {
              mbar_arrive_expect_tx(&full[slot], 2 * S::kTileBytes);
              const size_t off = (static_cast<size_t>(phys) * a.Hkv + pc.kvh) * kBlockSize * D +
                                 static_cast<size_t>(k % S::SUB) * TE;
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

  // The next piece's query rows are loaded while the current piece is merged.
  bool have = iter.next(pc);
  uint4 qraw[G];
  if (have) {
    const uint16_t* qp = a.q + (static_cast<size_t>(pc.qrow) * a.Hq + pc.kvh * G) * D + dl * 8;
#pragma unroll
    for (int g = 0; g < G; ++g) qraw[g] = *reinterpret_cast<const uint4*>(qp + g * D);
  }
  while (have) {
    float2 qf[G][4], acc[G][4];
    float m[G], ls[NVL];
    {
      const float2 qs2 = make_float2(qscale, qscale);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        unpack8x2(qraw[g], qf[g]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qf[g][e] = fmul2(qf[g][e], qs2);
          acc[g][e] = make_float2(0.f, 0.f);
        }
        m[g] = -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < NVL; ++j) ls[j] = 0.f;
    }

    // Tile T of the CTA's stream lives in slot T % NSLOT and belongs to warp
    // T % NW; NSLOT is a multiple of NW, so every slot has one owner warp that
    // consumes its phases in order (a phase-parity wait can never alias an
    // older phase of the same slot).
    const int nsub = pc.ntiles * S::SUB;
    const int i0 = static_cast<int>((warp - tile_base % NW + NW) % NW);
    for (int i = i0; i < nsub && ok; i += NW) {
      const long long T = tile_base + i;
      const int slot = static_cast<int>(T % NSLOT);
      const bool got = mbar_wait(&full[slot], static_cast<uint32_t>((T / NSLOT) & 1), a.err);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      const uint16_t* Kt = ring + static_cast<size_t>(slot) * 2 * TE;
      const uint16_t* Vt = Kt + TE;
      const int tok0 = (pc.j0 + i / S::SUB) * kBlockSize + (i % S::SUB) * S::TK;
      const bool edge = (tok0 < pc.t_lo || tok0 + S::TK - 1 > pc.pos);
      decode_tile<D, G, NW, NSLOT>(edge, Kt, Vt, qf, acc, m, ls, psm, lane, tok0, pc.t_lo, pc.pos,
                                   a.softcap, inv_cap);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    tile_base += nsub;

    Piece nx;
    const bool have_next = iter.next(nx);
    if (have_next) {
      const uint16_t* qp = a.q + (static_cast<size_t>(nx.qrow) * a.Hq + nx.kvh * G) * D + dl * 8;
#pragma unroll
      for (int g = 0; g < G; ++g) qraw[g] = *reinterpret_cast<const uint4*>(qp + g * D);
    }

    const bool split = a.split_blocks > 0;
    if (pc.ntiles > 0) {
      // ---- per-warp totals: sums per head, accumulators across key lanes
      float lt[G];
#pragma unroll
      for (int g = 0; g < G; ++g) lt[g] = 0.f;
#pragma unroll
      for (int j = 0; j < NVL; ++j) {
        const int gj = ((dl / S::DUP) * NVL + j) % G;
#pragma unroll
        for (int g = 0; g < G; ++g) lt[g] += opaque_sel(gj == g, ls[j], 0.f);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) lt[g] = warp_sum(lt[g]) * (1.f / S::DUP);
#pragma unroll
      for (int o = LPK; o < 32; o <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[g][e].x += __shfl_xor_sync(0xffffffffu, acc[g][e].x, o);
            acc[g][e].y += __shfl_xor_sync(0xffffffffu, acc[g][e].y, o);
          }

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
          dst[0] = make_float4(acc[g][0].x, acc[g][0].y, acc[g][1].x, acc[g][1].y);
          dst[1] = make_float4(acc[g][2].x, acc[g][2].y, acc[g][3].x, acc[g][3].y);
        }
      }
      consumer_sync(NW * 32);

      // ---- merge the warps' states and write this piece's result
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
        const int h = pc.kvh * G + g;
        if (split) {
          if (pc.slot < a.num_splits) {
            const size_t ph = (static_cast<size_t>(pc.b) * a.Hq + h) * a.num_splits + pc.slot;
            a.partial_o[ph * D + d] = o;
            if (d == 0) a.partial_lse[ph] = (den > 0.f) ? (M + log2f(den)) * kLn2 : -INFINITY;
          }
        } else {
          reinterpret_cast<uint16_t*>(a.out)[(static_cast<size_t>(pc.qrow) * a.Hq + h) * D + d] =
              f32_to_bf16_rn(o);
        }
      }
      consumer_sync(NW * 32);
    } else if (!split) {
      // a request with no visible key: output 0
      for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
        const int h = pc.kvh * G + idx / D;
        reinterpret_cast<uint16_t*>(a.out)[(static_cast<size_t>(pc.qrow) * a.Hq + h) * D +
                                           idx % D] = 0;
      }
    }
    // ---- split-K: slots of this segment no CTA fills get LSE = -inf
    if (split && pc.fill_from >= 0) {
      if (pc.fill_from > a.num_splits && threadIdx.x == 0) report(a.err, PKA_DEVERR_SEQ_LEN);
      const int nfill = a.num_splits - min(pc.fill_from, a.num_splits);
      for (int idx = threadIdx.x; idx < G * nfill; idx += NW * 32) {
        const int h = pc.kvh * G + idx / nfill;
        const int s = pc.fill_from + idx % nfill;
        a.partial_lse[(static_cast<size_t>(pc.b) * a.Hq + h) * a.num_splits + s] = -INFINITY;
      }
    }
    pc = nx;
    have = have_next;
  }
}

// ------------------------------------------------------------- launchers
namespace {

template <int D, int G>
struct DecodeTuning {
  // NW consumer warps + 1 producer warp, one CTA per SM: eight warps, two per
  // scheduler, so a thread may hold up to 255 registers (no spills).  The
  // ring has SPW slots per consumer warp (each slot owned by one warp).
  static constexpr int NW = 7;
  static constexpr int SPW = (G == 8) ? 2 : 3;
  static constexpr int NSLOT = NW * SPW;
};

template <int D, int G>
cudaError_t launch_decode_t(const DecodeArgs& a, int grid, cudaStream_t stream) {
  constexpr int NW = DecodeTuning<D, G>::NW;
  constexpr int NSLOT = DecodeTuning<D, G>::NSLOT;
  using S = DecodeShape<D, G, NW, NSLOT>;
  auto kern = paged_decode_kernel<D, G, NW, NSLOT>;
  cudaError_t e = set_smem_once(reinterpret_cast<const void*>(kern), S::kSmemBytes);
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
