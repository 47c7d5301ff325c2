// Paged prefill and mixed-batch attention on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), sm_103a.
//
// The chunked-prefill contractions are dense: a chunk of new tokens attends,
// causally, over its request's cached prefix and the chunk itself, K/V read
// through the block table ("Triton paged decode and prefill kernels reading
// K/V through block tables", inference-server README, engine feature list;
// mixed-batch chunked prefill, architecture page, "Phase status").  Decode
// rows (one token) may sit in the same varlen launch.
//
// Work item = (request, KV head, query tile).  A query tile packs TQ = 128/G
// tokens x the G query heads of one KV group into the 128 rows of the MMA
// (row = token * G + g), so all G heads share every K/V tile.  Per item:
//
//  * warps 4 and 7 (TMA): the Q tile (one 3-D box per 64-column chunk) and,
//    per key tile, one 2-D box per (pool block, 64-column chunk) of K into a
//    3-stage ring, each warp half of the blocks (a TMA copy costs the issuing
//    warp ~80 cycles whatever its size, and a tile has 16 such boxes); blocks
//    past the request's last block get an out-of-range row coordinate so TMA
//    fills zeros; a stage is refilled once S = Q K^T of the tile it held has
//    completed;
//  * warp 5 (TMA): V, one 3-D copy per block (block-major stages, which the
//    P V MMA reads one 16-key block at a time), 2 stages, refilled once P V
//    of its tile completed;
//  * warp 6 (MMA): allocates TMEM (2 S buffers + the O accumulator), issues
//    S_j = Q K_j^T (K-major A and B, 128B-swizzled) two tiles ahead, then
//    O += P_j V_j with P_j read from TMEM and V as an MN-major shared-memory
//    operand, committing each to mbarriers; it also zeroes V rows past
//    seq_len (stale slots of the last block, which may hold NaN) before they
//    reach P V;
//  * warps 0-3 (softmax): thread r owns row r.  It reads its S row from
//    TMEM, applies scale, softcap and the causal / window mask, keeps a
//    running max and sum in the exp2 domain, writes P (bf16 pairs) to its
//    own TMEM columns and signals the MMA warp (P never
//    touches shared memory, which holds Q and the K/V rings).  O is rescaled in TMEM only
//    when the row max grows by more than 2^8 (the stale reference max keeps
//    every P <= 256, and O and the sum share it, so the result is exact);
//  * epilogue: O / sum from TMEM to bf16 rows of the output.
//
// All waits are bounded; a timeout sets PKA_DEVERR_TIMEOUT, the roles stop,
// the CTA still frees its TMEM.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pka {

template <int D, int G>
struct PrefillShape {
  static constexpr int BM = 128;                    // MMA rows: tokens x heads
  static constexpr int TQ = BM / G;                 // tokens per query tile
  static constexpr int BN = (D == 256) ? 64 : 128;  // keys per key tile
  static constexpr int DC = D / 64;                 // 128-byte chunks of a K/V/Q row
  static constexpr int kBlocksPerTile = BN / kBlockSize;
  static constexpr int kQChunk = BM * 128;
  static constexpr int kKVChunk = BN * 128;        // K stage: [D/64 chunks][BN rows][128 B]
  static constexpr int kVBlock = kBlockSize * D * 2;  // V stage: [BN/16 blocks][D/64 chunks][16 rows][128 B]
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int kKVBytes = BN * D * 2;
  static constexpr int KST = 3;                     // K ring stages
  static constexpr int VST = 2;                     // V ring stages
  static constexpr int oQ = 0;
  static constexpr int oK = oQ + kQBytes;
  static constexpr int oV = oK + KST * kKVBytes;
  static constexpr int oBar = oV + VST * kKVBytes;
  static constexpr int kNumBars = 15;
  static constexpr int oMisc = oBar + kNumBars * 8;
  static constexpr int kSmemBytes = oMisc + 16 + 1024;  // + slack to align the base to 1 KiB
  // TMEM columns: S_j (fp32, BN columns) in buffer j % 2 at (j % 2) * BN;
  // O (fp32) at [256, 256 + D); P_j (bf16 pairs, BN / 2 columns), the A
  // operand of P_j V_j, in buffer j % 2 at kTmemP + (j % 2) * BN / 2.  P has
  // columns of its own: S_{j+2} may be written while P_j V_j still reads P_j
  // (consecutive MMAs overlap in the pipe), so P_j must not alias S_j.
  static constexpr uint32_t kTmemO = 256;
  static constexpr uint32_t kTmemP = (D == 256) ? 2 * BN : 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 8 * 32;
  // cost buckets of the heaviest-first ranking (scratch in the K stages)
  static constexpr int kCostBuckets = 4096;
  static_assert((kCostBuckets + 64) * 4 <= KST * kKVBytes, "ranking scratch");
  static_assert(BN % 64 == 0, "P is stored to TMEM 32 columns (64 keys) at a time");
  static_assert(kTmemP >= 2 * BN && (kTmemP + BN <= kTmemO || kTmemP >= kTmemO + D) &&
                    kTmemP + BN <= kTmemCols,
                "P buffers clear of S and O");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(2 * BN <= 256 && D <= 256, "TMEM columns");
};

// Built with -DPKA_TIMELINE (instrumented builds only), every prefill CTA
// records global-timer stamps: [rank][entry, first S tile ready, last P V
// done, exit, key tiles].  The default build compiles none of it.
constexpr int kPrefillStampRanks = 1024;
#ifdef PKA_TIMELINE
__device__ unsigned long long pka_timeline_prefill[kPrefillStampRanks * 5];
#define PKA_PF_SET(rank, f) \
  do { if ((rank) < kPrefillStampRanks) pka_timeline_prefill[(rank) * 5 + (f)] = timeline_now(); } while (0)
#define PKA_PF_VAL(rank, f, v) \
  do { if ((rank) < kPrefillStampRanks) pka_timeline_prefill[(rank) * 5 + (f)] = (v); } while (0)
#else
#define PKA_PF_SET(rank, f) do { } while (0)
#define PKA_PF_VAL(rank, f, v) do { } while (0)
#endif

namespace {

constexpr int kWarpTmaK = 4;
constexpr int kWarpTmaV = 5;
constexpr int kWarpMma = 6;
constexpr int kWarpTmaK2 = 7;
// named barrier of the four softmax warps (the epilogue's staged stores)
constexpr int kBarSoftmax = 1;

struct Item {
  int b, kvh, q0, n, L, it0, it1, kbase, ntiles, nblk;
};

// bar indices
// Every ring stage has its own "empty" barrier (K: B_KEMPTY, V: B_PV, whose
// two barriers are the two V stages), so a producer waiting for use r - 1 of
// a stage can never see the barrier one phase further on: use r cannot
// complete before the producer has loaded it.
enum { B_Q = 0, B_KFULL = 1, B_VFULL = 4, B_QK = 6, B_PV = 8, B_PRDY = 10, B_KEMPTY = 12 };

__device__ __forceinline__ bool stop_requested(const volatile int* flag) { return *flag != 0; }

__device__ __forceinline__ bool cta_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                         volatile int* failed) {
  if (mbar_wait(bar, parity, err)) return true;
  *failed = 1;
  return false;
}

// Every lane waits; the warp agrees on one outcome so that it never diverges.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int32_t* err,
                                          volatile int* failed) {
  const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, err));
  if (!ok) *failed = 1;
  return ok;
}

// Packed fp32 pairs (sm_100 family): one instruction computes both lanes of
// a float2, each rounded exactly as the scalar fmaf / a * b / a + b is.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// Three-input maximum and minimum (sm_100 family): fmaxf / fminf of three.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// exp2-based tanh: tanh(y) = 1 - 2 / (exp(2y) + 1); absolute error ~1e-7.
__device__ __forceinline__ float tanh_via_exp2(float y) {
  const float e = fast_exp2(fminf(2.f * kLog2e * y, 126.f));
  return 1.f - __fdividef(2.f, e + 1.f);
}

// tanh(y) for |y| < 0.5 from its odd Taylor series through y^11 (the first
// omitted term, 21844 y^13 / 6081075, is below 4.5e-7 there): FMA-pipe work
// only, where the exp2 form needs two MUFU operations.
// tanh(y) for |y| < 1/8 from y - y^3/3 + 2 y^5/15 (the first omitted term,
// 17 y^7 / 315, is below 2.6e-8 there): four FMA-pipe operations.
__device__ __forceinline__ float tanh_taylor_short(float y) {
  const float y2 = y * y;
  const float q = fmaf(y2, 2.f / 15.f, -1.f / 3.f);
  return fmaf(y * y2, q, y);
}

__device__ __forceinline__ float tanh_taylor(float y) {
  const float y2 = y * y;
  float q = fmaf(y2, -1382.f / 155925.f, 62.f / 2835.f);
  q = fmaf(y2, q, -17.f / 315.f);
  q = fmaf(y2, q, 2.f / 15.f);
  q = fmaf(y2, q, -1.f / 3.f);
  return fmaf(y * y2, q, y);
}

// Query rows [*q0, *q0 + n) of request b; returns n.  A request whose span
// is not 0 <= query_start_loc[b] <= query_start_loc[b+1] <= total_q, or is
// longer than max_query_len, gets n = -1: it has no tile and no row of it is
// written (the first pass over the requests reports it).
__device__ __forceinline__ int query_span(const PrefillArgs& a, int b, int* q0) {
  const int lo = a.query_start_loc[b], hi = a.query_start_loc[b + 1];
  *q0 = lo;
  if (lo < 0 || hi < lo || hi > a.total_q || hi - lo > a.max_query_len) return -1;
  return hi - lo;
}

// Cost in key tiles of query tile qt of a request with n query rows and
// context length L (clamped to the table) (0: no query row there).
template <int TQ, int BN>
__device__ __forceinline__ int tile_cost_nl(const PrefillArgs& a, int n, int L, int qt) {
  const int it0 = qt * TQ;
  if (n <= 0 || n > L || it0 >= n || (a.skip_decode_rows != 0 && n == 1)) return 0;
  const int it1 = min(n, it0 + TQ) - 1;
  const int p_first = L - n + it0;
  const int p_last = L - n + it1;
  const int t_lo = (a.window > 0) ? max(0, p_first - a.window + 1) : 0;
  return (p_last + 1 - (t_lo & ~(kBlockSize - 1)) + BN - 1) / BN + 1;
}

// Requests whose (n, L) the ranking keeps in shared memory (more: read from
// global memory at every use).
constexpr int kReqCache = 4096;
constexpr int kReqCacheOffset = 4224;  // ints, past the ranking's own scratch

// tile_cost_nl for request b, its (n, L) from the shared-memory copy when
// rn != nullptr.
template <int TQ, int BN>
__device__ __forceinline__ int tile_cost(const PrefillArgs& a, const int* rn, const int* rL,
                                         int b, int qt) {
  if (rn != nullptr) return tile_cost_nl<TQ, BN>(a, rn[b], rL[b], qt);
  int q0;
  const int n = query_span(a, b, &q0);
  const int L = min(a.seq_lens[b], a.max_blocks * kBlockSize);
  return tile_cost_nl<TQ, BN>(a, n, L, qt);
}

// Block-wide exclusive scan of one int per thread (blockDim.x <= 1024).
__device__ __forceinline__ int block_excl_scan(int x, int* warp_sums, int* total) {
  const int lane = threadIdx.x % 32, warp = threadIdx.x / 32, nw = (blockDim.x + 31) / 32;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (threadIdx.x == 0) {
    int run = 0;
    for (int w = 0; w < nw; ++w) {
      const int t = warp_sums[w];
      warp_sums[w] = run;
      run += t;
    }
    *total = run;
  }
  __syncthreads();
  const int r = warp_sums[warp] + incl - x;
  __syncthreads();
  return r;
}

// Longest-processing-time-first order of the (request, query tile) pairs.
// Every CTA ranks all pairs by cost (heaviest first, ties by index) with a
// counting sort in shared memory and returns the pair of rank `rank`; the
// hardware launches CTAs in blockIdx order, so the heaviest tiles start first
// and the light ones fill the tail.  All CTAs compute the same order.
template <int TQ, int BN>
__device__ int lpt_pair(const PrefillArgs& a, int qtiles, int rank, int* scratch, int nbuck,
                        const int* rn, const int* rL) {
  const int npairs = a.batch * qtiles;
  if (npairs <= static_cast<int>(blockDim.x)) {
    // Few pairs: one thread per pair counts the pairs ahead of it in the
    // same order (cost bucket descending, index ascending) -- the rank the
    // counting sort below gives, in one pass over shared memory.
    int* cost = scratch;                // [npairs]
    int* found = scratch + blockDim.x;  // [1]
    const int i = threadIdx.x;
    int c = 0;
    if (i < npairs) {
      c = min(tile_cost<TQ, BN>(a, rn, rL, i / qtiles, i % qtiles), nbuck - 1);
      cost[i] = c;
    }
    if (i == 0) *found = 0;
    __syncthreads();
    if (i < npairs) {
      int ahead = 0;
      for (int k = 0; k < npairs; ++k) {
        const int ck = cost[k];
        ahead += (ck > c || (ck == c && k < i)) ? 1 : 0;
      }
      if (ahead == rank) *found = i;
    }
    __syncthreads();
    const int pair = *found;
    __syncthreads();
    return pair;
  }
  int* hist = scratch;                  // [nbuck]
  int* warp_sums = scratch + nbuck;     // [32]
  int* misc = warp_sums + 32;           // [4]
  for (int k = threadIdx.x; k < nbuck; k += blockDim.x) hist[k] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < npairs; i += blockDim.x)
    atomicAdd(&hist[min(tile_cost<TQ, BN>(a, rn, rL, i / qtiles, i % qtiles), nbuck - 1)], 1);
  __syncthreads();
  // start of bucket k in the descending order: pairs in buckets > k.  Each
  // thread owns a run of buckets counted from the top.
  const int per = (nbuck + blockDim.x - 1) / blockDim.x;
  const int hi_k = nbuck - 1 - static_cast<int>(threadIdx.x) * per;  // first bucket of the run
  int mine = 0;
  for (int u = 0; u < per; ++u)
    if (hi_k - u >= 0) mine += hist[hi_k - u];
  int run = block_excl_scan(mine, warp_sums, &misc[0]);
  for (int u = 0; u < per; ++u) {
    const int k = hi_k - u;
    if (k < 0) break;
    const int c = hist[k];
    if (rank >= run && rank < run + c) {  // exactly one thread matches
      misc[1] = k;
      misc[2] = rank - run;
    }
    run += c;
  }
  __syncthreads();
  const int kb = misc[1], off = misc[2];
  // the off-th pair (in index order) of bucket kb
  const int chunk = (npairs + blockDim.x - 1) / blockDim.x;
  const int i0 = threadIdx.x * chunk, i1 = min(npairs, i0 + chunk);
  int cnt = 0;
  for (int i = i0; i < i1; ++i)
    cnt += (min(tile_cost<TQ, BN>(a, rn, rL, i / qtiles, i % qtiles), nbuck - 1) == kb);
  const int before = block_excl_scan(cnt, warp_sums, &misc[0]);
  if (off >= before && off < before + cnt) {
    int seen = before;
    for (int i = i0; i < i1; ++i) {
      if (min(tile_cost<TQ, BN>(a, rn, rL, i / qtiles, i % qtiles), nbuck - 1) == kb) {
        if (seen == off) {
          misc[3] = i;
          break;
        }
        ++seen;
      }
    }
  }
  __syncthreads();
  const int pair = misc[3];
  __syncthreads();
  return pair;
}

// ------------------------------------------------ one wave, split along keys
// When every (request, query tile, KV head) item fits in one wave of the
// CTAs that run at once (a.one_wave), the order of the items does not
// matter and no ranking is needed: CTA r takes unit r in index order.  With
// a split workspace, the items' key tiles are also cut into pieces, so that
// the units fill the wave: the smallest piece length theta (>= kMinPieceTiles
// tiles) for which sum over items of min(kMaxPieces, ceil(tiles / theta))
// pieces fits, found by bisection.  Piece k of an item of T tiles and P
// pieces takes tiles [k T / P, (k + 1) T / P).
constexpr int kMaxList = 256;         // (request, query tile) pairs the list holds
constexpr int kListOffset = 12416;    // ints, past the request cache
constexpr int kMinPieceTiles = 4;     // shortest piece worth a CTA of its own
constexpr int kMaxPieces = 8;         // pieces of one item at most

struct Unit {
  int b, qt, kvh, piece, npieces, slot0;  // slot0: the unit of the item's piece 0
};

__device__ __forceinline__ int pieces_of(int tiles, int theta) {
  return min(kMaxPieces, max(1, (tiles + theta - 1) / theta));
}

// Every thread of the CTA calls it (it uses __syncthreads); returns false
// (uniformly) when rank has no unit.  pairs: the pairs with work (<= kMaxList).
template <int TQ, int BN>
__device__ bool one_wave_unit(const PrefillArgs& a, int rank, int pairs, bool split,
                              int* scratch, const int* rn, const int* rL, Unit* u) {
  int* list = scratch + kListOffset;        // [kMaxList][4]: b, qt, tiles, pieces
  int* uoff = list + 4 * kMaxList;          // [kMaxList]: first unit of the pair
  int* misc = uoff + kMaxList;              // [4]
  const int lane = threadIdx.x % 32;
  if (threadIdx.x < 32) {
    // the pairs with work in index order: request-major, query tiles within
    int run = 0;
    for (int base = 0; base < a.batch; base += 32) {
      const int b = base + lane;
      int n = 0, L = 0;
      if (b < a.batch) {
        if (rn != nullptr) {
          n = rn[b];
          L = rL[b];
        } else {
          int q0;
          n = query_span(a, b, &q0);
          L = min(a.seq_lens[b], a.max_blocks * kBlockSize);
        }
      }
      const int t = (n > 0 && n <= L && !(a.skip_decode_rows != 0 && n == 1)) ? (n + TQ - 1) / TQ
                                                                              : 0;
      int incl = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int off = run + incl - t;
      for (int q = 0; q < t && off + q < kMaxList; ++q) {
        int* e = list + 4 * (off + q);
        e[0] = b;
        e[1] = q;
        e[2] = tile_cost_nl<TQ, BN>(a, n, L, q) - 1;  // key tiles of the pair
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    // pieces per pair: theta by bisection over [kMinPieceTiles, longest]
    int theta = 0x40000000;
    if (split) {
      int longest = 0;
      for (int e = lane; e < pairs; e += 32) longest = max(longest, list[4 * e + 2]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) longest = max(longest, __shfl_xor_sync(0xffffffffu, longest, o));
      const int budget = min(a.one_wave, a.split_slots);
      int lo = kMinPieceTiles, hi = max(kMinPieceTiles, longest);
      while (lo < hi) {
        const int mid = (lo + hi) / 2;
        int units = 0;
        for (int e = lane; e < pairs; e += 32) units += pieces_of(list[4 * e + 2], mid);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) units += __shfl_xor_sync(0xffffffffu, units, o);
        if (units * a.Hkv <= budget)
          hi = mid;
        else
          lo = mid + 1;
      }
      theta = hi;
    }
    run = 0;
    for (int base = 0; base < pairs; base += 32) {
      const int e = base + lane;
      const int pc = (e < pairs) ? (split ? pieces_of(list[4 * e + 2], theta) : 1) : 0;
      int incl = pc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < pairs) {
        list[4 * e + 3] = pc;
        uoff[e] = (run + incl - pc) * a.Hkv;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      misc[0] = run * a.Hkv;  // units
      misc[1] = -1;
    }
  }
  __syncthreads();
  const bool has = rank < misc[0];
  if (has) {
    for (int e = threadIdx.x; e < pairs; e += blockDim.x)
      if (rank >= uoff[e] && rank < uoff[e] + list[4 * e + 3] * a.Hkv) misc[1] = e;
  }
  __syncthreads();
  if (has) {
    const int e = misc[1];
    const int pc = list[4 * e + 3];
    const int r = rank - uoff[e];
    u->b = list[4 * e];
    u->qt = list[4 * e + 1];
    u->npieces = pc;
    u->kvh = r / pc;
    u->piece = r % pc;
    u->slot0 = uoff[e] + u->kvh * pc;
  }
  __syncthreads();  // the scratch is free again
  return has;
}

}  // namespace

// Ranks (CTAs) a prefill launch needs: one per (request, query tile, KV
// head) with work.  A request of n rows has ceil(n / TQ) <= 1 + (n - 1) / TQ
// query tiles (0 when n = 0), so B requests of total_q rows have at most
// B + (total_q - B) / TQ, and at most B * ceil(max_query_len / TQ).
inline long long prefill_ranks(const PrefillArgs& a, int TQ) {
  const long long qtiles = (a.max_query_len + TQ - 1) / TQ;
  long long pairs = static_cast<long long>(a.batch) * qtiles;
  const long long extra = static_cast<long long>(a.total_q) - a.batch;
  const long long bound = a.batch + (extra > 0 ? extra / TQ : 0);
  if (bound < pairs) pairs = bound;
  return pairs * a.Hkv;
}

// One prefill work item per CTA on the S::kSmemBytes of shared memory at
// smem_raw: the item of rank `rank` (heaviest first; ranks past the last
// item return at once).
// kSplit: the body can run pieces of items split along keys (the mixed
// launch); without it the merge code is not compiled in.
template <int D, int G, bool kSplit>
__device__ __forceinline__ void prefill_body(const PrefillArgs& a, const CUtensorMap* tm_q,
                                             const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                             const CUtensorMap* tm_out, uint8_t* smem_raw,
                                             int rank) {
  using S = PrefillShape<D, G>;
  constexpr int BN = S::BN, TQ = S::TQ, DC = S::DC;

  // ---------------------------------------------------------- work item
  // ------------------------------------------------------- shared memory
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));

  // ---------------------------------------------------------- work item
  // 1-D grid over (pair rank, KV head): CTA r takes the (r / Hkv)-th heaviest
  // (request, query tile) pair, KV head r % Hkv.  The K stage buffers are
  // free until the first TMA load, so the ranking uses them as scratch.
  Item it;
  const int qtiles = (a.max_query_len + TQ - 1) / TQ;
  // Ranks past the number of (request, query tile) pairs with work leave
  // before the ranking: a request of n query rows has ceil(n / TQ) such
  // pairs (the ones tile_cost rates above zero).
  // The same pass keeps every request's (n, L) in shared memory for the
  // ranking, which would otherwise read them once per query tile.
  int* scratch = reinterpret_cast<int*>(smem + S::oK);
  const bool cache = a.batch <= kReqCache;
  int* rn = cache ? scratch + kReqCacheOffset : nullptr;
  int* rL = cache ? rn + kReqCache : nullptr;
  static_assert((kReqCacheOffset + 2 * kReqCache) * 4 <= S::KST * S::kKVBytes,
                "the request cache fits in the K stages");
  static_assert(kListOffset >= kReqCacheOffset + 2 * kReqCache &&
                    (kListOffset + 5 * kMaxList + 4) * 4 <= S::KST * S::kKVBytes,
                "the pair list fits in the K stages, past the request cache");
  int pairs_with_work = 0;
  {
    int cnt = 0;
    for (int b = threadIdx.x; b < a.batch; b += blockDim.x) {
      int q0;
      const int n = query_span(a, b, &q0);
      if (n < 0 && rank == 0) report(a.err, PKA_DEVERR_QUERY_LOC);
      const int L = min(a.seq_lens[b], a.max_blocks * kBlockSize);
      if (cache) {
        rn[b] = n;
        rL[b] = L;
      }
      if (n > 0 && n <= L && !(a.skip_decode_rows != 0 && n == 1)) cnt += (n + TQ - 1) / TQ;
    }
    block_excl_scan(cnt, scratch, scratch + 32);  // also orders rn / rL for every thread
    pairs_with_work = scratch[32];
    __syncthreads();
  }
  // One wave: index order, and with a split workspace pieces along keys.
  // More items than CTAs at once: heaviest first, whole items.
  const long long items = static_cast<long long>(pairs_with_work) * a.Hkv;
  int qt;
  Unit un{0, 0, 0, 0, 1, 0};
  if (items <= a.one_wave && pairs_with_work <= kMaxList) {
    const bool split =
        kSplit && a.split_o != nullptr && items < a.one_wave && items <= a.split_slots;
    if (!one_wave_unit<TQ, BN>(a, rank, pairs_with_work, split, scratch, rn, rL, &un)) return;
    it.b = un.b;
    it.kvh = un.kvh;
    qt = un.qt;
  } else {
    if (rank / a.Hkv >= pairs_with_work) return;  // uniform
    // costs are at most ceil(max_seq_len / BN) + 1 key tiles
    const int nbuck = min(S::kCostBuckets, (a.max_seq_len + BN - 1) / BN + 2);
    const int pair = lpt_pair<TQ, BN>(a, qtiles, rank / a.Hkv, scratch, nbuck, rn, rL);
    it.b = pair / qtiles;
    it.kvh = rank % a.Hkv;
    qt = pair % qtiles;
  }
  it.n = query_span(a, it.b, &it.q0);
  if (it.n < 0) return;  // uniform (reported by the first pass)
  it.L = a.seq_lens[it.b];
  if (it.L > a.max_blocks * kBlockSize) {
    if (threadIdx.x == 0 && qt == 0 && it.kvh == 0) report(a.err, PKA_DEVERR_SEQ_LEN);
    it.L = a.max_blocks * kBlockSize;
  }
  if (it.n > it.L) {
    if (threadIdx.x == 0 && qt == 0 && it.kvh == 0) report(a.err, PKA_DEVERR_SEQ_LEN);
    return;
  }
  it.it0 = qt * TQ;
  // uniform: nothing to do for this tile (or a decode row left to the
  // decode pipelines of a mixed launch)
  if (it.n <= 0 || it.it0 >= it.n || (a.skip_decode_rows != 0 && it.n == 1)) return;
  it.it1 = min(it.n, it.it0 + TQ) - 1;
  const int p_first = it.L - it.n + it.it0;
  const int p_last = it.L - it.n + it.it1;
  const int t_lo = (a.window > 0) ? max(0, p_first - a.window + 1) : 0;
  it.kbase = t_lo & ~(kBlockSize - 1);
  it.ntiles = (p_last + 1 - it.kbase + BN - 1) / BN;
  it.nblk = (it.L + kBlockSize - 1) / kBlockSize;
  if (un.npieces > 1) {
    // this piece's key tiles
    const int j0 = un.piece * it.ntiles / un.npieces;
    const int j1 = (un.piece + 1) * it.ntiles / un.npieces;
    it.kbase += j0 * BN;
    it.ntiles = j1 - j0;
  }

  uint8_t* sQ = smem + S::oQ;
  uint8_t* sK = smem + S::oK;
  uint8_t* sV = smem + S::oV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::oBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::oMisc);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + S::oMisc + 4);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    PKA_PF_SET(rank, 0);
    PKA_PF_VAL(rank, 4, static_cast<unsigned long long>(it.ntiles));
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars[B_Q], 1);
    for (int i = 0; i < S::KST; ++i) {
      mbar_init(&bars[B_KFULL + i], 1);
      mbar_init(&bars[B_KEMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[B_VFULL + i], 1);
      mbar_init(&bars[B_QK + i], 1);
      mbar_init(&bars[B_PV + i], 1);
      mbar_init(&bars[B_PRDY + i], 128);
    }
    *failed = 0;
    mbar_fence_init();
  }
  if (warp == kWarpMma) tmem_alloc(tmem_slot, S::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t oob_row = static_cast<uint32_t>(a.num_blocks) * a.Hkv * kBlockSize;
  const int32_t* trow = a.tables + static_cast<size_t>(it.b) * a.max_blocks;

  if (warp == kWarpTmaK || warp == kWarpTmaK2 || warp == kWarpTmaV) {
    // ============================ TMA producers ============================
    // K stage j % KST is refilled once S_j = Q K_j^T has completed, V stage
    // j % VST once P_j V_j has.  Issuing a TMA copy costs its warp ~80 cycles
    // whatever the size, so the 16 boxes of a K tile are split over two
    // warps and V is read with one 3-D copy per block.
    const bool is_k = (warp != kWarpTmaV);
    const int kpart = (warp == kWarpTmaK2) ? 1 : 0;
    const int nst = is_k ? S::KST : S::VST;
    uint8_t* ring = is_k ? sK : sV;
    uint64_t* full = &bars[is_k ? B_KFULL : B_VFULL];
    static_assert(S::VST == 2, "the two P V barriers double as the V stages' empty barriers");
    uint64_t* freed = &bars[is_k ? B_KEMPTY : B_PV];
    int issued = 0;
    if (lane == 0) {
      prefetch_tensormap(is_k ? tm_k : tm_v);
      if (warp == kWarpTmaK) {
        prefetch_tensormap(tm_q);
        mbar_arrive_expect_tx(&bars[B_Q], S::kQBytes);
#pragma unroll
        for (int c = 0; c < DC; ++c)
          tma_load_3d(sQ + c * S::kQChunk, tm_q, c * 64, it.kvh * G, it.q0 + it.it0, &bars[B_Q]);
      }
    }
    // Pool rows of the item's blocks, read by the whole warp 32 at a time
    // (one coalesced load) into a window of 64 blocks held one per lane in
    // two registers (the second half is read ahead); the issuing lanes take
    // them by shuffle.  Block b (counted from the first key tile) maps to
    // TMA row (id * Hkv + kvh) * 16, or to an out-of-range row past the
    // request's last block (TMA fills zeros).
    constexpr int BPT = S::kBlocksPerTile;
    static_assert(32 % BPT == 0, "a tile's blocks never straddle two 32-block windows");
    const int jb0 = it.kbase / kBlockSize;
    auto load_rows = [&](int base) -> uint32_t {
      const int jb = jb0 + base + lane;
      uint32_t row = oob_row;
      if (jb < it.nblk) {
        const int id = trow[jb];
        if (static_cast<unsigned>(id) < static_cast<unsigned>(a.num_blocks))
          row = (static_cast<uint32_t>(id) * a.Hkv + it.kvh) * kBlockSize;
        else
          report(a.err, PKA_DEVERR_BAD_TABLE);
      }
      return row;
    };
    int win = 0;  // rows_lo: blocks [win, win + 32); rows_hi: the next 32
    uint32_t rows_lo = load_rows(0), rows_hi = load_rows(32);
    for (int j = 0; j < it.ntiles; ++j) {
      if (__any_sync(0xffffffffu, stop_requested(failed))) break;
      if (j * BPT >= win + 32) {
        rows_lo = rows_hi;
        rows_hi = load_rows(win + 64);
        win += 32;
      }
      uint32_t rl[BPT];
#pragma unroll
      for (int kb = 0; kb < BPT; ++kb)
        rl[kb] = __shfl_sync(0xffffffffu, rows_lo, (j * BPT + kb - win) & 31);
      const int st = j % nst;
      int good = 1;
      if (lane == 0) {
        if (j >= nst && !cta_wait(&freed[st], (j / nst - 1) & 1, a.err, failed)) good = 0;
        // one expect for the whole stage (the other K warp's copies count too)
        if (good && kpart == 0) mbar_arrive_expect_tx(&full[st], S::kKVBytes);
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) break;
      uint8_t* dst = ring + st * S::kKVBytes;
      if (is_k) {
        // K: chunk-major (the S MMA reads 64 keys of one 64-column chunk as
        // 8 uniformly strided 8-row groups), one box per (block, chunk); this
        // warp takes blocks [kpart * BPT / 2, (kpart + 1) * BPT / 2)
        if (lane < (BPT / 2) * DC) {
          const int kb = kpart * (BPT / 2) + lane / DC, c = lane % DC;
          uint32_t r = rl[0];
#pragma unroll
          for (int q = 1; q < BPT; ++q)
            if (kb == q) r = rl[q];
          tma_load_2d(dst + c * S::kKVChunk + kb * kBlockSize * 128, tm_k, c * 64,
                      static_cast<int>(r), &full[st]);
        }
      } else if (lane < BPT) {
        // V: block-major (each P V MMA reads one block's 16 keys), one 3-D
        // copy per block
        uint32_t r = rl[0];
#pragma unroll
        for (int q = 1; q < BPT; ++q)
          if (lane == q) r = rl[q];
        tma_load_3d(dst + lane * S::kVBlock, tm_v, 0, static_cast<int>(r), 0, &full[st]);
      }
      issued = j + 1;
    }
    if (lane == 0) {
      // every issued copy must land before the CTA may finish
      for (int j = issued - nst < 0 ? 0 : issued - nst; j < issued; ++j)
        mbar_wait(&full[j % nst], (j / nst) & 1, a.err);
      if (warp == kWarpTmaK && stop_requested(failed)) mbar_wait(&bars[B_Q], 0, a.err);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ================================ MMA ================================
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, BN, 0, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
    const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
    int committed_pv = 0;  // number of P V tiles issued
    bool ok = warp_wait(&bars[B_Q], 0, a.err, failed);
    auto issue_qk = [&](int j) -> bool {
      const int st = j & 1;  // S buffer
      const int ks = j % S::KST;
      if (!warp_wait(&bars[B_KFULL + ks], (j / S::KST) & 1, a.err, failed)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t kst = aK + ks * S::kKVBytes;
#pragma unroll
        for (int c = 0; c < DC; ++c)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t da = smem_desc_sw128(aQ + c * S::kQChunk + kk * 32, 16, 1024);
            const uint64_t db = smem_desc_sw128(kst + c * S::kKVChunk + kk * 32, 16, 1024);
            umma_bf16(tmem + st * BN, da, db, idesc_qk, (c | kk) != 0);
          }
        umma_commit(&bars[B_QK + st]);
        umma_commit(&bars[B_KEMPTY + ks]);
      }
      __syncwarp();
      return true;
    };
    if (ok) ok = issue_qk(0);
    if (ok && it.ntiles > 1) ok = issue_qk(1);
    for (int j = 0; ok && j < it.ntiles; ++j) {
      if (__any_sync(0xffffffffu, stop_requested(failed))) break;
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!warp_wait(&bars[B_VFULL + st], ph, a.err, failed)) break;
      // V rows at positions >= seq_len (stale slots of the last block) -> 0
      const int t0 = it.kbase + j * BN;
      const int z0 = it.L - t0;
      const int z1 = min(BN, it.nblk * kBlockSize - t0);
      if (z0 > 0 && z0 < z1) {
        uint8_t* vst = sV + st * S::kKVBytes;
        const int nrows = z1 - z0;
        for (int idx = lane; idx < nrows * DC * 8; idx += 32) {
          const int r = z0 + idx / (DC * 8);
          const int c = (idx / 8) % DC;
          const int q = idx % 8;
          *reinterpret_cast<uint4*>(vst + (r / kBlockSize) * S::kVBlock + c * (kBlockSize * 128) +
                                    (r % kBlockSize) * 128 + q * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (!warp_wait(&bars[B_PRDY + st], ph, a.err, failed)) break;
      tc_fence_after();
      if (lane == 0) {
        // A = P_j from TMEM (8 columns per 16 keys), B = V_j from the ring
        const uint32_t vst = aV + st * S::kKVBytes;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          // block k of the stage: 64-column chunks 16 x 128 B apart
          const uint64_t db = smem_desc_sw128(vst + k * S::kVBlock, kBlockSize * 128, 1024);
          umma_bf16_ts(tmem + S::kTmemO, tmem + S::kTmemP + st * (BN / 2) + k * 8, db, idesc_pv,
                       (j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&bars[B_PV + st]);
      }
      __syncwarp();
      committed_pv = j + 1;
      if (j + 2 < it.ntiles) ok = issue_qk(j + 2);
    }
    // the last P V must finish before TMEM is freed
    if (committed_pv > 0)
      mbar_wait(&bars[B_PV + ((committed_pv - 1) & 1)], ((committed_pv - 1) >> 1) & 1, a.err);
  } else {
    // ============================== softmax ==============================
    const int r = threadIdx.x;  // row of the tile, TMEM lane
    const int tok = r / G;
    const int g = r % G;
    const int qi = it.it0 + tok;
    const bool row_valid = qi <= it.it1;
    const int p = it.L - it.n + qi;
    const int kmin = (a.window > 0) ? p - a.window + 1 : -0x40000000;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const bool capped = a.softcap > 0.f;
    const float sl2 = a.scale * kLog2e;
    // The uncapped path masks the raw q.k and scales the row maximum, which is
    // the maximum of the scaled logits only for scale > 0.  For scale <= 0
    // (uniform over the launch) the logits are scaled before the mask, as the
    // capped path does.
    const bool prescale = capped || !(sl2 > 0.f);
    const float cap_in = capped ? a.scale / a.softcap : 0.f;
    const float cap_out = a.softcap * kLog2e;
    // The three-term form of cap_out * tanh(cap_in * s) written in s:
    // x(s) = s (k1 + s^2 (k3 + k5 s^2)), k1 = cap_in cap_out,
    // k3 = -cap_in^3 cap_out / 3, k5 = 2 cap_in^5 cap_out / 15.  For
    // cap_in > 0 it increases with s, so the row maximum of x is x(max s),
    // and a masked column (s = -inf) gives x = -inf, as long as k5 > 0
    // (no 0 * inf).
    const float k1 = cap_in * cap_out;
    const float k3 = -cap_in * cap_in * k1 * (1.f / 3.f);
    const float k5 = 2.f * cap_in * cap_in * cap_in * cap_in * k1 * (1.f / 15.f);
    const bool fold_ok = capped && cap_in > 0.f && k5 > 0.f;
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < it.ntiles; ++j) {
      if (__any_sync(0xffffffffu, stop_requested(failed))) {
        ok = false;
        break;
      }
      const int st = j & 1;
      const uint32_t ph = (j >> 1) & 1;
      if (!warp_wait(&bars[B_QK + st], ph, a.err, failed)) {
        ok = false;
        break;
      }
      if (j == 0 && threadIdx.x == 0) PKA_PF_SET(rank, 1);
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {  // 64 columns per load and wait
        float t[64];
        tmem_ld64(lane_base + st * BN + c * 64, t);
#pragma unroll
        for (int e = 0; e < 64; ++e) s[c * 64 + e] = t[e];
      }
      const int t0 = it.kbase + j * BN;
      const int c_hi = row_valid ? min(BN - 1, p - t0) : -1;
      const int c_lo = max(0, kmin - t0);
      // Only rows on a causal diagonal or a window edge need the per-column
      // mask; the warp takes the masked loop only if one of its rows does.
      const bool need_mask = __any_sync(0xffffffffu, c_lo > 0 || c_hi < BN - 1);
      bool folded = false;
      // Row maximum in column pairs (three-input max); the capped path takes
      // the minimum too, for the range of |s| that picks its form.  On a
      // tile with no masked column the raw maximum is the one the folded
      // form needs.
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      bool have_max = false;
      if (capped) {
        float n4[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          m4[c & 3] = max3f(m4[c & 3], s[2 * c], s[2 * c + 1]);
          n4[c & 3] = min3f(n4[c & 3], s[2 * c], s[2 * c + 1]);
        }
        const float amax = fmaxf(fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])),
                                 -fminf(fminf(n4[0], n4[1]), fminf(n4[2], n4[3])));
        // log2-domain logits cap * tanh(s * scale / cap) * log2(e); a
        // Taylor form when every |y| of the warp's rows is below 1/8 (three
        // terms) or 0.5 (six terms), else the exp2 form.  With scale > 0 the
        // three-term form stays folded (see k1, k3, k5) and s stays raw.
        if (fold_ok && __all_sync(0xffffffffu, amax * cap_in < 0.125f)) {
          folded = true;
          have_max = !need_mask;
        } else if (__all_sync(0xffffffffu, amax * cap_in < 0.125f)) {
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = cap_out * tanh_taylor_short(s[c] * cap_in);
        } else if (__all_sync(0xffffffffu, amax * cap_in < 0.5f)) {
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = cap_out * tanh_taylor(s[c] * cap_in);
        } else {
#pragma unroll
          for (int c = 0; c < BN; ++c) s[c] = cap_out * tanh_via_exp2(s[c] * cap_in);
        }
      } else if (prescale) {
#pragma unroll
        for (int c = 0; c < BN; c += 2) {
          const float2 v = mul2(make_float2(s[c], s[c + 1]), make_float2(sl2, sl2));
          s[c] = v.x;
          s[c + 1] = v.y;
        }
      }
      // (otherwise s stays raw; scale > 0, so the raw max scales to the max)
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (!(c >= c_lo && c <= c_hi)) s[c] = -INFINITY;
      }
      if (!have_max) {
#pragma unroll
        for (int e = 0; e < 4; ++e) m4[e] = -INFINITY;
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) m4[c & 3] = max3f(m4[c & 3], s[2 * c], s[2 * c + 1]);
      }
      float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      if (folded)
        mx = mx * fmaf(mx * mx, fmaf(mx * mx, k5, k3), k1);  // x(max s) = max x(s)
      else if (!prescale)
        mx *= sl2;
      const float m_new = fmaxf(m_ref, mx);
      const bool resc = (j > 0) && (m_new > m_ref + 8.f);
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled
        if (!warp_wait(&bars[B_PV + ((j - 1) & 1)], ((j - 1) >> 1) & 1, a.err, failed)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float f = resc ? fast_exp2(m_ref - m_new) : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(lane_base + S::kTmemO + c * 32, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= f;
          tmem_st32(lane_base + S::kTmemO + c * 32, o);
        }
      }
      if (resc) l *= fast_exp2(m_ref - m_new);
      if (j == 0 || resc) m_ref = m_new;
      const float ms = (m_ref == -INFINITY) ? 0.f : m_ref;
      // P_j (bf16 pairs) into P buffer j % 2.  Its last reader, P_{j-2}
      // V_{j-2}, was issued before S_j, whose completion this thread has
      // waited for (a commit covers every earlier MMA of the issuer).
      // p = 2^(x - ms), x the log2-domain logit (uncapped: x = s * scale * log2 e,
      // fused into one FMA)
      const float xs = prescale ? 1.f : sl2;
      // x - ms for each column: the folded capped form, or the (scaled)
      // logit; the two loops are compiled separately so that neither pays
      // for the other's arithmetic
      auto make_p = [&](auto arg2) {
        float2 lsum0 = make_float2(0.f, 0.f), lsum1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int h = 0; h < BN / 64; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 x = arg2(make_float2(s[h * 64 + 2 * e], s[h * 64 + 2 * e + 1]));
            const float2 pp = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            if (e & 1)
              lsum1 = add2(lsum1, pp);
            else
              lsum0 = add2(lsum0, pp);
            pk[e] = pack_bf16x2(pp.x, pp.y);
          }
          tmem_st32_u(lane_base + S::kTmemP + st * (BN / 2) + h * 32, pk);
        }
        const float2 ls = add2(lsum0, lsum1);
        return ls.x + ls.y;
      };
      const float2 nms = make_float2(-ms, -ms);
      const float lsum =
          folded ? make_p([&](float2 x) {
                     const float2 t = mul2(x, x);
                     const float2 u = fma2(t, fma2(t, make_float2(k5, k5), make_float2(k3, k3)),
                                           make_float2(k1, k1));
                     return fma2(x, u, nms);
                   })
                 : make_p([&](float2 x) { return fma2(x, make_float2(xs, xs), nms); });
      l += lsum;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[B_PRDY + st]);
    }
    // ------------------------------------------------------------ epilogue
    if (ok) {
      const int jl = it.ntiles - 1;
      ok = warp_wait(&bars[B_PV + (jl & 1)], (jl >> 1) & 1, a.err, failed);
    }
    if (ok && threadIdx.x == 0) PKA_PF_SET(rank, 2);
    const bool full = (it.it1 - it.it0 + 1 == TQ);  // uniform over the CTA
    // A piece of an item split along keys leaves its softmax-normalised rows
    // (fp32) and their log2-domain LSEs in its workspace slot; the piece that
    // arrives last on the item's counter merges every piece's slot, in piece
    // order (the same bits whichever piece merges), and writes the output.
    const bool split_item = kSplit && un.npieces > 1;  // uniform over the CTA
    bool write_out = true;
    if (split_item) {
      const int slot = un.slot0 + un.piece;
      if (ok) {
        tc_fence_after();
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        // [slot][D / 4][128 rows] float4: the 128 rows of a column group are
        // consecutive, so each store instruction of a warp is coalesced
        float4* po = reinterpret_cast<float4*>(a.split_o) + static_cast<size_t>(slot) * (D / 4) * 128 + r;
#pragma unroll 1
        for (int c = 0; c < D / 64; ++c) {
          float o[64];
          tmem_ld64(lane_base + S::kTmemO + c * 64, o);
#pragma unroll
          for (int e = 0; e < 16; ++e)
            po[(c * 16 + e) * 128] = make_float4(o[4 * e] * inv, o[4 * e + 1] * inv,
                                                 o[4 * e + 2] * inv, o[4 * e + 3] * inv);
        }
        a.split_lse[static_cast<size_t>(slot) * 128 + r] =
            (l > 0.f) ? m_ref + log2f(l) : -INFINITY;
      }
      volatile int* last = reinterpret_cast<volatile int*>(smem + S::oMisc + 8);
      asm volatile("bar.sync %0, %1;" ::"r"(kBarSoftmax), "r"(128) : "memory");
      if (threadIdx.x == 0) {
        fence_acq_rel_gpu();  // the CTA's rows (ordered by the barrier) before its arrival
        const int old = atomicAdd(a.split_cnt + un.slot0, 1);
        *last = (old == un.npieces - 1) ? 1 : 0;
        if (old == un.npieces - 1) a.split_cnt[un.slot0] = 0;  // for the next call
      }
      asm volatile("bar.sync %0, %1;" ::"r"(kBarSoftmax), "r"(128) : "memory");
      write_out = (*last != 0);
      if (write_out) fence_acq_rel_gpu();  // every piece's rows are visible now
    }
    if (write_out && ok) {
      tc_fence_after();
      float inv = (l > 0.f) ? 1.f / l : 0.f;
      // split item: the pieces' weights 2^(LSE_k - max LSE)
      float w[kMaxPieces];
      const float4* pk = split_item ? reinterpret_cast<const float4*>(a.split_o) +
                                          static_cast<size_t>(un.slot0) * (D / 4) * 128 + r
                                    : nullptr;
      if (split_item) {
        float lk[kMaxPieces];
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxPieces; ++k) {
          lk[k] = (k < un.npieces) ? __ldcg(a.split_lse + static_cast<size_t>(un.slot0 + k) * 128 + r)
                                   : -INFINITY;
          M = fmaxf(M, lk[k]);
        }
        float den = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxPieces; ++k) {
          w[k] = (M == -INFINITY) ? 0.f : fast_exp2(lk[k] - M);
          den += w[k];
        }
        inv = (den > 0.f) ? 1.f / den : 0.f;
      }
      // w[k] for a k known only at run time, by selects (w stays in registers)
      auto w_of = [&](int k) {
        float x = w[0];
#pragma unroll
        for (int kk = 1; kk < kMaxPieces; ++kk)
          if (k == kk) x = w[kk];
        return x;
      };
      // A tile of TQ tokens of this request leaves through TMA stores from
      // the Q tile's shared memory, which is free once the last MMA has
      // completed (the last P V commit covers every earlier MMA): each row
      // goes there in the 128-byte-swizzled layout the Q copies used, so the
      // output tensor map, of the same geometry, writes back whole 2 KB runs
      // (one token's G heads) instead of one 16-byte piece per row and
      // store.  A tile at the end of the request's rows, whose box would
      // cover the next request's rows, stores its valid rows one by one.
      uint16_t* orow = a.out + (static_cast<size_t>(it.q0 + qi) * a.Hq + it.kvh * G + g) * D;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {  // 64 columns per load and wait
        float o[64];
        if (split_item) {
          // piece by piece (the same order of terms for every element), the
          // 16 loads of a piece's 64 columns issued together
#pragma unroll
          for (int e = 0; e < 64; ++e) o[e] = 0.f;
#pragma unroll 1
          for (int k = 0; k < un.npieces; ++k) {
            const float4* src = pk + (static_cast<size_t>(k) * (D / 4) + c * 16) * 128;
            float4 v[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = __ldcg(src + e * 128);
            const float wk = w_of(k);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              o[4 * e] = fmaf(wk, v[e].x, o[4 * e]);
              o[4 * e + 1] = fmaf(wk, v[e].y, o[4 * e + 1]);
              o[4 * e + 2] = fmaf(wk, v[e].z, o[4 * e + 2]);
              o[4 * e + 3] = fmaf(wk, v[e].w, o[4 * e + 3]);
            }
          }
        } else {
          tmem_ld64(lane_base + S::kTmemO + c * 64, o);
        }
        uint8_t* srow = sQ + c * S::kQChunk + r * 128;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4 w = make_uint4(pack_bf16x2(o[q * 8 + 0] * inv, o[q * 8 + 1] * inv),
                                     pack_bf16x2(o[q * 8 + 2] * inv, o[q * 8 + 3] * inv),
                                     pack_bf16x2(o[q * 8 + 4] * inv, o[q * 8 + 5] * inv),
                                     pack_bf16x2(o[q * 8 + 6] * inv, o[q * 8 + 7] * inv));
          if (full)
            *reinterpret_cast<uint4*>(srow + ((q ^ (r & 7)) << 4)) = w;
          else if (row_valid)
            *reinterpret_cast<uint4*>(orow + c * 64 + q * 8) = w;
        }
      }
    }
    if (full && write_out) {
      // every softmax warp arrives, whatever its waits gave; the tile is
      // stored only if no wait of the CTA ran out
      fence_proxy_async_smem();
      asm volatile("bar.sync %0, %1;" ::"r"(kBarSoftmax), "r"(128) : "memory");
      if (threadIdx.x == 0 && !stop_requested(failed)) {
#pragma unroll
        for (int c = 0; c < DC; ++c)
          tma_store_3d(tm_out, sQ + c * S::kQChunk, c * 64, it.kvh * G, it.q0 + it.it0);
        bulk_commit();
        bulk_wait_read_all();  // the shared memory may go once the stores have read it
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, S::kTmemCols);
  if (threadIdx.x == 0) PKA_PF_SET(rank, 3);
}

}  // namespace pka
