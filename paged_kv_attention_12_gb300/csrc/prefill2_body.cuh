// Chunked prefill at D = 256 on CTA pairs (sm_103a): the tcgen05 MMAs of
// two SMs work as one, M = 256 rows over the pair.
//
// The same method as prefill_body.cuh ("Triton paged decode and prefill
// kernels reading K/V through block tables", inference-server README,
// engine feature list; causal attention over the cached prefix and the
// chunk), with the work item doubled: a cluster of two CTAs takes two
// consecutive query tiles of one (request, KV head) -- the rank-0 CTA the
// first 128 rows, the rank-1 CTA the next 128 -- and streams the keys both
// tiles see.  Every MMA is issued once, by the rank-0 CTA, for both
// (tcgen05.mma.cta_group::2), the S MMAs by one warp and the P V MMAs by
// another:
//
//  * S = Q K^T with M = 256 (each CTA's Q tile is its half of A) and the key
//    tile's 128 keys split between the CTAs' shared memory (N = 128: each
//    CTA holds 64 keys of every K stage);
//  * O += P V with P from each CTA's own TMEM and V split by columns (each
//    CTA holds 128 of the 256 columns of every V stage).
//
// So each SM receives and reads half of every K/V tile instead of all of
// it: at D = 256 a single SM's shared memory (a 64 KB Q tile plus the K/V
// rings) and its bandwidth set the pace of the one-CTA kernel, and the pair
// halves the ring bytes per key and doubles the stages that fit.  TMEM
// holds each CTA's own rows: one S buffer of 128 columns, two P buffers of
// 64 (bf16 pairs) and O (256).
//
// Cross-CTA signalling: both CTAs' TMA copies complete on the rank-0 CTA's
// "full" barriers (cp.async.bulk.tensor ... .cta_group::2), the MMA commits
// arrive on the barriers of both CTAs (multicast), and each CTA's softmax
// reports its P with one remote arrive on the rank-0 CTA's barrier.  All
// mbarrier waits are bounded; the TMEM allocation is a collective of the
// pair, which both CTAs reach unconditionally, and the pair meets at a
// cluster barrier before it frees TMEM and exits.
#pragma once

#include "prefill_body.cuh"

namespace pka {

template <int G>
struct Prefill2Shape {
  static constexpr int D = 256;
  static constexpr int BM = 128;                    // rows per CTA (256 per pair)
  static constexpr int TQ = BM / G;                 // query tokens per CTA tile
  static constexpr int BN = 128;                    // keys per key tile (pair)
  static constexpr int DC = D / 64;                 // 128-byte chunks of a row
  static constexpr int kHalfKeys = BN / 2;          // keys of a K stage per CTA
  static constexpr int kQChunk = BM * 128;
  static constexpr int kKChunk = kHalfKeys * 128;   // K stage: [DC][64 keys][128 B]
  static constexpr int kKStage = kHalfKeys * D * 2; // 32 KB
  static constexpr int kVBlock = kBlockSize * (DC / 2) * 128;  // [2 chunks][16 rows][128 B]
  static constexpr int kVStage = BN * (D / 2) * 2;  // 32 KB: 128 keys x 128 columns
  static constexpr int kQBytes = BM * D * 2;
  static constexpr int KST = 3;                     // K ring stages
  static constexpr int VST = 2;                     // V ring stages
  static constexpr int oQ = 0;
  static constexpr int oK = oQ + kQBytes;
  static constexpr int oV = oK + KST * kKStage;
  static constexpr int oBar = oV + VST * kVStage;
  // Q, K full/empty per stage, V full/empty per stage, S ready x2, P ready
  // x2, S read
  static constexpr int kNumBars = 1 + 2 * KST + 2 * VST + 2 + 2 + 1;
  static constexpr int oMisc = oBar + kNumBars * 8;
  static constexpr int kSmemBytes = oMisc + 16 + 1024;
  static constexpr uint32_t kTmemO = 256;
  // One S buffer (BN columns at 0), P_j (bf16 pairs, BN / 2 columns) in
  // buffer j % 2 at kTmemP, O at kTmemO: 128 + 2 x 64 + 256 = 512 columns.
  // S_{j+1} may be written as soon as every softmax warp has read S_j into
  // its registers, and P_{j+2} once P_j V_j has completed.
  static constexpr uint32_t kTmemP = BN;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr int kThreads = 8 * 32;
  static constexpr int kCostBuckets = 4096;
  static_assert((kCostBuckets + 64) * 4 <= KST * kKStage, "ranking scratch");
  static_assert((kReqCacheOffset + 2 * kReqCache) * 4 <= KST * kKStage, "request cache");
  static_assert(kListOffset >= kReqCacheOffset + 2 * kReqCache &&
                    (kListOffset + 5 * kMaxList + 4) * 4 <= KST * kKStage,
                "the pair list fits in the K stages, past the request cache");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(KST == 3 && VST == 2, "the barrier map below assumes 3 K and 2 V stages");
  static_assert(kTmemP + BN <= kTmemO && kTmemO + D <= kTmemCols, "TMEM columns");
};

namespace pair2 {

// Warp roles of a pair CTA: softmax 0-3, K copies kWarpTmaK, V copies
// kWarpTmaV, S MMAs kWarpMma (rank-0 CTA), P V MMAs kWarpPv (rank-0 CTA;
// the one-CTA kernel's second K warp).
constexpr int kWarpPv = kWarpTmaK2;

enum {
  PB_Q = 0,
  PB_KFULL = 1,                          // [KST], completed on the rank-0 CTA
  PB_KEMPTY = PB_KFULL + 3,               // [KST], both CTAs (multicast commit)
  PB_VFULL = PB_KEMPTY + 3,               // [VST], completed on the rank-0 CTA
  PB_VEMPTY = PB_VFULL + 2,               // [VST], both CTAs (multicast commit)
  PB_QK = PB_VEMPTY + 2,                  // [2] S_j ready, both CTAs
  PB_PRDY = PB_QK + 2,                    // [2] P_j ready, rank-0 CTA, 8 arrivals
  PB_SREAD = PB_PRDY + 2,                 // S_j read by every softmax warp, rank-0 CTA, 8 arrivals
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The shared::cluster address of this CTA's variable in the rank-0 CTA.
__device__ __forceinline__ uint32_t leader_addr(const void* p) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(a) : "r"(smem_u32(p)));
  return a;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}

// TMA copies into this CTA's shared memory completing on a barrier of the
// rank-0 CTA (a shared::cluster address).
__device__ __forceinline__ void tma2_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                             uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void tma2_load_3d(void* dst, const CUtensorMap* map, int x, int y,
                                             int z, uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar_cluster)
      : "memory");
}

__device__ __forceinline__ void umma2(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                      uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the barrier at this offset in both CTAs once every MMA issued
// so far by this thread has completed.
__device__ __forceinline__ void commit2_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// One arrival on a barrier of a CTA of the cluster (a shared::cluster
// address), with the default semantics of a remote arrive (release at CTA
// scope).  What it publishes is TMEM content the thread wrote with
// tcgen05.st, complete after tcgen05.wait::st and ordered before the arrive
// by tcgen05.fence::before_thread_sync; the waiting MMA thread orders its
// MMAs after the wait with tcgen05.fence::after_thread_sync.  A release at
// cluster scope would also order the thread's generic memory accesses for
// the other CTA, which the P V MMA does not read, and lengthens the path
// from P_j to P_j V_j (measured: 181 us for the chunked prefill workload
// against 201 us, with the same bits).  Every wait of the kernel, on the
// P-ready and Q barriers as well, acquires at CTA scope (the default of
// mbarrier.try_wait): what the barriers order is TMEM and TMA-written shared
// memory, ordered by the tcgen05 fences and the async proxy.
__device__ __forceinline__ void remote_arrive(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ void tmem2_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem2_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

}  // namespace pair2

// One pair item per cluster of two CTAs on the S::kSmemBytes of shared
// memory at smem_raw: the cluster of index (blockIdx.x - rank_base) / 2
// (rank_base even: the CTAs before it do other work) takes the pair item of
// that rank (heaviest first over (request, two query tiles) pairs),
// KV head rank % Hkv; ranks past the last item return at once (both CTAs of
// a cluster decide alike: everything up to the TMEM allocation depends on
// the arguments and the cluster's index only).  kSplit (the mixed launch,
// with its workspace): when every item fits the a.one_wave / 2 pair slots,
// rank r takes unit r in index order instead, and with room to spare the
// items are cut along keys into pieces merged through the workspace (two
// slots per piece, one per CTA; see one_wave_unit in prefill_body.cuh).
template <int G, bool kSplit>
__device__ __forceinline__ void prefill2_body(const PrefillArgs& a, const CUtensorMap* tm_q,
                                              const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                              const CUtensorMap* tm_out, uint8_t* smem_raw,
                                              int rank_base) {
  using S = Prefill2Shape<G>;
  using namespace pair2;
  constexpr int D = S::D, BN = S::BN, TQ = S::TQ, DC = S::DC;
  constexpr int TQ2 = 2 * TQ;  // query tokens of a pair item
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int crank = static_cast<int>(cluster_rank());
  const int rank = (static_cast<int>(blockIdx.x) - rank_base) / 2;  // the cluster's pair rank

  // ---------------------------------------------------------- work item
  Item it;
  const int qtiles = (a.max_query_len + TQ2 - 1) / TQ2;
  int* scratch = reinterpret_cast<int*>(smem + S::oK);
  const bool cache = a.batch <= kReqCache;
  int* rn = cache ? scratch + kReqCacheOffset : nullptr;
  int* rL = cache ? rn + kReqCache : nullptr;
  int pairs_with_work = 0;
  {
    int cnt = 0;
    for (int b = threadIdx.x; b < a.batch; b += blockDim.x) {
      int q0;
      const int n = query_span(a, b, &q0);
      if (n < 0 && rank == 0 && crank == 0) report(a.err, PKA_DEVERR_QUERY_LOC);
      const int L = min(a.seq_lens[b], a.max_blocks * kBlockSize);
      if (cache) {
        rn[b] = n;
        rL[b] = L;
      }
      if (a.window <= 0 && n > 0) {
        // without a window every item of the request starts at its first
        // block: bring the first 64 table entries into L2 while the items
        // are ranked (the K warp reads them right after)
        const int32_t* row = a.tables + static_cast<size_t>(b) * a.max_blocks;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row));
        if (a.max_blocks > 32) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + 32));
      }
      if (n > 0 && n <= L && !(a.skip_decode_rows != 0 && n == 1)) cnt += (n + TQ2 - 1) / TQ2;
    }
    block_excl_scan(cnt, scratch, scratch + 32);
    pairs_with_work = scratch[32];
    __syncthreads();
  }
  // With the split workspace (the mixed launch) and every pair item in one
  // wave of the pair slots (a.one_wave SMs, two per slot), the items go in
  // index order and are cut along keys into pieces that fill the wave, as
  // in the one-CTA body: counted in pair slots, each piece takes two
  // workspace slots, one per CTA of the pair (its 128 rows).  Otherwise the
  // items are ranked heaviest first and run whole.
  Unit un{0, 0, 0, 0, 1, 0};
  int qt2;
  const long long items = static_cast<long long>(pairs_with_work) * a.Hkv;
  if (kSplit && items <= a.one_wave / 2 && pairs_with_work <= kMaxList) {
    PrefillArgs ap = a;
    ap.one_wave = a.one_wave / 2;
    ap.split_slots = a.split_slots / 2;
    const bool split = a.split_o != nullptr && items < ap.one_wave && items <= ap.split_slots;
    if (!one_wave_unit<TQ2, BN>(ap, rank, pairs_with_work, split, scratch, rn, rL, &un)) return;
    it.b = un.b;
    it.kvh = un.kvh;
    qt2 = un.qt;
  } else {
    if (rank / a.Hkv >= pairs_with_work) return;  // uniform over the cluster
    const int nbuck = min(S::kCostBuckets, (a.max_seq_len + BN - 1) / BN + 2);
    const int pair = lpt_pair<TQ2, BN>(a, qtiles, rank / a.Hkv, scratch, nbuck, rn, rL);
    it.b = pair / qtiles;
    it.kvh = rank % a.Hkv;
    qt2 = pair % qtiles;
  }
  it.n = query_span(a, it.b, &it.q0);
  if (it.n < 0) return;  // uniform (reported by the first pass)
  it.L = a.seq_lens[it.b];
  if (it.L > a.max_blocks * kBlockSize) {
    if (threadIdx.x == 0 && crank == 0 && qt2 == 0 && it.kvh == 0) report(a.err, PKA_DEVERR_SEQ_LEN);
    it.L = a.max_blocks * kBlockSize;
  }
  if (it.n > it.L) {
    if (threadIdx.x == 0 && crank == 0 && qt2 == 0 && it.kvh == 0) report(a.err, PKA_DEVERR_SEQ_LEN);
    return;
  }
  it.it0 = qt2 * TQ2;
  if (it.n <= 0 || it.it0 >= it.n || (a.skip_decode_rows != 0 && it.n == 1)) return;
  it.it1 = min(it.n, it.it0 + TQ2) - 1;  // the pair's last query row
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
  const int my0 = it.it0 + crank * TQ;  // this CTA's first query row

  uint8_t* sQ = smem + S::oQ;
  uint8_t* sK = smem + S::oK;
  uint8_t* sV = smem + S::oV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::oBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::oMisc);
  volatile int* failed = reinterpret_cast<volatile int*>(smem + S::oMisc + 4);
  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const bool lead = (crank == 0);
  const int stamp = static_cast<int>(blockIdx.x);  // instrumented builds: one row per CTA
  if (threadIdx.x == 0) {
    PKA_PF_SET(stamp, 0);
    PKA_PF_VAL(stamp, 4, static_cast<unsigned long long>(it.ntiles));
  }

  if (threadIdx.x == 0) {
    mbar_init(&bars[PB_Q], 1);
    for (int i = 0; i < S::KST; ++i) {
      mbar_init(&bars[PB_KFULL + i], 1);
      mbar_init(&bars[PB_KEMPTY + i], 1);
    }
    for (int i = 0; i < S::VST; ++i) {
      mbar_init(&bars[PB_VFULL + i], 1);
      mbar_init(&bars[PB_VEMPTY + i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[PB_QK + i], 1);
      mbar_init(&bars[PB_PRDY + i], 8);  // each softmax warp of both CTAs
    }
    mbar_init(&bars[PB_SREAD], 8);
    *failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kWarpMma) tmem2_alloc(tmem_slot, S::kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any signal crosses
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t oob_row = static_cast<uint32_t>(a.num_blocks) * a.Hkv * kBlockSize;
  const int32_t* trow = a.tables + static_cast<size_t>(it.b) * a.max_blocks;

  if (warp == kWarpTmaK || warp == kWarpTmaV) {
    // ============================ TMA producers ============================
    // Each CTA loads its half of every stage -- K: 64 of the tile's 128 keys
    // (blocks 4 crank .. 4 crank + 3, one 2-D box per block and 64-column
    // chunk, one lane each), V: 128 of the 256 columns of all 128 keys (one
    // 3-D box of two chunks per block) -- completing on the rank-0 CTA's
    // "full" barrier, which expects both halves.  A stage is refilled once
    // the MMA that read it has committed (the commit reaches both CTAs).
    const bool is_k = (warp != kWarpTmaV);
    const int nst = is_k ? S::KST : S::VST;
    uint8_t* ring = is_k ? sK : sV;
    const int full_base = is_k ? PB_KFULL : PB_VFULL;
    const int empty_base = is_k ? PB_KEMPTY : PB_VEMPTY;
    const uint32_t stage_bytes = is_k ? S::kKStage : S::kVStage;
    int issued = 0;
    if (lane == 0) {
      prefetch_tensormap(is_k ? tm_k : tm_v);
      if (warp == kWarpTmaK) {
        prefetch_tensormap(tm_q);
        if (lead) mbar_arrive_expect_tx(&bars[PB_Q], 2 * S::kQBytes);
        const uint32_t qbar = leader_addr(&bars[PB_Q]);
#pragma unroll
        for (int c = 0; c < DC; ++c)
          tma2_load_3d(sQ + c * S::kQChunk, tm_q, c * 64, it.kvh * G, it.q0 + my0, qbar);
      }
    }
    // V is first read by P_0 V_0, a softmax after S_0: the V warp issues
    // its first stages once S_0 is done, so that Q and the first K stages,
    // which S_0 and S_1 need, do not share the memory system with them
    // (a failed wait sets the flag that ends the loop below).
    if (!is_k) warp_wait(&bars[PB_QK], 0, a.err, failed);
    // Pool rows of the item's blocks, 32 per coalesced load, in a window
    // of 64 blocks held one per lane in two registers (see prefill_body).
    constexpr int BPT = BN / kBlockSize;  // 8 blocks per key tile
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
    int win = 0;
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
        if (j >= nst &&
            !mbar_wait(&bars[empty_base + st], static_cast<uint32_t>((j / nst - 1) & 1), a.err)) {
          *failed = 1;
          good = 0;
        }
        if (good && lead) mbar_arrive_expect_tx(&bars[full_base + st], 2 * stage_bytes);
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) break;
      const uint32_t fbar = leader_addr(&bars[full_base + st]);
      uint8_t* dst = ring + st * stage_bytes;
      if (is_k) {
        if (lane < (BPT / 2) * DC) {
          // this CTA's keys: blocks 4 crank .. 4 crank + 3 of the tile, one
          // box per (block, 64-column chunk)
          const int kb = lane / DC, c = lane % DC;
          uint32_t r = rl[0];
#pragma unroll
          for (int q = 1; q < BPT; ++q)
            if ((BPT / 2) * crank + kb == q) r = rl[q];
          tma2_load_2d(dst + c * S::kKChunk + kb * kBlockSize * 128, tm_k, c * 64,
                       static_cast<int>(r), fbar);
        }
      } else if (lane < BPT) {
        uint32_t r = rl[0];
#pragma unroll
        for (int q = 1; q < BPT; ++q)
          if (lane == q) r = rl[q];
        tma2_load_3d(dst + lane * S::kVBlock, tm_v, 0, static_cast<int>(r), (DC / 2) * crank, fbar);
      }
      issued = j + 1;
    }
    if (lane == 0 && lead) {
      // every issued stage (both CTAs' halves) must land before the pair
      // may finish
      for (int j = issued - nst < 0 ? 0 : issued - nst; j < issued; ++j)
        mbar_wait(&bars[full_base + j % nst], (j / nst) & 1, a.err);
      if (warp == kWarpTmaK && stop_requested(failed)) mbar_wait(&bars[PB_Q], 0, a.err);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ============================== S MMAs ==============================
    // Issued by the rank-0 CTA only, for both (M = 256).  S has one TMEM
    // buffer: S_{j+1} waits until every softmax warp of both CTAs has read
    // S_j into registers.  Issuing a tile's 16 MMAs holds the issuing thread until the tensor
    // pipe has nearly run them, so the P V MMAs come from another warp
    // (below): P_j V_j goes to the pipe as soon as P_j is ready, even while
    // this warp is still issuing S_{j+1} (the two touch different TMEM
    // columns, so their MMAs may interleave).
    if (lead) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(256, BN, 0, 0);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK);
      bool ok = warp_wait(&bars[PB_Q], 0, a.err, failed);
      auto issue_qk = [&](int j) -> bool {
        const int st = j & 1;
        const int ks = j % S::KST;
        if (!warp_wait(&bars[PB_KFULL + ks], (j / S::KST) & 1, a.err, failed)) return false;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kst = aK + ks * S::kKStage;
#pragma unroll
          for (int c = 0; c < DC; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t da = smem_desc_sw128(aQ + c * S::kQChunk + kk * 32, 16, 1024);
              const uint64_t db = smem_desc_sw128(kst + c * S::kKChunk + kk * 32, 16, 1024);
              umma2(tmem, da, db, idesc_qk, (c | kk) != 0);
            }
          commit2_both(&bars[PB_QK + st]);
          commit2_both(&bars[PB_KEMPTY + ks]);
        }
        __syncwarp();
        return true;
      };
      if (ok) ok = issue_qk(0);
      for (int j = 0; ok && j + 1 < it.ntiles; ++j) {
        if (__any_sync(0xffffffffu, stop_requested(failed))) break;
        // S_{j+1} overwrites S_j: once all eight softmax warps have read it
        ok = warp_wait(&bars[PB_SREAD], j & 1, a.err, failed);
        if (ok) ok = issue_qk(j + 1);
      }
    }
  } else if (warp == kWarpPv) {
    // ============================= P V MMAs =============================
    // Rank-0 CTA only: P_j V_j as soon as P_j and V_j are there.
    if (lead) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(256, D, 0, 1);
      const uint32_t aV = smem_u32(sV);
      int committed_pv = 0;
      for (int j = 0; j < it.ntiles; ++j) {
        if (__any_sync(0xffffffffu, stop_requested(failed))) break;
        const int st = j & 1;
        const uint32_t ph = (j >> 1) & 1;
        const int vs = j % S::VST;
        if (!warp_wait(&bars[PB_VFULL + vs], (j / S::VST) & 1, a.err, failed)) break;
        // V rows at positions >= seq_len (stale slots of the last block,
        // which may hold NaN) -> 0 in both CTAs' halves, before P V reads
        // them (the peer's half through its cluster address)
        const int t0 = it.kbase + j * BN;
        const int z0 = it.L - t0;
        const int z1 = min(BN, it.nblk * kBlockSize - t0);
        if (z0 > 0 && z0 < z1) {
          uint8_t* vst = sV + vs * S::kVStage;
          const int per = (z1 - z0) * (DC / 2) * 8;  // 16-byte pieces per CTA
          for (int idx = lane; idx < 2 * per; idx += 32) {
            const int peer = idx / per;
            const int rem = idx % per;
            const int r = z0 + rem / ((DC / 2) * 8);
            const int c = (rem / 8) % (DC / 2);
            const int q = rem % 8;
            uint8_t* ptr = vst + (r / kBlockSize) * S::kVBlock + c * (kBlockSize * 128) +
                           (r % kBlockSize) * 128 + q * 16;
            if (peer == 0) {
              *reinterpret_cast<uint4*>(ptr) = make_uint4(0u, 0u, 0u, 0u);
            } else {
              uint32_t ra;
              asm volatile("mapa.shared::cluster.u32 %0, %1, 1;" : "=r"(ra) : "r"(smem_u32(ptr)));
              asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(ra), "r"(0u)
                           : "memory");
            }
          }
          fence_proxy_async_smem();
          asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
        }
        __syncwarp();
        if (!warp_wait(&bars[PB_PRDY + st], ph, a.err, failed)) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t vst = aV + vs * S::kVStage;
#pragma unroll
          for (int k = 0; k < BN / 16; ++k) {
            // block k: two 64-column chunks 16 x 128 B apart
            const uint64_t db = smem_desc_sw128(vst + k * S::kVBlock, kBlockSize * 128, 1024);
            umma2_ts(tmem + S::kTmemO, tmem + S::kTmemP + st * (BN / 2) + k * 8, db, idesc_pv,
                     (j > 0 || k > 0) ? 1u : 0u);
          }
          commit2_both(&bars[PB_VEMPTY + vs]);
        }
        __syncwarp();
        committed_pv = j + 1;
      }
      // the last P V must finish before TMEM is freed
      if (committed_pv > 0) {
        const int jl = committed_pv - 1;
        mbar_wait(&bars[PB_VEMPTY + jl % S::VST], (jl / S::VST) & 1, a.err);
      }
    }
  } else {
    // ============================== softmax ==============================
    const int r = threadIdx.x;  // row of the tile, TMEM lane
    const int tok = r / G;
    const int g = r % G;
    const int qi = my0 + tok;
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
      if (!warp_wait(&bars[PB_QK + st], ph, a.err, failed)) {
        ok = false;
        break;
      }
      if (j == 0 && threadIdx.x == 0) PKA_PF_SET(stamp, 1);
      tc_fence_after();
      float s[BN];
#pragma unroll
      for (int c = 0; c < BN / 64; ++c) {  // 64 columns per load and wait
        float t[64];
        tmem_ld64(lane_base + c * 64, t);
#pragma unroll
        for (int e = 0; e < 64; ++e) s[c * 64 + e] = t[e];
      }
      // S_j is in registers: the S warp may overwrite the buffer with S_{j+1}
      tc_fence_before();
      __syncwarp();
      if (lane == 0) remote_arrive(leader_addr(&bars[PB_SREAD]));
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
        if (!warp_wait(&bars[PB_VEMPTY + (j - 1) % S::VST], ((j - 1) / S::VST) & 1, a.err,
                               failed)) {
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
      // P_j (bf16 pairs) into P buffer j % 2, whose last reader P_{j-2} V_{j-2}
      // must have completed.
      if (j >= 2 && !warp_wait(&bars[PB_VEMPTY + j % S::VST], ((j - 2) / S::VST) & 1, a.err,
                               failed)) {
        ok = false;
        break;
      }
      tc_fence_after();
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
      // one arrival per warp on the rank-0 CTA's barrier once its 32 rows
      // have written P_j (a warp that gave up does not arrive, and the MMA
      // warp's bounded wait ends the item)
      __syncwarp();
      if (lane == 0) remote_arrive(leader_addr(&bars[PB_PRDY + st]));
    }
    // ------------------------------------------------------------ epilogue
    if (ok) {
      const int jl = it.ntiles - 1;
      ok = warp_wait(&bars[PB_VEMPTY + jl % S::VST], (jl / S::VST) & 1, a.err, failed);
    }
    if (ok && threadIdx.x == 0) PKA_PF_SET(stamp, 2);
    const bool full = (my0 + TQ - 1 <= it.it1);  // uniform over the CTA
    // A piece of an item split along keys leaves its softmax-normalised rows
    // (fp32) and their log2-domain LSEs in its workspace slot; the piece that
    // arrives last on the item's counter merges every piece's slot, in piece
    // order (the same bits whichever piece merges), and writes the output.
    const bool split_item = kSplit && un.npieces > 1;  // uniform over the CTA
    // workspace slot of piece k for this CTA's rows; the arrival counter of
    // the item's rows on this CTA
    auto slot_of = [&](int k) { return 2 * (un.slot0 + k) + crank; };
    bool write_out = true;
    if (split_item) {
      const int slot = slot_of(un.piece);
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
        const int old = atomicAdd(a.split_cnt + slot_of(0), 1);
        *last = (old == un.npieces - 1) ? 1 : 0;
        if (old == un.npieces - 1) a.split_cnt[slot_of(0)] = 0;  // for the next call
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
      const float4* pk = split_item ? reinterpret_cast<const float4*>(a.split_o) + r : nullptr;
      if (split_item) {
        float lk[kMaxPieces];
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kMaxPieces; ++k) {
          lk[k] = (k < un.npieces) ? __ldcg(a.split_lse + static_cast<size_t>(slot_of(k)) * 128 + r)
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
            const float4* src = pk + (static_cast<size_t>(slot_of(k)) * (D / 4) + c * 16) * 128;
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
          tma_store_3d(tm_out, sQ + c * S::kQChunk, c * 64, it.kvh * G, it.q0 + my0);
        bulk_commit();
        bulk_wait_read_all();  // the shared memory may go once the stores have read it
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs or signals may touch it
  tc_fence_after();
  if (warp == kWarpMma) tmem2_dealloc(tmem, S::kTmemCols);
  if (threadIdx.x == 0) PKA_PF_SET(stamp, 3);

}

}  // namespace pka
