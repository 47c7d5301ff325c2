// Paged decode attention, direct and split-K (sm_103a: TMA tensor tiles,
// mbarrier ring, warp-level tensor-core MMA, shuffle online softmax).
//
// One query token per request attends over its visible keys, read block by
// block through the request's block table ("Triton paged decode ... kernels
// reading K/V through block tables; split-K decode variant", inference-server
// README, engine feature list).  Decode is bound by HBM: every K/V byte is
// read once, so the design is about keeping enough bytes in flight, spreading
// them evenly over the SMs, and keeping the per-byte arithmetic far below the
// copy time.
//
// Work.  A segment is one (request, KV head): its visible blocks, each a
// 16-key "tile".  The pipelines are persistent (two per SM).
//  * split-K: the segments, laid end to end as work units (a fixed cost per
//    piece, then one unit per tile), are cut into equal contiguous chunks of
//    q = max(min_chunk, ceil(total / pipelines)) units, one chunk per
//    pipeline.  Each piece of a segment inside a chunk gives one partial
//    (normalised output, LSE) in slot (chunk index - chunk index of the
//    segment's first tile); the pipeline holding a segment's first tile also
//    writes LSE = -inf into the slots the segment does not use, so the LSE
//    combine needs nothing but the partials.  With a workspace of arrival
//    counters, the pipeline whose arrival completes a segment merges its
//    partials in the same launch (fused combine).
//  * direct: pipeline c takes whole segments c, c + pipelines, ... and
//    writes bf16.
//
// Inside a pipeline (a CTA of its own, or half of a mixed-batch CTA):
//  * one producer warp walks the pieces' block tables (32 ids per coalesced
//    load) and loads, per tile, the (block, head) K and V tiles with one
//    3-D TMA copy each (D / 64 boxes of 16 rows x 64 columns, 128-byte
//    swizzle) into a ring of
//    shared-memory slots, completion counted on a "full" mbarrier;
//  * NW consumer warps take the ring's tiles round robin; every slot has one
//    owner warp, so each slot's mbarrier phases are consumed in order.  A
//    warp computes S^T = K q^T and O^T += V^T P^T with m16n8k16 MMAs (keys
//    or head-dim rows on M, the G <= 8 query heads of the KV group on N, so
//    every K/V byte feeds all G heads), operands by conflict-free ldmatrix
//    from the swizzled tiles; the online softmax runs in the exp2 domain on
//    the accumulator fragments with shuffles; P goes to the PV operand
//    layout through shuffles, in bf16;
//  * at the end of a piece warps 1..NW-1 leave their (max, sum, acc) states
//    in shared memory and go straight on with the next piece; warp 0 merges
//    them in registers and writes the piece's result (through shared memory,
//    as coalesced 16-byte stores), while the producer streams on.
//
// Tiles with keys outside [first visible, query position] (window start,
// ragged tail) are masked on the fragments; V rows past the sequence end
// (stale slots that may hold NaN) are zeroed in shared memory before P V.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pka {

// ----------------------------------------------------------- timeline
// Built with -DPKA_TIMELINE (a separate, instrumented build of the library;
// see timeline.py beside the package), every decode pipeline records global
// timer stamps of its phases: [layer slot: 0 = full attention, 1 = sliding
// window][pipeline][kTimelineFields].  The default build compiles none of it.
enum TimelineField {
  TL_ENTRY = 0,        // pipeline starts (consumer thread 0)
  TL_PARTITION = 1,    // producer: partition known (iterator ready)
  TL_FIRST_ISSUE = 2,  // producer: first tile's copies issued
  TL_FIRST_TILE = 3,   // consumer warp 0: first tile landed
  TL_LAST_ISSUE = 4,   // producer: last tile's copies issued
  TL_LAST_TILE = 5,    // consumer warps: last tile consumed (latest warp)
  TL_EXIT = 6,         // consumer warps: pipeline done (latest warp)
  TL_TILES = 7,        // tiles streamed (a count, not a time)
  kTimelineFields = 8
};
constexpr int kTimelinePipes = 1024;
#ifdef PKA_TIMELINE
__device__ unsigned long long pka_timeline[2 * kTimelinePipes * kTimelineFields];
__device__ __forceinline__ unsigned long long* timeline_row(const DecodeArgs& a, int vcta) {
  return pka_timeline + ((a.window > 0 ? 1 : 0) * kTimelinePipes + vcta) * kTimelineFields;
}
#define PKA_TL_SET(a, vcta, f) \
  do { if ((vcta) < kTimelinePipes) timeline_row(a, vcta)[f] = timeline_now(); } while (0)
#define PKA_TL_MAX(a, vcta, f) \
  do { if ((vcta) < kTimelinePipes) atomicMax(&timeline_row(a, vcta)[f], timeline_now()); } while (0)
#define PKA_TL_VAL(a, vcta, f, v) \
  do { if ((vcta) < kTimelinePipes) timeline_row(a, vcta)[f] = (v); } while (0)
#else
#define PKA_TL_SET(a, vcta, f) do { } while (0)
#define PKA_TL_MAX(a, vcta, f) do { } while (0)
#define PKA_TL_VAL(a, vcta, f, v) do { } while (0)
#endif

namespace {

__device__ __forceinline__ int warp_incl_scan(int x, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  return x;
}

// Named barrier `id` over `nthreads` threads: the consumer warps only (the
// producer keeps streaming), or the whole (sub-)CTA.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Where one decode pipeline runs: a CTA of its own, or one of two pipelines
// sharing a CTA of the mixed-batch launch.  vcta / vgrid replace blockIdx.x /
// gridDim.x in the work partition, tid is the thread's index within the
// pipeline's (NW + 1) warps, and bar_all / bar_cons are the named barriers of
// the whole pipeline and of its consumer warps.
struct DecodeCtx {
  int vcta, vgrid, tid, bar_all, bar_cons, bar_merge;
};

// Arrival on named barrier `id` without waiting (the waiting side uses
// named_sync with the same thread count).  Memory accesses before the
// arrival are visible to the threads that complete the barrier.
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Visible keys of request b's decode query: positions [t_lo, pos], blocks
// [jlo, jlo + nb).
struct ReqGeo {
  int jlo, nb, t_lo, pos;
  bool skip;  // not a decode row of a mixed batch: no piece, no output
};

// The request's context length after the checks below (clamped to its
// table row), or -1 for a request the launch skips, from its
// query_start_loc pair (lo, hi; ignored without query_start_loc) and its
// seq_len L.
__device__ __forceinline__ int req_len_of(const DecodeArgs& a, int lo, int hi, int L) {
  if (a.query_start_loc != nullptr) {
    // a varlen batch: the request's query row is query_start_loc[b + 1] - 1;
    // a span outside [0, total_q] (or longer than max_query_len) is skipped
    // and reported, so no row outside the output is ever written
    if (lo < 0 || hi < lo || hi > a.total_q || hi - lo > a.max_query_len) {
      report(a.err, PKA_DEVERR_QUERY_LOC);
      return -1;
    }
    if (hi - lo != 1 && a.decode_rows_only != 0) return -1;
  }
  if (L > a.max_blocks * kBlockSize || L < 0) {
    report(a.err, PKA_DEVERR_SEQ_LEN);  // error path only: tables cannot hold it
    L = max(0, min(L, a.max_blocks * kBlockSize));
  }
  return L;
}

__device__ __forceinline__ int req_len(const DecodeArgs& a, int b) {
  const bool v = a.query_start_loc != nullptr;
  return req_len_of(a, v ? a.query_start_loc[b] : 0, v ? a.query_start_loc[b + 1] : 0,
                    a.seq_lens[b]);
}

// Visible blocks of a request from req_len's value (no memory access).
__device__ __forceinline__ ReqGeo geo_of_len(const DecodeArgs& a, int L) {
  ReqGeo g;
  g.skip = L < 0;
  if (g.skip) {
    g.pos = -1;
    g.t_lo = g.jlo = g.nb = 0;
    return g;
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
  int npieces;   // split-K: pieces (slots used) of this segment
};

// The split-K work line.  Segments (request, KV head) are laid end to end,
// in that order, on a line of work units: a segment with n > 0 visible tiles
// takes kPieceCost units followed by one unit per tile, an empty one none.
// The kPieceCost units stand for the fixed cost of a piece (merging the
// warps' states, writing the partial row): a pipeline whose range starts a
// new segment gets that many fewer tiles.  The T units are cut into chunks
// of q = max(min_chunk, ceil(T / pipelines)) units, chunk c for pipeline c;
// the piece of a segment in chunk c goes to partial slot
// c - floor(A / q), A the unit of the segment's first tile.  All quantities
// fit in 31 bits (checked on the host), so the arithmetic is 32-bit.
constexpr int kPieceCost = 4;
// Requests whose lengths a pipeline keeps in shared memory (the partition
// scans and the walk over segments read them there instead of going back to
// global memory, a round trip of several hundred ns each on the path to the
// first tile); longer batches read the rest from global memory.
constexpr int kLenCache = 128;

// Enumerates the pieces of one pipeline.  Every lane of a warp runs it in
// lockstep (it uses warp scans), and every warp of the pipeline sees the
// same sequence.
struct PieceIter {
  const DecodeArgs* a;
  const int* slen;  // req_len of the first min(B, kLenCache) requests (shared memory)
  int vcta, vgrid;  // this pipeline's index and the number of pipelines
  bool direct;
  // direct mode
  int item;
  // split mode: this pipeline's chunk [lo, hi) of the work line
  int q, lo, hi;
  bool last;    // the chunk holding the line's last unit: also takes the
                // empty segments at its end
  int b, kvh;
  int prefix;   // units of one KV head's segments of the requests before b
  ReqGeo geo;
  bool done;

  __device__ static int units(int nb) { return nb > 0 ? nb + kPieceCost : 0; }
  __device__ int len_of(int bb) const { return bb < kLenCache ? slen[bb] : req_len(*a, bb); }

  __device__ void init(const DecodeArgs& args, const int* slen_, int lane, int vcta_, int vgrid_) {
    a = &args;
    slen = slen_;
    vcta = vcta_;
    vgrid = vgrid_;
    direct = args.split_blocks <= 0;
    done = false;
    if (direct) {
      item = vcta;
      return;
    }
    // T = Hkv * sum_b units(nb_b); the units of 32 requests per step, kept
    // per lane for the search below when the batch has at most 32 requests
    int T = 0;
    int u_first = 0;
    int u_max = 0;
    for (int base = 0; base < args.batch; base += 32) {
      const int bb = base + lane;
      const int u = units(bb < args.batch ? geo_of_len(args, len_of(bb)).nb : 0);
      if (base == 0) u_first = u;
      T += __shfl_sync(0xffffffffu, warp_incl_scan(u, lane), 31);
      u_max = max(u_max, u);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) u_max = max(u_max, __shfl_xor_sync(0xffffffffu, u_max, o));
    T *= args.Hkv;
    q = max(max(args.split_blocks, 1), (T + vgrid - 1) / vgrid);
    // With the combine fused in and direct_slack > 0, a batch whose segments
    // all fit one per pipeline and are all short of the split's chunk plus
    // direct_slack units runs without splitting: each segment streams on its
    // own pipeline and writes its output directly, with no partials and no
    // merge (the merge at the end of the launch costs about as much as
    // streaming a couple of dozen tiles).
    if (args.seg_counters != nullptr && args.direct_slack > 0 &&
        args.batch * args.Hkv <= vgrid && u_max <= q + args.direct_slack) {
      direct = true;
      item = vcta;
      return;
    }
    const int nch = T > 0 ? (T + q - 1) / q : 1;
    if (vcta >= nch) {
      done = true;
      return;
    }
    lo = vcta * q;
    hi = min(T, lo + q);
    last = (vcta == nch - 1);
    // first request holding a segment this chunk touches: the first b with
    // Hkv * (prefix_b + u_b) + (u_b == 0) > lo
    int run = 0;
    b = args.batch;
    prefix = 0;
    for (int base = 0; base < args.batch; base += 32) {
      const int bb = base + lane;
      const int u = (base == 0) ? u_first
                                : units(bb < args.batch ? geo_of_len(args, len_of(bb)).nb : 0);
      const int incl = warp_incl_scan(u, lane);
      const int pre = run + incl - u;
      const bool hit = (bb < args.batch) && (args.Hkv * (pre + u) + (u == 0 ? 1 : 0) > lo);
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
    if (b < args.batch) geo = geo_of_len(args, len_of(b));
  }

  // The next piece.  `slots`: also its partial slot, the segment's number of
  // pieces and the slots to fill (the producer needs none of them).
  __device__ bool next(Piece& p, bool slots) {
    if (done) return false;
    const DecodeArgs& A = *a;
    if (direct) {
      const int nseg = A.batch * A.Hkv;
      ReqGeo g;
      while (true) {
        if (item >= nseg) {
          done = true;
          return false;
        }
        p.b = item / A.Hkv;
        p.kvh = item % A.Hkv;
        g = geo_of_len(A, len_of(p.b));
        if (!g.skip) break;
        item += vgrid;
      }
      p.j0 = g.jlo;
      p.ntiles = g.nb;
      p.t_lo = g.t_lo;
      p.pos = g.pos;
      p.slot = 0;
      p.fill_from = -1;
      p.npieces = 1;
      item += vgrid;
    } else {
      while (true) {
        if (b >= A.batch) {
          done = true;
          return false;
        }
        const int n = geo.nb;
        const int u = units(n);
        const int seg = A.Hkv * prefix + kvh * u;       // segment start
        const int s0 = seg + (n > 0 ? kPieceCost : 0);  // unit of its first tile
        const bool before = (n > 0 ? s0 + n : seg + 1) <= lo;  // wholly before this chunk
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
          prefix += u;
          ++b;
          if (b < A.batch) geo = geo_of_len(A, len_of(b));
        }
        if (before || g.skip) continue;
        const int t0 = max(s0, lo);
        const int t1 = min(s0 + n, hi);
        p.b = cur_b;
        p.kvh = cur_kvh;
        p.j0 = g.jlo + (t0 - s0);
        p.ntiles = max(0, t1 - t0);
        p.t_lo = g.t_lo;
        p.pos = g.pos;
        p.slot = 0;
        p.npieces = 0;
        p.fill_from = (n == 0) ? 0 : -1;
        if (n > 0 && slots) {
          // the chunk holding the first tile writes slot 0; a chunk whose
          // range holds only the segment's piece-cost units has no piece
          const int cfirst = s0 / q;
          p.slot = vcta - cfirst;
          p.npieces = (s0 + n - 1) / q - cfirst + 1;
          if (p.slot == 0) p.fill_from = p.npieces;
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

// ------------------------------------------------------ warp-level MMA
// mma.sync m16n8k16 (bf16 in, fp32 accumulate) and ldmatrix, as inline PTX.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

template <int D, int G, int NW, int NSLOT>
struct DecodeShape {
  static constexpr int DC = D / 64;                        // 64-column boxes of a key row
  static constexpr int kBoxBytes = kBlockSize * 128;       // one 16-row x 64-column box
  static constexpr int kTileBytes = kBlockSize * D * 2;    // one block's K (or V) tile
  static constexpr int KSTEPS = D / 16;                    // k-steps of S = K q^T
  static constexpr int MTILES = D / 16;                    // 16-row tiles of O^T = V^T P^T
  static constexpr int kRingBytes = NSLOT * 2 * kTileBytes;
  static constexpr int kBarBytes = (2 * NSLOT * 8 + 8 + 15) / 16 * 16;  // + staging_free
  // piece epilogue: warps 1..NW-1 leave their accumulator fragments (the
  // lanes whose columns are query heads: t < TG) and their (max, sum) here
  // for warp 0, which merges them in registers
  static constexpr int TG = (G + 1) / 2;
  static constexpr int kStageFrags = (NW - 1) * (D / 16) * 8 * TG;  // float4 each
  static constexpr int kStageML = (NW - 1) * TG;                      // float4 each
  static constexpr int kMergeBytes = (kStageFrags + kStageML) * 16;
  // fused combine: up to kMaxPend pieces whose arrival is deferred to the
  // end of the CTA's work, 4 ints each, and one "last piece" flag per entry
  static constexpr int kMaxPend = 4;
  static constexpr int kPendBytes = kMaxPend * 5 * 4;
  // the lengths of the first kLenCache requests
  static constexpr int kLenBytes = kLenCache * 4;
  // a piece's result on its way out: G rows of D fp32 (bulk-copied to the
  // partials, or converted to bf16 in place for a direct output)
  static constexpr int kOutBytes = G * D * 4;
  // + 1 KiB so the ring can start on a 1024-byte boundary (128B swizzle)
  static constexpr int kSmemBytes =
      1024 + kRingBytes + kBarBytes + kMergeBytes + kPendBytes + kLenBytes + kOutBytes;
  static_assert(G >= 1 && G <= 8, "the query heads of a group are the MMA's N = 8 columns");
  static_assert(kSmemBytes <= 232448 / 2 - 1024, "two CTAs per SM");
  static_assert(NSLOT % NW == 0, "each ring slot must have exactly one owner warp");
};

// One ring slot (a block's 16 keys) for one consumer warp, on the tensor
// cores at warp level: S^T[16 keys x 8] = K[16 x D] q^T[D x 8] (the G query
// heads are the N columns, the rest zero), online softmax on the fragments
// with shuffles, then O^T[D x 8] += V^T[D x 16] P^T[16 x 8].  K and V come
// from 128B-swizzled boxes, so every ldmatrix is bank-conflict free.
// Fragment roles (g = lane / 4, t = lane % 4): S^T holds keys g and g+8 of
// heads 2t and 2t+1; O^T tile mt holds rows mt*16 + g (+8) of heads 2t, 2t+1.
template <int D, int G, int NW, int NSLOT>
__device__ __forceinline__ void decode_slot(
    const bool edge, uint32_t k_addr, uint8_t* v_ptr, const uint32_t (&bq)[D / 16][2],
    float (&o)[D / 16][4], float (&m)[2], float (&l)[2], int lane, int tok0, int t_lo, int pos,
    float qscale, float softcap, float inv_cap, float* logits, int logit_stride) {
  using S = DecodeShape<D, G, NW, NSLOT>;
  const int g = lane >> 2, t = lane & 3;

  // ---- S^T = K q^T (even and odd k-steps in two accumulators: two
  // dependent MMA chains of half the length)
  float s[4] = {0.f, 0.f, 0.f, 0.f};
  float s2[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int row = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int hi = lane >> 4;
    const uint32_t rbase = k_addr + row * 128;
#pragma unroll
    for (int kk = 0; kk < S::KSTEPS; ++kk) {
      uint32_t a[4];
      const int j = (kk & 3) * 2 + hi;
      ldmatrix_x4(a, rbase + (kk >> 2) * S::kBoxBytes + ((j ^ (row & 7)) << 4));
      if (kk & 1)
        mma_bf16_16816(s2, a, bq[kk][0], bq[kk][1]);
      else
        mma_bf16_16816(s, a, bq[kk][0], bq[kk][1]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] += s2[i];
  }
  // ---- logits (log2 domain), mask, online softmax on the fragment
  const bool head_ok0 = (2 * t) < G, head_ok1 = (2 * t + 1) < G;
  bool key_ok_lo = true, key_ok_hi = true;
  if (edge) {
    key_ok_lo = (tok0 + g >= t_lo) && (tok0 + g <= pos);
    key_ok_hi = (tok0 + g + 8 >= t_lo) && (tok0 + g + 8 <= pos);
  }
  float x[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float v = s[i];
    if (softcap > 0.f) {
      // tanh(y) = 1 - 2 / (e^{2y} + 1); absolute error ~1e-7
      const float e = fast_exp2(fminf(2.f * kLog2e * (v * qscale * inv_cap), 126.f));
      v = softcap * (1.f - __fdividef(2.f, e + 1.f)) * kLog2e;
    }
    else v *= qscale;
    const bool ok = ((i & 1) ? head_ok1 : head_ok0) && ((i & 2) ? key_ok_hi : key_ok_lo);
    x[i] = ok ? v : -INFINITY;
    // optional: the visible keys' log2-domain logits of the G heads
    // (logits points at head kvh * G, key 0 of the request)
    if (logits != nullptr && ok)
      logits[(2 * t + (i & 1)) * logit_stride + tok0 + g + ((i & 2) ? 8 : 0)] = v;
  }
  float alpha[2], ms[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float mx = fmaxf(x[j], x[j + 2]);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float mn = fmaxf(m[j], mx);
    ms[j] = (mn == -INFINITY) ? 0.f : mn;
    alpha[j] = fast_exp2(m[j] - ms[j]);
    m[j] = mn;
  }
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = fast_exp2(x[i] - ms[i & 1]);
  l[0] = l[0] * alpha[0] + p[0] + p[2];
  l[1] = l[1] * alpha[1] + p[1] + p[3];
  if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < S::MTILES; ++mt) {
      o[mt][0] *= alpha[0];
      o[mt][1] *= alpha[1];
      o[mt][2] *= alpha[0];
      o[mt][3] *= alpha[1];
    }
  }
  // ---- P^T as the B fragment: this thread needs keys 2t, 2t+1 (+8) of head g
  const uint32_t wlo = pack_bf16x2(p[0], p[1]);  // key g,   heads 2t, 2t+1
  const uint32_t whi = pack_bf16x2(p[2], p[3]);  // key g+8, heads 2t, 2t+1
  const int src0 = 8 * t + (g >> 1), src1 = src0 + 4;
  const uint32_t a0 = __shfl_sync(0xffffffffu, wlo, src0);
  const uint32_t a1 = __shfl_sync(0xffffffffu, wlo, src1);
  const uint32_t c0 = __shfl_sync(0xffffffffu, whi, src0);
  const uint32_t c1 = __shfl_sync(0xffffffffu, whi, src1);
  const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
  const uint32_t pb0 = prmt(a0, a1, sel);
  const uint32_t pb1 = prmt(c0, c1, sel);
  // ---- stale slots past the sequence end may hold NaN: zero those V rows
  if (edge && tok0 + kBlockSize - 1 > pos) {
    const int z0 = max(0, pos - tok0 + 1);
    const int nz = (kBlockSize - z0) * S::DC * 8;
    for (int idx = lane; idx < nz; idx += 32) {
      const int r = z0 + idx / (S::DC * 8);
      const int c = (idx / 8) % S::DC;
      const int q = idx % 8;
      *reinterpret_cast<uint4*>(v_ptr + c * S::kBoxBytes + r * 128 + q * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    // the slot is refilled by TMA later: order these writes before it
    fence_proxy_async_smem();
    __syncwarp();
  }
  // ---- O^T += V^T P^T
  {
    const int mi = lane >> 3, rr = lane & 7;
    const int key = rr + 8 * (mi >> 1);
    const uint32_t vbase = smem_u32(v_ptr) + key * 128;
#pragma unroll
    for (int mt = 0; mt < S::MTILES; ++mt) {
      const int dch = mt * 2 + (mi & 1);  // 16-byte chunk along D
      uint32_t a[4];
      ldmatrix_x4_trans(a, vbase + (dch >> 3) * S::kBoxBytes + (((dch & 7) ^ (key & 7)) << 4));
      mma_bf16_16816(o[mt], a, pb0, pb1);
    }
  }
}

// One decode pipeline: a producer warp and NW consumer warps over the
// S::kSmemBytes of shared memory at smem_raw (aligned here to 1 KiB).
template <int D, int G, int NW, int NSLOT>
__device__ __forceinline__ void decode_body(const DecodeArgs& a, const CUtensorMap* tm_k,
                                            const CUtensorMap* tm_v, uint8_t* smem_raw,
                                            const DecodeCtx& cx) {
  using S = DecodeShape<D, G, NW, NSLOT>;

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kRingBytes);
  uint64_t* empty = full + NSLOT;
  uint64_t* staging_free = empty + NSLOT;  // warp 0 has read the staging area
  float4* stage = reinterpret_cast<float4*>(smem + S::kRingBytes + S::kBarBytes);
  float4* stage_ml = stage + S::kStageFrags;  // [NW-1][TG]: (m0, m1, l0, l1)
  int* pend = reinterpret_cast<int*>(smem + S::kRingBytes + S::kBarBytes + S::kMergeBytes);
  volatile int* pend_last = pend + S::kMaxPend * 4;  // [kMaxPend]
  int npend = 0;  // the same in every consumer thread
  int* slen = reinterpret_cast<int*>(smem + S::kRingBytes + S::kBarBytes + S::kMergeBytes +
                                     S::kPendBytes);  // [kLenCache]
  float* orow = reinterpret_cast<float*>(smem + S::kRingBytes + S::kBarBytes + S::kMergeBytes +
                                         S::kPendBytes + S::kLenBytes);  // [G][D]

  const int warp = cx.tid / 32;
  const int lane = cx.tid % 32;
  if (cx.tid == 0) PKA_TL_SET(a, cx.vcta, TL_ENTRY);

  if (warp == NW) {
    // the producer warp sets up the barriers (one lane each) and reads the
    // requests' lengths into shared memory for the whole pipeline
    for (int i = lane; i < 2 * NSLOT + 1; i += 32) mbar_init(full + i, 1);
    mbar_fence_init();
    // every load is issued before the first check, so that the lengths
    // take one memory round trip
    const int ncache = min(a.batch, kLenCache);
    const bool varlen = a.query_start_loc != nullptr;
    int lo[kLenCache / 32], hi[kLenCache / 32], sl[kLenCache / 32];
#pragma unroll
    for (int k = 0; k < kLenCache / 32; ++k) {
      const int bb = lane + 32 * k;
      const bool in = bb < ncache;
      lo[k] = (in && varlen) ? a.query_start_loc[bb] : 0;
      hi[k] = (in && varlen) ? a.query_start_loc[bb + 1] : 0;
      sl[k] = in ? a.seq_lens[bb] : 0;
    }
#pragma unroll
    for (int k = 0; k < kLenCache / 32; ++k) {
      const int bb = lane + 32 * k;
      if (bb < ncache) slen[bb] = req_len_of(a, lo[k], hi[k], sl[k]);
    }
  }
  named_sync(cx.bar_all, (NW + 1) * 32);

  PieceIter iter;
  iter.init(a, slen, lane, cx.vcta, cx.vgrid);
  Piece pc;

  if (warp == NW) {
    // ============================ producer warp ============================
    if (lane == 0) {
      prefetch_tensormap(tm_k);
      prefetch_tensormap(tm_v);
    }
    const uint32_t oob_row = static_cast<uint32_t>(a.num_blocks) * a.Hkv * kBlockSize;
    int issued = 0;
    bool ok = true;
    if (lane == 0) PKA_TL_SET(a, cx.vcta, TL_PARTITION);
    while (ok && iter.next(pc, false)) {
      const int32_t* trow = a.tables + static_cast<size_t>(pc.b) * a.max_blocks + pc.j0;
      for (int base = 0; base < pc.ntiles && ok; base += 32) {
        uint32_t row = oob_row;  // a bad id reads zeros (reported) instead of faulting
        if (base + lane < pc.ntiles) {
          const int id = trow[base + lane];
          if (static_cast<unsigned>(id) < static_cast<unsigned>(a.num_blocks))
            row = (static_cast<uint32_t>(id) * a.Hkv + pc.kvh) * kBlockSize;
          else
            report(a.err, PKA_DEVERR_BAD_TABLE);
        }
        const int cnt = min(32, pc.ntiles - base);
        for (int k = 0; k < cnt; ++k) {
          const uint32_t r0 = __shfl_sync(0xffffffffu, row, k);
          const int slot = issued % NSLOT;
          const int round = issued / NSLOT;
          int good = 1;
          if (lane == 0) {
            if (round > 0)
              good = mbar_wait(&empty[slot], static_cast<uint32_t>((round - 1) & 1), a.err);
            if (good) mbar_arrive_expect_tx(&full[slot], 2 * S::kTileBytes);
          }
          good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) {
            ok = false;
            break;
          }
          // one copy per tensor (the whole 16 x D block as DC boxes of 16 rows
          // x 64 columns), K from lane 0 and V from lane 1: one thread's
          // copies are processed one after another
          if (lane < 2) {
            uint8_t* dst =
                ring + static_cast<size_t>(slot) * 2 * S::kTileBytes + lane * S::kTileBytes;
            tma_load_3d(dst, lane == 0 ? tm_k : tm_v, 0, static_cast<int>(r0), 0, &full[slot]);
          }
          if (lane == 0 && issued == 0) PKA_TL_SET(a, cx.vcta, TL_FIRST_ISSUE);
          ++issued;
        }
      }
    }
    if (lane == 0) {
      PKA_TL_SET(a, cx.vcta, TL_LAST_ISSUE);
      PKA_TL_VAL(a, cx.vcta, TL_TILES, static_cast<unsigned long long>(issued));
    }
    // Every issued copy must have landed before the CTA may exit.
    if (lane == 0) {
      const int first = issued > NSLOT ? issued - NSLOT : 0;
      for (int i = first; i < issued; ++i)
        mbar_wait(&full[i % NSLOT], static_cast<uint32_t>((i / NSLOT) & 1), a.err);
    }
    return;
  }

  // ============================ consumer warps ============================
  const int g = lane >> 2, t = lane & 3;
  const float inv_cap = a.softcap > 0.f ? 1.f / a.softcap : 0.f;
  const float qscale = a.scale * (a.softcap > 0.f ? 1.f : kLog2e);
  int tile_base = 0;
  int nmerge = 0;  // pieces merged so far (phases of staging_free)
  bool ok = true;

  // q^T as B fragments: head g (zero for g >= G), elements 2t, 2t+1 (+8) of
  // every k-step.
  auto load_q = [&](const Piece& P, uint32_t (&bq)[D / 16][2]) {
    const uint32_t* qp = reinterpret_cast<const uint32_t*>(
        a.q + (static_cast<size_t>(P.qrow) * a.Hq + P.kvh * G + (g < G ? g : 0)) * D);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      bq[kk][0] = (g < G) ? qp[kk * 8 + t] : 0u;
      bq[kk][1] = (g < G) ? qp[kk * 8 + 4 + t] : 0u;
    }
  };

  // Arrivals of the pending pieces (one fence for all of them, the atomics
  // in flight together), then the merge of every segment they complete.
  auto flush_pending = [&]() {
    named_sync(cx.bar_cons, NW * 32);  // the pieces' partials and pend[] written
    if (cx.tid == 0) {
      bulk_wait_all();      // this thread's bulk copies of the partials have completed
      fence_acq_rel_gpu();  // the CTA's partials (ordered by the barrier) before its arrivals
      int old[S::kMaxPend];
#pragma unroll
      for (int i = 0; i < S::kMaxPend; ++i)
        if (i < npend) old[i] = atomicAdd(&a.seg_counters[pend[i * 4] * a.Hkv + pend[i * 4 + 1]], 1);
#pragma unroll
      for (int i = 0; i < S::kMaxPend; ++i)
        if (i < npend) pend_last[i] = (old[i] == pend[i * 4 + 2] - 1) ? 1 : 0;
      // the other CTAs' partials of every segment this CTA completes are
      // visible to the consumer threads after this fence and the barrier
      fence_acq_rel_gpu();
    }
    named_sync(cx.bar_cons, NW * 32);
    for (int i = 0; i < npend; ++i) {
      if (pend_last[i] == 0) continue;  // uniform
      const int cb = pend[i * 4], ckvh = pend[i * 4 + 1], np = pend[i * 4 + 2];
      const int cqrow = pend[i * 4 + 3];
      // One pass over the pieces (read from L2): four consecutive columns
      // of one head per item, the pieces' LSE and partial rows of four
      // pieces loaded together, merged with a running maximum.  Up to
      // kBatch of a thread's items go together, group by group, so that
      // their loads are in flight at once.
      constexpr int kItems = G * (D / 4);
      constexpr int kPerThread = (kItems + NW * 32 - 1) / (NW * 32);
      constexpr int kBatch = kPerThread < 2 ? kPerThread : 2;
#pragma unroll 1
      for (int k0 = 0; k0 < kPerThread; k0 += kBatch) {
        float M[kBatch], den[kBatch];
        float4 acc[kBatch];
        size_t ph0[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int item = cx.tid + (k0 + k) * NW * 32;
          M[k] = -INFINITY;
          den[k] = 0.f;
          acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          ph0[k] = (static_cast<size_t>(cb) * a.Hq + ckvh * G + min(item, kItems - 1) / (D / 4)) *
                   a.num_splits;
        }
        for (int s0 = 0; s0 < np; s0 += 4) {
          float lv[kBatch][4];
          float4 x[kBatch][4];
#pragma unroll
          for (int k = 0; k < kBatch; ++k) {
            const int item = cx.tid + (k0 + k) * NW * 32;
            const int d0 = (item % (D / 4)) * 4;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (k0 + k < kPerThread && item < kItems && s0 + u < np) {
                lv[k][u] = __ldcg(a.partial_lse + ph0[k] + s0 + u);
                x[k][u] = __ldcg(reinterpret_cast<const float4*>(a.partial_o +
                                                                 (ph0[k] + s0 + u) * D + d0));
              } else {
                lv[k][u] = -INFINITY;
                x[k][u] = make_float4(0.f, 0.f, 0.f, 0.f);
              }
            }
          }
#pragma unroll
          for (int k = 0; k < kBatch; ++k) lse_merge4(M[k], den[k], acc[k], lv[k], x[k]);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int item = cx.tid + (k0 + k) * NW * 32;
          if (k0 + k < kPerThread && item < kItems) {
            const int h = item / (D / 4);
            const int d0 = (item % (D / 4)) * 4;
            const float inv = den[k] > 0.f ? 1.f / den[k] : 0.f;
            uint16_t* dst = reinterpret_cast<uint16_t*>(a.out) +
                            (static_cast<size_t>(cqrow) * a.Hq + ckvh * G + h) * D + d0;
            *reinterpret_cast<uint2*>(dst) =
                make_uint2(pack_bf16x2(acc[k].x * inv, acc[k].y * inv),
                           pack_bf16x2(acc[k].z * inv, acc[k].w * inv));
          }
        }
      }
      named_sync(cx.bar_cons, NW * 32);
      if (cx.tid == 0) a.seg_counters[cb * a.Hkv + ckvh] = 0;
    }
    named_sync(cx.bar_cons, NW * 32);  // pend[] and pend_last[] free again
  };

  uint32_t bq[D / 16][2];
  bool have = iter.next(pc, true);
  if (have) load_q(pc, bq);
  while (have) {
    float o[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};

    // Tile T of the pipeline's stream lives in slot T % NSLOT and belongs to
    // warp T % NW; NSLOT is a multiple of NW, so every slot has one owner warp
    // that consumes its phases in order (a phase-parity wait can never alias
    // an older phase of the same slot), even when warps 1..NW-1 run ahead into
    // the next piece while warp 0 merges.  Warp w takes the piece's tiles
    // i = res (mod NW), res = (w - tile_base) mod NW; the merge adds the
    // warps' states in the order of res, so a piece gives the same bits
    // wherever in the stream it falls.
    const int rho = tile_base % NW;
    const int i0 = (warp - rho + NW) % NW;
    float* lg = (a.logits == nullptr)
                    ? nullptr
                    : a.logits + (static_cast<size_t>(pc.b) * a.Hq + pc.kvh * G) *
                                     (static_cast<size_t>(a.max_blocks) * kBlockSize);
    // ---- split-K: slots of this segment no pipeline fills get LSE = -inf,
    // written at the start of the piece by the last consumer warp (hidden
    // behind the wait for the piece's first tiles)
    if (!iter.direct && a.seg_counters == nullptr && pc.fill_from >= 0 && warp == NW - 1) {
      if (pc.fill_from > a.num_splits && lane == 0) report(a.err, PKA_DEVERR_SEQ_LEN);
      for (int h = 0; h < G; ++h)
        for (int sl = pc.fill_from + lane; sl < a.num_splits; sl += 32)
          a.partial_lse[(static_cast<size_t>(pc.b) * a.Hq + pc.kvh * G + h) * a.num_splits + sl] =
              -INFINITY;
    }
    for (int i = i0; i < pc.ntiles && ok; i += NW) {
      const int T = tile_base + i;
      const int slot = T % NSLOT;
      const bool got = mbar_wait(&full[slot], static_cast<uint32_t>((T / NSLOT) & 1), a.err);
      if (T == 0 && cx.tid == 0) PKA_TL_SET(a, cx.vcta, TL_FIRST_TILE);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      uint8_t* kp = ring + static_cast<size_t>(slot) * 2 * S::kTileBytes;
      const int tok0 = (pc.j0 + i) * kBlockSize;
      const bool edge = (tok0 < pc.t_lo || tok0 + kBlockSize - 1 > pc.pos);
      decode_slot<D, G, NW, NSLOT>(edge, smem_u32(kp), kp + S::kTileBytes, bq, o, m, l, lane,
                                   tok0, pc.t_lo, pc.pos, qscale, a.softcap, inv_cap, lg,
                                   a.max_blocks * kBlockSize);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
    tile_base += pc.ntiles;
    if (lane == 0) PKA_TL_MAX(a, cx.vcta, TL_LAST_TILE);

    Piece nx;
    const bool have_next = iter.next(nx, true);

    const bool split = !iter.direct;
    const bool fused = split && a.seg_counters != nullptr;
    if (pc.ntiles > 0) {
      // ---- per-warp totals: sums over the 8 key rows held by lanes g
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) l[j] += __shfl_xor_sync(0xffffffffu, l[j], off);
      if (warp != 0) {
        // ---- leave this warp's state for warp 0 and go on with the next
        // piece at once: the ring keeps flowing while warp 0 merges
        if (nmerge > 0 && ok) {
          const bool got = mbar_wait(staging_free, static_cast<uint32_t>((nmerge - 1) & 1), a.err);
          if (!__all_sync(0xffffffffu, got)) ok = false;
        }
        if (t < S::TG) {
          float4* st = stage + ((warp - 1) * (D / 16)) * 8 * S::TG + g * S::TG + t;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt)
            st[mt * 8 * S::TG] = make_float4(o[mt][0], o[mt][1], o[mt][2], o[mt][3]);
          if (g == 0) stage_ml[(warp - 1) * S::TG + t] = make_float4(m[0], m[1], l[0], l[1]);
        }
        named_arrive(cx.bar_merge, NW * 32);
      } else {
        // ---- warp 0: merge the other warps' states into its registers
        named_sync(cx.bar_merge, NW * 32);
        if (t < S::TG) {
          // the warps' (m0, m1, l0, l1); warp 0's own are in its registers
          const float4 own_ml = make_float4(m[0], m[1], l[0], l[1]);
          float M0 = m[0], M1 = m[1];
#pragma unroll
          for (int w = 1; w < NW; ++w) {
            const float4 x = stage_ml[(w - 1) * S::TG + t];
            M0 = fmaxf(M0, x.x);
            M1 = fmaxf(M1, x.y);
          }
          const float Ms0 = (M0 == -INFINITY) ? 0.f : M0;
          const float Ms1 = (M1 == -INFINITY) ? 0.f : M1;
          // residue r's state (warp (r + rho) % NW) is scaled by sc[r]
          float sc[NW][2];
          float den0 = 0.f, den1 = 0.f;
#pragma unroll
          for (int r = 0; r < NW; ++r) {
            const int w = (r + rho) % NW;
            const float4 x = (w == 0) ? own_ml : stage_ml[(w - 1) * S::TG + t];
            sc[r][0] = fast_exp2(x.x - Ms0);
            sc[r][1] = fast_exp2(x.y - Ms1);
            den0 = (r == 0) ? sc[r][0] * x.z : fmaf(sc[r][0], x.z, den0);
            den1 = (r == 0) ? sc[r][1] * x.w : fmaf(sc[r][1], x.w, den1);
          }
          m[0] = M0;
          m[1] = M1;
          l[0] = den0;
          l[1] = den1;
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            const float4 own = make_float4(o[mt][0], o[mt][1], o[mt][2], o[mt][3]);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < NW; ++r) {
              const int w = (r + rho) % NW;
              const float4 x =
                  (w == 0) ? own : stage[(((w - 1) * (D / 16) + mt) * 8 + g) * S::TG + t];
              if (r == 0) {
                acc = make_float4(sc[0][0] * x.x, sc[0][1] * x.y, sc[0][0] * x.z, sc[0][1] * x.w);
              } else {
                acc.x = fmaf(sc[r][0], x.x, acc.x);
                acc.y = fmaf(sc[r][1], x.y, acc.y);
                acc.z = fmaf(sc[r][0], x.z, acc.z);
                acc.w = fmaf(sc[r][1], x.w, acc.w);
              }
            }
            o[mt][0] = acc.x;
            o[mt][1] = acc.y;
            o[mt][2] = acc.z;
            o[mt][3] = acc.w;
          }
        }
        // the staging area may be refilled (its reads are done)
        __syncwarp();
        if (lane == 0) mbar_arrive(staging_free);
        // ---- this piece's result: each head's normalised row into the output
        // buffer (once the previous piece's bulk copies have read it), then
        // out through the async proxy: warp 0 does not wait for the copies to
        // reach memory behind the K/V stream
        if (lane == 0) bulk_wait_read_all();
        __syncwarp();
        const float inv0 = l[0] > 0.f ? 1.f / l[0] : 0.f;
        const float inv1 = l[1] > 0.f ? 1.f / l[1] : 0.f;
        const int h0 = 2 * t, h1 = 2 * t + 1;
        if (split) {
          if (t < S::TG) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              orow[h0 * D + mt * 16 + g] = o[mt][0] * inv0;
              orow[h0 * D + mt * 16 + g + 8] = o[mt][2] * inv0;
              if (h1 < G) {
                orow[h1 * D + mt * 16 + g] = o[mt][1] * inv1;
                orow[h1 * D + mt * 16 + g + 8] = o[mt][3] * inv1;
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (pc.slot < a.num_splits) {
            const size_t r0 = (static_cast<size_t>(pc.b) * a.Hq + pc.kvh * G) * a.num_splits +
                              pc.slot;  // row of head 0 of the group
            if (lane == 0) {
#pragma unroll
              for (int h = 0; h < G; ++h)
                bulk_s2g(a.partial_o + (r0 + static_cast<size_t>(h) * a.num_splits) * D,
                         orow + h * D, D * 4);
              bulk_commit();
            }
            if (t < S::TG && g == 0) {
              a.partial_lse[r0 + static_cast<size_t>(h0) * a.num_splits] =
                  l[0] > 0.f ? (m[0] + log2f(l[0])) * kLn2 : -INFINITY;
              if (h1 < G)
                a.partial_lse[r0 + static_cast<size_t>(h1) * a.num_splits] =
                    l[1] > 0.f ? (m[1] + log2f(l[1])) * kLn2 : -INFINITY;
            }
          }
        } else {
          // bf16 rows of the G heads, contiguous in out
          uint16_t* ob16 = reinterpret_cast<uint16_t*>(orow);
          if (t < S::TG) {
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
              ob16[h0 * D + mt * 16 + g] = f32_to_bf16_rn(o[mt][0] * inv0);
              ob16[h0 * D + mt * 16 + g + 8] = f32_to_bf16_rn(o[mt][2] * inv0);
              if (h1 < G) {
                ob16[h1 * D + mt * 16 + g] = f32_to_bf16_rn(o[mt][1] * inv1);
                ob16[h1 * D + mt * 16 + g + 8] = f32_to_bf16_rn(o[mt][3] * inv1);
              }
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            bulk_s2g(reinterpret_cast<uint16_t*>(a.out) +
                         (static_cast<size_t>(pc.qrow) * a.Hq + pc.kvh * G) * D,
                     ob16, G * D * 2);
            bulk_commit();
          }
        }
      }
      ++nmerge;
    } else if (!split && warp == 0) {
      // a request with no visible key: output 0
      for (int idx = lane; idx < G * D; idx += 32) {
        const int hq = pc.kvh * G + idx / D;
        reinterpret_cast<uint16_t*>(a.out)[(static_cast<size_t>(pc.qrow) * a.Hq + hq) * D +
                                           idx % D] = 0;
      }
    }
    // the next piece's q (after the merge, which needs the registers)
    if (have_next) load_q(nx, bq);
    // ---- fused LSE combine: a piece's arrival on its segment's counter is
    // deferred to the end of the CTA's work (or until kMaxPend pieces are
    // pending), so that a CTA with several pieces never stalls between them
    // on the fence, the atomic or a merge; the arrival that completes a
    // segment merges all of its pieces (the other CTAs' partials are read
    // from L2) and resets the counter for the next call.
    if (fused) {
      if (pc.npieces > a.num_splits && cx.tid == 0) report(a.err, PKA_DEVERR_SEQ_LEN);
      if (pc.ntiles > 0 && pc.slot < a.num_splits) {
        if (cx.tid == 0) {
          pend[npend * 4 + 0] = pc.b;
          pend[npend * 4 + 1] = pc.kvh;
          pend[npend * 4 + 2] = min(pc.npieces, a.num_splits);
          pend[npend * 4 + 3] = pc.qrow;
        }
        ++npend;
      } else if (pc.ntiles == 0 && pc.fill_from == 0 && warp == 0) {
        // a request with no visible key: output 0
        for (int idx = lane; idx < G * D; idx += 32) {
          const int hq = pc.kvh * G + idx / D;
          reinterpret_cast<uint16_t*>(a.out)[(static_cast<size_t>(pc.qrow) * a.Hq + hq) * D +
                                             idx % D] = 0;
        }
      }
    }
    if (fused && npend > 0 && (npend == S::kMaxPend || !have_next)) {
      flush_pending();
      npend = 0;
    }
    pc = nx;
    have = have_next;
  }
  // the bulk copies of the last results complete before the pipeline ends
  if (warp == 0 && lane == 0) bulk_wait_all();
  if (lane == 0) PKA_TL_MAX(a, cx.vcta, TL_EXIT);
}

}  // namespace pka
