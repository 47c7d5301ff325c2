// Append of new tokens' K and V rows into a block-paged pool (sm_103a).
//
// The step that precedes attention on every engine tick: the new tokens'
// keys and values are written into the cache blocks the scheduler gave them
// ("Block-paged per-layer KV with refcounted blocks, lazy allocation, and SDPA
// gather -- vLLM/PagedAttention layout", github README, "What's inside",
// Paged KV cache row).  Token t goes to slot s = slot_mapping[t], i.e. block
// s / bs, offset s % bs, of every KV head; s < 0 means "no slot" (padding).
//
// A pure copy: each thread moves one 16-byte chunk of one (token, head) row
// of K or V, consecutive threads covering consecutive chunks, so both the
// reads of the new rows and the writes into the pool are coalesced 16-byte
// accesses.  Bound by HBM (bytes read + written), and for a decode tick's few
// tokens by launch latency.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace pka {

namespace {

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
  const int cpr = a.head_dim / 8;  // 16-byte chunks per (token, head) row
  const long long per_tensor = static_cast<long long>(a.T) * a.Hkv * cpr;
  const long long total = 2 * per_tensor;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const bool is_v = i >= per_tensor;
    const long long r = is_v ? i - per_tensor : i;
    const int c = static_cast<int>(r % cpr);
    const long long th = r / cpr;  // token * Hkv + head
    const int h = static_cast<int>(th % a.Hkv);
    const int t = static_cast<int>(th / a.Hkv);
    const int s = a.slot_mapping[t];
    if (s < 0) continue;
    const int blk = s / a.block_size, off = s % a.block_size;
    if (blk >= a.num_blocks) {
      if (c == 0 && h == 0 && !is_v) report(a.err, PKA_DEVERR_BAD_TABLE);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(is_v ? a.v_new : a.k_new) + th * cpr + c;
    uint4* dst = reinterpret_cast<uint4*>(is_v ? a.v_pool : a.k_pool) +
                 ((static_cast<long long>(blk) * a.Hkv + h) * a.block_size + off) * cpr + c;
    *dst = __ldg(src);
  }
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs& a, int sm_count, cudaStream_t stream) {
  const long long total = 2LL * a.T * a.Hkv * (a.head_dim / 8);
  if (total == 0) return cudaSuccess;
  const long long want = (total + 255) / 256;
  const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  kv_append_kernel<<<grid, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pka

// ---------------------------------------------------------------------------
// Append with the pre-attention per-head math fused in: RMS norm of q and k
// (learned per-channel weight) and of v (no weight), then rotary position
// embedding of q and k ("Custom Gemma 4 forward -- Dual-RoPE, GQA with
// QK/V-norm + KV sharing", github README, "What's inside"; the two RoPE
// variants of the dual scheme are two calls with their own base and rotary
// width).  RoPE in the rotate-half form: for i < r/2 (r = rotary_dim) the pair
// (x_i, x_{i+r/2}) turns by the angle pos * base^(-2i/r); channels >= r stay.
// Each lane holds D/32 consecutive channels of a row; the pair partner r/2
// channels away sits r/(2 D/32) lanes away.
// Angles: positions reach 1e5 and more, where a float product pos * freq is
// off by ~1e-2 rad, so the host tabulates g_i = freq_i / (2 pi) as 64-bit
// fixed-point fractions (from double precision; passed with the arguments);
// pos * g_i modulo 1 is then the wrapping 64-bit integer product, exact to
// ~2^-39, and its top 24 bits give the reduced angle in [-pi, pi) for the
// sine and cosine.

namespace pka {

namespace {

// One warp per (token, group of up to RB rows): the group's rows are loaded
// together, and its lanes take the sines and cosines of their channels'
// angles once for all the group's rotated rows (the angles depend on the
// token and the channel, not on the head).
template <int D, int RB>
__global__ void __launch_bounds__(256, 3) kv_append_rope_kernel(const AppendRopeArgs a) {
  constexpr int EPL = D / 32;  // channels per lane
  using Chunk = typename std::conditional<EPL == 8, uint4, uint2>::type;
  const int lane = threadIdx.x & 31;
  // the fraction table into shared memory: lanes index it by channel, which
  // parameter memory would serve one distinct address at a time
  __shared__ unsigned long long gfrac[D / 2];
  for (int i = threadIdx.x; i < D / 2; i += blockDim.x) gfrac[i] = a.gfrac[i];
  __syncthreads();
  const int nq = (a.q != nullptr) ? a.Hq : 0;
  const int rows = nq + 2 * a.Hkv;  // q heads, then k heads, then v heads
  const int groups = (rows + RB - 1) / RB;
  const long long items = static_cast<long long>(a.T) * groups;
  const long long wstride = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
  const int half = a.rotary_dim / 2;
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
       w < items; w += wstride) {
    const int t = static_cast<int>(w / groups);
    const int r0 = static_cast<int>(w % groups) * RB;
    const int nr = min(RB, rows - r0);
    // the rows, the slot and the position are independent loads: issue them
    // together so that the group waits for one memory latency
    Chunk u[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (r >= nr) break;
      const int row = r0 + r;
      const uint16_t* src;
      if (row < nq)
        src = a.q + (static_cast<size_t>(t) * a.Hq + row) * D;
      else if (row < nq + a.Hkv)
        src = a.k_new + (static_cast<size_t>(t) * a.Hkv + (row - nq)) * D;
      else
        src = a.v_new + (static_cast<size_t>(t) * a.Hkv + (row - nq - a.Hkv)) * D;
      u[r] = __ldg(reinterpret_cast<const Chunk*>(src + lane * EPL));
    }
    const bool has_kv = r0 + nr > nq;
    const bool rot = a.rotary_dim > 0 && r0 < nq + a.Hkv;  // a q or k row in the group
    const int s = has_kv ? __ldg(a.slot_mapping + t) : 0;
    const int tpos = rot ? __ldg(a.positions + t) : 0;
    // sines and cosines of this lane's channels (channels >= rotary_dim stay)
    float cs[EPL], sn[EPL];
    if (rot) {
      const unsigned long long pos =
          static_cast<unsigned long long>(static_cast<unsigned int>(tpos));
#pragma unroll
      for (int j = 0; j < EPL; ++j) {
        const int e = lane * EPL + j;
        cs[j] = 1.f;
        sn[j] = 0.f;
        if (e < a.rotary_dim) {
          const int i = (e < half) ? e : e - half;
          // (pos * g_i) mod 1 as a 64-bit fraction; its top 24 bits, read as
          // a signed value, give the angle in [-pi, pi), where the hardware
          // sine and cosine are accurate to ~2^-21 absolute
          const unsigned long long ph = pos * gfrac[i];
          const float red = static_cast<float>(static_cast<long long>(ph) >> 40) *
                            (6.2831853071795865f / 16777216.f);
          __sincosf(red, &sn[j], &cs[j]);
          // rotate-half: the first half takes -x_{i+r/2} sin, the second +x_i sin
          if (e < half) sn[j] = -sn[j];
        }
      }
    }
    const int dl = half / EPL;  // lanes between pair partners
    // destination block of the k/v rows (q is rewritten in place)
    int blk = -1, off = 0;
    if (has_kv && s >= 0) {
      blk = s / a.block_size;
      off = s % a.block_size;
      if (blk >= a.num_blocks) {
        if (lane == 0) report(a.err, PKA_DEVERR_BAD_TABLE);
        blk = -1;
      }
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      if (r >= nr) break;
      const int row = r0 + r;
      const int kind = (row < nq) ? 0 : (row < nq + a.Hkv ? 1 : 2);
      const int h = (kind == 0) ? row : (kind == 1 ? row - nq : row - nq - a.Hkv);
      uint16_t* dst;
      if (kind == 0) {
        dst = a.q + (static_cast<size_t>(t) * a.Hq + h) * D;
      } else {
        if (blk < 0) continue;  // warp-uniform: no slot, or a bad one
        dst = (kind == 1 ? a.k_pool : a.v_pool) +
              ((static_cast<size_t>(blk) * a.Hkv + h) * a.block_size + off) * D;
      }
      float x[EPL];
      if constexpr (EPL == 8) {
        unpack8(u[r], x);
      } else {
        bf16x2_to_f32(u[r].x, x[0], x[1]);
        bf16x2_to_f32(u[r].y, x[2], x[3]);
      }
      // ---- RMS norm
      const float* wn = (kind == 0) ? a.q_norm_w : (kind == 1 ? a.k_norm_w : nullptr);
      const bool do_norm = (kind == 2) ? (a.v_norm != 0) : (wn != nullptr);
      if (do_norm) {
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j) ss = fmaf(x[j], x[j], ss);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float rn = rsqrtf(ss / D + a.eps);
        if (wn != nullptr) {
#pragma unroll
          for (int j = 0; j < EPL; ++j) x[j] *= rn * __ldg(wn + lane * EPL + j);
        } else {
#pragma unroll
          for (int j = 0; j < EPL; ++j) x[j] *= rn;
        }
      }
      // ---- rotary embedding (q and k)
      if (kind != 2 && rot) {
        float y[EPL];
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
          const float up = __shfl_sync(0xffffffffu, x[j], (lane + dl) & 31);
          const float dn = __shfl_sync(0xffffffffu, x[j], (lane - dl) & 31);
          const int e = lane * EPL + j;
          y[j] = (e < a.rotary_dim) ? fmaf(x[j], cs[j], (e < half ? up : dn) * sn[j]) : x[j];
        }
#pragma unroll
        for (int j = 0; j < EPL; ++j) x[j] = y[j];
      }
      if constexpr (EPL == 8) {
        *reinterpret_cast<uint4*>(dst + lane * 8) =
            make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                       pack_bf16x2(x[6], x[7]));
      } else {
        *reinterpret_cast<uint2*>(dst + lane * 4) =
            make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_append_rope(const AppendRopeArgs& a, int sm_count, cudaStream_t stream) {
  constexpr int kRB = 6;  // rows per warp
  const int rows = a.Hq * (a.q != nullptr ? 1 : 0) + 2 * a.Hkv;
  const long long items = static_cast<long long>(a.T) * ((rows + kRB - 1) / kRB);
  if (items == 0) return cudaSuccess;
  const long long want = (items + 7) / 8;  // 8 warps per block
  // one wave of 3 blocks per SM: a longer grid-stride loop per warp measured
  // faster than more, shorter-lived blocks
  const long long cap = static_cast<long long>(sm_count > 0 ? sm_count : 1) * 3;
  const int grid = static_cast<int>(want < cap ? want : cap);
  if (a.head_dim == 256)
    kv_append_rope_kernel<256, kRB><<<grid, 256, 0, stream>>>(a);
  else if (a.head_dim == 128)
    kv_append_rope_kernel<128, kRB><<<grid, 256, 0, stream>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace pka
