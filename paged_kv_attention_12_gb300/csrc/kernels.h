// Internal launch interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "paged_attn.h"

namespace pka {

// Arguments of the decode kernel (direct output or split-K partials).
struct DecodeArgs {
  const uint16_t* q;               // bf16 [rows][Hq][D]
  void* out;                       // bf16 [rows][Hq][D] (direct mode)
  float* partial_o;                // fp32 [B][Hq][S][D] (split mode)
  float* partial_lse;              // fp32 [B][Hq][S]    (split mode)
  const uint16_t* k;               // bf16 [num_blocks][Hkv][bs][D]
  const uint16_t* v;
  const int32_t* tables;           // int32 [B][max_blocks]
  const int32_t* seq_lens;         // int32 [B]
  const int32_t* query_start_loc;  // optional: the request's query row is qsl[b+1]-1
  int32_t* err;
  int32_t batch, Hq, Hkv, num_blocks, max_blocks;
  int32_t num_splits;              // items per (request, head); 1 in direct mode
  int32_t split_blocks;            // blocks per split; <= 0: direct mode (whole range)
  int32_t* seg_counters;           // split mode: non-null fuses the combine (zeroed [B*Hkv])
  int32_t direct_slack;            // with seg_counters: > 0 lets a batch whose segments fit one
                                   // per pipeline, none longer than the chunk + this many
                                   // units, stream unsplit (no partials, no merge); 0: never
  float* logits;                   // optional fp32 [B][Hq][max_blocks*bs]: log2-domain logits
  float scale, softcap;
  int32_t window;
  int32_t decode_rows_only;        // nonzero: requests whose query_start_loc span is not
                                   // one token are skipped (no output written for them)
  int32_t total_q, max_query_len;  // with query_start_loc: rows of q / out, longest span
};

cudaError_t launch_key_mass(const float* logits, const float* lse, const int32_t* seq_lens,
                            int32_t B, int32_t Hq, int32_t Hkv, int32_t max_keys, int32_t window,
                            float* key_mass, cudaStream_t stream);

cudaError_t launch_decode(const DecodeArgs& a, int head_dim, int group, int grid,
                          cudaStream_t stream);

struct CombineArgs {
  const float* partial_o;    // [B*Hq][S][D]
  const float* partial_lse;  // [B*Hq][S]
  uint16_t* out;             // bf16 [B*Hq][D]
  float* lse_out;            // [B*Hq] or null
  int32_t rows, num_splits, head_dim;
};

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

struct CheckArgs {
  const int32_t* tables;
  const int32_t* seq_lens;
  int32_t* err;
  int32_t batch, max_blocks, num_blocks, block_size;
};

cudaError_t launch_check_tables(const CheckArgs& a, cudaStream_t stream);

// Prefill / mixed varlen batch.
struct PrefillArgs {
  const uint16_t* q;               // bf16 [total_q][Hq][D]
  uint16_t* out;                   // bf16 [total_q][Hq][D]
  const uint16_t* k;
  const uint16_t* v;
  const int32_t* tables;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;  // [B+1]
  int32_t* err;
  int32_t batch, Hq, Hkv, num_blocks, max_blocks, total_q, max_query_len, max_seq_len;
  float scale, softcap;
  int32_t window;
  int32_t skip_decode_rows;        // nonzero: requests with one query token are left out
  int32_t one_wave;                // prefill CTAs that run at once: when every item fits,
                                   // items go in index order (no ranking) and, with the
                                   // split workspace below, are cut into pieces along keys
  float* split_o;                  // null: no pieces; else fp32 [split_slots][D/4][128][4]
  float* split_lse;                // fp32 [split_slots][128], log2 domain
  int32_t* split_cnt;              // int32 [split_slots], zeroed; left zero by every call
  int32_t split_slots;
};

cudaError_t launch_prefill(const PrefillArgs& a, int head_dim, int group, int sm_count,
                           cudaStream_t stream);

// Mixed batch in one launch: the prefill items of `pa` (skip_decode_rows set)
// on prefill CTAs, the decode rows of `da` (decode_rows_only set, split-K
// with the fused combine) on `decode_ctas` CTAs of two decode pipelines each.
// pairs (D = 256 only, decode_ctas even): the prefill items run on CTA
// pairs instead of one CTA each (pa.one_wave SMs give one_wave / 2 pair
// slots; a piece along keys takes two workspace slots, one per CTA).
// pair_pieces: the pair kernel that may cut its items along keys (else the
// items run whole, whatever their number).
cudaError_t launch_mixed(const PrefillArgs& pa, const DecodeArgs& da, int head_dim, int group,
                         int decode_ctas, bool pairs, bool pair_pieces, cudaStream_t stream);

// Query tokens per 128-row prefill tile (0: unsupported shape).
int mixed_query_tile(int head_dim, int group);

// Append of new tokens' K/V rows into a pool.
struct AppendArgs {
  const uint16_t* k_new;        // bf16 [T][Hkv][D]
  const uint16_t* v_new;
  uint16_t* k_pool;             // bf16 [num_blocks][Hkv][bs][D]
  uint16_t* v_pool;
  const int32_t* slot_mapping;  // [T]: block * bs + offset, < 0: skip
  int32_t* err;
  int32_t T, Hkv, head_dim, block_size, num_blocks;
};

cudaError_t launch_kv_append(const AppendArgs& a, int sm_count, cudaStream_t stream);

// Append with RMS norm and rotary embedding fused in.
struct AppendRopeArgs {
  uint16_t* q;                  // bf16 [T][Hq][D], normalised and rotated in place (or null)
  const uint16_t* k_new;        // bf16 [T][Hkv][D]
  const uint16_t* v_new;
  uint16_t* k_pool;             // bf16 [num_blocks][Hkv][bs][D]
  uint16_t* v_pool;
  const int32_t* slot_mapping;  // [T]
  const int32_t* positions;     // [T]: absolute position of token t
  const float* q_norm_w;        // [D] or null: no q norm
  const float* k_norm_w;        // [D] or null: no k norm
  int32_t* err;
  int32_t T, Hq, Hkv, head_dim, block_size, num_blocks;
  int32_t v_norm;               // nonzero: RMS-normalise v (no weight)
  int32_t rotary_dim;           // 0: no rotary embedding
  float eps, rope_theta;
  // freq_i / (2 pi) as a 64-bit fraction, freq_i = rope_theta^(-2i/rotary_dim)
  unsigned long long gfrac[128];
};

cudaError_t launch_kv_append_rope(const AppendRopeArgs& a, int sm_count, cudaStream_t stream);

int device_sm_count();

// The argument checks of paged_decode_attn (host only, nothing launched):
// PKA_OK or the pka_status the entry points return for these arguments.
int check_decode_call(const void* q, const void* out, const pka_kv_pool* kv,
                      const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                      int32_t B, int32_t Hq, int32_t max_seq_len, const pka_attn_params* params);

}  // namespace pka
