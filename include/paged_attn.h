/*
 * paged_attn.h -- C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * The operation is attention read through a block-paged KV cache, as the
 * inference-server pages describe it:
 *   - "Block-paged KV cache with refcounted blocks, window-aware sliding
 *     layers" and "Triton paged decode and prefill kernels reading K/V
 *     through block tables; split-K decode variant" (inference-server README,
 *     engine feature list);
 *   - "Block-paged per-layer KV with refcounted blocks, lazy allocation, and
 *     SDPA gather -- vLLM/PagedAttention layout" (github README, "What's
 *     inside", Paged KV cache row);
 *   - "GQA with QK/V-norm + KV sharing ... softcapping" (github README,
 *     "What's inside", Custom Gemma 4 forward row);
 *   - mixed-batch chunked prefill, "Needs custom attention path" (architecture
 *     page, "Phase status" table).
 *
 * Definitions shared by every entry point
 * ---------------------------------------
 *  B       requests; Hq / Hkv query / KV heads, G = Hq / Hkv in {1,2,4,8};
 *  D       head_dim in {128, 256}; bs = block_size = 16.
 *  KV pool bf16 [num_blocks][Hkv][bs][D] for K and for V (one pool per layer;
 *          "KV sharing" between layers is the same pool passed twice).  Each
 *          (block, head) tile is one contiguous bs*D*2-byte run.
 *  block_tables  int32 [B][max_blocks], device.  Token t of request b is in
 *          block block_tables[b][t / bs], slot t % bs.  Entries at
 *          j >= ceil(seq_len/bs), and entries of blocks that lie wholly
 *          before every query's sliding window, are never dereferenced (they
 *          may be -1 or point at freed blocks).  Shared prefix blocks are the
 *          same id in several rows; the library only reads them.
 *  seq_lens int32 [B], device: context length including the new tokens.
 *  Query i of request b (n_b new tokens) sits at position p = L_b - n_b + i
 *          and sees key t iff t <= p and (window <= 0 or t > p - window).
 *  Logit   s = scale * q.k; if softcap > 0, s = softcap * tanh(s / softcap).
 *  GQA     query head h reads KV head h / G.
 *  Output  softmax(s) . V over the visible keys, fp32 accumulation, stored
 *          bf16 (round to nearest even).  No visible key -> output 0.
 *
 * Ownership and threading: the caller owns every buffer (device memory unless
 * stated); the library allocates nothing, never synchronises, keeps no state
 * between calls except cached device attributes, and launches on the given
 * stream (a cudaStream_t passed as void*; NULL = legacy default stream).
 * Calls are asynchronous and may be captured in CUDA graphs.
 *
 * Errors: every entry point returns a pka_status.  Argument errors are found
 * on the host before any launch (nothing is written).  PKA_ERR_CUDA means a
 * launch failed; read cudaGetLastError() for the cause.  Kernels never fault
 * on a bad table entry: an id outside [0, num_blocks) is replaced by block 0
 * and bit PKA_DEVERR_BAD_TABLE is OR-ed into *params->err (when non-NULL);
 * a bounded wait that runs out sets PKA_DEVERR_TIMEOUT and the CTA returns.
 */
#ifndef PAGED_ATTN_H_
#define PAGED_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKA_OK = 0,
  PKA_ERR_NULL = -1,        /* a required pointer is NULL */
  PKA_ERR_SHAPE = -2,       /* inconsistent sizes (Hq % Hkv, negative sizes, ...) */
  PKA_ERR_ALIGN = -3,       /* q/out/pool pointer not 16-byte aligned */
  PKA_ERR_UNSUPPORTED = -4, /* head_dim, block_size or G outside the supported set */
  PKA_ERR_WORKSPACE = -5,   /* workspace too small (partials, slots or counters) */
  PKA_ERR_BAD_TABLE = -6,   /* (host view of PKA_DEVERR_BAD_TABLE) */
  PKA_ERR_TIMEOUT = -7,     /* (host view of PKA_DEVERR_TIMEOUT) */
  PKA_ERR_CUDA = -8         /* a CUDA runtime call or launch failed */
} pka_status;

/* Bits OR-ed into the optional device error word (pka_attn_params.err). */
#define PKA_DEVERR_BAD_TABLE 1  /* a table id was outside [0, num_blocks) */
#define PKA_DEVERR_TIMEOUT 2    /* a bounded mbarrier wait ran out */
#define PKA_DEVERR_SEQ_LEN 4    /* seq_len beyond max_blocks*bs or the split cover */
#define PKA_DEVERR_QUERY_LOC 8  /* query_start_loc span outside [0, total_q], negative,
                                   or longer than max_query_len (request skipped) */

/* One layer's K/V block pool.  k and v are device pointers, 16-byte aligned,
 * bf16 [num_blocks][num_kv_heads][block_size][head_dim]. */
typedef struct {
  const void* k;
  const void* v;
  int32_t num_blocks;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t head_dim;
} pka_kv_pool;

/* Attention parameters.  scale multiplies q.k and may be any finite value
 * (zero or negative included; NaN or infinite: PKA_ERR_SHAPE); softcap <= 0
 * or +infinity disables the tanh cap (NaN: PKA_ERR_SHAPE); window <= 0 is
 * full (causal) attention, else the W-key sliding window described above.
 * err: optional device int32 the kernels OR error bits into (never cleared by
 * the library). */
typedef struct {
  float scale;
  float softcap;
  int32_t window;
  int32_t* err;
} pka_attn_params;

/* Library version (major*10000 + minor*100 + patch). */
int pka_version(void);

/* Human-readable name of a pka_status (static string). */
const char* pka_status_string(int status);

/* Decode: one query token per request (engine feature list, "Triton paged
 * decode ... kernels reading K/V through block tables").
 * q   bf16 [B][Hq][D], out bf16 [B][Hq][D] (device, 16-byte aligned).
 * One CTA per (request, KV head) streams that request's visible blocks; use
 * the split-K entry points below when B*Hkv is small next to the SM count. */
int paged_decode_attn(const void* q, void* out, const pka_kv_pool* kv,
                      const int32_t* block_tables, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t B, int32_t Hq,
                      int32_t max_seq_len, const pka_attn_params* params,
                      void* stream);

/* Split-K plan (host only, makes no CUDA call): the workspace shape of a
 * split-K launch for requests of at most max_seq_len tokens.
 *   split_blocks (C): the smallest chunk of 16-key tiles one CTA streams;
 *   num_splits (S):   partial slots per (request, query head),
 *                     ceil(T / C) + 1 for T = most visible blocks of a query.
 * sm_count is accepted for compatibility and not needed: the partition
 * adapts to the GPU it runs on. */
int paged_decode_splitk_plan(int32_t B, int32_t Hkv, int32_t max_seq_len,
                             int32_t block_size, int32_t window, int32_t sm_count,
                             int32_t* num_splits, int32_t* split_blocks);

/* Bytes of fp32 partials a split-K launch writes: B*Hq*S*(D+1)*4. */
size_t paged_decode_splitk_workspace_bytes(int32_t B, int32_t Hq, int32_t D,
                                           int32_t num_splits);

/* Split-K decode ("split-K decode variant", engine feature list).
 * Work partition: a segment is one (request, KV head) with n_b visible
 * blocks ("tiles", blocks [jlo_b, jlo_b + n_b), jlo_b = block of the first
 * visible key).  Segments are laid end to end in (request, head) order on a
 * line of work units: a segment with n_b > 0 takes P = 4 units (the fixed
 * cost of one partial) followed by one unit per tile, an empty segment none.
 * The T units of the line are cut into chunks of q = max(C, ceil(T / grid))
 * units, grid = twice the GPU's SM count, and chunk c is streamed by CTA c.
 * The tiles of a segment whose first tile sits at unit A that fall in chunk
 * c form its piece c - floor(A / q), written to that slot: the piece's
 * softmax-normalised partial output partial_o fp32 [B][Hq][S][D] and its
 * natural-log LSE partial_lse fp32 [B][Hq][S].  Slots a segment does not use
 * get LSE -inf (their partial_o is left untouched).  Needs
 * S >= ceil(T_max / C) + 1 for T_max the visible blocks of max_seq_len (else
 * PKA_ERR_WORKSPACE).  The line's arithmetic is 32-bit: PKA_ERR_SHAPE if
 * B * Hkv * (visible blocks of a table row + 4) exceeds 2^30. */
int paged_decode_splitk(const void* q, float* partial_o, float* partial_lse,
                        const pka_kv_pool* kv, const int32_t* block_tables,
                        int32_t max_blocks, const int32_t* seq_lens, int32_t B,
                        int32_t Hq, int32_t max_seq_len, int32_t num_splits,
                        int32_t split_blocks, const pka_attn_params* params,
                        void* stream);

/* Split-K decode with the log-sum-exp combine fused into the same launch
 * (one launch instead of two).  Same partition and partials as
 * paged_decode_splitk with the plan's (S, C); the CTA that finishes a
 * segment's last piece merges its pieces and writes out bf16 [B][Hq][D].
 * Exception: when the B * Hkv segments (request, KV head) number at most
 * the decode pipelines (twice the GPU's SM count) and none has more than
 * q + 24 units on the split's line (q its chunk), every segment streams
 * whole on its own pipeline and writes its output with no partials and no
 * merge -- the result of paged_decode_attn, bit for bit.
 * workspace: device, 16-byte aligned, at least paged_decode_attn_ws_bytes()
 * bytes: partial outputs fp32 [B][Hq][S][D], partial LSEs [B][Hq][S] (padded
 * to 16 bytes), then B*Hkv int32 arrival counters.  The counters must be
 * zero before the first call (e.g. memset once at allocation); every call
 * that completes leaves them zero again.  After a call that reported
 * PKA_DEVERR_TIMEOUT, zero them before the next call.  Calls sharing one
 * workspace must not overlap on the GPU.  PKA_ERR_SHAPE if
 * B * Hkv * (visible blocks of a table row + 4) exceeds 2^30. */
size_t paged_decode_attn_ws_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                  int32_t max_seq_len, int32_t window);
int paged_decode_attn_ws(const void* q, void* out, const pka_kv_pool* kv,
                         const int32_t* block_tables, int32_t max_blocks,
                         const int32_t* seq_lens, int32_t B, int32_t Hq,
                         int32_t max_seq_len, const pka_attn_params* params,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Log-sum-exp merge of split partials (the merge a split-K softmax needs):
 * M = max_s LSE_s, w_s = exp(LSE_s - M),
 * out = sum_s w_s*O_s / sum_s w_s (bf16 [B][Hq][D]),
 * lse_out = M + ln sum_s w_s (fp32 [B][Hq], may be NULL).
 * Slots with LSE -inf are skipped without reading their partial_o. */
int paged_decode_splitk_combine(const float* partial_o, const float* partial_lse,
                                int32_t B, int32_t Hq, int32_t D, int32_t num_splits,
                                void* out, float* lse_out, void* stream);

/* Prefill / mixed batch ("Prefill in three modes: monolithic, chunked ...,
 * batched", engine feature list; mixed-batch chunked prefill, architecture
 * page "Phase status").  Varlen: request b owns query rows
 * [query_start_loc[b], query_start_loc[b+1]) of q bf16 [total_q][Hq][D]; rows
 * with one token (decode) and chunks of many tokens may be mixed in one
 * launch.  Causal over cached prefix + chunk.  out bf16 [total_q][Hq][D].
 * max_query_len / max_seq_len are host upper bounds.  query_start_loc is
 * device data: a request whose span is not 0 <= query_start_loc[b] <=
 * query_start_loc[b+1] <= total_q, or is longer than max_query_len, is
 * skipped (its rows are not written) and PKA_DEVERR_QUERY_LOC is OR-ed into
 * the error word; nothing outside out's total_q rows is ever written. */
int paged_prefill_attn(const void* q, void* out, const pka_kv_pool* kv,
                       const int32_t* block_tables, int32_t max_blocks,
                       const int32_t* query_start_loc, const int32_t* seq_lens,
                       int32_t B, int32_t Hq, int32_t total_q, int32_t max_query_len,
                       int32_t max_seq_len, const pka_attn_params* params,
                       void* stream);

/* Mixed batch in one launch with a workspace (mixed-batch chunked prefill,
 * architecture page "Phase status"): same arguments, result and errors as
 * paged_prefill_attn, but requests with exactly one query token (decode rows)
 * go to decode pipelines in the same launch -- split-K over their keys with
 * the log-sum-exp merge fused in, as paged_decode_attn_ws -- instead of
 * filling G of the 128 rows of a tensor-core tile; requests with more tokens
 * run the tensor-core prefill pipeline.  Exception: when the decode rows'
 * B * Hkv segments (request, KV head) number at most the decode pipelines
 * and none has more than q + 24 units on the split's line (q its chunk,
 * the paged_decode_splitk partition over the decode pipelines), every
 * segment streams whole on its own pipeline and writes its output with no
 * partials and no merge.
 * SMs: the prefill side gets P of the GPU's N SMs, the decode pipelines the
 * rest (two per SM).  P shares N in proportion to estimated SM time, from
 * sizes only: prefill E = ceil((total_q - B) / TQ) * Hkv items (TQ = 128/G
 * query tokens per tile) of ceil(K / BN) + 1 key tiles each at 2 us, with
 * K = min(max_seq_len, window + TQ) (max_seq_len without window) and BN = 64
 * at D = 256, 128 at D = 128; decode max(0, B - ceil((total_q - B) /
 * (max_query_len - 1))) rows of Hkv * ceil(K' / 16) blocks at 64 * D bytes
 * per block and 70 GB/s per SM, K' = min(max_seq_len, window).  With
 * share = round(N * prefill / (prefill + decode)), P = share if share >= 2E,
 * else E; then clamped to [1, N - N/4] (P = 0 without prefill rows).
 * Prefill items: one per (request, query tile, KV head) with work, on one
 * CTA each at D = 128; at D = 256 on CTA pairs, two query tiles per pair of
 * SMs, as in paged_prefill_attn (the decode CTAs then number N - P rounded
 * down to even, and the P SMs give S = P / 2 pair slots and 80 piece slots;
 * else S = P slots and 160 piece slots).  When the items are fewer than S
 * (and at most the piece slots; at D = 256 only when also the estimate
 * ceil((total_q - B) / (2 TQ)) * Hkv is below S and at most 80), they are
 * cut along their keys: with theta
 * the smallest piece length >= 4 key tiles for which sum over items of
 * min(8, ceil(tiles / theta)) <= min(S, piece slots), an item of T key
 * tiles runs as p = min(8, ceil(T / theta)) pieces on separate CTAs (CTA
 * pairs), piece k taking tiles [k T / p, (k + 1) T / p); each piece leaves
 * its normalised rows and their LSEs in the workspace (a CTA pair: each CTA
 * its 128 rows in a slot of its own) and the piece that arrives last on the
 * item's counter (at D = 256, each CTA's rows have their own) merges them
 * in piece order (the same result whichever piece merges).
 * workspace: device, 16-byte aligned, at least paged_prefill_attn_ws_bytes()
 * bytes: the layout of paged_decode_attn_ws for B requests, then 160 piece
 * slots of 128 fp32 rows of D columns, their 160 * 128 fp32 LSEs and 160
 * int32 piece counters (padded to 16 bytes).  All counters must be zero
 * before the first call and are left zero by every call that completes
 * (zero them again after a PKA_DEVERR_TIMEOUT).  Calls sharing one
 * workspace must not overlap on the GPU.  PKA_ERR_WORKSPACE if
 * workspace_bytes is too small. */
size_t paged_prefill_attn_ws_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                   int32_t max_seq_len, int32_t window);
int paged_prefill_attn_ws(const void* q, void* out, const pka_kv_pool* kv,
                          const int32_t* block_tables, int32_t max_blocks,
                          const int32_t* query_start_loc, const int32_t* seq_lens,
                          int32_t B, int32_t Hq, int32_t total_q, int32_t max_query_len,
                          int32_t max_seq_len, const pka_attn_params* params,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Checked mode: validates, on the device, every table entry a call would
 * dereference (j < ceil(seq_len/bs)) against [0, num_blocks), and seq_len
 * against [0, max_blocks*bs]; OR-s PKA_DEVERR_* bits into *err (device int32,
 * required).  Reads only the tables and seq_lens. */
int paged_attn_check_tables(const int32_t* block_tables, int32_t max_blocks,
                            const int32_t* seq_lens, int32_t B, int32_t num_blocks,
                            int32_t block_size, int32_t* err, void* stream);

/* Self-test of the bounded waits.  Launches one CTA whose thread waits, with
 * the wait routine of every kernel in this library, on an mbarrier phase
 * that nothing completes, for budget_cycles SM clock cycles (1 ..
 * 2e9; the kernels' own budget is 2e9, about a second).  The wait runs out,
 * PKA_DEVERR_TIMEOUT is OR-ed into *err (device int32, required) and the
 * kernel returns: a stalled pipeline ends with an error status and a usable
 * context instead of a hang.  PKA_ERR_NULL / PKA_ERR_SHAPE on bad arguments. */
int pka_selftest_bounded_wait(int32_t* err, int64_t budget_cycles, void* stream);

/* H2O attention mass.  The engine's cache offers an H2O eviction policy
 * ("Eviction policies -- Pluggable per-session: LRU, AttentionSink, H2O",
 * github README, "What's inside"; "H2O wiring deferred", architecture page,
 * "Phase status"), which keeps the keys that have drawn the most attention.
 * Two calls give what it needs from a decode step:
 *
 * paged_decode_splitk_logits: paged_decode_splitk that also stores every
 *   visible key's logit: logits fp32 [B][Hq][max_blocks*16] (device, caller
 *   owned), entry [b][h][t] = log2(e) * s_h(t) (s after scale and softcap)
 *   for the keys t query head h of request b sees; other entries are not
 *   written.  Arguments and errors otherwise as paged_decode_splitk.
 * paged_decode_key_mass: after paged_decode_splitk_combine with lse_out
 *   (natural-log LSE [B][Hq]), adds each visible key's attention probability,
 *   summed over the G query heads of its KV head, to key_mass fp32
 *   [B][Hkv][max_blocks*16] (device): key_mass[b][kvh][t] += sum_h
 *   exp(s_h(t) - LSE_h).  Invisible keys are left as they are; a head with
 *   LSE = -inf adds nothing.  Over the visible keys of one (b, kvh) the
 *   added mass sums to G. */
int paged_decode_splitk_logits(const void* q, float* partial_o, float* partial_lse,
                               float* logits, const pka_kv_pool* kv,
                               const int32_t* block_tables, int32_t max_blocks,
                               const int32_t* seq_lens, int32_t B, int32_t Hq,
                               int32_t max_seq_len, int32_t num_splits, int32_t split_blocks,
                               const pka_attn_params* params, void* stream);
int paged_decode_key_mass(const float* logits, const float* lse, const int32_t* seq_lens,
                          int32_t B, int32_t Hq, int32_t num_kv_heads, int32_t max_blocks,
                          int32_t block_size, int32_t window, float* key_mass, void* stream);

/* Append the new tokens' K and V rows to a pool: the cache write that comes
 * before attention on every tick ("Block-paged per-layer KV with refcounted
 * blocks, lazy allocation, and SDPA gather -- vLLM/PagedAttention layout",
 * github README, "What's inside", Paged KV cache row; one new token per
 * active request per tick, architecture page, "How a single request flows
 * through the system", step 7).
 *   k_new, v_new  bf16 [T][Hkv][D], device, contiguous, 16-byte aligned.
 *   k_pool, v_pool  bf16 [num_blocks][Hkv][block_size][D], device, written.
 *   slot_mapping  int32 [T], device: token t goes to slot s = slot_mapping[t]
 *                 = block * block_size + offset, for every KV head; s < 0
 *                 skips the token (padding).  Slots must be distinct (with a
 *                 repeated slot, which token's row lands there is undefined).
 *   err           optional device int32: a slot beyond num_blocks *
 *                 block_size is skipped and ORs PKA_DEVERR_BAD_TABLE into it.
 * Bit-exact copy; T = 0 is a no-op.  D in {128, 256}, block_size 16. */
int paged_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                    int32_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                    int32_t head_dim, const int32_t* slot_mapping, int32_t T, int32_t* err,
                    void* stream);

/* paged_kv_append with the per-head math before attention fused in
 * ("Custom Gemma 4 forward -- Dual-RoPE, GQA with QK/V-norm + KV sharing",
 * github README, "What's inside").  For each token t (position positions[t],
 * slot slot_mapping[t] as in paged_kv_append), in this order:
 *   RMS norm   x <- x / sqrt(mean_c(x_c^2) + eps) * w_c over the D channels of
 *              each head: q with q_norm_weight, k with k_norm_weight (fp32 [D],
 *              device; NULL = no norm for that tensor), v with unit weight when
 *              v_norm != 0;
 *   RoPE       q and k, rotate-half form: with r = rotary_dim and
 *              a_i = positions[t] * rope_theta^(-2i/r), for i < r/2:
 *              (x_i, x_{i+r/2}) <- (x_i cos a_i - x_{i+r/2} sin a_i,
 *                                   x_{i+r/2} cos a_i + x_i sin a_i);
 *              channels >= r unchanged; rotary_dim = 0 turns it off (the two
 *              RoPE variants of a dual scheme are two calls).
 * Then k and v rows go to the pool slots and q (bf16 [T][Hq][D], may be NULL)
 * is overwritten in place; everything is computed in fp32 from the bf16
 * inputs and stored bf16 (round to nearest even).
 * rotary_dim in [0, D], a multiple of 16; rope_theta > 1 when rotary_dim > 0;
 * eps >= 0.  Errors as paged_kv_append. */
int paged_kv_append_rope(void* q, const void* k_new, const void* v_new, void* k_pool,
                         void* v_pool, int32_t num_blocks, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t block_size, int32_t head_dim,
                         const int32_t* slot_mapping, const int32_t* positions, int32_t T,
                         const float* q_norm_weight, const float* k_norm_weight, int32_t v_norm,
                         float eps, float rope_theta, int32_t rotary_dim, int32_t* err,
                         void* stream);

/* Decode for callers that cannot allocate device memory.  The pages have no
 * counterpart: this is a service of this library.  Some callers cannot call
 * cudaMalloc -- a plugin running while another allocator owns all device
 * memory, code in a region where allocation calls are not allowed -- yet
 * split-K decode needs room for its fp32 partials.  This entry point gives
 * the same result as paged_decode_splitk_plan + paged_decode_splitk +
 * paged_decode_splitk_combine, with the partials in a 16 MiB array compiled
 * into the library, so it allocates nothing; q, out and the pool are the
 * caller's, as for paged_decode_attn.
 * Limit: B*Hq*S*(D+1)*4 bytes <= 16 MiB for the S paged_decode_splitk_plan
 * gives; larger calls return PKA_ERR_WORKSPACE before launching anything.
 * The first call on each device looks up the array's device address (make
 * that first call before any stream capture) and keeps it for the life of
 * the process: after cudaDeviceReset the library's module is loaded again at
 * another address, so a process that resets a device must not call this
 * entry point on that device afterwards.  Every GPU that loads the
 * library holds the array until the process exits.  All calls share the one
 * array: calls that overlap on the GPU (other streams, other threads) race
 * and must be serialised by the caller. */
int paged_decode_attn_noalloc(const void* q, void* out, const pka_kv_pool* kv,
                              const int32_t* block_tables, int32_t max_blocks,
                              const int32_t* seq_lens, int32_t B, int32_t Hq,
                              int32_t max_seq_len, const pka_attn_params* params,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_ATTN_H_ */
