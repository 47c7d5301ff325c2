// C-ABI layer: argument validation, split-K planning and kernel dispatch.
//
// Every argument error is found here, on the host, before anything is
// launched; the kernels themselves only guard against data-dependent faults
// (table ids, sequence lengths) and report those through the device error
// word.  Nothing here allocates or synchronises.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <stdint.h>

#include "kernels.h"
#include "paged_attn.h"

namespace {

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dim(int d) { return d == 128 || d == 256; }
bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

// Largest number of blocks a decode query's visible keys can span.
int max_visible_blocks(int max_seq_len, int window, int bs) {
  if (max_seq_len <= 0) return 0;
  const int full = (max_seq_len + bs - 1) / bs;
  if (window <= 0) return full;
  const int win = (window - 1) / bs + 2;
  return full < win ? full : win;
}

// The split-K work line (Hkv * sum over requests of (visible blocks + 4)
// units) fits in 31 bits with room to spare, so the kernels' partition
// arithmetic is 32-bit.
// (The kernels clamp a sequence to its table row, so a row's max_blocks
// bounds its visible blocks whatever the device lengths are.)
bool line_fits(int32_t B, int32_t Hkv, int32_t max_blocks, int32_t window) {
  int64_t per = max_blocks;
  if (window > 0) per = std::min<int64_t>(per, (window - 1) / 16 + 2);
  return static_cast<int64_t>(B) * Hkv * (per + 4) <= (int64_t(1) << 30);
}

int check_pool(const pka_kv_pool* kv, int Hq) {
  if (kv == nullptr || kv->k == nullptr || kv->v == nullptr) return PKA_ERR_NULL;
  if (kv->num_blocks <= 0 || kv->num_kv_heads <= 0 || Hq <= 0) return PKA_ERR_SHAPE;
  if (Hq % kv->num_kv_heads != 0) return PKA_ERR_SHAPE;
  if (kv->block_size != 16) return PKA_ERR_UNSUPPORTED;
  if (!supported_dim(kv->head_dim)) return PKA_ERR_UNSUPPORTED;
  if (!supported_group(Hq / kv->num_kv_heads)) return PKA_ERR_UNSUPPORTED;
  if (!aligned16(kv->k) || !aligned16(kv->v)) return PKA_ERR_ALIGN;
  return PKA_OK;
}

int check_common(const void* q, const pka_kv_pool* kv, const int32_t* block_tables,
                 int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t Hq,
                 int32_t max_seq_len, const pka_attn_params* params) {
  if (q == nullptr || block_tables == nullptr || seq_lens == nullptr || params == nullptr)
    return PKA_ERR_NULL;
  const int st = check_pool(kv, Hq);
  if (st != PKA_OK) return st;
  if (B < 0 || max_blocks <= 0 || max_seq_len < 0) return PKA_ERR_SHAPE;
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks) * kv->block_size)
    return PKA_ERR_SHAPE;
  if (!std::isfinite(params->scale) || std::isnan(params->softcap))
    return PKA_ERR_SHAPE;  // NaN or infinite scale, NaN cap
  if (!aligned16(q)) return PKA_ERR_ALIGN;
  return PKA_OK;
}

pka::DecodeArgs decode_args(const void* q, const pka_kv_pool* kv, const int32_t* block_tables,
                            int32_t max_blocks, const int32_t* seq_lens, int32_t B, int32_t Hq,
                            const pka_attn_params* p) {
  pka::DecodeArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(kv->k);
  a.v = static_cast<const uint16_t*>(kv->v);
  a.tables = block_tables;
  a.seq_lens = seq_lens;
  a.query_start_loc = nullptr;
  a.err = p->err;
  a.batch = B;
  a.Hq = Hq;
  a.Hkv = kv->num_kv_heads;
  a.num_blocks = kv->num_blocks;
  a.max_blocks = max_blocks;
  a.scale = p->scale;
  a.softcap = std::isinf(p->softcap) ? 0.f : p->softcap;  // an infinite cap is no cap
  a.window = p->window;
  return a;
}

}  // namespace

namespace pka {

int check_decode_call(const void* q, const void* out, const pka_kv_pool* kv,
                      const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                      int32_t B, int32_t Hq, int32_t max_seq_len, const pka_attn_params* params) {
  if (out == nullptr) return PKA_ERR_NULL;
  const int st =
      check_common(q, kv, block_tables, max_blocks, seq_lens, B, Hq, max_seq_len, params);
  if (st != PKA_OK) return st;
  return aligned16(out) ? PKA_OK : PKA_ERR_ALIGN;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev] = n;
  return n;
}

}  // namespace pka

extern "C" {

int pka_version(void) { return 100; }

const char* pka_status_string(int status) {
  switch (status) {
    case PKA_OK: return "ok";
    case PKA_ERR_NULL: return "null pointer argument";
    case PKA_ERR_SHAPE: return "inconsistent sizes";
    case PKA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case PKA_ERR_UNSUPPORTED: return "unsupported head_dim, block_size or GQA group";
    case PKA_ERR_WORKSPACE:
      return "split-K workspace too small (partials or slots for max_seq_len)";
    case PKA_ERR_BAD_TABLE: return "block table id out of range";
    case PKA_ERR_TIMEOUT: return "bounded device wait timed out";
    case PKA_ERR_CUDA: return "CUDA launch or runtime error";
    default: return "unknown status";
  }
}

int paged_decode_attn(const void* q, void* out, const pka_kv_pool* kv,
                      const int32_t* block_tables, int32_t max_blocks,
                      const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t max_seq_len,
                      const pka_attn_params* params, void* stream) {
  if (out == nullptr) return PKA_ERR_NULL;
  int st = check_common(q, kv, block_tables, max_blocks, seq_lens, B, Hq, max_seq_len, params);
  if (st != PKA_OK) return st;
  if (!aligned16(out)) return PKA_ERR_ALIGN;
  if (B == 0) return PKA_OK;
  pka::DecodeArgs a = decode_args(q, kv, block_tables, max_blocks, seq_lens, B, Hq, params);
  a.out = out;
  a.num_splits = 1;
  a.split_blocks = 0;
  const int items = B * kv->num_kv_heads;
  const int sms = pka::device_sm_count();
  if (sms <= 0) return PKA_ERR_CUDA;
  // launch_decode runs two CTAs per unit of grid
  const int grid = items < 2 * sms ? (items + 1) / 2 : sms;
  cudaError_t e = pka::launch_decode(a, kv->head_dim, Hq / kv->num_kv_heads, grid,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

int paged_decode_splitk_plan(int32_t B, int32_t Hkv, int32_t max_seq_len, int32_t block_size,
                             int32_t window, int32_t sm_count, int32_t* num_splits,
                             int32_t* split_blocks) {
  if (num_splits == nullptr || split_blocks == nullptr) return PKA_ERR_NULL;
  if (B <= 0 || Hkv <= 0 || max_seq_len < 0 || block_size <= 0) return PKA_ERR_SHAPE;
  (void)sm_count;  // the partition adapts to the SM count on the device
  const int T = max_visible_blocks(max_seq_len, window, block_size);
  if (T <= 0) {
    *num_splits = 1;
    *split_blocks = 1;
    return PKA_OK;
  }
  // Minimum chunk: at least four tiles, and long enough that one segment
  // never spans more than 33 slots (bounded workspace).
  int C = (T + 31) / 32;
  if (C < 4) C = 4;
  *split_blocks = C;
  *num_splits = (T + C - 1) / C + 1;
  return PKA_OK;
}

size_t paged_decode_splitk_workspace_bytes(int32_t B, int32_t Hq, int32_t D, int32_t num_splits) {
  if (B <= 0 || Hq <= 0 || D <= 0 || num_splits <= 0) return 0;
  return static_cast<size_t>(B) * Hq * num_splits * (static_cast<size_t>(D) + 1) * sizeof(float);
}

namespace {

int splitk_impl(const void* q, float* partial_o, float* partial_lse, float* logits,
                const pka_kv_pool* kv, const int32_t* block_tables, int32_t max_blocks,
                const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t max_seq_len,
                int32_t num_splits, int32_t split_blocks, const pka_attn_params* params,
                void* stream) {
  if (partial_o == nullptr || partial_lse == nullptr) return PKA_ERR_NULL;
  int st = check_common(q, kv, block_tables, max_blocks, seq_lens, B, Hq, max_seq_len, params);
  if (st != PKA_OK) return st;
  if (num_splits <= 0 || split_blocks <= 0) return PKA_ERR_SHAPE;
  if (!aligned16(partial_o)) return PKA_ERR_ALIGN;
  // a segment of up to T tiles spans at most ceil(T / split_blocks) + 1 chunks
  const int T = max_visible_blocks(max_seq_len, params->window, kv->block_size);
  if (T > 0 && static_cast<int64_t>(num_splits) < (T + split_blocks - 1) / split_blocks + 1)
    return PKA_ERR_WORKSPACE;
  if (B == 0) return PKA_OK;
  pka::DecodeArgs a = decode_args(q, kv, block_tables, max_blocks, seq_lens, B, Hq, params);
  a.partial_o = partial_o;
  a.partial_lse = partial_lse;
  a.num_splits = num_splits;
  a.split_blocks = split_blocks;
  a.logits = logits;
  if (static_cast<int64_t>(B) * Hq * num_splits > 0x7fffffffLL) return PKA_ERR_SHAPE;
  if (!line_fits(B, kv->num_kv_heads, max_blocks, params->window)) return PKA_ERR_SHAPE;
  const int sms = pka::device_sm_count();
  if (sms <= 0) return PKA_ERR_CUDA;
  // persistent: one CTA per SM, each streaming an equal share of the tiles
  const int grid = sms;
  cudaError_t e = pka::launch_decode(a, kv->head_dim, Hq / kv->num_kv_heads, grid,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

}  // namespace

int paged_decode_splitk(const void* q, float* partial_o, float* partial_lse,
                        const pka_kv_pool* kv, const int32_t* block_tables, int32_t max_blocks,
                        const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t max_seq_len,
                        int32_t num_splits, int32_t split_blocks,
                        const pka_attn_params* params, void* stream) {
  return splitk_impl(q, partial_o, partial_lse, nullptr, kv, block_tables, max_blocks, seq_lens,
                     B, Hq, max_seq_len, num_splits, split_blocks, params, stream);
}

int paged_decode_splitk_logits(const void* q, float* partial_o, float* partial_lse,
                               float* logits, const pka_kv_pool* kv,
                               const int32_t* block_tables, int32_t max_blocks,
                               const int32_t* seq_lens, int32_t B, int32_t Hq,
                               int32_t max_seq_len, int32_t num_splits, int32_t split_blocks,
                               const pka_attn_params* params, void* stream) {
  if (logits == nullptr) return PKA_ERR_NULL;
  if (static_cast<int64_t>(B) * Hq * max_blocks * 16 > (1LL << 40)) return PKA_ERR_SHAPE;
  return splitk_impl(q, partial_o, partial_lse, logits, kv, block_tables, max_blocks, seq_lens,
                     B, Hq, max_seq_len, num_splits, split_blocks, params, stream);
}

int paged_decode_key_mass(const float* logits, const float* lse, const int32_t* seq_lens,
                          int32_t B, int32_t Hq, int32_t num_kv_heads, int32_t max_blocks,
                          int32_t block_size, int32_t window, float* key_mass, void* stream) {
  if (B < 0 || Hq <= 0 || num_kv_heads <= 0 || max_blocks <= 0) return PKA_ERR_SHAPE;
  if (Hq % num_kv_heads != 0 || !supported_group(Hq / num_kv_heads)) return PKA_ERR_SHAPE;
  if (block_size != 16) return PKA_ERR_UNSUPPORTED;
  if (B == 0) return PKA_OK;
  if (logits == nullptr || lse == nullptr || seq_lens == nullptr || key_mass == nullptr)
    return PKA_ERR_NULL;
  const cudaError_t e =
      pka::launch_key_mass(logits, lse, seq_lens, B, Hq, num_kv_heads, max_blocks * block_size,
                           window, key_mass, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

// Workspace of the fused split-K decode: partial outputs, partial LSEs, then
// one arrival counter per (request, KV head).
struct FusedLayout {
  int32_t S, C;
  size_t o_bytes, lse_bytes, cnt_bytes;
  size_t total() const { return o_bytes + lse_bytes + cnt_bytes; }
};

int fused_layout(int32_t B, int32_t Hq, int32_t Hkv, int32_t D, int32_t max_seq_len,
                 int32_t window, FusedLayout* L) {
  int st = paged_decode_splitk_plan(B, Hkv, max_seq_len, 16, window, 0, &L->S, &L->C);
  if (st != PKA_OK) return st;
  L->o_bytes = static_cast<size_t>(B) * Hq * L->S * D * sizeof(float);
  L->lse_bytes = (static_cast<size_t>(B) * Hq * L->S * sizeof(float) + 15) / 16 * 16;
  L->cnt_bytes = (static_cast<size_t>(B) * Hkv * sizeof(int32_t) + 15) / 16 * 16;
  return PKA_OK;
}

size_t paged_decode_attn_ws_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                  int32_t max_seq_len, int32_t window) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return 0;
  FusedLayout L;
  if (fused_layout(B, Hq, Hkv, D, max_seq_len, window, &L) != PKA_OK) return 0;
  return L.total();
}

// With the combine fused in, a batch whose (request, KV head) segments fit
// one per decode pipeline and are at most this many work units beyond the
// split's chunk streams unsplit (no partials, no merge; the merge costs
// about as much as streaming a couple of dozen tiles).  Measured: a batch
// of 64 rows that all see a full 1024-key window beside prefill chunks,
// 47 us per launch this way against 51 us split and merged; 4 rows of up to
// 256 tokens, 8.7 us against 10.0 us.
constexpr int32_t kDirectSlackUnits = 24;

int paged_decode_attn_ws(const void* q, void* out, const pka_kv_pool* kv,
                         const int32_t* block_tables, int32_t max_blocks,
                         const int32_t* seq_lens, int32_t B, int32_t Hq, int32_t max_seq_len,
                         const pka_attn_params* params, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (out == nullptr || workspace == nullptr) return PKA_ERR_NULL;
  int st = check_common(q, kv, block_tables, max_blocks, seq_lens, B, Hq, max_seq_len, params);
  if (st != PKA_OK) return st;
  if (!aligned16(out) || !aligned16(workspace)) return PKA_ERR_ALIGN;
  if (B == 0) return PKA_OK;
  FusedLayout L;
  st = fused_layout(B, Hq, kv->num_kv_heads, kv->head_dim, max_seq_len, params->window, &L);
  if (st != PKA_OK) return st;
  if (workspace_bytes < L.total()) return PKA_ERR_WORKSPACE;
  if (!line_fits(B, kv->num_kv_heads, max_blocks, params->window)) return PKA_ERR_SHAPE;
  pka::DecodeArgs a = decode_args(q, kv, block_tables, max_blocks, seq_lens, B, Hq, params);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.out = out;
  a.partial_o = reinterpret_cast<float*>(ws);
  a.partial_lse = reinterpret_cast<float*>(ws + L.o_bytes);
  a.seg_counters = reinterpret_cast<int32_t*>(ws + L.o_bytes + L.lse_bytes);
  a.num_splits = L.S;
  a.split_blocks = L.C;
  a.direct_slack = kDirectSlackUnits;
  const int sms = pka::device_sm_count();
  if (sms <= 0) return PKA_ERR_CUDA;
  cudaError_t e = pka::launch_decode(a, kv->head_dim, Hq / kv->num_kv_heads, sms,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

int paged_decode_splitk_combine(const float* partial_o, const float* partial_lse, int32_t B,
                                int32_t Hq, int32_t D, int32_t num_splits, void* out,
                                float* lse_out, void* stream) {
  if (partial_o == nullptr || partial_lse == nullptr || out == nullptr) return PKA_ERR_NULL;
  if (B < 0 || Hq <= 0 || num_splits <= 0) return PKA_ERR_SHAPE;
  if (!supported_dim(D)) return PKA_ERR_UNSUPPORTED;
  if (!aligned16(partial_o) || !aligned16(out)) return PKA_ERR_ALIGN;
  if (B == 0) return PKA_OK;
  pka::CombineArgs a{};
  a.partial_o = partial_o;
  a.partial_lse = partial_lse;
  a.out = static_cast<uint16_t*>(out);
  a.lse_out = lse_out;
  a.rows = B * Hq;
  a.num_splits = num_splits;
  a.head_dim = D;
  cudaError_t e = pka::launch_combine(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

namespace {

pka::PrefillArgs prefill_args(const void* q, void* out, const pka_kv_pool* kv,
                              const int32_t* block_tables, int32_t max_blocks,
                              const int32_t* query_start_loc, const int32_t* seq_lens, int32_t B,
                              int32_t Hq, int32_t total_q, int32_t max_query_len,
                              int32_t max_seq_len, const pka_attn_params* params) {
  pka::PrefillArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.out = static_cast<uint16_t*>(out);
  a.k = static_cast<const uint16_t*>(kv->k);
  a.v = static_cast<const uint16_t*>(kv->v);
  a.tables = block_tables;
  a.seq_lens = seq_lens;
  a.query_start_loc = query_start_loc;
  a.err = params->err;
  a.batch = B;
  a.Hq = Hq;
  a.Hkv = kv->num_kv_heads;
  a.num_blocks = kv->num_blocks;
  a.max_blocks = max_blocks;
  a.total_q = total_q;
  a.max_query_len = max_query_len;
  a.max_seq_len = max_seq_len;
  a.scale = params->scale;
  a.softcap = std::isinf(params->softcap) ? 0.f : params->softcap;
  a.window = params->window;
  return a;
}

int check_prefill(const void* q, void* out, const pka_kv_pool* kv, const int32_t* block_tables,
                  int32_t max_blocks, const int32_t* query_start_loc, const int32_t* seq_lens,
                  int32_t B, int32_t Hq, int32_t total_q, int32_t max_query_len,
                  int32_t max_seq_len, const pka_attn_params* params) {
  if (out == nullptr || query_start_loc == nullptr) return PKA_ERR_NULL;
  int st = check_common(q, kv, block_tables, max_blocks, seq_lens, B, Hq, max_seq_len, params);
  if (st != PKA_OK) return st;
  if (total_q < 0 || max_query_len < 0 || max_query_len > max_seq_len) return PKA_ERR_SHAPE;
  if (!aligned16(out)) return PKA_ERR_ALIGN;
  return PKA_OK;
}

}  // namespace

int paged_prefill_attn(const void* q, void* out, const pka_kv_pool* kv,
                       const int32_t* block_tables, int32_t max_blocks,
                       const int32_t* query_start_loc, const int32_t* seq_lens, int32_t B,
                       int32_t Hq, int32_t total_q, int32_t max_query_len, int32_t max_seq_len,
                       const pka_attn_params* params, void* stream) {
  int st = check_prefill(q, out, kv, block_tables, max_blocks, query_start_loc, seq_lens, B, Hq,
                         total_q, max_query_len, max_seq_len, params);
  if (st != PKA_OK) return st;
  if (B == 0 || total_q == 0) return PKA_OK;
  const pka::PrefillArgs a = prefill_args(q, out, kv, block_tables, max_blocks, query_start_loc,
                                          seq_lens, B, Hq, total_q, max_query_len, max_seq_len,
                                          params);
  const int sms = pka::device_sm_count();
  if (sms <= 0) return PKA_ERR_CUDA;
  pka::PrefillArgs a1 = a;
  a1.one_wave = sms;  // one prefill CTA per SM
  cudaError_t e = pka::launch_prefill(a1, kv->head_dim, Hq / kv->num_kv_heads, sms,
                                      static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PKA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

// The prefill part of the mixed launch's workspace: kPrefillSplitSlots
// pieces of 128 rows (fp32 rows, then their LSEs), then one counter each.
constexpr int32_t kPrefillSplitSlots = 160;

size_t prefill_split_bytes(int32_t D) {
  const size_t o = static_cast<size_t>(kPrefillSplitSlots) * 128 * D * sizeof(float);
  const size_t lse = static_cast<size_t>(kPrefillSplitSlots) * 128 * sizeof(float);
  const size_t cnt = (static_cast<size_t>(kPrefillSplitSlots) * sizeof(int32_t) + 15) / 16 * 16;
  return o + lse + cnt;
}

size_t paged_prefill_attn_ws_bytes(int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                   int32_t max_seq_len, int32_t window) {
  const size_t dec = paged_decode_attn_ws_bytes(B, Hq, Hkv, D, max_seq_len, window);
  if (dec == 0) return 0;
  return dec + prefill_split_bytes(D);
}

int paged_prefill_attn_ws(const void* q, void* out, const pka_kv_pool* kv,
                          const int32_t* block_tables, int32_t max_blocks,
                          const int32_t* query_start_loc, const int32_t* seq_lens, int32_t B,
                          int32_t Hq, int32_t total_q, int32_t max_query_len,
                          int32_t max_seq_len, const pka_attn_params* params, void* workspace,
                          size_t workspace_bytes, void* stream) {
  int st = check_prefill(q, out, kv, block_tables, max_blocks, query_start_loc, seq_lens, B, Hq,
                         total_q, max_query_len, max_seq_len, params);
  if (st != PKA_OK) return st;
  if (workspace == nullptr) return PKA_ERR_NULL;
  if (!aligned16(workspace)) return PKA_ERR_ALIGN;
  if (B == 0 || total_q == 0) return PKA_OK;
  const int D = kv->head_dim, Hkv = kv->num_kv_heads, G = Hq / Hkv;
  FusedLayout L;
  st = fused_layout(B, Hq, Hkv, D, max_seq_len, params->window, &L);
  if (st != PKA_OK) return st;
  if (workspace_bytes < L.total() + prefill_split_bytes(D)) return PKA_ERR_WORKSPACE;
  if (!line_fits(B, Hkv, max_blocks, params->window)) return PKA_ERR_SHAPE;
  pka::PrefillArgs pa = prefill_args(q, out, kv, block_tables, max_blocks, query_start_loc,
                                     seq_lens, B, Hq, total_q, max_query_len, max_seq_len, params);
  pa.skip_decode_rows = 1;
  pka::DecodeArgs da = decode_args(q, kv, block_tables, max_blocks, seq_lens, B, Hq, params);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  da.out = out;
  da.query_start_loc = query_start_loc;
  da.decode_rows_only = 1;
  da.total_q = total_q;
  da.max_query_len = max_query_len;
  da.partial_o = reinterpret_cast<float*>(ws);
  da.partial_lse = reinterpret_cast<float*>(ws + L.o_bytes);
  da.seg_counters = reinterpret_cast<int32_t*>(ws + L.o_bytes + L.lse_bytes);
  da.num_splits = L.S;
  da.split_blocks = L.C;
  da.direct_slack = kDirectSlackUnits;
  const int sms = pka::device_sm_count();
  if (sms <= 0) return PKA_ERR_CUDA;
  // Decode CTAs and prefill SMs.  The host sees only sizes, so both sides'
  // work is estimated from them: the prefill items from the query tokens
  // beyond one per request, each streaming at most the keys a query tile
  // can see (max_seq_len, or the window and the tile); the decode rows are
  // the requests the chunks leave, each streaming at most as many keys.  The
  // SMs are shared in proportion to the estimated SM time (measured rates on
  // GB300: ~2 us per 64-key prefill tile, ~70 GB/s of decode K/V per SM),
  // with every prefill item in one wave when a quarter of the SMs is left
  // to the decode rows.  The prefill side cuts its items along keys when
  // they fill less than that wave.
  const int tq = pka::mixed_query_tile(D, G);
  if (tq <= 0) return PKA_ERR_UNSUPPORTED;
  const long long extra = static_cast<long long>(total_q) - B;
  const long long est_items = extra > 0 ? (extra + tq - 1) / tq * Hkv : 0;
  const int window = params->window;
  const long long keys = (window > 0) ? std::min<long long>(max_seq_len, window + tq) : max_seq_len;
  const int bn = (D == 256) ? 64 : 128;
  const double prefill_us = static_cast<double>(est_items) * ((keys + bn - 1) / bn + 1) * 2.0;
  const long long chunks = (extra > 0 && max_query_len > 1) ? (extra + max_query_len - 2) /
                                                                   (max_query_len - 1)
                                                             : 0;
  const long long dec_rows = std::max<long long>(0, B - chunks);
  const long long dec_keys = (window > 0) ? std::min<long long>(max_seq_len, window) : max_seq_len;
  const double decode_us = static_cast<double>(dec_rows) * Hkv * ((dec_keys + 15) / 16) *
                           (64.0 * D) / 70.0e3;
  long long prefill_sms = 0;
  if (est_items > 0) {
    // the proportional share, taken only when it gives every item room for
    // two pieces or more (measured on the mixed workload: 83 prefill SMs for
    // its 64 items of ~17 key tiles ran 59 us, 64 SMs 53 us)
    const long long share =
        static_cast<long long>(sms * prefill_us / (prefill_us + decode_us) + 0.5);
    prefill_sms = (share >= 2 * est_items) ? share : est_items;
    prefill_sms = std::min<long long>(std::max<long long>(prefill_sms, 1), sms - sms / 4);
  }
  long long decode_ctas = static_cast<long long>(sms) - prefill_sms;
  if (decode_ctas < 1) decode_ctas = 1;
  // At D = 256 the items run on CTA pairs (two query tiles per pair of SMs,
  // as in paged_prefill_attn, cut along keys as below when they fit the
  // pair slots with room to spare), which needs an even number of decode
  // CTAs before them.
  const bool pairs = (D == 256) && est_items > 0;
  if (pairs && (decode_ctas & 1) != 0) --decode_ctas;
  // The prefill items run in the SMs the decode CTAs leave; when they fit
  // in one wave with room to spare, they are cut along keys into pieces
  // that fill it (the pieces' rows and counters after the decode part).
  uint8_t* split = ws + L.total();
  pa.one_wave = static_cast<int32_t>(sms - decode_ctas);
  pa.split_o = reinterpret_cast<float*>(split);
  pa.split_lse =
      reinterpret_cast<float*>(split + static_cast<size_t>(kPrefillSplitSlots) * 128 * D * 4);
  pa.split_cnt = reinterpret_cast<int32_t*>(split + static_cast<size_t>(kPrefillSplitSlots) * 128 *
                                                        (D + 1) * 4);
  pa.split_slots = kPrefillSplitSlots;
  // The pair kernel that can cut its items along keys only when the items
  // the sizes suggest (the query tokens beyond one per request, in pair
  // items of 2 TQ) are fewer than the pair slots: the merge code it carries
  // slows its softmax, and with as many items as slots it would not cut.
  const long long est_pair_items = extra > 0 ? (extra + 2 * tq - 1) / (2 * tq) * Hkv : 0;
  const bool pair_pieces =
      pairs && est_pair_items < pa.one_wave / 2 && est_pair_items <= kPrefillSplitSlots / 2;
  cudaError_t e = pka::launch_mixed(pa, da, D, G, static_cast<int>(decode_ctas), pairs,
                                    pair_pieces, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PKA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

int paged_kv_append(const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                    int32_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                    int32_t head_dim, const int32_t* slot_mapping, int32_t T, int32_t* err,
                    void* stream) {
  if (T < 0 || num_blocks <= 0 || num_kv_heads <= 0) return PKA_ERR_SHAPE;
  if (block_size != 16) return PKA_ERR_UNSUPPORTED;
  if (!supported_dim(head_dim)) return PKA_ERR_UNSUPPORTED;
  if (T == 0) return PKA_OK;
  if (k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr ||
      slot_mapping == nullptr)
    return PKA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
    return PKA_ERR_ALIGN;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return PKA_ERR_SHAPE;
  pka::AppendArgs a;
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_pool = static_cast<uint16_t*>(k_pool);
  a.v_pool = static_cast<uint16_t*>(v_pool);
  a.slot_mapping = slot_mapping;
  a.err = err;
  a.T = T;
  a.Hkv = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  const cudaError_t e =
      pka::launch_kv_append(a, pka::device_sm_count(), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

int paged_kv_append_rope(void* q, const void* k_new, const void* v_new, void* k_pool,
                         void* v_pool, int32_t num_blocks, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t block_size, int32_t head_dim,
                         const int32_t* slot_mapping, const int32_t* positions, int32_t T,
                         const float* q_norm_weight, const float* k_norm_weight, int32_t v_norm,
                         float eps, float rope_theta, int32_t rotary_dim, int32_t* err,
                         void* stream) {
  if (T < 0 || num_blocks <= 0 || num_kv_heads <= 0) return PKA_ERR_SHAPE;
  if (q != nullptr && (num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)) return PKA_ERR_SHAPE;
  if (block_size != 16) return PKA_ERR_UNSUPPORTED;
  if (!supported_dim(head_dim)) return PKA_ERR_UNSUPPORTED;
  if (rotary_dim < 0 || rotary_dim > head_dim || rotary_dim % 16 != 0) return PKA_ERR_SHAPE;
  if (rotary_dim > 0 && !(rope_theta > 1.f)) return PKA_ERR_SHAPE;
  if (!(eps >= 0.f)) return PKA_ERR_SHAPE;
  if (T == 0) return PKA_OK;
  if (k_new == nullptr || v_new == nullptr || k_pool == nullptr || v_pool == nullptr ||
      slot_mapping == nullptr || (rotary_dim > 0 && positions == nullptr))
    return PKA_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (q != nullptr && !aligned16(q)))
    return PKA_ERR_ALIGN;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return PKA_ERR_SHAPE;
  pka::AppendRopeArgs a;
  a.q = static_cast<uint16_t*>(q);
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.k_pool = static_cast<uint16_t*>(k_pool);
  a.v_pool = static_cast<uint16_t*>(v_pool);
  a.slot_mapping = slot_mapping;
  a.positions = positions;
  a.q_norm_w = q_norm_weight;
  a.k_norm_w = k_norm_weight;
  a.err = err;
  a.T = T;
  a.Hq = (q != nullptr) ? num_q_heads : 0;
  a.Hkv = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.v_norm = v_norm;
  a.rotary_dim = rotary_dim;
  a.eps = eps;
  a.rope_theta = rope_theta;
  for (int i = 0; i < 128; ++i) {
    a.gfrac[i] = 0;
    if (i < rotary_dim / 2) {
      const double f = std::pow(static_cast<double>(rope_theta), -2.0 * i / rotary_dim);
      a.gfrac[i] = static_cast<unsigned long long>(
          f * (18446744073709551616.0 / 6.283185307179586476925286766559));  // f / 2pi < 1
    }
  }
  const cudaError_t e =
      pka::launch_kv_append_rope(a, pka::device_sm_count(), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

int paged_attn_check_tables(const int32_t* block_tables, int32_t max_blocks,
                            const int32_t* seq_lens, int32_t B, int32_t num_blocks,
                            int32_t block_size, int32_t* err, void* stream) {
  if (block_tables == nullptr || seq_lens == nullptr || err == nullptr) return PKA_ERR_NULL;
  if (B < 0 || max_blocks <= 0 || num_blocks <= 0 || block_size <= 0) return PKA_ERR_SHAPE;
  if (B == 0) return PKA_OK;
  pka::CheckArgs a{};
  a.tables = block_tables;
  a.seq_lens = seq_lens;
  a.err = err;
  a.batch = B;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  cudaError_t e = pka::launch_check_tables(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}

}  // extern "C"
