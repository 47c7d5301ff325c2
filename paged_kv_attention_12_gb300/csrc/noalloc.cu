// Split-K decode for callers that cannot allocate device memory.
//
// paged_decode_splitk needs a workspace for its fp32 partials, which the
// caller normally allocates.  Some callers cannot: code that runs while
// another allocator owns all device memory (a framework plugin that must not
// grow the process's footprint), code inside a region where allocation calls
// are not allowed, or a host program without a device allocator of its own.
// This entry point takes its partials from a fixed array compiled into the
// library instead, so it allocates nothing; the caller still passes the
// inputs and the output.
//
// The array is a file-scope __device__ variable.  In host code its name is
// only a stand-in for the device object, never a device address, so the
// address is obtained once per device with cudaGetSymbolAddress (with that
// device current) and cached.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "kernels.h"
#include "paged_attn.h"

namespace {

// 16 MiB of fp32 partials.  Every GPU that loads the library holds this
// array until the process exits.
constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr size_t kScratchFloats = kScratchBytes / sizeof(float);
__device__ __align__(256) float g_decode_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call per device).
int scratch_for_current_device(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return PKA_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return PKA_OK;
}

}  // namespace

extern "C" {

int paged_decode_attn_noalloc(const void* q, void* out, const pka_kv_pool* kv,
                              const int32_t* block_tables, int32_t max_blocks,
                              const int32_t* seq_lens, int32_t B, int32_t Hq,
                              int32_t max_seq_len, const pka_attn_params* params,
                              void* stream) {
  // the same argument checks as every other decode entry point, before the
  // empty batch returns
  int st = pka::check_decode_call(q, out, kv, block_tables, max_blocks, seq_lens, B, Hq,
                                  max_seq_len, params);
  if (st != PKA_OK) return st;
  if (B == 0) return PKA_OK;
  int32_t S = 0, C = 0;
  st = paged_decode_splitk_plan(B, kv->num_kv_heads, max_seq_len, kv->block_size,
                                params->window, 0, &S, &C);
  if (st != PKA_OK) return st;
  // partial outputs [B][Hq][S][D] first, then the LSEs [B][Hq][S]
  const size_t n_o = static_cast<size_t>(B) * Hq * S * kv->head_dim;
  const size_t n_lse = static_cast<size_t>(B) * Hq * S;
  if (kv->head_dim <= 0 || n_o + n_lse > kScratchFloats) return PKA_ERR_WORKSPACE;
  float* scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != PKA_OK) return st;
  float* partial_o = scratch;
  float* partial_lse = scratch + n_o;
  // The split-K kernel writes every slot's LSE (-inf where unused) and the
  // output of every used slot, so nothing in the array needs clearing.
  st = paged_decode_splitk(q, partial_o, partial_lse, kv, block_tables, max_blocks, seq_lens, B,
                           Hq, max_seq_len, S, C, params, stream);
  if (st != PKA_OK) return st;
  return paged_decode_splitk_combine(partial_o, partial_lse, B, Hq, kv->head_dim, S, out,
                                     nullptr, stream);
}

}  // extern "C"
