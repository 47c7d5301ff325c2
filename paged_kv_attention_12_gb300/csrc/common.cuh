// Device helpers shared by the paged-attention kernels (sm_103a).
//
// mbarrier + bulk-copy (TMA) wrappers written as inline PTX, bounded waits
// that report a timeout instead of hanging, and bf16 unpacking.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "paged_attn.h"

namespace pka {

#ifdef PKA_TIMELINE
// Instrumented builds only (-DPKA_TIMELINE): the global timer, in ns.
__device__ __forceinline__ unsigned long long timeline_now() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Each translation unit has its own copy of a __device__ array; a unit
// whose kernels record stamps exports its copy under its own names.
#define PKA_TIMELINE_EXPORT(name, array)                                                    \
  extern "C" int pka_timeline_copy##name(void* dst) {                                       \
    return static_cast<int>(                                                                 \
        cudaMemcpyFromSymbol(dst, array, sizeof(array), 0, cudaMemcpyDeviceToDevice));       \
  }                                                                                          \
  extern "C" int pka_timeline_clear##name(void* stream) {                                   \
    void* p = nullptr;                                                                       \
    if (cudaGetSymbolAddress(&p, array) != cudaSuccess) return -1;                           \
    return static_cast<int>(cudaMemsetAsync(p, 0, sizeof(array),                              \
                                            static_cast<cudaStream_t>(stream)));             \
  }
#endif

constexpr int kBlockSize = 16;        // tokens per KV block (the only supported size)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// A bounded wait gives up after this many SM clock cycles (about a second).
constexpr long long kWaitBudgetCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void report(int32_t* err, int bits) {
  if (err != nullptr) atomicOr(err, bits);
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Gives up after
// `budget` SM clock cycles, reports PKA_DEVERR_TIMEOUT and returns false.
__device__ __forceinline__ bool mbar_wait_budget(uint64_t* bar, uint32_t parity, int32_t* err,
                                                 long long budget) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > budget) {
      report(err, PKA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Every wait of the library's kernels: a budget of kWaitBudgetCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* err) {
  return mbar_wait_budget(bar, parity, err, kWaitBudgetCycles);
}

// ------------------------------------------------------- bulk copy (TMA)
// 1-D bulk copy global -> shared, completion counted on an mbarrier.  Both
// addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                        uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Same, with an L2 evict-first hint: K/V tiles are streamed once.
__device__ __forceinline__ void bulk_g2s_stream(void* dst_smem, const void* src_gmem,
                                               uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], "
      "[%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Bulk copy shared -> global through the async (TMA) proxy, in the issuing
// thread's bulk groups: both addresses 16-byte aligned, bytes a multiple of
// 16.  The smem writes it reads must be fenced into the async proxy first
// (fence.proxy.async.shared::cta by the writing threads).
__device__ __forceinline__ void bulk_s2g(void* dst_gmem, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
               "r"(smem_u32(src_smem)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The thread's bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// The thread's bulk groups have completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// GPU-scope acquire-release fence: with a relaxed atomic after it, the
// release half of a flag handshake; after an atomic, the acquire half.
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// ------------------------------------------------------------ arithmetic
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One step of the split-K log-sum-exp merge: folds four pieces (natural-log
// LSE lv[u], normalised partial row x[u]) into a running state (max M,
// denominator den, numerator acc) taken relative to M.  Pieces with
// lv = -inf must come with x = 0; a group of four such pieces leaves the
// state untouched.  The split-K combine launch and the decode kernel's fused
// combine both merge groups [0, 4), [4, 8), ... of a row's pieces with this
// step, so the two paths give identical results.
__device__ __forceinline__ void lse_merge4(float& M, float& den, float4& acc, const float* lv,
                                          const float4* x) {
  const float gm = fmaxf(fmaxf(lv[0], lv[1]), fmaxf(lv[2], lv[3]));
  if (gm == -INFINITY) return;
  const float nm = fmaxf(M, gm);
  const float r = fast_exp2((M - nm) * 1.4426950408889634f);  // 0 while M = -inf
  den *= r;
  acc.x *= r;
  acc.y *= r;
  acc.z *= r;
  acc.w *= r;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float w = fast_exp2((lv[u] - nm) * 1.4426950408889634f);
    den += w;
    acc.x = fmaf(w, x[u].x, acc.x);
    acc.y = fmaf(w, x[u].y, acc.y);
    acc.z = fmaf(w, x[u].z, acc.z);
    acc.w = fmaf(w, x[u].w, acc.w);
  }
  M = nm;
}

// bf16 pair (packed in a 32-bit word) -> two fp32, exact.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  bf16x2_to_f32(u.x, f[0], f[1]);
  bf16x2_to_f32(u.y, f[2], f[3]);
  bf16x2_to_f32(u.z, f[4], f[5]);
  bf16x2_to_f32(u.w, f[6], f[7]);
}

// Two fp32 -> packed bf16x2 (round to nearest even), one hardware convert.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  return static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xffffu);
}

// Raises a kernel's dynamic shared-memory limit once per (kernel, device):
// the call takes a driver lock, so it stays off the per-launch path.
inline cudaError_t set_smem_once(const void* kernel, int bytes) {
  struct Entry {
    const void* kernel;
    int device;
  };
  static std::mutex mu;
  static Entry done[256];
  static int count = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < count; ++i)
    if (done[i].kernel == kernel && done[i].device == dev) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && count < 256) done[count++] = Entry{kernel, dev};
  return e;
}

}  // namespace pka
