// Self-test of the bounded wait (sm_103a): one thread waits, with the wait
// routine every kernel of the library uses, on an mbarrier phase that
// nothing completes.  The wait runs out after the given budget, reports
// PKA_DEVERR_TIMEOUT into the error word and the kernel returns -- the
// behaviour every pipeline relies on to end with an error status instead of
// hanging when a copy or a partner never arrives.
#include "common.cuh"

namespace pka {

namespace {

__global__ void bounded_wait_probe_kernel(int32_t* err, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);  // one arrival expected; none ever comes
  mbar_fence_init();
  mbar_wait_budget(&bar, 0, err, budget);
}

}  // namespace

}  // namespace pka

extern "C" int pka_selftest_bounded_wait(int32_t* err, int64_t budget_cycles, void* stream) {
  if (err == nullptr) return PKA_ERR_NULL;
  if (budget_cycles <= 0 || budget_cycles > 2000000000LL) return PKA_ERR_SHAPE;
  pka::bounded_wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      err, static_cast<long long>(budget_cycles));
  return cudaGetLastError() == cudaSuccess ? PKA_OK : PKA_ERR_CUDA;
}
