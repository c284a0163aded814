// Self-tests of the device-side error paths.  Bounded waits: a kernel waits
// on an mbarrier that nothing completes, gives up after the caller's limit
// and records TIMEOUT in the device status word, leaving the context usable.
// Every wait in the library's kernels has this form (with a limit of about
// 2 s), so this shows the give-up path without faulting or hanging the GPU.
// Index checks: one write through the check of the bounds-checked build.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

__global__ void wait_timeout_kernel(unsigned long long limit_ns, int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);          // one arrival completes phase 0; none ever comes
  fence_barrier_init();
  if (!mbar_wait(b, 0, limit_ns)) record_error(err, FP4MOE_ERR_TIMEOUT);
}

// Slot `index` of a 64-entry array, written through the checked-build index
// check (forced on here).
__device__ int g_bounds_probe[64];

__global__ void bounds_check_kernel(int64_t index, int* err) {
  if (threadIdx.x != 0) return;
  if (in_bounds<true>(err, index, 64)) g_bounds_probe[index] = 1;
}

}  // namespace

cudaError_t launch_bounds_check(int64_t index, int* err, cudaStream_t st) {
  bounds_check_kernel<<<1, 32, 0, st>>>(index, err);
  return cudaGetLastError();
}

cudaError_t launch_wait_timeout(unsigned long long limit_ns, int* err,
                                cudaStream_t st) {
  wait_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, err);
  return cudaGetLastError();
}

}  // namespace fp4moe

extern "C" int fp4moe_test_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull) return FP4MOE_ERR_INVALID_ARG;
  int* err = fp4moe::status_word();
  if (!err) return FP4MOE_ERR_CUDA;
  return fp4moe::launch_wait_timeout(limit_ns, err,
                                     static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_ERR_CUDA;
}

extern "C" int fp4moe_test_bounds_check(int64_t index, void* stream) {
  int* err = fp4moe::status_word();
  if (!err) return FP4MOE_ERR_CUDA;
  return fp4moe::launch_bounds_check(index, err, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FP4MOE_OK
             : FP4MOE_ERR_CUDA;
}

extern "C" int fp4moe_build_flags(void) {
  return fp4moe::kBoundsCheck ? FP4MOE_BUILD_BOUNDS_CHECK : 0;
}
