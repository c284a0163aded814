// Allocation-free variant of the routing + permutation call.
//
// Some callers cannot allocate device memory at the point where they route
// tokens: a plugin running inside a framework whose own allocator owns the
// device memory pool (a raw cudaMalloc there can fail or fragment it), or a
// latency-critical loop where cudaMalloc may synchronise the device.  For
// them this entry point keeps its scratch (the per-block expert histogram,
// the per-block scatter bases and the token-chunk prefix) in one fixed-size
// array in device global memory that the library owns for the life of the
// process.  Every GPU that loads the library holds this array until exit.
#include <mutex>

#include "common.cuh"
#include "internal.h"

using namespace fp4moe;

namespace {

// Scratch for fp4moe_route_noalloc (FP4MOE_NOALLOC_SCRATCH_BYTES, 4 MiB).
constexpr size_t kScratchBytes = FP4MOE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device with that device current, and cached.
void* scratch_on_current_device(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = FP4MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || !p) {
      *status = FP4MOE_ERR_CUDA;
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  *status = FP4MOE_OK;
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" size_t fp4moe_route_noalloc_scratch_bytes(int T, int E) {
  if (T < 0 || E < 1 || E > kMaxE) return 0;
  const size_t nblk = (static_cast<size_t>(T) + kTokPerBlk - 1) / kTokPerBlk;
  return 2 * align256(nblk * E * 4) + align256((static_cast<size_t>(E) + 1) * 4);
}

extern "C" int fp4moe_route_noalloc(const float* logits, int T, int E,
                                    int top_k, int32_t* ids, float* w,
                                    int32_t* counts, int32_t* offsets,
                                    int32_t* perm, int32_t* inv,
                                    void* stream) {
  if (T < 0 || E < 1 || E > kMaxE || top_k < 1 || top_k > E || top_k > kMaxTopK)
    return FP4MOE_ERR_INVALID_ARG;
  if (!counts || !offsets) return FP4MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !ids || !w || !perm || !inv)) return FP4MOE_ERR_INVALID_ARG;
  const size_t need = fp4moe_route_noalloc_scratch_bytes(T, E);
  if (need > kScratchBytes) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;
  int st_code = FP4MOE_OK;
  char* scratch = static_cast<char*>(scratch_on_current_device(&st_code));
  if (!scratch) return st_code;
  const size_t nblk = (static_cast<size_t>(T) + kTokPerBlk - 1) / kTokPerBlk;
  int32_t* hist = reinterpret_cast<int32_t*>(scratch);
  int32_t* base = reinterpret_cast<int32_t*>(scratch + align256(nblk * E * 4));
  int32_t* cstart = reinterpret_cast<int32_t*>(scratch + 2 * align256(nblk * E * 4));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The kernels overwrite every scratch word they later read (each routing
  // block writes its whole histogram row, the scan writes every base and
  // prefix entry), so nothing left by an earlier call needs clearing.
  cudaError_t e = launch_route(logits, T, E, top_k, ids, w, hist, status_word(), st);
  if (e == cudaSuccess)
    e = launch_scan(T, E, hist, base, counts, offsets, cstart, gemm_chunk_max(T), st);
  if (e == cudaSuccess)
    e = launch_scatter(ids, T, E, top_k, base, perm, inv, nullptr, nullptr, 0,
                       FP4MOE_ACT_BF16, nullptr, status_word(), st);
  return e == cudaSuccess ? FP4MOE_OK : FP4MOE_ERR_CUDA;
}
