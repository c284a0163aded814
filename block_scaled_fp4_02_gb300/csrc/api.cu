// C-ABI entry points of libfp4moe (declared in include/fp4moe.h): argument
// checks, workspace layout, tensor maps and the launch sequence of each call.
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

using namespace fp4moe;

struct fp4moe_packed {
  int E, K, I, gran, act_mode, w13_layout, device;
  bool mx;       // block-scaled path: plain codes + scale words
  uint8_t* w13;
  size_t w13_bytes;
  uint8_t* w2;
  size_t w2_bytes;
  uint32_t* s13;  // block-scaled path: scale words [E][2I/128][K/128][128]
  size_t s13_bytes;
  uint32_t* s2;   //                    [E][K/128][I/128][128]
  size_t s2_bytes;
  float* alpha;  // [2E]: FC1 then FC2
  uint32_t smul, sadd;
};

// Per-device status word: kernels record the first data-dependent error.
__device__ int g_fp4moe_status;

namespace fp4moe {
int* status_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_fp4moe_status) != cudaSuccess) return nullptr;
  return static_cast<int*>(p);
}

int device_sm_count() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> g(mu);
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}
}  // namespace fp4moe

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP4MOE_OK : FP4MOE_ERR_CUDA; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major [rows, cols] of E2M1 codes (two per byte) read in 128 x 128
// boxes with the 16U4_ALIGN16B type (each 16 codes widened to 16 bytes in
// shared memory) and the 128-byte swizzle: the kind::mxf8f6f4 operand form.
bool make_e2m1_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto fn = encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols / 2};
  cuuint32_t box[2] = {128, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bytes [rows, cols] (E4M3) read in boxes of box_rows x 128 with
// the 128-byte swizzle.
bool make_u8_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                  uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major bf16 [rows, cols] read in boxes of box_rows rows x 64 columns
// with the 128-byte swizzle (the UMMA K-major operand layout).
bool make_row_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn || rows == 0) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct RouteLayout {
  size_t hist, base, cstart, total;
};

RouteLayout route_layout(int T, int E, size_t start = 0) {
  const size_t nblk = (static_cast<size_t>(T) + kTokPerBlk - 1) / kTokPerBlk;
  RouteLayout L;
  size_t off = start;
  L.hist = off; off = align_up(off + nblk * E * 4);
  L.base = off; off = align_up(off + nblk * E * 4);
  L.cstart = off; off = align_up(off + (static_cast<size_t>(E) + 1) * 4);
  L.total = off;
  return L;
}

struct MoeLayout {
  RouteLayout r;
  size_t ids, wts, counts, offsets, perm, inv, xperm, xs, h, hs, h32, o, total;
  int64_t pitch;  // block-scaled path: scale words per step row
};

// Words per step row of the block-scaled path's scale arrays: P rounded up
// to 4 plus the over-read of the aligned bulk copies of the last chunk.
int64_t mx_pitch(int64_t P) { return ((P + 3) & ~3LL) + 264; }

MoeLayout moe_layout(const fp4moe_packed* p, int T, int k) {
  const size_t P = static_cast<size_t>(T) * k;
  MoeLayout L;
  L.r = route_layout(T, p->E, 0);
  size_t off = L.r.total;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes); return o; };
  L.ids = take(P * 4);
  L.wts = take(P * 4);
  L.counts = take(static_cast<size_t>(p->E) * 4);
  L.offsets = take((static_cast<size_t>(p->E) + 1) * 4);
  L.perm = take(P * 4);
  L.inv = take(P * 4);
  L.pitch = 0;
  L.xs = L.hs = L.h32 = 0;
  if (p->mx) {
    L.pitch = mx_pitch(static_cast<int64_t>(P));
    L.xperm = take(P * p->K);
    L.xs = take(static_cast<size_t>(p->K / kMxK) * L.pitch * 4);
    L.h = take(P * p->I);
    L.hs = take(static_cast<size_t>(p->I / kMxK) * L.pitch * 4);
  } else {
    L.xperm = take(P * p->K * 2);
    L.h = take(P * p->I * 2);
    L.h32 = (p->act_mode == FP4MOE_ACT_FP8) ? take(P * p->I * 4) : 0;
  }
  L.o = take(P * p->K * 4);
  L.total = off;
  return L;
}

// Stage events handed over by fp4moe_set_stage_events for the next forward.
thread_local cudaEvent_t t_stage_ev[FP4MOE_STAGE_EVENTS];
thread_local bool t_stage_on = false;

void stage_mark(int i, cudaStream_t st) {
  if (t_stage_on) cudaEventRecord(t_stage_ev[i], st);
}

// S2 + S3 without the gather: ids, w, counts, offsets, cstart (chunks of at
// most `chunk` tokens), perm and inv.  Up to kTokPerBlk tokens take one
// launch; more take route, scan and scatter (the same values).  Marks the
// route and scan stages.
cudaError_t route_permute(const float* logits, int T, int E, int k, int chunk, int32_t* hist,
                          int32_t* base, int32_t* ids, float* w, int32_t* counts,
                          int32_t* offsets, int32_t* cstart, int32_t* perm, int32_t* inv,
                          int* err, cudaStream_t st) {
  if (T <= kTokPerBlk) {
    const cudaError_t e = launch_route_small(logits, T, E, k, chunk, ids, w, counts, offsets,
                                             cstart, perm, inv, err, st);
    stage_mark(1, st);
    stage_mark(2, st);
    return e;
  }
  cudaError_t e = launch_route(logits, T, E, k, ids, w, hist, err, st);
  stage_mark(1, st);
  if (e == cudaSuccess) e = launch_scan(T, E, hist, base, counts, offsets, cstart, chunk, st);
  stage_mark(2, st);
  if (e == cudaSuccess)
    e = launch_scatter(ids, T, E, k, base, perm, inv, nullptr, nullptr, 0, FP4MOE_ACT_BF16,
                       nullptr, err, st);
  return e;
}

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

void free_packed(fp4moe_packed* p) {
  if (!p) return;
  cudaFree(p->w13);
  cudaFree(p->w2);
  cudaFree(p->s13);
  cudaFree(p->s2);
  cudaFree(p->alpha);
  delete p;
}

// The MoE layer on the block-scaled path (FP8 activations over group32
// weights): routing, permutation, gather of the E4M3 rows and their scale
// words, FC1 + SwiGLU with the FP8 rounding of h in its epilogue, FC2 and the
// combine; stage events as in fp4moe_moe_forward (no separate rounding of h,
// so events 4 and 5 coincide).
int mx_forward(const fp4moe_packed* p, const MoeLayout& L, char* ws, const void* x,
               const uint8_t* x_scales, const float* router_logits, int T, int top_k,
               void* y, cudaStream_t st) {
  auto at = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  int32_t *hist = at(L.r.hist), *base = at(L.r.base), *cstart = at(L.r.cstart);
  int32_t *ids = at(L.ids), *counts = at(L.counts), *offsets = at(L.offsets);
  int32_t *perm = at(L.perm), *inv = at(L.inv);
  float* wts = reinterpret_cast<float*>(ws + L.wts);
  uint8_t* xperm = reinterpret_cast<uint8_t*>(ws + L.xperm);
  uint32_t* xs = reinterpret_cast<uint32_t*>(ws + L.xs);
  uint8_t* h8 = reinterpret_cast<uint8_t*>(ws + L.h);
  uint32_t* hs = reinterpret_cast<uint32_t*>(ws + L.hs);
  float* o = reinterpret_cast<float*>(ws + L.o);
  int* err = status_word();
  const int64_t P = static_cast<int64_t>(T) * top_k;
  const int sms = device_sm_count();
  struct StageOff {
    ~StageOff() { t_stage_on = false; }
  } stage_off;
  stage_mark(0, st);
  cudaError_t e = route_permute(router_logits, T, p->E, top_k, kMxChunk, hist, base, ids, wts,
                                counts, offsets, cstart, perm, inv, err, st);
  if (e == cudaSuccess)
    e = launch_gather_mx(inv, T, top_k, static_cast<const uint8_t*>(x), x_scales, p->K,
                         L.pitch, xperm, xs, err, st);
  stage_mark(3, st);
  if (e != cudaSuccess) return FP4MOE_ERR_CUDA;

  MxMaps m1, m2;
  bool ok = make_e2m1_tmap(&m1.w, p->w13, static_cast<uint64_t>(p->E) * 2 * p->I, p->K) &&
            make_e2m1_tmap(&m2.w, p->w2, static_cast<uint64_t>(p->E) * p->K, p->I);
  for (int i = 0; i < kMxBoxes && ok; ++i)
    ok = make_u8_tmap(&m1.x[i], xperm, P, p->K, 32u * (i + 1)) &&
         make_u8_tmap(&m2.x[i], h8, P, p->I, 32u * (i + 1));
  if (!ok) return FP4MOE_ERR_CUDA;
  MxGemmArgs a1{};
  a1.wscale = p->s13; a1.xscale = xs; a1.alpha = p->alpha; a1.offsets = offsets;
  a1.cstart = cstart; a1.out = h8; a1.hscale = reinterpret_cast<uint8_t*>(hs); a1.err = err;
  a1.rows = P;
  a1.E = p->E; a1.nblocks = p->I / 128; a1.ksteps = p->K / kMxK;
  a1.rows_per_expert = 2 * p->I; a1.tiles_per_expert = 2 * p->I / 128;
  a1.xscale_pitch = L.pitch; a1.hscale_pitch = L.pitch; a1.ldo = p->I;
  a1.mode = kGemmModeFc1;
  e = gemm_mx_pair_supported(a1) ? launch_gemm_mx_pair(m1, a1, sms, st)
                                 : launch_gemm_mx(m1, a1, sms, st);
  stage_mark(4, st);
  stage_mark(5, st);
  MxGemmArgs a2 = a1;
  a2.wscale = p->s2; a2.xscale = hs; a2.alpha = p->alpha + p->E; a2.out = o;
  a2.hscale = nullptr; a2.nblocks = p->K / 128; a2.ksteps = p->I / kMxK;
  a2.rows_per_expert = p->K; a2.tiles_per_expert = p->K / 128; a2.ldo = p->K;
  a2.mode = kGemmModeFc2;
  if (e == cudaSuccess)
    e = gemm_mx_pair_supported(a2) ? launch_gemm_mx_pair(m2, a2, sms, st)
                                   : launch_gemm_mx(m2, a2, sms, st);
  stage_mark(6, st);
  if (e == cudaSuccess)
    e = launch_combine(o, inv, wts, T, top_k, p->K, static_cast<uint16_t*>(y), err, st);
  stage_mark(7, st);
  return cuda_status(e);
}

}  // namespace

extern "C" {

const char* fp4moe_status_string(int s) {
  switch (s) {
    case FP4MOE_OK: return "ok";
    case FP4MOE_ERR_INVALID_ARG: return "invalid argument";
    case FP4MOE_ERR_UNSUPPORTED: return "unsupported";
    case FP4MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FP4MOE_ERR_CUDA: return "CUDA error";
    case FP4MOE_ERR_TIMEOUT: return "device wait timed out";
    case FP4MOE_ERR_BOUNDS: return "index out of bounds (bounds-checked build)";
    default: return "unknown status";
  }
}

int fp4moe_last_device_error(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return FP4MOE_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_fp4moe_status, sizeof(int)) != cudaSuccess)
    return FP4MOE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_fp4moe_status, &zero, sizeof(int)) != cudaSuccess)
    return FP4MOE_ERR_CUDA;
  return v;
}

int fp4moe_set_stage_events(void* const* events, int n) {
  if (!events) {
    t_stage_on = false;
    return FP4MOE_OK;
  }
  if (n != FP4MOE_STAGE_EVENTS) return FP4MOE_ERR_INVALID_ARG;
  for (int i = 0; i < n; ++i) {
    if (!events[i]) return FP4MOE_ERR_INVALID_ARG;
    t_stage_ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  t_stage_on = true;
  return FP4MOE_OK;
}

int fp4moe_requant_fp4_gran_k(const uint8_t* fp4, const uint8_t* e4m3_s,
                              int64_t rows, int64_t K, int src_gran,
                              int dst_gran, uint8_t* fp4_out,
                              uint8_t* ue8m0_out, void* stream) {
  if (rows < 0 || K <= 0 || K % 32 != 0) return FP4MOE_ERR_INVALID_ARG;
  if (src_gran != 16 || dst_gran != 32) {
    if ((src_gran != 16 && src_gran != 32) || (dst_gran != 16 && dst_gran != 32))
      return FP4MOE_ERR_INVALID_ARG;
    return FP4MOE_ERR_UNSUPPORTED;
  }
  if (rows == 0) return FP4MOE_OK;
  if (!fp4 || !e4m3_s || !fp4_out || !ue8m0_out) return FP4MOE_ERR_INVALID_ARG;
  if (!aligned(fp4, 16) || !aligned(fp4_out, 16) || !aligned(e4m3_s, 2))
    return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_requant(fp4, e4m3_s, rows, K, fp4_out, ue8m0_out,
                                    status_word(),
                                    static_cast<cudaStream_t>(stream)));
}

int fp4moe_act_quant(const void* x_bf16, int64_t T, int64_t K, uint8_t* xq,
                     uint8_t* xs, void* stream) {
  if (T < 0 || K <= 0 || K % 32 != 0) return FP4MOE_ERR_INVALID_ARG;
  if (T == 0) return FP4MOE_OK;
  if (!x_bf16 || !xq || !xs || !aligned(x_bf16, 16) || !aligned(xq, 16))
    return FP4MOE_ERR_INVALID_ARG;
  return cuda_status(launch_act_quant(static_cast<const uint16_t*>(x_bf16), T,
                                      K, xq, xs, status_word(),
                                      static_cast<cudaStream_t>(stream)));
}

size_t fp4moe_route_workspace_size(int T, int E, int top_k) {
  if (T < 0 || E < 1 || E > kMaxE || top_k < 1 || top_k > std::min(E, kMaxTopK))
    return 0;
  return route_layout(T, E).total;
}

int fp4moe_route_debug(const float* logits, int T, int E, int top_k,
                       int32_t* ids, float* w, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv,
                       void* workspace, size_t ws_bytes, void* stream) {
  if (T < 0 || E < 1 || E > kMaxE || top_k < 1 || top_k > std::min(E, kMaxTopK))
    return FP4MOE_ERR_INVALID_ARG;
  if (!counts || !offsets || !workspace) return FP4MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !ids || !w || !perm || !inv)) return FP4MOE_ERR_INVALID_ARG;
  const RouteLayout L = route_layout(T, E);
  if (ws_bytes < L.total) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, kAlign)) return FP4MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int32_t* hist = reinterpret_cast<int32_t*>(ws + L.hist);
  int32_t* base = reinterpret_cast<int32_t*>(ws + L.base);
  int32_t* cstart = reinterpret_cast<int32_t*>(ws + L.cstart);
  cudaError_t e = launch_route(logits, T, E, top_k, ids, w, hist, status_word(), st);
  if (e == cudaSuccess)
    e = launch_scan(T, E, hist, base, counts, offsets, cstart, gemm_chunk_max(T), st);
  if (e == cudaSuccess)
    e = launch_scatter(ids, T, E, top_k, base, perm, inv, nullptr, nullptr, 0,
                       FP4MOE_ACT_BF16, nullptr, status_word(), st);
  return cuda_status(e);
}

int fp4moe_prepare_weights(const uint8_t* w13, const uint8_t* w13_s,
                           const float* w13_gs, const uint8_t* w2,
                           const uint8_t* w2_s, const float* w2_gs, int E,
                           int K, int I, int gran_k, int w13_layout,
                           int act_mode, void* stream, fp4moe_packed** out) {
  if (!out) return FP4MOE_ERR_INVALID_ARG;
  *out = nullptr;
  const int mode = act_mode & 0xFF;
  const bool no_requant = (act_mode & FP4MOE_FLAG_NO_REQUANT) != 0;
  const bool keep16 = (act_mode & FP4MOE_FLAG_KEEP_GROUP16) != 0;
  const bool gs_inv = (act_mode & FP4MOE_FLAG_GS_INVERTED) != 0;
  if ((act_mode & ~(0xFF | FP4MOE_FLAG_NO_REQUANT | FP4MOE_FLAG_KEEP_GROUP16 |
                    FP4MOE_FLAG_GS_INVERTED)) != 0)
    return FP4MOE_ERR_INVALID_ARG;
  if (mode != FP4MOE_ACT_BF16 && mode != FP4MOE_ACT_FP8) return FP4MOE_ERR_INVALID_ARG;
  if (gran_k != 16 && gran_k != 32) return FP4MOE_ERR_INVALID_ARG;
  if (w13_layout != FP4MOE_W13_GATE_UP && w13_layout != FP4MOE_W13_UP_GATE)
    return FP4MOE_ERR_INVALID_ARG;
  if (E < 1 || E > kMaxE || K <= 0 || I <= 0 || K % 128 || I % 128)
    return FP4MOE_ERR_INVALID_ARG;
  if (!w13 || !w13_s || !w13_gs || !w2 || !w2_s || !w2_gs) return FP4MOE_ERR_INVALID_ARG;
  if (!aligned(w13, 16) || !aligned(w2, 16)) return FP4MOE_ERR_INVALID_ARG;
  // FP8 over group16: lossy requant to group32, unless the exact group16
  // conversion is asked for (KEEP_GROUP16) or refused (NO_REQUANT).
  const bool requant = (mode == FP4MOE_ACT_FP8 && gran_k == 16 && !keep16);
  if (requant && no_requant) return FP4MOE_ERR_UNSUPPORTED;
  const int g = requant ? 32 : gran_k;
  // FP8 activations over group32 weights (given, or from the requant) run
  // on the block-scaled tensor-core path; kept group16 weights and bf16
  // activations on the bf16 path.
  const bool mx = (mode == FP4MOE_ACT_FP8 && g == 32);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  fp4moe_packed* p = new fp4moe_packed{};
  p->E = E; p->K = K; p->I = I; p->gran = g; p->act_mode = mode;
  p->w13_layout = w13_layout;
  p->mx = mx;
  cudaGetDevice(&p->device);
  p->smul = mx ? 0u : (g == 16) ? 16u : 128u;
  p->sadd = (!mx && g == 16) ? 0x7680u : 0u;
  const int64_t n13 = 2LL * I, n2 = K;
  if (mx) {
    p->w13_bytes = static_cast<size_t>(E) * n13 * (K / 2);
    p->w2_bytes = static_cast<size_t>(E) * n2 * (I / 2);
    p->s13_bytes = static_cast<size_t>(E) * n13 * (K / kMxK) * 4;
    p->s2_bytes = static_cast<size_t>(E) * n2 * (I / kMxK) * 4;
  } else {
    p->w13_bytes = static_cast<size_t>(E) * (n13 / kTileN) * (K / kTileK) * tile_bytes(g);
    p->w2_bytes = static_cast<size_t>(E) * (n2 / kTileN) * (I / kTileK) * tile_bytes(g);
  }

  uint8_t* tmp = nullptr;   // requant output, if any
  int32_t* bmax = nullptr;  // [2E]
  int* err = nullptr;
  auto fail = [&](int code) {
    cudaStreamSynchronize(st);
    cudaFree(tmp);
    cudaFree(bmax);
    cudaFree(err);
    free_packed(p);
    return code;
  };
  if (cudaMalloc(&p->w13, p->w13_bytes) != cudaSuccess ||
      cudaMalloc(&p->w2, p->w2_bytes) != cudaSuccess ||
      (mx && cudaMalloc(&p->s13, p->s13_bytes) != cudaSuccess) ||
      (mx && cudaMalloc(&p->s2, p->s2_bytes) != cudaSuccess) ||
      cudaMalloc(&p->alpha, 2 * E * sizeof(float)) != cudaSuccess ||
      cudaMalloc(&bmax, 2 * E * sizeof(int32_t)) != cudaSuccess ||
      cudaMalloc(&err, sizeof(int)) != cudaSuccess)
    return fail(FP4MOE_ERR_CUDA);
  if (cudaMemsetAsync(bmax, 0, 2 * E * sizeof(int32_t), st) != cudaSuccess ||
      cudaMemsetAsync(err, 0, sizeof(int), st) != cudaSuccess)
    return fail(FP4MOE_ERR_CUDA);

  const uint8_t *c13 = w13, *s13 = w13_s, *c2 = w2, *s2 = w2_s;
  cudaError_t e = cudaSuccess;
  if (requant) {
    // Lossy group16 -> group32 conversion (the requantization path of the
    // group16 notes page), then pack the group32 result.
    const size_t b13 = static_cast<size_t>(E) * n13 * (K / 2);
    const size_t q13 = static_cast<size_t>(E) * n13 * (K / 32);
    const size_t b2 = static_cast<size_t>(E) * n2 * (I / 2);
    const size_t q2 = static_cast<size_t>(E) * n2 * (I / 32);
    if (cudaMalloc(&tmp, align_up(b13) + align_up(q13) + align_up(b2) + q2) != cudaSuccess)
      return fail(FP4MOE_ERR_CUDA);
    uint8_t* t = tmp;
    uint8_t* rc13 = t; t += align_up(b13);
    uint8_t* rs13 = t; t += align_up(q13);
    uint8_t* rc2 = t; t += align_up(b2);
    uint8_t* rs2 = t;
    e = launch_requant(w13, w13_s, static_cast<int64_t>(E) * n13, K, rc13, rs13, err, st);
    if (e == cudaSuccess)
      e = launch_requant(w2, w2_s, static_cast<int64_t>(E) * n2, I, rc2, rs2, err, st);
    c13 = rc13; s13 = rs13; c2 = rc2; s2 = rs2;
  }
  if (mx) {
    // Plain codes (FC1 rows reordered into gate/up tiles) and scale words.
    if (e == cudaSuccess)
      e = launch_mx_rows(c13, E, static_cast<int>(n13), K, true, w13_layout, p->w13, st);
    if (e == cudaSuccess)
      e = launch_mx_rows(c2, E, static_cast<int>(n2), I, false, 0, p->w2, st);
    if (e == cudaSuccess)
      e = launch_mx_scales(s13, E, static_cast<int>(n13), K, true, w13_layout, p->s13, err, st);
    if (e == cudaSuccess)
      e = launch_mx_scales(s2, E, static_cast<int>(n2), I, false, 0, p->s2, err, st);
    if (e == cudaSuccess) e = launch_alpha(w13_gs, nullptr, E, 0, gs_inv, p->alpha, st);
    if (e == cudaSuccess) e = launch_alpha(w2_gs, nullptr, E, 0, gs_inv, p->alpha + E, st);
  } else {
    if (e == cudaSuccess && g == 32) {
      e = launch_scale_max(s13, E, n13 * (K / 32), bmax, err, st);
      if (e == cudaSuccess) e = launch_scale_max(s2, E, n2 * (I / 32), bmax + E, err, st);
    }
    if (e == cudaSuccess)
      e = launch_pack(c13, s13, E, static_cast<int>(n13), K, g, true, w13_layout, bmax,
                      p->w13, err, st);
    if (e == cudaSuccess)
      e = launch_pack(c2, s2, E, static_cast<int>(n2), I, g, false, 0, bmax + E, p->w2,
                      err, st);
    if (e == cudaSuccess) e = launch_alpha(w13_gs, bmax, E, g, gs_inv, p->alpha, st);
    if (e == cudaSuccess) e = launch_alpha(w2_gs, bmax + E, E, g, gs_inv, p->alpha + E, st);
  }
  if (e != cudaSuccess) return fail(FP4MOE_ERR_CUDA);
  if (cudaStreamSynchronize(st) != cudaSuccess) return fail(FP4MOE_ERR_CUDA);
  int h_err = 0;
  if (cudaMemcpy(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(FP4MOE_ERR_CUDA);
  if (h_err != 0) return fail(FP4MOE_ERR_INVALID_ARG);
  cudaFree(tmp);
  cudaFree(bmax);
  cudaFree(err);
  *out = p;
  return FP4MOE_OK;
}

void fp4moe_free_packed(fp4moe_packed* p) {
  if (!p) return;
  cudaDeviceSynchronize();
  free_packed(p);
}

int fp4moe_packed_info(const fp4moe_packed* p, fp4moe_packed_desc* d) {
  if (!p || !d) return FP4MOE_ERR_INVALID_ARG;
  d->E = p->E; d->K = p->K; d->I = p->I; d->gran_k = p->gran;
  d->act_mode = p->act_mode; d->w13_layout = p->w13_layout;
  d->k_tile = p->mx ? kMxK : kTileK; d->n_tile = kTileN;
  d->tile_bytes = p->mx ? 0 : tile_bytes(p->gran);
  d->w13 = p->w13; d->w13_bytes = p->w13_bytes;
  d->w2 = p->w2; d->w2_bytes = p->w2_bytes;
  d->alpha13 = p->alpha; d->alpha2 = p->alpha + p->E;
  d->scale_mul = p->smul; d->scale_add = p->sadd;
  d->layout = p->mx ? 1 : 0;
  d->w13_scales = p->s13; d->w13_scales_bytes = p->s13_bytes;
  d->w2_scales = p->s2; d->w2_scales_bytes = p->s2_bytes;
  return FP4MOE_OK;
}

size_t fp4moe_moe_workspace_size(const fp4moe_packed* p, int T, int top_k) {
  if (!p || T < 0 || top_k < 1 || top_k > std::min(p->E, kMaxTopK)) return 0;
  return moe_layout(p, T, top_k).total;
}

int fp4moe_moe_workspace_offsets(const fp4moe_packed* p, int T, int top_k,
                                 size_t* out, int n) {
  if (!p || !out || n < 10 || T < 0 || top_k < 1 ||
      top_k > std::min(p->E, kMaxTopK))
    return FP4MOE_ERR_INVALID_ARG;
  const MoeLayout L = moe_layout(p, T, top_k);
  const size_t v[13] = {L.ids, L.wts, L.counts, L.offsets, L.perm,
                        L.inv, L.xperm, L.h, L.o, L.total,
                        L.hs, p->mx ? 1u : 0u, static_cast<size_t>(L.pitch)};
  for (int i = 0; i < std::min(n, 13); ++i) out[i] = v[i];
  return FP4MOE_OK;
}

int fp4moe_moe_forward(const void* x, const uint8_t* x_scales,
                       const float* router_logits, int T,
                       const fp4moe_packed* p, int top_k, void* y,
                       void* workspace, size_t ws_bytes, void* stream) {
  if (!p || T < 0 || top_k < 1 || top_k > std::min(p->E, kMaxTopK))
    return FP4MOE_ERR_INVALID_ARG;
  if (T == 0) return FP4MOE_OK;
  if (!x || !router_logits || !y || !workspace) return FP4MOE_ERR_INVALID_ARG;
  if (p->act_mode == FP4MOE_ACT_BF16 && x_scales) return FP4MOE_ERR_INVALID_ARG;
  if (p->act_mode == FP4MOE_ACT_FP8 && !x_scales) return FP4MOE_ERR_INVALID_ARG;
  if (p->mx && !aligned(x_scales, 4)) return FP4MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(workspace, kAlign))
    return FP4MOE_ERR_INVALID_ARG;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev != p->device) return FP4MOE_ERR_INVALID_ARG;
  const MoeLayout L = moe_layout(p, T, top_k);
  if (ws_bytes < L.total) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  auto at = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  int32_t *hist = at(L.r.hist), *base = at(L.r.base), *cstart = at(L.r.cstart);
  int32_t *ids = at(L.ids), *counts = at(L.counts), *offsets = at(L.offsets);
  int32_t *perm = at(L.perm), *inv = at(L.inv);
  float* wts = reinterpret_cast<float*>(ws + L.wts);
  if (p->mx) return mx_forward(p, L, ws, x, x_scales, router_logits, T, top_k, y, st);
  uint16_t* xperm = reinterpret_cast<uint16_t*>(ws + L.xperm);
  uint16_t* h = reinterpret_cast<uint16_t*>(ws + L.h);
  float* h32 = reinterpret_cast<float*>(ws + L.h32);
  float* o = reinterpret_cast<float*>(ws + L.o);
  int* err = status_word();
  const int64_t P = static_cast<int64_t>(T) * top_k;
  const int chunk = gemm_chunk_max(T);
  const int sms = device_sm_count();

  struct StageOff {  // the hand-over covers exactly one forward call
    ~StageOff() { t_stage_on = false; }
  } stage_off;
  stage_mark(0, st);
  cudaError_t e = route_permute(router_logits, T, p->E, top_k, chunk, hist, base, ids, wts,
                                counts, offsets, cstart, perm, inv, err, st);
  if (e == cudaSuccess)
    e = launch_gather(inv, T, top_k, x, x_scales, p->K, p->act_mode, xperm, err, st);
  stage_mark(3, st);
  if (e != cudaSuccess) return FP4MOE_ERR_CUDA;

  GemmArgs a1{};
  a1.wpack = p->w13; a1.alpha = p->alpha; a1.offsets = offsets; a1.cstart = cstart;
  a1.err = err; a1.rows = P; a1.E = p->E; a1.nblocks = 2 * p->I / kTileN;
  a1.ksteps = p->K / kTileK;
  a1.tile_bytes = tile_bytes(p->gran); a1.gran = p->gran; a1.smul = p->smul;
  a1.sadd = p->sadd; a1.ldo = p->I;
  if (p->act_mode == FP4MOE_ACT_BF16) {
    a1.out = h;
    a1.mode = kGemmModeFc1;
  } else {
    a1.out = h32;
    a1.mode = kGemmModeFc1Fp8;
  }
  GemmArgs a2 = a1;
  a2.wpack = p->w2; a2.alpha = p->alpha + p->E; a2.nblocks = p->K / kTileN;
  a2.ksteps = p->I / kTileK; a2.out = o; a2.ldo = p->K; a2.mode = kGemmModeFc2;
  // Many tokens per expert: the CTA-pair kernel where the block and step
  // counts split evenly, else the one-CTA kernel.  Each has its own box rows.
  const bool pair1 = chunk > 32 && gemm_pair_supported(a1);
  const bool pair2 = chunk > 32 && gemm_pair_supported(a2);
  CUtensorMap tm_x, tm_h;
  if (!make_row_tmap(&tm_x, xperm, P, p->K,
                     static_cast<uint32_t>(pair1 ? kPairBoxRows : gemm_box_rows(chunk))) ||
      !make_row_tmap(&tm_h, h, P, p->I,
                     static_cast<uint32_t>(pair2 ? kPairBoxRows : gemm_box_rows(chunk))))
    return FP4MOE_ERR_CUDA;
  e = pair1 ? launch_gemm_pair(tm_x, a1, sms, st) : launch_gemm(tm_x, a1, chunk, sms, st);
  stage_mark(4, st);
  if (e == cudaSuccess && p->act_mode == FP4MOE_ACT_FP8)
    e = launch_h_fp8_round(h32, P, p->I, h, st);
  stage_mark(5, st);
  if (e == cudaSuccess)
    e = pair2 ? launch_gemm_pair(tm_h, a2, sms, st) : launch_gemm(tm_h, a2, chunk, sms, st);
  stage_mark(6, st);
  if (e == cudaSuccess)
    e = launch_combine(o, inv, wts, T, top_k, p->K, static_cast<uint16_t*>(y), err, st);
  stage_mark(7, st);
  return cuda_status(e);
}

size_t fp4moe_moe_workspace_size_host(const fp4moe_packed* p, int T, int top_k) {
  const size_t base = fp4moe_moe_workspace_size(p, T, top_k);
  if (base == 0) return 0;
  const size_t TK = static_cast<size_t>(T) * p->K;
  const size_t xb = (p->act_mode == FP4MOE_ACT_FP8) ? TK : 2 * TK;
  const size_t sb = (p->act_mode == FP4MOE_ACT_FP8) ? TK / 32 : 0;
  return base + align_up(xb) + align_up(sb) + align_up(static_cast<size_t>(T) * p->E * 4) +
         align_up(2 * TK);
}

int fp4moe_moe_forward_host(const void* x_host, const uint8_t* x_scales_host,
                            const float* logits_host, int T,
                            const fp4moe_packed* p, int top_k, void* y_host,
                            void* workspace, size_t ws_bytes, void* stream) {
  if (!p || T < 0 || top_k < 1 || top_k > std::min(p->E, kMaxTopK))
    return FP4MOE_ERR_INVALID_ARG;
  if (T == 0) return FP4MOE_OK;
  if (!x_host || !logits_host || !y_host || !workspace) return FP4MOE_ERR_INVALID_ARG;
  if ((p->act_mode == FP4MOE_ACT_FP8) != (x_scales_host != nullptr))
    return FP4MOE_ERR_INVALID_ARG;
  const size_t need = fp4moe_moe_workspace_size_host(p, T, top_k);
  if (ws_bytes < need) return FP4MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(workspace, kAlign)) return FP4MOE_ERR_INVALID_ARG;
  const size_t base = fp4moe_moe_workspace_size(p, T, top_k);
  const size_t TK = static_cast<size_t>(T) * p->K;
  const size_t xb = (p->act_mode == FP4MOE_ACT_FP8) ? TK : 2 * TK;
  const size_t sb = (p->act_mode == FP4MOE_ACT_FP8) ? TK / 32 : 0;
  const size_t lb = static_cast<size_t>(T) * p->E * 4;
  char* ws = static_cast<char*>(workspace);
  char* dx = ws + base;
  char* ds = dx + align_up(xb);
  char* dl = ds + align_up(sb);
  char* dy = dl + align_up(lb);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(dx, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return FP4MOE_ERR_CUDA;
  if (sb && cudaMemcpyAsync(ds, x_scales_host, sb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return FP4MOE_ERR_CUDA;
  if (cudaMemcpyAsync(dl, logits_host, lb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return FP4MOE_ERR_CUDA;
  const int rc = fp4moe_moe_forward(dx, sb ? reinterpret_cast<uint8_t*>(ds) : nullptr,
                                    reinterpret_cast<float*>(dl), T, p, top_k, dy, ws,
                                    base, stream);
  if (rc != FP4MOE_OK) return rc;
  if (cudaMemcpyAsync(y_host, dy, 2 * TK, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FP4MOE_ERR_CUDA;
  return FP4MOE_OK;
}

}  // extern "C"
