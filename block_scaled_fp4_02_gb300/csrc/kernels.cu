// Memory-bound kernels of the block-scaled FP4 MoE path (sm_103a): the
// group16 -> group32 requant, FP8 activation quantization, routing, the
// expert-major permutation and activation gather, the weighted combine, and
// the weight packing of prepare_weights.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;

int num_sms() { return device_sm_count(); }

// ================================================================ requant
//
// group16 -> group32 requant ("glm52_nvfp4_group16_notes.md", section
// "Requantization path").  One thread owns one 32-element group: 16 bytes of
// codes and two E4M3 scales in, 16 bytes of codes and one UE8M0 byte out.
// The codes are widened to exact f16 pairs with the hardware E2M1
// conversion, the group maximum |e2m1| * |s| picks the UE8M0 exponent e, each
// half is multiplied by s / 2^e in f16 (exact: at most six significant bits)
// and converted back with round-to-nearest-even, which keeps the sign (also
// of zero) and flips it for a negative scale.

// Four packed E2M1 pairs (the bytes of w) -> four f16x2 (exact).
__device__ __forceinline__ void e2m1x8_to_f16x8(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Four f16x2 -> four packed E2M1 pairs (RNE, saturating; sign of zero kept).
__device__ __forceinline__ uint32_t f16x8_to_e2m1x8(const uint32_t (&h)[4]) {
  uint32_t w;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f16x2 b0, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f16x2 b1, %2;\n\t"
      "cvt.rn.satfinite.e2m1x2.f16x2 b2, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f16x2 b3, %4;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(w)
      : "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]));
  return w;
}

__device__ __forceinline__ uint32_t hmax_abs2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ void requant_group(uint4 d, uint32_t sc, uint4& o,
                                              uint32_t& byte, int* err) {
  const uint32_t sb0 = sc & 0xFFu, sb1 = sc >> 8;
  if ((sb0 & 0x7Fu) == 0x7Fu || (sb1 & 0x7Fu) == 0x7Fu) {
    record_error(err, FP4MOE_ERR_INVALID_ARG);
    o = make_uint4(0, 0, 0, 0);
    byte = 0xFFu;
    return;
  }
  // Elements as exact f16 pairs (first half: words x, y; second: z, w).
  uint32_t hx[4], hy[4], hz[4], hw[4];
  e2m1x8_to_f16x8(d.x, hx);
  e2m1x8_to_f16x8(d.y, hy);
  e2m1x8_to_f16x8(d.z, hz);
  e2m1x8_to_f16x8(d.w, hw);
  // Largest |e2m1| of each half.
  uint32_t m0 = hmax_abs2(hmax_abs2(hmax_abs2(hx[0], hx[1]), hmax_abs2(hx[2], hx[3])),
                          hmax_abs2(hmax_abs2(hy[0], hy[1]), hmax_abs2(hy[2], hy[3])));
  uint32_t m1 = hmax_abs2(hmax_abs2(hmax_abs2(hz[0], hz[1]), hmax_abs2(hz[2], hz[3])),
                          hmax_abs2(hmax_abs2(hw[0], hw[1]), hmax_abs2(hw[2], hw[3])));
  const float2 mm0 = __half22float2(*reinterpret_cast<__half2*>(&m0));
  const float2 mm1 = __half22float2(*reinterpret_cast<__half2*>(&m1));
  const float2 s = e4m3x2_to_f32x2(sc);
  const float amax = fmaxf(fmaxf(fabsf(mm0.x), fabsf(mm0.y)) * fabsf(s.x),
                           fmaxf(fabsf(mm1.x), fabsf(mm1.y)) * fabsf(s.y));
  int e = 0;
  if (amax > 0.0f) {
    const uint32_t bits = __float_as_uint(amax);
    const int E = static_cast<int>(bits >> 23) - 127;
    e = ((bits & 0x7FFFFFu) <= 0x400000u) ? E - 2 : E - 1;
  }
  e = max(-126, min(127, e));
  byte = static_cast<uint32_t>(e + 127);
  // s / 2^e per half as an f16 pair: exact, since e is in [-13, 9] for any
  // finite non-zero group and s has at most four significant bits.  A half
  // with nonzero codes has |s| / 2^e <= 12; an all-zero half may exceed f16
  // range, so the factor is clamped to +-16 (its products stay +-0).
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
  const __half2 f = __floats2half2_rn(fminf(fmaxf(s.x * inv, -16.0f), 16.0f),
                                      fminf(fmaxf(s.y * inv, -16.0f), 16.0f));
  const uint32_t fb = *reinterpret_cast<const uint32_t*>(&f);
  const uint32_t f0 = __byte_perm(fb, fb, 0x1010), f1 = __byte_perm(fb, fb, 0x3232);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    hx[i] = hmul2(hx[i], f0);
    hy[i] = hmul2(hy[i], f0);
    hz[i] = hmul2(hz[i], f1);
    hw[i] = hmul2(hw[i], f1);
  }
  o.x = f16x8_to_e2m1x8(hx);
  o.y = f16x8_to_e2m1x8(hy);
  o.z = f16x8_to_e2m1x8(hz);
  o.w = f16x8_to_e2m1x8(hw);
}

// Each thread takes kRqUnroll groups per iteration with all loads issued
// first, so that enough bytes are in flight to cover HBM latency.
constexpr int kRqUnroll = 4;

__global__ void __launch_bounds__(256) requant_kernel(
    const uint8_t* __restrict__ fp4, const uint8_t* __restrict__ s16,
    int64_t groups, uint8_t* __restrict__ out, uint8_t* __restrict__ s32,
    int* err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       g0 < groups; g0 += kRqUnroll * stride) {
    uint4 d[kRqUnroll];
    uint32_t sc[kRqUnroll];
#pragma unroll
    for (int i = 0; i < kRqUnroll; ++i) {
      const int64_t g = g0 + i * stride;
      if (g < groups) {
        d[i] = __ldcs(reinterpret_cast<const uint4*>(fp4) + g);
        sc[i] = __ldcs(reinterpret_cast<const uint16_t*>(s16) + g);
      }
    }
#pragma unroll
    for (int i = 0; i < kRqUnroll; ++i) {
      const int64_t g = g0 + i * stride;
      if (g < groups) {
        uint4 o;
        uint32_t byte;
        requant_group(d[i], sc[i], o, byte, err);
        __stcs(reinterpret_cast<uint4*>(out) + g, o);
        s32[g] = static_cast<uint8_t>(byte);
      }
    }
  }
}

// ============================================================== act quant
//
// Recipe (1,1,32) of the group16 notes page: per token and 32 consecutive K
// elements, UE8M0 e = min{e : amax <= 448 * 2^e}, q = E4M3(x / 2^e).

__global__ void __launch_bounds__(256) act_quant_kernel(
    const uint16_t* __restrict__ x, int64_t groups, uint8_t* __restrict__ q,
    uint8_t* __restrict__ s, int* err) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       g < groups; g += stride) {
    const uint4* src = reinterpret_cast<const uint4*>(x + g * 32);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = src[i];
      w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    if (!(amax <= 3.402823466e38f)) {  // inf or NaN
      record_error(err, FP4MOE_ERR_INVALID_ARG);
      amax = 0.0f;
    }
    const uint32_t byte = ue8m0_for_e4m3(amax);
    const int e = static_cast<int>(byte) - 127;   // <= 120 for bf16 inputs
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t lo = f32x2_to_e4m3x2(bf16_lo(w[2 * i]) * inv,
                                          bf16_hi(w[2 * i]) * inv);
      const uint32_t hi = f32x2_to_e4m3x2(bf16_lo(w[2 * i + 1]) * inv,
                                          bf16_hi(w[2 * i + 1]) * inv);
      o[i] = lo | (hi << 16);
    }
    uint4* dst = reinterpret_cast<uint4*>(q + g * 32);
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    s[g] = static_cast<uint8_t>(byte);
  }
}

// FP8 rounding of the FC1 output h (FP8 activation path): per row and 32
// consecutive columns, the same UE8M0 + E4M3 rule as the activation
// quantization, stored back as the exact bf16 value q * 2^e for FC2.
__global__ void __launch_bounds__(256) h_fp8_round_kernel(
    const float* __restrict__ h, int64_t groups, uint16_t* __restrict__ out) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       g < groups; g += stride) {
    const float4* src = reinterpret_cast<const float4*>(h + g * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 t = src[i];
      v[4 * i] = t.x, v[4 * i + 1] = t.y, v[4 * i + 2] = t.z, v[4 * i + 3] = t.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const int e = static_cast<int>(ue8m0_for_e4m3(amax)) - 127;
    const float inv = pow2_any(-e), sc = pow2_any(e);
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 q = e4m3x2_to_f32x2(f32x2_to_e4m3x2(v[2 * i] * inv, v[2 * i + 1] * inv));
      o[i] = pack_bf16x2(q.x * sc, q.y * sc);
    }
    uint4* dst = reinterpret_cast<uint4*>(out + g * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
  }
}

// ================================================================ routing
//
// Softmax top-k with renormalised weights.  One warp per token; each lane
// holds EPL logits (expert lane + 32 i).  k rounds of a warp arg-max
// (larger value wins, equal values go to the lower expert id) select the
// experts on the raw logits; w_j = exp(l_j - l_0) / sum over the k.

// Top-k of token t by one warp: lane j < k receives the j-th expert and its
// renormalised weight.
template <int EPL>
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int t, int E,
                                            int k, int lane, int* err, int& my_id,
                                            float& my_w) {
  float v[EPL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      v[i] = logits[static_cast<int64_t>(t) * E + e];
      if (v[i] != v[i]) {
        record_error(err, FP4MOE_ERR_INVALID_ARG);
        v[i] = -INFINITY;
      }
    } else {
      v[i] = -INFINITY;
      taken |= 1u << i;
    }
  }
  float my_v = 0.0f;
  my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7FFFFFFF;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (!((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
        bv = v[i];
        bi = e;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, off);
      const int oi = __shfl_xor_sync(kFull, bi, off);
      if (ov > bv || (ov == bv && oi < bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == j) {
      my_v = bv;
      my_id = bi;
    }
  }
  const float v0 = __shfl_sync(kFull, my_v, 0);
  const float ex = (lane < k) ? expf(my_v - v0) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
  my_w = ex / sum;
}

template <int EPL>
__global__ void __launch_bounds__(1024) route_kernel(
    const float* __restrict__ logits, int T, int E, int k,
    int32_t* __restrict__ ids, float* __restrict__ w,
    int32_t* __restrict__ hist, int* err) {
  __shared__ int cnt[kMaxE];
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTokPerBlk + warp;
  if (t < T && warp < kTokPerBlk) {
    int my_id;
    float my_w;
    route_token<EPL>(logits, t, E, k, lane, err, my_id, my_w);
    if (lane < k && in_bounds(err, my_id, E)) {
      ids[static_cast<int64_t>(t) * k + lane] = my_id;
      w[static_cast<int64_t>(t) * k + lane] = my_w;
      atomicAdd(&cnt[my_id], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    hist[static_cast<int64_t>(blockIdx.x) * E + e] = cnt[e];
}

// Exclusive block scan over blockDim.x (== 1024) values; returns the
// exclusive prefix and writes the total to *total.
__device__ int block_exclusive_scan(int v, int* total) {
  __shared__ int wsum[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(kFull, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = wsum[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, s, off);
      if (lane >= off) s += y;
    }
    wsum[lane] = s;
  }
  __syncthreads();
  const int incl = x + (warp > 0 ? wsum[warp - 1] : 0);
  *total = wsum[31];
  __syncthreads();
  return incl - v;
}

__global__ void __launch_bounds__(1024) scan_kernel(
    int nblk, int E, const int32_t* __restrict__ hist, int32_t* __restrict__ base,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ cstart, int chunk_max) {
  const int e = threadIdx.x;
  int tot = 0;
  if (e < E)
    for (int b = 0; b < nblk; ++b) tot += hist[static_cast<int64_t>(b) * E + e];
  int total;
  const int off = block_exclusive_scan(e < E ? tot : 0, &total);
  const int nch = (e < E) ? (tot + chunk_max - 1) / chunk_max : 0;
  int ctotal;
  const int coff = block_exclusive_scan(nch, &ctotal);
  if (e < E) {
    counts[e] = tot;
    offsets[e] = off;
    cstart[e] = coff;
    int run = off;
    for (int b = 0; b < nblk; ++b) {
      const int64_t i = static_cast<int64_t>(b) * E + e;
      const int c = hist[i];
      base[i] = run;
      run += c;
    }
  }
  if (e == 0) {
    offsets[E] = total;
    cstart[E] = ctotal;
  }
}

// Routing, scan and stable scatter of at most kTokPerBlk tokens in one
// launch (the three kernels above and below do the same for any T, in
// three): one warp per token as in route_kernel, the expert counts in
// shared memory, the two block scans of scan_kernel, and the rank of pair p
// among the pairs of its expert = the number of lower-indexed pairs of that
// expert, so every output equals the three-kernel path's bit for bit.
template <int EPL>
__global__ void __launch_bounds__(1024) route_small_kernel(
    const float* __restrict__ logits, int T, int E, int k, int chunk_max,
    int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ cstart,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int* err) {
  __shared__ int cnt[kMaxE];
  __shared__ int pid[kTokPerBlk * kMaxTopK];   // expert of each pair, -1 if invalid
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp < T) {
    int my_id;
    float my_w;
    route_token<EPL>(logits, warp, E, k, lane, err, my_id, my_w);
    if (lane < k) {
      const bool ok = in_bounds(err, my_id, E);
      pid[warp * k + lane] = ok ? my_id : -1;
      if (ok) {
        ids[warp * k + lane] = my_id;
        w[warp * k + lane] = my_w;
        atomicAdd(&cnt[my_id], 1);
      }
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int tot = e < E ? cnt[e] : 0;
  int total;
  const int off = block_exclusive_scan(tot, &total);
  const int nch = (e < E) ? (tot + chunk_max - 1) / chunk_max : 0;
  int ctotal;
  const int coff = block_exclusive_scan(nch, &ctotal);
  if (e < E) {
    counts[e] = tot;
    offsets[e] = off;
    cstart[e] = coff;
  }
  if (e == 0) {
    offsets[E] = total;
    cstart[E] = ctotal;
  }
  __syncthreads();                 // every count read before cnt becomes the base
  if (e < E) cnt[e] = off;
  __syncthreads();
  const int P = T * k;
  const int p = threadIdx.x;
  if (p < P && pid[p] >= 0) {
    const int ep = pid[p];
    int rank = 0;
    for (int q = 0; q < p; ++q) rank += (pid[q] == ep) ? 1 : 0;
    const int pos = cnt[ep] + rank;
    if (in_bounds(err, pos, P)) {
      perm[pos] = p;
      inv[p] = pos;
    }
  }
}

// Stable scatter: within block b (tokens [32b, 32b+32)), the rank of pair p
// among the block's pairs of the same expert is the number of lower-indexed
// pairs of that expert: earlier warps (per-warp counts in shared memory) plus
// lower lanes of this warp (match mask).
__global__ void __launch_bounds__(512) scatter_kernel(
    const int32_t* __restrict__ ids, int T, int E, int k,
    const int32_t* __restrict__ base, int32_t* __restrict__ perm,
    int32_t* __restrict__ inv, int* err) {
  extern __shared__ int wcnt[];   // [16 warps][E]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t P = static_cast<int64_t>(T) * k;
  const int64_t p0 = static_cast<int64_t>(blockIdx.x) * kTokPerBlk * k;
  const int np = static_cast<int>(min(P - p0, static_cast<int64_t>(kTokPerBlk) * k));
  for (int i = tid; i < 16 * E; i += blockDim.x) wcnt[i] = 0;
  __syncthreads();
  bool act = tid < np;
  const int e = act ? ids[p0 + tid] : -1;
  if (act && !in_bounds(err, e, E)) act = false;
  const unsigned m = __match_any_sync(kFull, e);
  const int rank = __popc(m & ((1u << lane) - 1u));
  if (act && rank == 0) wcnt[warp * E + e] = __popc(m);
  __syncthreads();
  if (act) {
    int pre = 0;
    for (int w2 = 0; w2 < warp; ++w2) pre += wcnt[w2 * E + e];
    const int pos = base[static_cast<int64_t>(blockIdx.x) * E + e] + pre + rank;
    if (in_bounds(err, pos, P)) {
      perm[pos] = static_cast<int32_t>(p0 + tid);
      inv[p0 + tid] = pos;
    }
  }
}

// Activation gather: row p of the pair list goes to expert-major slot inv[p]
// (blocks (p, c) for c < gridDim.y share a row's 16-byte groups c,
// c + gridDim.y, ...; grid-stride over rows), as bf16; FP8 inputs are
// dequantized exactly on the way.
__global__ void __launch_bounds__(256) gather_kernel(
    const int32_t* __restrict__ inv, int64_t P, int k, const void* __restrict__ x,
    const uint8_t* __restrict__ xs, int K, int act_mode, uint16_t* __restrict__ xperm,
    int* err) {
  const int c0 = blockIdx.y * blockDim.x + threadIdx.x, cs = gridDim.y * blockDim.x;
  for (int64_t p = blockIdx.x; p < P; p += gridDim.x) {
    const int64_t t = p / k;
    const int64_t row = inv[p];
    if (!in_bounds(err, row, P)) continue;
    uint4* dst = reinterpret_cast<uint4*>(xperm + row * K);
    if (act_mode == FP4MOE_ACT_BF16) {
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + t * K);
      for (int c = c0; c < K / 8; c += cs) dst[c] = __ldg(src + c);
    } else {
      // FP8: bf16(e4m3 * 2^(xs - 127)), exact for scaled values in the
      // bf16 normal range.
      const uint2* src = reinterpret_cast<const uint2*>(static_cast<const uint8_t*>(x) + t * K);
      const uint8_t* srow = xs + t * (K / 32);
      for (int c = c0; c < K / 8; c += cs) {
        const uint2 q = src[c];
        const uint32_t sb = srow[c / 4];
        const float sc = (sb == 0)     ? __uint_as_float(0x00400000u)
                         : (sb == 255) ? __uint_as_float(0x7FC00000u)
                                       : __uint_as_float(sb << 23);
        const float2 a = e4m3x2_to_f32x2(q.x), b = e4m3x2_to_f32x2(q.x >> 16);
        const float2 c2 = e4m3x2_to_f32x2(q.y), d2 = e4m3x2_to_f32x2(q.y >> 16);
        dst[c] = make_uint4(pack_bf16x2(a.x * sc, a.y * sc), pack_bf16x2(b.x * sc, b.y * sc),
                            pack_bf16x2(c2.x * sc, c2.y * sc),
                            pack_bf16x2(d2.x * sc, d2.y * sc));
      }
    }
  }
}

// ================================================================ combine

__global__ void __launch_bounds__(256) combine_kernel(
    const float* __restrict__ o, const int32_t* __restrict__ inv,
    const float* __restrict__ w, int k, int K, uint16_t* __restrict__ y, int* err) {
  const int64_t t = blockIdx.x;
  int pos[kMaxTopK];
  float wt[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      pos[j] = inv[t * k + j];
      wt[j] = w[t * k + j];
      // bounds-checked build: a slot outside [0, P) reads row 0 instead
      if (!in_bounds(err, pos[j], static_cast<int64_t>(gridDim.x) * k)) pos[j] = 0;
    }
  }
  // Block (t, c) takes the 8-column groups c, c + gridDim.y, ... of token t.
  const int stride = gridDim.y * blockDim.x * 8;
  for (int n = (blockIdx.y * blockDim.x + threadIdx.x) * 8; n < K; n += stride) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (j < k) {
        const float4* row =
            reinterpret_cast<const float4*>(o + static_cast<int64_t>(pos[j]) * K + n);
        const float4 a = row[0], b = row[1];
        acc[0] = fmaf(wt[j], a.x, acc[0]);
        acc[1] = fmaf(wt[j], a.y, acc[1]);
        acc[2] = fmaf(wt[j], a.z, acc[2]);
        acc[3] = fmaf(wt[j], a.w, acc[3]);
        acc[4] = fmaf(wt[j], b.x, acc[4]);
        acc[5] = fmaf(wt[j], b.y, acc[5]);
        acc[6] = fmaf(wt[j], b.z, acc[6]);
        acc[7] = fmaf(wt[j], b.w, acc[7]);
      }
    }
    *reinterpret_cast<uint4*>(y + t * K + n) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                   pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
  }
}

// ================================================================ prepare
//
// Packed tile (e, nb, ks): 128 weight rows x 64 K elements, contiguous:
//   [0, 4096)      E2M1 data: [2 halves of 32 K][128 rows][16 bytes]; each
//                  16-byte row half is 4 words of 8 elements whose bits are
//                  placed so that the GEMM's dequantizer needs only shifts
//                  and masks (see dequant8 in gemm.cu);
//   [4096, ...)    scale codes: [128 rows][64 / gran bytes].
// FC1 tiles interleave gate and up rows: in row r = 32 q + l, l < 16 is gate
// row i = 64 nb + 16 q + l and l >= 16 is up row i = 64 nb + 16 q + (l - 16).
// Scale codes: gran 16 -> c with bf16(s * 2^119) = c * 16 + 0x7680 (the E4M3
// exponent renormalised so subnormal scales are exact; a negative scale
// flips the codes' signs; a zero scale zeroes the codes); gran 32 ->
// c = b - bmax + 254 with bf16 bits c * 128 (scales more than 2^126 below the
// matrix maximum flush to zero).

// Bit positions of element j (k offset 0..7) in a packed word, for its
// magnitude bits m, e0, e1 (E2M1 bits 0..2) and its sign.  The dequantizer
// extracts the four bf16 pairs (s, e1, e0, m at bits 15, 8, 7, 6 and 31, 24,
// 23, 22) as: elements 0, 1 by one right shift (m) and the word itself (the
// rest); 2, 3 by a left shift of 6; 4, 5 by a rotate of 12; 6, 7 by a left
// shift of 2, each followed by one mask: seven logic operations per eight
// elements, the fewest of any layout with this extraction pattern.
__constant__ uint8_t kBitPos[8][4] = {
    {14, 7, 8, 15},  {30, 23, 24, 31}, {0, 1, 2, 9},    {16, 17, 18, 25},
    {26, 27, 28, 3}, {10, 11, 12, 19}, {4, 5, 6, 13},   {20, 21, 22, 29}};

__device__ __forceinline__ uint32_t pack8(const uint8_t* c) {
  uint32_t x = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int b = 0; b < 4; ++b)
      x |= static_cast<uint32_t>((c[j] >> b) & 1u) << kBitPos[j][b];
  return x;
}

__global__ void scale_max_kernel(const uint8_t* __restrict__ s,
                                 int64_t per_expert, int32_t* bmax, int* err) {
  const int e = blockIdx.y;
  const uint8_t* p = s + static_cast<int64_t>(e) * per_expert;
  int m = 0;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       i < per_expert; i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int b = p[i];
    if (b == 255)
      record_error(err, FP4MOE_ERR_INVALID_ARG);
    else
      m = max(m, b);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = max(m, __shfl_xor_sync(kFull, m, off));
  if ((threadIdx.x & 31) == 0) atomicMax(bmax + e, m);
}

__global__ void __launch_bounds__(128) pack_kernel(
    const uint8_t* __restrict__ w, const uint8_t* __restrict__ s, int E, int N,
    int Kd, int gran, int gated, int layout, const int32_t* __restrict__ bmax,
    uint8_t* __restrict__ out, int* err) {
  const int nblocks = N / kTileN, ksteps = Kd / kTileK;
  const int64_t tile = blockIdx.x;
  const int r = threadIdx.x;
  const int ks = static_cast<int>(tile % ksteps);
  const int64_t t2 = tile / ksteps;
  const int nb = static_cast<int>(t2 % nblocks);
  const int e = static_cast<int>(t2 / nblocks);
  int src;
  if (gated) {
    const int I = N / 2, q = r >> 5, l = r & 31;
    const int i = 64 * nb + 16 * q + (l & 15);
    const int gate0 = (layout == FP4MOE_W13_GATE_UP) ? 0 : I;
    const int up0 = (layout == FP4MOE_W13_GATE_UP) ? I : 0;
    src = ((l < 16) ? gate0 : up0) + i;
  } else {
    src = kTileN * nb + r;
  }
  const int64_t row = static_cast<int64_t>(e) * N + src;
  const uint4* wsrc =
      reinterpret_cast<const uint4*>(w + row * (Kd / 2) + ks * (kTileK / 2));
  const uint4 b0 = wsrc[0], b1 = wsrc[1];
  const uint32_t bw[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
  uint8_t codes[64];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) codes[8 * i + j] = (bw[i] >> (4 * j)) & 0xFu;
  const int ng = kTileK / gran;
  const uint8_t* srow = s + row * (Kd / gran) + ks * ng;
  uint8_t* tp = out + tile * tile_bytes(gran);
  for (int g = 0; g < ng; ++g) {
    const uint32_t sb = srow[g];
    uint32_t code = 0;
    bool zero = false, neg = false;
    if (gran == 16) {
      const uint32_t v = sb & 0x7Fu;
      neg = (sb & 0x80u) != 0;
      if (v == 0x7Fu) {
        record_error(err, FP4MOE_ERR_INVALID_ARG);
        zero = true;
      } else if (v == 0) {
        zero = true;
      } else if (v >= 8) {
        code = v + 16;                          // normal: exponent + 2
      } else {
        const int msb = 31 - __clz(v);           // subnormal m * 2^-9
        code = static_cast<uint32_t>((msb << 3) | ((v << (3 - msb)) & 7u));
      }
    } else {
      if (sb == 0xFFu) {
        record_error(err, FP4MOE_ERR_INVALID_ARG);
        zero = true;
      } else {
        const int bm = bmax[e];
        code = (static_cast<int>(sb) >= bm - 126)
                   ? static_cast<uint32_t>(static_cast<int>(sb) - bm + 254)
                   : 0u;
      }
    }
    for (int i = g * gran; i < (g + 1) * gran; ++i) {
      if (zero) codes[i] = 0;
      else if (neg) codes[i] ^= 8u;
    }
    tp[kTileDataBytes + r * ng + g] = static_cast<uint8_t>(code);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 o;
    o.x = pack8(codes + 32 * h + 0);
    o.y = pack8(codes + 32 * h + 8);
    o.z = pack8(codes + 32 * h + 16);
    o.w = pack8(codes + 32 * h + 24);
    *reinterpret_cast<uint4*>(tp + h * 2048 + r * 16) = o;
  }
}

__global__ void alpha_kernel(const float* __restrict__ gs,
                             const int32_t* __restrict__ bmax, int E, int gran,
                             int inverted, float* __restrict__ alpha) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const float g = inverted ? 1.0f / gs[e] : gs[e];   // IEEE division
  alpha[e] = (gran == 16) ? g * 128.0f : (gran == 32) ? ldexpf(g, bmax[e] - 128) : g;
}

// ============================================= block-scaled (FP8 x FP4) path
//
// Weights for kind::mxf8f6f4 stay plain E2M1 codes, two per byte (the TMA
// widens them on the way into shared memory); only the rows are reordered
// and the UE8M0 scales regrouped.  FC1 rows of block b (128 intermediate
// columns): gate rows 128 b .. 128 b + 127 at 256 b, the up rows of the same
// columns at 256 b + 128.  Scale words: one 32-bit word per row and 128-wide
// K step holding the four UE8M0 bytes of its 32-wide blocks, ordered
// [expert][128-row tile][step][row].

// One block per destination row (gated: reordered), 16 bytes per thread.
__global__ void __launch_bounds__(256) mx_rows_kernel(
    const uint8_t* __restrict__ w, int N, int64_t row_bytes, int gated,
    int layout, uint8_t* __restrict__ out) {
  const int64_t R = blockIdx.x;                  // destination row (all experts)
  const int e = static_cast<int>(R / N), r = static_cast<int>(R % N);
  int src = r;
  if (gated) {
    const int I = N / 2, b = r >> 8, t = (r >> 7) & 1, rr = r & 127;
    const int gate0 = (layout == FP4MOE_W13_GATE_UP) ? 0 : I;
    const int up0 = (layout == FP4MOE_W13_GATE_UP) ? I : 0;
    src = (t ? up0 : gate0) + 128 * b + rr;
  }
  const uint4* s4 = reinterpret_cast<const uint4*>(w + (static_cast<int64_t>(e) * N + src) * row_bytes);
  uint4* d4 = reinterpret_cast<uint4*>(out + R * row_bytes);
  for (int64_t c = threadIdx.x; c < row_bytes / 16; c += blockDim.x) d4[c] = s4[c];
}

// One thread per (expert, destination row, step): four scale bytes -> word.
__global__ void __launch_bounds__(256) mx_scales_kernel(
    const uint8_t* __restrict__ s, int E, int N, int ksteps, int gated,
    int layout, uint32_t* __restrict__ out, int* err) {
  const int64_t n = static_cast<int64_t>(E) * N * ksteps;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int r = static_cast<int>(idx % 128);
    const int64_t rest = idx / 128;
    const int ks = static_cast<int>(rest % ksteps);
    const int64_t tg = rest / ksteps;            // tile over all experts
    const int tiles = N / 128;
    const int e = static_cast<int>(tg / tiles), tile = static_cast<int>(tg % tiles);
    const int R = 128 * tile + r;                 // destination row in the expert
    int src = R;
    if (gated) {
      const int I = N / 2, b = R >> 8, t = (R >> 7) & 1, rr = R & 127;
      const int gate0 = (layout == FP4MOE_W13_GATE_UP) ? 0 : I;
      const int up0 = (layout == FP4MOE_W13_GATE_UP) ? I : 0;
      src = (t ? up0 : gate0) + 128 * b + rr;
    }
    const uint32_t word = __ldg(reinterpret_cast<const uint32_t*>(
        s + (static_cast<int64_t>(e) * N + src) * (4 * ksteps)) + ks);
    // UE8M0 0xFF is NaN: reject.
    if (((word & 0xFFu) == 0xFFu) || (((word >> 8) & 0xFFu) == 0xFFu) ||
        (((word >> 16) & 0xFFu) == 0xFFu) || ((word >> 24) == 0xFFu))
      record_error(err, FP4MOE_ERR_INVALID_ARG);
    out[idx] = word;
  }
}

// Activation gather of the block-scaled path: row p of the pair list goes to
// expert-major slot inv[p] as E4M3 bytes, and its UE8M0 scale words to
// xs_perm[step][inv[p]].
__global__ void __launch_bounds__(256) gather_mx_kernel(
    const int32_t* __restrict__ inv, int64_t P, int k, const uint8_t* __restrict__ x,
    const uint8_t* __restrict__ xs, int K, int64_t pitch, uint8_t* __restrict__ xperm,
    uint32_t* __restrict__ xsperm, int* err) {
  for (int64_t p = blockIdx.x; p < P; p += gridDim.x) {
    const int64_t t = p / k;
    const int64_t row = inv[p];
    if (!in_bounds(err, row, P) || !in_bounds(err, row, pitch)) continue;
    const uint4* src = reinterpret_cast<const uint4*>(x + t * K);
    uint4* dst = reinterpret_cast<uint4*>(xperm + row * K);
    for (int c = threadIdx.x; c < K / 16; c += blockDim.x) dst[c] = __ldg(src + c);
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(xs + t * (K / 32));
    for (int c = threadIdx.x; c < K / 128; c += blockDim.x) xsperm[c * pitch + row] = __ldg(sw + c);
  }
}

}  // namespace

// ============================================================== launchers

cudaError_t launch_requant(const uint8_t* fp4, const uint8_t* s16,
                           int64_t rows, int64_t K, uint8_t* fp4_out,
                           uint8_t* s32_out, int* err, cudaStream_t st) {
  const int64_t groups = rows * (K / 32);
  if (groups == 0) return cudaSuccess;
  const int64_t want = (groups + 256 * kRqUnroll - 1) / (256 * kRqUnroll);
  const int blocks = static_cast<int>(std::min<int64_t>(want, num_sms() * 8));
  requant_kernel<<<blocks, 256, 0, st>>>(fp4, s16, groups, fp4_out, s32_out,
                                         err);
  return cudaGetLastError();
}

cudaError_t launch_act_quant(const uint16_t* x, int64_t T, int64_t K,
                             uint8_t* xq, uint8_t* xs, int* err,
                             cudaStream_t st) {
  const int64_t groups = T * (K / 32);
  if (groups == 0) return cudaSuccess;
  const int64_t want = (groups + 255) / 256;
  const int blocks = static_cast<int>(std::min<int64_t>(want, num_sms() * 8));
  act_quant_kernel<<<blocks, 256, 0, st>>>(x, groups, xq, xs, err);
  return cudaGetLastError();
}

cudaError_t launch_h_fp8_round(const float* h, int64_t rows, int64_t I,
                               uint16_t* out, cudaStream_t st) {
  const int64_t groups = rows * (I / 32);
  if (groups == 0) return cudaSuccess;
  const int64_t want = (groups + 255) / 256;
  const int blocks = static_cast<int>(std::min<int64_t>(want, num_sms() * 8));
  h_fp8_round_kernel<<<blocks, 256, 0, st>>>(h, groups, out);
  return cudaGetLastError();
}

cudaError_t launch_route(const float* logits, int T, int E, int k,
                         int32_t* ids, float* w, int32_t* hist, int* err,
                         cudaStream_t st) {
  const int nblk = (T + kTokPerBlk - 1) / kTokPerBlk;
  if (nblk == 0) return cudaSuccess;
  const int epl = (E + 31) / 32;
#define FP4MOE_ROUTE(N)                                                   \
  route_kernel<N><<<nblk, kTokPerBlk * 32, 0, st>>>(logits, T, E, k, ids, w, \
                                                    hist, err)
  if (epl <= 1) FP4MOE_ROUTE(1);
  else if (epl <= 2) FP4MOE_ROUTE(2);
  else if (epl <= 4) FP4MOE_ROUTE(4);
  else if (epl <= 8) FP4MOE_ROUTE(8);
  else if (epl <= 16) FP4MOE_ROUTE(16);
  else FP4MOE_ROUTE(32);
#undef FP4MOE_ROUTE
  return cudaGetLastError();
}

cudaError_t launch_route_small(const float* logits, int T, int E, int k, int chunk_max,
                               int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                               int32_t* cstart, int32_t* perm, int32_t* inv, int* err,
                               cudaStream_t st) {
  if (T < 1 || T > kTokPerBlk || k > kMaxTopK || E > kMaxE) return cudaErrorInvalidValue;
  const int epl = (E + 31) / 32;
#define FP4MOE_ROUTE_SMALL(N)                                                        \
  route_small_kernel<N><<<1, 1024, 0, st>>>(logits, T, E, k, chunk_max, ids, w, counts, \
                                            offsets, cstart, perm, inv, err)
  if (epl <= 1) FP4MOE_ROUTE_SMALL(1);
  else if (epl <= 2) FP4MOE_ROUTE_SMALL(2);
  else if (epl <= 4) FP4MOE_ROUTE_SMALL(4);
  else if (epl <= 8) FP4MOE_ROUTE_SMALL(8);
  else if (epl <= 16) FP4MOE_ROUTE_SMALL(16);
  else FP4MOE_ROUTE_SMALL(32);
#undef FP4MOE_ROUTE_SMALL
  return cudaGetLastError();
}

cudaError_t launch_scan(int T, int E, const int32_t* hist, int32_t* base,
                        int32_t* counts, int32_t* offsets, int32_t* cstart,
                        int chunk_max, cudaStream_t st) {
  const int nblk = (T + kTokPerBlk - 1) / kTokPerBlk;
  scan_kernel<<<1, 1024, 0, st>>>(nblk, E, hist, base, counts, offsets, cstart,
                                  chunk_max);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const int32_t* ids, int T, int E, int k,
                           const int32_t* base, int32_t* perm, int32_t* inv,
                           const void* x, const uint8_t* xs, int K,
                           int act_mode, uint16_t* xperm, int* err, cudaStream_t st) {
  const int nblk = (T + kTokPerBlk - 1) / kTokPerBlk;
  if (nblk == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(16) * E * sizeof(int);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(
        scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  scatter_kernel<<<nblk, 512, smem, st>>>(ids, T, E, k, base, perm, inv, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || xperm == nullptr) return e;
  return launch_gather(inv, T, k, x, xs, K, act_mode, xperm, err, st);
}

cudaError_t launch_gather(const int32_t* inv, int T, int k, const void* x, const uint8_t* xs,
                          int K, int act_mode, uint16_t* xperm, int* err, cudaStream_t st) {
  const int64_t P = static_cast<int64_t>(T) * k;
  if (P == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<int64_t>(P, static_cast<int64_t>(num_sms()) * 64));
  // Few rows: each row's 16-byte groups are split over several blocks, so
  // that about two blocks per SM copy.
  const int64_t groups = (K / 8 + 255) / 256;
  const int split = static_cast<int>(
      std::max<int64_t>(1, std::min<int64_t>(groups, (2 * num_sms() + P - 1) / P)));
  gather_kernel<<<dim3(grid, split), 256, 0, st>>>(inv, P, k, x, xs, K, act_mode, xperm, err);
  return cudaGetLastError();
}

cudaError_t launch_mx_rows(const uint8_t* w, int E, int N, int Kd, bool gated, int layout,
                           uint8_t* out, cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(E) * N;
  if (rows == 0) return cudaSuccess;
  if (rows > 0x7FFFFFFF) return cudaErrorInvalidValue;
  mx_rows_kernel<<<static_cast<unsigned>(rows), 256, 0, st>>>(w, N, Kd / 2, gated ? 1 : 0,
                                                              layout, out);
  return cudaGetLastError();
}

cudaError_t launch_mx_scales(const uint8_t* s, int E, int N, int Kd, bool gated, int layout,
                             uint32_t* out, int* err, cudaStream_t st) {
  const int64_t n = static_cast<int64_t>(E) * N * (Kd / kMxK);
  if (n == 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, num_sms() * 8));
  mx_scales_kernel<<<blocks, 256, 0, st>>>(s, E, N, Kd / kMxK, gated ? 1 : 0, layout, out,
                                           err);
  return cudaGetLastError();
}

cudaError_t launch_gather_mx(const int32_t* inv, int T, int k, const uint8_t* x,
                             const uint8_t* xs, int K, int64_t pitch, uint8_t* xperm,
                             uint32_t* xsperm, int* err, cudaStream_t st) {
  const int64_t P = static_cast<int64_t>(T) * k;
  if (P == 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<int64_t>(P, static_cast<int64_t>(num_sms()) * 64));
  gather_mx_kernel<<<grid, 256, 0, st>>>(inv, P, k, x, xs, K, pitch, xperm, xsperm, err);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float* o, const int32_t* inv, const float* w,
                           int T, int k, int K, uint16_t* y, int* err, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  // A few tokens: each token's columns are split over several blocks, so
  // that about two blocks per SM read the k rows (each output element is
  // still summed by one thread in top-k order).
  const int groups = (K + 2047) / 2048;
  const int split = std::max(1, std::min(groups, (2 * num_sms() + T - 1) / T));
  combine_kernel<<<dim3(T, split), 256, 0, st>>>(o, inv, w, k, K, y, err);
  return cudaGetLastError();
}

cudaError_t launch_scale_max(const uint8_t* s, int E, int64_t per_expert,
                             int32_t* bmax, int* err, cudaStream_t st) {
  const int bx = static_cast<int>(std::min<int64_t>((per_expert + 255) / 256, 64));
  scale_max_kernel<<<dim3(bx, E), 256, 0, st>>>(s, per_expert, bmax, err);
  return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t* w, const uint8_t* s, int E, int N,
                        int Kd, int gran, bool gated, int layout,
                        const int32_t* bmax, uint8_t* out, int* err,
                        cudaStream_t st) {
  const int64_t tiles =
      static_cast<int64_t>(E) * (N / kTileN) * (Kd / kTileK);
  if (tiles == 0) return cudaSuccess;
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidValue;
  pack_kernel<<<static_cast<unsigned>(tiles), 128, 0, st>>>(
      w, s, E, N, Kd, gran, gated ? 1 : 0, layout, bmax, out, err);
  return cudaGetLastError();
}

cudaError_t launch_alpha(const float* gs, const int32_t* bmax, int E, int gran, bool inverted,
                         float* alpha, cudaStream_t st) {
  alpha_kernel<<<(E + 255) / 256, 256, 0, st>>>(gs, bmax, E, gran, inverted ? 1 : 0, alpha);
  return cudaGetLastError();
}

}  // namespace fp4moe
