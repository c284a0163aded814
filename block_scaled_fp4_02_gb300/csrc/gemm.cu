// Grouped GEMM of the MoE expert FFN over packed block-scaled FP4 weights
// (sm_103a, tcgen05): FC1 gate|up with the SwiGLU epilogue and FC2.
//
// Formulation (weights as the UMMA M side): for each work unit (expert e,
// 128-row weight block nb, chunk of up to NT tokens of e),
//     D[128 x n] = W_tile[128 x Kd] * X_chunk[n x Kd]^T    (FP32 in TMEM)
// W is dequantized FP4 -> bf16 into shared memory in the 128-byte swizzled
// K-major layout; X (bf16 activations in expert-major order) arrives by TMA
// in the same layout.  Warp roles, one CTA per SM, persistent over units:
//   warp 0      : weight producer -- bulk copies of the packed FP4 tiles
//                 (one per 64-wide K step) into a deep ring of F stages;
//   warp 1      : TMEM allocation and the single UMMA-issuing thread
//                 (kind::f16, M = 128, N = tokens rounded up to 16, K = 16);
//   warp 2      : activation producer -- TMA of the token rows of each K step
//                 into the B half of a ring of A/B stages;
//   warps 3..10 : dequantizers (warp w owns rows 32*(w%4).. and one 32-wide
//                 K half of each step), writing the A half of the A/B stage;
//   warps 11..14: epilogue, reading one of two TMEM accumulators while the
//                 MMA fills the other.
// The weight ring runs ahead of the A/B ring, so weight bytes in flight are
// bounded by the F ring depth, not by the (larger) operand stages.  All waits
// are bounded (about 2 s); a timeout records FP4MOE_ERR_TIMEOUT in the device
// status word and the CTA winds down and frees its TMEM.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kWarps = 15;
constexpr int kThreads = kWarps * 32;
constexpr int kDqWarps = 8;
constexpr int kEpiWarps = 4;
constexpr int kWarpFProd = 0, kWarpMma = 1, kWarpBProd = 2, kWarpDq0 = 3,
              kWarpEpi0 = 11;
constexpr uint32_t kABytes = kTileN * kTileK * 2;  // 16 KB bf16 tile
constexpr uint32_t kFBytes = 4608;                 // >= largest packed tile
constexpr uint32_t kTmemCols = 512;                // two 256-column buffers

template <int NT>
struct Cfg {
  static constexpr uint32_t kBBytes = NT * 128;  // NT rows x 64 bf16
  static constexpr uint32_t kABStage = kABytes + kBBytes;
  static constexpr int kSA = NT >= 256 ? 4 : 3;
  static constexpr int kSF = NT >= 256 ? 6 : 32;
  static constexpr uint32_t kFOff = kABStage * kSA;
  static constexpr uint32_t kBarOff = kFOff + kFBytes * kSF;
  static constexpr int kNumBars = 2 * kSF + 3 * kSA + 5;
  static constexpr uint32_t kSmem = kBarOff + 8 * kNumBars + 16 + 1024;
};

struct Unit {
  int e, nb, row0, ntok;
};

// Units are ordered (expert, weight block, token chunk); expert e owns
// nblocks * (cstart[e+1] - cstart[e]) consecutive units.
__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, int u) {
  int lo = 0, hi = a.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.nblocks * __ldg(a.cstart + mid) <= u) lo = mid; else hi = mid;
  }
  const int c0 = __ldg(a.cstart + lo), nch = __ldg(a.cstart + lo + 1) - c0;
  const int local = u - a.nblocks * c0;
  const int o0 = __ldg(a.offsets + lo), cnt = __ldg(a.offsets + lo + 1) - o0;
  const int cs = (cnt + nch - 1) / nch;
  const int c = local % nch;
  Unit U;
  U.e = lo;
  U.nb = local / nch;
  U.row0 = o0 + c * cs;
  U.ntok = min(cs, cnt - c * cs);
  return U;
}

// 8 packed E2M1 codes -> 8 bf16 (4 words, element 0 in the low half of
// word 0), each multiplied by the bf16 pair s2.  The packer places element
// j's magnitude bits (m, e0, e1) and sign so that one or two rotates and a
// mask put them at bf16 bits 6..8 and 15 (or 22..24 and 31): read as bf16,
// (s, e1, e0, m) there is e2m1 * 2^-126 (code 1 = 0.5 lands on a subnormal),
// and the multiply by s * 2^119 gives e2m1 * s * 2^-7 exactly.
__device__ __forceinline__ uint4 dequant8(uint32_t x, uint32_t s2) {
  const uint32_t w0 = x & 0x81C081C0u;
  const uint32_t w1 = (rotl32(x, 3) & 0x01C001C0u) | (rotl32(x, 1) & 0x80008000u);
  const uint32_t w2 = rotl32(x, 6) & 0x81C081C0u;
  const uint32_t w3 = (rotl32(x, 11) & 0x01C001C0u) | (rotl32(x, 5) & 0x80008000u);
  return make_uint4(bf16x2_mul(w0, s2), bf16x2_mul(w1, s2), bf16x2_mul(w2, s2),
                    bf16x2_mul(w3, s2));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <int NT, int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
  using C = Cfg<NT>;
  constexpr int SA = C::kSA, SF = C::kSF;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = sbase + C::kBarOff;
  auto fullF = [&](int s) { return bars + 8u * s; };
  auto emptyF = [&](int s) { return bars + 8u * (SF + s); };
  auto fullB = [&](int s) { return bars + 8u * (2 * SF + s); };
  auto aready = [&](int s) { return bars + 8u * (2 * SF + SA + s); };
  auto emptyAB = [&](int s) { return bars + 8u * (2 * SF + 2 * SA + s); };
  auto accFull = [&](int b) { return bars + 8u * (2 * SF + 3 * SA + b); };
  auto accEmpty = [&](int b) { return bars + 8u * (2 * SF + 3 * SA + 2 + b); };
  const uint32_t done_bar = bars + 8u * (2 * SF + 3 * SA + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + 8 * C::kNumBars);

  if (threadIdx.x == 0) {
    for (int s = 0; s < SF; ++s) {
      mbar_init(fullF(s), 1);
      mbar_init(emptyF(s), kDqWarps);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(fullB(s), 1);
      mbar_init(aready(s), kDqWarps);
      mbar_init(emptyAB(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accFull(b), 1);
      mbar_init(accEmpty(b), kEpiWarps);
    }
    mbar_init(done_bar, 1);
    fence_barrier_init();
  }
  if (warp == kWarpBProd && lane == 0) prefetch_tensormap(&tmB);
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = a.nblocks * __ldg(a.cstart + a.E);

  if (warp == kWarpFProd) {
    // ------------------------------------------------- weight producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit U = decode_unit(a, u);
        const uint8_t* wt = a.wpack + (static_cast<int64_t>(U.e) * a.nblocks + U.nb) *
                                          a.ksteps * a.tile_bytes;
        for (int ks = 0; ks < a.ksteps; ++ks) {
          if (!mbar_wait(emptyF(s), ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(fullF(s), a.tile_bytes);
          bulk_load(sbase + C::kFOff + s * kFBytes,
                    wt + static_cast<int64_t>(ks) * a.tile_bytes, a.tile_bytes, fullF(s));
          issued |= 1u << (s & 31);
          issued_ph = (issued_ph & ~(1u << (s & 31))) | (ph << (s & 31));
          if (++s == SF) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      // Copies still in flight must land before the CTA exits.
      for (int t = 0; t < SF && t < 32; ++t)
        if ((issued >> t) & 1u) mbar_wait(fullF(t), (issued_ph >> t) & 1u);
    }
  } else if (warp == kWarpBProd) {
    // --------------------------------------------- activation producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit U = decode_unit(a, u);
        const int nbox = (U.ntok + 15) >> 4;
        for (int ks = 0; ks < a.ksteps; ++ks) {
          if (!mbar_wait(emptyAB(s), ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(fullB(s), nbox * 2048u);
          const uint32_t dst = sbase + s * C::kABStage + kABytes;
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(dst + b * 2048u, &tmB, ks * kTileK, U.row0 + 16 * b, fullB(s));
          issued |= 1u << s;
          issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
          if (++s == SA) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      for (int t = 0; t < SA; ++t)
        if ((issued >> t) & 1u) mbar_wait(fullB(t), (issued_ph >> t) & 1u);
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      int s = 0, buf = 0;
      uint32_t ph = 0, acc_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit U = decode_unit(a, u);
        const uint32_t n = static_cast<uint32_t>((U.ntok + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(128, n);
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf) * 256u;
        if (!mbar_wait(accEmpty(buf), acc_ph ^ 1u)) { ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < a.ksteps; ++ks) {
          if (!mbar_wait(fullB(s), ph) || !mbar_wait(aready(s), ph)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = sbase + s * C::kABStage;
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk)
            umma_f16(d_tmem, sw128_kmajor_desc(st + kk * 32),
                     sw128_kmajor_desc(st + kABytes + kk * 32), idesc,
                     (ks | kk) != 0 ? 1u : 0u);
          umma_commit(emptyAB(s));
          if (++s == SA) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        umma_commit(accFull(buf));
        if (++buf == 2) { buf = 0; acc_ph ^= 1u; }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      // Let every issued MMA finish before TMEM is released.
      umma_commit(done_bar);
      if (!mbar_wait(done_bar, 0)) record_error(a.err, FP4MOE_ERR_TIMEOUT);
    }
  } else if (warp < kWarpEpi0) {
    // ---------------------------------------------------------- dequant
    const int dq = warp - kWarpDq0;   // 0..7
    const int q = warp & 3;           // row quarter
    const int khalf = dq >> 2;        // 32-wide K half of each step
    const int r = 32 * q + lane;      // weight row in the tile
    const uint32_t smul = a.smul, sadd = a.sadd;
    const uint32_t a_row_off = (r >> 3) * 1024u + (r & 7) * 128u;
    const uint32_t sw = r & 7, cb = 4 * khalf;
    int sf = 0, sa = 0;
    uint32_t phf = 0, pha = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      for (int ks = 0; ks < a.ksteps; ++ks) {
        if (!mbar_wait(fullF(sf), phf)) { ok = false; break; }
        const uint8_t* f = smem + C::kFOff + sf * kFBytes;
        const uint4 d = *reinterpret_cast<const uint4*>(f + khalf * 2048 + r * 16);
        uint32_t c0, c1;
        if (a.gran == 16) {
          const uint32_t sc =
              *reinterpret_cast<const uint16_t*>(f + kTileDataBytes + r * 4 + khalf * 2);
          c0 = sc & 0xFFu;
          c1 = sc >> 8;
        } else {
          c0 = c1 = f[kTileDataBytes + r * 2 + khalf];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(emptyF(sf));
        if (++sf == SF) { sf = 0; phf ^= 1u; }
        uint32_t s0 = c0 * smul + sadd, s1 = c1 * smul + sadd;
        s0 |= s0 << 16;
        s1 |= s1 << 16;
        const uint4 w0 = dequant8(d.x, s0), w1 = dequant8(d.y, s0);
        const uint4 w2 = dequant8(d.z, s1), w3 = dequant8(d.w, s1);
        if (!mbar_wait(emptyAB(sa), pha ^ 1u)) { ok = false; break; }
        const uint32_t arow = sbase + sa * C::kABStage + a_row_off;
        st_shared_v4(arow + (((cb + 0) ^ sw) << 4), w0);
        st_shared_v4(arow + (((cb + 1) ^ sw) << 4), w1);
        st_shared_v4(arow + (((cb + 2) ^ sw) << 4), w2);
        st_shared_v4(arow + (((cb + 3) ^ sw) << 4), w3);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(aready(sa));
        if (++sa == SA) { sa = 0; pha ^= 1u; }
      }
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int r = 32 * q + lane;      // weight row in the tile
    int buf = 0;
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit U = decode_unit(a, u);
      if (!mbar_wait(accFull(buf), acc_ph)) { ok = false; break; }
      tc_fence_after();
      const float alpha = __ldg(a.alpha + U.e);
      const int nchunks = (U.ntok + 15) >> 4;
      const uint32_t t_base = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                              static_cast<uint32_t>(buf) * 256u;
      for (int j = 0; j < nchunks; ++j) {
        uint32_t v[16];
        tmem_ld16(t_base + 16 * j, v);
        tmem_ld_wait();
        if (MODE == kGemmModeFc2) {
          float* o = static_cast<float*>(a.out);
          const int64_t n = static_cast<int64_t>(U.nb) * kTileN + r;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int col = 16 * j + c;
            if (col < U.ntok)
              o[static_cast<int64_t>(U.row0 + col) * a.ldo + n] = __uint_as_float(v[c]) * alpha;
          }
        } else {
          // Lanes 0..15 hold gate rows, 16..31 the up rows of the same 16
          // intermediate columns; one exchange per column pair.
          const int i = U.nb * 64 + 16 * q + (lane & 15);
          const bool is_gate = lane < 16;
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float a0 = __uint_as_float(v[2 * m]), a1 = __uint_as_float(v[2 * m + 1]);
            const float recv = __shfl_xor_sync(kFull, is_gate ? a1 : a0, 16);
            const float g = (is_gate ? a0 : recv) * alpha;
            const float up = (is_gate ? recv : a1) * alpha;
            const float h = g / (1.0f + expf(-g)) * up;
            const int col = 16 * j + 2 * m + (is_gate ? 0 : 1);
            if (col < U.ntok) {
              const int64_t idx = static_cast<int64_t>(U.row0 + col) * a.ldo + i;
              if (MODE == kGemmModeFc1)
                static_cast<uint16_t*>(a.out)[idx] = static_cast<uint16_t>(f32_to_bf16_bits(h));
              else
                static_cast<float*>(a.out)[idx] = h;
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accEmpty(buf));
      if (++buf == 2) { buf = 0; acc_ph ^= 1u; }
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  }

  // ---- teardown: the MMA thread has waited (bounded) for its final commit,
  // so no UMMA is still writing TMEM; free it.
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int NT, int MODE>
cudaError_t launch_one(const CUtensorMap& tmB, const GemmArgs& a, int grid,
                       cudaStream_t st) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<NT, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Cfg<NT>::kSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  moe_gemm_kernel<NT, MODE><<<grid, kThreads, Cfg<NT>::kSmem, st>>>(tmB, a);
  return cudaGetLastError();
}

template <int NT>
cudaError_t launch_nt(const CUtensorMap& tmB, const GemmArgs& a, int grid,
                      cudaStream_t st) {
  switch (a.mode) {
    case kGemmModeFc1: return launch_one<NT, kGemmModeFc1>(tmB, a, grid, st);
    case kGemmModeFc2: return launch_one<NT, kGemmModeFc2>(tmB, a, grid, st);
    default: return launch_one<NT, kGemmModeFc1Fp8>(tmB, a, grid, st);
  }
}

}  // namespace

int gemm_chunk_max(int T) { return T <= 64 ? 64 : 256; }

cudaError_t launch_gemm(const CUtensorMap& tmB, const GemmArgs& a, int nt,
                        int num_sms, cudaStream_t st) {
  const int grid = num_sms > 0 ? num_sms : 1;
  if (nt <= 64) return launch_nt<64>(tmB, a, grid, st);
  return launch_nt<256>(tmB, a, grid, st);
}

}  // namespace fp4moe
