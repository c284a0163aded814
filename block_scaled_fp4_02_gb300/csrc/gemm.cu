// Grouped GEMM of the MoE expert FFN over packed block-scaled FP4 weights
// (sm_103a, tcgen05): FC1 gate|up with the SwiGLU epilogue and FC2.
//
// Formulation (weights as the UMMA M side): for each work unit (expert e,
// 128-row weight block nb, chunk of up to NT tokens of e),
//     D[128 x n] = W_tile[128 x Kd] * X_chunk[n x Kd]^T    (FP32 in TMEM)
// W is dequantized FP4 -> bf16 into shared memory in the 128-byte swizzled
// K-major layout; X (bf16 activations in expert-major order) arrives by TMA
// in the same layout.  Warp roles, one CTA per SM, persistent over units:
//   warp 0     : producer -- bulk copy of the packed FP4 tile + TMA of the
//                token rows for each 64-wide K step into a ring of stages;
//   warp 1     : TMEM allocation and the single UMMA-issuing thread
//                (kind::f16, M = 128, N = tokens rounded up to 16, K = 16);
//   warps 2..9 : dequantizers (warp w owns rows 32*(w%4).. and one 32-wide K
//                half of each step), then the epilogue reading TMEM.
// All waits are bounded (about 2 s); a timeout records FP4MOE_ERR_TIMEOUT in
// the device status word and the CTA winds down and frees its TMEM.
#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kWarps = 10;
constexpr int kThreads = kWarps * 32;
constexpr int kDqWarps = 8;
constexpr uint32_t kABytes = kTileN * kTileK * 2;  // 16 KB bf16 tile
constexpr uint32_t kFBytes = 5120;  // >= largest packed tile, 1 KB multiple
constexpr uint32_t kTmemCols = 256;

template <int NT>
struct Cfg {
  static constexpr uint32_t kBBytes = NT * 128;  // NT rows x 64 bf16
  static constexpr uint32_t kStage = kABytes + kBBytes + kFBytes;
  static constexpr int kStages = NT >= 256 ? 4 : (NT >= 128 ? 5 : 7);
  static constexpr uint32_t kBarOff = kStage * kStages;
  static constexpr uint32_t kSmem = kBarOff + 256 + 1024;
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
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = sbase + C::kBarOff;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto aready_bar = [&](int s) { return bars + 8u * (S + s); };
  auto empty_bar = [&](int s) { return bars + 8u * (2 * S + s); };
  const uint32_t acc_full = bars + 8u * (3 * S);
  const uint32_t acc_empty = bars + 8u * (3 * S + 1);
  const uint32_t done_bar = bars + 8u * (3 * S + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + 8 * (3 * S + 3));

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(aready_bar(s), kDqWarps);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, kDqWarps);
    mbar_init(done_bar, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = a.nblocks * __ldg(a.cstart + a.E);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_parity = 0;  // per-stage bit masks
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit U = decode_unit(a, u);
        const uint8_t* wt = a.wpack + (static_cast<int64_t>(U.e) * a.nblocks + U.nb) *
                                          a.ksteps * a.tile_bytes;
        const int nbox = (U.ntok + 15) >> 4;
        const uint32_t bytes = a.tile_bytes + nbox * 2048u;
        for (int ks = 0; ks < a.ksteps; ++ks) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u)) { ok = false; break; }
          const uint32_t st = sbase + stage * C::kStage;
          mbar_arrive_expect_tx(full_bar(stage), bytes);
          bulk_load(st + kABytes + C::kBBytes, wt + static_cast<int64_t>(ks) * a.tile_bytes,
                    a.tile_bytes, full_bar(stage));
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(st + kABytes + b * 2048u, &tmB, ks * kTileK, U.row0 + 16 * b,
                        full_bar(stage));
          issued |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      // Copies still in flight must land before the CTA exits.
      for (int s = 0; s < S; ++s)
        if ((issued >> s) & 1u) mbar_wait(full_bar(s), (issued_parity >> s) & 1u);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit U = decode_unit(a, u);
        const uint32_t n = static_cast<uint32_t>((U.ntok + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(128, n);
        if (!mbar_wait(acc_empty, acc_phase ^ 1u)) { ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < a.ksteps; ++ks) {
          if (!mbar_wait(aready_bar(stage), phase)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = sbase + stage * C::kStage;
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk)
            umma_f16(tmem, sw128_kmajor_desc(st + kk * 32),
                     sw128_kmajor_desc(st + kABytes + kk * 32), idesc,
                     (ks | kk) != 0 ? 1u : 0u);
          umma_commit(empty_bar(stage));
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        umma_commit(acc_full);
        acc_phase ^= 1u;
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      // Let every issued MMA finish before TMEM is released.
      umma_commit(done_bar);
      if (!mbar_wait(done_bar, 0)) record_error(a.err, FP4MOE_ERR_TIMEOUT);
    }
  } else {
    // ------------------------------------------------ dequant + epilogue
    const int dq = warp - 2;          // 0..7
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int khalf = dq >> 2;        // 32-wide K half of each step
    const int r = 32 * q + lane;      // weight row in the tile
    const uint32_t smul = a.smul, sadd = a.sadd;
    const uint32_t a_row_off = (r >> 3) * 1024u + (r & 7) * 128u;
    int stage = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit U = decode_unit(a, u);
      for (int ks = 0; ks < a.ksteps; ++ks) {
        if (!mbar_wait(full_bar(stage), phase)) { ok = false; break; }
        const uint8_t* f = smem + stage * C::kStage + kABytes + C::kBBytes;
        const uint4 d = *reinterpret_cast<const uint4*>(f + khalf * 2048 + r * 16);
        uint32_t c0, c1;
        if (a.gran == 16) {
          const uint32_t sc = *reinterpret_cast<const uint16_t*>(f + kTileDataBytes + r * 4 + khalf * 2);
          c0 = sc & 0xFFu;
          c1 = sc >> 8;
        } else {
          c0 = c1 = f[kTileDataBytes + r * 2 + khalf];
        }
        uint32_t s0 = c0 * smul + sadd, s1 = c1 * smul + sadd;
        s0 |= s0 << 16;
        s1 |= s1 << 16;
        const uint32_t arow = sbase + stage * C::kStage + a_row_off;
        const uint32_t sw = r & 7;
        const uint32_t cb = 4 * khalf;
        st_shared_v4(arow + (((cb + 0) ^ sw) << 4), dequant8(d.x, s0));
        st_shared_v4(arow + (((cb + 1) ^ sw) << 4), dequant8(d.y, s0));
        st_shared_v4(arow + (((cb + 2) ^ sw) << 4), dequant8(d.z, s1));
        st_shared_v4(arow + (((cb + 3) ^ sw) << 4), dequant8(d.w, s1));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(aready_bar(stage));
        if (++stage == S) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      // ---- epilogue: columns in chunks of 16, alternating between the two
      // groups of four warps.
      if (!mbar_wait(acc_full, acc_phase)) { ok = false; break; }
      tc_fence_after();
      const float alpha = __ldg(a.alpha + U.e);
      const int nchunks = (U.ntok + 15) >> 4;
      for (int j = khalf; j < nchunks; j += 2) {
        uint32_t v[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q) << 16) + 16 * j, v);
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
      if (lane == 0) mbar_arrive(acc_empty);
      acc_phase ^= 1u;
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  }

  // ---- teardown: the MMA thread has waited (bounded) for its final commit,
  // so no UMMA is still writing TMEM; free it.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
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
