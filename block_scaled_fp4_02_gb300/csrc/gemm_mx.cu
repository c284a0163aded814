// Grouped GEMM of the MoE expert FFN with FP8 activations over group32 FP4
// weights on the block-scaled tensor-core path (sm_103a, tcgen05
// kind::mxf8f6f4): recipe (1,1,32) of the group16 notes page (section
// "Context"; section "Remaining kernel work" places this compute on the
// block-scaled MMA with the UE8M0 scales in tensor memory).
//
//     D_t[128 x n] = (W_t x SW_t)[128 x K] * (X x SX)[n x K]^T      (FP32)
//
// W: E2M1 codes, copied by TMA with the 16U4_ALIGN16B type, which widens
// each 16 packed codes (8 bytes) to 16 bytes in shared memory, the operand
// form the MMA reads for E2M1 under kind::mxf8f6f4; no conversion runs on
// the SM.  X: E4M3 rows (gathered activations for FC1, the FP8 intermediate
// h for FC2) by TMA.  SW, SX: one UE8M0 byte per row and 32 K elements, in
// step-major arrays (one 32-bit word = four 32-wide blocks per row and
// 128-wide K step), bulk-copied into the stage and moved to tensor memory by
// four scale warps; the MMA's scale id picks the block.
//
// A work unit is (expert e, block b, chunk of up to 224 tokens of e); the K
// loop runs in steps of 128.  FC1: the unit's two tiles are the gate rows and
// the up rows of the same 128 intermediate columns i = 128 b + r, so the
// epilogue finds G and U of one i in one TMEM lane (two accumulators) and
// the 32-wide FP8 group of h in one warp; it stores h as E4M3 bytes plus one
// UE8M0 byte per token and 32 columns (the (1,1,32) rule), which FC2
// consumes directly.  FC2: the two tiles are consecutive 128-row blocks of
// w2; the epilogue stores FP32 o.
//
// Warps (one CTA per SM, persistent over units):
//   0      weight producer: TMA of the unit's weight tiles and bulk copy of
//          their scale words, per step, into a ring of stages;
//   1, 3   MMA issuers of tile 0 and tile 1 (one elected thread each);
//   2      activation producer: TMA of the chunk's rows (one box of 32..256
//          rows) and bulk copy of their scale words;
//   4..7   scale warps (TMEM lane quarters 0..3): scale words -> TMEM;
//   8..23  epilogue (lane quarter = warp % 4; four warps per quarter share
//          the accumulator columns, so the single-buffered accumulators drain
//          quickly between units).
// All waits are bounded (about 2 s); a timeout records FP4MOE_ERR_TIMEOUT in
// the device status word and the CTA winds down and frees its TMEM.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr int kWarps = 24, kThreads = kWarps * 32;
constexpr int kWarpA = 0, kWarpMma0 = 1, kWarpB = 2, kWarpMma1 = 3, kWarpSf0 = 4,
              kWarpEpi0 = 8, kEpiWarps = 16;
constexpr int kStages = 3;
constexpr uint32_t kATile = 128 * 128;             // 128 rows x 128 B (widened E2M1)
constexpr uint32_t kATileTx = 128 * 64;            // bytes the TMA reads (packed)
constexpr uint32_t kBBytes = kMxChunk256Rows * 128;  // up to 256 rows x 128 B
constexpr uint32_t kSfaBytes = 128 * 4;            // one word per row
constexpr uint32_t kSfbBytes = (kMxChunk256Rows + 16) * 4;
constexpr uint32_t kOffA = 0, kOffB = 2 * kATile, kOffSfa = kOffB + kBBytes,
                   kOffSfb = kOffSfa + 2 * kSfaBytes;
constexpr uint32_t kStage = (kOffSfb + kSfbBytes + 1023) & ~1023u;
// Barriers per stage: full (TMA bytes), ready (scale factors of the stage in
// its TMEM slot: implies full), empty (both MMA issuers' commits: frees the
// shared-memory stage and its scale slot).
constexpr int kNumBars = 3 * kStages + 2 + 1;
static_assert(kStages <= kMxSfSlots, "one TMEM scale slot per stage");
constexpr uint32_t kBarOff = kStage * kStages;
constexpr uint32_t kTabOff = kBarOff + 8 * kNumBars + 16;
constexpr uint32_t kSmem = kTabOff + 8 * (kMaxE + 1) + 1024;
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kOffB % 1024 == 0 && kStage % 1024 == 0, "swizzled operands need 1 KB alignment");
static_assert(kOffSfa % 16 == 0 && kOffSfb % 16 == 0, "bulk copies need 16 B alignment");
// TMEM: accumulators at columns 0 and 256 (N <= 224 each); four scale slots
// of 16 columns in the two gaps, at 224, 240, 480 and 496 (tile 0 SFA:
// +0..3, tile 1 SFA: +4..7, SFB: +8..15).
constexpr uint32_t kAcc1Col = 256, kTmemCols = 512;
__host__ __device__ constexpr uint32_t sf_col(int j) {
  return j < 2 ? 224u + 16u * j : 480u + 16u * (j - 2);
}
static_assert(kMxChunk <= 224 && kAcc1Col + kMxChunk <= sf_col(2) &&
              sf_col(1) + 16 <= kAcc1Col && sf_col(kMxSfSlots - 1) + 16 <= kTmemCols,
              "TMEM budget");
static_assert(kMxChunk % 32 == 0 && (kMxChunk + 31) / 32 <= 8, "SFB columns");

struct Unit {
  int e, nb, row0, ntok;
};

__device__ __forceinline__ Unit decode_unit(const MxGemmArgs& a, int nbu, const int* cs_,
                                            const int* os, int u) {
  constexpr int max_tok = kMxChunk;
  int lo = 0, hi = a.E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (nbu * cs_[mid] <= u) lo = mid; else hi = mid;
  }
  const int c0 = cs_[lo];
  int nch = cs_[lo + 1] - c0;
  if (!in_bounds(a.err, nch - 1, INT32_MAX)) nch = 1;
  const int local = u - nbu * c0;
  const int o0 = os[lo], cnt = os[lo + 1] - o0;
  const int cs = (cnt + nch - 1) / nch;
  const int c = local % nch;
  Unit U;
  U.e = lo;
  U.nb = local / nch;          // FC1: block of 128 columns; FC2: pair of row blocks
  U.row0 = o0 + c * cs;
  U.ntok = min(cs, cnt - c * cs);
  // Bounds-checked build: a unit outside the expert-major rows, or larger
  // than a chunk, records BOUNDS and shrinks to row 0 alone, so that every
  // role still walks the same (in-bounds) schedule.
  if (!(in_bounds(a.err, U.e, a.E) && in_bounds(a.err, U.ntok - 1, max_tok) &&
        in_bounds(a.err, U.row0, a.rows) && in_bounds(a.err, U.row0 + U.ntok - 1, a.rows))) {
    U.row0 = 0;
    U.ntok = 1;
  }
  return U;
}

__device__ __forceinline__ uint64_t desc_at(uint32_t saddr) {
  return sw128_kmajor_desc(saddr);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_mx_kernel(const __grid_constant__ MxMaps maps, const MxGemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = sbase + kBarOff;
  auto fullS = [&](int s) { return bars + 8u * s; };
  auto emptyS = [&](int s) { return bars + 8u * (kStages + s); };
  auto readyS = [&](int s) { return bars + 8u * (2 * kStages + s); };
  const uint32_t accFull = bars + 8u * (3 * kStages);
  const uint32_t accEmpty = accFull + 8u;
  const uint32_t done_bar = accFull + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kNumBars);
  int* tab_cs = reinterpret_cast<int*>(smem + kTabOff);
  int* tab_os = tab_cs + (kMaxE + 1);
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) {
    tab_cs[i] = __ldg(a.cstart + i);
    tab_os[i] = __ldg(a.offsets + i);
  }
  // FC1: one unit per 128-column block (two tiles: gate, up); FC2: one unit
  // per pair of 128-row blocks (the last may hold one).
  const int nbu = (MODE == kGemmModeFc2) ? (a.nblocks + 1) / 2 : a.nblocks;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(fullS(s), 2);     // weight and activation producers
      mbar_init(readyS(s), 4);    // four scale warps
      mbar_init(emptyS(s), 2);    // both MMA issuers
    }
    mbar_init(accFull, 2);
    mbar_init(accEmpty, kEpiWarps);
    mbar_init(done_bar, 2);
    fence_barrier_init();
  }
  if (warp == kWarpA && lane == 0) prefetch_tensormap(&maps.w);
  if (warp == kWarpB && lane < kMxBoxes) prefetch_tensormap(&maps.x[lane]);
  if (warp == kWarpMma0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = nbu * tab_cs[a.E];

  if (warp == kWarpA || warp == kWarpB) {
    // ------------------------------------------------------ producers
    if (lane == 0) {
      const bool isA = warp == kWarpA;
      uint32_t n = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit U = decode_unit(a, nbu, tab_cs, tab_os, u);
        const int tiles = (MODE == kGemmModeFc2) ? min(2, a.nblocks - 2 * U.nb) : 2;
        // FC1 rows of block b: gate tile at 256 b, up tile at 256 b + 128;
        // FC2 rows: tiles at 128 (2 nb) and 128 (2 nb + 1).
        const int wrow0 = U.e * a.rows_per_expert + 256 * U.nb;
        const int brows = (U.ntok + 31) & ~31;        // box rows: 32 .. 256
        const CUtensorMap* tmX = &maps.x[brows / 32 - 1];
        const int lead = U.row0 & 3;                   // scale words before row0
        const uint32_t sfb_bytes = static_cast<uint32_t>(((lead + brows + 3) & ~3) * 4);
        for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
          const int s = static_cast<int>(n % kStages);
          const uint32_t ph = (n / kStages) & 1u;
          if (!mbar_wait(emptyS(s), ph ^ 1u)) { ok = false; break; }
          const uint32_t st = sbase + s * kStage;
          if (isA) {
            mbar_arrive_expect_tx(fullS(s), tiles * (kATileTx + kSfaBytes));
            for (int t = 0; t < tiles; ++t) {
              tma_load_2d(st + kOffA + t * kATile, &maps.w, ks * kMxK, wrow0 + 128 * t,
                          fullS(s));
              // scale words of tile t at step ks: [tile group][ks][128 rows]
              const int64_t tg = static_cast<int64_t>(U.e) * a.tiles_per_expert + 2 * U.nb + t;
              bulk_load(st + kOffSfa + t * kSfaBytes,
                        a.wscale + (tg * a.ksteps + ks) * 128, kSfaBytes, fullS(s));
            }
          } else {
            mbar_arrive_expect_tx(fullS(s), brows * 128u + sfb_bytes);
            tma_load_2d(st + kOffB, tmX, ks * kMxK, U.row0, fullS(s));
            bulk_load(st + kOffSfb,
                      a.xscale + static_cast<int64_t>(ks) * a.xscale_pitch + (U.row0 - lead),
                      sfb_bytes, fullS(s));
          }
          issued |= 1u << s;
          issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      for (int t = 0; t < kStages; ++t)
        if ((issued >> t) & 1u) mbar_wait(fullS(t), (issued_ph >> t) & 1u);
    }
  } else if (warp == kWarpMma0 || warp == kWarpMma1) {
    // ------------------------------------------------------------ MMA
    const int t = (warp == kWarpMma0) ? 0 : 1;
    if (lane == 0) {
      uint32_t n = 0, acc_ph = 0;
      bool ok = true;
      const uint32_t d_tmem = tmem + (t ? kAcc1Col : 0u);
      for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
        const Unit U = decode_unit(a, nbu, tab_cs, tab_os, u);
        const int tiles = (MODE == kGemmModeFc2) ? min(2, a.nblocks - 2 * U.nb) : 2;
        const uint32_t nn = static_cast<uint32_t>((U.ntok + 15) & ~15);
        if (!mbar_wait(accEmpty, acc_ph ^ 1u)) { ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
          // One wait per step: the scale warps arrive on ready(s) only after
          // the stage's copies landed (full(s)) and its scales are in TMEM.
          const int s = static_cast<int>(n % kStages);
          if (!mbar_wait(readyS(s), (n / kStages) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (t < tiles) {
            const uint32_t st = sbase + s * kStage;
            const uint64_t ad = desc_at(st + kOffA + t * kATile);
            const uint64_t bd = desc_at(st + kOffB);
            const uint32_t sfa = tmem + sf_col(s) + 4u * t;
            const uint32_t sfb = tmem + sf_col(s) + 8u;
#pragma unroll
            for (int kk = 0; kk < kMxK / 32; ++kk)
              umma_mx(d_tmem, ad + 2u * kk, bd + 2u * kk,
                      idesc_mx_e2m1_e4m3(128, nn, kk, kk), sfa, sfb,
                      (ks > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(emptyS(s));
        }
        if (!ok) break;
        umma_commit(accFull);
        acc_ph ^= 1u;
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      umma_commit(done_bar);
      if (!mbar_wait(done_bar, 0)) record_error(a.err, FP4MOE_ERR_TIMEOUT);
    }
  } else if (warp >= kWarpSf0 && warp < kWarpEpi0) {
    // ----------------------------------------------------- scale warps
    // Warp q (= warp % 4) owns TMEM lanes 32q..32q+31.  SFA of tile t: row
    // m = 32q + lane goes to lane m, column q (the column of its 32-row
    // block).  SFB: row n = 32c + lane goes to column c of every lane
    // quarter, so each quarter of the accumulator reads its own copy.
    const int q = warp & 3;
    uint32_t n = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit U = decode_unit(a, nbu, tab_cs, tab_os, u);
      const int tiles = (MODE == kGemmModeFc2) ? min(2, a.nblocks - 2 * U.nb) : 2;
      const int lead = U.row0 & 3;
      for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
        // The stage's scale slot is free: the producers reloaded the stage,
        // which needed the MMAs that last read the slot to complete.
        const int s = static_cast<int>(n % kStages);
        if (!mbar_wait(fullS(s), (n / kStages) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* st = smem + s * kStage;
        const uint32_t* sfa = reinterpret_cast<const uint32_t*>(st + kOffSfa);
        const uint32_t* sfb = reinterpret_cast<const uint32_t*>(st + kOffSfb) + lead;
        const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t col = tmem + lanes + sf_col(s);
        for (int t = 0; t < tiles; ++t) tmem_st1(col + 4u * t + q, sfa[t * 128 + 32 * q + lane]);
        uint32_t v[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) v[c] = sfb[32 * c + lane];
        tmem_st8(col + 8u, v);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(readyS(s));
      }
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  } else {
    // --------------------------------------------------------- epilogue
    const int ew = warp - kWarpEpi0;   // 0..15
    const int q = warp & 3;            // TMEM lane quarter
    const int part = ew >> 2;          // 0..3: FC1 column part; FC2 tile + half
    const int tile = part & 1;         // FC2: the accumulator (weight tile) it drains
    const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      const Unit U = decode_unit(a, nbu, tab_cs, tab_os, u);
      if (!mbar_wait(accFull, acc_ph)) { ok = false; break; }
      tc_fence_after();
      const float alpha = __ldg(a.alpha + U.e);
      const int nchunks = (U.ntok + 15) >> 4;
      if (MODE == kGemmModeFc2) {
        const int nb = 2 * U.nb + tile;
        if (nb < a.nblocks) {
          float* o = static_cast<float*>(a.out);
          const int64_t col_n = static_cast<int64_t>(nb) * 128 + 32 * q + lane;
          const uint32_t tb = tmem + lanes + (tile ? kAcc1Col : 0u);
          // Pairs of chunks (32 columns) per TMEM load; the two warps of a
          // tile and lane quarter take alternate pairs.
          for (int c0 = 2 * (part >> 1); c0 < nchunks; c0 += 4) {
            uint32_t v[32];
            tmem_ld32(tb + 16 * c0, v);
            tmem_ld_wait(v);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int col = 16 * c0 + c;
              if (col < U.ntok)
                o[static_cast<int64_t>(U.row0 + col) * a.ldo + col_n] =
                    __uint_as_float(v[c]) * alpha;
            }
          }
        }
      } else {
        // h for i = 128 b + 32 q + lane; the 32 lanes are one (1,1,32) group.
        // Per chunk of 16 tokens each lane packs its 16 codes four per word;
        // a transpose over the warp then gives lane L the codes of token
        // 4k + L/8 for i = 4 (L % 8) .. + 3, stored as one 32-bit word, and
        // lanes 0..15 store the 16 tokens' scale bytes at once.
        uint8_t* h8 = static_cast<uint8_t*>(a.out);
        const int tr = lane >> 3, tm = lane & 7;
        const int64_t i4 = static_cast<int64_t>(U.nb) * 128 + 32 * q + 4 * tm;
        const uint32_t sel = static_cast<uint32_t>(tr) | (static_cast<uint32_t>(tr + 4) << 4);
        for (int c0 = part; c0 < nchunks; c0 += 4) {
          uint32_t g[16], up[16];
          tmem_ld16(tmem + lanes + 16 * c0, g);
          tmem_ld16(tmem + lanes + kAcc1Col + 16 * c0, up);
          tmem_ld_wait(g);
          tmem_ld_wait(up);
          uint32_t packed[4] = {0u, 0u, 0u, 0u};
          uint32_t my_sb = 0u;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float gv = __uint_as_float(g[c]) * alpha;
            const float uv = __uint_as_float(up[c]) * alpha;
            const float h = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            // group maximum of |h| over the warp: non-negative floats order
            // like their bit patterns
            const float amax = __uint_as_float(redux_max_u32(__float_as_uint(fabsf(h))));
            const uint32_t byte = ue8m0_for_e4m3(amax);   // <= 247 for finite h
            const float inv = __uint_as_float((254u - byte) << 23);   // 2^(127 - byte)
            const uint32_t code = f32x2_to_e4m3x2(h * inv, 0.0f) & 0xFFu;
            packed[c >> 2] |= code << (8 * (c & 3));
            if (lane == c) my_sb = byte;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t b0 = __shfl_sync(kFullMask, packed[k], 4 * tm + 0);
            const uint32_t b1 = __shfl_sync(kFullMask, packed[k], 4 * tm + 1);
            const uint32_t b2 = __shfl_sync(kFullMask, packed[k], 4 * tm + 2);
            const uint32_t b3 = __shfl_sync(kFullMask, packed[k], 4 * tm + 3);
            const uint32_t w = __byte_perm(__byte_perm(b0, b1, sel), __byte_perm(b2, b3, sel),
                                           0x5410);
            const int col = 16 * c0 + 4 * k + tr;
            if (col < U.ntok)
              *reinterpret_cast<uint32_t*>(h8 + static_cast<int64_t>(U.row0 + col) * a.ldo + i4) = w;
          }
          if (lane < 16 && 16 * c0 + lane < U.ntok)
            a.hscale[(static_cast<int64_t>(U.nb) * a.hscale_pitch + U.row0 + 16 * c0 + lane) * 4 +
                     q] = static_cast<uint8_t>(my_sb);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accEmpty);
      acc_ph ^= 1u;
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  }

  // ---- teardown: both MMA threads waited (bounded) for their last commits.
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int MODE>
cudaError_t launch_mx_mode(const MxMaps& maps, const MxGemmArgs& a, int grid,
                           cudaStream_t st) {
  static std::mutex mu;
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!attr_set[dev]) {
      e = cudaFuncSetAttribute(moe_gemm_mx_kernel<MODE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmem));
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  moe_gemm_mx_kernel<MODE><<<grid, kThreads, kSmem, st>>>(maps, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_mx(const MxMaps& maps, const MxGemmArgs& a, int num_sms,
                           cudaStream_t st) {
  const int grid = num_sms > 0 ? num_sms : 1;
  if (a.mode == kGemmModeFc2) return launch_mx_mode<kGemmModeFc2>(maps, a, grid, st);
  return launch_mx_mode<kGemmModeFc1>(maps, a, grid, st);
}

}  // namespace fp4moe
