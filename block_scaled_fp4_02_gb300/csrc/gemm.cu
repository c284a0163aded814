// Grouped GEMM of the MoE expert FFN over packed block-scaled FP4 weights
// (sm_103a, tcgen05): FC1 gate|up with the SwiGLU epilogue and FC2.
//
// Formulation (weights as the UMMA M side): for each work unit (expert e,
// MT consecutive 128-row weight blocks, chunk of up to NT tokens of e),
//     D_t[128 x n] = W_tile_t[128 x Kd] * X_chunk[n x Kd]^T   (FP32, TMEM)
// W is dequantized FP4 -> bf16 into shared memory (or TMEM) in the UMMA
// K-major layout; X (bf16 activations in expert-major order) arrives by TMA
// in the 128-byte swizzled layout.  Two variants:
//   NT = 256 (many tokens per expert): MT = 2 weight tiles share each
//     activation tile, which halves activation traffic per MMA; A in shared
//     memory; two accumulators of 256 columns fill TMEM; one MMA warp per
//     tile.
//   NT = 32 (decode): MT = 1; A lives in TMEM.  One thread issues an
//     asynchronous instruction (tcgen05.mma, a TMA copy) only every ~100
//     cycles or more, far below what the tensor and TMA units take, so the
//     issue is spread and amortized: the unit of hand-off is a pair of K
//     steps (128 wide: one weight copy, one TMEM A stage of 64 columns, eight
//     MMAs); four MMA warps take pairs m = 0..3 (mod 4) into their own
//     accumulators (summed in the epilogue, double-buffered), and four
//     threads load the activation rows (steps n = 0..3 (mod 4)).
// Warp roles, one CTA per SM, persistent over units:
//   warp 0      : weight producer -- bulk copies of the packed FP4 tiles
//                 (MT per K step, or two K steps with NT = 32) into a ring of
//                 F stages;
//   warp 1      : TMEM allocation; with NT = 256 the UMMA-issuing thread of
//                 tile 0 (kind::f16, M = 128, N = tokens rounded up to 16,
//                 K = 16), with NT = 32 the activation producer of steps
//                 n = 1 (mod 4);
//   warp 2      : activation producer -- TMA of the token rows of each K step
//                 (steps n = 0 (mod 4) with NT = 32) into the B part of a ring
//                 of A/B stages;
//   warps 3..18 : dequantizers: NT = 256, two groups of eight (warp w owns
//                 rows 32*(w%4).. and one 32-wide K half; group g fills
//                 weight tile g of every step); NT = 32, four groups of four
//                 (group g converts the pairs m = g (mod 4) into A stage g);
//   warps 19..  : epilogue (twelve warps for NT = 256, three per lane
//                 quarter; four for NT = 32), reading the TMEM accumulators;
//                 then NT = 256 has the MMA
//                 warp of tile 1, NT = 32 its four MMA warps (one per SM
//                 sub-partition) and the activation producers of steps
//                 n = 2, 3 (mod 4).
// All waits are bounded (about 2 s); a timeout records FP4MOE_ERR_TIMEOUT in
// the device status word and the CTA winds down and frees its TMEM.
#include <mutex>

#include "common.cuh"
#include "gemm_parts.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr int kMaxDevices = 64;

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kDqGroups = 2;     // dequant groups (A in shared memory)
constexpr int kDqWarps = 8;      // warps per dequant group (A in shared memory)
constexpr int kWarpFProd = 0, kWarpMma = 1, kWarpBProd = 2, kWarpDq0 = 3,
              kWarpEpi0 = kWarpDq0 + kDqGroups * kDqWarps;
constexpr uint32_t kABytes = kTileN * kTileK * 2;  // 16 KB bf16 tile
constexpr uint32_t kFBytes = 4608;                 // >= largest packed tile
constexpr uint32_t kTmemCols = 512;

template <int NT>
struct Cfg {
  static_assert(NT == 32 || NT == 256, "the two variants of the kernel");
  static constexpr bool kATmem = NT == 32;         // A stages in TMEM
  static constexpr int kMT = kATmem ? 1 : 2;       // weight tiles per unit
  // One thread issues a tcgen05.mma about every 55 cycles whatever its size,
  // while the tensor pipe takes a short (N <= 32, A in TMEM) one every ~14:
  // with A in TMEM four warps issue, one per SM sub-partition (warp % 4),
  // and split the pairs of K steps; with A in shared memory two MMA warps
  // each own one weight tile (all K steps).
  static constexpr int kMmaWarps = kATmem ? 4 : 2;
  // Epilogue: NT = 32, one warp per TMEM lane quarter; NT = 256, three per
  // quarter, which take the (tile, pair of chunks) items round robin so the
  // single-buffered accumulators drain quickly between units.
  static constexpr int kEpiWarps = kATmem ? 4 : 12;
  // The warps after the epilogue: TMEM A, the four MMA warps and then two
  // activation producers; shared-memory A, the MMA warp of tile 1 (warp 1
  // issues tile 0).
  static constexpr int kWarpMmaX0 = kWarpEpi0 + kEpiWarps;
  static constexpr int kWarpBX0 = kWarpMmaX0 + kMmaWarps;   // extra B producers
  static constexpr int kExtraB = kATmem ? 2 : 0;
  static constexpr int kWarps = kATmem ? kWarpBX0 + kExtraB : kWarpMmaX0 + 1;
  static constexpr int kThreads = kWarps * 32;
  // Rings: F (packed weights, from HBM), A (dequantized weights, shared
  // memory or TMEM), B (activation rows, from L2 by TMA).  With A in TMEM
  // an F stage and an A stage hold a pair of K steps, a B stage one step.
  static constexpr int kStepsPerF = kATmem ? 2 : 1;  // K steps per F stage
  static constexpr int kSF = kATmem ? 12 : 6;
  // TMEM A: four stages of 64 columns (a pair of K tiles each), stage g
  // owned by dequant group g and by MMA warp g: every waiter on a stage's
  // barriers sees each of its phases in turn (a waiter that skipped a phase
  // could mistake an old phase for the one it waits for).
  static constexpr int kSAa = kATmem ? 4 : 2;
  static constexpr int kSB = kATmem ? 2 * kSAa : 3;
  static constexpr uint32_t kFStage = kFBytes * kMT * kStepsPerF;
  static constexpr uint32_t kAStage = kATmem ? 0 : kABytes * kMT;
  static constexpr uint32_t kBStage = NT * 128;    // NT rows x 64 bf16
  // Activation rows per TMA box (the tensor map is built to match): boxes
  // of 64 rows cut the copies per step four-fold for many-token chunks.
  static constexpr int kBoxRows = kATmem ? 16 : 64;
  // TMEM A: the four MMA warps' double-buffered accumulators in columns
  // 0..255, A from 256.
  static constexpr uint32_t kATmemCol = 256;       // first TMEM column of A
  static constexpr int kAccBufs = kATmem ? 2 : 1;
  static constexpr uint32_t kAccCols = kATmem ? NT * kMmaWarps : 512;  // per buffer
  // Dequant warps per stage: TMEM A splits the 16 warps into four groups of
  // four (one row quarter and a whole pair of K steps each), NT=256 into
  // two groups of eight (row quarter x K half) that fill one tile each.
  static constexpr int kDqPerStage = kATmem ? 4 : kDqGroups * kDqWarps;
  static constexpr int kDqPerF = kATmem ? 4 : kDqGroups * kDqWarps;
  static constexpr uint32_t kAOff = 0;
  static constexpr uint32_t kBOff = kAOff + kAStage * kSAa;
  static constexpr uint32_t kFOff = kBOff + kBStage * kSB;
  static constexpr uint32_t kBarOff = kFOff + kFStage * kSF;
  static constexpr int kNumBars = 2 * kSF + 2 * kSAa + 2 * kSB + 2 * kAccBufs + 1;
  // cstart[0..E] and offsets[0..E] copied to shared memory for the per-unit
  // lookups of every role.
  static constexpr uint32_t kTabOff = kBarOff + 8 * kNumBars + 16;
  // TMEM A: the CTA's work units (expert, block, first row, tokens), decoded
  // once at the start for up to kUnitTab units: every role then reads a
  // unit instead of searching the expert table at each unit boundary, where
  // the search sat on the MMA and activation producers' hand-off chain.
  static constexpr int kUnitTab = kATmem ? 640 : 0;
  static constexpr uint32_t kUnitOff = (kTabOff + 8 * (kMaxE + 1) + 15) & ~15u;
  static constexpr uint32_t kSmem = kUnitOff + 16 * kUnitTab + 1024;
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(kATmem ? (kAccBufs * kAccCols <= kATmemCol &&
                          kATmemCol + 64 * kSAa <= kTmemCols)
                       : kAccCols <= kTmemCols, "TMEM budget");
  static_assert(!kATmem || (kSB == 2 * kSAa && kSF % 4 == 0 && kSAa == 4 && kMmaWarps == 4),
                "TMEM A rings: stage g belongs to dequant group g and MMA warp g; "
                "B stages released with their pair's A stage");
  static_assert(kAOff % 1024 == 0 && kBOff % 1024 == 0 && kBStage % 1024 == 0,
                "swizzled operands need 1 KB alignment");
};

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

template <int NT, int MODE>
__global__ void __launch_bounds__(Cfg<NT>::kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
  using C = Cfg<NT>;
  constexpr int SF = C::kSF, SAa = C::kSAa, SB = C::kSB, MT = C::kMT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bars = sbase + C::kBarOff;
  auto fullF = [&](int s) { return bars + 8u * s; };
  auto emptyF = [&](int s) { return bars + 8u * (SF + s); };
  auto aready = [&](int s) { return bars + 8u * (2 * SF + s); };
  auto emptyA = [&](int s) { return bars + 8u * (2 * SF + SAa + s); };
  auto fullB = [&](int s) { return bars + 8u * (2 * SF + 2 * SAa + s); };
  auto emptyB = [&](int s) { return bars + 8u * (2 * SF + 2 * SAa + SB + s); };
  constexpr int kAccBar0 = 2 * SF + 2 * SAa + 2 * SB;
  auto accFull = [&](int b) { return bars + 8u * (kAccBar0 + b); };
  auto accEmpty = [&](int b) { return bars + 8u * (kAccBar0 + C::kAccBufs + b); };
  const uint32_t done_bar = bars + 8u * (kAccBar0 + 2 * C::kAccBufs);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + 8 * C::kNumBars);
  int* tab_cs = reinterpret_cast<int*>(smem + C::kTabOff);
  int* tab_os = tab_cs + (kMaxE + 1);
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) {
    tab_cs[i] = __ldg(a.cstart + i);
    tab_os[i] = __ldg(a.offsets + i);
  }
  const int nbu = (a.nblocks + MT - 1) / MT;   // weight-block groups per chunk

  if (threadIdx.x == 0) {
    for (int s = 0; s < SF; ++s) {
      mbar_init(fullF(s), 1);
      mbar_init(emptyF(s), C::kDqPerF);
    }
    for (int s = 0; s < SAa; ++s) {
      // TMEM A: aready(g) also takes the two activation producers' arrivals
      // (and TMA bytes) of the pair's K steps, so an MMA warp waits on one
      // barrier per pair.
      mbar_init(aready(s), C::kDqPerStage + (C::kATmem ? 2 : 0));
      mbar_init(emptyA(s), C::kATmem ? 1 : C::kMmaWarps);
    }
    for (int s = 0; s < SB; ++s) {
      mbar_init(fullB(s), 1);
      mbar_init(emptyB(s), C::kATmem ? 1 : C::kMmaWarps);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(accFull(b), C::kMmaWarps);
      mbar_init(accEmpty(b), C::kEpiWarps);
    }
    mbar_init(done_bar, C::kMmaWarps);
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
  const int total = nbu * tab_cs[a.E];
  const int nloc = static_cast<int>(blockIdx.x) < total
                       ? (total - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                       : 0;
  const bool utab = nloc <= C::kUnitTab;   // uniform over the block
  int4* utab_s = reinterpret_cast<int4*>(smem + C::kUnitOff);
  if (utab) {
    for (int i = threadIdx.x; i < nloc; i += blockDim.x) {
      const Unit U = decode_unit(a, nbu, MT, NT, tab_cs, tab_os, blockIdx.x + i * gridDim.x);
      utab_s[i] = make_int4(U.e, U.nb, U.row0, U.ntok);
    }
    __syncthreads();
  }
  // Unit u, the iu-th of this CTA.
  auto unit_at = [&](int iu, int u) -> Unit {
    if (utab) {
      const int4 v = utab_s[iu];
      return Unit{v.x, v.y, v.z, v.w};
    }
    return decode_unit(a, nbu, MT, NT, tab_cs, tab_os, u);
  };

  if (warp == kWarpFProd) {
    // ------------------------------------------------- weight producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x, iu = 0; u < total && ok; u += gridDim.x, ++iu) {
        const Unit U = unit_at(iu, u);
        const int tiles = min(MT, a.nblocks - U.nb);
        const uint8_t* wt = a.wpack + (static_cast<int64_t>(U.e) * a.nblocks + U.nb) *
                                          a.ksteps * a.tile_bytes;
        const int64_t tstride = static_cast<int64_t>(a.ksteps) * a.tile_bytes;
        // TMEM A: one copy of two consecutive K-step tiles per stage (one
        // 4.6 KB copy per step cannot keep HBM busy; ksteps is even).
        for (int ks = 0; ks < a.ksteps; ks += C::kStepsPerF) {
          if (!mbar_wait(emptyF(s), ph ^ 1u)) { ok = false; break; }
          if (C::kATmem) {
            mbar_arrive_expect_tx(fullF(s), 2 * a.tile_bytes);
            bulk_load(sbase + C::kFOff + s * C::kFStage,
                      wt + static_cast<int64_t>(ks) * a.tile_bytes, 2 * a.tile_bytes,
                      fullF(s));
          } else {
            mbar_arrive_expect_tx(fullF(s), tiles * a.tile_bytes);
            for (int t = 0; t < tiles; ++t)
              bulk_load(sbase + C::kFOff + s * C::kFStage + t * kFBytes,
                        wt + t * tstride + static_cast<int64_t>(ks) * a.tile_bytes,
                        a.tile_bytes, fullF(s));
          }
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
  } else if (warp == kWarpBProd || (C::kATmem && (warp == kWarpMma || warp >= C::kWarpBX0))) {
    // --------------------------------------------- activation producer(s)
    if (lane == 0) {
      const int nprod = C::kATmem ? 2 + C::kExtraB : 1;
      const int bp = (warp == kWarpBProd) ? 0 : (warp == kWarpMma) ? 1 : 2 + (warp - C::kWarpBX0);
      uint32_t n = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int u = blockIdx.x, iu = 0; u < total && ok; u += gridDim.x, ++iu) {
        const Unit U = unit_at(iu, u);
        const int nbox = (U.ntok + C::kBoxRows - 1) / C::kBoxRows;
        constexpr uint32_t kBoxBytes = C::kBoxRows * 128u;
        for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
          if (static_cast<int>(n % nprod) != bp) continue;
          const int s = static_cast<int>(n % SB);
          const uint32_t ph = (n / SB) & 1u;
          // TMEM A: the stage is free once the MMAs of the pair (n / 2) that
          // last used it completed (released with that pair's A stage).
          const bool fr = C::kATmem
              ? mbar_wait(emptyA(static_cast<int>((n >> 1) % SAa)),
                          (((n >> 1) / SAa) & 1u) ^ 1u)
              : mbar_wait(emptyB(s), ph ^ 1u);
          if (!fr) { ok = false; break; }
          // Completion barrier: fullB(s), or with TMEM A the pair's aready.
          const int cb = C::kATmem ? static_cast<int>((n >> 1) % SAa) : s;
          const uint32_t cph = C::kATmem ? ((n >> 1) / SAa) & 1u : ph;
          const uint32_t full = C::kATmem ? aready(cb) : fullB(cb);
          mbar_arrive_expect_tx(full, nbox * kBoxBytes);
          const uint32_t dst = sbase + C::kBOff + s * C::kBStage;
          // Rows past the chunk (up to the box) are loaded but not used;
          // rows past the tensor are zero-filled by the TMA unit.
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(dst + b * kBoxBytes, &tmB, ks * kTileK, U.row0 + C::kBoxRows * b,
                        full);
          issued |= 1u << cb;
          issued_ph = (issued_ph & ~(1u << cb)) | (cph << cb);
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      for (int t = 0; t < SB; ++t)
        if ((issued >> t) & 1u)
          mbar_wait(C::kATmem ? aready(t) : fullB(t), (issued_ph >> t) & 1u);
    }
  } else if (C::kATmem ? warp >= C::kWarpMmaX0
                        : (warp == kWarpMma || warp == C::kWarpMmaX0)) {
    // ---------------------------------------------------------------- MMA
    // TMEM A: warp mi takes the pairs of K steps m = n / 2 with
    // m % kMmaWarps == mi; shared-memory A: warp mi issues the MMAs of weight
    // tile mi in every step.
    const int mi = C::kATmem ? warp - C::kWarpMmaX0 : (warp == kWarpMma ? 0 : 1);
    if (lane == 0) {
      int buf = 0;
      uint32_t n = 0, acc_ph = 0;
      bool ok = true;
      const uint64_t adesc0 = sw128_kmajor_desc(sbase + C::kAOff);
      const uint64_t bdesc0 = sw128_kmajor_desc(sbase + C::kBOff);
      for (int u = blockIdx.x, iu = 0; u < total && ok; u += gridDim.x, ++iu) {
        const Unit U = unit_at(iu, u);
        const int tiles = min(MT, a.nblocks - U.nb);
        const uint32_t nn = static_cast<uint32_t>((U.ntok + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(128, nn);
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf) * C::kAccCols +
                                static_cast<uint32_t>(mi * NT);
        if (!mbar_wait(accEmpty(buf), acc_ph ^ 1u)) { ok = false; break; }
        tc_fence_after();
        uint32_t acc = 0;
        for (int ks = 0; ks < a.ksteps; ks += (C::kATmem ? 2 : 1), n += (C::kATmem ? 2 : 1)) {
          // TMEM A: pair m = n / 2 of K tiles, taken by MMA warp m % 4.
          const uint32_t m = n >> 1;
          if (C::kATmem && static_cast<int>(m % C::kMmaWarps) != mi) continue;
          const int sa = static_cast<int>(C::kATmem ? m % SAa : n % SAa);
          const uint32_t pa = C::kATmem ? (m / SAa) & 1u : (n / SAa) & 1u;
          const int sb = static_cast<int>(n % SB);
          // TMEM A: aready(sa) also covers both K steps' activation rows.
          if ((!C::kATmem && !mbar_wait(fullB(sb), (n / SB) & 1u)) ||
              !mbar_wait(aready(sa), pa)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // Descriptors advance by the stage offset and 32 B per K=16 step
          // (2 in the descriptor's 16-byte address units).
          const uint64_t bd = bdesc0 + static_cast<uint64_t>((sb * C::kBStage) >> 4);
          if (C::kATmem) {
            const uint32_t at = tmem + C::kATmemCol + sa * 64u;
            const uint64_t bd1 = bdesc0 + static_cast<uint64_t>((((sb + 1) % SB) * C::kBStage) >> 4);
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk) {
              umma_f16_ta(d_tmem, at + kk * 8u, bd + 2u * kk, idesc, acc);
              acc = 1u;
            }
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk)
              umma_f16_ta(d_tmem, at + 32u + kk * 8u, bd1 + 2u * kk, idesc, 1u);
          } else if (mi < tiles) {
            // Tile mi -> accumulator columns 256 mi (d_tmem).
            const uint64_t ad = adesc0 + static_cast<uint64_t>((sa * C::kAStage) >> 4) +
                                (kABytes >> 4) * static_cast<uint32_t>(mi);
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk) {
              umma_f16(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc, acc);
              acc = 1u;
            }
          }
          umma_commit(emptyA(sa));
          if (!C::kATmem) umma_commit(emptyB(sb));
        }
        if (!ok) break;
        umma_commit(accFull(buf));
        if (++buf == C::kAccBufs) { buf = 0; acc_ph ^= 1u; }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      // Let every issued MMA finish before TMEM is released.
      umma_commit(done_bar);
      if (!mbar_wait(done_bar, 0)) record_error(a.err, FP4MOE_ERR_TIMEOUT);
    }
  } else if (warp < kWarpEpi0 && C::kATmem) {
    // ------------------------------------------- dequant, A in TMEM (NT=32)
    // Group g (four warps) takes the pairs of K tiles m = g (mod 4): the F
    // stage m % SF holds both tiles, A stage g (64 columns) receives them.
    // Warp q of the group converts rows 32q.. into TMEM lanes 32q.. (the
    // lane quarter its warp may write).
    const int grp = (warp - kWarpDq0) >> 2;
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t smul2 = a.smul * 0x10001u, sadd2 = a.sadd * 0x10001u;
    const uint32_t t_st = tmem + (static_cast<uint32_t>(32 * q) << 16) + C::kATmemCol +
                          static_cast<uint32_t>(grp) * 64u;
    uint32_t pha = 0;
    uint32_t n = 0;                   // K steps of this CTA before the unit
    bool ok = true;
    for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
      for (int ks = 2 * ((grp - static_cast<int>(n >> 1)) & 3); ks < a.ksteps; ks += 8) {
        // CTA-wide pair index m (m = grp mod 4): weight stage m % SF.
        const uint32_t m = (n + static_cast<uint32_t>(ks)) >> 1;
        const int sf = static_cast<int>(m % SF);
        const uint32_t phf = (m / SF) & 1u;
        if (!mbar_wait(fullF(sf), phf)) { ok = false; break; }
        // Both tiles' packed words and scale pairs are read into registers
        // first, so the F stage is released before the A-stage wait.
        const uint8_t* f0 = smem + C::kFOff + sf * C::kFStage;
        uint4 d[4];
        uint32_t sc2[8];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint8_t* f = f0 + t * a.tile_bytes;
          d[2 * t] = *reinterpret_cast<const uint4*>(f + r * 16);
          d[2 * t + 1] = *reinterpret_cast<const uint4*>(f + 2048 + r * 16);
          if (a.gran == 16) {
            const uint8_t* sc = f + kTileDataBytes + r * 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) sc2[4 * t + j] = sc[j] * smul2 + sadd2;
          } else {
            const uint8_t* sc = f + kTileDataBytes + r * 2;
            sc2[4 * t] = sc2[4 * t + 1] = sc[0] * smul2 + sadd2;
            sc2[4 * t + 2] = sc2[4 * t + 3] = sc[1] * smul2 + sadd2;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(emptyF(sf));
        auto convert = [&](int t, uint32_t (&va)[16], uint32_t (&vb)[16]) {
          const uint4 d0 = d[2 * t], d1 = d[2 * t + 1];
          const uint32_t s0 = sc2[4 * t], s1 = sc2[4 * t + 1], s2 = sc2[4 * t + 2],
                         s3 = sc2[4 * t + 3];
          const uint4 w0 = dequant8(d0.x, s0), w1 = dequant8(d0.y, s0);
          const uint4 w2 = dequant8(d0.z, s1), w3 = dequant8(d0.w, s1);
          const uint4 w4 = dequant8(d1.x, s2), w5 = dequant8(d1.y, s2);
          const uint4 w6 = dequant8(d1.z, s3), w7 = dequant8(d1.w, s3);
          const uint4 wa[4] = {w0, w1, w2, w3}, wb[4] = {w4, w5, w6, w7};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            va[4 * x] = wa[x].x; va[4 * x + 1] = wa[x].y;
            va[4 * x + 2] = wa[x].z; va[4 * x + 3] = wa[x].w;
            vb[4 * x] = wb[x].x; vb[4 * x + 1] = wb[x].y;
            vb[4 * x + 2] = wb[x].z; vb[4 * x + 3] = wb[x].w;
          }
        };
        uint32_t va[16], vb[16];
        convert(0, va, vb);
        if (!mbar_wait(emptyA(grp), pha ^ 1u)) { ok = false; break; }
        tc_fence_after();             // after the MMA that last read this stage
        tmem_st16(t_st, va);
        tmem_st16(t_st + 16u, vb);
        convert(1, va, vb);
        tmem_st16(t_st + 32u, va);
        tmem_st16(t_st + 48u, vb);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(aready(grp));
        pha ^= 1u;
      }
      n += static_cast<uint32_t>(a.ksteps);
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  } else if (warp < kWarpEpi0) {
    // ------------------------------------ dequant, A in shared memory (NT=256)
    const int dq = warp - kWarpDq0;   // 0 .. 15
    const int grp = dq / kDqWarps;
    const int w8 = dq % kDqWarps;
    const int q = warp & 3;           // row quarter = TMEM lane quarter
    const int khalf = w8 >> 2;        // 32-wide K half of each step
    const int r = 32 * q + lane;      // weight row in the tile
    const uint32_t smul2 = a.smul * 0x10001u, sadd2 = a.sadd * 0x10001u;
    const uint32_t a_row_off = (r >> 3) * 1024u + (r & 7) * 128u;
    const uint32_t sw = r & 7, cb = 4 * khalf;
    // Group g fills weight tile g of every step (nothing to load when the
    // unit's second block does not exist: odd block count).
    const int tile = grp;
    uint32_t n = 0;                   // global K-step counter of this CTA
    bool ok = true;
    for (int u = blockIdx.x, iu = 0; u < total && ok; u += gridDim.x, ++iu) {
      const bool live = unit_at(iu, u).nb + tile < a.nblocks;
      for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
        const int sf = static_cast<int>(n % SF), sa = static_cast<int>(n % SAa);
        const uint32_t phf = (n / SF) & 1u, pha = (n / SAa) & 1u;
        uint4 w0, w1, w2, w3;
        if (live) {
          if (!mbar_wait(fullF(sf), phf)) { ok = false; break; }
          const uint8_t* f = smem + C::kFOff + sf * C::kFStage + tile * kFBytes;
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
          // (c * smul + sadd) * 0x10001: the bf16 scale in both halves.
          const uint32_t s0 = c0 * smul2 + sadd2, s1 = c1 * smul2 + sadd2;
          w0 = dequant8(d.x, s0); w1 = dequant8(d.y, s0);
          w2 = dequant8(d.z, s1); w3 = dequant8(d.w, s1);
        } else {
          // No second weight block (odd block count): nothing to load.
          if (!mbar_wait(fullF(sf), phf)) { ok = false; break; }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(emptyF(sf));
        if (!mbar_wait(emptyA(sa), pha ^ 1u)) { ok = false; break; }
        if (live) {
          if (C::kATmem) {
            tc_fence_after();   // after the MMA that last read this stage
            // Row r of A -> TMEM lane r; this K half -> 16 columns.
            const uint32_t v[16] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w,
                                    w2.x, w2.y, w2.z, w2.w, w3.x, w3.y, w3.z, w3.w};
            tmem_st16(tmem + (static_cast<uint32_t>(32 * q) << 16) + C::kATmemCol +
                          sa * 32u + khalf * 16u, v);
            tmem_st_wait();
            tc_fence_before();
          } else {
            const uint32_t arow = sbase + C::kAOff + sa * C::kAStage + tile * kABytes + a_row_off;
            st_shared_v4(arow + (((cb + 0) ^ sw) << 4), w0);
            st_shared_v4(arow + (((cb + 1) ^ sw) << 4), w1);
            st_shared_v4(arow + (((cb + 2) ^ sw) << 4), w2);
            st_shared_v4(arow + (((cb + 3) ^ sw) << 4), w3);
            fence_proxy_async_smem();
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(aready(sa));
      }
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  } else {
    // --------------------------------------------------------- epilogue
    const int ew = warp - kWarpEpi0;  // 0 .. kEpiWarps-1
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    constexpr int kParts = C::kEpiWarps / 4;
    const int part = ew >> 2;         // this warp's share of the quarter's work
    const int r = 32 * q + lane;      // weight row in the tile
    int buf = 0;
    uint32_t acc_ph = 0;
    uint32_t n_unit = 0;              // K steps of this CTA before the unit
    bool ok = true;
    for (int u = blockIdx.x, iu = 0; u < total && ok;
         u += gridDim.x, ++iu, n_unit += a.ksteps) {
      const Unit U = unit_at(iu, u);
      if (!mbar_wait(accFull(buf), acc_ph)) { ok = false; break; }
      tc_fence_after();
      const float alpha = __ldg(a.alpha + U.e);
      const int nchunks = (U.ntok + 15) >> 4;
      const uint32_t t_base = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                              static_cast<uint32_t>(buf) * C::kAccCols;
      // Stores one 16-column chunk j of accumulator values v of weight
      // block nb.
      auto emit16 = [&](const uint32_t (&v)[16], int j, int nb) {
        if (MODE == kGemmModeFc2) {
          float* o = static_cast<float*>(a.out);
          const int64_t col_n = static_cast<int64_t>(nb) * kTileN + r;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int col = 16 * j + c;
            if (col < U.ntok)
              o[static_cast<int64_t>(U.row0 + col) * a.ldo + col_n] =
                  __uint_as_float(v[c]) * alpha;
          }
        } else {
          // Lanes 0..15 hold gate rows, 16..31 the up rows of the same 16
          // intermediate columns; one exchange per column pair.
          const int i = nb * 64 + 16 * q + (lane & 15);
          const bool is_gate = lane < 16;
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float a0 = __uint_as_float(v[2 * m]), a1 = __uint_as_float(v[2 * m + 1]);
            const float recv = __shfl_xor_sync(kFull, is_gate ? a1 : a0, 16);
            const float g = (is_gate ? a0 : recv) * alpha;
            const float up = (is_gate ? recv : a1) * alpha;
            // silu(g) = g / (1 + e^-g); fast exp and division keep the
            // relative error within a few 1e-6.
            const float h = __fdividef(g, 1.0f + __expf(-g)) * up;
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
      };
      if (MT > 1) {
        // Items (tile, pair of chunks), tiles interleaved, taken round robin
        // by the kParts warps of this lane quarter; one TMEM load and wait
        // per item (32 columns).  (Releasing each tile on its own gained
        // nothing: the two tiles' MMA warps share the activation ring.)
        const int npairs = (nchunks + 1) >> 1;
        for (int it = part; it < 2 * npairs; it += kParts) {
          const int tile = it & 1, j = 2 * (it >> 1);
          const int nb = U.nb + tile;
          if (nb >= a.nblocks) continue;   // odd block count: no second tile
          uint32_t v[32];
          tmem_ld32(t_base + 256u * tile + 16 * j, v);
          tmem_ld_wait(v);
          uint32_t v0[16], v1[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) { v0[x] = v[x]; v1[x] = v[16 + x]; }
          emit16(v0, j, nb);
          if (j + 1 < nchunks) emit16(v1, j + 1, nb);
        }
      } else {
        const int nb = U.nb;
        const bool live = nb < a.nblocks;
        // Sum the partial accumulators (NT columns apart) of the MMA warps
        // that had K steps in this unit: warp m took the steps with
        // (n_unit + ks) % kMmaWarps == m, none when ksteps is short.
        const int m0 = static_cast<int>((n_unit >> 1) % C::kMmaWarps);
        const int nparts = min(C::kMmaWarps, a.ksteps / 2);
        for (int j = part; live && j < nchunks; j += kParts) {
          uint32_t v[16];
          tmem_ld16(t_base + static_cast<uint32_t>(m0 * NT) + 16 * j, v);
          tmem_ld_wait(v);
          for (int p = 1; p < nparts; ++p) {
            const int m = (m0 + p) % C::kMmaWarps;
            uint32_t w[16];
            tmem_ld16(t_base + static_cast<uint32_t>(m * NT) + 16 * j, w);
            tmem_ld_wait(w);
#pragma unroll
            for (int x = 0; x < 16; ++x)
              v[x] = __float_as_uint(__uint_as_float(v[x]) + __uint_as_float(w[x]));
          }
          emit16(v, j, nb);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(accEmpty(buf));
      if (++buf == C::kAccBufs) { buf = 0; acc_ph ^= 1u; }
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  }

  // ---- teardown: the MMA threads have waited (bounded) for their final
  // commits, so no UMMA is still writing TMEM; free it.
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// The dynamic shared-memory opt-in is a per-device function attribute: it is
// set once per device (and kernel instantiation), under a lock.
template <int NT, int MODE>
cudaError_t launch_one(const CUtensorMap& tmB, const GemmArgs& a, int grid,
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
      e = cudaFuncSetAttribute(moe_gemm_kernel<NT, MODE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(Cfg<NT>::kSmem));
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  moe_gemm_kernel<NT, MODE><<<grid, Cfg<NT>::kThreads, Cfg<NT>::kSmem, st>>>(tmB, a);
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

int gemm_chunk_max(int T) { return T <= 64 ? 32 : 256; }

int gemm_box_rows(int chunk) { return chunk <= 32 ? Cfg<32>::kBoxRows : Cfg<256>::kBoxRows; }

cudaError_t launch_gemm(const CUtensorMap& tmB, const GemmArgs& a, int nt,
                        int num_sms, cudaStream_t st) {
  const int grid = num_sms > 0 ? num_sms : 1;
  if (nt <= 32) return launch_nt<32>(tmB, a, grid, st);
  return launch_nt<256>(tmB, a, grid, st);
}

}  // namespace fp4moe
