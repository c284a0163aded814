// Grouped GEMM of the MoE expert FFN with FP8 activations over group32 FP4
// weights on the block-scaled tensor-core path, on CTA pairs (sm_103a,
// tcgen05 kind::mxf8f6f4 with cta_group::2): recipe (1,1,32) of the group16
// notes page (section "Context"; section "Remaining kernel work" places this
// compute on the block-scaled MMA with the UE8M0 scales in tensor memory).
//
// The arithmetic is that of the one-CTA kernel (gemm_mx.cu): E2M1 weights
// widened by TMA (16U4_ALIGN16B), E4M3 rows, one UE8M0 byte per row and 32 K
// elements moved into TMEM by four scale warps, FP32 accumulators, the FC1
// epilogue applying SwiGLU and the (1,1,32) FP8 rounding of h.  Here two CTAs
// of a cluster share a work unit and every MMA has M = 256:
//   FC1  unit (expert e, pair of 128-column blocks 2p and 2p+1, chunk of up
//        to 224 tokens): CTA r holds the gate and the up tile of block
//        2p + r; MMA t (t = 0 gate, 1 up) takes A rows from both CTAs' tile t,
//        so each CTA receives G and U of its own block and runs its own
//        SwiGLU epilogue;
//   FC2  unit (expert e, four 128-row blocks 4p..4p+3, chunk): CTA r holds
//        blocks 4p + 2r + t, t = 0, 1.
// Each CTA loads half of the chunk's token rows (its half of the B columns)
// but the scale words of all of them: a pair MMA reads SFB for all N columns
// from each CTA's own TMEM (probed on the GB300, like the rest of the pair
// protocol).  One thread per MMA of CTA 0 issues (two threads, one per
// accumulator); their commits are multicast to both CTAs.  CTA 1 forwards
// its stage readiness with one relaxed remote arrive per K step.
//
// Warps (per CTA, 24):
//   0      weight producer: TMA of the CTA's two tiles and bulk copies of
//          their scale words, per 128-wide K step, into a ring of stages;
//   1, 3   CTA 0: MMA issuers of accumulators 0 and 1; CTA 1: warp 1 is the
//          forwarder;
//   2      activation producer: TMA of the CTA's half of the chunk's rows and
//          bulk copy of the scale words of all the chunk's rows;
//   4..7   scale warps (TMEM lane quarters): scale words -> TMEM slot of the
//          stage;
//   8..23  epilogue (lane quarter = warp % 4).
// All waits are bounded (about 2 s); a timeout records FP4MOE_ERR_TIMEOUT and
// the pair winds down, frees its TMEM and leaves the cluster together.
#include <algorithm>
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
constexpr int kStages = 4;
constexpr uint32_t kATile = 128 * 128;             // 128 rows x 128 B (widened E2M1)
constexpr uint32_t kATileTx = 128 * 64;            // bytes the TMA reads (packed)
constexpr uint32_t kBHalfRows = 128;               // largest half-chunk box
constexpr uint32_t kBBytes = kBHalfRows * 128;
constexpr uint32_t kSfaBytes = 128 * 4;            // one word per row
constexpr uint32_t kSfbBytes = (kMxChunk256Rows + 16) * 4;
constexpr uint32_t kOffA = 0, kOffB = 2 * kATile, kOffSfa = kOffB + kBBytes,
                   kOffSfb = kOffSfa + 2 * kSfaBytes;
constexpr uint32_t kStage = (kOffSfb + kSfbBytes + 1023) & ~1023u;
// Barriers per stage: full (TMA bytes), ready (scale warps; in CTA 0 also
// CTA 1's forwarded arrival), empty (both issuers' multicast commits).
constexpr int kNumBars = 3 * kStages + 3;
constexpr uint32_t kBarOff = kStage * kStages;
constexpr uint32_t kTabOff = kBarOff + 8 * kNumBars + 16;
constexpr uint32_t kSmem = kTabOff + 8 * (kMaxE + 1) + 1024;
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kOffB % 1024 == 0 && kStage % 1024 == 0, "swizzled operands need 1 KB alignment");
static_assert(kOffSfa % 16 == 0 && kOffSfb % 16 == 0, "bulk copies need 16 B alignment");
static_assert(kMxChunk / 2 <= static_cast<int>(kBHalfRows), "half-chunk box");
// TMEM: accumulators at columns 0 and 256 (N <= 224 each); the scale slot of
// stage s (16 columns: tile 0 SFA +0..3, tile 1 SFA +4..7, SFB +8..15) in
// the two gaps, at 224, 240, 480, 496.
constexpr uint32_t kAcc1Col = 256, kTmemCols = 512;
__host__ __device__ constexpr uint32_t sf_col(int j) {
  return j < 2 ? 224u + 16u * j : 480u + 16u * (j - 2);
}
static_assert(kStages <= kMxSfSlots && kMxChunk <= 224 && kAcc1Col + kMxChunk <= sf_col(2) &&
              sf_col(1) + 16 <= kAcc1Col && sf_col(kStages - 1) + 16 <= kTmemCols,
              "TMEM budget");
static_assert(kWarpSf0 % 4 == 0 && kWarpEpi0 % 4 == 0,
              "warp w may only touch TMEM lane quarter w % 4");

struct Unit {
  int e, p, row0, ntok;   // p: block pair (FC1) or block quad (FC2)
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
  U.p = local / nch;
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

// Weight tile t of CTA r in unit U: FC1, tile t of column block 2p + r (gate
// rows, then up rows: tile index 2 b + t within the expert); FC2, row block
// 4p + 2r + t.
template <int MODE>
__device__ __forceinline__ int tile_index(const Unit& U, uint32_t rank, int t) {
  return MODE == kGemmModeFc2 ? 4 * U.p + 2 * static_cast<int>(rank) + t
                              : 2 * (2 * U.p + static_cast<int>(rank)) + t;
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    moe_gemm_mx_pair_kernel(const __grid_constant__ MxMaps maps, const MxGemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const uint32_t bars = sbase + kBarOff;
  auto fullS = [&](int s) { return bars + 8u * s; };
  auto readyS = [&](int s) { return bars + 8u * (kStages + s); };
  auto emptyS = [&](int s) { return bars + 8u * (2 * kStages + s); };
  const uint32_t accFull = bars + 8u * (3 * kStages);
  const uint32_t accEmpty = accFull + 8u, done_bar = accFull + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kNumBars);
  int* tab_cs = reinterpret_cast<int*>(smem + kTabOff);
  int* tab_os = tab_cs + (kMaxE + 1);
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) {
    tab_cs[i] = __ldg(a.cstart + i);
    tab_os[i] = __ldg(a.offsets + i);
  }
  // Units per chunk: FC1 block pairs, FC2 block quads (the counts divide).
  const int nbu = (MODE == kGemmModeFc2) ? a.nblocks / 4 : a.nblocks / 2;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(fullS(s), 2);                          // weight, activation producers
      mbar_init(readyS(s), 4 + (rank == 0 ? 1 : 0));   // scale warps (+ CTA 1)
      mbar_init(emptyS(s), 2);                         // both issuers (multicast)
    }
    mbar_init(accFull, 2);
    mbar_init(accEmpty, 2 * kEpiWarps);                // CTA 0: both CTAs' epilogues
    mbar_init(done_bar, 2);
    fence_barrier_init();
  }
  if (warp == kWarpA && lane == 0) prefetch_tensormap(&maps.w);
  if (warp == kWarpB && lane < kMxBoxes) prefetch_tensormap(&maps.x[lane]);
  if (warp == kWarpMma0) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers initialized, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = nbu * tab_cs[a.E];
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == kWarpA || warp == kWarpB) {
    // ------------------------------------------------------ producers
    if (lane == 0) {
      const bool isA = warp == kWarpA;
      uint32_t n = 0, issued = 0, issued_ph = 0;
      bool ok = true;
      for (int u = pair; u < total && ok; u += npairs) {
        const Unit U = decode_unit(a, nbu, tab_cs, tab_os, u);
        const int half = ((U.ntok + 15) & ~15) >> 1;   // B rows per CTA
        const int hrows = (half + 31) & ~31;           // its box: 32 .. 128 rows
        const CUtensorMap* tmX = &maps.x[hrows / 32 - 1];
        // Scale words of all the chunk's rows, from a 16-byte-aligned start.
        const int lead = U.row0 & 3;
        const int brows = (U.ntok + 31) & ~31;
        const uint32_t sfb_bytes = static_cast<uint32_t>(((lead + brows + 3) & ~3) * 4);
        for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
          const int s = static_cast<int>(n % kStages);
          const uint32_t ph = (n / kStages) & 1u;
          if (!mbar_wait(emptyS(s), ph ^ 1u)) { ok = false; break; }
          const uint32_t st = sbase + s * kStage;
          if (isA) {
            mbar_arrive_expect_tx(fullS(s), 2 * (kATileTx + kSfaBytes));
            for (int t = 0; t < 2; ++t) {
              const int ti = tile_index<MODE>(U, rank, t);
              tma_load_2d(st + kOffA + t * kATile, &maps.w, ks * kMxK,
                          U.e * a.rows_per_expert + 128 * ti, fullS(s));
              // scale words of the tile at step ks: [tile group][ks][128 rows]
              const int64_t tg = static_cast<int64_t>(U.e) * a.tiles_per_expert + ti;
              bulk_load(st + kOffSfa + t * kSfaBytes, a.wscale + (tg * a.ksteps + ks) * 128,
                        kSfaBytes, fullS(s));
            }
          } else {
            mbar_arrive_expect_tx(fullS(s), static_cast<uint32_t>(hrows) * 128u + sfb_bytes);
            tma_load_2d(st + kOffB, tmX, ks * kMxK, U.row0 + static_cast<int>(rank) * half,
                        fullS(s));
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
    const int t = (warp == kWarpMma0) ? 0 : 1;
    if (lane == 0 && rank == 0) {
      // -------------------------------------------------- MMA (CTA 0)
      uint32_t n = 0, acc_ph = 0;
      bool ok = true;
      const uint32_t d_tmem = tmem + (t ? kAcc1Col : 0u);
      for (int u = pair; u < total && ok; u += npairs) {
        const Unit U = decode_unit(a, nbu, tab_cs, tab_os, u);
        const uint32_t nn = static_cast<uint32_t>((U.ntok + 15) & ~15);
        if (!mbar_wait_cluster(accEmpty, acc_ph ^ 1u)) { ok = false; break; }
        tc_fence_after();
        for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
          // ready(s): both CTAs' copies landed and scales are in their TMEM.
          const int s = static_cast<int>(n % kStages);
          if (!mbar_wait(readyS(s), (n / kStages) & 1u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * kStage;
          const uint64_t ad = sw128_kmajor_desc(st + kOffA + t * kATile);
          const uint64_t bd = sw128_kmajor_desc(st + kOffB);
          const uint32_t sfa = tmem + sf_col(s) + 4u * t;
          const uint32_t sfb = tmem + sf_col(s) + 8u;
#pragma unroll
          for (int kk = 0; kk < kMxK / 32; ++kk)
            umma_mx_pair(d_tmem, ad + 2u * kk, bd + 2u * kk, idesc_mx_e2m1_e4m3(256, nn, kk, kk),
                         sfa, sfb, (ks > 0 || kk > 0) ? 1u : 0u);
          umma_commit_pair(emptyS(s));
        }
        if (!ok) break;
        umma_commit_pair(accFull);
        acc_ph ^= 1u;
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      // Every MMA issued has completed once `done` fires (in both CTAs).
      umma_commit_pair(done_bar);
      if (!mbar_wait(done_bar, 0)) record_error(a.err, FP4MOE_ERR_TIMEOUT);
    } else if (lane == 0 && t == 0) {
      // -------------------------------------------- forwarder (CTA 1)
      uint32_t n = 0;
      bool ok = true;
      for (int u = pair; u < total && ok; u += npairs) {
        for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
          const int s = static_cast<int>(n % kStages);
          if (!mbar_wait(readyS(s), (n / kStages) & 1u)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(readyS(s), 0);
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      mbar_wait(done_bar, 0);   // CTA 0's last MMAs have completed
    }
  } else if (warp >= kWarpSf0 && warp < kWarpEpi0) {
    // ----------------------------------------------------- scale warps
    // Warp q (= warp % 4) owns TMEM lanes 32q..32q+31.  SFA of tile t: row
    // m = 32q + lane goes to lane m, column q (the column of its 32-row
    // block).  SFB: row n = 32c + lane of the whole chunk goes to column c of
    // every lane quarter, so each quarter of the accumulator reads its own
    // copy.
    const int q = warp & 3;
    uint32_t n = 0;
    bool ok = true;
    for (int u = pair; u < total && ok; u += npairs) {
      const Unit U = decode_unit(a, nbu, tab_cs, tab_os, u);
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
        for (int t = 0; t < 2; ++t) tmem_st1(col + 4u * t + q, sfa[t * 128 + 32 * q + lane]);
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
  } else if (warp >= kWarpEpi0) {
    // --------------------------------------------------------- epilogue
    const int ew = warp - kWarpEpi0;   // 0..15
    const int q = warp & 3;            // TMEM lane quarter
    const int part = ew >> 2;          // 0..3: FC1 column part; FC2 tile + half
    const int tile = part & 1;         // FC2: the accumulator (weight tile) it drains
    const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int u = pair; u < total && ok; u += npairs) {
      const Unit U = decode_unit(a, nbu, tab_cs, tab_os, u);
      if (!mbar_wait(accFull, acc_ph)) { ok = false; break; }
      tc_fence_after();
      const float alpha = __ldg(a.alpha + U.e);
      const int nchunks = (U.ntok + 15) >> 4;
      if (MODE == kGemmModeFc2) {
        const int nb = tile_index<MODE>(U, rank, tile);   // 128-row block of o's columns
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
      } else {
        // h for i = 128 b + 32 q + lane (b = 2p + rank); the 32 lanes are one
        // (1,1,32) group.  Per chunk of 16 tokens each lane packs its 16
        // codes four per word; a transpose over the warp then gives lane L
        // the codes of token 4k + L/8 for i = 4 (L % 8) .. + 3, stored as one
        // 32-bit word, and lanes 0..15 store the 16 tokens' scale bytes.
        const int b = 2 * U.p + static_cast<int>(rank);
        uint8_t* h8 = static_cast<uint8_t*>(a.out);
        const int tr = lane >> 3, tm = lane & 7;
        const int64_t i4 = static_cast<int64_t>(b) * 128 + 32 * q + 4 * tm;
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
            a.hscale[(static_cast<int64_t>(b) * a.hscale_pitch + U.row0 + 16 * c0 + lane) * 4 +
                     q] = static_cast<uint8_t>(my_sb);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) mbar_arrive(accEmpty);
        else mbar_arrive_cluster(accEmpty, 0);
      }
      acc_ph ^= 1u;
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  }

  // ---- teardown: CTA 0's issuers and CTA 1's forwarder waited (bounded)
  // for the final commits, so no MMA still reads or writes either CTA; the
  // cluster barrier keeps both CTAs alive until both are done.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == kWarpMma0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// The dynamic shared-memory opt-in and the number of CTA pairs that fit at
// once are per device: found once per device, under a lock.
template <int MODE>
cudaError_t launch_mx_pair_mode(const MxMaps& maps, const MxGemmArgs& a, int num_sms,
                                cudaStream_t st) {
  static std::mutex mu;
  static int pairs_fit[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int fit = 0;
  {
    std::lock_guard<std::mutex> g(mu);
    if (pairs_fit[dev] == 0) {
      e = cudaFuncSetAttribute(moe_gemm_mx_pair_kernel<MODE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmem));
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * static_cast<unsigned>(num_sms / 2));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmem;
      cfg.stream = st;
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, moe_gemm_mx_pair_kernel<MODE>, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters < 1) return cudaErrorInvalidConfiguration;
      pairs_fit[dev] = clusters;
    }
    fit = pairs_fit[dev];
  }
  // A persistent grid: every pair must be resident at once.
  const int pairs = std::max(1, std::min(num_sms / 2, fit));
  moe_gemm_mx_pair_kernel<MODE><<<2 * pairs, kThreads, kSmem, st>>>(maps, a);
  return cudaGetLastError();
}

}  // namespace

bool gemm_mx_pair_supported(const MxGemmArgs& a) {
  return a.mode == kGemmModeFc2 ? a.nblocks % 4 == 0 : a.nblocks % 2 == 0;
}

cudaError_t launch_gemm_mx_pair(const MxMaps& maps, const MxGemmArgs& a, int num_sms,
                                cudaStream_t st) {
  if (a.mode == kGemmModeFc2) return launch_mx_pair_mode<kGemmModeFc2>(maps, a, num_sms, st);
  return launch_mx_pair_mode<kGemmModeFc1>(maps, a, num_sms, st);
}

}  // namespace fp4moe
