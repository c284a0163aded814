// Grouped GEMM of the MoE expert FFN over packed FP4 weights on CTA pairs
// (sm_103a, tcgen05 with cta_group::2): the many-token variant of FC1 (gate|up
// with the SwiGLU epilogue) and FC2.
//
// A work unit is (expert e, pair of 128-row weight blocks 2bp and 2bp+1,
// chunk of up to 256 tokens of e).  The two CTAs of a cluster share it:
//     D[256 x n] = W[blocks 2bp, 2bp+1][256 x Kd] * X_chunk[n x Kd]^T
// CTA r dequantizes weight block 2bp + r (FP4 -> bf16) into its own TMEM --
// the A rows of the M = 256 MMA -- and loads token rows [r n/2, (r+1) n/2) of
// the chunk by TMA into its shared memory -- its half of the B columns.  One
// thread of CTA 0 issues every MMA (kind::f16, M = 256, N = n, K = 16, A from
// TMEM); each CTA receives its 128 rows of D in its own TMEM and runs its own
// epilogue.  Against the one-CTA kernel this halves the activation traffic
// into each SM, takes the dequantized weights out of shared memory entirely
// (shared memory holds only the packed weights and the activation halves),
// and doubles the work of each issued MMA.
//
// Hand-offs run on mbarriers in each CTA; the ones the MMA thread needs from
// CTA 1 are forwarded: a thread of CTA 1 waits for its A stage and B halves of
// each pair of K steps and then arrives on CTA 0's barrier (one remote arrive
// per pair).  The MMA thread's commits are multicast to the barriers of both
// CTAs (A stage with its B stages, accumulator full, done); CTA 1's epilogue warps
// arrive on CTA 0's accumulator-empty barrier directly.
//
// Warp roles (32 warps, one CTA per SM):
//   warp 0       weight producer: one bulk copy per pair of K steps of the
//                CTA's packed tile into a ring of F stages;
//   warp 1       TMEM allocation (both CTAs, collectively); CTA 0: the MMA
//                thread; CTA 1: the forwarder;
//   warps 2, 3   activation producers (K steps n = 0, 1 mod 2): TMA of the
//                CTA's 128-row box of the chunk into a ring of B stages (two
//                per A stage, released with it);
//   warps 4..19  dequantizers, four groups of four; group g converts the
//                pairs of K steps m = g (mod 4) into TMEM A stage g (every
//                waiter on a stage sees each of its phases in turn);
//   warps 20..31 epilogue, three per TMEM lane quarter.
// TMEM (512 columns): the accumulator in columns 0..255 (single-buffered),
// A stage g (a pair of K steps, 128 K) in columns 256 + 64 g.
// All waits are bounded (about 2 s); a timeout records FP4MOE_ERR_TIMEOUT and
// the pair winds down, frees its TMEM and leaves the cluster together.
#include <mutex>

#include "common.cuh"
#include "gemm_parts.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned kFullMask = 0xFFFFFFFFu;

constexpr int kNMax = 256;                 // tokens per unit (MMA N)
constexpr int kWarpF = 0, kWarpMma = 1, kWarpB0 = 2, kWarpDq0 = 4, kWarpEpi0 = 20;
constexpr int kEpiWarps = 12, kEpiParts = kEpiWarps / 4;
constexpr int kWarps = kWarpEpi0 + kEpiWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kStagesA = 4;                // TMEM A stages = dequant groups
// B (activation halves, from L2): one slot of two K-step stages per A stage,
// released with it (a slot released by its own commit instead costs the MMA
// thread a commit per pair, more than a deeper B ring gains).  F (packed
// weights, from HBM): pairs of K steps, deep enough to cover HBM latency.
constexpr int kSB = 2 * kStagesA;          // B stages (one K step each)
constexpr int kSF = 8;                     // F stages (pairs of K steps)
constexpr uint32_t kBoxRows = 128;         // activation rows per CTA and step
constexpr uint32_t kBStage = kBoxRows * 128;          // 16 KB
constexpr uint32_t kFBytesPair = 2 * 4608;            // two packed tiles
constexpr uint32_t kTmemCols = 512, kATmemCol = 256;
constexpr uint32_t kBOff = 0;
constexpr uint32_t kFOff = kBOff + kBStage * kSB;
constexpr uint32_t kBarOff = kFOff + kFBytesPair * kSF;
constexpr int kNumBars = 2 * kSF + 2 * kStagesA + 3;
constexpr uint32_t kTabOff = kBarOff + 8 * kNumBars + 16;
constexpr uint32_t kSmem = kTabOff + 8 * (kMaxE + 1) + 1024;
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kATmemCol >= kNMax && kATmemCol + 64 * kStagesA <= kTmemCols, "TMEM budget");
static_assert(kWarpDq0 % 4 == 0 && kWarpEpi0 % 4 == 0,
              "warp w may only touch TMEM lane quarter w % 4");
static_assert(kSF % kStagesA == 0, "F stage m % kSF belongs to dequant group m % 4");
static_assert(kBOff % 1024 == 0 && kBStage % 1024 == 0, "swizzled B needs 1 KB alignment");

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_cta_rank();
  const uint32_t bars = sbase + kBarOff;
  auto fullF = [&](int s) { return bars + 8u * s; };
  auto emptyF = [&](int s) { return bars + 8u * (kSF + s); };
  // pairFull(g): A stage g converted (four dequant warps) and its two B
  // stages loaded (two producer arrivals with the TMA bytes) in this CTA;
  // in CTA 0 also the forwarded arrival of CTA 1 (the same, there).
  auto pairFull = [&](int g) { return bars + 8u * (2 * kSF + g); };
  auto emptyA = [&](int g) { return bars + 8u * (2 * kSF + kStagesA + g); };
  const uint32_t accFull = bars + 8u * (2 * kSF + 2 * kStagesA);
  const uint32_t accEmpty = accFull + 8u, done_bar = accFull + 16u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kNumBars);
  int* tab_cs = reinterpret_cast<int*>(smem + kTabOff);
  int* tab_os = tab_cs + (kMaxE + 1);
  for (int i = threadIdx.x; i <= a.E; i += blockDim.x) {
    tab_cs[i] = __ldg(a.cstart + i);
    tab_os[i] = __ldg(a.offsets + i);
  }
  const int nbp = a.nblocks / 2;   // block pairs per chunk (nblocks is even)

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSF; ++s) {
      mbar_init(fullF(s), 1);
      mbar_init(emptyF(s), 4);       // the four warps of the stage's group
    }
    for (int g = 0; g < kStagesA; ++g) {
      mbar_init(pairFull(g), 4 + 2 + (rank == 0 ? 1 : 0));
      mbar_init(emptyA(g), 1);       // multicast commit
    }
    mbar_init(accFull, 1);
    mbar_init(accEmpty, 2 * kEpiWarps);   // CTA 0: both CTAs' epilogue warps
    mbar_init(done_bar, 1);
    fence_barrier_init();
  }
  if (warp == kWarpB0 && lane == 0) prefetch_tensormap(&tmB);
  if (warp == kWarpMma) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // both CTAs' barriers initialized, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = nbp * tab_cs[a.E];
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == kWarpF) {
    // ------------------------------------------------- weight producer
    if (lane == 0) {
      uint32_t m = 0, issued = 0, issued_ph = 0;   // m: pairs of K steps so far
      bool ok = true;
      for (int u = pair; u < total && ok; u += npairs) {
        const Unit U = decode_unit(a, nbp, 2, kNMax, tab_cs, tab_os, u);
        const uint8_t* wt = a.wpack +
            (static_cast<int64_t>(U.e) * a.nblocks + U.nb + static_cast<int>(rank)) *
                a.ksteps * a.tile_bytes;
        for (int ks = 0; ks < a.ksteps; ks += 2, ++m) {
          const int s = static_cast<int>(m % kSF);
          const uint32_t ph = (m / kSF) & 1u;
          if (!mbar_wait(emptyF(s), ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(fullF(s), 2 * a.tile_bytes);
          bulk_load(sbase + kFOff + s * kFBytesPair, wt + static_cast<int64_t>(ks) * a.tile_bytes,
                    2 * a.tile_bytes, fullF(s));
          issued |= 1u << s;
          issued_ph = (issued_ph & ~(1u << s)) | (ph << s);
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      // Copies still in flight must land before the CTA exits.
      for (int t = 0; t < kSF; ++t)
        if ((issued >> t) & 1u) mbar_wait(fullF(t), (issued_ph >> t) & 1u);
    }
  } else if (warp == kWarpB0 || warp == kWarpB0 + 1) {
    // --------------------------------------------- activation producers
    if (lane == 0) {
      const uint32_t bp = static_cast<uint32_t>(warp - kWarpB0);
      uint32_t n = 0, issued = 0, issued_ph = 0;   // n: K steps so far
      bool ok = true;
      for (int u = pair; u < total && ok; u += npairs) {
        const Unit U = decode_unit(a, nbp, 2, kNMax, tab_cs, tab_os, u);
        const int half = ((U.ntok + 15) & ~15) >> 1;   // B rows per CTA
        const int row = U.row0 + static_cast<int>(rank) * half;
        for (int ks = 0; ks < a.ksteps; ++ks, ++n) {
          if ((n & 1u) != bp) continue;
          // Pair m = n / 2 uses the slot of its A stage g = m % 4: stage
          // 2 g + (n % 2), free once the MMAs of the pair that last used it
          // completed (released with that pair's A stage).
          const uint32_t m = n >> 1;
          const int g = static_cast<int>(m % kStagesA), s = 2 * g + static_cast<int>(bp);
          const uint32_t ph = (m / kStagesA) & 1u;
          if (!mbar_wait(emptyA(g), ph ^ 1u)) { ok = false; break; }
          mbar_arrive_expect_tx(pairFull(g), kBStage);
          // Rows past this CTA's half (up to the box) are loaded but not
          // used; rows past the tensor are zero-filled by the TMA unit.
          tma_load_2d(sbase + kBOff + s * kBStage, &tmB, ks * kTileK, row, pairFull(g));
          issued |= 1u << g;
          issued_ph = (issued_ph & ~(1u << g)) | (ph << g);
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      for (int t = 0; t < kStagesA; ++t)
        if ((issued >> t) & 1u) mbar_wait(pairFull(t), (issued_ph >> t) & 1u);
    }
  } else if (warp == kWarpMma) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------- MMA (CTA 0)
      uint32_t m = 0, acc_ph = 0;
      bool ok = true;
      for (int u = pair; u < total && ok; u += npairs) {
        const Unit U = decode_unit(a, nbp, 2, kNMax, tab_cs, tab_os, u);
        const uint32_t nn = static_cast<uint32_t>((U.ntok + 15) & ~15);
        const uint32_t idesc = idesc_bf16_f32(256, nn);
        if (!mbar_wait_cluster(accEmpty, acc_ph ^ 1u)) { ok = false; break; }
        tc_fence_after();
        uint32_t acc = 0;
        for (int ks = 0; ks < a.ksteps; ks += 2, ++m) {
          const int g = static_cast<int>(m % kStagesA);
          const uint32_t ph = (m / kStagesA) & 1u;
          if (!mbar_wait(pairFull(g), ph)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t at = tmem + kATmemCol + 64u * static_cast<uint32_t>(g);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint64_t bd = sw128_kmajor_desc(sbase + kBOff + (2 * g + t) * kBStage);
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk) {
              umma_f16_ta_pair(tmem, at + 32u * t + 8u * kk, bd + 2u * kk, idesc, acc);
              acc = 1u;
            }
          }
          umma_commit_pair(emptyA(g));
        }
        if (!ok) break;
        umma_commit_pair(accFull);
        acc_ph ^= 1u;
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      // Every MMA issued has completed once `done` fires (in both CTAs).
      umma_commit_pair(done_bar);
      mbar_wait(done_bar, 0);
    } else if (lane == 0) {
      // -------------------------------------------- forwarder (CTA 1)
      uint32_t m = 0;
      bool ok = true;
      for (int u = pair; u < total && ok; u += npairs) {
        for (int ks = 0; ks < a.ksteps; ks += 2, ++m) {
          const int g = static_cast<int>(m % kStagesA);
          const uint32_t ph = (m / kStagesA) & 1u;
          if (!mbar_wait(pairFull(g), ph)) {
            ok = false;
            break;
          }
          mbar_arrive_cluster(pairFull(g), 0);
        }
      }
      if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
      mbar_wait(done_bar, 0);   // CTA 0's last MMA has completed
    }
  } else if (warp < kWarpEpi0) {
    // ---------------------------- dequant: FP4 -> bf16 into TMEM A stages
    const int grp = (warp - kWarpDq0) >> 2;
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const uint32_t smul2 = a.smul * 0x10001u, sadd2 = a.sadd * 0x10001u;
    const uint32_t t_st = tmem + (static_cast<uint32_t>(32 * q) << 16) + kATmemCol +
                          static_cast<uint32_t>(grp) * 64u;
    uint32_t pha = 0;
    uint32_t n = 0;                   // K steps of this CTA before the unit
    bool ok = true;
    for (int u = pair; u < total && ok; u += npairs) {
      for (int ks = 2 * ((grp - static_cast<int>(n >> 1)) & 3); ks < a.ksteps; ks += 8) {
        // CTA-wide pair index m (m = grp mod 4): weight stage m % kSF.
        const uint32_t m = (n + static_cast<uint32_t>(ks)) >> 1;
        const int sf = static_cast<int>(m % kSF);
        if (!mbar_wait(fullF(sf), (m / kSF) & 1u)) { ok = false; break; }
        // Converts packed tile t of the stage: the 16 words of K columns
        // 0..31 into va and those of 32..63 into vb.
        auto convert = [&](int t, uint32_t (&va)[16], uint32_t (&vb)[16]) {
          const uint8_t* f = smem + kFOff + sf * kFBytesPair + t * a.tile_bytes;
          const uint4 d0 = *reinterpret_cast<const uint4*>(f + r * 16);
          const uint4 d1 = *reinterpret_cast<const uint4*>(f + 2048 + r * 16);
          uint32_t s0, s1, s2, s3;    // bf16 scale pairs of the 16-wide groups
          if (a.gran == 16) {
            const uint8_t* sc = f + kTileDataBytes + r * 4;
            s0 = sc[0] * smul2 + sadd2;
            s1 = sc[1] * smul2 + sadd2;
            s2 = sc[2] * smul2 + sadd2;
            s3 = sc[3] * smul2 + sadd2;
          } else {
            const uint8_t* sc = f + kTileDataBytes + r * 2;
            s0 = s1 = sc[0] * smul2 + sadd2;
            s2 = s3 = sc[1] * smul2 + sadd2;
          }
          const uint4 wa[4] = {dequant8(d0.x, s0), dequant8(d0.y, s0), dequant8(d0.z, s1),
                               dequant8(d0.w, s1)};
          const uint4 wb[4] = {dequant8(d1.x, s2), dequant8(d1.y, s2), dequant8(d1.z, s3),
                               dequant8(d1.w, s3)};
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            va[4 * x] = wa[x].x; va[4 * x + 1] = wa[x].y;
            va[4 * x + 2] = wa[x].z; va[4 * x + 3] = wa[x].w;
            vb[4 * x] = wb[x].x; vb[4 * x + 1] = wb[x].y;
            vb[4 * x + 2] = wb[x].z; vb[4 * x + 3] = wb[x].w;
          }
        };
        // The first tile is converted before waiting for the A stage, so
        // the conversion overlaps the MMAs that still read the stage.
        uint32_t va[16], vb[16];
        convert(0, va, vb);
        if (!mbar_wait(emptyA(grp), pha ^ 1u)) { ok = false; break; }
        tc_fence_after();             // after the MMAs that last read this stage
        tmem_st16(t_st, va);
        tmem_st16(t_st + 16u, vb);
        convert(1, va, vb);
        tmem_st16(t_st + 32u, va);
        tmem_st16(t_st + 48u, vb);
        __syncwarp();
        if (lane == 0) mbar_arrive(emptyF(sf));
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pairFull(grp));
        pha ^= 1u;
      }
      n += static_cast<uint32_t>(a.ksteps);
    }
    if (!ok) record_error(a.err, FP4MOE_ERR_TIMEOUT);
  } else {
    // --------------------------------------------------------- epilogue
    const int q = warp & 3;           // TMEM lane quarter this warp may access
    const int part = (warp - kWarpEpi0) >> 2;
    const int r = 32 * q + lane;      // weight row in this CTA's tile
    const uint32_t t_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
    uint32_t acc_ph = 0;
    bool ok = true;
    for (int u = pair; u < total && ok; u += npairs) {
      const Unit U = decode_unit(a, nbp, 2, kNMax, tab_cs, tab_os, u);
      if (!mbar_wait(accFull, acc_ph)) { ok = false; break; }
      tc_fence_after();
      const float alpha = __ldg(a.alpha + U.e);
      const int nb = U.nb + static_cast<int>(rank);   // this CTA's weight block
      const int nchunks = (U.ntok + 15) >> 4;
      // Stores one 16-column chunk j of accumulator values v.
      auto emit16 = [&](const uint32_t (&v)[16], int j) {
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
          for (int mm = 0; mm < 8; ++mm) {
            const float a0 = __uint_as_float(v[2 * mm]), a1 = __uint_as_float(v[2 * mm + 1]);
            const float recv = __shfl_xor_sync(kFullMask, is_gate ? a1 : a0, 16);
            const float gv = (is_gate ? a0 : recv) * alpha;
            const float up = (is_gate ? recv : a1) * alpha;
            // silu(g) = g / (1 + e^-g); fast exp and division keep the
            // relative error within a few 1e-6.
            const float h = __fdividef(gv, 1.0f + __expf(-gv)) * up;
            const int col = 16 * j + 2 * mm + (is_gate ? 0 : 1);
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
      // Pairs of 16-column chunks, taken round robin by the three warps of
      // this lane quarter; one TMEM load and wait per pair (32 columns,
      // inside the allocation even past the accumulator's last column).
      // (Loading 16 columns at a time with the next load in flight drained
      // more slowly.)
      for (int j = 2 * part; j < nchunks; j += 2 * kEpiParts) {
        uint32_t v[32];
        tmem_ld32(t_base + 16u * j, v);
        tmem_ld_wait(v);
        uint32_t v0[16], v1[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) { v0[x] = v[x]; v1[x] = v[16 + x]; }
        emit16(v0, j);
        if (j + 1 < nchunks) emit16(v1, j + 1);
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

  // ---- teardown: CTA 0's MMA thread and CTA 1's forwarder have waited
  // (bounded) for the final commit, so no MMA still reads or writes either
  // CTA; the cluster barrier keeps both CTAs (their shared memory, the
  // barriers the other CTA arrives on) alive until both are done.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// The dynamic shared-memory opt-in and the number of CTA pairs that fit at
// once are per device: found once per device, under a lock.
template <int MODE>
cudaError_t launch_pair_mode(const CUtensorMap& tmB, const GemmArgs& a, int num_sms,
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
      e = cudaFuncSetAttribute(moe_gemm_pair_kernel<MODE>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmem));
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * static_cast<unsigned>(num_sms / 2));
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kSmem;
      cfg.stream = st;
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, moe_gemm_pair_kernel<MODE>, &cfg);
      if (e != cudaSuccess) return e;
      if (clusters < 1) return cudaErrorInvalidConfiguration;
      pairs_fit[dev] = clusters;
    }
    fit = pairs_fit[dev];
  }
  // A persistent grid: every pair must be resident at once.
  const int pairs = std::max(1, std::min(num_sms / 2, fit));
  moe_gemm_pair_kernel<MODE><<<2 * pairs, kThreads, kSmem, st>>>(tmB, a);
  return cudaGetLastError();
}

}  // namespace

bool gemm_pair_supported(const GemmArgs& a) {
  return a.nblocks % 2 == 0 && a.tile_bytes <= 4608 && a.ksteps % 2 == 0;
}

cudaError_t launch_gemm_pair(const CUtensorMap& tmB, const GemmArgs& a, int num_sms,
                             cudaStream_t st) {
  switch (a.mode) {
    case kGemmModeFc1: return launch_pair_mode<kGemmModeFc1>(tmB, a, num_sms, st);
    case kGemmModeFc2: return launch_pair_mode<kGemmModeFc2>(tmB, a, num_sms, st);
    default: return launch_pair_mode<kGemmModeFc1Fp8>(tmB, a, num_sms, st);
  }
}

}  // namespace fp4moe
