// Host-side declarations shared by the fp4moe translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fp4moe {

constexpr int kTokPerBlk = 32;   // tokens per routing / scatter block
constexpr int kMaxE = 1024;      // experts supported by the routing kernels
constexpr int kMaxTopK = 16;
constexpr int kTileN = 128;      // packed weight tile rows (UMMA M)
constexpr int kTileK = 64;       // packed weight tile K (one 128-B bf16 row)
constexpr int kTileDataBytes = kTileN * kTileK / 2;  // 4096

// Packed tile bytes for a scale granularity: E2M1 data + one scale code per
// group and row.
constexpr int tile_bytes(int gran) {
  return kTileDataBytes + kTileN * (kTileK / gran);
}

// ---------------------------------------------------------------- kernels
cudaError_t launch_requant(const uint8_t* fp4, const uint8_t* s16,
                           int64_t rows, int64_t K, uint8_t* fp4_out,
                           uint8_t* s32_out, int* err, cudaStream_t st);

cudaError_t launch_act_quant(const uint16_t* x, int64_t T, int64_t K,
                             uint8_t* xq, uint8_t* xs, int* err,
                             cudaStream_t st);

// FP8 rounding of FP32 h [rows, I] to exact-bf16 E4M3 x UE8M0/32 values.
cudaError_t launch_h_fp8_round(const float* h, int64_t rows, int64_t I,
                               uint16_t* out, cudaStream_t st);

// S2: ids/w per pair and a per-block expert histogram hist[nblk][E].
cudaError_t launch_route(const float* logits, int T, int E, int k,
                         int32_t* ids, float* w, int32_t* hist, int* err,
                         cudaStream_t st);

// S3 (scan): counts, offsets, per-block bases, and the GEMM token-chunk
// prefix cstart[E+1] for chunks of at most chunk_max tokens.
cudaError_t launch_scan(int T, int E, const int32_t* hist, int32_t* base,
                        int32_t* counts, int32_t* offsets, int32_t* cstart,
                        int chunk_max, cudaStream_t st);

// S3 (scatter): perm/inv and, if xperm != nullptr, the gathered activation
// rows in expert-major order as bf16 (FP8 inputs are dequantized exactly).
cudaError_t launch_scatter(const int32_t* ids, int T, int E, int k,
                           const int32_t* base, int32_t* perm, int32_t* inv,
                           const void* x, const uint8_t* xs, int K,
                           int act_mode, uint16_t* xperm, int* err, cudaStream_t st);

// S3 (gather alone): the activation rows in expert-major order, as above.
cudaError_t launch_gather(const int32_t* inv, int T, int k, const void* x, const uint8_t* xs,
                          int K, int act_mode, uint16_t* xperm, int* err, cudaStream_t st);

// S2 + S3 (route, scan, scatter) for 1 <= T <= kTokPerBlk tokens in one
// launch, with the outputs of launch_route + launch_scan + launch_scatter
// (hist and base are not written).
cudaError_t launch_route_small(const float* logits, int T, int E, int k, int chunk_max,
                               int32_t* ids, float* w, int32_t* counts, int32_t* offsets,
                               int32_t* cstart, int32_t* perm, int32_t* inv, int* err,
                               cudaStream_t st);

// S7: y[t] = sum_j w[t,j] * o[inv[t,j]] -> bf16.
cudaError_t launch_combine(const float* o, const int32_t* inv, const float* w,
                           int T, int k, int K, uint16_t* y, int* err, cudaStream_t st);

// S0: pack one weight matrix [E, N, Kd] into tiles.  gated: FC1 gate/up
// interleave with `layout` giving the source half order.  bmax: per-expert
// maximum UE8M0 byte (gran 32) or nullptr.
cudaError_t launch_scale_max(const uint8_t* s, int E, int64_t per_expert,
                             int32_t* bmax, int* err, cudaStream_t st);
cudaError_t launch_pack(const uint8_t* w, const uint8_t* s, int E, int N,
                        int Kd, int gran, bool gated, int layout,
                        const int32_t* bmax, uint8_t* out, int* err,
                        cudaStream_t st);
// alpha = gs (or 1 / gs when the global scales are stored inverted) times
// the power of two that the packed scale codes leave out (gran 16, 32);
// gran 0: gs alone (block-scaled path, whose scales the MMA applies).
cudaError_t launch_alpha(const float* gs, const int32_t* bmax, int E,
                         int gran, bool inverted, float* alpha, cudaStream_t st);

// S5 / S6: grouped GEMM over packed weights.
struct GemmArgs {
  const uint8_t* wpack;    // packed tiles [E][N/128][Kd/64]
  const float* alpha;      // [E] epilogue scale
  const int32_t* offsets;  // [E+1] token offsets (expert-major rows)
  const int32_t* cstart;   // [E+1] token-chunk prefix
  void* out;               // FC1: h [P, N/2]; FC2: o f32 [P, N]
  int* err;
  int64_t rows;            // P: rows of the expert-major buffers
  int E, nblocks, ksteps, tile_bytes, gran;
  uint32_t smul, sadd;     // scale code -> bf16 bits
  int ldo;                 // output row stride in elements
  int mode;                // 0: FC1 + SwiGLU (bf16 h), 1: FC2 (f32 o),
                           // 2: FC1 + SwiGLU writing FP32 h (rounded to
                           //    E4M3 x UE8M0/32 by launch_h_fp8_round)
};
constexpr int kGemmModeFc1 = 0, kGemmModeFc2 = 1, kGemmModeFc1Fp8 = 2;

cudaError_t launch_gemm(const CUtensorMap& tmB, const GemmArgs& a, int nt,
                        int num_sms, cudaStream_t st);
// The same GEMM on CTA pairs (tcgen05 cta_group::2, chunks of up to 256
// tokens, activation boxes of kPairBoxRows rows): for an even number of
// 128-row blocks and of K steps.
constexpr int kPairBoxRows = 128;
bool gemm_pair_supported(const GemmArgs& a);
cudaError_t launch_gemm_pair(const CUtensorMap& tmB, const GemmArgs& a, int num_sms,
                             cudaStream_t st);

// S5 / S6 on the block-scaled path (FP8 activations over group32 weights):
// kind::mxf8f6f4, E2M1 weights widened by TMA, E4M3 rows, UE8M0 scales.
constexpr int kMxK = 128;             // K elements per step
constexpr int kMxChunk = 224;         // tokens per unit (accumulator columns)
constexpr int kMxChunk256Rows = 256;  // largest activation box (rows)
constexpr int kMxSfSlots = 4;         // scale-factor slots in TMEM
struct MxGemmArgs {
  const uint32_t* wscale;  // [E][tiles][ksteps][128] UE8M0 words (4 blocks)
  const uint32_t* xscale;  // [ksteps][xscale_pitch] words of the B rows
  const float* alpha;      // [E] epilogue scale (global scale)
  const int32_t* offsets;  // [E+1] token offsets (expert-major rows)
  const int32_t* cstart;   // [E+1] token-chunk prefix (chunks <= kMxChunk)
  void* out;               // FC1: h E4M3 [P, ldo]; FC2: o f32 [P, ldo]
  uint8_t* hscale;         // FC1: h scale words [I/128][hscale_pitch]
  int* err;
  int64_t rows;            // P: rows of the expert-major buffers
  int E, nblocks, ksteps, rows_per_expert, tiles_per_expert;
  int64_t xscale_pitch, hscale_pitch;  // words per step row
  int ldo;
  int mode;                // kGemmModeFc1 (SwiGLU, FP8 h) or kGemmModeFc2
};
// S0 of the block-scaled path: rows of one weight matrix [E, N, Kd/2] copied
// (FC1 reordered: per 128-column block the gate rows then the up rows), and
// its UE8M0 scales [E, N, Kd/32] regrouped as one word per row and 128-wide
// step, [E][N/128][Kd/128][128].
cudaError_t launch_mx_rows(const uint8_t* w, int E, int N, int Kd, bool gated, int layout,
                           uint8_t* out, cudaStream_t st);
cudaError_t launch_mx_scales(const uint8_t* s, int E, int N, int Kd, bool gated, int layout,
                             uint32_t* out, int* err, cudaStream_t st);
// S3 gather of the block-scaled path: E4M3 rows to xperm [P, K] and their
// scale words to xsperm [K/128][pitch].
cudaError_t launch_gather_mx(const int32_t* inv, int T, int k, const uint8_t* x,
                             const uint8_t* xs, int K, int64_t pitch, uint8_t* xperm,
                             uint32_t* xsperm, int* err, cudaStream_t st);
// Tensor maps of one block-scaled GEMM: the weights (16U4_ALIGN16B, 128 x
// 128 boxes) and the activation rows with boxes of 32, 64, ..., 256 rows
// (E4M3, 128-byte swizzle).
constexpr int kMxBoxes = 8;
struct MxMaps {
  CUtensorMap w;
  CUtensorMap x[kMxBoxes];   // x[j]: boxes of 32 (j + 1) rows
};
cudaError_t launch_gemm_mx(const MxMaps& maps, const MxGemmArgs& a, int num_sms,
                           cudaStream_t st);
// The same GEMM on CTA pairs (tcgen05 cta_group::2): FC1 needs an even
// number of 128-column blocks, FC2 a number of 128-row blocks divisible by 4.
bool gemm_mx_pair_supported(const MxGemmArgs& a);
cudaError_t launch_gemm_mx_pair(const MxMaps& maps, const MxGemmArgs& a, int num_sms,
                                cudaStream_t st);

// Chunk size (tokens) a GEMM launch for T tokens uses; the scan needs it.
int gemm_chunk_max(int T);
// Rows per TMA box of the activation tensor map for that chunk size.
int gemm_box_rows(int chunk);

// Device address of the per-device status word (kernels record errors there).
int* status_word();

// Number of SMs of the current device (cached per device, thread-safe).
int device_sm_count();

// Test helper: one thread waits, with a bounded wait of limit_ns, on an
// mbarrier that nothing completes, and records TIMEOUT in *err.
cudaError_t launch_wait_timeout(unsigned long long limit_ns, int* err,
                                cudaStream_t st);
// Test helper: one write of slot `index` of a 64-entry device array through
// the index check; out of range records BOUNDS in *err and writes nothing.
cudaError_t launch_bounds_check(int64_t index, int* err, cudaStream_t st);

}  // namespace fp4moe
