/*
 * fp4moe -- fused Mixture-of-Experts expert FFN over block-scaled FP4 weights,
 * and the FP4 group16 -> group32 requantization, for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Every pointer argument is a DEVICE pointer owned by the caller unless
 * the comment says "host".  `stream` is a cudaStream_t passed as void* (NULL =
 * the legacy default stream).  Every call that takes a stream is asynchronous
 * on it (no host synchronisation) unless its comment says otherwise, and
 * returns a status code (fp4moe_status).  Argument checks happen on the host
 * before anything is launched; a non-zero status means nothing was launched.
 * Data-dependent errors found by a kernel (a NaN scale or logit, a bounded
 * device wait that gave up) are recorded in a per-device status word that
 * fp4moe_last_device_error() returns after the caller has synchronised.
 *
 * Formats (page "b12x/moe/fused/w4a16/prepare.py" unless noted):
 *   E2M1 FP4 codes: two per byte, the LOW nibble holds the even k element;
 *     code bit 3 = sign, bits 2..1 = exponent, bit 0 = mantissa, magnitudes
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 *   NVFP4 (gran_k 16): one E4M3 ("fn") scale byte per 16 K elements plus an
 *     FP32 global scale per expert matrix; weight = e2m1 * e4m3 * gs.
 *   MX (gran_k 32): one UE8M0 byte (2^(b-127)) per 32 K elements; the FP32
 *     global scale still multiplies in (1.0 for plain MX weights).
 *   bfloat16 tensors are passed as raw 16-bit words.
 */
#ifndef FP4MOE_H_
#define FP4MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  INVALID_ARG mirrors the prepare page's validation errors
 * (shape, dtype, divisibility); UNSUPPORTED mirrors the capability gate of
 * the group16 notes page (section "Current patch scope": a recipe the fused
 * compute refuses); TIMEOUT and CUDA_ERROR have no counterpart there. */
enum fp4moe_status {
  FP4MOE_OK = 0,
  FP4MOE_ERR_INVALID_ARG = 1,         /* bad shape, pointer, enum or value  */
  FP4MOE_ERR_UNSUPPORTED = 2,         /* valid request this build refuses   */
  FP4MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes below the *_size() query  */
  FP4MOE_ERR_CUDA = 4,                /* a CUDA runtime call failed         */
  FP4MOE_ERR_TIMEOUT = 5,             /* a bounded device wait gave up      */
  FP4MOE_ERR_BOUNDS = 6               /* an index check of the bounds-checked
                                         build failed (the access was skipped) */
};

/* Row order of the fused FC1 weight w13 [E, 2I, K].  "w31"/gate_up is the
 * kernel-native order (rows [0,I) = gate); "w13"/up_gate is the checkpoint
 * order (rows [0,I) = up), per the W13 layout notes of prepare.py. */
enum fp4moe_w13_layout { FP4MOE_W13_GATE_UP = 0, FP4MOE_W13_UP_GATE = 1 };

/* Activation format of moe_forward.  BF16 = W4A16.  FP8 = E4M3 values with a
 * per-token 1x32 UE8M0 scale (recipe (1,1,32) of the group16 notes page). */
enum fp4moe_act_mode { FP4MOE_ACT_BF16 = 0, FP4MOE_ACT_FP8 = 1 };

/* Flag OR-ed into act_mode of fp4moe_prepare_weights: refuse the lossy
 * group16 -> group32 requant that the FP8 path otherwise runs, mirroring the
 * capability gate of the group16 notes page (group16 scales are accepted by
 * the layout transform but not by the fused FP8 compute):
 * FP8 + gran_k 16 + this flag -> UNSUPPORTED. */
#define FP4MOE_FLAG_NO_REQUANT 0x100

/* Flag OR-ed into act_mode of fp4moe_prepare_weights: FP8 activations over
 * group16 (E4M3-scaled) weights without the lossy requant.  The GEMM converts
 * e2m1 * E4M3 exactly, as in the bf16 path, so the result is the exact
 * group16 product (the group16 notes page's "remaining kernel work" of a
 * software group16 path in the FP8 kernel).  Takes precedence over
 * FP4MOE_FLAG_NO_REQUANT; no effect unless act_mode is FP8 and gran_k 16. */
#define FP4MOE_FLAG_KEEP_GROUP16 0x200

/* Flag OR-ed into act_mode of fp4moe_prepare_weights: w13_gs and w2_gs are
 * stored inverted (the compressed-tensors checkpoint convention of the
 * prepare page); the scale applied is 1 / gs, an FP32 division. */
#define FP4MOE_FLAG_GS_INVERTED 0x400

/* Opaque prepared weights.  Owned by the library until fp4moe_free_packed. */
typedef struct fp4moe_packed fp4moe_packed;

/* Read-only description of a prepared weight set (for tests and tools). */
typedef struct fp4moe_packed_desc {
  int32_t E, K, I, gran_k, act_mode, w13_layout;
  int32_t k_tile, n_tile;        /* packed tile shape: 128 rows x 64 K      */
  int32_t tile_bytes;            /* bytes per packed tile                   */
  const uint8_t* w13;            /* device: packed FC1 tiles                */
  size_t w13_bytes;
  const uint8_t* w2;             /* device: packed FC2 tiles                */
  size_t w2_bytes;
  const float* alpha13;          /* device [E]: FC1 epilogue scale          */
  const float* alpha2;           /* device [E]: FC2 epilogue scale          */
  uint32_t scale_mul, scale_add; /* scale code c -> bf16 bits c*mul + add   */
  /* layout 0: tiles of 128 rows x 64 K with scale codes (bf16 path);
   * layout 1: block-scaled path (FP8 activations over group32 weights):
   *   w13 [E][2I][K/2] plain E2M1 codes, rows per 128-column block b: the
   *   gate rows of columns 128b..128b+127 at 256b, their up rows at
   *   256b+128; w2 [E][K][I/2] as given; w13_scales / w2_scales: one 32-bit
   *   word per row and 128-wide K step holding its four UE8M0 bytes (block
   *   j of the step in byte j), ordered [E][rows/128][K/128][128]; alpha is
   *   the global scale (gs, or 1/gs with FP4MOE_FLAG_GS_INVERTED). */
  int32_t layout;
  const uint32_t* w13_scales;
  size_t w13_scales_bytes;
  const uint32_t* w2_scales;
  size_t w2_scales_bytes;
} fp4moe_packed_desc;

/* ------------------------------------------------------------------ S1 --
 * group16 -> group32 FP4 requantization (page "glm52_nvfp4_group16_notes.md",
 * section "Requantization path"; the requant commit of the DeepGEMM branch
 * "cch/deepgemm-glm52-nvfp4-group16"): per 32-element group of a row,
 * dequantize v = e2m1 * e4m3(scale16), recompute a UE8M0 scale
 * e = min{e : max|v| <= 6 * 2^e} (byte e + 127; an all-zero group gives 127),
 * and round v / 2^e to E2M1, nearest, ties to the even mantissa bit, sign of
 * zero kept.  Lossy.  The FP32 global scale is not an input: it applies
 * unchanged to the output.  A group with an E4M3 NaN scale gets UE8M0 0xFF
 * and codes 0, and records FP4MOE_ERR_INVALID_ARG in the device status word.
 *   fp4       [rows, K/2]  E2M1 codes            (16-byte aligned)
 *   e4m3_s    [rows, K/16] E4M3 scales
 *   fp4_out   [rows, K/2]  E2M1 codes            (16-byte aligned)
 *   ue8m0_out [rows, K/32] UE8M0 scales
 * K % 32 == 0, src_gran == 16, dst_gran == 32 (else INVALID_ARG /
 * UNSUPPORTED).  rows == 0 is a no-op.  In and out must not overlap. */
int fp4moe_requant_fp4_gran_k(const uint8_t* fp4, const uint8_t* e4m3_s,
                              int64_t rows, int64_t K, int src_gran,
                              int dst_gran, uint8_t* fp4_out,
                              uint8_t* ue8m0_out, void* stream);

/* ------------------------------------------------------------------ S4 --
 * FP8 activation quantization, recipe (1,1,32) (group16 notes page): per
 * token and 32 consecutive K elements, UE8M0 e = min{e : amax <= 448 * 2^e}
 * (byte clamped to [0,254]; an all-zero group gives 127) and
 * q = E4M3(x / 2^e), nearest-even, saturating, sign of zero kept.
 *   x_bf16 [T, K] bfloat16 words; xq [T, K] E4M3; xs [T, K/32] UE8M0.
 * K % 32 == 0.  Non-finite inputs record INVALID_ARG in the status word. */
int fp4moe_act_quant(const void* x_bf16, int64_t T, int64_t K, uint8_t* xq,
                     uint8_t* xs, void* stream);

/* ------------------------------------------------------------------ S0 --
 * Prepare raw grouped FP4 weights for moe_forward (the "prepare FP4 weights
 * for MegaMoE" commit: raw weights + scales -> optional requant -> layout
 * transform; and the NVFP4 preparation of prepare.py).  Inputs:
 *   w13 [E, 2I, K/2] codes, w13_s [E, 2I, K/gran_k], w13_gs [E] FP32,
 *   w2  [E, K, I/2]  codes, w2_s  [E, K, I/gran_k],  w2_gs  [E] FP32.
 * gran_k 16 -> E4M3 scales, 32 -> UE8M0 scales.  act_mode FP4MOE_ACT_BF16
 * or FP4MOE_ACT_FP8, optionally OR FP4MOE_FLAG_NO_REQUANT or
 * FP4MOE_FLAG_KEEP_GROUP16, and FP4MOE_FLAG_GS_INVERTED.  With FP8 and
 * gran_k 16 the weights are requantized to group32 first (lossy, as above)
 * unless KEEP_GROUP16 is set.  FP8 activations over group32 weights (given,
 * or from that requant) run on the block-scaled tensor-core path
 * (kind::mxf8f6f4 with UE8M0 scales in TMEM, layout 1 of the description);
 * bf16 activations and kept group16 weights run on the bf16 path.
 * Requires K % 128 == 0, I % 128 == 0, E >= 1.
 * SYNCHRONOUS: allocates device memory for the packed weights, runs the
 * packing kernels on `stream`, synchronises it, and returns INVALID_ARG if a
 * scale was NaN.  On success *out owns the packed weights (free with
 * fp4moe_free_packed); on failure *out is NULL. */
int fp4moe_prepare_weights(const uint8_t* w13, const uint8_t* w13_s,
                           const float* w13_gs, const uint8_t* w2,
                           const uint8_t* w2_s, const float* w2_gs, int E,
                           int K, int I, int gran_k, int w13_layout,
                           int act_mode, void* stream, fp4moe_packed** out);

/* Frees packed weights (NULL is a no-op).  Synchronises the device first. */
void fp4moe_free_packed(fp4moe_packed* p);

/* Fills *desc (host struct) for packed weights.  INVALID_ARG on NULL. */
int fp4moe_packed_info(const fp4moe_packed* p, fp4moe_packed_desc* desc);

/* -------------------------------------------------------------- S2..S7 --
 * Sources of the MoE layer.  The pages print no kernel for routing,
 * permutation, SwiGLU or combine; these calls follow the benchmark
 * description of the MoE workloads (the tiny layer E8 K256 I128 T16 top-2,
 * the decode layer E256 K6144 I2048 T64 top-8, the prefill layer T8192, the
 * FP8 x FP4 layer E128 K7168 I2048 T4096 top-8): router logits FP32, softmax
 * then top-k with the k weights renormalised, SwiGLU(gate, up), FP32
 * accumulation, bfloat16 output; the expert FFN is routing -> top-k
 * permutation (per-expert histogram, prefix-sum offsets, scatter) -> FC1
 * gate|up grouped GEMM with SwiGLU -> FC2 grouped GEMM -> weighted top-k
 * combine.  The gate/up row order is the prepare page's (W13 layout notes);
 * the FP8 activation format is recipe (1,1,32) of the group16 notes page
 * (section "Context").
 *
 * Bytes of device workspace moe_forward needs for T tokens and top_k: the
 * routing scratch, ids and weights, counts and offsets, perm and inv, the
 * gathered activation rows, h and the FC2 output (FP32), laid out for the
 * steps above.  Returns 0 for invalid arguments. */
size_t fp4moe_moe_workspace_size(const fp4moe_packed* p, int T, int top_k);

/* MoE layer forward: softmax top-k routing with renormalised weights (S2),
 * stable expert-major permutation (S3), FC1 gate|up grouped GEMM + SwiGLU
 * (S5), FC2 grouped GEMM (S6) and the weighted top-k combine (S7), all on
 * `stream`.  FP32 accumulation; h = silu(G) * U is rounded to bfloat16
 * (BF16 mode) or to E4M3 with a per-32 UE8M0 scale (FP8 mode) before FC2.
 *   x:            BF16 mode: bfloat16 [T, K];  FP8 mode: E4M3 [T, K]
 *   x_scales:     FP8 mode: UE8M0 [T, K/32]; BF16 mode: must be NULL
 *   router_logits FP32 [T, E]
 *   y             bfloat16 [T, K] output
 *   workspace     >= fp4moe_moe_workspace_size(p, T, top_k) bytes, 256-byte
 *                 aligned; contents are scratch.
 * T >= 0 (T == 0 is a no-op), 1 <= top_k <= min(E, 16).  The mode is the
 * act_mode the weights were prepared for.  Asynchronous: no host
 * synchronisation, and after the first call on a device (which sets the
 * kernels' per-device attributes) no allocation either, so the call may be
 * captured into a CUDA graph.  Calls that can run at once (other streams)
 * need their own workspace and y; the status word is shared. */
int fp4moe_moe_forward(const void* x, const uint8_t* x_scales,
                       const float* router_logits, int T,
                       const fp4moe_packed* p, int top_k, void* y,
                       void* workspace, size_t ws_bytes, void* stream);

/* End-to-end variant of moe_forward (same steps and sources as above) for
 * callers holding HOST buffers: x_host, x_scales_host
 * (FP8 mode) and logits_host are copied to the device, moe_forward runs, and
 * y is copied back to y_host, all asynchronously on `stream` (use pinned host
 * memory; synchronise the stream before reading y_host).  The device
 * workspace must hold fp4moe_moe_workspace_size_host(p, T, top_k) bytes. */
size_t fp4moe_moe_workspace_size_host(const fp4moe_packed* p, int T,
                                      int top_k);
int fp4moe_moe_forward_host(const void* x_host, const uint8_t* x_scales_host,
                            const float* logits_host, int T,
                            const fp4moe_packed* p, int top_k, void* y_host,
                            void* workspace, size_t ws_bytes, void* stream);

/* Test export (no counterpart on the pages; it exposes moe_forward's own
 * intermediates so tests can check each step): byte offsets, inside the
 * moe_forward workspace for (p, T,
 * top_k), of its intermediates, so a test can read them back after a call:
 * out[0] ids int32 [T*top_k], [1] routing weights FP32 [T*top_k], [2] counts
 * int32 [E], [3] offsets int32 [E+1], [4] perm int32 [P], [5] inv int32 [P],
 * [6] gathered activations [P, K] (bf16; E4M3 bytes on the block-scaled
 * path), [7] h [P, I] (FC2's input, in expert-major order: bf16 values, or
 * E4M3 bytes on the block-scaled path), [8] FC2 output FP32 [P, K], [9] total
 * size; with n >= 13 also [10] the block-scaled path's h scale words
 * [I/128][pitch] (word row p holds the four UE8M0 bytes of h row p's 32-wide
 * groups in that 128-column step; 0 otherwise), [11] the h format (0 bf16,
 * 1 E4M3 bytes + scale words), [12] that pitch in words.  n >= 10 (host
 * array); INVALID_ARG otherwise. */
int fp4moe_moe_workspace_offsets(const fp4moe_packed* p, int T, int top_k,
                                 size_t* out, int n);

/* Test export of S2 + S3 alone (bit-exact checks), defined by the routing of
 * the benchmark description's MoE workloads (softmax then top-k with
 * renormalised weights) and its top-k permutation (per-expert histogram,
 * prefix-sum offsets, scatter): ids [T, top_k] int32,
 * w [T, top_k] FP32, counts [E], offsets [E+1], perm [T*top_k],
 * inv [T*top_k], with workspace >= fp4moe_route_workspace_size(T, E, top_k).
 * Ties between equal logits go to the lower expert id; pairs p = t*top_k + j
 * keep ascending order within an expert. */
size_t fp4moe_route_workspace_size(int T, int E, int top_k);
int fp4moe_route_debug(const float* logits, int T, int E, int top_k,
                       int32_t* ids, float* w, int32_t* counts,
                       int32_t* offsets, int32_t* perm, int32_t* inv,
                       void* workspace, size_t ws_bytes, void* stream);

/* Stage timing for profiling: hands the NEXT fp4moe_moe_forward (or
 * fp4moe_moe_forward_host) call on this host thread n cudaEvent_t handles
 * (n must be FP4MOE_STAGE_EVENTS; host array, events owned by the caller,
 * created with timing enabled).  That call records them on its stream at the
 * stage boundaries: [0] start, [1] after routing, [2] after the scan,
 * [3] after the scatter/gather, [4] after FC1, [5] after the FP8 rounding of
 * h (same point as [4] in BF16 mode), [6] after FC2, [7] after the combine;
 * then the hand-over is cleared.  Up to 32 tokens, routing, scan and scatter
 * are one launch, which [1] and [2] both follow.  events == NULL clears it.
 * INVALID_ARG if n is wrong. */
#define FP4MOE_STAGE_EVENTS 8
int fp4moe_set_stage_events(void* const* events, int n);

/* Allocation-free routing + permutation, for callers that cannot allocate
 * device memory where they route tokens: for example a plugin inside a
 * framework whose own allocator owns the device memory pool, or a
 * latency-critical loop where cudaMalloc could synchronise the device.  The
 * pages have no counterpart: this is a library convenience.
 * It computes exactly what fp4moe_route_debug computes (same outputs, same
 * argument rules) but takes no workspace: its scratch lives in one array of
 * FP4MOE_NOALLOC_SCRATCH_BYTES in device global memory that the library
 * owns, which every GPU that loads the library keeps until the process exits.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - The first call on a device looks up that array's device address (once
 *     per device, with the device current); make that first call before any
 *     stream capture.
 *   - All calls share the one array, and each call overwrites what it uses,
 *     so calls whose kernels overlap on the GPU (other streams, other host
 *     threads) race on it: serialise them.
 *   - The looked-up address belongs to the device's current context: after
 *     cudaDeviceReset (or anything else that destroys that context) it is
 *     stale, so do not call this entry point across a device reset.
 *   - Sizes whose scratch (fp4moe_route_noalloc_scratch_bytes) exceeds the
 *     array return FP4MOE_ERR_WORKSPACE_TOO_SMALL before launching anything;
 *     the scratch is about 8 * ceil(T/32) * E bytes, so 4 MiB covers, e.g.,
 *     T = 8192 tokens with E = 1024 experts or T = 32768 with E = 256. */
#define FP4MOE_NOALLOC_SCRATCH_BYTES (4u << 20)
size_t fp4moe_route_noalloc_scratch_bytes(int T, int E);
int fp4moe_route_noalloc(const float* logits, int T, int E, int top_k,
                         int32_t* ids, float* w, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv,
                         void* stream);

/* Test export of the bounded device waits (no counterpart on the pages):
 * launches one thread that waits on an mbarrier nothing completes; the wait
 * gives up after limit_ns nanoseconds (1 .. 1e9, else INVALID_ARG) and records
 * FP4MOE_ERR_TIMEOUT in the device status word, which
 * fp4moe_last_device_error() then returns.  Every wait inside the library's
 * kernels is bounded the same way (about 2 s).  Asynchronous on `stream`. */
int fp4moe_test_wait_timeout(uint64_t limit_ns, void* stream);

/* Build variant (no counterpart on the pages).  The library is built twice
 * from the same sources: libfp4moe.so and libfp4moe_checked.so, the latter
 * compiled with FP4MOE_BOUNDS_CHECK, where every data-dependent index (expert
 * ids, permutation slots, work-unit rows and columns, scale offsets) is
 * checked against its buffer before the access; a failed check records
 * FP4MOE_ERR_BOUNDS in the device status word and skips the access (a
 * GEMM work unit with a bad expert index is computed from expert 0 and its
 * stores are checked as well).  Returns FP4MOE_BUILD_BOUNDS_CHECK in the
 * checked build, 0 otherwise. */
#define FP4MOE_BUILD_BOUNDS_CHECK 1
int fp4moe_build_flags(void);

/* Test export of the index check (no counterpart on the pages): one thread
 * writes slot `index` of a 64-entry device array through the same check the
 * checked build applies (in both builds); an index outside [0, 64) records
 * FP4MOE_ERR_BOUNDS in the device status word and writes nothing.
 * Asynchronous on `stream`. */
int fp4moe_test_bounds_check(int64_t index, void* stream);

/* Static text for a status code (never NULL); see the status codes above. */
const char* fp4moe_status_string(int status);

/* Device-side error reporting (no counterpart on the pages, whose code only
 * raises host exceptions): reads and clears the status word of the current
 * device: the first error a
 * kernel recorded since the last call (FP4MOE_OK if none).  Synchronises the
 * device.  Returns FP4MOE_ERR_CUDA if the read itself fails. */
int fp4moe_last_device_error(void);

#ifdef __cplusplus
}
#endif
#endif /* FP4MOE_H_ */
