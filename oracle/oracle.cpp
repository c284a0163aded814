// Oracle: a plain, slow, FP64 CPU statement of what the block-scaled FP4 MoE
// hot path computes.  TEST INFRASTRUCTURE ONLY: it exists so that tests, the
// smoke check and the benchmark's CPU-baseline leg can check the CUDA path
// against an independent implementation.  The product never calls it, and it
// shares no source with the CUDA library (no headers, tables or helpers).
//
// Sources (page title, then section):
//  * "DeepGEMM commits, branch cch/deepgemm-glm52-nvfp4-group16" -- the
//    requant commit: group16 -> group32 recomputes UE8M0 scales.
//  * "glm52_nvfp4_group16_notes.md", section "Requantization path": the
//    group16 values are restored with their own scales and re-encoded with
//    one new scale per 32 values, which changes the codes (a lossy step).
//  * "b12x/moe/fused/w4a16/prepare.py": E2M1 packing (two codes per byte, low
//    nibble = even k), NVFP4 E4M3 scales per 16, per-tensor FP32 global scale,
//    E8M0 scales per 32, and the gate/up order of the fused FC1 weight
//    ("w13" arrives up/gate, "w31" is gate/up).
//  * Steps the pages leave open (routing, permutation, SwiGLU, combine, the
//    requant rounding rule) follow the plainest reading; each is marked
//    READING below.
//
// Parity status of each function is stated in its comment; all are pinned by
// closed forms, invariants or brute force in tests/test_oracle_pins.py.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {
template <class F>
static void parallel_for(int64_t n, int nthreads, F f) {
  if (nthreads <= 1 || n < 64) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> th;
  int64_t chunk = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    int64_t a = t * chunk, b = std::min(n, a + chunk);
    if (a >= b) break;
    th.emplace_back([=] { for (int64_t i = a; i < b; ++i) f(i); });
  }
  for (auto& x : th) x.join();
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------- formats

// E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.  The
// magnitudes are the codebook {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_value(uint8_t code) {
  double m = kE2M1Mag[code & 7];
  return (code & 8) ? -m : m;
}

// E4M3 ("fn" variant): bias 7, subnormals, no infinities; 0x7F/0xFF are NaN.
double orc_e4m3_value(uint8_t b) {
  int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? std::ldexp((double)m / 8.0, -6)
                      : std::ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

// UE8M0: a power of two 2^(b-127); 0xFF is NaN.
double orc_ue8m0_value(uint8_t b) {
  if (b == 255) return NAN;
  return std::ldexp(1.0, (int)b - 127);
}

// bfloat16 bits -> value.
double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Round-half-to-even of a non-negative double to an integer-valued double.
static double rne_int(double x) {
  double r = std::floor(x);
  double frac = x - r;
  if (frac > 0.5) return r + 1.0;
  if (frac < 0.5) return r;
  return (std::fmod(r, 2.0) == 0.0) ? r : r + 1.0;
}

// Round to E2M1, nearest, ties to the code with an even mantissa bit, |v| > 6
// saturates to 6.  The sign is kept, so -0 and negative values that round to
// zero give code 0x8 (READING: IEEE sign of zero).  Written as a search over
// the eight magnitudes so it can be checked by eye.
uint8_t orc_e2m1_rne(double v) {
  double a = std::fabs(v);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = std::fabs(a - kE2M1Mag[c]);
    if (d < bestd || (d == bestd && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      bestd = d;
    }
  }
  return (uint8_t)(best | (std::signbit(v) ? 8 : 0));
}

// Round to E4M3 (fn), nearest-even, saturating to +-448 (no NaN produced for
// finite input).  Sign kept.
uint8_t orc_e4m3_rne_sat(double v) {
  double a = std::fabs(v);
  uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  if (a >= 448.0) return sign | 0x7E;
  if (a < std::ldexp(1.0, -6)) {               // subnormal range, step 2^-9
    double q = rne_int(a / std::ldexp(1.0, -9)); // 0..8; 8 is the first normal
    return sign | (uint8_t)q;
  }
  int E;
  std::frexp(a, &E);          // a = f * 2^E, f in [0.5, 1)
  E -= 1;                     // a = g * 2^E, g in [1, 2)
  double q = rne_int(a / std::ldexp(1.0, E - 3));   // in [8, 16]
  if (q == 16.0) { q = 8.0; E += 1; }
  if (E > 8) return sign | 0x7E;
  int field = E + 7;
  return sign | (uint8_t)((field << 3) | ((int)q - 8));
}

// Round to bfloat16, nearest-even, directly from double (no double rounding
// through float).  Overflow gives infinity.
uint16_t orc_bf16_rne(double v) {
  uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  if (std::isnan(v)) return 0x7FC0;
  if (a == 0.0) return sign;
  if (std::isinf(a)) return sign | 0x7F80;
  if (a < std::ldexp(1.0, -126)) {                 // subnormal, step 2^-133
    double q = rne_int(a / std::ldexp(1.0, -133)); // 0..128 (128 = min normal)
    return sign | (uint16_t)q;
  }
  int E;
  std::frexp(a, &E);
  E -= 1;                                           // a = g * 2^E, g in [1,2)
  double q = rne_int(a / std::ldexp(1.0, E - 7));   // in [128, 256]
  if (q == 256.0) { q = 128.0; E += 1; }
  if (E > 127) return sign | 0x7F80;
  return sign | (uint16_t)(((E + 127) << 7) | ((int)q - 128));
}

// Smallest integer e with amax <= limit * 2^e, by exact comparison (no log).
static int min_pow2_exponent(double amax, double limit) {
  int e = 0;
  while (limit * std::ldexp(1.0, e) < amax) ++e;
  while (limit * std::ldexp(1.0, e - 1) >= amax) --e;
  return e;
}

// ----------------------------------------------------------------- requant
//
// S1.  group16 -> group32 requantization ("glm52_nvfp4_group16_notes.md",
// section "Requantization path"; the requant commit of the DeepGEMM branch).
// Per 32-element group of a row:
//   v_i  = e2m1(code_i) * e4m3(scale16[i/16])     (exact in FP64)
//   amax = max |v_i|
//   e    = min { e : amax <= 6 * 2^e }             (READING: no element clips)
//   byte = clamp(e + 127, 0, 254); amax == 0 gives byte 127
//   q_i  = RNE_E2M1(v_i / 2^(byte-127))
// The per-tensor global scale is not an input: it passes through unchanged
// (READING).  A group whose group16 scales include an E4M3 NaN gets the
// UE8M0 NaN byte 0xFF and codes 0 (READING).
// fp4: [rows, K/2] bytes, low nibble = even k.  s16: [rows, K/16].
// Outputs fp4_out [rows, K/2], s32_out [rows, K/32].  K % 32 == 0 required.
static void requant_rows(const uint8_t* fp4, const uint8_t* s16, int64_t r0,
                         int64_t r1, int64_t K, uint8_t* fp4_out,
                         uint8_t* s32_out) {
  const int64_t kb = K / 2, k16 = K / 16, k32 = K / 32;
  for (int64_t r = r0; r < r1; ++r) {
    for (int64_t g = 0; g < k32; ++g) {
      double v[32];
      bool nan_scale = false;
      for (int i = 0; i < 32; ++i) {
        int64_t k = g * 32 + i;
        uint8_t byte = fp4[r * kb + k / 2];
        uint8_t code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
        double s = orc_e4m3_value(s16[r * k16 + k / 16]);
        if (std::isnan(s)) nan_scale = true;
        v[i] = orc_e2m1_value(code) * s;
      }
      uint8_t* out = fp4_out + r * kb + g * 16;
      if (nan_scale) {
        s32_out[r * k32 + g] = 0xFF;
        std::memset(out, 0, 16);
        continue;
      }
      double amax = 0.0;
      for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(v[i]));
      int e = (amax == 0.0) ? 0 : min_pow2_exponent(amax, 6.0);
      int byte = std::min(254, std::max(0, e + 127));
      s32_out[r * k32 + g] = (uint8_t)byte;
      double inv = std::ldexp(1.0, -(byte - 127));
      for (int i = 0; i < 16; ++i) {
        uint8_t lo = orc_e2m1_rne(v[2 * i] * inv);
        uint8_t hi = orc_e2m1_rne(v[2 * i + 1] * inv);
        out[i] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
}

int orc_requant(const uint8_t* fp4, const uint8_t* s16, int64_t rows, int64_t K,
                uint8_t* fp4_out, uint8_t* s32_out, int nthreads) {
  if (rows < 0 || K <= 0 || K % 32 != 0) return 1;
  if (nthreads < 1) nthreads = 1;
  std::vector<std::thread> th;
  int64_t chunk = (rows + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    int64_t r0 = t * chunk, r1 = std::min(rows, r0 + chunk);
    if (r0 >= r1) break;
    th.emplace_back(requant_rows, fp4, s16, r0, r1, K, fp4_out, s32_out);
  }
  for (auto& x : th) x.join();
  return 0;
}

// ----------------------------------------------------------------- routing
//
// S2.  Softmax top-k routing with renormalised weights (the pages are silent;
// this is the plain reading of "softmax then top-k with renormalised
// weights").  Softmax is monotone, so the k experts are chosen on the raw
// logits: descending value, equal values to the lower expert id (READING).
// w_j = exp(l_j - l_max) / sum_{i in top-k} exp(l_i - l_max), which equals
// softmax over all experts, restricted to the top-k and renormalised.
// Returns 1 (and writes nothing for that token onward) on a NaN logit.
int orc_route(const float* logits, int64_t T, int E, int k, int32_t* ids,
              double* w) {
  if (k < 1 || k > E) return 1;
  std::vector<int> idx(E);
  for (int64_t t = 0; t < T; ++t) {
    const float* l = logits + t * E;
    for (int e = 0; e < E; ++e) {
      if (std::isnan(l[e])) return 1;
      idx[e] = e;
    }
    std::stable_sort(idx.begin(), idx.end(),
                     [&](int a, int b) { return l[a] > l[b]; });
    double lmax = l[idx[0]];
    double sum = 0.0;
    for (int j = 0; j < k; ++j) sum += std::exp((double)l[idx[j]] - lmax);
    for (int j = 0; j < k; ++j) {
      ids[t * k + j] = idx[j];
      w[t * k + j] = std::exp((double)l[idx[j]] - lmax) / sum;
    }
  }
  return 0;
}

// S3.  Permutation: per-expert histogram, exclusive prefix-sum offsets and a
// stable scatter of routed pairs p = t*k + j into expert-major order
// (ascending p within an expert); inv is the inverse map p -> position.
int orc_permute(const int32_t* ids, int64_t T, int k, int E, int32_t* counts,
                int32_t* offsets, int32_t* perm, int32_t* inv) {
  int64_t P = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t p = 0; p < P; ++p) {
    if (ids[p] < 0 || ids[p] >= E) return 1;
    counts[ids[p]]++;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> cursor(offsets, offsets + E);
  for (int64_t p = 0; p < P; ++p) {
    int32_t pos = cursor[ids[p]]++;
    perm[pos] = (int32_t)p;
    inv[p] = pos;
  }
  return 0;
}

// S4.  FP8 activation quantization, recipe (1,1,32): per token, per 32
// consecutive K elements, a UE8M0 scale e = min { e : amax <= 448 * 2^e }
// (byte = clamp(e + 127, 0, 254), amax == 0 gives 127) and E4M3 values
// q = RNE_E4M3_satfinite(x / 2^(byte-127)).  x is bfloat16 bits [T, K].
int orc_act_quant(const uint16_t* x, int64_t T, int64_t K, uint8_t* q,
                  uint8_t* s) {
  if (K % 32 != 0) return 1;
  for (int64_t t = 0; t < T; ++t) {
    for (int64_t g = 0; g < K / 32; ++g) {
      double v[32], amax = 0.0;
      for (int i = 0; i < 32; ++i) {
        v[i] = orc_bf16_value(x[t * K + g * 32 + i]);
        if (!std::isfinite(v[i])) return 1;
        amax = std::max(amax, std::fabs(v[i]));
      }
      int e = (amax == 0.0) ? 0 : min_pow2_exponent(amax, 448.0);
      int byte = std::min(254, std::max(0, e + 127));
      s[t * (K / 32) + g] = (uint8_t)byte;
      double inv = std::ldexp(1.0, -(byte - 127));
      for (int i = 0; i < 32; ++i)
        q[t * K + g * 32 + i] = orc_e4m3_rne_sat(v[i] * inv);
    }
  }
  return 0;
}

// ------------------------------------------------------------------- MoE
//
// S5-S7 for a list of tokens.  Weights are E2M1 codes [E, N, Kd/2] with
// per-group scales [E, N, Kd/gran]: gran 16 -> E4M3 bytes (NVFP4), gran 32 ->
// UE8M0 bytes (MX); times the per-expert FP32 global scale.  The dequantized
// weight is e2m1 * scale * gs ("b12x/moe/fused/w4a16/prepare.py", NVFP4
// preparation, where the ModelOpt global scale multiplies in).
//
//   w13 [E, 2I, K]: w13_layout 0 = "w31"/gate_up (rows [0,I) gate),
//                   w13_layout 1 = "w13"/up_gate (rows [0,I) up) -- the
//                   checkpoint order, per the prepare.py layout notes.
//   G = gs13 * sum_k x_k * w_gate[i,k],  U likewise with the up rows.
//   h_i = silu(G_i) * U_i = G_i / (1 + exp(-G_i)) * U_i        (SwiGLU)
//   h is rounded before FC2: act_mode 0 (BF16 activations) -> bfloat16 RNE;
//   act_mode 1 (FP8 activations) -> E4M3 with a per-32 UE8M0 scale by the S4
//   rule, then back to its exact value (READING).
//   o_n = gs2 * sum_i h_i * w2[n, i]
//   y_t = sum_j w_{t,j} * o_{(t,j)}, in top-k order.  Returned in FP64; the
//   product rounds y to bfloat16 (orc_bf16_rne gives that rounding).
//   If h_out is set, the unrounded h of each (token, slot) is stored there;
//   aux_out receives G, U, the sums of |terms| behind them and the sums of
//   |running sums| after each 16-wide K chunk (error-analysis quantities for
//   the tests' FP32 tolerance; they do not enter y).
// act_mode 0 reads x_bf16 [T, K]; act_mode 1 reads xq [T, K] (E4M3) and
// xs [T, K/32] (UE8M0).
struct OrcMoe {
  const uint8_t* w13;
  const uint8_t* w13_s;
  const float* w13_gs;
  const uint8_t* w2;
  const uint8_t* w2_s;
  const float* w2_gs;
  int32_t E, K, I, gran, w13_layout, act_mode, top_k, nthreads;
  const uint16_t* x_bf16;
  const uint8_t* xq;
  const uint8_t* xs;
  const float* logits;
  int64_t T;
  double* h_out;  // optional [ntok, top_k, I]: h before its rounding
  double* aux_out;  // optional [ntok, top_k, I, 6]: G, U, sum|G terms|,
                    // sum|U terms|, sum over 16-wide K chunks of |G running
                    // sum|, the same for U (the scale of FP32 rounding in G
                    // and U); global scale included in all but G and U
};

static double weight_value(const uint8_t* w, const uint8_t* s, int gran,
                           int64_t Kd, int64_t row, int64_t k) {
  uint8_t byte = w[row * (Kd / 2) + k / 2];
  uint8_t code = (k % 2 == 0) ? (byte & 0xF) : (byte >> 4);
  uint8_t sb = s[row * (Kd / gran) + k / gran];
  double sc = (gran == 16) ? orc_e4m3_value(sb) : orc_ue8m0_value(sb);
  return orc_e2m1_value(code) * sc;
}

// One row dot product: sum_k x[k] * dequant(w[row, k]) (FP64); *abs_sum
// (if given) receives sum_k |x[k] * dequant(w[row, k])| and *run_sum the sum,
// over the chunks of 16 consecutive k, of |the running sum after the chunk|.
static double row_dot(const uint8_t* w, const uint8_t* s, int gran, int64_t Kd,
                      int64_t row, const double* x, double* abs_sum = nullptr,
                      double* run_sum = nullptr) {
  double acc = 0.0, a = 0.0, r = 0.0;
  for (int64_t k = 0; k < Kd; ++k) {
    const double t = x[k] * weight_value(w, s, gran, Kd, row, k);
    acc += t;
    a += std::fabs(t);
    if (k % 16 == 15) r += std::fabs(acc);
  }
  if (abs_sum) *abs_sum = a;
  if (run_sum) *run_sum = r;
  return acc;
}

// Rounds h the way the intermediate activation is stored (see above).
static void round_intermediate(std::vector<double>& h, int act_mode) {
  if (act_mode == 0) {
    for (auto& v : h) v = orc_bf16_value(orc_bf16_rne(v));
    return;
  }
  for (size_t g = 0; g < h.size() / 32; ++g) {
    double amax = 0.0;
    for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(h[g * 32 + i]));
    int e = (amax == 0.0) ? 0 : min_pow2_exponent(amax, 448.0);
    int byte = std::min(254, std::max(0, e + 127));
    double sc = std::ldexp(1.0, byte - 127);
    for (int i = 0; i < 32; ++i)
      h[g * 32 + i] = orc_e4m3_value(orc_e4m3_rne_sat(h[g * 32 + i] / sc)) * sc;
  }
}

// Rounds n values of h the way the intermediate is stored (act_mode 0:
// bfloat16; act_mode 1: E4M3 with a per-32 UE8M0 scale, n % 32 == 0).
int orc_round_intermediate(const double* h, int64_t n, int act_mode,
                           double* out) {
  if (act_mode == 1 && n % 32) return 1;
  std::vector<double> v(h, h + n);
  round_intermediate(v, act_mode);
  std::copy(v.begin(), v.end(), out);
  return 0;
}

// The UE8M0 exponent (byte - 127) the FP8 rounding picks for 32 values.
int orc_fp8_group_exponent(const double* h32) {
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(h32[i]));
  int e = (amax == 0.0) ? 0 : min_pow2_exponent(amax, 448.0);
  return std::min(254, std::max(0, e + 127)) - 127;
}

// y_out: [ntok, K] FP64 for the tokens listed in `tokens`.
int orc_moe_rows(const OrcMoe* a, const int64_t* tokens, int64_t ntok,
                 double* y_out) {
  const int64_t E = a->E, K = a->K, I = a->I;
  if (a->gran != 16 && a->gran != 32) return 1;
  if (K % a->gran || I % a->gran) return 1;
  if (a->act_mode == 1 && (K % 32 || I % 32)) return 1;
  std::vector<int32_t> ids(a->top_k);
  std::vector<double> w(a->top_k), x(K), g(I), u(I), h(I), o(K), sg(I), su(I),
      pg(I), pu(I);
  for (int64_t n = 0; n < ntok; ++n) {
    int64_t t = tokens[n];
    if (t < 0 || t >= a->T) return 1;
    if (orc_route(a->logits + t * E, 1, (int)E, a->top_k, ids.data(), w.data()))
      return 1;
    for (int64_t k = 0; k < K; ++k) {
      if (a->act_mode == 0)
        x[k] = orc_bf16_value(a->x_bf16[t * K + k]);
      else
        x[k] = orc_e4m3_value(a->xq[t * K + k]) *
               orc_ue8m0_value(a->xs[t * (K / 32) + k / 32]);
    }
    double* y = y_out + n * K;
    for (int64_t c = 0; c < K; ++c) y[c] = 0.0;
    for (int j = 0; j < a->top_k; ++j) {
      const int64_t e = ids[j];
      const uint8_t* w13 = a->w13 + e * (2 * I) * (K / 2);
      const uint8_t* w13s = a->w13_s + e * (2 * I) * (K / a->gran);
      const uint8_t* w2 = a->w2 + e * K * (I / 2);
      const uint8_t* w2s = a->w2_s + e * K * (I / a->gran);
      const int64_t gate0 = (a->w13_layout == 0) ? 0 : I;
      const int64_t up0 = (a->w13_layout == 0) ? I : 0;
      const double gs13 = a->w13_gs[e], gs2 = a->w2_gs[e];
      parallel_for(I, a->nthreads, [&](int64_t i) {
        g[i] = gs13 * row_dot(w13, w13s, a->gran, K, gate0 + i, x.data(), &sg[i],
                              &pg[i]);
        u[i] = gs13 * row_dot(w13, w13s, a->gran, K, up0 + i, x.data(), &su[i],
                              &pu[i]);
        h[i] = g[i] / (1.0 + std::exp(-g[i])) * u[i];
      });
      if (a->h_out)
        std::copy(h.begin(), h.end(), a->h_out + (n * a->top_k + j) * I);
      if (a->aux_out) {
        double* ax = a->aux_out + (n * a->top_k + j) * I * 6;
        for (int64_t i = 0; i < I; ++i) {
          ax[6 * i] = g[i];
          ax[6 * i + 1] = u[i];
          ax[6 * i + 2] = std::fabs(gs13) * sg[i];
          ax[6 * i + 3] = std::fabs(gs13) * su[i];
          ax[6 * i + 4] = std::fabs(gs13) * pg[i];
          ax[6 * i + 5] = std::fabs(gs13) * pu[i];
        }
      }
      round_intermediate(h, a->act_mode);
      parallel_for(K, a->nthreads, [&](int64_t c) {
        o[c] = gs2 * row_dot(w2, w2s, a->gran, I, c, h.data());
      });
      for (int64_t c = 0; c < K; ++c) y[c] += w[j] * o[c];
    }
  }
  return 0;
}

}  // extern "C"
