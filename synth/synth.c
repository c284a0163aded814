/* Seeded synthetic weights for the block-scaled FP4 MoE workloads.
 *
 * Random numbers: a counter-based generator -- the SplitMix64 output function
 * (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014) applied to key + (i + 1) * 0x9E3779B97F4A7C15 -- so element i
 * of a stream is a pure function of (key, i) and experts generate in parallel.
 * Normals come from the Box-Muller transform of two 24-bit uniforms.
 *
 * Encoding recipe (an input recipe, not the method: nearest with ties away
 * from zero, through a table search):
 *   gs   = amax(W_e) / (6 * 448) per expert matrix (1 if all zero)
 *   s16  = nearest E4M3 value to amax(group of 16) / (6 * gs)
 *   code = nearest E2M1 value to w * (1 / (s16 * gs)) (the reciprocal in
 *          float); s16 == 0 gives code 0.
 * Portable C (no intrinsics); built with -ffp-contract=off.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static uint64_t ctr(uint64_t key, uint64_t i) {
  return mix64(key + (i + 1) * 0x9E3779B97F4A7C15ULL);
}

static float u01(uint32_t x) { /* in (0, 1] */
  return (float)((x >> 8) + 1) * (1.0f / 16777216.0f);
}

static void normal2(uint64_t key, uint64_t i, float* a, float* b) {
  uint64_t r = ctr(key, i);
  float u1 = u01((uint32_t)r), u2 = u01((uint32_t)(r >> 32));
  float rad = sqrtf(-2.0f * logf(u1));
  float th = 6.2831853071795864f * u2;
  *a = rad * cosf(th);
  *b = rad * sinf(th);
}

/* Non-negative finite E4M3 values by code 0..126. */
static double g_e4m3[127];
static double g_e4m3_mid[126];
static pthread_once_t g_once = PTHREAD_ONCE_INIT;

static void init_tables(void) {
  for (int b = 0; b < 127; ++b) {
    int e = b >> 3, m = b & 7;
    g_e4m3[b] = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  }
  for (int b = 0; b < 126; ++b) g_e4m3_mid[b] = 0.5 * (g_e4m3[b] + g_e4m3[b + 1]);
}

/* Index of the nearest table entry, ties to the larger (away from zero). */
static int nearest_e4m3(double t) {
  int lo = 0, hi = 126; /* count of midpoints <= t */
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (g_e4m3_mid[mid] <= t) lo = mid + 1; else hi = mid;
  }
  return lo;
}

static uint8_t nearest_e2m1(float y) {
  float a = fabsf(y);
  uint8_t m = a < 0.25f ? 0 : a < 0.75f ? 1 : a < 1.25f ? 2 : a < 1.75f ? 3
            : a < 2.5f ? 4 : a < 3.5f ? 5 : a < 5.0f ? 6 : 7;
  return (uint8_t)(m | (y < 0.0f ? 8 : 0));
}

/* w [N, Kd] -> codes [N, Kd/2], scales [N, Kd/16]; returns gs. */
static float encode(const float* w, int64_t N, int64_t Kd, uint8_t* codes,
                    uint8_t* scales) {
  float amax = 0.0f;
  for (int64_t i = 0; i < N * Kd; ++i) amax = fmaxf(amax, fabsf(w[i]));
  float gs = amax > 0.0f ? (float)(amax / (6.0 * 448.0)) : 1.0f;
  for (int64_t r = 0; r < N; ++r) {
    for (int64_t g = 0; g < Kd / 16; ++g) {
      const float* v = w + r * Kd + g * 16;
      float ga = 0.0f;
      for (int i = 0; i < 16; ++i) ga = fmaxf(ga, fabsf(v[i]));
      int si = nearest_e4m3((double)ga / (6.0 * (double)gs));
      scales[r * (Kd / 16) + g] = (uint8_t)si;
      const double sv = g_e4m3[si] * (double)gs;
      const float inv = sv > 0 ? (float)(1.0 / sv) : 0.0f;
      uint8_t* out = codes + r * (Kd / 2) + g * 8;
      for (int i = 0; i < 8; ++i) {
        uint8_t lo = sv > 0 ? nearest_e2m1(v[2 * i] * inv) : 0;
        uint8_t hi = sv > 0 ? nearest_e2m1(v[2 * i + 1] * inv) : 0;
        out[i] = (uint8_t)(lo | (hi << 4));
      }
    }
  }
  return gs;
}

typedef struct {
  uint64_t seed;
  int E;
  int64_t N, Kd;
  float std, outlier_mul;
  double outlier_p;
  uint8_t* codes;
  uint8_t* scales;
  float* gs;
  int next; /* next expert to take */
  pthread_mutex_t mu;
} Job;

static void* worker(void* arg) {
  Job* j = (Job*)arg;
  const int64_t n = j->N * j->Kd;
  float* w = (float*)malloc((size_t)n * sizeof(float));
  if (!w) return NULL;
  for (;;) {
    pthread_mutex_lock(&j->mu);
    int e = j->next++;
    pthread_mutex_unlock(&j->mu);
    if (e >= j->E) break;
    const uint64_t key = mix64(j->seed ^ mix64((uint64_t)e + 1));
    const uint64_t okey = mix64(key ^ 0x5DEECE66DULL);
    for (int64_t i = 0; i < n; i += 2) {
      float a, b;
      normal2(key, (uint64_t)(i / 2), &a, &b);
      w[i] = a * j->std;
      if (i + 1 < n) w[i + 1] = b * j->std;
    }
    if (j->outlier_p > 0) {
      const uint32_t thr = (uint32_t)(j->outlier_p * 4294967296.0);
      for (int64_t i = 0; i < n; ++i)
        if ((uint32_t)ctr(okey, (uint64_t)i) < thr) w[i] *= j->outlier_mul;
    }
    j->gs[e] = encode(w, j->N, j->Kd, j->codes + (int64_t)e * j->N * (j->Kd / 2),
                      j->scales + (int64_t)e * j->N * (j->Kd / 16));
  }
  free(w);
  return NULL;
}

/* E expert matrices [N, Kd] ~ N(0, std) (with outliers), NVFP4 group16. */
int synth_nvfp4_weights(uint64_t seed, int E, int64_t N, int64_t Kd, float std,
                        double outlier_p, float outlier_mul, uint8_t* codes,
                        uint8_t* scales, float* gs, int nthreads) {
  if (E < 0 || N < 0 || Kd <= 0 || Kd % 16) return 1;
  pthread_once(&g_once, init_tables);
  Job j;
  memset(&j, 0, sizeof j);
  j.seed = seed; j.E = E; j.N = N; j.Kd = Kd; j.std = std;
  j.outlier_p = outlier_p; j.outlier_mul = outlier_mul;
  j.codes = codes; j.scales = scales; j.gs = gs;
  pthread_mutex_init(&j.mu, NULL);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > E) nthreads = E > 0 ? E : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, worker, &j);
  for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  free(th);
  pthread_mutex_destroy(&j.mu);
  return 0;
}
