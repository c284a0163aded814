// Pieces shared by the two grouped-GEMM kernels over packed FP4 weights
// (gemm.cu: one CTA per unit; gemm_pair.cu: a CTA pair per unit): the work
// unit decoder and the FP4 -> bf16 conversion.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace fp4moe {
namespace {

struct Unit {
  int e, nb, row0, ntok;   // nb: first 128-row weight block of the unit
};

// Units are ordered (expert, weight-block group, token chunk); expert e owns
// nbu * (cstart[e+1] - cstart[e]) consecutive units, nbu = ceil(nblocks/MT).
// cs_/os are the shared-memory copies of cstart and offsets.
__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, int nbu,
                                            int mt, int max_tok, const int* cs_,
                                            const int* os, int u) {
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
  U.nb = (local / nch) * mt;
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

// 8 packed E2M1 codes -> 8 bf16 (4 words, element 0 in the low half of
// word 0), each multiplied by the bf16 pair s2.  The packer places each
// element's magnitude bits (m, e0, e1) and sign so that a shift (or rotate)
// and a mask put them at bf16 bits 6..8 and 15 (or 22..24 and 31): read as
// bf16, (s, e1, e0, m) there is e2m1 * 2^-126 (code 1 = 0.5 lands on a
// subnormal), and the multiply by s * 2^119 gives e2m1 * s * 2^-7 exactly.
// Seven logic operations per eight elements; the compiler can put the two
// left shifts on the multiply-add pipe, which is less loaded than the logic
// pipe.
__device__ __forceinline__ uint4 dequant8(uint32_t x, uint32_t s2) {
  const uint32_t w0 = ((x >> 8) & 0x00400040u) | (x & 0x81808180u);
  const uint32_t w1 = (x << 6) & 0x81C081C0u;
  const uint32_t w2 = __funnelshift_l(x, x, 12) & 0x81C081C0u;
  const uint32_t w3 = (x << 2) & 0x81C081C0u;
  return make_uint4(bf16x2_mul(w0, s2), bf16x2_mul(w1, s2), bf16x2_mul(w2, s2),
                    bf16x2_mul(w3, s2));
}


}  // namespace
}  // namespace fp4moe
