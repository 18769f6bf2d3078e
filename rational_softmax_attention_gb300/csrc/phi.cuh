// phi of the rational soft-argmax on the FMA pipe, shared by the forward kernels, and the
// attention-mask chunk vote shared by every masked tensor-core kernel.
//
// Page "Ra-Family: Rational Neural Architecture", section 3, ra_softmax: u = (x_max - x)/16,
// q = (1-u)/(1+u), phi = q^8 for u < 1 and exactly 0 otherwise.  With w = (1+u)/2 computed
// by one saturating FMA from the raw score (so every u >= 1, and every masked entry fed as
// -inf, gives w = 1), q = 1/w - 1 and phi = ((q^2)^2)^2; at w = 1 the computed q is below
// 3e-7 and phi rounds to exactly 0.0.
#pragma once

#include "common.cuh"

namespace raattn {

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// phi for four scores of a row (columns c .. c+3): w = sat(base - c2 s) = (1+u)/2.  The
// reciprocals come from one packed product of the pairs A = (w0, w1), B = (w2, w3):
// R = 1/(A B) = (1/(w0 w2), 1/(w1 w3)), so R B = (1/w0, 1/w1) and R A = (1/w2, 1/w3);
// q = 1/w - 1 is one packed FMA per pair and phi = ((q^2)^2)^2 three packed products.
__device__ __forceinline__ void phi_quad(float s0, float s1, float s2, float s3, float c2, float base,
                                         float2& pa, float2& pb) {
  const float2 A = make_float2(fma_sat(s0, -c2, base), fma_sat(s1, -c2, base));
  const float2 B = make_float2(fma_sat(s2, -c2, base), fma_sat(s3, -c2, base));
  const float2 P = __fmul2_rn(A, B);
  const float2 R = make_float2(rcp_approx(P.x), rcp_approx(P.y));
  const float2 minus1 = make_float2(-1.0f, -1.0f);
  float2 qa = __ffma2_rn(R, B, minus1);
  float2 qb = __ffma2_rn(R, A, minus1);
  qa = __fmul2_rn(qa, qa);
  qb = __fmul2_rn(qb, qb);
  qa = __fmul2_rn(qa, qa);
  qb = __fmul2_rn(qb, qb);
  pa = __fmul2_rn(qa, qa);
  pb = __fmul2_rn(qb, qb);
}

// Lowest column of a 32-column chunk whose score equals m (visible columns only: at most
// `lim`, attention-mask bit set in mword), or 32.
__device__ __forceinline__ int find_in_chunk(const uint32_t (&v)[32], float m, int col0, int lim, uint32_t mword) {
  int idx = 32;
#pragma unroll
  for (int c = 31; c >= 0; --c) idx = (u2f(v[c]) == m && col0 + c <= lim && ((mword >> c) & 1u)) ? c : idx;
  return idx;
}

// How a warp's 32-entry chunk of an attention-mask row is masked, voted over the warp: every
// lane may see all 32 entries, none may see any, or mixed.  `all_vis` / `none_vis` are this
// lane's answers (its mask word all ones / zero, and the causal or ragged limit).  Key padding
// and block masks make the first two the rule away from their edges.  A warp vote: call it
// only where all 32 lanes of the warp execute it together.
constexpr int kChunkAll = 0, kChunkNone = 1, kChunkMixed = 2;
__device__ __forceinline__ int chunk_vote(bool all_vis, bool none_vis) {
  if (__all_sync(0xffffffffu, all_vis)) return kChunkAll;
  if (__all_sync(0xffffffffu, none_vis)) return kChunkNone;
  return kChunkMixed;
}
// The chunk of keys col0 .. col0 + 31 of a query row: mask word w, last visible key lim.
__device__ __forceinline__ int chunk_kind(uint32_t w, int col0, int lim) {
  return chunk_vote(w == ~0u && col0 + 31 <= lim, w == 0u || col0 > lim);
}

}  // namespace raattn
