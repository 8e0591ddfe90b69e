// attn_common.cuh — pieces the forward and the backward must share bit for
// bit: the score-to-logit arithmetic, the causal/document mask and the P^
// quantizer.  FLAMIA (paper summary), §3.3 Forward–Backward Numerical
// Consistency: the backward recomputes scores from the same quantized Q and K
// with the same tiling, diagonal decisions and exponent evaluation.  Both
// kernels call these functions on the same 128x128 tiles with the same
// operands, so the recomputed P^ codes equal the forward's.
#pragma once
#include "common.cuh"

namespace flamia {

constexpr int kTile = 128;                      // queries and keys per tile
constexpr float kLog2_448 = 8.807354922057604f;  // log2(448), E4M3 max

// y = acc * (rowc * kf) + vf with rowc = softmax_scale * log2(e) * 2^eQ(i),
// kf = 2^eK(j), vf = eV(j): the base-2 logit with the V fold.  rowc * kf is
// exact (a power-of-two scaling); the two remaining ops are rounded once
// each, never contracted into an FMA, so every kernel gets the same bits.
__device__ __forceinline__ float score_to_y(float acc, float rowc, float kf, float vf) {
  return __fadd_rn(__fmul_rn(acc, __fmul_rn(rowc, kf)), vf);
}

// Visibility of doc-local key j for doc-local query i (document length len).
__device__ __forceinline__ bool visible(int i, int j, int len, int causal) {
  return j < len && (!causal || j <= i);
}

// Exponent of a 32-key P^ block from its largest logit M (M finite): the
// smallest e with 2^M <= 448 * 2^e, i.e. ceil(M - log2 448).  No clamp.
__device__ __forceinline__ int phat_block_exp(float M) { return (int)ceilf(__fsub_rn(M, kLog2_448)); }

// p = 2^(y - E) (<= 448 up to the approximation of ex2; the cvt saturates).
__device__ __forceinline__ float phat_value(float y, int E) { return ex2_approx(__fsub_rn(y, (float)E)); }

constexpr int kEmptyBlock = -(1 << 30);

// x * 2^e for any integer e (exact while the result stays normal).
__device__ __forceinline__ float ldexp_f(float x, int e) {
  if (e >= -126 && e <= 127) return x * exp2i(e);
  if (e < -252) return 0.f * x;
  if (e < -126) return (x * exp2i(-126)) * exp2i(e + 126);
  if (e > 254) return x * exp2i(127) * exp2i(127);
  return (x * exp2i(127)) * exp2i(e - 127);
}

// 2^e for e in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2_127(int e) { return e >= -126 ? exp2i(e) : exp2i(-126) * 0.5f; }

}  // namespace flamia
