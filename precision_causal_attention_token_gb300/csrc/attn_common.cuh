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
// exact (a power-of-two scaling); the fused multiply-add rounds once.  Every
// kernel evaluates it through phat_block_logits, so all get the same bits.
__device__ __forceinline__ float score_to_y(float acc, float scale, float vf) { return __fmaf_rn(acc, scale, vf); }

// Visibility of doc-local key j for doc-local query i (document length len).
__device__ __forceinline__ bool visible(int i, int j, int len, int causal) {
  return j < len && (!causal || j <= i);
}

// Exponent of a 32-key P^ block from its largest logit M (M finite): the
// smallest e with 2^M <= 448 * 2^e, i.e. ceil(M - log2 448).  No clamp.
__device__ __forceinline__ int phat_block_exp(float M) { return (int)ceilf(__fsub_rn(M, kLog2_448)); }

constexpr int kEmptyBlock = -(1 << 30);

// Logits of one 32-key block of one query row, in place (a: S accumulator in,
// y out; masked keys -> -inf), and the block's P^ exponent (kEmptyBlock when
// every key is masked).  `kf`, `vf` point at the block's 32 per-key factors.
// In the default option 2^eK is constant over the block (document-local
// 32-token blocks), so one scale serves all 32 keys; the exact option has a
// per-key scale.  The value of every visible y is the same either way.
// Only the tile on the diagonal (and a document's last, partial tile) needs
// the mask: NEED_MASK is false on the tiles every key of which is visible,
// and the visible logits are computed identically in both forms.
template <bool EXACT, bool NEED_MASK>
__device__ __forceinline__ int phat_block_logits(float (&a)[32], float rowc, const float* kf, const float* vf,
                                                 int i_loc, int key, int len, int causal) {
  // pairs of keys go through the packed fp32 FMA (same rounding as fmaf)
  float m2[2] = {-INFINITY, -INFINITY};
  const float sb = __fmul_rn(rowc, kf[0]);
  const uint64_t sb2 = f2_pack(sb, sb);
#pragma unroll
  for (int j4 = 0; j4 < 8; ++j4) {
    const float4 v4 = *reinterpret_cast<const float4*>(vf + 4 * j4);  // 16-byte aligned factor vectors
    uint64_t sc2[2] = {sb2, sb2};
    if constexpr (EXACT) {
      const float4 k4 = *reinterpret_cast<const float4*>(kf + 4 * j4);
      const uint64_t r2 = f2_pack(rowc, rowc);
      sc2[0] = f2_mul(r2, f2_pack(k4.x, k4.y));
      sc2[1] = f2_mul(r2, f2_pack(k4.z, k4.w));
    }
    const uint64_t vv2[2] = {f2_pack(v4.x, v4.y), f2_pack(v4.z, v4.w)};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int jj = 4 * j4 + 2 * h;
      float y0, y1;
      f2_unpack(f2_fma(f2_pack(a[jj], a[jj + 1]), sc2[h], vv2[h]), y0, y1);
      if (NEED_MASK && !visible(i_loc, key + jj, len, causal)) y0 = -INFINITY;
      if (NEED_MASK && !visible(i_loc, key + jj + 1, len, causal)) y1 = -INFINITY;
      a[jj] = y0;
      a[jj + 1] = y1;
      m2[h] = fmax3(m2[h], y0, y1);
    }
  }
  const float M = fmaxf(m2[0], m2[1]);
  return (M == -INFINITY) ? kEmptyBlock : phat_block_exp(M);
}

// p = 2^(y - E) for two keys (<= 448 up to the approximation of ex2; the cvt
// saturates), with nE2 = phat_neg_exp(E).  An empty block (E = kEmptyBlock)
// has y = -inf everywhere, so p = 0 with no test; a caller that wants zeros
// for finite y passes E = kZeroCodes.  y + (-E) is the IEEE difference y - E.
__device__ __forceinline__ uint64_t phat_neg_exp(int E) {
  const float nE = -(float)E;
  return f2_pack(nE, nE);
}
__device__ __forceinline__ void phat_values2(float y0, float y1, uint64_t nE2, float& p0, float& p1) {
  float d0, d1;
  f2_unpack(f2_add(f2_pack(y0, y1), nE2), d0, d1);
  p0 = ex2_approx(d0);
  p1 = ex2_approx(d1);
}
constexpr int kZeroCodes = 1 << 30;  // 2^(y - 2^30) = 0 for every finite logit

// P^ codes of one 32-key block from its logits and exponent, as 8 words of
// 4 E4M3 bytes.
__device__ __forceinline__ void phat_block_codes(const float (&y)[32], int E, uint32_t (&codes)[8]) {
  const uint64_t nE2 = phat_neg_exp(E);
#pragma unroll
  for (int q4 = 0; q4 < 8; ++q4) {
    float pv[4];
    phat_values2(y[4 * q4], y[4 * q4 + 1], nE2, pv[0], pv[1]);
    phat_values2(y[4 * q4 + 2], y[4 * q4 + 3], nE2, pv[2], pv[3]);
    codes[q4] = pack_e4m3x4(pv[0], pv[1], pv[2], pv[3]);
  }
}

// One 32-key block of logits for one row, read from tensor memory.
template <bool EXACT, bool NEED_MASK>
__device__ __forceinline__ int phat_logits1(uint32_t t_s, float (&y)[32], float rowc, const float* kf,
                                            const float* vf, int i_loc, int key, int len, int causal) {
  uint32_t rr[32];
  tmem_ld32(t_s, rr);
  tmem_ld_wait_regs(rr);
#pragma unroll
  for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(rr[j]);
  return phat_block_logits<EXACT, NEED_MASK>(y, rowc, kf, vf, i_loc, key, len, causal);
}

// Bytes of one 128-token score-operand tile: E4M3 codes (MXFP8 path) or
// packed E2M1 codes, two to a byte (mixed path).
template <int HD, bool NV4>
constexpr int score_tile_bytes() {
  return NV4 ? kTile * HD / 2 : kTile * HD;
}

// Mixed path: the 16-element block scales of a 128-token tile, staged for
// copy_scales_x4 in HD/64 blocks of 512 bytes (block s: K-elements
// 64s..64s+63); row r of a block holds the 4-byte scale words of tokens r,
// r + 32, r + 64, r + 96.  One warp; tokens at or past T get zero scales (their
// codes are zero-filled).  The writes are made visible to the tensor core's
// copies (async proxy) before the caller's arrival.
template <int HD>
__device__ __forceinline__ void stage_nv_scales(uint32_t* dst, const uint8_t* bs, int heads, int h, int tok0, int T,
                                                int lane) {
  constexpr int NS = HD / 64;  // scale words per token-head
  uint32_t wv[4][NS];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int tok = tok0 + lane + 32 * c;
    const uint8_t* src = bs + ((size_t)tok * heads + h) * (HD / 16);
    if constexpr (NS == 2) {
      const uint2 v = tok < T ? *reinterpret_cast<const uint2*>(src) : make_uint2(0u, 0u);
      wv[c][0] = v.x;
      wv[c][1] = v.y;
    } else {
      wv[c][0] = tok < T ? *reinterpret_cast<const uint32_t*>(src) : 0u;
    }
  }
#pragma unroll
  for (int s = 0; s < NS; ++s)
    *reinterpret_cast<uint4*>(dst + s * 128 + lane * 4) = make_uint4(wv[0][s], wv[1][s], wv[2][s], wv[3][s]);
  fence_proxy_async_smem();
}

// Mixed path: copy a staged tile's scales (stage_nv_scales) to tensor memory
// columns col..col + 4 HD/64 - 1 (MMA thread).
template <int HD>
__device__ __forceinline__ void copy_nv_scales(uint32_t col_tmem, const uint32_t* src) {
#pragma unroll
  for (int s = 0; s < HD / 64; ++s) copy_scales_x4(col_tmem + 4 * s, src + s * 128);
}

// S = Q K^T for one 128 x 128 tile into TMEM column d_s.
//  MXFP8: E4M3 tiles with rows of HD bytes (swizzle = HD bytes), kind::f8f6f4,
//         32 K-elements per instruction.
//  Mixed: packed E2M1 tiles with rows of HD/2 bytes (swizzle = HD/2 bytes),
//         kind::mxf4nvf4 with the E4M3 16-element block scales in tensor
//         memory (sfa: Q's, sfb: K's, as copy_nv_scales puts them), 64
//         K-elements per instruction, fp32 accumulation.
template <int HD, bool NV4>
__device__ __forceinline__ void issue_scores(uint32_t d_s, const uint8_t* qt, const uint8_t* kt, uint32_t sfa = 0,
                                             uint32_t sfb = 0) {
  const uint32_t qa = smem_u32(qt), ka = smem_u32(kt);
  if constexpr (NV4) {
    const uint32_t id = idesc_mxf4nvf4(128, 128);
    constexpr uint32_t rb = HD / 2, swz = HD == 128 ? kSwz64 : kSwz32;
#pragma unroll
    for (int s = 0; s < HD / 64; ++s)
      mma_mxf4nvf4(d_s, smem_desc(qa + 32 * s, 16, 8 * rb, swz), smem_desc(ka + 32 * s, 16, 8 * rb, swz), id,
                   sfa + 4 * s, sfb + 4 * s, s > 0);
  } else {
    const uint32_t id = idesc_f8(128, 128, 0, 0);
    constexpr uint32_t swz = HD == 128 ? kSwz128 : kSwz64;
#pragma unroll
    for (int kk = 0; kk < HD / 32; ++kk)
      mma_f8(d_s, smem_desc(qa + 32 * kk, 16, 8 * HD, swz), smem_desc(ka + 32 * kk, 16, 8 * HD, swz), id, kk > 0);
  }
}

// TMA of one 128-token score-operand tile (row `tok0`, head `head`).
template <int HD, bool NV4>
__device__ __forceinline__ void load_score_tile(uint8_t* dst, const CUtensorMap* map8, const CUtensorMap* mapn,
                                                uint64_t* bar, int head, int tok0) {
  if constexpr (NV4) {
    tma_load_3d(dst, mapn, bar, 0, head, tok0);
  } else {
    tma_load_3d(dst, map8, bar, 0, head, tok0);
  }
}

// x * 2^e for e <= 127, flushed to 0 below 2^-126 (for normaliser terms and
// rescale factors, where such terms are far below fp32 resolution).
__device__ __forceinline__ float ldexp_fast(float x, int e) { return e >= -126 ? x * exp2i(min(e, 127)) : 0.f; }

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
