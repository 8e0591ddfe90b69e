// quantize.cu — the fused quantizer: token-block E4M3 codes with UE8M0
// scales (per document-local 32-token block, or per token), the NVFP4 operand
// of the mixed path, and D for the dO role.
//
// FLAMIA (paper summary), §3.1 Token-Block Scaling: one power-of-two exponent
// per 32 consecutive tokens across the whole head dimension, so the codes are
// valid in both MMA orientations; §3.2 Causally Safe Scales: the exponent is
// rounded up so no element clamps; §3.6.2: blocks are document-local and the
// scale is stored per token; §3.3: D comes from the same quantized dO as dP.
// Close reading 4.4: a single fused launch produces codes and scales (here one
// launch covers Q, K and V together).
//
// One warp handles one (document-local 32-token block, head) unit: lane l
// holds elements [l*EPL, l*EPL + EPL) of each of the block's tokens (EPL =
// d/32), so every token row is read with one vector load per lane (256 or 512
// contiguous bytes per warp) and written as one contiguous 128-byte segment.
// The block is kept as raw input words (bf16 pairs stay packed); three
// blocks of 128 threads fit on an SM, each warp with 32 loads in flight.
#include "kernels.h"

namespace flamia {

// 2^e for e in [-127, 127] as a product of two normal factors (one multiply
// each, no branch): x * 2^e is exact unless the result is subnormal.
__device__ __forceinline__ float2 pow2_pair(int e) {
  const int e1 = e >> 1;
  return make_float2(exp2i(e1), exp2i(e - e1));
}

// Reduce v[0..31] (one partial per token, per lane) across the warp so that
// lane t ends with the reduction over all lanes of token t (31 shuffles).
template <bool IS_MAX>
__device__ __forceinline__ float transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool upper = (lane & s) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      float send = upper ? v[i] : v[i + s];
      float keep = upper ? v[i + s] : v[i];
      float recv = __shfl_xor_sync(0xffffffffu, send, s);
      v[i] = IS_MAX ? fmaxf(keep, recv) : (keep + recv);
    }
  }
  return v[0];
}

// Largest magnitude among a lane's packed bf16 words (max of |x| taken on the
// bf16 pairs, exact), as fp32.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t m, uint32_t w) {
  uint32_t r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(w & 0x7FFF7FFFu));
  return r;
}
__device__ __forceinline__ float bf16x2_hmax_f32(uint32_t m) {
  return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
}

// transpose_reduce<true> on 32 non-negative bf16 values packed in pairs
// (w[j] holds tokens 2j, 2j+1): four stages move whole registers (both
// tokens of a pair at once), the last splits the pair.  Lane t ends with the
// maximum of token t over all lanes (16 shuffles).
__device__ __forceinline__ float transpose_max_bf16x2(uint32_t (&w)[16], int lane) {
#pragma unroll
  for (int s = 8; s >= 1; s >>= 1) {  // token stride 2s
    const bool upper = (lane & (2 * s)) != 0;
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const uint32_t send = upper ? w[i] : w[i + s];
      const uint32_t keep = upper ? w[i + s] : w[i];
      w[i] = bf16x2_absmax(keep, __shfl_xor_sync(0xffffffffu, send, 2 * s));
    }
  }
  const bool odd = (lane & 1) != 0;  // lane 2k + 1 keeps token 2k + 1 (the high half)
  const float keep = __uint_as_float(odd ? (w[0] & 0xFFFF0000u) : (w[0] << 16));
  const float send = __uint_as_float(odd ? (w[0] << 16) : (w[0] & 0xFFFF0000u));
  return fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 1));
}

// Smallest E4M3FN code whose value is >= r (r > 0), saturating at 448.
__device__ __forceinline__ uint32_t e4m3_roundup(float r) {
  uint32_t c = pack_e4m3x2(r, 0.f) & 0xFFu;
  float v = unpack_e4m3x2((uint16_t)c).x;
  if (v < r) c += 1;
  return c > 0x7Eu ? 0x7Eu : c;
}

// Value of one E2M1 code (sign bit 3; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6).
__device__ __forceinline__ float e2m1_value(uint32_t n) {
  const uint32_t m = n & 7u, e = m >> 1, f = m & 1u;
  const float mag = (e == 0u) ? 0.5f * (float)f : (1.0f + 0.5f * (float)f) * exp2i((int)e - 1);
  return (n & 8u) ? -mag : mag;
}

// One lane's EPL input elements of one token, as raw 32-bit words, and their
// fp32 values.  bf16 -> fp32 is exact (the bf16 bits are the high half).
template <typename T, int EPL>
struct RawRow {
  static constexpr int kWords = (int)sizeof(T) * EPL / 4;
  uint32_t w[kWords];
  __device__ __forceinline__ void load(const T* p) {
    if constexpr (kWords == 4) {
      const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
      w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else if constexpr (kWords == 2) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
      w[0] = u.x; w[1] = u.y;
    } else {
      w[0] = __ldg(reinterpret_cast<const uint32_t*>(p));
    }
  }
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < kWords; ++i) w[i] = 0u;
  }
  __device__ __forceinline__ float at(int e) const {
    if constexpr (sizeof(T) == 4) return __uint_as_float(w[e]);
    else return __uint_as_float((e & 1) ? (w[e >> 1] & 0xFFFF0000u) : (w[e >> 1] << 16));
  }
};

// Hadamard rotation of one token's d-vector across the warp (FLAMIA summary
// §4.3 and close reading 四 4.4: the fused quantizer rotates Q and K to
// spread outlier channels): x -> x H_d with the Sylvester matrix (entries
// +-1), by the fast Walsh-Hadamard transform in fp32 with stages h = 1, 2,
// ..., d/2 in that order; each stage turns the pair (x[i], x[i + h]) (bit h
// of i clear) into (x[i] + x[i + h], x[i] - x[i + h]).  Lane l holds
// elements [l EPL, l EPL + EPL): the stages below EPL are in-lane, the
// others pair lane l with lane l ^ m (one shuffle per element and stage).
template <int EPL>
__device__ __forceinline__ void fwht_warp(float (&v)[EPL], int lane) {
#pragma unroll
  for (int h = 1; h < EPL; h <<= 1)
#pragma unroll
    for (int e = 0; e < EPL; ++e)
      if ((e & h) == 0) {
        const float a = v[e], b = v[e + h];
        v[e] = a + b;
        v[e + h] = a - b;
      }
  // lower lane: o + v = x[i] + x[i + h]; upper lane: o - v = x[i] - x[i + h]
  // (one fused multiply-add by +-1: the product is exact, the sum rounds once)
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] = fmaf(sgn, v[e], __shfl_xor_sync(0xffffffffu, v[e], m));
  }
}

// First token and token count of document-local 32-token block g: the
// document is the last one with blk_prefix[doc] <= g.  A 32-way search:
// every lane probes one position of the current range (blk_prefix is
// non-decreasing, so the probes at or below g form a prefix of the lanes),
// so a pass costs one load round trip and up to 32 documents take one pass.
__device__ __forceinline__ int2 block_tokens(int g, const int32_t* __restrict__ cu,
                                             const int32_t* __restrict__ blk_prefix, int n_seq, int lane) {
  int lo = 0, hi = n_seq;  // blk_prefix[lo] <= g < blk_prefix[hi]
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;
    const int pidx = lo + (lane + 1) * step;
    const bool le = pidx < hi && __ldg(blk_prefix + pidx) <= g;
    const int k = __popc(__ballot_sync(0xffffffffu, le));
    hi = min(hi, lo + (k + 1) * step);
    lo += k * step;
  }
  const int doc_start = __ldg(cu + lo), doc_end = __ldg(cu + lo + 1);
  const int t0 = doc_start + 32 * (g - __ldg(blk_prefix + lo));
  return make_int2(t0, min(32, doc_end - t0));
}

// Quantize one (32-token block g, head h) unit of one tensor.  ROT: the
// launch holds a rotated tensor; units with a.rotate quantize x H_d (fp32)
// instead of x.  The exponent pass stages each token's values (rotated or
// not) in the warp's shared-memory slice `stage` ([32 tokens][32 lanes][EPL]
// fp32, each lane reading back only what it wrote), and the code pass reads
// them from there, so 32 rotated rows never sit in registers.
// `loc` is the unit's (first token, token count); the next unit's block
// `g_next` (or -1) is located while this unit's rows are in flight.
template <typename TIn, typename TO, int HD, bool WITH_D, bool NVFP4, bool ROT>
__device__ __forceinline__ void quantize_unit(const QuantArgs& a, int2 loc, int h, int g_next,
                                              int2& loc_next, const int32_t* __restrict__ cu,
                                              const int32_t* __restrict__ blk_prefix, int n_seq, int lane,
                                              float* stage) {
  constexpr int EPL = HD / 32;  // elements per lane: 4 (d=128) or 2 (d=64)
  const TIn* __restrict__ x = static_cast<const TIn*>(a.x);
  const size_t row = (size_t)a.heads * HD;  // elements between consecutive tokens
  const int t0 = loc.x, ntok = loc.y;

  RawRow<TIn, EPL> raw[32];
#pragma unroll
  for (int t = 0; t < 32; ++t) {
    if (t < ntok) raw[t].load(x + (size_t)(t0 + t) * row + (size_t)h * HD + lane * EPL);
    else raw[t].zero();
  }
  // dO role: O's rows are read in two chunks; the first is requested now, so
  // its latency overlaps the exponent and code passes
  constexpr int kOChunk = 16;
  const TO* __restrict__ Ob = static_cast<const TO*>(a.O) + (size_t)t0 * row + (size_t)h * HD + lane * EPL;
  RawRow<TO, EPL> oa[WITH_D ? kOChunk : 1];
  if constexpr (WITH_D) {
#pragma unroll
    for (int t8 = 0; t8 < kOChunk; ++t8) {
      if (t8 < ntok) oa[t8].load(Ob + (size_t)t8 * row);
      else oa[t8].zero();
    }
  }
  if (g_next >= 0) loc_next = block_tokens(g_next, cu, blk_prefix, n_seq, lane);
  static_assert(!ROT || (!WITH_D && !NVFP4), "only Q/K/V launches of the MXFP8 path rotate");
  // token t's EPL values of this lane (rotated when the unit rotates; a zero
  // row stays zero).  ROT: `fresh` computes and stages them, else they are
  // read back from the stage.
  auto row_vals = [&](int t, float (&v)[EPL], bool fresh) {
    if constexpr (ROT) {
      float* s = stage + (t * 32 + lane) * EPL;
      if (fresh) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[e] = raw[t].at(e);
        if (a.rotate) fwht_warp<EPL>(v, lane);
        if constexpr (EPL == 4) *reinterpret_cast<float4*>(s) = make_float4(v[0], v[1], v[2], v[3]);
        else *reinterpret_cast<float2*>(s) = make_float2(v[0], v[1]);
      } else {
        if constexpr (EPL == 4) {
          const float4 u = *reinterpret_cast<const float4*>(s);
          v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
        } else {
          const float2 u = *reinterpret_cast<const float2*>(s);
          v[0] = u.x; v[1] = u.y;
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[e] = raw[t].at(e);
    }
  };
  if constexpr (!NVFP4) {
    // MXFP8 codes.  Token-block units: one exponent from the lane maxima and a
    // single warp reduction.  Per-token units (V, exact option): one warp
    // reduction per token, so every lane holds that token's exponent.
    // bf16 input, no rotation: maxima taken on the packed bf16 pairs
    constexpr bool kPackedMax = sizeof(TIn) == 2 && !ROT;
    int e_blk = 0;
    if (!a.per_token) {
      // four partial maxima (short dependency chains), three-input max
      float lm[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (kPackedMax) {
        uint32_t m2[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int t = 0; t < 32; ++t)
#pragma unroll
          for (int k = 0; k < RawRow<TIn, EPL>::kWords; ++k) m2[t & 3] = bf16x2_absmax(m2[t & 3], raw[t].w[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k) lm[k] = bf16x2_hmax_f32(m2[k]);
      } else {
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          float v[EPL];
          row_vals(t, v, true);
#pragma unroll
          for (int e = 0; e < EPL; e += 2) lm[t & 3] = fmax3(lm[t & 3], fabsf(v[e]), fabsf(v[e + 1]));
        }
      }
      e_blk = noclamp_exp_clamped(warp_max(fmaxf(fmaxf(lm[0], lm[1]), fmaxf(lm[2], lm[3]))));
    }
    int my_e = e_blk;  // exponent of token `lane`
    if (a.per_token) {
      // per-token maxima: each lane's maximum of every token, then one
      // transpose-reduce leaves token `lane`'s maximum in lane `lane` (31
      // shuffles for the unit instead of a warp reduction per token)
      if constexpr (kPackedMax) {
        // a token's lane maximum is a bf16 value: two tokens per register
        uint32_t pm2[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          uint32_t m0 = 0u, m1 = 0u;
#pragma unroll
          for (int k = 0; k < RawRow<TIn, EPL>::kWords; ++k) {
            m0 = bf16x2_absmax(m0, raw[2 * j].w[k]);
            m1 = bf16x2_absmax(m1, raw[2 * j + 1].w[k]);
          }
          // fold each token's pair of halves, then pack token 2j low, 2j+1 high
          const uint32_t f0 = bf16x2_absmax(m0, (m0 >> 16) | (m0 << 16));
          const uint32_t f1 = bf16x2_absmax(m1, (m1 >> 16) | (m1 << 16));
          pm2[j] = (f0 & 0xFFFFu) | (f1 << 16);
        }
        my_e = noclamp_exp_clamped(transpose_max_bf16x2(pm2, lane));
      } else {
        float pm[32];
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          float v[EPL];
          row_vals(t, v, true);
          float lm = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) lm = fmaxf(lm, fabsf(v[e]));
          pm[t] = lm;
        }
        my_e = noclamp_exp_clamped(transpose_reduce<true>(pm, lane));
      }
    }
    const float my_inv = exp2i(max(-my_e, -126));
    // dO role: each token's code word is kept for D, and the dO values die
    // as the codes are made, so O's rows are read afterwards (below) without
    // both blocks held in registers at once
    uint32_t cws[WITH_D ? 32 : 1];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      float v[EPL];
      row_vals(t, v, false);  // staged by the exponent pass (rotated units)
      // 2^-e is a normal fp32 for every exponent of finite data (e <= 120),
      // so one multiply per element is exact down to the E4M3 range
      const float inv_s = __shfl_sync(0xffffffffu, my_inv, a.per_token ? t : 0);
      if constexpr (WITH_D) cws[t] = 0u;
      if (t < ntok) {
        const uint64_t s2 = f2_pack(inv_s, inv_s);
        float qv[EPL];
#pragma unroll
        for (int e = 0; e < EPL; e += 2) f2_unpack(f2_mul(f2_pack(v[e], v[e + 1]), s2), qv[e], qv[e + 1]);
        uint8_t* dst = a.codes + (size_t)(t0 + t) * row + (size_t)h * HD + lane * EPL;
        uint32_t cw;
        if constexpr (EPL == 4) {
          cw = pack_e4m3x4(qv[0], qv[1], qv[2], qv[3]);
          *reinterpret_cast<uint32_t*>(dst) = cw;
        } else {
          cw = pack_e4m3x2(qv[0], qv[1]);
          *reinterpret_cast<uint16_t*>(dst) = (uint16_t)cw;
        }
        if constexpr (WITH_D) cws[t] = cw;
      }
    }
    if (lane < ntok) a.scales[(size_t)h * a.T + t0 + lane] = (uint8_t)(my_e + 127);
    if constexpr (WITH_D) {
      // D's terms are code * O (products exact in fp32); the exponent is
      // applied to the lane's partial sum (per token) or to the token's sum
      // (token block).  The second chunk of O's rows is requested before the
      // first chunk's sums.
      float dpart[32];
      RawRow<TO, EPL> ob[kOChunk];
#pragma unroll
      for (int t8 = 0; t8 < kOChunk; ++t8) {
        if (kOChunk + t8 < ntok) ob[t8].load(Ob + (size_t)(kOChunk + t8) * row);
        else ob[t8].zero();
      }
      auto d_term = [&](int t, const RawRow<TO, EPL>& orow) {
        const uint32_t cw = cws[t];
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
          const float2 d2 = unpack_e4m3x2((uint16_t)(cw >> (8 * e)));
          acc = fmaf(d2.x, orow.at(e), acc);
          acc = fmaf(d2.y, orow.at(e + 1), acc);
        }
        if (a.per_token) {
          const float2 s2 = pow2_pair(__shfl_sync(0xffffffffu, my_e, t));
          acc = (acc * s2.x) * s2.y;
        }
        dpart[t] = acc;
      };
#pragma unroll
      for (int t8 = 0; t8 < kOChunk; ++t8) d_term(t8, oa[t8]);
#pragma unroll
      for (int t8 = 0; t8 < kOChunk; ++t8) d_term(kOChunk + t8, ob[t8]);
      float dsum = transpose_reduce<false>(dpart, lane);
      if (!a.per_token) {
        const float2 s2 = pow2_pair(e_blk);
        dsum = (dsum * s2.x) * s2.y;
      }
      if (lane < ntok) a.D[(size_t)h * a.T + t0 + lane] = dsum;
    }
    return;
  } else {
    // The mixed path's quantizer: MXFP8 codes as above from per-token maxima
    // (lane t <- token t), which also feed the NVFP4 token scale.
    float pmax[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      float m = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) m = fmaxf(m, fabsf(raw[t].at(e)));
      pmax[t] = m;
    }
    float tok_amax_arr[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) tok_amax_arr[t] = pmax[t];
    const float my_tok_amax = transpose_reduce<true>(tok_amax_arr, lane);
    const int my_e = noclamp_exp_clamped(a.per_token ? my_tok_amax : warp_max(my_tok_amax));
    if (lane < ntok) a.scales[(size_t)h * a.T + t0 + lane] = (uint8_t)(my_e + 127);
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const int e_t = __shfl_sync(0xffffffffu, my_e, t);
      if (t < ntok) {
        const float inv_s = exp2i(max(-e_t, -126));
        float qv[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) qv[e] = raw[t].at(e) * inv_s;
        uint8_t* dst = a.codes + (size_t)(t0 + t) * row + (size_t)h * HD + lane * EPL;
        if constexpr (EPL == 4) *reinterpret_cast<uint32_t*>(dst) = pack_e4m3x4(qv[0], qv[1], qv[2], qv[3]);
        else *reinterpret_cast<uint16_t*>(dst) = pack_e4m3x2(qv[0], qv[1]);
      }
    }
    if (a.codes4 == nullptr) return;  // V has no NVFP4 operand
    // NVFP4 operand for the mixed path's QK^T (FLAMIA summary §3.4, §3.2):
    // per-token fp32 scale g = amax / (6 * 448), 16-element E4M3 block
    // scales rounded up so nothing exceeds 6, E2M1 codes; IEEE fp32 ops.
    constexpr int LPB = 16 / EPL;  // lanes per 16-element block
    const float my_g = (my_tok_amax == 0.f) ? 1.f : __fdiv_rn(my_tok_amax, 2688.f);
    if (lane < ntok) a.gscale4[(size_t)h * a.T + t0 + lane] = my_g;
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      const float gs = __shfl_sync(0xffffffffu, my_g, t);
      float bm = pmax[t];
#pragma unroll
      for (int s = 1; s < LPB; s <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, s));
      if (t < ntok) {
        uint32_t sc = 0u;
        if (bm > 0.f) sc = e4m3_roundup(__fdiv_rn(bm, __fmul_rn(6.f, gs)));
        const float sv = unpack_e4m3x2((uint16_t)sc).x;
        const float sg = __fmul_rn(sv, gs);
        uint32_t packed = 0u;
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
          uint32_t byte = (sc == 0u) ? 0u
                                     : pack_e2m1x2(__fdiv_rn(raw[t].at(e), sg), __fdiv_rn(raw[t].at(e + 1), sg));
          packed |= byte << (8 * (e / 2));
        }
        uint8_t* dst4 = a.codes4 + (size_t)(t0 + t) * a.heads * (HD / 2) + (size_t)h * (HD / 2) + lane * (EPL / 2);
        if constexpr (EPL == 4) *reinterpret_cast<uint16_t*>(dst4) = (uint16_t)packed;
        else *dst4 = (uint8_t)packed;
        if ((lane % LPB) == 0)
          a.scales4[(size_t)(t0 + t) * a.heads * (HD / 16) + (size_t)h * (HD / 16) + lane / LPB] = (uint8_t)sc;
      }
    }
  }
}

// Resident 128-thread blocks per SM for each variant: the register
// footprint is set by the unit held in registers (bf16 pairs packed; with D
// also O's rows; the mixed path also the per-token maxima).
template <typename TIn, typename TO, bool WITH_D, bool NVFP4, bool ROT>
constexpr int quant_blocks_per_sm() {
  if constexpr (NVFP4 || ROT) return 3;
  else if constexpr (WITH_D) return (sizeof(TIn) == 2 && sizeof(TO) == 2) ? 4 : 2;
  else return sizeof(TIn) == 2 ? 5 : 3;
}

// Grid-stride over the units of up to three tensors (Q, K, V share a launch).
template <typename TIn, typename TO, int HD, bool WITH_D, bool NVFP4, bool ROT>
__global__ void __launch_bounds__(128, (quant_blocks_per_sm<TIn, TO, WITH_D, NVFP4, ROT>())) quantize_kernel(const __grid_constant__ QuantBatch qb,
                                                          const int32_t* __restrict__ cu,
                                                          const int32_t* __restrict__ blk_prefix, int n_seq,
                                                          WsHeader* hdr) {
  extern __shared__ float4 quant_stage[];  // ROT: 32 * HD fp32 per warp
  float* const stage = ROT ? reinterpret_cast<float*>(quant_stage) + (threadIdx.x >> 5) * (32 * HD) : nullptr;
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int n_blk = hdr->n_blk32;
  int total = 0;
  for (int r = 0; r < qb.n; ++r) total += n_blk * qb.a[r].heads;
  // unit -> (tensor r, block g, head h)
  auto split = [&](int unit, int& r, int& g, int& h) {
    int u = unit;
    r = 0;
    while (r + 1 < qb.n && u >= n_blk * qb.a[r].heads) {
      u -= n_blk * qb.a[r].heads;
      ++r;
    }
    g = u / qb.a[r].heads;
    h = u - g * qb.a[r].heads;
  };
  int unit = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (unit >= total) return;
  int r, g, h;
  split(unit, r, g, h);
  int2 loc = block_tokens(g, cu, blk_prefix, n_seq, lane);
  for (; unit < total; unit += warps_total) {
    const int nxt = unit + warps_total;
    int r2 = 0, g2 = -1, h2 = 0;
    if (nxt < total) split(nxt, r2, g2, h2);
    int2 loc2 = loc;
    quantize_unit<TIn, TO, HD, WITH_D, NVFP4, ROT>(qb.a[r], loc, h, g2, loc2, cu, blk_prefix, n_seq, lane, stage);
    r = r2;
    h = h2;
    loc = loc2;
  }
}

// Raise a kernel's dynamic shared-memory limit once per device (a function
// attribute, not a stream operation).
template <auto Kernel>
static cudaError_t raise_smem_once(int smem) {
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (done[dev]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  done[dev] = e == cudaSuccess;
  return e;
}

// Grid size in waves of resident blocks (one, four and eight measured within
// 3% of each other on the batched workload; four kept).
constexpr int kQuantWaves = 4;

// Host-side launcher (called by api.cu).
cudaError_t launch_quantize(const QuantBatch& qb, int d, int in_bf16, int o_bf16, bool with_D, bool nvfp4,
                            const int32_t* cu, const int32_t* blk_prefix, int n_seq, WsHeader* hdr,
                            int max_units, int n_sms, cudaStream_t st) {
  const int want = (max_units + 3) / 4;  // four warps per block, one unit per warp
  bool rot = false;
  for (int i = 0; i < qb.n; ++i) rot = rot || qb.a[i].rotate;
  // at most kQuantWaves waves of resident blocks; the warps stride over the rest
#define FLAMIA_QL_R(TIN, TO_, HD_, WD, NV, RT)                                                            \
  do {                                                                                                    \
    const int cap = quant_blocks_per_sm<TIN, TO_, WD, NV, RT>() * n_sms * kQuantWaves;                    \
    const int blocks = want < 1 ? 1 : (want > cap ? cap : want);                                          \
    const int smem = RT ? 4 * 32 * HD_ * (int)sizeof(float) : 0;                                          \
    if (RT) {                                                                                             \
      const cudaError_t ea =                                                                              \
          raise_smem_once<quantize_kernel<TIN, TO_, HD_, WD, NV, RT>>(smem);                              \
      if (ea != cudaSuccess) return ea;                                                                   \
    }                                                                                                     \
    quantize_kernel<TIN, TO_, HD_, WD, NV, RT><<<blocks, 128, smem, st>>>(qb, cu, blk_prefix, n_seq, hdr); \
  } while (0)
#define FLAMIA_QL(TIN, TO_, HD_, WD, NV) FLAMIA_QL_R(TIN, TO_, HD_, WD, NV, false)
#define FLAMIA_QL_D(TIN, HD_, WD, NV)                           \
  do {                                                          \
    if (o_bf16) FLAMIA_QL(TIN, __nv_bfloat16, HD_, WD, NV);     \
    else FLAMIA_QL(TIN, float, HD_, WD, NV);                    \
  } while (0)
#define FLAMIA_QL_V(TIN, HD_)                                   \
  do {                                                          \
    if (with_D) FLAMIA_QL_D(TIN, HD_, true, false);             \
    else if (nvfp4) FLAMIA_QL(TIN, float, HD_, false, true);    \
    else if (rot) FLAMIA_QL_R(TIN, float, HD_, false, false, true); \
    else FLAMIA_QL(TIN, float, HD_, false, false);              \
  } while (0)
  if (in_bf16) {
    if (d == 128) FLAMIA_QL_V(__nv_bfloat16, 128); else FLAMIA_QL_V(__nv_bfloat16, 64);
  } else {
    if (d == 128) FLAMIA_QL_V(float, 128); else FLAMIA_QL_V(float, 64);
  }
#undef FLAMIA_QL_V
#undef FLAMIA_QL_D
#undef FLAMIA_QL
#undef FLAMIA_QL_R
  return cudaGetLastError();
}

}  // namespace flamia
