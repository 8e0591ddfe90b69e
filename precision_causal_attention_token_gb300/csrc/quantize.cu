// quantize.cu — the fused quantizer: token-block E4M3 codes with UE8M0
// scales (per document-local 32-token block, or per token), the NVFP4 operand
// of the mixed path, and D for the dO role.
//
// FLAMIA (paper summary), §3.1 Token-Block Scaling: one power-of-two exponent
// per 32 consecutive tokens across the whole head dimension, so the codes are
// valid in both MMA orientations; §3.2 Causally Safe Scales: the exponent is
// rounded up so no element clamps; §3.6.2: blocks are document-local and the
// scale is stored per token; §3.3: D comes from the same quantized dO as dP.
// Close reading 4.4: a single fused launch produces codes and scales.
//
// One warp handles one (document-local 32-token block, head) unit: lane l
// holds elements [l*EPL, l*EPL + EPL) of each of the block's tokens (EPL =
// d/32), so every token row is read and written as one contiguous segment.
#include "kernels.h"

namespace flamia {

// x * 2^e for e in [-127, 127] (exact unless the result is subnormal).
__device__ __forceinline__ float mul_pow2(float x, int e) {
  return (e >= -126) ? x * exp2i(e) : (x * exp2i(e + 64)) * exp2i(-64);
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

// Smallest E4M3FN code whose value is >= r (r > 0), saturating at 448.
__device__ __forceinline__ uint32_t e4m3_roundup(float r) {
  uint32_t c = pack_e4m3x2(r, 0.f) & 0xFFu;
  float v = unpack_e4m3x2((uint16_t)c).x;
  if (v < r) c += 1;
  return c > 0x7Eu ? 0x7Eu : c;
}

template <typename TIn, typename TO, int HD, bool WITH_D, bool NVFP4>
__global__ void __launch_bounds__(256) quantize_kernel(QuantArgs a, const int32_t* __restrict__ cu,
                                                       const int32_t* __restrict__ blk_prefix, int n_seq,
                                                       WsHeader* hdr) {
  constexpr int EPL = HD / 32;  // elements per lane: 4 (d=128) or 2 (d=64)
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int n_units = hdr->n_blk32 * a.heads;
  const TIn* __restrict__ x = static_cast<const TIn*>(a.x);
  const size_t row = (size_t)a.heads * HD;  // elements between consecutive tokens

  for (int unit = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); unit < n_units; unit += warps_total) {
    const int g = unit / a.heads, h = unit - g * a.heads;
    // document of block g: last doc with blk_prefix[doc] <= g
    int lo = 0, hi = n_seq;  // blk_prefix[lo] <= g < blk_prefix[hi]
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (__ldg(blk_prefix + mid) <= g) lo = mid; else hi = mid;
    }
    const int doc_start = __ldg(cu + lo), doc_end = __ldg(cu + lo + 1);
    const int t0 = doc_start + 32 * (g - __ldg(blk_prefix + lo));
    const int ntok = min(32, doc_end - t0);

    float v[32][EPL];
    float pmax[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      pmax[t] = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[t][e] = 0.f;
      if (t < ntok) {
        const TIn* p = x + (size_t)(t0 + t) * row + (size_t)h * HD + lane * EPL;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          v[t][e] = to_f32(p[e]);
          pmax[t] = fmaxf(pmax[t], fabsf(v[t][e]));
        }
      }
    }
    // per-token maxima (lane t <- token t) also feed the NVFP4 token scale
    float tok_amax_arr[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) tok_amax_arr[t] = pmax[t];
    const float my_tok_amax = transpose_reduce<true>(tok_amax_arr, lane);
    int my_e;  // exponent of token `lane`
    if (a.per_token) {
      my_e = noclamp_exp_clamped(my_tok_amax);
    } else {
      float bmax = my_tok_amax;
#pragma unroll
      for (int s = 16; s >= 1; s >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, s));
      my_e = noclamp_exp_clamped(bmax);
    }
    if (lane < ntok) a.scales[(size_t)h * a.T + t0 + lane] = (uint8_t)(my_e + 127);

    float dpart[32];
#pragma unroll
    for (int t = 0; t < 32; ++t) {
      dpart[t] = 0.f;
      const int e_t = __shfl_sync(0xffffffffu, my_e, t);
      if (t < ntok) {
        float q[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) q[e] = mul_pow2(v[t][e], -e_t);
        uint8_t* dst = a.codes + (size_t)(t0 + t) * row + (size_t)h * HD + lane * EPL;
        if constexpr (EPL == 4) {
          const uint32_t c4 = pack_e4m3x4(q[0], q[1], q[2], q[3]);
          *reinterpret_cast<uint32_t*>(dst) = c4;
          if constexpr (WITH_D) {
            const TO* op = static_cast<const TO*>(a.O) + (size_t)(t0 + t) * row + (size_t)h * HD + lane * EPL;
            float2 d01 = unpack_e4m3x2((uint16_t)(c4 & 0xFFFFu));
            float2 d23 = unpack_e4m3x2((uint16_t)(c4 >> 16));
            float acc = mul_pow2(d01.x, e_t) * to_f32(op[0]);
            acc = fmaf(mul_pow2(d01.y, e_t), to_f32(op[1]), acc);
            acc = fmaf(mul_pow2(d23.x, e_t), to_f32(op[2]), acc);
            acc = fmaf(mul_pow2(d23.y, e_t), to_f32(op[3]), acc);
            dpart[t] = acc;
          }
        } else {
          const uint16_t c2 = pack_e4m3x2(q[0], q[1]);
          *reinterpret_cast<uint16_t*>(dst) = c2;
          if constexpr (WITH_D) {
            const TO* op = static_cast<const TO*>(a.O) + (size_t)(t0 + t) * row + (size_t)h * HD + lane * EPL;
            float2 d01 = unpack_e4m3x2(c2);
            float acc = mul_pow2(d01.x, e_t) * to_f32(op[0]);
            acc = fmaf(mul_pow2(d01.y, e_t), to_f32(op[1]), acc);
            dpart[t] = acc;
          }
        }
      }
    }
    if constexpr (WITH_D) {
      const float dsum = transpose_reduce<false>(dpart, lane);
      if (lane < ntok) a.D[(size_t)h * a.T + t0 + lane] = dsum;
    }
    if constexpr (NVFP4) {
      // NVFP4 operand for the mixed path's QK^T (FLAMIA summary §3.4, §3.2):
      // per-token fp32 scale g = amax / (6 * 448), 16-element E4M3 block
      // scales rounded up so nothing exceeds 6, E2M1 codes; IEEE fp32 ops.
      constexpr int LPB = 16 / EPL;  // lanes per 16-element block
      const float my_g = (my_tok_amax == 0.f) ? 1.f : __fdiv_rn(my_tok_amax, 2688.f);
      if (lane < ntok) a.gscale4[(size_t)h * a.T + t0 + lane] = my_g;
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const float g = __shfl_sync(0xffffffffu, my_g, t);
        float bm = pmax[t];
#pragma unroll
        for (int s = 1; s < LPB; s <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, s));
        if (t < ntok) {
          uint32_t sc = 0u;
          if (bm > 0.f) sc = e4m3_roundup(__fdiv_rn(bm, __fmul_rn(6.f, g)));
          const float sg = __fmul_rn(unpack_e4m3x2((uint16_t)sc).x, g);
          uint32_t packed = 0u;
#pragma unroll
          for (int e = 0; e < EPL; e += 2) {
            uint32_t byte = (sc == 0u) ? 0u : pack_e2m1x2(__fdiv_rn(v[t][e], sg), __fdiv_rn(v[t][e + 1], sg));
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
}

// Host-side launcher (called by api.cu).
cudaError_t launch_quantize(const QuantArgs& a, int d, int in_bf16, int o_bf16, bool with_D, bool nvfp4,
                            const int32_t* cu, const int32_t* blk_prefix, int n_seq, WsHeader* hdr,
                            int max_units, cudaStream_t st) {
  int blocks = (max_units + 7) / 8;
  blocks = blocks < 1 ? 1 : (blocks > 152 * 8 ? 152 * 8 : blocks);
#define FLAMIA_QL(TIN, TO_, HD_, WD, NV) \
  quantize_kernel<TIN, TO_, HD_, WD, NV><<<blocks, 256, 0, st>>>(a, cu, blk_prefix, n_seq, hdr)
#define FLAMIA_QL_D(TIN, HD_, WD, NV)                           \
  do {                                                          \
    if (o_bf16) FLAMIA_QL(TIN, __nv_bfloat16, HD_, WD, NV);     \
    else FLAMIA_QL(TIN, float, HD_, WD, NV);                    \
  } while (0)
#define FLAMIA_QL_V(TIN, HD_)                                   \
  do {                                                          \
    if (with_D) FLAMIA_QL_D(TIN, HD_, true, false);             \
    else if (nvfp4) FLAMIA_QL(TIN, float, HD_, false, true);    \
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
  return cudaGetLastError();
}

}  // namespace flamia
