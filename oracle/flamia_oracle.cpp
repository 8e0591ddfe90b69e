// flamia_oracle.cpp — test infrastructure, NOT part of the product path.
//
// A plain, slow, single-threaded fp64 restatement of the FLAMIA training call
// (quantize -> forward -> quantize dO + D -> backward) used only to check the
// CUDA library.  Nothing here is blocked, fused or reordered beyond what the
// method's definitions state; every function says which passage it follows.
// It shares no code, header, table or constant with the CUDA path.  Only the
// tests, __graft_entry__.smoke() and bench.py's CPU-baseline leg load it.
//
// Sources (pages describing FLAMIA; cited by title and section):
//   [SUM]  "FLAMIA: FLAsh MIcroscaling Attention for Fast and Causally Safe
//          Training on Blackwell" (paper summary page), claim bullets under
//          §3.1 Token-Block Scaling, §3.2 Causally Safe Scales,
//          §3.3 Forward–Backward Numerical Consistency, §3.4 Paths,
//          §3.6.2 Load-Balanced Scheduling, §4.5 Causality.
//   [READ] "因果安全的低精度注意力——FLAMIA Blackwell 训练内核精读"
//          (close reading), 一 (background: MX formats), 四 4.1 token-block
//          scaling, 4.2 causally safe scales, 4.3 forward/backward
//          consistency, 五 5.1 metrics (leakage probe).
// Where the pages leave a step open the reading taken is named at the step.
//
// Conventions: packed THD tensors [T][H][d]; per-token metadata [H][T];
// cu_seqlens[0..nseq] with cu_seqlens[nseq] == T.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <vector>
#include <algorithm>

extern "C" {

// ---------------------------------------------------------------------------
// Codecs, written from the format definitions ([READ] 一, MX formats: E4M3
// codes, E2M1 codes, UE8M0 power-of-two scales, E4M3 block scales for NVFP4).
// ---------------------------------------------------------------------------

// OCP E4M3FN: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field
// 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity.
double orc_e4m3_decode(unsigned code) {
  unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  if (e == 15u && m == 7u) return NAN;
  double mag = (e == 0u) ? std::ldexp((double)m, -9)                // m/8 * 2^-6
                         : std::ldexp(8.0 + (double)m, (int)e - 10); // (1+m/8) * 2^(e-7)
  return s ? -mag : mag;
}

// Round-to-nearest-even into E4M3FN.  The non-negative finite codes 0x00..0x7E
// are monotone in value, so the nearest code is found by bisection over the
// decoded values; a tie picks the code with an even mantissa (even code).
// Magnitudes at or above 448 saturate to 448 (the quantizers below never
// produce them: their exponent rule keeps every scaled magnitude <= 448).
unsigned orc_e4m3_encode(double x) {
  if (std::isnan(x)) return 0x7Fu;
  unsigned sign = std::signbit(x) ? 0x80u : 0u;
  double a = std::fabs(x);
  if (a >= 448.0) return sign | 0x7Eu;
  unsigned lo = 0, hi = 0x7E;  // invariant: value(lo) <= a
  while (lo < hi) {
    unsigned mid = (lo + hi + 1) / 2;
    if (orc_e4m3_decode(mid) <= a) lo = mid; else hi = mid - 1;
  }
  double vl = orc_e4m3_decode(lo);
  if (vl == a) return sign | lo;
  unsigned up = lo + 1;
  double dl = a - vl, du = orc_e4m3_decode(up) - a;
  unsigned c = (dl < du) ? lo : (du < dl) ? up : ((lo & 1u) ? up : lo);
  return sign | c;
}

// Smallest positive E4M3FN value >= r (a "rounded up" E4M3 scale, used for the
// NVFP4 16-element block scales so that no element clamps).  r <= 0 -> code 0;
// r above 448 saturates to 448.
unsigned orc_e4m3_roundup(double r) {
  if (!(r > 0.0)) return 0u;
  if (r >= 448.0) return 0x7Eu;
  for (unsigned c = 1; c <= 0x7E; ++c)
    if (orc_e4m3_decode(c) >= r) return c;
  return 0x7Eu;
}

// E2M1 (FP4): sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no NaN or infinity.
double orc_e2m1_decode(unsigned code) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[code & 7u];
  return (code & 8u) ? -v : v;
}

// Round-to-nearest-even into E2M1 (ties to the even code), saturating at 6.
unsigned orc_e2m1_encode(double x) {
  unsigned sign = std::signbit(x) ? 8u : 0u;
  double a = std::fabs(x);
  if (a >= 6.0) return sign | 7u;
  unsigned lo = 0;
  while (lo < 7 && orc_e2m1_decode(lo + 1) <= a) ++lo;
  double vl = orc_e2m1_decode(lo);
  if (vl == a) return sign | lo;
  unsigned up = lo + 1;
  double dl = a - vl, du = orc_e2m1_decode(up) - a;
  unsigned c = (dl < du) ? lo : (du < dl) ? up : ((lo & 1u) ? up : lo);
  return sign | c;
}

// UE8M0 scale byte b encodes 2^(b-127); 255 is NaN.
double orc_ue8m0_decode(unsigned b) {
  if ((b & 255u) == 255u) return NAN;
  return std::ldexp(1.0, (int)(b & 255u) - 127);
}

// The "rounded-up" (no-clamp) block exponent ([SUM] §3.2; [READ] 4.2): the
// smallest integer e with amax <= 448 * 2^e, so that the largest scaled
// magnitude never exceeds E4M3's 448.  (The MX reference rule floor(log2 amax)
// - 8 can push the block maximum past 448, where it clamps and leaks.)
// amax = f * 2^k with f in [0.5, 1) and 448 = 0.875 * 2^9, hence
//   e = k - 9 when f <= 0.875, else k - 8.
// Not clamped here; callers that store a UE8M0 byte clamp to [-127, 127].
// An all-zero block takes e = 0 (reading: its codes are zero either way).
int orc_noclamp_exponent(double amax) {
  if (amax == 0.0) return 0;
  int k = 0;
  double f = std::frexp(amax, &k);
  return (f <= 0.875) ? k - 9 : k - 8;
}

static int clamp127(int e) { return e < -127 ? -127 : (e > 127 ? 127 : e); }

// Exponent stored as a UE8M0 byte: the no-clamp exponent clamped to the byte's
// range [-127, 127].
int orc_scale_exponent(double amax) { return clamp127(orc_noclamp_exponent(amax)); }

// bf16 round-to-nearest-even of a double (through fp32, the GPU's own order:
// outputs are accumulated in fp32 and cast once).
double orc_round_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u) return (double)f;  // inf / nan
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  u &= 0xFFFF0000u;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// IEEE binary16 round-to-nearest-even of a double: 11 significant bits down
// to 2^-14, a fixed step of 2^-24 below (subnormals), infinity from 65520 up.
double orc_round_f16(double x) {
  if (std::isnan(x)) return x;
  double a = std::fabs(x);
  if (a >= 65520.0) return std::copysign(INFINITY, x);
  int e = 0;
  std::frexp(a, &e);                       // a = f * 2^e, f in [0.5, 1)
  int step = (a >= std::ldexp(1.0, -14)) ? e - 11 : -24;
  double q = std::nearbyint(std::ldexp(a, -step));  // ties to even (default rounding mode)
  return std::copysign(std::ldexp(q, step), x);
}

// Bit-level exponential for inference ([SUM] §3.7 and §4.4; [READ] 4.5: the
// Schraudolph variant for the 8-bit P^ evaluates the piecewise-linear
// 2^floor(z) (1 + frac(z)) in the bf16 bit field, written there by a fused
// multiply-add as a fixed-point number, with a shift that makes its error
// zero-mean).  Reading: the bf16 pattern is n = RNE(128 z) + 128 * 127 - 7,
// i.e. the fraction rounded to 7 bits and moved down by 7 units of the last
// place: the mean of log2((1 + f) / 2^f) over f in [0, 1) is
// 2 - 1/ln 2 - 1/2 = 0.0573, or 7.3 such units.  z is first raised to
// z_lo = -126.9453125, where n = 0, so z <= z_lo gives exactly 0 and n never
// goes negative.
double orc_bitexp2(double z) {
  const double z_lo = -126.9453125;
  if (!(z > z_lo)) z = z_lo;  // also -inf and NaN
  const long n = (long)std::nearbyint(128.0 * z) + 128L * 127 - 7;  // RNE: the default mode
  const int e = (int)(n >> 7), mant = (int)(n & 127);
  return e == 0 ? std::ldexp((double)mant, -133) : std::ldexp(128.0 + mant, e - 134);
}

// Hadamard rotation of Q and K before quantization ([SUM] abstract and §4.3
// Ablation Study: the fused quantizer applies a Hadamard rotation; [READ] 四
// 4.4, fused quantization: QuIP-style incoherence processing mixes the
// head-dimension channels to spread outliers, and an orthogonal transform
// keeps the dot products).  Reading: the Sylvester matrix H_d (entries +-1,
// H_2n = [[H_n, H_n], [H_n, -H_n]]), unnormalised, applied to each token's
// d-vector (x -> x H_d); the 1/d of H_d H_d = d I goes into the softmax scale.
// The rotated values are what gets quantized, so they are formed in fp32, the
// precision the kernel decides the codes in, by the fast Walsh-Hadamard
// transform: stages h = 1, 2, 4, ..., d/2, each replacing the pair
// (x[i], x[i + h]) (i with bit h clear) by (x[i] + x[i + h], x[i] - x[i + h]),
// every sum rounded to fp32.  x: n rows of d floats, in place.
void orc_fwht_f32(float* x, int n, int d) {
  for (int r = 0; r < n; ++r) {
    float* v = x + (size_t)r * d;
    for (int h = 1; h < d; h <<= 1)
      for (int i = 0; i < d; ++i)
        if ((i & h) == 0) {
          const float a = v[i], b = v[i + h];
          v[i] = a + b;
          v[i + h] = a - b;
        }
  }
}

// ---------------------------------------------------------------------------
// Quantizers.
// ---------------------------------------------------------------------------

// Token-block quantization ([SUM] §3.1; [READ] 4.1; document-local blocks,
// [SUM] §3.6.2): inside each document, consecutive runs of `block` tokens
// (the last run of a document may be shorter) share one power-of-two exponent
// per head, taken over the whole run and the full head dimension.  block = 32
// is the default; block = 1 is the per-token scaling of the exact option and of
// V (one exponent per key).  Blocks never cross a cu_seqlens boundary.
//   x:      [T][H][d] values
//   codes:  [T][H][d] E4M3FN codes of x * 2^-e
//   scales: [H][T]    UE8M0 byte e + 127, replicated for every token of a block
void orc_quantize_blocks(const double* x, int T, int H, int d, const int* cu, int nseq,
                         int block, unsigned char* codes, unsigned char* scales) {
  for (int doc = 0; doc < nseq; ++doc) {
    for (int s = cu[doc]; s < cu[doc + 1]; s += block) {
      int e_end = std::min(s + block, cu[doc + 1]);
      for (int h = 0; h < H; ++h) {
        double amax = 0.0;
        for (int t = s; t < e_end; ++t)
          for (int k = 0; k < d; ++k)
            amax = std::max(amax, std::fabs(x[((size_t)t * H + h) * d + k]));
        int e = orc_scale_exponent(amax);
        for (int t = s; t < e_end; ++t) {
          scales[(size_t)h * T + t] = (unsigned char)(e + 127);
          for (int k = 0; k < d; ++k) {
            size_t i = ((size_t)t * H + h) * d + k;
            codes[i] = (unsigned char)orc_e4m3_encode(std::ldexp(x[i], -e));
          }
        }
      }
    }
  }
}

// Value of an E4M3 payload with per-token UE8M0 bytes: code * 2^(byte-127).
void orc_dequantize_blocks(const unsigned char* codes, const unsigned char* scales, int T,
                           int H, int d, double* out) {
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      int e = (int)scales[(size_t)h * T + t] - 127;
      for (int k = 0; k < d; ++k) {
        size_t i = ((size_t)t * H + h) * d + k;
        out[i] = std::ldexp(orc_e4m3_decode(codes[i]), e);
      }
    }
}

// Mixed-path Q/K quantization (NVFP4) ([SUM] §3.4 and §3.2: per-token NVFP4
// scales for Q and K, one scale per 16 head-dimension elements; [READ] 一:
// NVFP4 = 16-element blocks with an E4M3 scale plus an fp32 second-level
// scale).  Reading (the pages fix neither the fp32 granularity nor the op
// order): the second level is per token, g = fl32(amax_token / 2688) with
// 2688 = 6 * 448 (g = 1 for an all-zero token); each 16-block takes the
// rounded-up E4M3 scale s = roundup(fl32(amax_block / fl32(6 g))) so that no
// element exceeds 6 after scaling; codes = RNE_E2M1(fl32(x / fl32(s g))).
// Every step is an IEEE fp32 operation in this order.  An all-zero block takes
// s = 0 and zero codes.
//   codes:  [T][H][d] one E2M1 code per byte (low nibble)
//   bscale: [T][H][d/16] E4M3 codes
//   gscale: [H][T] fp32 second-level scale
void orc_quantize_nvfp4(const double* x, int T, int H, int d, unsigned char* codes,
                        unsigned char* bscale, float* gscale) {
  int nb = d / 16;
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      const double* row = x + ((size_t)t * H + h) * d;
      float amax_t = 0.0f;
      for (int k = 0; k < d; ++k) amax_t = std::max(amax_t, (float)std::fabs(row[k]));
      float g = (amax_t == 0.0f) ? 1.0f : amax_t / 2688.0f;
      gscale[(size_t)h * T + t] = g;
      float six_g = 6.0f * g;
      for (int b = 0; b < nb; ++b) {
        float amax_b = 0.0f;
        for (int k = 16 * b; k < 16 * b + 16; ++k) amax_b = std::max(amax_b, (float)std::fabs(row[k]));
        unsigned sc = (amax_b == 0.0f) ? 0u : orc_e4m3_roundup((double)(amax_b / six_g));
        bscale[((size_t)t * H + h) * nb + b] = (unsigned char)sc;
        float sg = (float)orc_e4m3_decode(sc) * g;
        for (int k = 16 * b; k < 16 * b + 16; ++k) {
          size_t i = ((size_t)t * H + h) * d + k;
          codes[i] = (sc == 0u) ? 0u : (unsigned char)orc_e2m1_encode((double)((float)row[k] / sg));
        }
      }
    }
}

// Value of an NVFP4 payload: e2m1(code) * e4m3(bscale) * g.
void orc_dequantize_nvfp4(const unsigned char* codes, const unsigned char* bscale,
                          const float* gscale, int T, int H, int d, double* out) {
  int nb = d / 16;
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      for (int k = 0; k < d; ++k) {
        size_t i = ((size_t)t * H + h) * d + k;
        double s = orc_e4m3_decode(bscale[((size_t)t * H + h) * nb + k / 16]);
        out[i] = orc_e2m1_decode(codes[i]) * s * (double)gscale[(size_t)h * T + t];
      }
}

// D_i = sum_d dO^_id * O_id, with dO^ the same quantized dO that feeds dP and
// O as stored ([SUM] §3.3; [READ] 4.3).
void orc_compute_D(const double* dOq, const double* O_stored, int T, int H, int d, double* D) {
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int k = 0; k < d; ++k) {
        size_t i = ((size_t)t * H + h) * d + k;
        acc += dOq[i] * O_stored[i];
      }
      D[(size_t)h * T + t] = acc;
    }
}

// ---------------------------------------------------------------------------
// Attention forward + backward over packed documents, fp64.
// ---------------------------------------------------------------------------

struct orc_attn_cfg {
  int T, H, Hkv, d, nseq;
  int causal;            // 1: key j visible to query i iff j <= i (same document)
  double softmax_scale;  // S_ij = softmax_scale * <q_i, k_j>
  int quant_p;           // quantize P^ per (row, 32-key block) with the V fold
  int quant_ds;          // quantize dS (32x32 blocks; exact option: see below)
  int quant_pt;          // quantize the dV operand P~ in 32x32 blocks
  int exact;             // exact option: per-row dS exponents for dQ ([SUM] §4.5)
  int out_round;         // O as stored: 0 kept in fp64, 1 rounded to bf16, 2 to fp32
  int bitexp;            // inference: 2^z by the bit-level approximation on 5 of every 8 key pairs
  int dq_fp16;           // dQ partials of each 128-key tile in FP16 with a row prescale
  int dq_causal_scale;   // the prescale from keys j <= i only (else the whole document)
};

// The power-of-two dQ prescale of one query row ([READ] 四 4.4: FP16 dQ
// partials with a data-dependent power-of-two prescale, since a fixed one
// overflows on outlier K channels; [SUM] §4.5: the optional causal dQ scale).
// Reading: a bound of |dQ_i| from the exponent bytes alone.  With
// |dO^_i|_2 <= sqrt(d) 448 2^edO(i), |V^_j|_2 <= sqrt(d) 448 2^eV(j) and
// |K^_j|_inf <= 448 2^eK(j) (no element clamps), |dP_ij - D_i| stays below
// 2 (1 + 2^-4) d 448^2 2^(edO + eV) and
//   |dQ_i| <= 2.5 d 448^3 scale 2^(edO(i) + MK + MV) =: 2^(c0 + edO + MK + MV)
// with MK, MV the largest eK, eV over the keys the rule looks at: the whole
// document by default (a sequence-range dependency), keys j <= i with the
// causal dQ scale.  The prescale 2^p, p = 15 - c0 - (edO + MK + MV) clamped
// to [-126, 127], keeps every partial sum of 2^p dQ_i within 2^15 < 65504.
int orc_dq_prescale_c0(int d, double softmax_scale) {
  int e = 0;
  double f = std::frexp(2.5 * d * 448.0 * 448.0 * 448.0 * softmax_scale, &e);
  return f > 0.5 ? e : e - 1;  // ceil(log2(.)), exact
}
int orc_dq_prescale(int c0, int edO, int mk, int mv) {
  int p = 15 - c0 - (edO + mk + mv);
  return p < -126 ? -126 : (p > 127 ? 127 : p);
}

// The prescale exponent of every query row: p [H][T] from the exponent bytes
// eK, eV [Hkv][T] and edO [H][T].  MK, MV run over the row's document, or
// over keys j <= i when causal and causal_scale are both set.
void orc_dq_prescales(int T, int H, int Hkv, const int* cu, int nseq, const int* eK, const int* eV,
                      const int* edO, int c0, int causal, int causal_scale, int* p) {
  const int G = H / Hkv;
  for (int doc = 0; doc < nseq; ++doc) {
    const int s0 = cu[doc], L = cu[doc + 1] - cu[doc];
    for (int h = 0; h < H; ++h) {
      const int hk = h / G;
      int mk_doc = -1000, mv_doc = -1000;
      for (int j = 0; j < L; ++j) {
        mk_doc = std::max(mk_doc, eK[(size_t)hk * T + s0 + j]);
        mv_doc = std::max(mv_doc, eV[(size_t)hk * T + s0 + j]);
      }
      int mk = -1000, mv = -1000;
      for (int i = 0; i < L; ++i) {
        mk = std::max(mk, eK[(size_t)hk * T + s0 + i]);
        mv = std::max(mv, eV[(size_t)hk * T + s0 + i]);
        const bool pre = causal && causal_scale;
        p[(size_t)h * T + s0 + i] = orc_dq_prescale(c0, edO[(size_t)h * T + s0 + i], pre ? mk : mk_doc,
                                                    pre ? mv : mv_doc);
      }
    }
  }
}

// Quantize v (values of one block) to E4M3 codes with the no-clamp exponent of
// the block's max-abs and return the dequantized values in place.  `clampexp`
// selects the UE8M0 byte clamp [-127, 127] (dS, P~) or none (P^, whose
// exponent is kept relative to a row anchor).
static void quantize_block_inplace(std::vector<double*>& v, bool clampexp) {
  double amax = 0.0;
  for (double* p : v) amax = std::max(amax, std::fabs(*p));
  int e = clampexp ? orc_scale_exponent(amax) : orc_noclamp_exponent(amax);
  for (double* p : v) *p = std::ldexp(orc_e4m3_decode(orc_e4m3_encode(std::ldexp(*p, -e))), e);
}

// One training call's attention part.  Inputs are the values of the quantized
// operands (Q^, K^, V^, dO^ dequantized; or unquantized values for the
// identity reference).  Qs/Ks are the operands of the scores (S and its
// recompute); Q/K those of dK and dQ.  They are the same arrays on the MXFP8
// path and differ on the mixed path, where QK^T alone runs in NVFP4 ([SUM]
// §3.4).  The integer exponents that the folds use:
//   eQ [H][T], eK [Hkv][T], eV [Hkv][T], edO [H][T].
// Outputs: O [T][H][d] as stored (rounded per out_round), D [H][T],
// lse2 [H][T] = log2 of the row's normaliser (base-2 log-sum-exp of x),
// dQ [T][H][d], dK/dV [T][Hkv][d].  dO == nullptr runs the forward only.
//
// Per (document, query head), with keys counted from the document start:
//  1. S_ij = scale * <Q^_i, K^_j>, x_ij = S_ij * log2(e); masked unless i, j
//     are in the same document and (non-causal or j <= i).
//  2. P^ ([SUM] §3.1–§3.3; reading: one exponent per (query row, 32-key
//     block), blocks counted from the document start; masked keys excluded):
//     y_ij = x_ij + eV(j) (the V fold: V's per-key factor moved into P along
//     the contraction axis), a_ij = 2^y_ij, E_ib = no-clamp exponent of the
//     block max of a, codes RNE_E4M3(a_ij 2^-E_ib).  Evaluated relative to the
//     integer anchor m_i = ceil(max_j x_ij): the no-clamp rule commutes with
//     integer shifts, so the codes are the same as for the absolute values.
//  3. l_i = sum_j 2^(x_ij - m_i) over unmasked keys (reading: the normaliser
//     uses the unquantized probabilities, as FlashAttention does).
//  4. O_i = sum_j P^_ij 2^-eV(j) V^_j / l_i.
//  5. D_i = <dO^_i, O_i as stored>.
//  6. dP_ij = <dO^_i, V^_j>; Pn_ij = P^_ij 2^-eV(j) / l_i; dS_ij = Pn_ij (dP_ij - D_i)
//     (straight-through: quantizers act as identity in the derivative).
//  7. dS^ ([SUM] §3.3, [READ] 4.3: one exponent per 32x32 block from the
//     block's max-abs; the single payload serves dQ and dK).  Exact option
//     ([SUM] §4.5: per-query-row dS exponent): the dQ operand is quantized per
//     (query row, 32-key block) on dS_ij 2^eK(j) and the fold removed; the dK
//     operand is a separate 32x32 encoding of dS_ij 2^eQ(i), fold removed.
//     (Reading: every factor that varies along a contraction is folded into the
//     other operand before that operand's block quantization.)
//  8. dQ_i = scale * sum_j dS^_ij K^_j;  dK_j = scale * sum_i dS^_ij Q^_i.
//  9. P~ (reading; the pages give no layout for the dV operand): a 32x32
//     block quantization of Pn_ij 2^edO(i), fold removed; dV_j = sum_i P~_ij dO^_i.
// 10. GQA: dK and dV summed over the query heads that share a KV head.
void orc_attention(const orc_attn_cfg* cfg, const int* cu, const double* Qs, const double* Ks,
                   const double* Q, const double* K,
                   const double* V, const double* dO, const int* eQ, const int* eK,
                   const int* eV, const int* edO, double* O, double* D, double* lse2,
                   double* dQ, double* dK, double* dV) {
  const int T = cfg->T, H = cfg->H, Hkv = cfg->Hkv, d = cfg->d;
  const int G = H / Hkv;
  const double LOG2E = 1.4426950408889634073599246810019;
  const bool bwd = (dO != nullptr);
  std::vector<int> pq((size_t)T * H, 0);  // dQ prescale exponents (FP16 partials)
  if (bwd && cfg->dq_fp16)
    orc_dq_prescales(T, H, Hkv, cu, cfg->nseq, eK, eV, edO, orc_dq_prescale_c0(d, cfg->softmax_scale),
                     cfg->causal, cfg->dq_causal_scale, pq.data());
  if (bwd) {
    std::fill(dQ, dQ + (size_t)T * H * d, 0.0);
    std::fill(dK, dK + (size_t)T * Hkv * d, 0.0);
    std::fill(dV, dV + (size_t)T * Hkv * d, 0.0);
  }
  for (int doc = 0; doc < cfg->nseq; ++doc) {
    const int s0 = cu[doc], L = cu[doc + 1] - cu[doc];
    if (L <= 0) continue;
    std::vector<double> x((size_t)L * L), P((size_t)L * L), dS((size_t)L * L);
    std::vector<char> vis((size_t)L * L);
    std::vector<double> l(L);
    std::vector<int> m(L);
    for (int h = 0; h < H; ++h) {
      const int hk = h / G;
      auto q = [&](int i, int k) { return Q[((size_t)(s0 + i) * H + h) * d + k]; };
      auto kk = [&](int j, int k) { return K[((size_t)(s0 + j) * Hkv + hk) * d + k]; };
      auto vv = [&](int j, int k) { return V[((size_t)(s0 + j) * Hkv + hk) * d + k]; };
      auto qs = [&](int i, int k) { return Qs[((size_t)(s0 + i) * H + h) * d + k]; };
      auto ks = [&](int j, int k) { return Ks[((size_t)(s0 + j) * Hkv + hk) * d + k]; };
      // 1. scores and mask
      for (int i = 0; i < L; ++i)
        for (int j = 0; j < L; ++j) {
          bool ok = !cfg->causal || j <= i;
          vis[(size_t)i * L + j] = ok;
          double acc = 0.0;
          if (ok)
            for (int k = 0; k < d; ++k) acc += qs(i, k) * ks(j, k);
          x[(size_t)i * L + j] = cfg->softmax_scale * acc * LOG2E;
        }
      // 2.-4. P^, l, O
      for (int i = 0; i < L; ++i) {
        double xmax = -INFINITY;
        for (int j = 0; j < L; ++j)
          if (vis[(size_t)i * L + j]) xmax = std::max(xmax, x[(size_t)i * L + j]);
        m[i] = (int)std::ceil(xmax);
        double li = 0.0;
        for (int j = 0; j < L; ++j)
          if (vis[(size_t)i * L + j]) li += std::exp2(x[(size_t)i * L + j] - m[i]);
        if (cfg->bitexp) {
          // Inference forward with bit-level exponentials ([SUM] §3.7): in
          // each (row, 32-key block), z = y - E with E = ceil(max y - log2 448)
          // (the block's P^ exponent); keys of pairs 0-4 of every 8 pairs take
          // orc_bitexp2(z), pairs 5-7 the exact 2^z (reading of "five of every
          // eight pairs").  P^ codes come from these values and the normaliser
          // is their sum, l = sum_j p~_ij 2^(E - eV(j) - m).
          li = 0.0;
          for (int b = 0; b < L; b += 32) {
            double ymax = -INFINITY;
            for (int j = b; j < std::min(b + 32, L); ++j)
              if (vis[(size_t)i * L + j])
                ymax = std::max(ymax, x[(size_t)i * L + j] + eV[(size_t)hk * T + s0 + j]);
            const int E = (int)std::ceil(ymax - std::log2(448.0));
            for (int j = b; j < std::min(b + 32, L); ++j) {
              double& p = P[(size_t)i * L + j];
              if (!vis[(size_t)i * L + j]) { p = 0.0; continue; }
              const int ev = eV[(size_t)hk * T + s0 + j];
              const double z = x[(size_t)i * L + j] + ev - E;
              const double pt = (((j - b) / 2) % 8 < 5) ? orc_bitexp2(z) : std::exp2(z);
              li += std::ldexp(pt, E - ev - m[i]);
              const double q = cfg->quant_p ? orc_e4m3_decode(orc_e4m3_encode(pt)) : pt;
              p = std::ldexp(q, E - m[i]);
            }
          }
        }
        l[i] = li;
        for (int b = 0; !cfg->bitexp && b < L; b += 32) {
          std::vector<double*> blk;
          for (int j = b; j < std::min(b + 32, L); ++j) {
            double& p = P[(size_t)i * L + j];
            if (!vis[(size_t)i * L + j]) { p = 0.0; continue; }
            p = std::exp2(x[(size_t)i * L + j] + eV[(size_t)hk * T + s0 + j] - m[i]);
            blk.push_back(&p);
          }
          if (cfg->quant_p && !blk.empty()) quantize_block_inplace(blk, false);
        }
        if (lse2) lse2[(size_t)h * T + s0 + i] = m[i] + std::log2(li);
        for (int k = 0; k < d; ++k) {
          double acc = 0.0;
          for (int j = 0; j < L; ++j)
            if (vis[(size_t)i * L + j])
              acc += P[(size_t)i * L + j] * std::ldexp(1.0, -eV[(size_t)hk * T + s0 + j]) * vv(j, k);
          double o = acc / li;
          O[((size_t)(s0 + i) * H + h) * d + k] =
              cfg->out_round == 1 ? orc_round_bf16(o) : cfg->out_round == 2 ? (double)(float)o : o;
        }
      }
      if (!bwd) continue;
      auto dOv = [&](int i, int k) { return dO[((size_t)(s0 + i) * H + h) * d + k]; };
      // 5. D from the quantized dO and O as stored
      std::vector<double> Dl(L);
      for (int i = 0; i < L; ++i) {
        double acc = 0.0;
        for (int k = 0; k < d; ++k) acc += dOv(i, k) * O[((size_t)(s0 + i) * H + h) * d + k];
        Dl[i] = acc;
        D[(size_t)h * T + s0 + i] = acc;
      }
      // 6. dP, Pn, dS   (Pn kept in P, scaled by 2^-eV / l)
      for (int i = 0; i < L; ++i)
        for (int j = 0; j < L; ++j) {
          size_t ij = (size_t)i * L + j;
          if (!vis[ij]) { P[ij] = 0.0; dS[ij] = 0.0; continue; }
          double dp = 0.0;
          for (int k = 0; k < d; ++k) dp += dOv(i, k) * vv(j, k);
          P[ij] = P[ij] * std::ldexp(1.0, -eV[(size_t)hk * T + s0 + j]) / l[i];
          dS[ij] = P[ij] * (dp - Dl[i]);
        }
      // 7. dS^ payload(s)
      std::vector<double> dSq(dS), dSk(dS);
      if (cfg->quant_ds) {
        if (!cfg->exact) {
          for (int ib = 0; ib < L; ib += 32)
            for (int jb = 0; jb < L; jb += 32) {
              std::vector<double*> blk;
              for (int i = ib; i < std::min(ib + 32, L); ++i)
                for (int j = jb; j < std::min(jb + 32, L); ++j) blk.push_back(&dSq[(size_t)i * L + j]);
              quantize_block_inplace(blk, true);
            }
          dSk = dSq;
        } else {
          // dQ operand: per (query row, 32-key block), fold 2^eK(j)
          for (int i = 0; i < L; ++i)
            for (int jb = 0; jb < L; jb += 32) {
              std::vector<double*> blk;
              for (int j = jb; j < std::min(jb + 32, L); ++j) {
                dSq[(size_t)i * L + j] = std::ldexp(dS[(size_t)i * L + j], eK[(size_t)hk * T + s0 + j]);
                blk.push_back(&dSq[(size_t)i * L + j]);
              }
              quantize_block_inplace(blk, true);
              for (int j = jb; j < std::min(jb + 32, L); ++j)
                dSq[(size_t)i * L + j] = std::ldexp(dSq[(size_t)i * L + j], -eK[(size_t)hk * T + s0 + j]);
            }
          // dK operand: 32x32 blocks, fold 2^eQ(i)
          for (int ib = 0; ib < L; ib += 32)
            for (int jb = 0; jb < L; jb += 32) {
              std::vector<double*> blk;
              for (int i = ib; i < std::min(ib + 32, L); ++i)
                for (int j = jb; j < std::min(jb + 32, L); ++j) {
                  dSk[(size_t)i * L + j] = std::ldexp(dS[(size_t)i * L + j], eQ[(size_t)h * T + s0 + i]);
                  blk.push_back(&dSk[(size_t)i * L + j]);
                }
              quantize_block_inplace(blk, true);
              for (int i = ib; i < std::min(ib + 32, L); ++i)
                for (int j = jb; j < std::min(jb + 32, L); ++j)
                  dSk[(size_t)i * L + j] = std::ldexp(dSk[(size_t)i * L + j], -eQ[(size_t)h * T + s0 + i]);
            }
        }
      }
      // 9. P~ for dV: 32x32 blocks of Pn * 2^edO(i), fold removed
      std::vector<double> Pt(P);
      if (cfg->quant_pt) {
        for (int ib = 0; ib < L; ib += 32)
          for (int jb = 0; jb < L; jb += 32) {
            std::vector<double*> blk;
            for (int i = ib; i < std::min(ib + 32, L); ++i)
              for (int j = jb; j < std::min(jb + 32, L); ++j) {
                Pt[(size_t)i * L + j] = std::ldexp(P[(size_t)i * L + j], edO[(size_t)h * T + s0 + i]);
                blk.push_back(&Pt[(size_t)i * L + j]);
              }
            quantize_block_inplace(blk, true);
            for (int i = ib; i < std::min(ib + 32, L); ++i)
              for (int j = jb; j < std::min(jb + 32, L); ++j)
                Pt[(size_t)i * L + j] = std::ldexp(Pt[(size_t)i * L + j], -edO[(size_t)h * T + s0 + i]);
          }
      }
      // 8., 9., 10. gradients
      for (int i = 0; i < L; ++i) {
        const int p = pq[(size_t)h * T + s0 + i];
        for (int k = 0; k < d; ++k) {
          double acc = 0.0;
          if (!cfg->dq_fp16) {
            for (int j = 0; j < L; ++j) acc += dSq[(size_t)i * L + j] * kk(j, k);
          } else {
            // each 128-key tile's partial sum, scaled by 2^p and rounded to
            // FP16, is added to an FP16 accumulator (each sum rounded), in
            // the order of the key tiles
            for (int j0 = 0; j0 < L; j0 += 128) {
              double part = 0.0;
              for (int j = j0; j < std::min(j0 + 128, L); ++j) part += dSq[(size_t)i * L + j] * kk(j, k);
              acc = orc_round_f16(acc + orc_round_f16(std::ldexp(part, p)));
            }
            acc = std::ldexp(acc, -p);
          }
          dQ[((size_t)(s0 + i) * H + h) * d + k] = cfg->softmax_scale * acc;
        }
      }
      for (int j = 0; j < L; ++j)
        for (int k = 0; k < d; ++k) {
          double ak = 0.0, av = 0.0;
          for (int i = 0; i < L; ++i) {
            ak += dSk[(size_t)i * L + j] * q(i, k);
            av += Pt[(size_t)i * L + j] * dOv(i, k);
          }
          dK[((size_t)(s0 + j) * Hkv + hk) * d + k] += cfg->softmax_scale * ak;
          dV[((size_t)(s0 + j) * Hkv + hk) * d + k] += av;
        }
    }
  }
}

// Array forms of the codecs, for exhaustive tests.
void orc_e4m3_encode_array(const double* x, long n, unsigned char* out) {
  for (long i = 0; i < n; ++i) out[i] = (unsigned char)orc_e4m3_encode(x[i]);
}
void orc_e2m1_encode_array(const double* x, long n, unsigned char* out) {
  for (long i = 0; i < n; ++i) out[i] = (unsigned char)orc_e2m1_encode(x[i]);
}
void orc_noclamp_exponent_array(const double* x, long n, int* out) {
  for (long i = 0; i < n; ++i) out[i] = orc_noclamp_exponent(x[i]);
}

}  // extern "C"
