// bwd.cu — backward of the block-scaled causal attention (MXFP8 path).
//
// FLAMIA (paper summary), §3.3 Forward–Backward Numerical Consistency: the
// backward recomputes the scores from the same quantized Q and K with the
// forward's tiling, diagonal decisions and exponent evaluation, forms D from
// the same quantized dO as dP, and quantizes dS with one exponent per 32x32
// block taken from the block's max-abs (so one payload serves dQ and dK).
// §4.5 / close reading 4.2: the exact option uses per-(row, 32-key) dS
// exponents for dQ.  dQ, dK and dV accumulate in fp32.
//
// Persistent grid over the longest-first list of (document, 128-key tile) x
// KV heads.  A CTA keeps dK and dV of its 128 keys in TMEM and loops over the
// query heads of the GQA group and over the query tiles that see its keys.
// Thread r of warps 0-3 owns query row r of the current query tile (= TMEM
// lane r), exactly as in the forward, so P^ is recomputed by the same code on
// the same values.  Per query tile (five MMAs):
//   S  = Q^ K^T    -> TMEM X0        (kind::f8f6f4, A = Q K-major, B = K K-major)
//   dP = dO^ V^T   -> TMEM X1
//   compute warps: P^ (recomputed), Pn = P^ 2^-eV / l, dS = Pn (dP - D),
//     dS^ (32x32 blocks), P~ (32x32 blocks of Pn 2^edO), block exponents
//     written to TMEM (in X0, free once S is read) as MMA scale factors
//   dV += P~^T dO^ (A = P~ MN-major, B = dO MN-major)   block-scaled
//   dK += dS^T Q^  (A = dS MN-major, B = Q MN-major)    block-scaled
//   dQ  = dS K^    -> TMEM X1 in two 64-column halves (A = dS K-major,
//     B = K MN-major); the drain warps stage each half in 128B-swizzled boxes
//     and the reducer warp adds them into the dQ accumulator with bulk tensor
//     reduce-adds (the addition happens in L2): fp32 partials by default, or
//     (DQ16) each row scaled by its power-of-two prescale and rounded to FP16
//     (close reading 4.4: FP16 dQ partials with a data-dependent
//     power-of-two prescale).
// Every per-token factor that varies along a contraction (2^eQ, 2^eK, 2^edO,
// 2^-eV) is folded into the other operand before its block quantization, so
// all B operands run with unit scale factors.
#include "kernels.h"
#include "attn_common.cuh"

namespace flamia {

// Compute warps 0-7 (two per TMEM lane quarter: warp w owns query rows
// 32(w%4)..+31 and key blocks 2(w/4), 2(w/4)+1).
// Warpgroups: 0-1 compute (warps 0-7), 2 dQ drain (warps 8-11, one per TMEM
// lane quarter), 3 producer (12), MMA issuer (13), dQ reducer (14), idle (15).
// Registers are rebalanced per warpgroup after launch (512 x 128 in total):
// 2 x 128 x 160 + 128 x 112 + 128 x 80 = 65536.
constexpr int kBwdCompute = 256;
constexpr int kBwdThreads = 512;
constexpr int kWarpDrain0 = 8, kWarpProd = 12, kWarpMma = 13, kWarpRed = 14;
constexpr uint32_t kRegCompute = 160, kRegDrain = 112, kRegCtl = 80;
static_assert(2 * 128 * kRegCompute + 128 * kRegDrain + 128 * kRegCtl <= 65536, "register split");
// TMEM: dV, dK accumulators; X0 = S; X1 = dP, then (once dP is read) the
// scale factors at X1 + 64.. and the dQ tile, 64 columns at a time, at X1 + 0.
// Keeping the scale factors out of X0 lets the next tile's S start as soon as
// the compute warps have read this tile's S.
constexpr uint32_t kColDV = 0, kColDK = 128, kColX0 = 256, kColX1 = 384;
constexpr uint32_t kColSfDV = kColX1 + 64, kColSfDK = kColX1 + 68, kColSfDQ = kColX1 + 72, kColSfOne = kColX1 + 76;

// NV4 (mixed path): the scores' operands are packed E2M1 codes (k holds K's,
// qn Q's) with their block scales staged in ksf / qsf; dK and dQ still
// contract with the E4M3 Q and K codes (q, k8).
// K/V tiles of consecutive work items are double-buffered so the next item's
// copies land while this one is processed (one buffer on the mixed path,
// whose extra E4M3 K tile leaves no room for a second).
template <bool NV4>
constexpr int bwd_kv_stages() {
  return NV4 ? 1 : 2;
}

template <int HD, bool EXACT, bool NV4>
struct __align__(1024) BwdTiles {
  uint8_t k[bwd_kv_stages<NV4>()][score_tile_bytes<HD, NV4>()];
  uint8_t v[bwd_kv_stages<NV4>()][kTile * HD];
  uint8_t q[2][kTile * HD];
  uint8_t dO[2][kTile * HD];
  uint8_t pt[kTile * kTile];   // P~ codes   [query][key]
  uint8_t ds[kTile * kTile];   // dS^ codes  [query][key] (dQ payload; also dK's in the default option)
  uint8_t dsk[EXACT ? kTile * kTile : 1024];  // exact option: dK payload
  // one half (64 columns) of a dQ tile staged for the bulk reduce-adds: two
  // boxes of [128 rows][32 fp32], or one of [128 rows][64 FP16] (DQ16);
  // 128B-swizzled
  uint8_t dqs[kTile * 256];
  uint8_t qn[2][NV4 ? score_tile_bytes<HD, NV4>() : 16];  // mixed path: Q's score operand
  uint32_t qsf[2][NV4 ? 256 : 4];                          // mixed path: its block scales
  uint32_t ksf[bwd_kv_stages<NV4>()][NV4 ? 256 : 4];       // and K's
  // mixed path: K's E4M3 codes for the dQ MMA.  Last, after members that
  // are whole KB on the mixed path: every tile above must stay at a
  // 1024-byte boundary (swizzled TMA destinations, MMA operands)
  uint8_t k8[NV4 ? bwd_kv_stages<NV4>() : 1][NV4 ? kTile * HD : 16];
};
// every tile's offset is a multiple of 1024 bytes on every variant used
template <int HD, bool EXACT, bool NV4>
constexpr bool bwd_tiles_aligned() {
  using T = BwdTiles<HD, EXACT, NV4>;
  return offsetof(T, q) % 1024 == 0 && offsetof(T, dO) % 1024 == 0 && offsetof(T, pt) % 1024 == 0 &&
         offsetof(T, ds) % 1024 == 0 && offsetof(T, dsk) % 1024 == 0 && offsetof(T, dqs) % 1024 == 0 &&
         offsetof(T, v) % 1024 == 0 && (!NV4 || (offsetof(T, qn) % 1024 == 0 && offsetof(T, qsf) % 1024 == 0 &&
                                                 offsetof(T, ksf) % 1024 == 0)) &&
         (!NV4 || offsetof(T, k8) % 1024 == 0);
}

// Per-row values of one query tile, staged in shared memory by the producer
// next to the tile's Q / dO codes (off the compute warps' critical path).
struct RowStage {
  float rowc, hdo, inv_l, nDp;  // nDp = -D 2^-edO
  int mi, eq;
};

struct BwdCtl {
  RowStage rows[2][kTile];  // [Q/dO stage][query row]
  float kf[2][kTile];    // [K/V stage] 2^eK(j) (mixed path: g_K(j))
  float vf[2][kTile];    // eV(j)
  float vinv[2][kTile];  // 2^-eV(j)
  int ekb[2][4];         // eK of each 32-key block (default option)
  uint8_t xch[2][2][4][4];   // [parity][dV, dK][query block][key block] scale bytes
  uint8_t xdq[2][kTile][4];  // [parity][query row][key block] dQ scale bytes
  uint64_t kv_full[2], kv_empty[2], qd_full[2], qd_empty[2];
  uint64_t s_full, dp_full, ds_full, mm_done, x1_free, acc_full, acc_free, xch_bar, dqs_full, dqs_free;
  uint64_t x0_free, dq_lo_full, dq_lo_free;
  ItemRing ring;  // this CTA's work items, in the order all roles process them
  uint32_t tmem_base;
  int abort_flag;
};

template <int HD, bool EXACT, bool NV4>
constexpr size_t bwd_smem_bytes() {
  return sizeof(BwdTiles<HD, EXACT, NV4>) + sizeof(BwdCtl) + 1024;
}

__device__ __forceinline__ uint64_t bdesc_k(const uint8_t* t, uint32_t off, uint32_t rb) {
  return smem_desc(smem_u32(t) + off, 16, 8 * rb, rb == 128 ? kSwz128 : kSwz64);
}
__device__ __forceinline__ uint64_t bdesc_mn(const uint8_t* t, uint32_t off, uint32_t rb) {
  return smem_desc(smem_u32(t) + off, 8 * rb, 8 * rb, rb == 128 ? kSwz128 : kSwz64);
}

__device__ __forceinline__ uint32_t sf_byte(int e) { return (uint32_t)min(max(e + 127, 0), 254); }

// Per-(row, key block) factor of dS and P~: with gb = 2^(Eb - m) / l (0 for
// an empty block or a row outside the document), Pn = P^ 2^-eV / l =
// code * gb * 2^-eV, so with gbh = gb 2^edO and nDp = -D 2^-edO
//   dS  = Pn (dP - D) = gbh * code * (accdP + nDp 2^-eV(j))      = gbh * w
//   P~ input = Pn 2^edO = gbh * code * 2^-eV(j)                    = gbh * u
// (the dO factor folded in).  gbh is a row constant of the block, so it is
// applied once per block: to the max-abs and to the encoding scale.
__device__ __forceinline__ float ds_gbh(int Eb_b, int mi, float inv_l, float hdo) {
  return (Eb_b == kEmptyBlock) ? 0.f : ldexp_f(inv_l, Eb_b - mi) * hdo;
}

// w and u (above) of one 32-key block of this thread's row from the dP
// accumulator values `acc` (fp32 bits), and their max-abs.
__device__ __forceinline__ void ds_block(const uint32_t (&acc)[32], const uint32_t (&pcode_b)[8], float nDp,
                                         const float* vinv_b, float (&wv)[32], float (&uv)[32], float& amax_w,
                                         float& amax_u) {
  // key pairs through the packed fp32 instructions; max |w| in two partial
  // chains of three-input max (the absolute values fold into its operands)
  float a_w[2] = {0.f, 0.f}, a_u[2] = {0.f, 0.f};
  const uint64_t nD2 = f2_pack(nDp, nDp);
#pragma unroll
  for (int q4 = 0; q4 < 8; ++q4) {
    const uint32_t cw = pcode_b[q4];
    const float2 p01 = unpack_e4m3x2((uint16_t)(cw & 0xFFFFu));
    const float2 p23 = unpack_e4m3x2((uint16_t)(cw >> 16));
    const float4 vi = *reinterpret_cast<const float4*>(vinv_b + 4 * q4);
    const uint64_t pd2[2] = {f2_pack(p01.x, p01.y), f2_pack(p23.x, p23.y)};
    const uint64_t vv2[2] = {f2_pack(vi.x, vi.y), f2_pack(vi.z, vi.w)};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int jj = 4 * q4 + 2 * h;
      const uint64_t y2 = f2_fma(nD2, vv2[h], f2_pack(__uint_as_float(acc[jj]), __uint_as_float(acc[jj + 1])));
      f2_unpack(f2_mul(pd2[h], y2), wv[jj], wv[jj + 1]);
      f2_unpack(f2_mul(pd2[h], vv2[h]), uv[jj], uv[jj + 1]);
      a_w[h] = fmax3(a_w[h], fabsf(wv[jj]), fabsf(wv[jj + 1]));
      a_u[h] = fmax3(a_u[h], uv[jj], uv[jj + 1]);
    }
  }
  amax_w = fmaxf(a_w[0], a_w[1]);
  amax_u = fmaxf(a_u[0], a_u[1]);
}

// 2^-e for a block exponent e (e <= 120 for any finite max-abs, so the
// factor is a normal fp32 and x * 2^-e is exact down to the E4M3 range).
__device__ __forceinline__ float inv_pow2(int e) { return exp2i(-min(e, 126)); }

// Codes of 32 values times s (a power of two), as 8 words of 4 E4M3 bytes.
__device__ __forceinline__ void encode32(const float (&v)[32], float s, uint32_t (&out)[8]) {
  const uint64_t s2 = f2_pack(s, s);
#pragma unroll
  for (int q4 = 0; q4 < 8; ++q4) {
    float x[4];
    f2_unpack(f2_mul(f2_pack(v[4 * q4], v[4 * q4 + 1]), s2), x[0], x[1]);
    f2_unpack(f2_mul(f2_pack(v[4 * q4 + 2], v[4 * q4 + 3]), s2), x[2], x[3]);
    out[q4] = pack_e4m3x4(x[0], x[1], x[2], x[3]);
  }
}

// Store 32 codes (keys 32b..32b+31) of row r into a 128B-swizzled [128][128] tile.
__device__ __forceinline__ void store_row_block(uint8_t* tile, int r, int b, const uint32_t (&w)[8]) {
  *reinterpret_cast<uint4*>(tile + sw128_off(r, 2 * b)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(tile + sw128_off(r, 2 * b + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
}

// Store 32 fp32 values (times f) of one row at out + off, in the output dtype.
template <bool OUT_BF16>
__device__ __forceinline__ void store_row32(void* out, size_t off, const uint32_t (&rr)[32], float f) {
  if constexpr (OUT_BF16) {
    uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + off);
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      uint32_t wv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 b2 =
            __floats2bfloat162_rn(__uint_as_float(rr[8 * c8 + 2 * e]) * f, __uint_as_float(rr[8 * c8 + 2 * e + 1]) * f);
        wv[e] = *reinterpret_cast<uint32_t*>(&b2);
      }
      d4[c8] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
  } else {
    float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(out) + off);
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4)
      d4[c4] = make_float4(__uint_as_float(rr[4 * c4]) * f, __uint_as_float(rr[4 * c4 + 1]) * f,
                           __uint_as_float(rr[4 * c4 + 2]) * f, __uint_as_float(rr[4 * c4 + 3]) * f);
  }
}

// Store 32 fp32 values of row r into one 128B-swizzled [128 rows][32 fp32] box.
__device__ __forceinline__ void store_row_box(uint8_t* box, int r, const uint32_t (&rr)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(box + sw128_off(r, c)) = make_uint4(rr[4 * c], rr[4 * c + 1], rr[4 * c + 2], rr[4 * c + 3]);
}

// 32 fp32 values times s, rounded to FP16 (RNE), as 16-byte chunks c0..c0+3
// of row r of a 128B-swizzled [128 rows][64 FP16] box.
__device__ __forceinline__ void store_row_f16(uint8_t* box, int r, int c0, const uint32_t (&rr)[32], float s) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 h2 = __floats2half2_rn(__uint_as_float(rr[8 * c + 2 * e]) * s,
                                           __uint_as_float(rr[8 * c + 2 * e + 1]) * s);
      w[e] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    *reinterpret_cast<uint4*>(box + sw128_off(r, c0 + c)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Per-row values the backward needs for query row i of head h.
struct RowVals {
  int eq, edo, mi;
  float li, Di, rowc, hdo;
};
// `tok_valid` is any token index inside the array (the loads are issued
// unconditionally, so several rows' loads can be in flight at once).
// NV4: the score's row factor is Q's per-token NVFP4 scale instead of 2^eQ.
template <bool NV4>
__device__ __forceinline__ RowVals load_row(const AttnParams& p, int h, int tok, bool row_ok, int tok_valid) {
  const size_t mt = (size_t)h * p.T + (row_ok ? tok : tok_valid);
  const int eq = (int)__ldg(p.q_sc + mt) - 127, edo = (int)__ldg(p.do_sc + mt) - 127;
  const int mi = __ldg(p.m + mt);
  const float li = __ldg(p.l + mt), Di = __ldg(p.D + mt);
  const float gq = NV4 ? __ldg(p.q_g + mt) : 1.f;
  RowVals v{0, 0, 0, 1.f, 0.f, 0.f, 1.f};
  if (row_ok) {
    v.eq = eq;
    v.edo = edo;
    v.mi = mi;
    v.li = li;
    v.Di = Di;
  }
  v.rowc = p.c_log2 * (NV4 ? (row_ok ? gq : 1.f) : pow2_127(v.eq));
  v.hdo = pow2_127(v.edo);
  return v;
}

// The dQ operand of key block b from dS = gbh * w.  Default option: one
// exponent per 32x32 block (reduced over the warp's 32 rows) and scale byte
// e + eK(block).  Exact option: one exponent per (row, 32 keys) of
// dS * 2^eK(j), scale byte e.  Returns the default option's block exponent
// (reused for dK) in e_blk.
template <bool EXACT>
__device__ __forceinline__ uint32_t dq_operand(const float (&wv)[32], float amax_w, float gbh, const float* kf_b,
                                               int ekb, uint32_t (&codes)[8], int& e_blk) {
  if constexpr (!EXACT) {
    e_blk = noclamp_exp_clamped(warp_max(amax_w * gbh));
    encode32(wv, gbh * inv_pow2(e_blk), codes);
    return sf_byte(e_blk + ekb);
  } else {
    float f[32];
    float am = 0.f;
#pragma unroll
    for (int jj = 0; jj < 32; ++jj) {
      f[jj] = wv[jj] * (gbh * kf_b[jj]);
      am = fmaxf(am, fabsf(f[jj]));
    }
    const int e = noclamp_exp_clamped(am);
    encode32(f, inv_pow2(e), codes);
    e_blk = 0;
    return sf_byte(e);
  }
}

// ============================================================================
// Backward kernel (DQ16: FP16 dQ partials): one CTA per (document, 128-key
// tile, KV head), looping over the group's query heads and tiles.  dK and dV
// accumulate in TMEM; each query tile's dQ = dS^ K^ lands in TMEM, is staged
// in shared memory by the drain warps and added to the dQ buffer by the
// reducer warp with bulk tensor reduce-adds (whole 128-byte lines, the
// addition done in L2).
// ============================================================================
template <int HD, bool OUT_BF16, bool EXACT, bool NV4, bool DQ16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const AttnParams p, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
               const __grid_constant__ CUtensorMap map_dq, const __grid_constant__ CUtensorMap map_qn,
               const __grid_constant__ CUtensorMap map_kn) {
  static_assert(bwd_tiles_aligned<HD, EXACT, NV4>(), "tile alignment");
  constexpr int kKvStages = bwd_kv_stages<NV4>();
  constexpr bool PERKEY = EXACT || NV4;
  constexpr int kQKBytes = score_tile_bytes<HD, NV4>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_base_1k(smem_raw);
  using Tiles = BwdTiles<HD, EXACT, NV4>;
  Tiles& tl = *reinterpret_cast<Tiles*>(base);
  BwdCtl& c = *reinterpret_cast<BwdCtl*>(base + sizeof(Tiles));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.H / p.Hkv;
  const int n_work = p.hdr->n_items * p.Hkv;
  volatile int* abort_flag = &c.abort_flag;
  WsHeader* hdr = p.hdr;

  if (tid == 0) {
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(&c.kv_full[s2], 32);
      mbar_init(&c.kv_empty[s2], 1 + kBwdCompute);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&c.qd_full[s], 32);
      mbar_init(&c.qd_empty[s], 1);
    }
    mbar_init(&c.s_full, 1);
    mbar_init(&c.dp_full, 1);
    mbar_init(&c.ds_full, kBwdCompute);
    mbar_init(&c.mm_done, 1);
    mbar_init(&c.x1_free, 128);     // drain warps: the dQ tile has left X1
    mbar_init(&c.x0_free, kBwdCompute);  // compute warps: S has been read
    mbar_init(&c.dq_lo_full, 1);
    mbar_init(&c.dq_lo_free, 128);
    mbar_init(&c.acc_full, 1);
    mbar_init(&c.acc_free, 128);  // the drain warpgroup stores dK / dV
    mbar_init(&c.xch_bar, kBwdCompute);
    mbar_init(&c.dqs_full, 128);
    mbar_init(&c.dqs_free, 1);
    // readers: the MMA thread, the dQ reducer, four drain and eight compute warps
    item_ring_init(c.ring, 1 + 1 + 4 + kBwdCompute / 32);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(&c.tmem_base, 512);
  if (warp == kWarpProd && lane == 0) {
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_k);
    prefetch_tensormap(&map_v);
    prefetch_tensormap(&map_do);
    prefetch_tensormap(&map_dq);
    if (NV4) {
      prefetch_tensormap(&map_qn);
      prefetch_tensormap(&map_kn);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = c.tmem_base;

  if (warp >= kWarpProd) {
   // Warpgroup 3: producer, MMA issuer, dQ reducer (and one idle warp).
   setmaxnreg_dec<kRegCtl>();
   if (warp == kWarpProd) {
    // ------------------------------------------------------------ producer
    uint32_t ic = 0, ii = 0;
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it, ++ic) {
      const int w = item_publish(c.ring, n_it, &hdr->bwd_counter, n_work, lane, abort_flag, hdr, 0x304, ok, p.dbg_withhold, p.clc);
      if (w < 0) break;
      const int pair = w / p.Hkv, hk = w - pair * p.Hkv;
      const int2 it = p.bwd_items[pair];
      const int ds = __ldg(p.cu + it.x), len = __ldg(p.cu + it.x + 1) - ds;
      const int k0 = ds + kTile * it.y;
      const int n_t = (len + kTile - 1) / kTile, q_first = p.causal ? it.y : 0;
      const int kvs = ic % kKvStages;
      if (!(ok = mbar_wait_warp(&c.kv_empty[kvs], ((ic / kKvStages) & 1) ^ 1, abort_flag, hdr, 0x301))) break;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = lane * 4 + jj, key = kTile * it.y + j;
        int ek = 0, ev = 0;
        float gk = 1.f;
        if (key < len) {
          ek = (int)__ldg(p.k_sc + (size_t)hk * p.T + ds + key) - 127;
          ev = (int)__ldg(p.v_sc + (size_t)hk * p.T + ds + key) - 127;
          if (NV4) gk = __ldg(p.k_g + (size_t)hk * p.T + ds + key);
        }
        c.kf[kvs][j] = NV4 ? gk : pow2_127(ek);
        c.vf[kvs][j] = (float)ev;
        c.vinv[kvs][j] = pow2_127(-ev);
        if ((j & 31) == 0) c.ekb[kvs][j >> 5] = ek;
      }
      if constexpr (NV4) stage_nv_scales<HD>(tl.ksf[kvs], p.k_bs, p.Hkv, hk, k0, p.T, lane);
      if (lane == 0) {
        mbar_arrive_expect_tx(&c.kv_full[kvs], kQKBytes + kTile * HD + (NV4 ? kTile * HD : 0));
        load_score_tile<HD, NV4>(tl.k[kvs], &map_k, &map_kn, &c.kv_full[kvs], hk, k0);
        tma_load_3d(tl.v[kvs], &map_v, &c.kv_full[kvs], 0, hk, k0);
        if (NV4) tma_load_3d(tl.k8[kvs], &map_k, &c.kv_full[kvs], 0, hk, k0);
      } else {
        mbar_arrive(&c.kv_full[kvs]);
      }
      for (int g = 0; ok && g < G; ++g) {
        const int h = hk * G + g;
        for (int qt = q_first; qt < n_t; ++qt, ++ii) {
          const int qs = ii & 1;
          // the per-row values are read from global memory before waiting for
          // the stage, so their latency overlaps the wait
          RowVals v[4];
#pragma unroll
          for (int rr4 = 0; rr4 < 4; ++rr4) {
            const int i_loc = kTile * qt + lane * 4 + rr4;
            v[rr4] = load_row<NV4>(p, h, ds + i_loc, i_loc < len, ds);
          }
          if (!(ok = mbar_wait_warp(&c.qd_empty[qs], ((ii >> 1) & 1) ^ 1, abort_flag, hdr, 0x302))) break;
          if constexpr (NV4) stage_nv_scales<HD>(tl.qsf[qs], p.q_bs, p.H, h, ds + kTile * qt, p.T, lane);
          if (lane == 0) {
            mbar_expect_tx(&c.qd_full[qs], 2 * kTile * HD + (NV4 ? kQKBytes : 0));
            tma_load_3d(tl.q[qs], &map_q, &c.qd_full[qs], 0, h, ds + kTile * qt);
            tma_load_3d(tl.dO[qs], &map_do, &c.qd_full[qs], 0, h, ds + kTile * qt);
            if (NV4) load_score_tile<HD, NV4>(tl.qn[qs], &map_q, &map_qn, &c.qd_full[qs], h, ds + kTile * qt);
          }
#pragma unroll
          for (int rr4 = 0; rr4 < 4; ++rr4)
            c.rows[qs][lane * 4 + rr4] = RowStage{v[rr4].rowc, v[rr4].hdo, 1.0f / v[rr4].li,
                                                  ldexp_f(-v[rr4].Di, -v[rr4].edo), v[rr4].mi, v[rr4].eq};
          mbar_arrive(&c.qd_full[qs]);
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      uint32_t ic = 0, ii = 0;
      bool ok = true;
      const uint32_t id_sp = idesc_f8(128, 128, 0, 0);
      for (uint32_t n_it = 0; ok; ++n_it, ++ic) {
        const int w = item_get(c.ring, n_it, abort_flag, hdr, 0x318, ok);
        if (w < 0) break;
        const int pair = w / p.Hkv;
        const int2 it = p.bwd_items[pair];
        const int len = __ldg(p.cu + it.x + 1) - __ldg(p.cu + it.x);
        const int n_t = (len + kTile - 1) / kTile, q_first = p.causal ? it.y : 0;
        const int n_iter = G * (n_t - q_first);
        const int kvs = ic % kKvStages;
        if (!(ok = mbar_wait(&c.kv_full[kvs], (ic / kKvStages) & 1, abort_flag, hdr, 0x311))) break;
        // S of query tile ii into X0 (Q^ of stage ii & 1, K^ of this item)
        auto issue_s = [&](uint32_t i_s) -> bool {
          const int qs_s = i_s & 1;
          if (!mbar_wait(&c.qd_full[qs_s], (i_s >> 1) & 1, abort_flag, hdr, 0x312)) return false;
          // X0 is free once the compute warps have read the previous S
          if (!mbar_wait(&c.x0_free, (i_s & 1) ^ 1, abort_flag, hdr, 0x313)) return false;
          tc_fence_after();
          if constexpr (NV4) {  // the block scales go to X1's last 16 columns (see below)
            copy_nv_scales<HD>(tb + kColX1 + 112, tl.qsf[qs_s]);
            copy_nv_scales<HD>(tb + kColX1 + 120, tl.ksf[kvs]);
          }
          issue_scores<HD, NV4>(tb + kColX0, NV4 ? tl.qn[qs_s] : tl.q[qs_s], tl.k[kvs], tb + kColX1 + 112,
                                tb + kColX1 + 120);
          tc_commit(&c.s_full);
          return true;
        };
        // dP of query tile ii into X1
        auto issue_dp = [&](uint32_t i_p) -> bool {
          // X1 is free once the previous tile's MMAs have read their scale
          // factors there and its dQ tile has been drained
          if (!mbar_wait(&c.x1_free, (i_p & 1) ^ 1, abort_flag, hdr, 0x314)) return false;
          // d = 64: the single dQ tile may drain before dV / dK have read the scale factors
          if (HD == 64 && i_p > 0 && !mbar_wait(&c.mm_done, (i_p - 1) & 1, abort_flag, hdr, 0x319)) return false;
          // mixed path: S(i_p) has read its scale factors in X1
          if (NV4 && !mbar_wait(&c.s_full, i_p & 1, abort_flag, hdr, 0x31a)) return false;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 32; ++kk)
            mma_f8(tb + kColX1, bdesc_k(tl.dO[i_p & 1], 32 * kk, HD), bdesc_k(tl.v[kvs], 32 * kk, HD), id_sp, kk > 0);
          tc_commit(&c.dp_full);
          return true;
        };
        // the first tile of the item: S and dP; later tiles' S and dP are
        // issued one tile ahead (S as soon as X0 is read, dP once X1 is free).
        // Mixed path: S's block scales sit in X1, so S(t + 1) waits until
        // dS(t) is done (dP(t) read); it is needed only after dS(t + 1)'s
        // inputs anyway, and dP(t + 1) follows the MMAs that precede it.
        if (!(ok = issue_s(ii) && issue_dp(ii))) break;
        for (int t = 0; ok && t < n_iter; ++t, ++ii) {
          const int qs = ii & 1;
          if (!NV4 && t + 1 < n_iter && !(ok = issue_s(ii + 1))) break;
          if (!(ok = mbar_wait(&c.ds_full, ii & 1, abort_flag, hdr, 0x315))) break;
          if (NV4 && t + 1 < n_iter && !(ok = issue_s(ii + 1))) break;
          if (t == 0 && !(ok = mbar_wait(&c.acc_free, (ic & 1) ^ 1, abort_flag, hdr, 0x316))) break;
          tc_fence_after();
          const uint8_t* dsk = EXACT ? tl.dsk : tl.ds;
          // dQ = dS^ K^ in halves of 64 columns through X1[0, 64); the first
          // half goes first so that its drain overlaps the dV / dK MMAs
          auto issue_dq = [&](int half) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // contraction over the 128 keys
              mma_mxf8(tb + kColX1, bdesc_k(tl.ds, 32 * kk, 128),
                       bdesc_mn(NV4 ? tl.k8[kvs] : tl.k[kvs], kk * 32 * HD + 64 * half, HD),
                       idesc_mxf8(128, 64, 0, 1, kk, kk), tb + kColSfDQ, tb + kColSfOne, kk > 0 ? 1u : 0u);
          };
          issue_dq(0);
          tc_commit(&c.dq_lo_full);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // contraction over the 128 queries
            const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
            mma_mxf8(tb + kColDV, bdesc_mn(tl.pt, kk * 32 * 128, 128), bdesc_mn(tl.dO[qs], kk * 32 * HD, HD),
                     idesc_mxf8(128, HD, 1, 1, kk, kk), tb + kColSfDV, tb + kColSfOne, acc);
            mma_mxf8(tb + kColDK, bdesc_mn(dsk, kk * 32 * 128, 128), bdesc_mn(tl.q[qs], kk * 32 * HD, HD),
                     idesc_mxf8(128, HD, 1, 1, kk, kk), tb + kColSfDK, tb + kColSfOne, acc);
          }
          if constexpr (HD == 128) {
            if (!(ok = mbar_wait(&c.dq_lo_free, ii & 1, abort_flag, hdr, 0x317))) break;
            tc_fence_after();
            issue_dq(1);
          }
          tc_commit(&c.mm_done);
          tc_commit(&c.qd_empty[qs]);
          if (t + 1 < n_iter && !(ok = issue_dp(ii + 1))) break;
          if (t == n_iter - 1) {
            tc_commit(&c.acc_full);
            tc_commit(&c.kv_empty[kvs]);
          }
        }
      }
    }
    __syncwarp();
   } else if (warp == kWarpRed) {
    // ------------------------------------------------------------ dQ reducer
    // Each staged half is added into the accumulator by bulk tensor
    // reduce-adds (rows past the document's end hold zeros; rows past T are
    // clipped by the copy).  Ordered (deterministic and exact options): the
    // partials of a (query tile, head) go in key-tile order.  A counter per
    // (query tile, head) holds how many have been added: this CTA (key tile
    // kt) waits for it to read kt (the load is issued a tile ahead, so in the
    // steady state it has long returned),
    // and sets it to kt + 1 once its adds have completed: a tile's counter
    // is released when the tile after next is staged (or at the item's end),
    // by then its adds, issued a tile earlier, have completed and the wait
    // for them costs nothing; releasing never waits on another CTA.  Every
    // wait points at a key tile with more query tiles, which the
    // longest-first list hands out earlier: no cycle.
    if (lane == 0) {
      constexpr int kHalves = HD / 64;
      uint32_t ii = 0, hc = 0;  // hc: staged halves
      bool ok = true;
      // counters of the two previous tiles, released once their adds completed
      uint32_t* pend[2] = {nullptr, nullptr};
      uint32_t pend_val[2] = {0u, 0u};
      auto release = [&](int k) {
        if (pend[k] != nullptr) {
          fence_proxy_async_global();  // the completed reduce-adds before the counter
          st_release_gpu(pend[k], pend_val[k]);
          pend[k] = nullptr;
        }
      };
      for (uint32_t n_it = 0; ok; ++n_it) {
        const int w = item_get(c.ring, n_it, abort_flag, hdr, 0x332, ok);
        if (w < 0) break;
        const int pair = w / p.Hkv, hk = w - pair * p.Hkv;
        const int2 it = p.bwd_items[pair];
        const int ds = __ldg(p.cu + it.x), len = __ldg(p.cu + it.x + 1) - ds;
        const int n_t = (len + kTile - 1) / kTile, q_first = p.causal ? it.y : 0;
        const int tile0 = p.dq_ordered ? __ldg(p.tile_prefix + it.x) : 0;
        // key tiles 0, 1, ... add in turn (causal: those <= qt; else all)
        const uint32_t want = (uint32_t)it.y;
        uint32_t seen = p.dq_ordered ? ld_acquire_gpu(p.dq_order + (size_t)(tile0 + q_first) * p.H + hk * G) : 0u;
        for (int g = 0; ok && g < G; ++g) {
          const int h = hk * G + g;
          for (int qt = q_first; ok && qt < n_t; ++qt, ++ii) {
            uint32_t* const ctr = p.dq_ordered ? p.dq_order + (size_t)(tile0 + qt) * p.H + h : nullptr;
            // one staged half (64 columns) at a time
            for (int half = 0; ok && half < kHalves; ++half, ++hc) {
              if (!(ok = mbar_wait(&c.dqs_full, hc & 1, abort_flag, hdr, 0x331))) break;
              if (p.dq_ordered && half == 0) {
                // the tile before last: every group but the last tile's has completed
                bulk_wait_group<kHalves>();
                release(0);
                if (seen != want && !(ok = counter_wait(ctr, want, abort_flag, hdr, 0x333))) break;
                fence_proxy_async_global();  // the reduce-adds below come after the acquire
              }
              if constexpr (DQ16) {
                tma_reduce_add_3d(&map_dq, tl.dqs, 64 * half, h, ds + kTile * qt);
              } else {
#pragma unroll
                for (int cb = 0; cb < 2; ++cb)
                  tma_reduce_add_3d(&map_dq, tl.dqs + cb * (kTile * 128), 64 * half + 32 * cb, h, ds + kTile * qt);
              }
              bulk_commit_group();
              bulk_wait_group_read0();
              mbar_arrive(&c.dqs_free);
            }
            if (p.dq_ordered && ok) {
              pend[0] = pend[1];
              pend_val[0] = pend_val[1];
              pend[1] = ctr;
              pend_val[1] = want + 1u;
              // the next tile's counter, read now (its value is used a tile later)
              const int qn = qt + 1 < n_t ? qt + 1 : q_first, hn = qt + 1 < n_t ? h : h + 1;
              if (qt + 1 < n_t || g + 1 < G) seen = ld_acquire_gpu(p.dq_order + (size_t)(tile0 + qn) * p.H + hn);
            }
          }
        }
        if (ok) {  // before the next item: its waits may depend on this one
          bulk_wait_group0();
          release(0);
          release(1);
        }
      }
      bulk_wait_group0();
      if (ok) {
        release(0);
        release(1);
      }
    }
    __syncwarp();
   }
  } else if (warp >= kWarpDrain0) {
    setmaxnreg_dec<kRegDrain>();
    // ------------------------------------------------------------ drain
    // Warp 8 + qq reads TMEM lane quarter qq.  Per query tile: rows
    // 32qq..32qq+31 of the finished dQ tile are staged for the reducer, 32
    // columns at a time, into the 128B-swizzled [128 rows][32 fp32] boxes.
    // Rows outside the document hold exact zeros (their dS row is zero), so
    // whole boxes are added.  Per work item: keys 32qq..32qq+31 of dK and dV
    // go to global memory, so the compute warps start the next item at once.
    const int qq = warp - kWarpDrain0, r = 32 * qq + lane;
    const float sm_scale = p.softmax_scale;
    uint32_t ic = 0, ii = 0, hc = 0;  // hc: staged dQ halves
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it, ++ic) {
      const int w = item_get_warp(c.ring, n_it, lane, abort_flag, hdr, 0x344, ok);
      if (w < 0) break;
      const int pair = w / p.Hkv, hk = w - pair * p.Hkv;
      const int2 it = p.bwd_items[pair];
      const int ds = __ldg(p.cu + it.x), len = __ldg(p.cu + it.x + 1) - ds;
      const int n_t = (len + kTile - 1) / kTile, q_first = p.causal ? it.y : 0;
      const int n_iter = G * (n_t - q_first);
      {  // the dQ tiles of this item
        const int per_g = n_t - q_first;
        for (int t = 0; ok && t < n_iter; ++t, ++ii) {
          // this iteration's query tile and head (the order of every role)
          const int g = t / per_g, qt = q_first + (t - g * per_g);
          const int i_loc = kTile * qt + r;
          // DQ16: the row's power-of-two prescale (rows past the document: zeros)
          float sp = 0.f;
          if constexpr (DQ16)
            if (i_loc < len) sp = exp2i((int)__ldg(p.pexp + (size_t)(hk * G + g) * p.T + ds + i_loc));
          // the dQ tile arrives in X1[0, 64) in halves of 64 columns (d = 128)
          // or whole (d = 64); each half is staged as FP16.  The first half is
          // committed before the dV / dK MMAs, the second with them.
#pragma unroll
          for (int half = 0; half < HD / 64; ++half) {
            if (half == 0) {  // the first (d = 64: only) half is committed on its own
              if (!(ok = mbar_wait_warp(&c.dq_lo_full, ii & 1, abort_flag, hdr, 0x343))) break;
            } else {
              if (!(ok = mbar_wait_warp(&c.mm_done, ii & 1, abort_flag, hdr, 0x341))) break;
            }
            tc_fence_after();
            uint32_t rq[2][32];  // both 32-column blocks with one wait
            tmem_ld32(taddr(tb, qq * 32, kColX1), rq[0]);
            tmem_ld32(taddr(tb, qq * 32, kColX1 + 32), rq[1]);
            tmem_ld_wait_regs(rq[0], rq[1]);
            tc_fence_before();
            if (half == 0 && HD == 128) mbar_arrive(&c.dq_lo_free);  // X1[0, 64) may take the second half
            if (half == HD / 64 - 1) mbar_arrive(&c.x1_free);         // the dQ tile has left X1
            // the staging half is free once the reducer has read the previous one
            if (!(ok = mbar_wait_warp(&c.dqs_free, (hc & 1) ^ 1, abort_flag, hdr, 0x342))) break;
            if constexpr (DQ16) {
              store_row_f16(tl.dqs, r, 0, rq[0], sp);
              store_row_f16(tl.dqs, r, 4, rq[1], sp);
            } else {
              store_row_box(tl.dqs, r, rq[0]);
              store_row_box(tl.dqs + kTile * 128, r, rq[1]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&c.dqs_full);
            ++hc;
          }
          if (!ok) break;
        }
        if (!ok) break;
      }
      // ---- dK, dV of this key tile (TMEM lane = key)
      if (!(ok = mbar_wait_warp(&c.acc_full, ic & 1, abort_flag, hdr, 0x325))) break;
      tc_fence_after();
      const int j_loc = kTile * it.y + r;
      const bool key_ok = j_loc < len;
      const size_t koff = ((size_t)(ds + j_loc) * p.Hkv + hk) * HD;
#pragma unroll 1
      for (int cc = 0; cc < 2 * (HD / 32); ++cc) {
        const int which = cc / (HD / 32), cb = cc % (HD / 32);  // which: 0 = dK, 1 = dV
        uint32_t rr[32];
        tmem_ld32(taddr(tb, qq * 32, (which == 0 ? kColDK : kColDV) + 32 * cb), rr);
        tmem_ld_wait_regs(rr);
        if (!key_ok) continue;
        if (which == 0 && p.hadamard)  // dK of the rotated Q, in fp32 until the back-rotation
          store_row32<false>(p.rot_dk, koff + 32 * cb, rr, sm_scale);
        else
          store_row32<OUT_BF16>(which == 0 ? p.dK : p.dV, koff + 32 * cb, rr, which == 0 ? sm_scale : 1.0f);
      }
      tc_fence_before();
      mbar_arrive(&c.acc_free);
    }
  } else {
    setmaxnreg_inc<kRegCompute>();
    // ------------------------------------------------------------ compute warps
    const int q = warp & 3, hf = warp >> 2;  // lane quarter (query rows), key-block half
    const int r = 32 * q + lane;             // query row of the tile = TMEM lane
    const int b0 = 2 * hf;                   // first of this thread's two key blocks
    uint8_t* const dbg_c = hdr->dbg_phat;
    int32_t* const dbg_e = hdr->dbg_eb;
    uint32_t ic = 0, ii = 0;
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it, ++ic) {
      const int w = item_get_warp(c.ring, n_it, lane, abort_flag, hdr, 0x329, ok);
      if (w < 0) break;
      const int pair = w / p.Hkv, hk = w - pair * p.Hkv;
      const int2 it = p.bwd_items[pair];
      const int ds = __ldg(p.cu + it.x), len = __ldg(p.cu + it.x + 1) - ds;
      const int n_t = (len + kTile - 1) / kTile, q_first = p.causal ? it.y : 0;
      const int kvs = ic % kKvStages;
      if (!(ok = mbar_wait_warp(&c.kv_full[kvs], (ic / kKvStages) & 1, abort_flag, hdr, 0x321))) break;
      const int key0 = kTile * it.y;
      for (int g = 0; ok && g < G; ++g) {
        const int h = hk * G + g;
        for (int qt = q_first; ok && qt < n_t; ++qt, ++ii) {
          const int i_loc = kTile * qt + r;
          const bool row_ok = i_loc < len;
          const int qs = ii & 1;
          if (!(ok = mbar_wait_warp(&c.qd_full[qs], (ii >> 1) & 1, abort_flag, hdr, 0x328))) break;
          const RowStage rv = c.rows[qs][r];
          if (!(ok = mbar_wait_warp(&c.s_full, ii & 1, abort_flag, hdr, 0x322))) break;
          tc_fence_after();
          uint32_t pcode[2][8];
          int Eb[2];
          // the diagonal tile (and a document's last key tile) needs the mask
          const bool need_mask = p.causal ? (qt == it.y) : (it.y == n_t - 1);
          // P^ of the two key blocks, one block at a time through one copy of
          // the code (as the dS blocks below)
#pragma unroll 1
          for (int bb = 0; bb < 2; ++bb) {
            const int b = b0 + bb;
            uint32_t sr[32], cw[8];
            tmem_ld32(taddr(tb, q * 32, kColX0 + 32 * b), sr);
            tmem_ld_wait_regs(sr);
            float y[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) y[j] = __uint_as_float(sr[j]);
            int e;
            if (need_mask)
              e = phat_block_logits<PERKEY, true>(y, rv.rowc, c.kf[kvs] + 32 * b, c.vf[kvs] + 32 * b, i_loc,
                                                  key0 + 32 * b, len, p.causal);
            else
              e = phat_block_logits<PERKEY, false>(y, rv.rowc, c.kf[kvs] + 32 * b, c.vf[kvs] + 32 * b, i_loc,
                                                   key0 + 32 * b, len, p.causal);
            if (!row_ok) e = kEmptyBlock;
            // rows outside the document: finite logits, zero codes
            phat_block_codes(y, row_ok ? e : kZeroCodes, cw);
            if (bb == 0) {
              Eb[0] = e;
#pragma unroll
              for (int k = 0; k < 8; ++k) pcode[0][k] = cw[k];
            } else {
              Eb[1] = e;
#pragma unroll
              for (int k = 0; k < 8; ++k) pcode[1][k] = cw[k];
            }
          }
          tc_fence_before();
          mbar_arrive(&c.x0_free);  // S has been read: X0 may take the next S
          if (dbg_c != nullptr && row_ok) {
            PhatDump d;
#pragma unroll
            for (int k = 0; k < 16; ++k) d.w[k] = pcode[k >> 3][k & 7];
            d.e[0] = Eb[0];
            d.e[1] = Eb[1];
            dbg_dump_phat(dbg_c, dbg_e, p.T, h, ds + i_loc, ds + key0, b0, 2, d);
          }
          if (!(ok = mbar_wait_warp(&c.dp_full, ii & 1, abort_flag, hdr, 0x323))) break;
          // the previous iteration's MMAs must be done with the P~ / dS tiles
          if (ii > 0 && !(ok = mbar_wait_warp(&c.mm_done, (ii - 1) & 1, abort_flag, hdr, 0x326))) break;
          tc_fence_after();
          const int par = ii & 1;
          // The two key blocks go through one copy of the block code (a loop
          // that is not unrolled): unrolled, the backward's hot loop no longer
          // fit the instruction cache.
#pragma unroll 1
          for (int bb = 0; bb < 2; ++bb) {
            const int b = b0 + bb;
            uint32_t dp[32], pc[8];
            tmem_ld32(taddr(tb, q * 32, kColX1 + 32 * b), dp);
#pragma unroll
            for (int k = 0; k < 8; ++k) pc[k] = bb ? pcode[1][k] : pcode[0][k];
            const int eb = bb ? Eb[1] : Eb[0];
            tmem_ld_wait_regs(dp);
            float wv[32], uv[32];
            float amax_w, amax_u;
            const float gbh = ds_gbh(eb, rv.mi, rv.inv_l, rv.hdo);
            ds_block(dp, pc, rv.nDp, c.vinv[kvs] + 32 * b, wv, uv, amax_w, amax_u);
            // P~: 32 x 32 block (this warp's 32 queries x key block b)
            const int e_pt = noclamp_exp_clamped(warp_max(amax_u * gbh));
            uint32_t codes[8];
            encode32(uv, gbh * inv_pow2(e_pt), codes);
            store_row_block(tl.pt, r, b, codes);
            uint32_t kbyte, qbyte = 0;
            if constexpr (!EXACT) {
              int e_ds;
              qbyte = dq_operand<false>(wv, amax_w, gbh, c.kf[kvs] + 32 * b, c.ekb[kvs][b], codes, e_ds);
              store_row_block(tl.ds, r, b, codes);
              kbyte = sf_byte(e_ds + rv.eq);  // dK operand: the same codes, Q's block exponent folded in
            } else {
              int unused;
              qbyte = dq_operand<true>(wv, amax_w, gbh, c.kf[kvs] + 32 * b, c.ekb[kvs][b], codes, unused);
              store_row_block(tl.ds, r, b, codes);
              // dK operand: 32 x 32 block of dS * 2^eQ(i)
              const float gq = gbh * pow2_127(rv.eq);
              float f[32];
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) f[jj] = wv[jj] * gq;
              const int e_k = noclamp_exp_clamped(warp_max(amax_w * gq));
              encode32(f, inv_pow2(e_k), codes);
              store_row_block(tl.dsk, r, b, codes);
              kbyte = sf_byte(e_k);
            }
            c.xdq[par][r][b] = (uint8_t)qbyte;
            if (lane == 0) {
              c.xch[par][0][q][b] = (uint8_t)sf_byte(e_pt);
              c.xch[par][1][q][b] = (uint8_t)kbyte;
            }
          }
          // exchange the block exponents among the compute warps (an mbarrier
          // with a bounded wait, so an aborting warp cannot strand the others)
          mbar_arrive(&c.xch_bar);
          if (!(ok = mbar_wait_warp(&c.xch_bar, ii & 1, abort_flag, hdr, 0x327))) break;
          if (hf == 0) {
            // dV / dK rows are keys: lane quarter q = key block q, one byte per query block
            uint32_t wdv = 0, wdk = 0;
#pragma unroll
            for (int qb = 0; qb < 4; ++qb) {
              wdv |= (uint32_t)c.xch[par][0][qb][q] << (8 * qb);
              wdk |= (uint32_t)c.xch[par][1][qb][q] << (8 * qb);
            }
            tmem_st4(taddr(tb, q * 32, kColSfDV), wdv, wdv, wdv, wdv);
            tmem_st4(taddr(tb, q * 32, kColSfDK), wdk, wdk, wdk, wdk);
          } else {
            // dQ rows are queries: this thread's row, one byte per key block
            const uint32_t wdq = *reinterpret_cast<const uint32_t*>(c.xdq[par][r]);
            tmem_st4(taddr(tb, q * 32, kColSfDQ), wdq, wdq, wdq, wdq);
            tmem_st4(taddr(tb, q * 32, kColSfOne), 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
          }
          fence_proxy_async_smem();
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&c.ds_full);
        }
      }
      if (!ok) break;
      mbar_arrive(&c.kv_empty[kvs]);  // key vectors no longer read
    }
  }
  tc_fence_before();
  __syncthreads();
  drain_after_abort(abort_flag);
  if (warp == kWarpMma) tmem_dealloc(tb, 512);
}

// The fp32 dQ accumulator (sums of dS^ K^ over key tiles) times the softmax
// scale -> output dtype.
template <bool OUT_BF16>
__global__ void dq_convert_kernel(const float* __restrict__ acc, void* out, size_t n4, float scale) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    float4 v = reinterpret_cast<const float4*>(acc)[i];
    v.x *= scale;
    v.y *= scale;
    v.z *= scale;
    v.w *= scale;
    if constexpr (OUT_BF16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
      reinterpret_cast<uint2*>(out)[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    } else {
      reinterpret_cast<float4*>(out)[i] = v;
    }
  }
}

// FP16 dQ accumulator (prescaled partial sums) -> dQ: each element times the
// softmax scale and 2^-p of its row -> output dtype.  A row of HD FP16 values
// is HD/8 lanes' 16-byte loads; a warp takes 32/(HD/8) rows at a time and two
// such groups per loop trip, so each lane keeps 32 bytes of loads in flight.
template <bool OUT_BF16, int HD>
__global__ void __launch_bounds__(256) dq16_convert_kernel(const __half* __restrict__ acc,
                                                           const int8_t* __restrict__ pexp, void* out, size_t rows,
                                                           float scale, int T, int H) {
  constexpr int LPR = HD / 8;   // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp and group
  const int lane = threadIdx.x & 31, sub = lane / LPR, col = (lane % LPR) * 8;
  const size_t warp = blockIdx.x * (size_t)(blockDim.x >> 5) + (threadIdx.x >> 5);
  const size_t stride = (size_t)gridDim.x * (blockDim.x >> 5) * RPW;
#pragma unroll 2
  for (size_t r0 = warp * RPW; r0 < rows; r0 += stride) {
    const size_t r = r0 + sub;
    if (r >= rows) continue;
    const int t = (int)(r / (size_t)H), h = (int)(r - (size_t)t * H);
    const float f = scale * pow2_127(-(int)__ldg(pexp + (size_t)h * T + t));
    const size_t o = r * HD + (size_t)col;
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(acc + o));
    const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
    float v[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&uw[k]));
      v[2 * k] = x.x * f;
      v[2 * k + 1] = x.y * f;
    }
    if constexpr (OUT_BF16) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + o) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + o);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

// Back-rotation of the gradients of rotated operands (Hadamard option):
// with Q_r = Q H_d, dL/dQ = (dL/dQ_r) H_d (H_d symmetric), likewise for K.
// One warp per row of `rows` d-vectors: the row (fp32, or FP16 with the
// row's prescale 2^-pexp when F16) times f, the fast Walsh-Hadamard transform
// in fp32, then the output dtype.  Lane l holds elements [l EPL, l EPL + EPL).
template <bool OUT_BF16, int HD, bool F16>
__global__ void __launch_bounds__(256) rot_back_kernel(const void* __restrict__ src, const int8_t* __restrict__ pexp,
                                                       void* out, size_t rows, float f, int T, int heads) {
  constexpr int EPL = HD / 32;
  const int lane = threadIdx.x & 31;
  const size_t warps = (size_t)gridDim.x * (blockDim.x >> 5);
  for (size_t r = blockIdx.x * (size_t)(blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const size_t o = r * HD + (size_t)lane * EPL;
    float v[EPL];
    float fr = f;
    if constexpr (F16) {
      const int t = (int)(r / (size_t)heads), h = (int)(r - (size_t)t * heads);
      fr = f * pow2_127(-(int)__ldg(pexp + (size_t)h * T + t));
      const __half* s16 = static_cast<const __half*>(src) + o;
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const float2 x = __half22float2(*reinterpret_cast<const __half2*>(s16 + e));
        v[e] = x.x;
        v[e + 1] = x.y;
      }
    } else {
      const float* s32 = static_cast<const float*>(src) + o;
      if constexpr (EPL == 4) {
        const float4 x = *reinterpret_cast<const float4*>(s32);
        v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(s32);
        v[0] = x.x; v[1] = x.y;
      }
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) v[e] *= fr;
#pragma unroll
    for (int h = 1; h < EPL; h <<= 1)
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        if ((e & h) == 0) {
          const float a = v[e], b = v[e + h];
          v[e] = a + b;
          v[e + h] = a - b;
        }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {  // lower lane: x + v; upper lane: x - v
      const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[e] = fmaf(sgn, v[e], __shfl_xor_sync(0xffffffffu, v[e], m));
    }
    if constexpr (OUT_BF16) {
      uint32_t w[EPL / 2];
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(v[e], v[e + 1]);
        w[e / 2] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      if constexpr (EPL == 4) *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + o) = make_uint2(w[0], w[1]);
      else *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(out) + o) = w[0];
    } else {
      if constexpr (EPL == 4) *reinterpret_cast<float4*>(static_cast<float*>(out) + o) = make_float4(v[0], v[1], v[2], v[3]);
      else *reinterpret_cast<float2*>(static_cast<float*>(out) + o) = make_float2(v[0], v[1]);
    }
  }
}

template <bool OB, int HD, bool F16>
static cudaError_t launch_rot_back(const void* src, const int8_t* pexp, void* out, size_t rows, float f, int T,
                                   int heads, int nsm, cudaStream_t st) {
  const size_t want = (rows + 7) / 8;  // eight warps a block, a row a warp
  const int blocks = (int)(want < (size_t)nsm * 8 ? (want < 1 ? 1 : want) : (size_t)nsm * 8);
  rot_back_kernel<OB, HD, F16><<<blocks, 256, 0, st>>>(src, pexp, out, rows, f, T, heads);
  return cudaGetLastError();
}

// The prescale exponent of every query row's FP16 dQ partials, pexp [H][T]:
// p_i = 15 - c0 - (edO(i) + MK + MV), clamped to [-126, 127], with MK, MV
// the largest key and value exponents over the row's document, or over keys
// j <= i (a running maximum) with the causal dQ scale.  Then every partial
// sum of 2^p_i dQ_i stays within 2^15 (close reading 4.4; FLAMIA summary §4.5).
// One CTA per (document, KV head), kPrescaleThreads threads.
constexpr int kPrescaleThreads = 1024;
__global__ void __launch_bounds__(kPrescaleThreads) dq_prescale_kernel(const AttnParams p) {
  __shared__ int s_k[kPrescaleThreads / 32], s_v[kPrescaleThreads / 32];
  __shared__ int carry_k, carry_v;
  const int doc = blockIdx.x, hk = blockIdx.y, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int s0 = __ldg(p.cu + doc), len = __ldg(p.cu + doc + 1) - s0;
  // an inconsistent cu_seqlens (reported by the plan) touches nothing here
  if (s0 < 0 || len <= 0 || s0 + len > p.T || p.hdr->n_items == 0) return;
  const int G = p.H / p.Hkv;
  const bool prefix = p.causal && p.causal_dq_scale;
  const uint8_t* ksc = p.k_sc + (size_t)hk * p.T + s0;
  const uint8_t* vsc = p.v_sc + (size_t)hk * p.T + s0;
  if (tid == 0) {
    carry_k = -1000;
    carry_v = -1000;
  }
  __syncthreads();
  if (!prefix) {  // the document's maxima
    int mk = -1000, mv = -1000;
    for (int j = tid; j < len; j += kPrescaleThreads) {
      mk = max(mk, (int)__ldg(ksc + j) - 127);
      mv = max(mv, (int)__ldg(vsc + j) - 127);
    }
    mk = __reduce_max_sync(0xffffffffu, mk);
    mv = __reduce_max_sync(0xffffffffu, mv);
    if (lane == 0) {
      atomicMax(&carry_k, mk);
      atomicMax(&carry_v, mv);
    }
    __syncthreads();
    mk = carry_k;
    mv = carry_v;
    // every token independently (no chunk barriers): the loads of all of a
    // thread's tokens and heads can be in flight together
    for (int j = tid; j < len; j += kPrescaleThreads)
      for (int g = 0; g < G; ++g) {
        const int h = hk * G + g;
        const int edo = (int)__ldg(p.do_sc + (size_t)h * p.T + s0 + j) - 127;
        const int e = 15 - p.c0 - (edo + mk + mv);
        p.pexp[(size_t)h * p.T + s0 + j] = (int8_t)(e < -126 ? -126 : (e > 127 ? 127 : e));
      }
    return;
  }
  // causal dQ scale: running maxima over keys j <= i, kPrescaleThreads tokens
  // at a time (inclusive scan in each warp, then across the warps' totals)
  for (int c = 0; c < len; c += kPrescaleThreads) {
    const int j = c + tid;
    int mk = j < len ? (int)__ldg(ksc + j) - 127 : -1000;
    int mv = j < len ? (int)__ldg(vsc + j) - 127 : -1000;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int uk = __shfl_up_sync(0xffffffffu, mk, o), uv = __shfl_up_sync(0xffffffffu, mv, o);
      if (lane >= o) {
        mk = max(mk, uk);
        mv = max(mv, uv);
      }
    }
    if (lane == 31) {
      s_k[wid] = mk;
      s_v[wid] = mv;
    }
    __syncthreads();
    if (wid == 0) {  // exclusive scan of the warps' totals, with the carry of earlier chunks
      int tk = lane < kPrescaleThreads / 32 ? s_k[lane] : -1000;
      int tv = lane < kPrescaleThreads / 32 ? s_v[lane] : -1000;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int uk = __shfl_up_sync(0xffffffffu, tk, o), uv = __shfl_up_sync(0xffffffffu, tv, o);
        if (lane >= o) {
          tk = max(tk, uk);
          tv = max(tv, uv);
        }
      }
      int ek = __shfl_up_sync(0xffffffffu, tk, 1), ev = __shfl_up_sync(0xffffffffu, tv, 1);
      if (lane == 0) ek = ev = -1000;
      const int ck = carry_k, cv = carry_v;
      __syncwarp();
      if (lane < kPrescaleThreads / 32) {
        s_k[lane] = max(ek, ck);
        s_v[lane] = max(ev, cv);
      }
      if (lane == 31) {
        carry_k = max(ck, tk);
        carry_v = max(cv, tv);
      }
    }
    __syncthreads();
    mk = max(mk, s_k[wid]);
    mv = max(mv, s_v[wid]);
    if (j < len) {
      for (int g = 0; g < G; ++g) {
        const int h = hk * G + g;
        const int edo = (int)__ldg(p.do_sc + (size_t)h * p.T + s0 + j) - 127;
        const int e = 15 - p.c0 - (edo + mk + mv);
        p.pexp[(size_t)h * p.T + s0 + j] = (int8_t)(e < -126 ? -126 : (e > 127 ? 127 : e));
      }
    }
    __syncthreads();
  }
}

int sm_count();

// Raise a kernel's dynamic shared-memory limit once per kernel (not a stream
// operation, so it is kept out of launches that may be captured in a graph).
template <auto Kernel>
static cudaError_t set_smem(size_t smem) {
  static bool done[64] = {};  // one flag per kernel and device
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (done[dev]) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  done[dev] = e == cudaSuccess;
  return e;
}

template <int HD, bool OB, bool EX, bool NV4>
static cudaError_t launch_bwd_t(const AttnParams& p_in, const AttnMaps& m, cudaStream_t st) {
  // the deterministic and exact options add the dQ partials in key-tile
  // order (fixed-order sums)
  AttnParams p = p_in;
  p.dq_ordered = (p.exact || p.deterministic) ? 1 : 0;
  const int nsm = sm_count();
  const int grid = attn_grid((long)p.max_items * p.Hkv, nsm, p.clc);
  cudaError_t e;
  const size_t smem = bwd_smem_bytes<HD, EX, NV4>();
  static_assert(bwd_smem_bytes<HD, EX, NV4>() <= 232448, "shared memory");
  const size_t n4 = (size_t)p.T * p.H * HD / 4;
  int cg = (int)((n4 + 255) / 256);
  if (cg > nsm * 8) cg = nsm * 8;
  if ((e = cudaMemsetAsync(&p.hdr->bwd_counter, 0, sizeof(uint32_t), st)) != cudaSuccess) return e;
  if (p.dq_ordered &&
      (e = cudaMemsetAsync(p.dq_order, 0, sizeof(uint32_t) * (size_t)p.max_items * p.H, st)) != cudaSuccess)
    return e;
  if (p.dq_fp16) {  // FP16 partials (never with the exact option), unordered or in key-tile order
    if ((e = set_smem<bwd_kernel<HD, OB, EX, NV4, true>>(attn_smem_max(smem))) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(p.dq16, 0, 2 * (size_t)p.T * p.H * HD, st)) != cudaSuccess) return e;
    if (p.n_seq > 0) dq_prescale_kernel<<<dim3(p.n_seq, p.Hkv), kPrescaleThreads, 0, st>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_kernel<HD, OB, EX, NV4, true><<<grid, kBwdThreads, attn_smem(smem, p.clc), st>>>(
        p, m.q, m.k, m.v, m.dO, m.dq, m.qn, m.kn);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (!NV4 && p.hadamard) {
      if ((e = launch_rot_back<OB, HD, true>(p.dq16, p.pexp, p.dQ, (size_t)p.T * p.H, p.softmax_scale, p.T, p.H,
                                             nsm, st)) != cudaSuccess)
        return e;
      return launch_rot_back<OB, HD, false>(p.rot_dk, nullptr, p.dK, (size_t)p.T * p.Hkv, 1.f, p.T, p.Hkv, nsm,
                                            st);
    }
    const size_t rows = (size_t)p.T * p.H;
    const size_t want = (rows + 8 * (32 / (HD / 8)) - 1) / (8 * (32 / (HD / 8)));  // eight warps a block
    const int blocks = (int)(want < (size_t)nsm * 16 ? (want < 1 ? 1 : want) : (size_t)nsm * 16);
    dq16_convert_kernel<OB, HD><<<blocks, 256, 0, st>>>(p.dq16, p.pexp, p.dQ, rows, p.softmax_scale, p.T, p.H);
    return cudaGetLastError();
  }
  if ((e = set_smem<bwd_kernel<HD, OB, EX, NV4, false>>(attn_smem_max(smem))) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(p.dq_acc, 0, 4 * (size_t)p.T * p.H * HD, st)) != cudaSuccess) return e;
  bwd_kernel<HD, OB, EX, NV4, false><<<grid, kBwdThreads, attn_smem(smem, p.clc), st>>>(
      p, m.q, m.k, m.v, m.dO, m.dq, m.qn, m.kn);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (!NV4 && p.hadamard) {
    if ((e = launch_rot_back<OB, HD, false>(p.dq_acc, nullptr, p.dQ, (size_t)p.T * p.H, p.softmax_scale, p.T, p.H,
                                            nsm, st)) != cudaSuccess)
      return e;
    return launch_rot_back<OB, HD, false>(p.rot_dk, nullptr, p.dK, (size_t)p.T * p.Hkv, 1.f, p.T, p.Hkv, nsm, st);
  }
  if (OB) dq_convert_kernel<true><<<cg, 256, 0, st>>>(p.dq_acc, p.dQ, n4, p.softmax_scale);
  else dq_convert_kernel<false><<<cg, 256, 0, st>>>(p.dq_acc, p.dQ, n4, p.softmax_scale);
  return cudaGetLastError();
}

template <int HD, bool OB, bool EX>
static cudaError_t launch_bwd_n(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  if constexpr (EX) {  // the exact option is not offered on the mixed path (the host rejects it)
    return p.nvfp4 ? cudaErrorNotSupported : launch_bwd_t<HD, OB, EX, false>(p, m, st);
  } else {
    return p.nvfp4 ? launch_bwd_t<HD, OB, EX, true>(p, m, st) : launch_bwd_t<HD, OB, EX, false>(p, m, st);
  }
}

template <int HD, bool OB>
static cudaError_t launch_bwd_e(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  return p.exact ? launch_bwd_n<HD, OB, true>(p, m, st) : launch_bwd_n<HD, OB, false>(p, m, st);
}

cudaError_t launch_bwd(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  if (p.d == 128) return p.out_bf16 ? launch_bwd_e<128, true>(p, m, st) : launch_bwd_e<128, false>(p, m, st);
  return p.out_bf16 ? launch_bwd_e<64, true>(p, m, st) : launch_bwd_e<64, false>(p, m, st);
}

}  // namespace flamia
