// fwd.cu — forward of the block-scaled causal attention (MXFP8 path).
//
// FLAMIA (paper summary), abstract and §3.1–§3.3; close reading 4.1 (scale
// factorisation S_ij = 2^(eQ(i)+eK(j)) * <codes>), 4.4 (warp specialisation
// after FlashAttention-4, tiles on chip, tensor cores kept busy).
//
// Persistent grid over the longest-first work list (document, 128-query tile)
// x query heads.  Warp roles:
//   warps 0-15 softmax: four warps per TMEM lane quarter; thread (warp w,
//              lane) owns query row 32(w%4)+lane of the tile (= its TMEM
//              lane) and key block w/4 of each 128-key tile.
//              Reads S from TMEM, forms y = x + eV(j) (the per-key V factor
//              folded into P along the contraction axis), quantizes P^ with
//              one no-clamp exponent per (row, 32-key block), keeps the
//              row's integer reference m and normaliser l, writes P^ codes to
//              shared memory and the block exponents (relative to m) to TMEM
//              as the A-operand scale factors of the P^V MMA.
//   warp 16    producer: TMA loads of Q, K, V code tiles (128 x d, swizzled)
//              and the per-key scale vectors of each K/V stage (mixed path:
//              also Q's and K's NVFP4 block scales, staged for tcgen05.cp).
//   warp 17    MMA issuer: S = Q^ K^T (kind::f8f6f4, or on the mixed path
//              kind::mxf4nvf4 with the block scales copied to TMEM; fp32 in
//              TMEM, double buffered) and O += P^ V^ (kind::mxf8f6f4
//              block-scaled, scale A = P^ block exponents, scale B = 1: V's
//              own scale is folded).
// The next tile's S is issued before the current tile's P^V so the tensor
// core works while the softmax warps quantize.
#include "kernels.h"
#include "attn_common.cuh"

namespace flamia {

constexpr int kFwdStages = 3;
constexpr int kFwdSoftmax = 512;
// Warpgroups 0-3 softmax, warpgroup 4: producer (warp 16), MMA issuer (17),
// two idle warps.  Registers are rebalanced after launch (640 x 96 in total):
// 4 x 128 x 104 + 128 x 64 = 61440.
constexpr int kFwdThreads = kFwdSoftmax + 128;
constexpr int kFwdWarpProd = 16, kFwdWarpMma = 17;
constexpr uint32_t kFwdRegSoftmax = 104, kFwdRegCtl = 64;
static_assert(4 * 128 * kFwdRegSoftmax + 128 * kFwdRegCtl <= kFwdThreads * 96, "register split");
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256, kColSFA0 = 384, kColSFA1 = 392, kColSFB = 400;
// mixed path: the scores' block scales, Q's per item and K's per S buffer,
// each double-buffered (8 columns a buffer: two 64-element steps at d = 128)
constexpr uint32_t kColQSF = 416, kColKSF = 432;

template <int HD, bool NV4>
struct __align__(1024) FwdTiles {
  uint8_t q[score_tile_bytes<HD, NV4>()];
  uint8_t k[kFwdStages][score_tile_bytes<HD, NV4>()];
  uint8_t v[kFwdStages][kTile * HD];
  uint8_t p[2][kTile * kTile];
  // mixed path: Q's and each K stage's block scales staged for the copy to
  // tensor memory (stage_nv_scales)
  uint32_t qsf[NV4 ? 256 : 4];
  uint32_t ksf[kFwdStages][NV4 ? 256 : 4];
};
// the tiles sit at 1024-byte boundaries (swizzled TMA destinations, MMA operands)
template <int HD, bool NV4>
constexpr bool fwd_tiles_aligned() {
  using T = FwdTiles<HD, NV4>;
  return offsetof(T, k) % 1024 == 0 && offsetof(T, v) % 1024 == 0 && offsetof(T, p) % 1024 == 0 &&
         (!NV4 || (offsetof(T, qsf) % 16 == 0 && offsetof(T, ksf) % 16 == 0));
}

struct FwdCtl {
  float kf[kFwdStages][kTile];    // 2^eK(j)
  float vf[kFwdStages][kTile];    // eV(j)
  float vinv[kFwdStages][kTile];  // 2^-eV(j)
  uint64_t q_full, q_empty;
  uint64_t k_full[kFwdStages], k_empty[kFwdStages], v_full[kFwdStages], v_empty[kFwdStages];
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2], o_full, o_free;
  uint64_t eb_bar[4], l_bar[4];  // per TMEM lane quarter: the four warps that share its rows
  int ebx[2][kTile][4];  // [tile parity][row][key block] P^ block exponents, shared by a row's four threads
  float lx[kTile][4];    // [row][key block] partial normalisers for the epilogue
  ItemRing ring;  // this CTA's work items, in the order all roles process them
  uint32_t tmem_base;
  int abort_flag;
};

template <int HD, bool NV4>
constexpr size_t fwd_smem_bytes() {
  return sizeof(FwdTiles<HD, NV4>) + sizeof(FwdCtl) + 1024;
}

// K-major operand with rows of `row_bytes` (128 or 64), swizzle = row size.
__device__ __forceinline__ uint64_t desc_kmajor(const uint8_t* tile, uint32_t byte_off, uint32_t row_bytes) {
  return smem_desc(smem_u32(tile) + byte_off, 16, 8 * row_bytes, row_bytes == 128 ? kSwz128 : kSwz64);
}
// MN-major operand: rows are K indices, `row_bytes` of M/N per row.
__device__ __forceinline__ uint64_t desc_mnmajor(const uint8_t* tile, uint32_t byte_off, uint32_t row_bytes) {
  return smem_desc(smem_u32(tile) + byte_off, 8 * row_bytes, 8 * row_bytes, row_bytes == 128 ? kSwz128 : kSwz64);
}

// 2^z by the bit-level approximation (FLAMIA summary, §3.7 Bit-Level
// Exponentials for Inference): one fused multiply-add writes 128 z + 16249
// as an integer n into the low mantissa bits of a float in [2^23, 2^24)
// (1.5 * 2^23 + 16249 = 12599161; the float's bits are 0x4B400000 + n and
// the ulp there is 1, so n is 128 z + 16249 rounded to nearest even), and a
// 16-bit shift moves n into the bf16 half of an fp32: exponent n >> 7,
// mantissa n & 127, i.e. 2^floor(z) (1 + frac z) with the fraction rounded to
// 7 bits and taken 7 units down (zero mean error).  z is first raised to
// -126.9453125, where n = 0, so n stays in [0, 17376] (z <= log2 448 in a
// P^ block) and -inf, NaN and the underflow give +0.
__device__ __forceinline__ float bitexp2(float z) {
  const float f = __fmaf_rn(fmaxf(z, -126.9453125f), 128.f, 12599161.f);
  return __uint_as_float(__float_as_uint(f) << 16);
}
// phat_values2 with the bit-level exponential: p = bitexp2(y - E).
__device__ __forceinline__ void phat_bitexp2(float y0, float y1, uint64_t nE2, float& p0, float& p1) {
  float d0, d1;
  f2_unpack(f2_add(f2_pack(y0, y1), nE2), d0, d1);
  p0 = bitexp2(d0);
  p1 = bitexp2(d1);
}

// NV4: the mixed path (scores from the NVFP4 payload: packed E2M1 tiles and
// E4M3 block scales in a block-scaled MMA; per-token fp32 factors
// g_Q(i) g_K(j) applied with the softmax scale).
// BX: the inference forward with bit-level exponentials on key pairs 0-4 of
// every 8 in a 32-key block (the other pairs keep ex2); MXFP8 default option.
template <int HD, bool OUT_BF16, bool EXACT, bool NV4, bool BX>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const AttnParams p, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_qn,
               const __grid_constant__ CUtensorMap map_kn) {
  constexpr bool PERKEY = EXACT || NV4;  // the key factor varies within a 32-key block
  constexpr int kQKBytes = score_tile_bytes<HD, NV4>();
  static_assert(fwd_tiles_aligned<HD, NV4>(), "tile alignment");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = smem_base_1k(smem_raw);
  FwdTiles<HD, NV4>& tl = *reinterpret_cast<FwdTiles<HD, NV4>*>(base);
  FwdCtl& c = *reinterpret_cast<FwdCtl*>(base + sizeof(FwdTiles<HD, NV4>));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.H / p.Hkv;
  const int n_work = p.hdr->n_items * p.H;
  volatile int* abort_flag = &c.abort_flag;
  WsHeader* hdr = p.hdr;

  if (tid == 0) {
    mbar_init(&c.q_full, NV4 ? 32 : 1);  // mixed path: every producer lane stages Q's scales
    mbar_init(&c.q_empty, 1);
    for (int s = 0; s < kFwdStages; ++s) {
      mbar_init(&c.k_full[s], 32);
      mbar_init(&c.k_empty[s], 1 + kFwdSoftmax);
      mbar_init(&c.v_full[s], 1);
      mbar_init(&c.v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c.s_full[b], 1);
      mbar_init(&c.s_free[b], kFwdSoftmax);
      mbar_init(&c.p_full[b], kFwdSoftmax);
      mbar_init(&c.p_free[b], 1);
    }
    mbar_init(&c.o_full, 1);
    mbar_init(&c.o_free, kFwdSoftmax);
    for (int qq = 0; qq < 4; ++qq) {
      mbar_init(&c.eb_bar[qq], 128);
      mbar_init(&c.l_bar[qq], 128);
    }
    item_ring_init(c.ring, 1 + kFwdSoftmax / 32);  // the MMA thread and each softmax warp
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kFwdWarpMma) tmem_alloc(&c.tmem_base, 512);
  if (warp == kFwdWarpProd && lane == 0) {
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_k);
    prefetch_tensormap(&map_v);
    if (NV4) {
      prefetch_tensormap(&map_qn);
      prefetch_tensormap(&map_kn);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = c.tmem_base;
  if (warp < 4) {  // scale factors of V in the P^V MMA: 2^0 (V's factor is folded into P)
    tmem_st4(taddr(tb, warp * 32, kColSFB), 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp >= kFwdWarpProd) {
   setmaxnreg_dec<kFwdRegCtl>();
   if (warp == kFwdWarpProd) {
    // ------------------------------------------------------------ producer
    uint32_t kv = 0, qc = 0;
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it) {
      const int w = item_publish(c.ring, n_it, &hdr->fwd_counter, n_work, lane, abort_flag, hdr, 0x204, ok, p.dbg_withhold, p.clc);
      if (w < 0) break;
      const int pair = w / p.H, h = w - pair * p.H, hk = h / G;
      const int2 it = p.fwd_items[pair];
      const int ds = __ldg(p.cu + it.x), len = __ldg(p.cu + it.x + 1) - ds;
      const int q0 = ds + kTile * it.y;
      const int n_kt = p.causal ? it.y + 1 : (len + kTile - 1) / kTile;
      if (!(ok = mbar_wait_warp(&c.q_empty, (qc & 1) ^ 1, abort_flag, hdr, 0x201))) break;
      if constexpr (NV4) stage_nv_scales<HD>(tl.qsf, p.q_bs, p.H, h, q0, p.T, lane);
      if (lane == 0) {
        mbar_arrive_expect_tx(&c.q_full, kQKBytes);
        load_score_tile<HD, NV4>(tl.q, &map_q, &map_qn, &c.q_full, h, q0);
      } else if (NV4) {
        mbar_arrive(&c.q_full);
      }
      ++qc;
      for (int kt = 0; kt < n_kt; ++kt, ++kv) {
        const int st = kv % kFwdStages;
        const uint32_t ph = (kv / kFwdStages) & 1;
        if (!(ok = mbar_wait_warp(&c.k_empty[st], ph ^ 1, abort_flag, hdr, 0x202))) break;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int j = lane * 4 + jj, key = kTile * kt + j;
          int ek = 0, ev = 0;
          float gk = 1.f;
          if (key < len) {
            ek = (int)__ldg(p.k_sc + (size_t)hk * p.T + ds + key) - 127;
            ev = (int)__ldg(p.v_sc + (size_t)hk * p.T + ds + key) - 127;
            if (NV4) gk = __ldg(p.k_g + (size_t)hk * p.T + ds + key);
          }
          c.kf[st][j] = NV4 ? gk : pow2_127(ek);
          c.vf[st][j] = (float)ev;
          c.vinv[st][j] = pow2_127(-ev);
        }
        if constexpr (NV4) stage_nv_scales<HD>(tl.ksf[st], p.k_bs, p.Hkv, hk, ds + kTile * kt, p.T, lane);
        if (lane == 0) {
          mbar_arrive_expect_tx(&c.k_full[st], kQKBytes);
          load_score_tile<HD, NV4>(tl.k[st], &map_k, &map_kn, &c.k_full[st], hk, ds + kTile * kt);
        } else {
          mbar_arrive(&c.k_full[st]);
        }
        if (!(ok = mbar_wait_warp(&c.v_empty[st], ph ^ 1, abort_flag, hdr, 0x203))) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&c.v_full[st], kTile * HD);
          tma_load_3d(tl.v[st], &map_v, &c.v_full[st], 0, hk, ds + kTile * kt);
        }
      }
    }
  } else if (warp == kFwdWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      uint32_t kv = 0, qc = 0, sc = 0, pc = 0, ic = 0;
      bool ok = true;
      for (uint32_t n_it = 0; ok; ++n_it) {
        const int w = item_get(c.ring, n_it, abort_flag, hdr, 0x217, ok);
        if (w < 0) break;
        const int pair = w / p.H;
        const int2 it = p.fwd_items[pair];
        const int len = __ldg(p.cu + it.x + 1) - __ldg(p.cu + it.x);
        const int n_kt = p.causal ? it.y + 1 : (len + kTile - 1) / kTile;
        if (!(ok = mbar_wait(&c.q_full, qc & 1, abort_flag, hdr, 0x211))) break;
        const uint32_t qsf = tb + kColQSF + 8 * (qc & 1);
        if constexpr (NV4) {
          tc_fence_after();
          copy_nv_scales<HD>(qsf, tl.qsf);
        }
        // S runs two tiles ahead of P^V: the softmax warps release S(t)'s
        // buffer a full tile before they hand over P^(t), so S(t + 2) can be
        // issued as soon as P^V(t - 1) is, and is ready a tile later.
        auto issue_s = [&](int t) -> bool {
          const uint32_t kvt = kv + t, sct = sc + t;
          const int st = kvt % kFwdStages;
          const uint32_t ph = (kvt / kFwdStages) & 1;
          const uint32_t sb = sct & 1, sph = (sct >> 1) & 1;
          if (!mbar_wait(&c.k_full[st], ph, abort_flag, hdr, 0x212)) return false;
          if (!mbar_wait(&c.s_free[sb], sph ^ 1, abort_flag, hdr, 0x213)) return false;
          tc_fence_after();
          const uint32_t ksf = tb + kColKSF + 8 * sb;
          if constexpr (NV4) copy_nv_scales<HD>(ksf, tl.ksf[st]);
          issue_scores<HD, NV4>(tb + (sb ? kColS1 : kColS0), tl.q, tl.k[st], qsf, ksf);
          tc_commit(&c.s_full[sb]);
          tc_commit(&c.k_empty[st]);
          if (t == n_kt - 1) tc_commit(&c.q_empty);
          return true;
        };
        if (!(ok = issue_s(0))) break;
        if (n_kt > 1 && !(ok = issue_s(1))) break;
        for (int j = 0; ok && j < n_kt; ++j) {
          if (j + 2 < n_kt && !(ok = issue_s(j + 2))) break;
          const uint32_t vidx = kv + j, pct = pc + j;
          const int vst = vidx % kFwdStages;
          const uint32_t vph = (vidx / kFwdStages) & 1;
          const uint32_t pb = pct & 1, pph = (pct >> 1) & 1;
          if (!(ok = mbar_wait(&c.p_full[pb], pph, abort_flag, hdr, 0x214))) break;
          if (!(ok = mbar_wait(&c.v_full[vst], vph, abort_flag, hdr, 0x215))) break;
          if (j == 0 && !(ok = mbar_wait(&c.o_free, (ic & 1) ^ 1, abort_flag, hdr, 0x216))) break;
          tc_fence_after();
          const uint32_t sfa = tb + (pb ? kColSFA1 : kColSFA0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_mxf8(tb + kColO, desc_kmajor(tl.p[pb], 32 * kk, 128), desc_mnmajor(tl.v[vst], 32 * kk * HD, HD),
                     idesc_mxf8(128, HD, 0, 1, kk, kk), sfa, tb + kColSFB, (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&c.p_free[pb]);
          tc_commit(&c.v_empty[vst]);
          if (j == n_kt - 1) tc_commit(&c.o_full);
        }
        if (!ok) break;
        kv += n_kt;
        sc += n_kt;
        pc += n_kt;
        ++qc;
        ++ic;
      }
    }
    __syncwarp();
   }
  } else {
    setmaxnreg_inc<kFwdRegSoftmax>();
    // ------------------------------------------------------------ softmax
    const int q = warp & 3, blk = warp >> 2;  // lane quarter, key block
    const int r = 32 * q + lane;              // query row of the tile = TMEM lane
    constexpr int OC = HD / 4;                // O columns handled by this thread
    uint8_t* const dbg_c = hdr->dbg_phat;
    int32_t* const dbg_e = hdr->dbg_eb;
    uint32_t kv = 0, sc = 0, pc = 0, ic = 0;
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it) {
      const int w = item_get_warp(c.ring, n_it, lane, abort_flag, hdr, 0x228, ok);
      if (w < 0) break;
      const int pair = w / p.H, h = w - pair * p.H;
      const int2 it = p.fwd_items[pair];
      const int ds = __ldg(p.cu + it.x), len = __ldg(p.cu + it.x + 1) - ds;
      const int q0 = ds + kTile * it.y;
      const int n_kt = p.causal ? it.y + 1 : (len + kTile - 1) / kTile;
      const int i_loc = kTile * it.y + r;
      const bool row_ok = i_loc < len;
      float rowc;
      if constexpr (NV4) {
        rowc = p.c_log2 * (row_ok ? __ldg(p.q_g + (size_t)h * p.T + q0 + r) : 1.f);
      } else {
        const int eq = row_ok ? (int)__ldg(p.q_sc + (size_t)h * p.T + q0 + r) - 127 : 0;
        rowc = p.c_log2 * pow2_127(eq);
      }
      int m_ref = kEmptyBlock;
      float l_run = 0.f;  // this thread's share of the normaliser (its key block)
      // Software pipeline over the key tiles: the logits, P^ codes and block
      // exponent of tile t + 1 are computed while the exponents of tile t
      // are being exchanged among the row's four threads, so the exchange
      // latency overlaps work.  Tile t uses counters kv + t, sc + t, pc + t.
      // Part A (tile t): S and the per-key vectors in, codes / Eb / partial
      // normaliser out, S buffer and key vectors released.
      auto part_a = [&](int t, uint32_t (&codes)[8], int& Eb, float& lb) -> bool {
        const uint32_t kvt = kv + t, sct = sc + t;
        const int st = kvt % kFwdStages;
        const uint32_t kph = (kvt / kFwdStages) & 1;
        const uint32_t sb = sct & 1, sph = (sct >> 1) & 1;
        if (!mbar_wait_warp(&c.k_full[st], kph, abort_flag, hdr, 0x221)) return false;
        if (!mbar_wait_warp(&c.s_full[sb], sph, abort_flag, hdr, 0x222)) return false;
        tc_fence_after();
        const int key0 = kTile * t;
        float y[32];
        const uint32_t t_s = taddr(tb, q * 32, (sb ? kColS1 : kColS0) + 32 * blk);
        const float* kfb = c.kf[st] + 32 * blk;
        const float* vfb = c.vf[st] + 32 * blk;
        // the diagonal tile (or a document's last tile) is the only one with masked keys
        if (t == n_kt - 1)
          Eb = phat_logits1<PERKEY, true>(t_s, y, rowc, kfb, vfb, i_loc, key0 + 32 * blk, len, p.causal);
        else
          Eb = phat_logits1<PERKEY, false>(t_s, y, rowc, kfb, vfb, i_loc, key0 + 32 * blk, len, p.causal);
        tc_fence_before();
        mbar_arrive(&c.s_free[sb]);
        const float* vi = c.vinv[st] + 32 * blk;
        const uint64_t nE2 = phat_neg_exp(Eb);
        uint64_t l2[2] = {0ull, 0ull};  // four partial sums, two per packed pair
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 v4 = *reinterpret_cast<const float4*>(vi + 4 * q4);
          float pv[4];  // 0 on an empty block (y = -inf)
          // key pairs 2 q4 and 2 q4 + 1 of the block; with BX the pairs
          // whose index mod 8 is below 5 take the bit-level exponential
          if (BX && (2 * q4) % 8 < 5)
            phat_bitexp2(y[4 * q4], y[4 * q4 + 1], nE2, pv[0], pv[1]);
          else
            phat_values2(y[4 * q4], y[4 * q4 + 1], nE2, pv[0], pv[1]);
          if (BX && (2 * q4 + 1) % 8 < 5)
            phat_bitexp2(y[4 * q4 + 2], y[4 * q4 + 3], nE2, pv[2], pv[3]);
          else
            phat_values2(y[4 * q4 + 2], y[4 * q4 + 3], nE2, pv[2], pv[3]);
          l2[0] = f2_fma(f2_pack(pv[0], pv[1]), f2_pack(v4.x, v4.y), l2[0]);
          l2[1] = f2_fma(f2_pack(pv[2], pv[3]), f2_pack(v4.z, v4.w), l2[1]);
          codes[q4] = pack_e4m3x4(pv[0], pv[1], pv[2], pv[3]);
        }
        mbar_arrive(&c.k_empty[st]);  // key vectors no longer read
        float l4[4];
        f2_unpack(l2[0], l4[0], l4[1]);
        f2_unpack(l2[1], l4[2], l4[3]);
        lb = (l4[0] + l4[1]) + (l4[2] + l4[3]);
        return true;
      };
      // the row's reference needs all four block exponents: each thread
      // publishes its own to the row's other three (an mbarrier per lane
      // quarter, one phase per tile, with a bounded wait)
      auto publish = [&](int t, int Eb) {
        c.ebx[(sc + t) & 1][r][blk] = Eb;
        mbar_arrive(&c.eb_bar[q]);
      };
      uint32_t codes[8], codes_n[8];
      int Eb = 0, Eb_n = 0;
      float lb = 0.f, lb_n = 0.f;
      if (!(ok = part_a(0, codes, Eb, lb))) break;
      publish(0, Eb);
      for (int kt = 0; ok && kt < n_kt; ++kt) {
        const bool more = kt + 1 < n_kt;
        if (more && !(ok = part_a(kt + 1, codes_n, Eb_n, lb_n))) break;
        const uint32_t sct = sc + kt, pct = pc + kt;
        const int par = sct & 1;
        if (!(ok = mbar_wait_warp(&c.eb_bar[q], sct & 1, abort_flag, hdr, 0x226))) break;
        const int4 e4 = *reinterpret_cast<const int4*>(c.ebx[par][r]);
        const int Eall[4] = {e4.x, e4.y, e4.z, e4.w};
        const int Emax = max(max(Eall[0], Eall[1]), max(Eall[2], Eall[3]));
        int m_new = m_ref;
        if (Emax != kEmptyBlock && (m_ref == kEmptyBlock || Emax > m_ref + 8)) m_new = Emax;
        const float lsum = (Eb != kEmptyBlock) ? ldexp_fast(lb, Eb - m_new) : 0.f;
        // the row's scale word (one byte per key block, relative to m) is
        // built and stored by the row's block-0 thread
        uint32_t word = 0;
        if (blk == 0) {
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (Eall[b] != kEmptyBlock) word |= (uint32_t)min(max(Eall[b] - m_new + 127, 0), 254) << (8 * b);
        }
        if (dbg_c != nullptr && row_ok) {
          PhatDump d;
#pragma unroll
          for (int k = 0; k < 16; ++k) d.w[k] = k < 8 ? codes[k & 7] : 0u;
          d.e[0] = Eb;
          d.e[1] = 0;
          dbg_dump_phat(dbg_c, dbg_e, p.T, h, q0 + r, ds + kTile * kt, blk, 1, d);
        }
        l_run = (m_ref == kEmptyBlock) ? lsum : ldexp_fast(l_run, m_ref - m_new) + lsum;
        // rescale this thread's quarter of the O accumulator row once the
        // previous P^V has landed (warp-uniform: tcgen05.ld/st are
        // warp-collective; lanes whose reference did not move scale by 1)
        if (__any_sync(0xffffffffu, kt > 0 && m_new != m_ref)) {
          const uint32_t pp = pct - 1;
          if (!(ok = mbar_wait_warp(&c.p_free[pp & 1], (pp >> 1) & 1, abort_flag, hdr, 0x223))) break;
          tc_fence_after();
          const float f = (m_new != m_ref) ? ldexp_fast(1.0f, m_ref - m_new) : 1.0f;
          const uint32_t t_o = taddr(tb, q * 32, kColO + blk * OC);
          if constexpr (OC == 32) {
            uint32_t rr[32];
            tmem_ld32(t_o, rr);
            tmem_ld_wait_regs(rr);
#pragma unroll
            for (int j = 0; j < 32; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * f);
            tmem_st32(t_o, rr);
          } else {
            uint32_t rr[16];
            tmem_ld16(t_o, rr);
            tmem_ld_wait_regs(rr);
#pragma unroll
            for (int j = 0; j < 16; ++j) rr[j] = __float_as_uint(__uint_as_float(rr[j]) * f);
            tmem_st16(t_o, rr);
          }
          tmem_st_wait();
        }
        m_ref = m_new;
        const uint32_t pb = pct & 1;
        if (!(ok = mbar_wait_warp(&c.p_free[pb], ((pct >> 1) & 1) ^ 1, abort_flag, hdr, 0x224))) break;
        uint8_t* prow = tl.p[pb];
        *reinterpret_cast<uint4*>(prow + sw128_off(r, 2 * blk)) = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        *reinterpret_cast<uint4*>(prow + sw128_off(r, 2 * blk + 1)) =
            make_uint4(codes[4], codes[5], codes[6], codes[7]);
        // the row's scale word goes to all four columns
        if (blk == 0) tmem_st4(taddr(tb, q * 32, pb ? kColSFA1 : kColSFA0), word, word, word, word);
        fence_proxy_async_smem();
        if (blk == 0) tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&c.p_full[pb]);
        if (more) {
          publish(kt + 1, Eb_n);
#pragma unroll
          for (int k = 0; k < 8; ++k) codes[k] = codes_n[k];
          Eb = Eb_n;
          lb = lb_n;
        }
      }
      kv += n_kt;
      sc += n_kt;
      pc += n_kt;
      if (!ok) break;
      // epilogue: O = acc / l (this thread: a quarter of the row)
      c.lx[r][blk] = l_run;
      mbar_arrive(&c.l_bar[q]);
      if (!(ok = mbar_wait_warp(&c.l_bar[q], ic & 1, abort_flag, hdr, 0x227))) break;
      const float4 l4 = *reinterpret_cast<const float4*>(c.lx[r]);
      const float l_tot = (l4.x + l4.y) + (l4.z + l4.w);
      const float inv = 1.0f / l_tot;
      if (!(ok = mbar_wait_warp(&c.o_full, ic & 1, abort_flag, hdr, 0x225))) break;
      tc_fence_after();
      uint32_t rr[OC];
      if constexpr (OC == 32) tmem_ld32(taddr(tb, q * 32, kColO + blk * OC), rr);
      else tmem_ld16(taddr(tb, q * 32, kColO + blk * OC), rr);
      tmem_ld_wait_regs(rr);
      tc_fence_before();
      mbar_arrive(&c.o_free);
      if (row_ok) {
        const size_t off = ((size_t)(q0 + r) * p.H + h) * HD + blk * OC;
        if constexpr (OUT_BF16) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.O) + off);
#pragma unroll
          for (int c8 = 0; c8 < OC / 8; ++c8) {
            uint32_t wv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(rr[8 * c8 + 2 * e]) * inv,
                                                        __uint_as_float(rr[8 * c8 + 2 * e + 1]) * inv);
              wv[e] = *reinterpret_cast<uint32_t*>(&b2);
            }
            dst[c8] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + off);
#pragma unroll
          for (int c4 = 0; c4 < OC / 4; ++c4)
            dst[c4] = make_float4(__uint_as_float(rr[4 * c4]) * inv, __uint_as_float(rr[4 * c4 + 1]) * inv,
                                  __uint_as_float(rr[4 * c4 + 2]) * inv, __uint_as_float(rr[4 * c4 + 3]) * inv);
        }
        if (blk == 0) {
          p.m[(size_t)h * p.T + q0 + r] = m_ref;
          p.l[(size_t)h * p.T + q0 + r] = l_tot;
        }
      }
      ++ic;
    }
  }
  tc_fence_before();
  __syncthreads();
  drain_after_abort(abort_flag);
  if (warp == kFwdWarpMma) tmem_dealloc(tb, 512);
}

static int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int HD, bool OB, bool EX, bool NV4, bool BX = false>
static cudaError_t launch_fwd_t(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  const size_t smem = fwd_smem_bytes<HD, NV4>();
  static_assert(fwd_smem_bytes<HD, NV4>() <= 232448, "shared memory");
  static bool attr_set[64] = {};  // per device: raised once, outside any graph capture
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  if (!attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<HD, OB, EX, NV4, BX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem_max(smem));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int grid = attn_grid((long)p.max_items * p.H, num_sms(), p.clc);
  cudaError_t e = cudaMemsetAsync(&p.hdr->fwd_counter, 0, sizeof(uint32_t), st);  // work counter of this launch
  if (e != cudaSuccess) return e;
  fwd_kernel<HD, OB, EX, NV4, BX><<<grid, kFwdThreads, attn_smem(smem, p.clc), st>>>(p, m.q, m.k, m.v, m.qn, m.kn);
  return cudaGetLastError();
}

template <int HD, bool OB, bool EX>
static cudaError_t launch_fwd_n(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  if constexpr (EX) {  // neither the mixed path nor bitexp has the exact option (the host rejects both)
    return (p.nvfp4 || p.bitexp) ? cudaErrorNotSupported : launch_fwd_t<HD, OB, EX, false>(p, m, st);
  } else {
    if (p.bitexp)  // MXFP8 only (the host rejects it on the mixed path)
      return p.nvfp4 ? cudaErrorNotSupported : launch_fwd_t<HD, OB, EX, false, true>(p, m, st);
    return p.nvfp4 ? launch_fwd_t<HD, OB, EX, true>(p, m, st) : launch_fwd_t<HD, OB, EX, false>(p, m, st);
  }
}

template <int HD, bool OB>
static cudaError_t launch_fwd_e(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  return p.exact ? launch_fwd_n<HD, OB, true>(p, m, st) : launch_fwd_n<HD, OB, false>(p, m, st);
}

cudaError_t launch_fwd(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  if (p.d == 128) return p.out_bf16 ? launch_fwd_e<128, true>(p, m, st) : launch_fwd_e<128, false>(p, m, st);
  return p.out_bf16 ? launch_fwd_e<64, true>(p, m, st) : launch_fwd_e<64, false>(p, m, st);
}

int sm_count() { return num_sms(); }

}  // namespace flamia
