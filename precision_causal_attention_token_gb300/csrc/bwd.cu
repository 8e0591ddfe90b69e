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
//   dQ  = dS K^    -> TMEM X1 (A = dS K-major, B = K MN-major), added to
//     an fp32 buffer with vector reductions by the compute warps.
// Every per-token factor that varies along a contraction (2^eQ, 2^eK, 2^edO,
// 2^-eV) is folded into the other operand before its block quantization, so
// all B operands run with unit scale factors.
#include "kernels.h"
#include "attn_common.cuh"

namespace flamia {

constexpr int kBwdThreads = 192;
constexpr uint32_t kColDV = 0, kColDK = 128, kColX0 = 256, kColX1 = 384;
constexpr uint32_t kColSfDV = kColX0 + 0, kColSfDK = kColX0 + 4, kColSfDQ = kColX0 + 8, kColSfOne = kColX0 + 12;

template <int HD>
struct __align__(1024) BwdTiles {
  uint8_t k[kTile * HD];
  uint8_t v[kTile * HD];
  uint8_t q[2][kTile * HD];
  uint8_t dO[2][kTile * HD];
  uint8_t pt[kTile * kTile];   // P~ codes   [query][key]
  uint8_t ds[kTile * kTile];   // dS^ codes  [query][key] (dQ payload; also dK's in the default option)
  uint8_t dsk[kTile * kTile];  // exact option: dK payload
};

struct BwdCtl {
  float kf[kTile];     // 2^eK(j)
  float vf[kTile];     // eV(j)
  float vinv[kTile];   // 2^-eV(j)
  int ekb[4];          // eK of each 32-key block (default option)
  uint32_t xch[2][2][4];  // [parity][dV, dK][query block]: 4 scale bytes (one per key block)
  uint64_t kv_full, kv_empty, qd_full[2], qd_empty[2];
  uint64_t s_full, dp_full, ds_full, mm_done, x1_free, acc_full, acc_free;
  uint32_t tmem_base;
  int abort_flag;
};

template <int HD>
constexpr size_t bwd_smem_bytes() {
  return sizeof(BwdTiles<HD>) + sizeof(BwdCtl) + 1024;
}

__device__ __forceinline__ uint64_t bdesc_k(const uint8_t* t, uint32_t off, uint32_t rb) {
  return smem_desc(smem_u32(t) + off, 16, 8 * rb, rb == 128 ? kSwz128 : kSwz64);
}
__device__ __forceinline__ uint64_t bdesc_mn(const uint8_t* t, uint32_t off, uint32_t rb) {
  return smem_desc(smem_u32(t) + off, 8 * rb, 8 * rb, rb == 128 ? kSwz128 : kSwz64);
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.relaxed.gpu.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d) : "memory");
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
  return v;
}

__device__ __forceinline__ uint32_t sf_byte(int e) { return (uint32_t)min(max(e + 127, 0), 254); }

template <int HD, bool OUT_BF16, bool EXACT>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const AttnParams p, const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  BwdTiles<HD>& tl = *reinterpret_cast<BwdTiles<HD>*>(base);
  BwdCtl& c = *reinterpret_cast<BwdCtl*>(base + sizeof(BwdTiles<HD>));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.H / p.Hkv;
  const int n_work = p.hdr->n_items * p.Hkv;
  volatile int* abort_flag = &c.abort_flag;
  WsHeader* hdr = p.hdr;

  if (tid == 0) {
    mbar_init(&c.kv_full, 32);
    mbar_init(&c.kv_empty, 1 + 128);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&c.qd_full[s], 1);
      mbar_init(&c.qd_empty[s], 1);
    }
    mbar_init(&c.s_full, 1);
    mbar_init(&c.dp_full, 1);
    mbar_init(&c.ds_full, 128);
    mbar_init(&c.mm_done, 1);
    mbar_init(&c.x1_free, 128);
    mbar_init(&c.acc_full, 1);
    mbar_init(&c.acc_free, 128);
    c.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) tmem_alloc(&c.tmem_base, 512);
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_k);
    prefetch_tensormap(&map_v);
    prefetch_tensormap(&map_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = c.tmem_base;

  // number of query tiles a (document, key tile) item visits, per query head
  auto q_range = [&](int kt, int len, int& q_first, int& n_t) {
    n_t = (len + kTile - 1) / kTile;
    q_first = p.causal ? kt : 0;
  };

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    uint32_t ic = 0, ii = 0;
    bool ok = true;
    for (int w = blockIdx.x; ok && w < n_work; w += gridDim.x, ++ic) {
      const int pair = w / p.Hkv, hk = w - pair * p.Hkv;
      const int2 it = p.bwd_items[pair];
      const int ds = __ldg(p.cu + it.x), len = __ldg(p.cu + it.x + 1) - ds;
      const int k0 = ds + kTile * it.y;
      int q_first, n_t;
      q_range(it.y, len, q_first, n_t);
      if (!(ok = mbar_wait(&c.kv_empty, (ic & 1) ^ 1, abort_flag, hdr, 0x301))) break;
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = lane * 4 + jj, key = kTile * it.y + j;
        int ek = 0, ev = 0;
        if (key < len) {
          ek = (int)__ldg(p.k_sc + (size_t)hk * p.T + ds + key) - 127;
          ev = (int)__ldg(p.v_sc + (size_t)hk * p.T + ds + key) - 127;
        }
        c.kf[j] = pow2_127(ek);
        c.vf[j] = (float)ev;
        c.vinv[j] = pow2_127(-ev);
        if ((j & 31) == 0) c.ekb[j >> 5] = ek;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&c.kv_full, 2 * kTile * HD);
        tma_load_3d(tl.k, &map_k, &c.kv_full, 0, hk, k0);
        tma_load_3d(tl.v, &map_v, &c.kv_full, 0, hk, k0);
      } else {
        mbar_arrive(&c.kv_full);
      }
      for (int g = 0; ok && g < G; ++g) {
        const int h = hk * G + g;
        for (int qt = q_first; qt < n_t; ++qt, ++ii) {
          const int qs = ii & 1;
          if (!(ok = mbar_wait(&c.qd_empty[qs], ((ii >> 1) & 1) ^ 1, abort_flag, hdr, 0x302))) break;
          if (lane == 0) {
            mbar_arrive_expect_tx(&c.qd_full[qs], 2 * kTile * HD);
            tma_load_3d(tl.q[qs], &map_q, &c.qd_full[qs], 0, h, ds + kTile * qt);
            tma_load_3d(tl.dO[qs], &map_do, &c.qd_full[qs], 0, h, ds + kTile * qt);
          }
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      uint32_t ic = 0, ii = 0;
      bool ok = true;
      const uint32_t id_sp = idesc_f8(128, 128, 0, 0);
      for (int w = blockIdx.x; ok && w < n_work; w += gridDim.x, ++ic) {
        const int pair = w / p.Hkv;
        const int2 it = p.bwd_items[pair];
        const int len = __ldg(p.cu + it.x + 1) - __ldg(p.cu + it.x);
        int q_first, n_t;
        q_range(it.y, len, q_first, n_t);
        const int n_iter = G * (n_t - q_first);
        if (!(ok = mbar_wait(&c.kv_full, ic & 1, abort_flag, hdr, 0x311))) break;
        for (int t = 0; ok && t < n_iter; ++t, ++ii) {
          const int qs = ii & 1;
          if (!(ok = mbar_wait(&c.qd_full[qs], (ii >> 1) & 1, abort_flag, hdr, 0x312))) break;
          // X0 still holds the previous iteration's scale factors until its MMAs finish
          if (ii > 0 && !(ok = mbar_wait(&c.mm_done, (ii - 1) & 1, abort_flag, hdr, 0x313))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 32; ++kk)
            mma_f8(tb + kColX0, bdesc_k(tl.q[qs], 32 * kk, HD), bdesc_k(tl.k, 32 * kk, HD), id_sp, kk > 0);
          tc_commit(&c.s_full);
          if (!(ok = mbar_wait(&c.x1_free, (ii & 1) ^ 1, abort_flag, hdr, 0x314))) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 32; ++kk)
            mma_f8(tb + kColX1, bdesc_k(tl.dO[qs], 32 * kk, HD), bdesc_k(tl.v, 32 * kk, HD), id_sp, kk > 0);
          tc_commit(&c.dp_full);
          if (!(ok = mbar_wait(&c.ds_full, ii & 1, abort_flag, hdr, 0x315))) break;
          if (t == 0 && !(ok = mbar_wait(&c.acc_free, (ic & 1) ^ 1, abort_flag, hdr, 0x316))) break;
          tc_fence_after();
          const uint8_t* dsk = EXACT ? tl.dsk : tl.ds;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {  // contraction over the 128 queries
            const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
            mma_mxf8(tb + kColDV, bdesc_mn(tl.pt, kk * 32 * 128, 128), bdesc_mn(tl.dO[qs], kk * 32 * HD, HD),
                     idesc_mxf8(128, HD, 1, 1, kk, kk), tb + kColSfDV, tb + kColSfOne, acc);
            mma_mxf8(tb + kColDK, bdesc_mn(dsk, kk * 32 * 128, 128), bdesc_mn(tl.q[qs], kk * 32 * HD, HD),
                     idesc_mxf8(128, HD, 1, 1, kk, kk), tb + kColSfDK, tb + kColSfOne, acc);
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // contraction over the 128 keys
            mma_mxf8(tb + kColX1, bdesc_k(tl.ds, 32 * kk, 128), bdesc_mn(tl.k, kk * 32 * HD, HD),
                     idesc_mxf8(128, HD, 0, 1, kk, kk), tb + kColSfDQ, tb + kColSfOne, kk > 0 ? 1u : 0u);
          tc_commit(&c.mm_done);
          tc_commit(&c.qd_empty[qs]);
          if (t == n_iter - 1) {
            tc_commit(&c.acc_full);
            tc_commit(&c.kv_empty);
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    const int r = tid;
    uint32_t ic = 0, ii = 0;
    bool ok = true;
    const float sm_scale = p.softmax_scale;
    for (int w = blockIdx.x; ok && w < n_work; w += gridDim.x, ++ic) {
      const int pair = w / p.Hkv, hk = w - pair * p.Hkv;
      const int2 it = p.bwd_items[pair];
      const int ds = __ldg(p.cu + it.x), len = __ldg(p.cu + it.x + 1) - ds;
      int q_first, n_t;
      q_range(it.y, len, q_first, n_t);
      if (!(ok = mbar_wait(&c.kv_full, ic & 1, abort_flag, hdr, 0x321))) break;
      const int key0 = kTile * it.y;
      for (int g = 0; ok && g < G; ++g) {
        const int h = hk * G + g;
        for (int qt = q_first; ok && qt < n_t; ++qt, ++ii) {
          const int i_loc = kTile * qt + r;
          const bool row_ok = i_loc < len;
          const size_t mt = (size_t)h * p.T + ds + i_loc;
          int eq = 0, edo = 0, mi = 0;
          float li = 1.f, Di = 0.f;
          if (row_ok) {
            eq = (int)__ldg(p.q_sc + mt) - 127;
            edo = (int)__ldg(p.do_sc + mt) - 127;
            mi = __ldg(p.m + mt);
            li = __ldg(p.l + mt);
            Di = __ldg(p.D + mt);
          }
          const float rowc = p.c_log2 * pow2_127(eq);
          const float hdo = pow2_127(edo);
          // ---- recompute P^ exactly as the forward does
          if (!(ok = mbar_wait(&c.s_full, ii & 1, abort_flag, hdr, 0x322))) break;
          tc_fence_after();
          uint32_t pcode[32];
          int Eb[4];
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t rr[32];
            tmem_ld32(taddr(tb, warp * 32, kColX0 + 32 * b), rr);
            tmem_ld_wait();
            float yv[32];
            float M = -INFINITY;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const int j = 32 * b + jj;
              yv[jj] = (row_ok && visible(i_loc, key0 + j, len, p.causal))
                           ? score_to_y(__uint_as_float(rr[jj]), rowc, c.kf[j], c.vf[j])
                           : -INFINITY;
              M = fmaxf(M, yv[jj]);
            }
            Eb[b] = (M == -INFINITY) ? kEmptyBlock : phat_block_exp(M);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              float pv[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) pv[e] = (Eb[b] == kEmptyBlock) ? 0.f : phat_value(yv[4 * q4 + e], Eb[b]);
              pcode[8 * b + q4] = pack_e4m3x4(pv[0], pv[1], pv[2], pv[3]);
            }
          }
          // ---- dS, P~ per 32-key block
          if (!(ok = mbar_wait(&c.dp_full, ii & 1, abort_flag, hdr, 0x323))) break;
          tc_fence_after();
          const float inv_l = 1.0f / li;
          uint32_t word_dq = 0;
          const int par = ii & 1;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            uint32_t rr[32];
            tmem_ld32(taddr(tb, warp * 32, kColX1 + 32 * b), rr);
            tmem_ld_wait();
            // Pn = P^ 2^-eV / l = code * 2^(Eb - m) / l * 2^-eV ; dS = Pn (dP - D)
            const float gb = (Eb[b] == kEmptyBlock) ? 0.f : ldexp_f(inv_l, Eb[b] - mi);
            float dsv[32], ptv[32];
            float amax_ds = 0.f, amax_pt = 0.f;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const uint32_t cw = pcode[8 * b + q4];
              const float2 p01 = unpack_e4m3x2((uint16_t)(cw & 0xFFFFu));
              const float2 p23 = unpack_e4m3x2((uint16_t)(cw >> 16));
              const float pd[4] = {p01.x, p01.y, p23.x, p23.y};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int jj = 4 * q4 + e, j = 32 * b + jj;
                const float pn = pd[e] * gb * c.vinv[j];
                const float dpv = __uint_as_float(rr[jj]) * hdo;  // dP * 2^-eV(j)
                const float d_s = (pd[e] * gb) * (dpv - Di * c.vinv[j]);
                dsv[jj] = row_ok ? d_s : 0.f;
                ptv[jj] = row_ok ? pn * hdo : 0.f;
                amax_ds = fmaxf(amax_ds, fabsf(dsv[jj]));
                amax_pt = fmaxf(amax_pt, ptv[jj]);
              }
            }
            // 32 x 32 block exponents (this warp's 32 queries x key block b)
            const int e_pt = noclamp_exp_clamped(warp_max(amax_pt));
            uint32_t ptc[8], dsc[8];
            if constexpr (!EXACT) {
              const int e_ds = noclamp_exp_clamped(warp_max(amax_ds));
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                ptc[q4] = pack_e4m3x4(ldexp_f(ptv[4 * q4], -e_pt), ldexp_f(ptv[4 * q4 + 1], -e_pt),
                                      ldexp_f(ptv[4 * q4 + 2], -e_pt), ldexp_f(ptv[4 * q4 + 3], -e_pt));
                dsc[q4] = pack_e4m3x4(ldexp_f(dsv[4 * q4], -e_ds), ldexp_f(dsv[4 * q4 + 1], -e_ds),
                                      ldexp_f(dsv[4 * q4 + 2], -e_ds), ldexp_f(dsv[4 * q4 + 3], -e_ds));
              }
              word_dq |= sf_byte(e_ds + c.ekb[b]) << (8 * b);
              if (lane == 0) {
                c.xch[par][0][warp] = (c.xch[par][0][warp] & ~(0xFFu << (8 * b))) | (sf_byte(e_pt) << (8 * b));
                c.xch[par][1][warp] = (c.xch[par][1][warp] & ~(0xFFu << (8 * b))) | (sf_byte(e_ds + eq) << (8 * b));
              }
            } else {
              // dQ payload: per (row, 32 keys) on dS * 2^eK(j); dK payload: 32x32 on dS * 2^eQ(i)
              float amq = 0.f;
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) amq = fmaxf(amq, fabsf(dsv[jj] * c.kf[32 * b + jj]));
              const int e_q = noclamp_exp_clamped(amq);
              const float feq = pow2_127(eq);
              const int e_k = noclamp_exp_clamped(warp_max(amax_ds * feq));
              uint32_t dkc[8];
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                float a4[4], b4[4], p4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int jj = 4 * q4 + e;
                  a4[e] = ldexp_f(dsv[jj] * c.kf[32 * b + jj], -e_q);
                  b4[e] = ldexp_f(dsv[jj] * feq, -e_k);
                  p4[e] = ldexp_f(ptv[jj], -e_pt);
                }
                dsc[q4] = pack_e4m3x4(a4[0], a4[1], a4[2], a4[3]);
                dkc[q4] = pack_e4m3x4(b4[0], b4[1], b4[2], b4[3]);
                ptc[q4] = pack_e4m3x4(p4[0], p4[1], p4[2], p4[3]);
              }
              word_dq |= sf_byte(e_q) << (8 * b);
              if (lane == 0) {
                c.xch[par][0][warp] = (c.xch[par][0][warp] & ~(0xFFu << (8 * b))) | (sf_byte(e_pt) << (8 * b));
                c.xch[par][1][warp] = (c.xch[par][1][warp] & ~(0xFFu << (8 * b))) | (sf_byte(e_k) << (8 * b));
              }
#pragma unroll
              for (int h16 = 0; h16 < 2; ++h16)
                *reinterpret_cast<uint4*>(tl.dsk + sw128_off(r, 2 * b + h16)) =
                    make_uint4(dkc[4 * h16], dkc[4 * h16 + 1], dkc[4 * h16 + 2], dkc[4 * h16 + 3]);
            }
#pragma unroll
            for (int h16 = 0; h16 < 2; ++h16) {
              *reinterpret_cast<uint4*>(tl.pt + sw128_off(r, 2 * b + h16)) =
                  make_uint4(ptc[4 * h16], ptc[4 * h16 + 1], ptc[4 * h16 + 2], ptc[4 * h16 + 3]);
              *reinterpret_cast<uint4*>(tl.ds + sw128_off(r, 2 * b + h16)) =
                  make_uint4(dsc[4 * h16], dsc[4 * h16 + 1], dsc[4 * h16 + 2], dsc[4 * h16 + 3]);
            }
          }
          // scale-factor words: dV / dK rows are keys (key block = this warp),
          // one byte per query block; dQ rows are queries (this thread's row)
          named_bar_sync(1, 128);
          uint32_t wdv = 0, wdk = 0;
#pragma unroll
          for (int qb = 0; qb < 4; ++qb) {
            wdv |= ((c.xch[par][0][qb] >> (8 * warp)) & 0xFFu) << (8 * qb);
            wdk |= ((c.xch[par][1][qb] >> (8 * warp)) & 0xFFu) << (8 * qb);
          }
          tmem_st4(taddr(tb, warp * 32, kColSfDV), wdv, wdv, wdv, wdv);
          tmem_st4(taddr(tb, warp * 32, kColSfDK), wdk, wdk, wdk, wdk);
          tmem_st4(taddr(tb, warp * 32, kColSfDQ), word_dq, word_dq, word_dq, word_dq);
          tmem_st4(taddr(tb, warp * 32, kColSfOne), 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
          fence_proxy_async_smem();
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&c.ds_full);
          // ---- dQ tile -> fp32 buffer
          if (!(ok = mbar_wait(&c.mm_done, ii & 1, abort_flag, hdr, 0x324))) break;
          tc_fence_after();
          float* dst = p.dq_acc + ((size_t)(ds + i_loc) * p.H + h) * HD;
#pragma unroll
          for (int cb = 0; cb < HD / 32; ++cb) {
            uint32_t rr[32];
            tmem_ld32(taddr(tb, warp * 32, kColX1 + 32 * cb), rr);
            tmem_ld_wait();
            if (row_ok) {
#pragma unroll
              for (int e = 0; e < 32; e += 4)
                red_add_v4(dst + 32 * cb + e, __uint_as_float(rr[e]) * sm_scale, __uint_as_float(rr[e + 1]) * sm_scale,
                           __uint_as_float(rr[e + 2]) * sm_scale, __uint_as_float(rr[e + 3]) * sm_scale);
            }
          }
          tc_fence_before();
          mbar_arrive(&c.x1_free);
        }
      }
      if (!ok) break;
      mbar_arrive(&c.kv_empty);  // key vectors no longer read
      // ---- dK, dV of this key tile (TMEM lane = key)
      if (!(ok = mbar_wait(&c.acc_full, ic & 1, abort_flag, hdr, 0x325))) break;
      tc_fence_after();
      const int j_loc = key0 + r;
      const bool key_ok = j_loc < len;
      const size_t koff = ((size_t)(ds + j_loc) * p.Hkv + hk) * HD;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const float f = which == 0 ? sm_scale : 1.0f;
        void* outp = which == 0 ? p.dK : p.dV;
        const uint32_t col = which == 0 ? kColDK : kColDV;
#pragma unroll
        for (int cb = 0; cb < HD / 32; ++cb) {
          uint32_t rr[32];
          tmem_ld32(taddr(tb, warp * 32, col + 32 * cb), rr);
          tmem_ld_wait();
          if (key_ok) {
            if constexpr (OUT_BF16) {
              uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(outp) + koff + 32 * cb);
#pragma unroll
              for (int c8 = 0; c8 < 4; ++c8) {
                uint32_t wv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(rr[8 * c8 + 2 * e]) * f,
                                                            __uint_as_float(rr[8 * c8 + 2 * e + 1]) * f);
                  wv[e] = *reinterpret_cast<uint32_t*>(&b2);
                }
                d4[c8] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
              }
            } else {
              float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(outp) + koff + 32 * cb);
#pragma unroll
              for (int c4 = 0; c4 < 8; ++c4)
                d4[c4] = make_float4(__uint_as_float(rr[4 * c4]) * f, __uint_as_float(rr[4 * c4 + 1]) * f,
                                     __uint_as_float(rr[4 * c4 + 2]) * f, __uint_as_float(rr[4 * c4 + 3]) * f);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&c.acc_free);
    }
  }
  tc_fence_before();
  __syncthreads();
  drain_after_abort(abort_flag);
  if (warp == 5) tmem_dealloc(tb, 512);
}

// dQ buffer (fp32, already scaled) -> output dtype.
template <bool OUT_BF16>
__global__ void dq_convert_kernel(const float* __restrict__ acc, void* out, size_t n4) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(acc)[i];
    if constexpr (OUT_BF16) {
      __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
      uint2 u = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
      reinterpret_cast<uint2*>(out)[i] = u;
    } else {
      reinterpret_cast<float4*>(out)[i] = v;
    }
  }
}

int sm_count();

template <int HD, bool OB, bool EX>
static cudaError_t launch_bwd_t(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  const size_t smem = bwd_smem_bytes<HD>();
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel<HD, OB, EX>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  long work = (long)p.max_items * p.Hkv;
  int grid = (int)(work < sm_count() ? work : sm_count());
  bwd_kernel<HD, OB, EX><<<grid, kBwdThreads, smem, st>>>(p, m.q, m.k, m.v, m.dO);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const AttnParams& p, const AttnMaps& m, cudaStream_t st) {
  if (p.d == 128) {
    if (p.exact) return p.out_bf16 ? launch_bwd_t<128, true, true>(p, m, st) : launch_bwd_t<128, false, true>(p, m, st);
    return p.out_bf16 ? launch_bwd_t<128, true, false>(p, m, st) : launch_bwd_t<128, false, false>(p, m, st);
  }
  if (p.exact) return p.out_bf16 ? launch_bwd_t<64, true, true>(p, m, st) : launch_bwd_t<64, false, true>(p, m, st);
  return p.out_bf16 ? launch_bwd_t<64, true, false>(p, m, st) : launch_bwd_t<64, false, false>(p, m, st);
}

cudaError_t launch_dq_convert(const AttnParams& p, cudaStream_t st) {
  const size_t n4 = (size_t)p.T * p.H * p.d / 4;
  int grid = (int)((n4 + 255) / 256);
  if (grid > sm_count() * 8) grid = sm_count() * 8;
  if (p.out_bf16) dq_convert_kernel<true><<<grid, 256, 0, st>>>(p.dq_acc, p.dQ, n4);
  else dq_convert_kernel<false><<<grid, 256, 0, st>>>(p.dq_acc, p.dQ, n4);
  return cudaGetLastError();
}

}  // namespace flamia
