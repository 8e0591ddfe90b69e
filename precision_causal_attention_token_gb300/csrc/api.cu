// api.cu — the C ABI (include/flamia.h): host-side validation, workspace
// layout, TMA descriptors and kernel launches.  No allocation, no host
// synchronisation on the plan/quantize/fwd/bwd paths.
#include <cmath>
#include <cstddef>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <cudaTypedefs.h>

#include "kernels.h"

using namespace flamia;

namespace {

// Test hook (flamia_debug_withhold_first_item): process-wide, copied into the
// parameters of the next attention launches, cleared by flamia_plan.
std::atomic<int> g_dbg_withhold{0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

flamia_status_t validate(const flamia_problem_t* p) {
  if (!p) return FLAMIA_ERR_INVALID_ARG;
  if (p->T < 1 || p->H < 1 || p->Hkv < 1 || p->n_seq < 1 || !p->cu_seqlens) return FLAMIA_ERR_INVALID_ARG;
  if (p->H % p->Hkv != 0) return FLAMIA_ERR_INVALID_ARG;
  if (p->d != 64 && p->d != 128) return FLAMIA_ERR_UNSUPPORTED;
  if ((int64_t)p->T * p->H * p->d >= (int64_t)1 << 40) return FLAMIA_ERR_UNSUPPORTED;
  if (p->T > (1 << 30) || p->n_seq > p->T + 1) return FLAMIA_ERR_INVALID_ARG;
  if (p->path != FLAMIA_PATH_MXFP8 && p->path != FLAMIA_PATH_NVFP4_FP8) return FLAMIA_ERR_UNSUPPORTED;
  if (p->path == FLAMIA_PATH_NVFP4_FP8 && p->exact) return FLAMIA_ERR_UNSUPPORTED;
  if (p->bitexp && (p->path != FLAMIA_PATH_MXFP8 || p->exact)) return FLAMIA_ERR_UNSUPPORTED;
  if (p->hadamard && p->path != FLAMIA_PATH_MXFP8) return FLAMIA_ERR_UNSUPPORTED;
  // cluster launch control: not with the ordered dQ reduction (its waits need
  // the items taken in list order); the grid (a CTA per item) must fit in x
  if (p->clc && (p->exact || p->deterministic)) return FLAMIA_ERR_UNSUPPORTED;
  if (p->clc && ((int64_t)(p->T + 127) / 128 + p->n_seq) * p->H > INT32_MAX) return FLAMIA_ERR_UNSUPPORTED;
  if ((p->in_dtype != FLAMIA_F32 && p->in_dtype != FLAMIA_BF16) ||
      (p->out_dtype != FLAMIA_F32 && p->out_dtype != FLAMIA_BF16))
    return FLAMIA_ERR_UNSUPPORTED;
  if (!(p->softmax_scale >= 0.f) || std::isinf(p->softmax_scale)) return FLAMIA_ERR_INVALID_ARG;
  if (!aligned16(p->cu_seqlens) && (reinterpret_cast<uintptr_t>(p->cu_seqlens) & 3u)) return FLAMIA_ERR_INVALID_ARG;
  return FLAMIA_OK;
}

flamia_status_t check_ws(const flamia_problem_t* p, void* ws, size_t ws_bytes, WsLayout* L) {
  *L = ws_layout(*p);
  if (!ws || !aligned16(ws)) return FLAMIA_ERR_INVALID_ARG;
  if (ws_bytes < L->total) return FLAMIA_ERR_WORKSPACE_TOO_SMALL;
  return FLAMIA_OK;
}

// The scale the kernels apply to the scores: with the Hadamard rotation the
// rotated dot products are d times the originals (H_d H_d = d I), so 1/d
// (a power of two) joins the softmax scale.
float softmax_scale_of(const flamia_problem_t* p) {
  const float s = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / std::sqrt((float)p->d);
  return p->hadamard ? s / (float)p->d : s;
}

// The constant of the FP16 dQ prescale: c0 = ceil(log2(2.5 d 448^3 scale)),
// so that |dQ_i| <= 2^(c0 + edO(i) + max eK + max eV) (close reading, 4.4: a
// data-dependent power-of-two prescale of the FP16 dQ partials).  frexp keeps
// it exact: x = f 2^e with f in [0.5, 1), ceil(log2 x) = e unless f = 0.5.
int dq_prescale_c0(int d, float scale) {
  int e = 0;
  const double f = std::frexp(2.5 * d * 448.0 * 448.0 * 448.0 * (double)scale, &e);
  return f > 0.5 ? e : e - 1;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 3-D map over E4M3 codes [T][heads][d]: box = 128 tokens x 1 head x d bytes,
// swizzle = d bytes (128B or 64B), out-of-range rows read as zero.
bool make_codes_map(CUtensorMap* m, const void* ptr, int d, int heads, int T) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)heads * d};
  cuuint32_t box[3] = {(cuuint32_t)d, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   d == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over the dQ accumulator [T][heads][d], the target of bulk
// reduce-adds: box = 128 tokens x 1 head x 128 bytes of values (32 fp32, or
// 64 FP16 with dq_fp16), 128B swizzle.
bool make_dq_map(CUtensorMap* m, void* ptr, int d, int heads, int T, bool fp16) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t es = fp16 ? 2 : 4;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)d * es, (cuuint64_t)heads * d * es};
  cuuint32_t box[3] = {fp16 ? 64u : 32u, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims,
                   strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D map over the mixed path's packed E2M1 codes [T][heads][d/2]: box = 128
// tokens x 1 head x d/2 bytes, swizzle = d/2 bytes (64B or 32B), out-of-range
// rows read as zero.
bool make_nv_map(CUtensorMap* m, const void* ptr, int d, int heads, int T) {
  auto enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t rb = (cuuint64_t)d / 2;
  cuuint64_t dims[3] = {rb, (cuuint64_t)heads, (cuuint64_t)T};
  cuuint64_t strides[2] = {rb, (cuuint64_t)heads * rb};
  cuuint32_t box[3] = {(cuuint32_t)rb, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE,
                   d == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Null members of the NVFP4 payload are allowed here (the MXFP8 path does
// not use them); every pointer given must be 16-byte aligned.
bool operand_ok(const flamia_operand_t* o) {
  return o && o->codes && o->scales && aligned16(o->codes) && aligned16(o->scales) && aligned16(o->codes4) &&
         aligned16(o->scales4) && aligned16(o->gscale4);
}

}  // namespace

extern "C" {

size_t flamia_workspace_size(const flamia_problem_t* p) {
  if (validate(p) != FLAMIA_OK) return 0;
  return ws_layout(*p).total;
}

const char* flamia_status_string(flamia_status_t s) {
  switch (s) {
    case FLAMIA_OK: return "ok";
    case FLAMIA_ERR_INVALID_ARG: return "invalid argument";
    case FLAMIA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FLAMIA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FLAMIA_ERR_CUDA: return "CUDA launch error";
    case FLAMIA_ERR_TIMEOUT: return "device wait timed out";
    case FLAMIA_ERR_BAD_SEQLENS: return "cu_seqlens inconsistent with T";
  }
  return "unknown status";
}

flamia_status_t flamia_plan(const flamia_problem_t* p, void* ws, size_t ws_bytes, cudaStream_t stream) {
  flamia_status_t s = validate(p);
  if (s != FLAMIA_OK) return s;
  WsLayout L;
  if ((s = check_ws(p, ws, ws_bytes, &L)) != FLAMIA_OK) return s;
  g_dbg_withhold.store(0);
  return launch_plan(*p, L, static_cast<uint8_t*>(ws), stream) == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

flamia_status_t flamia_quantize(const flamia_problem_t* p, int32_t role, const void* const* in, const void* O,
                                const flamia_operand_t* out, float* D, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  flamia_status_t s = validate(p);
  if (s != FLAMIA_OK) return s;
  WsLayout L;
  if ((s = check_ws(p, ws, ws_bytes, &L)) != FLAMIA_OK) return s;
  if (!in || !out) return FLAMIA_ERR_INVALID_ARG;
  uint8_t* w = static_cast<uint8_t*>(ws);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(w + L.header);
  const int32_t* blk = reinterpret_cast<const int32_t*>(w + L.blk32_prefix);
  const int max_blk = (p->T + 31) / 32 + p->n_seq;
  const int in_bf16 = p->in_dtype == FLAMIA_BF16, o_bf16 = p->out_dtype == FLAMIA_BF16;
  if (role == FLAMIA_ROLE_QKV) {
    for (int i = 0; i < 3; ++i) {
      if (!in[i] || !aligned16(in[i]) || !operand_ok(&out[i])) return FLAMIA_ERR_INVALID_ARG;
    }
    const bool nv = p->path == FLAMIA_PATH_NVFP4_FP8;
    QuantBatch qb{};
    qb.n = 3;
    int units = 0;
    for (int i = 0; i < 3; ++i) {
      QuantArgs& a = qb.a[i];
      a.x = in[i];
      a.codes = static_cast<uint8_t*>(out[i].codes);
      a.scales = static_cast<uint8_t*>(out[i].scales);
      a.heads = i == 0 ? p->H : p->Hkv;
      a.T = p->T;
      a.per_token = (i == 2 || p->exact) ? 1 : 0;
      a.rotate = (i < 2 && p->hadamard) ? 1 : 0;
      if (nv && i < 2) {
        if (!out[i].codes4 || !out[i].scales4 || !out[i].gscale4) return FLAMIA_ERR_INVALID_ARG;
        a.codes4 = static_cast<uint8_t*>(out[i].codes4);
        a.scales4 = static_cast<uint8_t*>(out[i].scales4);
        a.gscale4 = static_cast<float*>(out[i].gscale4);
      }
      units += max_blk * a.heads;
    }
    return launch_quantize(qb, p->d, in_bf16, o_bf16, false, nv, p->cu_seqlens, blk, p->n_seq, hdr, units,
                           sm_count(), stream) == cudaSuccess
               ? FLAMIA_OK
               : FLAMIA_ERR_CUDA;
  }
  if (role == FLAMIA_ROLE_DO) {
    if (!in[0] || !aligned16(in[0]) || !O || !aligned16(O) || !D || !aligned16(D) || !operand_ok(&out[0]))
      return FLAMIA_ERR_INVALID_ARG;
    QuantBatch qb{};
    qb.n = 1;
    QuantArgs& a = qb.a[0];
    a.x = in[0];
    a.codes = static_cast<uint8_t*>(out[0].codes);
    a.scales = static_cast<uint8_t*>(out[0].scales);
    a.O = O;
    a.D = D;
    a.heads = p->H;
    a.T = p->T;
    a.per_token = p->exact ? 1 : 0;
    return launch_quantize(qb, p->d, in_bf16, o_bf16, true, false, p->cu_seqlens, blk, p->n_seq, hdr,
                           max_blk * p->H, sm_count(), stream) == cudaSuccess
               ? FLAMIA_OK
               : FLAMIA_ERR_CUDA;
  }
  return FLAMIA_ERR_INVALID_ARG;
}

static flamia_status_t fill_params(const flamia_problem_t* p, const WsLayout& L, void* ws, AttnParams* a) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  std::memset(a, 0, sizeof(*a));
  a->T = p->T; a->H = p->H; a->Hkv = p->Hkv; a->d = p->d; a->n_seq = p->n_seq;
  a->causal = p->causal ? 1 : 0;
  a->exact = p->exact ? 1 : 0;
  a->deterministic = p->deterministic ? 1 : 0;
  a->out_bf16 = p->out_dtype == FLAMIA_BF16;
  a->max_items = L.max_items;
  a->softmax_scale = softmax_scale_of(p);
  a->c_log2 = (float)((double)a->softmax_scale * 1.4426950408889634);
  a->cu = p->cu_seqlens;
  a->tile_prefix = reinterpret_cast<const int32_t*>(w + L.tile_prefix);
  a->fwd_items = reinterpret_cast<const int2*>(w + L.fwd_items);
  a->bwd_items = reinterpret_cast<const int2*>(w + L.bwd_items);
  a->hdr = reinterpret_cast<WsHeader*>(w + L.header);
  a->dq_acc = reinterpret_cast<float*>(w + L.dq_acc);
  a->dq16 = reinterpret_cast<__half*>(w + L.dq_acc);
  // FP16 partials: the default option, unordered or (deterministic) in
  // key-tile order; the exact option adds fp32 partials in key-tile order
  a->dq_fp16 = (p->dq_fp16 && !p->exact) ? 1 : 0;
  a->pexp = reinterpret_cast<int8_t*>(w + L.pexp);
  a->c0 = dq_prescale_c0(p->d, a->softmax_scale);
  a->causal_dq_scale = p->causal_dq_scale ? 1 : 0;
  a->nvfp4 = p->path == FLAMIA_PATH_NVFP4_FP8 ? 1 : 0;
  a->bitexp = p->bitexp ? 1 : 0;
  a->hadamard = p->hadamard ? 1 : 0;
  a->rot_dk = p->hadamard ? reinterpret_cast<float*>(w + L.rot_dk) : nullptr;
  a->dq_order = reinterpret_cast<uint32_t*>(w + L.dq_order);
  a->clc = p->clc ? 1 : 0;
  a->dbg_withhold = g_dbg_withhold.load();
  return FLAMIA_OK;
}

flamia_status_t flamia_fwd(const flamia_problem_t* p, const flamia_operand_t* q, const flamia_operand_t* k,
                           const flamia_operand_t* v, void* O, int32_t* m, float* l, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  flamia_status_t s = validate(p);
  if (s != FLAMIA_OK) return s;
  WsLayout L;
  if ((s = check_ws(p, ws, ws_bytes, &L)) != FLAMIA_OK) return s;
  if (!operand_ok(q) || !operand_ok(k) || !operand_ok(v) || !O || !aligned16(O) || !m || !aligned16(m) || !l ||
      !aligned16(l))
    return FLAMIA_ERR_INVALID_ARG;
  if (p->path == FLAMIA_PATH_NVFP4_FP8 && (!q->codes4 || !q->scales4 || !q->gscale4 || !k->codes4 ||
                                           !k->scales4 || !k->gscale4))
    return FLAMIA_ERR_INVALID_ARG;
  AttnParams a;
  fill_params(p, L, ws, &a);
  a.q_sc = static_cast<const uint8_t*>(q->scales);
  a.k_sc = static_cast<const uint8_t*>(k->scales);
  a.v_sc = static_cast<const uint8_t*>(v->scales);
  a.O = O; a.m = m; a.l = l;
  AttnMaps maps;
  if (!make_codes_map(&maps.q, q->codes, p->d, p->H, p->T) || !make_codes_map(&maps.k, k->codes, p->d, p->Hkv, p->T) ||
      !make_codes_map(&maps.v, v->codes, p->d, p->Hkv, p->T))
    return FLAMIA_ERR_CUDA;
  maps.dO = maps.q;
  maps.dq = maps.q;
  maps.qn = maps.q;
  maps.kn = maps.k;
  if (a.nvfp4) {
    a.q_g = static_cast<const float*>(q->gscale4);
    a.k_g = static_cast<const float*>(k->gscale4);
    a.q_bs = static_cast<const uint8_t*>(q->scales4);
    a.k_bs = static_cast<const uint8_t*>(k->scales4);
    if (!make_nv_map(&maps.qn, q->codes4, p->d, p->H, p->T) || !make_nv_map(&maps.kn, k->codes4, p->d, p->Hkv, p->T))
      return FLAMIA_ERR_CUDA;
  }
  return launch_fwd(a, maps, stream) == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

flamia_status_t flamia_bwd(const flamia_problem_t* p, const flamia_operand_t* q, const flamia_operand_t* k,
                           const flamia_operand_t* v, const flamia_operand_t* dO, const float* D, const int32_t* m,
                           const float* l, void* dQ, void* dK, void* dV, void* ws, size_t ws_bytes,
                           cudaStream_t stream) {
  flamia_status_t s = validate(p);
  if (s != FLAMIA_OK) return s;
  // the bit-level exponential forward is for inference: the backward cannot
  // rebuild its P^ ([SUM] §3.7)
  if (p->bitexp) return FLAMIA_ERR_UNSUPPORTED;
  WsLayout L;
  if ((s = check_ws(p, ws, ws_bytes, &L)) != FLAMIA_OK) return s;
  if (!operand_ok(q) || !operand_ok(k) || !operand_ok(v) || !operand_ok(dO) || !D || !m || !l || !dQ || !dK ||
      !dV || !aligned16(D) || !aligned16(m) || !aligned16(l) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
    return FLAMIA_ERR_INVALID_ARG;
  if (p->path == FLAMIA_PATH_NVFP4_FP8 && (!q->codes4 || !q->scales4 || !q->gscale4 || !k->codes4 ||
                                           !k->scales4 || !k->gscale4))
    return FLAMIA_ERR_INVALID_ARG;
  AttnParams a;
  fill_params(p, L, ws, &a);
  a.q_sc = static_cast<const uint8_t*>(q->scales);
  a.k_sc = static_cast<const uint8_t*>(k->scales);
  a.v_sc = static_cast<const uint8_t*>(v->scales);
  a.do_sc = static_cast<const uint8_t*>(dO->scales);
  a.D = D;
  a.m = const_cast<int32_t*>(m);
  a.l = const_cast<float*>(l);
  a.dQ = dQ; a.dK = dK; a.dV = dV;
  AttnMaps maps;
  if (!make_codes_map(&maps.q, q->codes, p->d, p->H, p->T) || !make_codes_map(&maps.k, k->codes, p->d, p->Hkv, p->T) ||
      !make_codes_map(&maps.v, v->codes, p->d, p->Hkv, p->T) || !make_codes_map(&maps.dO, dO->codes, p->d, p->H, p->T) ||
      !make_dq_map(&maps.dq, a.dq_acc, p->d, p->H, p->T, a.dq_fp16 != 0))
    return FLAMIA_ERR_CUDA;
  maps.qn = maps.q;
  maps.kn = maps.k;
  if (a.nvfp4) {
    a.q_g = static_cast<const float*>(q->gscale4);
    a.k_g = static_cast<const float*>(k->gscale4);
    a.q_bs = static_cast<const uint8_t*>(q->scales4);
    a.k_bs = static_cast<const uint8_t*>(k->scales4);
    if (!make_nv_map(&maps.qn, q->codes4, p->d, p->H, p->T) || !make_nv_map(&maps.kn, k->codes4, p->d, p->Hkv, p->T))
      return FLAMIA_ERR_CUDA;
  }
  return launch_bwd(a, maps, stream) == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

flamia_status_t flamia_get_device_status(const void* ws, cudaStream_t stream) {
  if (!ws) return FLAMIA_ERR_INVALID_ARG;
  uint32_t st = 0;
  if (cudaMemcpyAsync(&st, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FLAMIA_ERR_CUDA;
  return static_cast<flamia_status_t>(st);
}

flamia_status_t flamia_debug_set_phat_dump(void* ws, size_t ws_bytes, void* codes, int32_t* exps,
                                           cudaStream_t stream) {
  if (!ws || ws_bytes < sizeof(WsHeader) || (codes == nullptr) != (exps == nullptr)) return FLAMIA_ERR_INVALID_ARG;
  static thread_local void* ptrs[2];
  ptrs[0] = codes;
  ptrs[1] = exps;
  uint8_t* dst = static_cast<uint8_t*>(ws) + offsetof(WsHeader, dbg_phat);
  if (cudaMemcpyAsync(dst, ptrs, sizeof(ptrs), cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return FLAMIA_ERR_CUDA;
  return FLAMIA_OK;
}

size_t flamia_debug_workspace_offset(const flamia_problem_t* p, int32_t region) {
  if (validate(p) != FLAMIA_OK) return 0;
  const WsLayout L = ws_layout(*p);
  switch (region) {
    case FLAMIA_WS_FWD_ITEMS: return L.fwd_items;
    case FLAMIA_WS_BWD_ITEMS: return L.bwd_items;
    case FLAMIA_WS_DQ_PRESCALE: return L.pexp;
  }
  return 0;
}

flamia_status_t flamia_debug_withhold_first_item(int32_t on) {
  g_dbg_withhold.store(on ? 1 : 0);
  return FLAMIA_OK;
}

flamia_status_t flamia_debug_mma_idesc(int32_t kind, uint32_t M, uint32_t N, int32_t a_mn, int32_t b_mn,
                                       int32_t a_sf_id, int32_t b_sf_id, uint32_t* out) {
  const uint32_t n_step = M == 64 ? 8u : 16u;
  if (!out || (M != 64 && M != 128) || N < n_step || N > 256 || N % n_step) return FLAMIA_ERR_INVALID_ARG;
  if ((a_mn | b_mn) & ~1 || (a_sf_id | b_sf_id) & ~3) return FLAMIA_ERR_INVALID_ARG;
  switch (kind) {
    case FLAMIA_MMA_F8F6F4:
      if (a_sf_id || b_sf_id) return FLAMIA_ERR_INVALID_ARG;
      *out = idesc_f8(M, N, (uint32_t)a_mn, (uint32_t)b_mn);
      return FLAMIA_OK;
    case FLAMIA_MMA_MXF8F6F4:
      *out = idesc_mxf8(M, N, (uint32_t)a_mn, (uint32_t)b_mn, (uint32_t)a_sf_id, (uint32_t)b_sf_id);
      return FLAMIA_OK;
    case FLAMIA_MMA_MXF4NVF4:
      if (a_mn || b_mn || a_sf_id || b_sf_id) return FLAMIA_ERR_INVALID_ARG;
      *out = idesc_mxf4nvf4(M, N);
      return FLAMIA_OK;
  }
  return FLAMIA_ERR_INVALID_ARG;
}

flamia_status_t flamia_debug_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, int32_t swizzle,
                                       uint64_t* out) {
  if (!out || ((saddr | lbo | sbo) & 15u) || saddr >= (1u << 18) || lbo >= (1u << 18) || sbo >= (1u << 18))
    return FLAMIA_ERR_INVALID_ARG;
  if (swizzle != FLAMIA_SWZ_NONE && swizzle != FLAMIA_SWZ_128B && swizzle != FLAMIA_SWZ_64B &&
      swizzle != FLAMIA_SWZ_32B)
    return FLAMIA_ERR_INVALID_ARG;
  *out = smem_desc(saddr, lbo, sbo, (uint32_t)swizzle);
  return FLAMIA_OK;
}

flamia_status_t flamia_clear_device_status(void* ws, cudaStream_t stream) {
  if (!ws) return FLAMIA_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, 2 * sizeof(uint32_t), stream) == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

}  // extern "C"
