// kernels.h — host-side launch interfaces between api.cu and the kernels.
#pragma once
#include "common.cuh"

namespace flamia {

struct QuantArgs {
  const void* x;     // [T][heads][d]
  uint8_t* codes;    // [T][heads][d]
  uint8_t* scales;   // [heads][T]
  uint8_t* codes4;   // [T][heads][d/2]   (NVFP4 operand)
  uint8_t* scales4;  // [T][heads][d/16]
  float* gscale4;    // [heads][T]
  const void* O;     // [T][heads][d]     (dO role)
  float* D;          // [heads][T]
  int T, heads;
  int per_token;
  int rotate;        // Hadamard rotation of each token's d-vector before quantization
};

// Up to three tensors quantized by one launch (Q, K, V; or dO alone).
struct QuantBatch {
  QuantArgs a[3];
  int n;
};

cudaError_t launch_quantize(const QuantBatch& qb, int d, int in_bf16, int o_bf16, bool with_D, bool nvfp4,
                            const int32_t* cu, const int32_t* blk_prefix, int n_seq, WsHeader* hdr, int max_units,
                            int n_sms, cudaStream_t st);
int sm_count();

// Grid of an attention kernel over `work` items: one CTA per SM (persistent,
// items from a global counter) or, with cluster launch control, one CTA per
// item.  Such a CTA asks for at least kClcMinSmem bytes of shared memory so
// that no two share an SM: each holds all of the SM's tensor memory.
constexpr size_t kClcMinSmem = 116 * 1024;
inline int attn_grid(long work, int nsm, int clc) { return clc ? (int)work : (int)(work < nsm ? work : nsm); }
inline size_t attn_smem(size_t smem, int clc) { return clc && smem < kClcMinSmem ? kClcMinSmem : smem; }
inline size_t attn_smem_max(size_t smem) { return smem < kClcMinSmem ? kClcMinSmem : smem; }
cudaError_t launch_plan(const flamia_problem_t& p, const WsLayout& L, uint8_t* ws, cudaStream_t st);

// Everything the attention kernels need for one call (host-built).
struct AttnParams {
  int T, H, Hkv, d, n_seq, causal, exact, deterministic, out_bf16, max_items;
  int dbg_withhold;     // test hook: each CTA's producer withholds its first work item
  float softmax_scale;  // c' (scores)
  float c_log2;         // softmax_scale * log2(e)
  const int32_t* cu;
  const int32_t* tile_prefix;
  const int2* fwd_items;
  const int2* bwd_items;
  WsHeader* hdr;
  const uint8_t* q_sc;  // [H][T]
  const uint8_t* k_sc;  // [Hkv][T]
  const uint8_t* v_sc;  // [Hkv][T]
  const uint8_t* do_sc; // [H][T]
  const float* q_g;     // mixed path: per-token fp32 scale of Q's NVFP4 payload [H][T]
  const float* k_g;     // mixed path: of K's [Hkv][T]
  int nvfp4;            // 1: scores from the NVFP4 payload (block-scaled E2M1 MMAs)
  const uint8_t* q_bs;  // mixed path: Q's E4M3 16-element block scales [T][H][d/16]
  const uint8_t* k_bs;  // mixed path: K's [T][Hkv][d/16]
  int bitexp;           // 1: forward with bit-level exponentials (inference only)
  int hadamard;         // 1: Q, K rotated; dQ, dK go through fp32 buffers and are rotated back
  float* rot_dk;        // hadamard: fp32 [T][Hkv][d] dK (times the softmax scale), rotated basis
  uint32_t* dq_order;   // [tiles][H]: dQ partials already added to each (query tile, head), in key-tile order
  int dq_ordered;       // 1: the partials are added in key-tile order (deterministic and exact options)
  int clc;              // 1: a CTA per work item, items taken over by cluster launch control
  const float* D;       // [H][T]
  int32_t* m;           // [H][T]
  float* l;             // [H][T]
  void* O;              // [T][H][d]
  float* dq_acc;        // [T][H][d] fp32 dQ accumulator (dq_fp16 = 0)
  __half* dq16;         // [T][H][d] binary16 dQ accumulator, prescaled FP16 partials (dq_fp16 = 1)
  int dq_fp16;
  int8_t* pexp;         // [H][T] dQ prescale exponent of each query row
  int c0;               // ceil(log2(2.5 d 448^3 softmax_scale)): the constant of the prescale bound
  int causal_dq_scale;  // 1: the prescale from keys j <= i only (causal); 0: the whole document
  void* dQ;             // [T][H][d]
  void* dK;             // [T][Hkv][d]
  void* dV;             // [T][Hkv][d]
};

struct AttnMaps {
  CUtensorMap q, k, v, dO;
  CUtensorMap qn, kn;  // mixed path: packed E2M1 codes, boxes of 128 tokens x d/2 bytes
  CUtensorMap dq;      // dQ accumulator [T][H][d], the reduce-add target: fp32 boxes of 128 rows x 32
                       // values, or (dq_fp16) FP16 boxes of 128 rows x 64 values; 128B swizzle
};

cudaError_t launch_fwd(const AttnParams& p, const AttnMaps& maps, cudaStream_t st);
cudaError_t launch_bwd(const AttnParams& p, const AttnMaps& maps, cudaStream_t st);

}  // namespace flamia
