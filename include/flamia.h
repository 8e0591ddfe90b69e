/*
 * flamia.h — C ABI of the block-scaled causal attention training call
 * (FLAMIA-style MXFP8 and mixed NVFP4/FP8 paths) for one GB300 (sm_103a).
 *
 * Sources, by page title and section:
 *   [SUM]  "FLAMIA: FLAsh MIcroscaling Attention for Fast and Causally Safe
 *          Training on Blackwell" (paper summary), bullets under §3.1–§3.7,
 *          §4.1–§4.6.
 *   [READ] "因果安全的低精度注意力——FLAMIA Blackwell 训练内核精读"
 *          (close reading), 四 4.1–4.6 and 五 5.1–5.3.
 *
 * One training call is, in this order, on one CUDA stream:
 *   flamia_plan        -> work lists and document tables (once per cu_seqlens)
 *   flamia_quantize    -> role QKV: Q^, K^, V^ codes and scales
 *   flamia_fwd         -> O, per-row (m, l)
 *   flamia_quantize    -> role DO: dO^ codes and scales, D = rowsum(dO^ * O)
 *   flamia_bwd         -> dQ, dK, dV
 * ([READ] 五 5.1: the training call is forward + backward + quantization.)
 *
 * Conventions for every entry point:
 *   - Every pointer named "device" is a CUDA device pointer owned by the
 *     caller; the library never allocates, frees or synchronises inside
 *     plan/quantize/fwd/bwd, so the sequence can be captured in a CUDA graph.
 *   - Packed token-major layouts: activations [T][heads][d] (row-major, d
 *     contiguous); per-token metadata [heads][T].
 *   - Every device pointer must be 16-byte aligned (cu_seqlens: 4-byte);
 *     tensors are contiguous.
 *   - Arguments are validated on the host before any launch; a violation
 *     returns FLAMIA_ERR_INVALID_ARG or FLAMIA_ERR_UNSUPPORTED and launches
 *     nothing.  Launch failures return FLAMIA_ERR_CUDA.  Device-side
 *     conditions (a bounded wait that expired, an inconsistent cu_seqlens
 *     seen by a kernel) set the device status word in the workspace, read
 *     with flamia_get_device_status().
 *   - The workspace `ws` (size from flamia_workspace_size) holds the plan,
 *     the dQ accumulator (fp32, or FP16 with its prescale exponents), and
 *     the status word.  It must stay the same buffer from flamia_plan through
 *     flamia_bwd of one call.
 */
#ifndef FLAMIA_H_
#define FLAMIA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLAMIA_OK = 0,
  FLAMIA_ERR_INVALID_ARG = 1,
  FLAMIA_ERR_UNSUPPORTED = 2,
  FLAMIA_ERR_WORKSPACE_TOO_SMALL = 3,
  FLAMIA_ERR_CUDA = 4,
  FLAMIA_ERR_TIMEOUT = 5,
  FLAMIA_ERR_BAD_SEQLENS = 6
} flamia_status_t;

/* [SUM] §3.4: the two default training paths. */
typedef enum { FLAMIA_PATH_MXFP8 = 0, FLAMIA_PATH_NVFP4_FP8 = 1 } flamia_path_t;

typedef enum { FLAMIA_F32 = 0, FLAMIA_BF16 = 1 } flamia_dtype_t;

typedef enum { FLAMIA_ROLE_QKV = 0, FLAMIA_ROLE_DO = 1 } flamia_role_t;

/* Problem description (host struct; cu_seqlens is a device pointer).
 *   T            total packed tokens (>= 1)
 *   H, Hkv       query heads and key/value heads; H % Hkv == 0 (GQA)
 *   d            head dimension: 64 or 128
 *   n_seq        documents; cu_seqlens[0] = 0, cu_seqlens[n_seq] = T,
 *                non-decreasing (device int32 [n_seq + 1]); an empty document
 *                is allowed.  Batched equal-length input is
 *                {0, L, 2L, ...} ([SUM] §3.6.2: packed documents in place).
 *   causal       1: query i sees keys j <= i of its own document; 0: the whole
 *                document.
 *   exact        1: the exact option ([SUM] §4.5): per-token Q, K and dO
 *                scales, per-(row, 32-key) dS exponents for dQ, deterministic
 *                dQ.  0: token-block scales over 32 document-local tokens.
 *   causal_dq_scale  with dq_fp16: 1 takes the power-of-two prescale of
 *                row i's FP16 dQ partials from keys j <= i only ([SUM] §4.5:
 *                removes the sequence-range dependency of the dQ
 *                accumulator); 0 from the whole document.
 *   dq_fp16      1: the default option's dQ partials (one per 128-key tile)
 *                are prescaled by a power of two per query row, rounded to
 *                FP16 and reduced into an FP16 accumulator ([READ] 四 4.4;
 *                the setting the Python training call uses by default: as
 *                fast as fp32 on short documents, faster on long and packed
 *                ones, where it halves the accumulator's traffic);
 *                0: fp32 partials into an fp32 accumulator.  No effect on the
 *                exact option and the mixed path, whose dQ sums in fp32 in
 *                a fixed order.
 *   deterministic 1: dQ's partials (one per 128-key tile) are added in
 *                key-tile order (a counter per query tile and head orders the
 *                bulk reduce-adds of the CTAs), so dQ is reproducible bit for
 *                bit; FP16 partials with dq_fp16 (then every FP16 addition
 *                happens in the order the per-tile model of [READ] 四 4.4
 *                states), else fp32.
 *   softmax_scale  0 selects 1/sqrt(d).
 *   path         flamia_path_t.
 *   in_dtype     dtype of Q, K, V, dO, O inputs (FLAMIA_BF16 or FLAMIA_F32).
 *   out_dtype    dtype of O, dQ, dK, dV outputs.
 *   bitexp       1: inference forward with bit-level exponentials ([SUM] §3.7
 *                Bit-Level Exponentials for Inference, §4.4): on key pairs 0-4
 *                of every 8 in each 32-key block, 2^z is the bf16 bit-field
 *                approximation 2^floor(z) (1 + frac z), fraction rounded to 7
 *                bits, with a zero-mean shift of 7 units (pattern
 *                RNE(128 z) + 16249, 0 for z <= -126.9453125); the other
 *                pairs use the hardware exponential.  l sums the same values.
 *                MXFP8 path, default option only (else
 *                FLAMIA_ERR_UNSUPPORTED); flamia_bwd rejects it
 *                (FLAMIA_ERR_UNSUPPORTED): the backward must rebuild the
 *                forward's P^ exactly.
 *   hadamard     1: Q and K are rotated by the Sylvester Hadamard matrix H_d
 *                (entries +-1) before quantization ([SUM] §4.3 Ablation Study
 *                and abstract: the fused quantizer's Hadamard rotation;
 *                [READ] 四 4.4: it spreads outlier channels and keeps dot
 *                products).  The rotated values are formed in fp32 by the
 *                fast Walsh-Hadamard transform (stages h = 1, 2, ..., d/2)
 *                inside flamia_quantize, the 1/d of H_d H_d = d I is folded
 *                into the softmax scale, and flamia_bwd rotates dQ and dK
 *                back, so O, dQ, dK, dV keep their meaning.  The Q/K payloads
 *                hold rotated codes.  MXFP8 path only (else
 *                FLAMIA_ERR_UNSUPPORTED); the workspace grows by
 *                4 T Hkv d bytes.
 *   clc          how flamia_fwd and flamia_bwd hand out the longest-first
 *                work items ([SUM] §3.6.2 Load-Balanced Scheduling and
 *                [READ] 四 4.4, GPU-side scheduling: cluster launch control
 *                for skewed and causal calls).  1: the grid has one CTA per
 *                item (item = blockIdx.x, (ceil(T/128) + n_seq) * heads CTAs,
 *                those past the plan's item count exit at once); a CTA that
 *                finishes its item cancels a CTA not yet launched
 *                (clusterlaunchcontrol.try_cancel) and takes that item, and
 *                stops when none is left.  0: a persistent grid of one CTA
 *                per SM takes items from a global counter.  Results are the
 *                same up to the order of the dQ partials' additions.  Not
 *                with the exact or deterministic options
 *                (FLAMIA_ERR_UNSUPPORTED): their ordered dQ reduction waits
 *                on items earlier in the list, which the counter hands out
 *                first and cancellation need not.
 */
typedef struct {
  int32_t T, H, Hkv, d, n_seq;
  const int32_t* cu_seqlens;
  int32_t causal, exact, causal_dq_scale, deterministic;
  float softmax_scale;
  int32_t path, in_dtype, out_dtype;
  int32_t dq_fp16;
  int32_t bitexp;
  int32_t hadamard;
  int32_t clc;
} flamia_problem_t;

/* A quantized operand (device pointers, caller-owned).
 *   codes    uint8 [T][heads][d] E4M3FN codes.  One payload serves both MMA
 *            orientations ([SUM] §3.1).
 *   scales   uint8 [heads][T] UE8M0 exponent byte (e + 127) of each token's
 *            block, replicated per token ([SUM] §3.6.2: per-token scale
 *            metadata).  V always has one exponent per key ([SUM] abstract).
 *   codes4   mixed path, Q and K only: uint8 [T][heads][d/2], two E2M1 codes
 *            per byte, element 2k in the low nibble.
 *   scales4  mixed path, Q and K only: uint8 [T][heads][d/16] E4M3 block scales.
 *   gscale4  mixed path, Q and K only: float [heads][T] per-token fp32 scale.
 *   On the mixed path flamia_fwd and flamia_bwd read codes4 and scales4 of Q
 *   and K directly as the operands of the block-scaled NVFP4 score MMA
 *   ([SUM] §3.4: QK^T and its recompute in NVFP4, one E4M3 scale per 16
 *   head-dimension elements), so they must stay unchanged between the calls.
 * Unused members may be NULL. */
typedef struct {
  void* codes;
  void* scales;
  void* codes4;
  void* scales4;
  void* gscale4;
} flamia_operand_t;

/* Bytes of device workspace needed by plan/quantize/fwd/bwd for `p`
 * (0 if `p` is invalid). */
size_t flamia_workspace_size(const flamia_problem_t* p);

/* Builds, on the GPU, the document tables and the longest-first work lists
 * ([SUM] §3.6.2 and [READ] 4.4: a fixed-pass merge sort on the GPU, once per
 * microbatch, items issued in descending cost to a persistent grid or, with
 * clc, by cluster launch control).  One launch when each list fits one sort
 * block (ceil(T/128) + n_seq <= 2048).
 * Forward items are (document, 128-query tile) with cost = key tiles visited;
 * backward items are (document, 128-key tile) with cost = query tiles
 * visited; ties keep document order.  Reads cu_seqlens on the device only.
 * Also clears the workspace's device status word and test hooks: the status
 * read after flamia_bwd covers one call, plan through backward. */
flamia_status_t flamia_plan(const flamia_problem_t* p, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Fused quantizer ([SUM] §3.1, §3.2; [READ] 4.4 fused quantization).
 * role FLAMIA_ROLE_QKV: in = {Q [T][H][d], K [T][Hkv][d], V [T][Hkv][d]},
 *   out = {Q^, K^, V^} operands.  Q and K: token-block exponent over 32
 *   document-local tokens x d (per token in the exact option); V: per key.
 *   Exponent = smallest e with max|x| <= 448 * 2^e (nothing clamps), clamped
 *   to [-127, 127]; all-zero blocks take e = 0; codes RNE(x * 2^-e).
 *   Mixed path: Q and K also get the NVFP4 payload (codes4/scales4/gscale4).
 * role FLAMIA_ROLE_DO: in = {dO [T][H][d]}, O = the forward output as stored
 *   (out_dtype), out = {dO^}; also writes D (device float [H][T]),
 *   D_i = sum_d dO^_id * O_id from the same dO^ that feeds dP ([SUM] §3.3).
 * Requires flamia_plan on the same workspace. */
flamia_status_t flamia_quantize(const flamia_problem_t* p, int32_t role, const void* const* in, const void* O,
                                const flamia_operand_t* out, float* D, void* ws, size_t ws_bytes,
                                cudaStream_t stream);

/* Forward ([SUM] §3.1–§3.3; [READ] 4.1–4.4): S = Q^ K^T (mixed path:
 * g_Q(i) g_K(j) sum_d (e2m1 s)_Q (e2m1 s)_K from the NVFP4 payload, [SUM]
 * §3.4), online softmax over key tiles with an integer row reference, P^ quantized to E4M3 with one
 * exponent per (row, 32-key block) after the per-key V factor is folded in,
 * O += P^ V^ by a block-scaled MMA, O = acc / l.
 *   O  device [T][H][d] out_dtype
 *   m  device int32 [H][T]: the row's integer reference exponent
 *   l  device float [H][T]: sum_j 2^(x_ij - m_i), x = S * softmax_scale * log2(e)
 * Requires flamia_plan on the same workspace. */
flamia_status_t flamia_fwd(const flamia_problem_t* p, const flamia_operand_t* q, const flamia_operand_t* k,
                           const flamia_operand_t* v, void* O, int32_t* m, float* l, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* Backward ([SUM] §3.3; [READ] 4.3): recomputes S and P^ from the same Q^/K^
 * with the forward's tiling and exponent evaluation, dP = dO^ V^T,
 * dS = P (dP - D), dS quantized with one exponent per 32x32 block (the exact
 * option: per (row, 32 keys) for dQ), dV += P~^T dO^, dK += dS^T Q^,
 * dQ += dS K^; dK and dV accumulate in fp32; dQ's per-key-tile partials are
 * summed by bulk reduce-adds, in fp32, or (dq_fp16) prescaled by a power of
 * two per query row and summed in FP16 ([READ] 四 4.4); the exact and
 * deterministic options add the partials in key-tile order (the exact
 * option's in fp32); the mixed path takes the same route.
 * GQA sums dK/dV over the group.
 *   dQ device [T][H][d], dK/dV device [T][Hkv][d], out_dtype.
 * D, m, l as produced by flamia_quantize(DO) and flamia_fwd. */
flamia_status_t flamia_bwd(const flamia_problem_t* p, const flamia_operand_t* q, const flamia_operand_t* k,
                           const flamia_operand_t* v, const flamia_operand_t* dO, const float* D, const int32_t* m,
                           const float* l, void* dQ, void* dK, void* dV, void* ws, size_t ws_bytes,
                           cudaStream_t stream);

/* Reads and returns the device status word of `ws` (FLAMIA_OK,
 * FLAMIA_ERR_TIMEOUT or FLAMIA_ERR_BAD_SEQLENS).  Synchronises `stream`:
 * for tests and diagnostics, not for the hot path. */
flamia_status_t flamia_get_device_status(const void* ws, cudaStream_t stream);

/* Clears the device status word (stream-ordered, no synchronisation). */
flamia_status_t flamia_clear_device_status(void* ws, cudaStream_t stream);

/* Test hook (not for the hot path): make the next flamia_fwd / flamia_bwd
 * calls on workspace `ws` record, for every (query head h, query token i,
 * key token j) they evaluate, the P^ code in codes[(h*T + i)*T + j] (device
 * uint8 [H][T][T]) and each 32-key block's exponent in
 * exps[(h*T + i)*T + j0] at the block's first key j0 (device int32 [H][T][T]).
 * Both kernels write the P^ they use, so a caller can check that the backward
 * rebuilds the forward's P^ bit for bit ([SUM] §3.3).  NULL, NULL switches the
 * hook off.  Must be called after flamia_plan (which does not touch it) and
 * synchronises `stream`. */
flamia_status_t flamia_debug_set_phat_dump(void* ws, size_t ws_bytes, void* codes, int32_t* exps,
                                           cudaStream_t stream);

/* Regions of the workspace that tests read back (flamia_debug_workspace_offset). */
typedef enum {
  FLAMIA_WS_FWD_ITEMS = 0,    /* int32 pairs (document, 128-query tile), longest first */
  FLAMIA_WS_BWD_ITEMS = 1,    /* int32 pairs (document, 128-key tile), longest first */
  FLAMIA_WS_DQ_PRESCALE = 2   /* int8 [H][T]: exponent p of the FP16 dQ partials' prescale 2^p */
} flamia_ws_region_t;

/* Test hook: byte offset of a region inside the workspace of problem `p`
 * (0 for an invalid problem or region).  The dQ prescale exponents are
 * written by flamia_bwd on the dq_fp16 path. */
size_t flamia_debug_workspace_offset(const flamia_problem_t* p, int32_t region);

/* Test hook (not for the hot path): exercise the bounded waits.  While on,
 * each CTA of the next flamia_fwd / flamia_bwd launches withholds its first
 * work item, so its other roles' waits for that item run out after the
 * bounded-wait limit (about 2 s): the kernel records FLAMIA_ERR_TIMEOUT in the
 * device status word, every role leaves its loop and the CTA releases its
 * tensor memory and exits (nothing was issued, so no copy or MMA is in
 * flight).  The outputs of such a call are undefined.  Process-wide (not per
 * workspace); flamia_plan switches it off.  Always returns FLAMIA_OK. */
flamia_status_t flamia_debug_withhold_first_item(int32_t on);

/* Test hooks (no device call): the tensor-core descriptors the kernels issue,
 * as the library's own builders encode them, so that a host test can check
 * each bit field against the field tables of the PTX ISA's tcgen05
 * "Instruction descriptor" and "Shared memory descriptor" sections.
 *
 * flamia_debug_mma_idesc: the 32-bit instruction descriptor of one
 *   tcgen05.mma of kind
 *     FLAMIA_MMA_F8F6F4   kind::f8f6f4, E4M3 x E4M3, fp32 accumulator;
 *     FLAMIA_MMA_MXF8F6F4 kind::mxf8f6f4.block_scale.scale_vec::1X, E4M3
 *                         operands, UE8M0 scales (one per 32 K-elements);
 *     FLAMIA_MMA_MXF4NVF4 kind::mxf4nvf4.block_scale.scale_vec::4X, E2M1
 *                         operands, UE4M3 scales (one per 16 K-elements);
 *   for an M x N tile (cta_group::1: M = 64 with N a multiple of 8, or
 *   M = 128 with N a multiple of 16; 8 or 16 <= N <= 256).  a_mn / b_mn = 1
 *   selects an MN-major operand (0 or 1; 0 for the E2M1 kind), a_sf_id /
 *   b_sf_id the scale-factor ids of the block-scaled kinds (0..3; 0 for the
 *   E2M1 kind, 0 for kind::f8f6f4).  Writes *out and returns FLAMIA_OK;
 *   FLAMIA_ERR_INVALID_ARG for a NULL out or an argument outside these
 *   ranges (then *out is untouched).
 * flamia_debug_smem_desc: the 64-bit shared-memory matrix descriptor for a
 *   tile at shared address saddr with leading- and stride-dimension byte
 *   offsets lbo / sbo (all multiples of 16 below 2^18) and swizzle mode
 *   FLAMIA_SWZ_NONE / _128B / _64B / _32B.  Same return rules. */
typedef enum { FLAMIA_MMA_F8F6F4 = 0, FLAMIA_MMA_MXF8F6F4 = 1, FLAMIA_MMA_MXF4NVF4 = 2 } flamia_mma_kind_t;
typedef enum { FLAMIA_SWZ_NONE = 0, FLAMIA_SWZ_128B = 2, FLAMIA_SWZ_64B = 4, FLAMIA_SWZ_32B = 6 } flamia_swizzle_t;
flamia_status_t flamia_debug_mma_idesc(int32_t kind, uint32_t M, uint32_t N, int32_t a_mn, int32_t b_mn,
                                       int32_t a_sf_id, int32_t b_sf_id, uint32_t* out);
flamia_status_t flamia_debug_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, int32_t swizzle,
                                       uint64_t* out);

/* Allocation-free work-list builder (this library's own addition; the
 * method's pages have no counterpart).  For callers that cannot allocate
 * device memory: code inside a CUDA graph under capture (cudaMalloc cannot be
 * captured), embeddings without an allocator, or frameworks that forbid
 * allocations outside their own caching allocator.  It builds the same two
 * longest-first work lists as flamia_plan, but its scratch (document
 * prefix tables, sort keys) lives in a file-scope device array of the library
 * (about 2.5 MiB, held by every GPU that loads the library until the process
 * exits) instead of a caller workspace; it calls no allocating routine.
 *   fwd_items, bwd_items  device int32 pairs (document, 128-token tile),
 *                         each [ceil(T/128) + n_seq] entries, caller-owned;
 *                         the first *n_items entries are written.
 *   n_items               device int32, receives the number of tiles (0 when
 *                         cu_seqlens is inconsistent with T).
 * Limits: ceil(T/128) + n_seq <= 65536 and n_seq <= 65536, else
 * FLAMIA_ERR_UNSUPPORTED.  The first call on each device looks up the array's
 * device address with that device current (make that first call before any
 * stream capture) and keeps it for the life of the process, so the entry
 * point must not be used on a device after cudaDeviceReset.  All calls share
 * the array and it keeps the last call's
 * contents: calls whose kernels may overlap on the GPU race with each other
 * and must be serialised by the caller. */
flamia_status_t flamia_plan_noalloc(const flamia_problem_t* p, int2* fwd_items, int2* bwd_items, int32_t* n_items,
                                    cudaStream_t stream);

/* Static description of a status code. */
const char* flamia_status_string(flamia_status_t s);

#ifdef __cplusplus
}
#endif
#endif /* FLAMIA_H_ */
