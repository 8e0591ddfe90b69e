// common.cuh — device helpers shared by the kernels: workspace layout,
// status word, fp8/fp4 conversions, mbarrier, TMA and tcgen05 wrappers.
// Everything is sm_103a inline PTX written against the PTX ISA (CUDA 13.0).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda.h>

#include "../../include/flamia.h"

namespace flamia {

// ---------------------------------------------------------------------------
// Workspace layout (device bytes, all offsets 256-aligned).
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t status;         // flamia_status_t of the first device-side failure
  uint32_t status_where;   // kernel tag + site of that failure
  int32_t n_items;         // tiles (document, 128-token tile) in the plan
  int32_t n_blk32;         // document-local 32-token blocks
  uint32_t fwd_counter;    // persistent-grid work counters (reset per launch)
  uint32_t bwd_counter;
  uint32_t pad0[2];
  uint8_t* dbg_phat;       // test hook: P^ codes [H][T][T] (null: off)
  int32_t* dbg_eb;         // test hook: P^ block exponents [H][T][T] at each block's first key
  uint32_t pad[52];
};
static_assert(sizeof(WsHeader) == 256, "header");

// Test hook: record one row's P^ codes and block exponents for `nb` 32-key
// blocks starting at block b0 of a 128-key tile (w[8 * i + k] = word k of
// block i).  Out of line, not unrolled and taking its data by value: it runs
// only when the hook is set, and the hot loops keep their registers and a
// small code footprint.  Callers test `dc` first.
struct PhatDump {
  uint32_t w[16];
  int e[2];
};
static __device__ __noinline__ void dbg_dump_phat(uint8_t* dc, int32_t* de, int T, int h, int tok, int key_tok0, int b0,
                                          int nb, const PhatDump d) {
  const size_t row = ((size_t)h * T + tok) * (size_t)T;
  const int k0 = key_tok0 + 32 * b0;
#pragma unroll 1
  for (int j = 0; j < 32 * nb; ++j)
    if (k0 + j < T) dc[row + k0 + j] = (uint8_t)(d.w[j >> 2] >> (8 * (j & 3)));
#pragma unroll 1
  for (int b = 0; b < nb; ++b)
    if (k0 + 32 * b < T) de[row + k0 + 32 * b] = d.e[b];
}

struct WsLayout {
  size_t header, tile_prefix, blk32_prefix, fwd_items, bwd_items, keys_a, keys_b;
  size_t dq_acc;           // [T][H][d] dQ accumulator: fp32, or binary16 with dq_fp16
  size_t pexp;             // int8 [H][T]: the dQ prescale exponent of each query row
  size_t rot_dk;           // hadamard: fp32 [T][Hkv][d] dK before the back-rotation
  size_t dq_order;         // uint32 [max_items][H]: ordered dQ reduction counters
  size_t total;
  int32_t max_items;       // upper bound of tiles: ceil(T/128) + n_seq
  int32_t sort_n;          // max_items rounded up to the block-sort size
};

constexpr int kSortBlock = 2048;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline WsLayout ws_layout(const flamia_problem_t& p) {
  WsLayout L{};
  L.max_items = (p.T + 127) / 128 + p.n_seq;
  L.sort_n = ((L.max_items + kSortBlock - 1) / kSortBlock) * kSortBlock;
  size_t o = 0;
  L.header = o; o = align256(o + sizeof(WsHeader));
  L.tile_prefix = o; o = align256(o + sizeof(int32_t) * (p.n_seq + 1));
  L.blk32_prefix = o; o = align256(o + sizeof(int32_t) * (p.n_seq + 1));
  L.fwd_items = o; o = align256(o + sizeof(int2) * L.max_items);
  L.bwd_items = o; o = align256(o + sizeof(int2) * L.max_items);
  L.keys_a = o; o = align256(o + sizeof(uint64_t) * L.sort_n * 2);
  L.keys_b = o; o = align256(o + sizeof(uint64_t) * L.sort_n * 2);
  // fp32 unless the FP16 partials alone use it (the rotation's back-transform
  // reads every dQ path's result from here in fp32; the exact option sums
  // fp32 partials)
  const bool acc16 = p.dq_fp16 && !p.hadamard && !p.exact;
  L.dq_acc = o; o = align256(o + (acc16 ? 2 : 4) * (size_t)p.T * p.H * p.d);
  L.pexp = o; o = align256(o + (size_t)p.T * p.H);
  L.dq_order = o; o = align256(o + sizeof(uint32_t) * (size_t)L.max_items * p.H);
  L.rot_dk = 0;
  if (p.hadamard) {  // dK in the rotated basis, fp32, before the back-rotation
    L.rot_dk = o; o = align256(o + 4 * (size_t)p.T * p.Hkv * p.d);
  }
  L.total = o;
  return L;
}

// Device-side failure report: first writer wins.
__device__ __forceinline__ void report(WsHeader* hdr, uint32_t code, uint32_t where) {
  if (atomicCAS(&hdr->status, 0u, code) == 0u) hdr->status_where = where;
}

// ---------------------------------------------------------------------------
// Numeric helpers.
// ---------------------------------------------------------------------------
// 2^e as fp32 for e in [-126, 127] (built from the exponent field).
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// The no-clamp exponent of a non-negative fp32 amax: the smallest integer e
// with amax <= 448 * 2^e, clamped to [-127, 127]; 0 for amax == 0.
// amax = 1.m * 2^(E-127) = (1.m / 2) * 2^(E-126): e = E-135 when 1.m <= 1.75,
// else E-134.  Subnormal amax lies far below 448 * 2^-127 and clamps to -127.
__device__ __forceinline__ int noclamp_exp_clamped(float amax) {
  uint32_t b = __float_as_uint(amax);
  if (b == 0u) return 0;
  int E = (int)(b >> 23);
  if (E == 0) return -127;
  int e = ((b & 0x7FFFFFu) <= 0x600000u) ? E - 135 : E - 134;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Two fp32 values in one 64-bit register for the packed FP32 instructions
// of sm_100-class SMs (fma/mul/add .rn.f32x2): each lane is rounded exactly
// as the scalar instruction rounds it, so results are bit-identical to the
// scalar forms with half the instructions.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// max(a, b, c) in one instruction (exact, as two fmaxf); an fabsf on an
// operand folds into it.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Max over the warp of a non-negative float (no NaN): with the sign bit
// cleared (a -0 counts as 0) the bit patterns order like unsigned integers,
// so one integer warp reduction replaces a five-step shuffle chain.
__device__ __forceinline__ float warp_max(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7FFFFFFFu));
}

// Two fp32 -> two E4M3FN codes (RNE, saturating), `lo` in the low byte.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  return (uint32_t)pack_e4m3x2(a, b) | ((uint32_t)pack_e4m3x2(c, d) << 16);
}
// Two E4M3FN codes (low byte first) -> two fp32 values (exact).
__device__ __forceinline__ float2 unpack_e4m3x2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}
// Two fp32 -> two E2M1 codes in one byte (RNE, saturating), `lo` in the low nibble.
__device__ __forceinline__ uint32_t pack_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers (bounded waits), TMA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The dynamic shared-memory buffer rounded up to a 1024-byte boundary (the
// 128-byte swizzle pattern repeats every 1024 bytes).  The array pointer is
// offset, rather than an integer copy of its address rounded, so the result
// stays in the shared address space and every access through it compiles to
// a shared-memory instruction instead of a generic one.
__device__ __forceinline__ uint8_t* smem_base_1k(uint8_t* raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes) : "memory");
}
// Announce `bytes` of asynchronous copies on `bar` without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Non-blocking test of a phase (the common case on the hot path: the phase
// has already completed when the consumer arrives).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// One poll.  The suspend-time hint lets the hardware park the warp until the
// phase completes (or 1 ms passes) instead of spinning on issue slots that
// the other warps of the same sub-partition need.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u) : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait.  Every wait in these kernels goes through here: after about
// two seconds without progress it records FLAMIA_ERR_TIMEOUT, raises the
// CTA's abort flag and returns false; a wait that finds the abort flag raised
// returns false at once, so every role leaves its loop and the CTA reaches
// its teardown (TMEM release) normally.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          WsHeader* hdr, uint32_t where) {
  if (mbar_test_wait(bar, parity)) return true;  // already complete: no suspend
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      report(hdr, FLAMIA_ERR_TIMEOUT, where);
      return false;
    }
  }
}

// Bounded wait (one thread) for a counter in global memory, written by other
// CTAs, to reach `want` (acquire): the ordered dQ reduction.  Same limit and
// abort protocol as mbar_wait.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Orders earlier generic-proxy accesses before later async-proxy (bulk copy)
// accesses of global memory, and the reverse.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ bool counter_wait(const uint32_t* ctr, uint32_t want, volatile int* abort_flag,
                                             WsHeader* hdr, uint32_t where) {
  if (ld_acquire_gpu(ctr) == want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    __nanosleep(64);
    if (ld_acquire_gpu(ctr) == want) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      report(hdr, FLAMIA_ERR_TIMEOUT, where);
      return false;
    }
  }
}

// Warp-uniform bounded wait: every lane polls, and the warp continues only if
// every lane saw the phase complete.  Warps that go on to warp-collective
// instructions (tcgen05.ld/st are .sync.aligned) use this form, so a timeout
// can never leave part of a warp behind.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                               WsHeader* hdr, uint32_t where) {
  const bool ok = mbar_wait(bar, parity, abort_flag, hdr, where);
  return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------------------
// Dynamic work distribution: the producer warp takes the next item of the
// longest-first list and publishes it in a small shared-memory ring; every
// other warp role reads the items in the same order from the ring, so all
// roles of a CTA agree on its items.  -1 marks the end.  Slots are released
// as soon as they are read.  Two ways to take the next item:
//  * persistent grid (one CTA per SM): a global counter (atomicAdd);
//  * cluster launch control (one CTA per item, blockIdx.x = the item): the
//    CTA starts with its own item, then asks the hardware to cancel a CTA of
//    the grid that has not been launched yet and takes that CTA's item; when
//    no CTA is left to cancel, the CTA is done.  Every item is processed
//    once: by its own CTA if that one is launched, else by the CTA that
//    cancelled it.
// ---------------------------------------------------------------------------
constexpr int kItemRing = 4;
struct ItemRing {
  int item[kItemRing];
  uint64_t full[kItemRing], empty[kItemRing];
  uint64_t clc_bar;                   // completion of a cancellation request
  alignas(16) uint32_t clc_resp[4];  // its 16-byte response
};

__device__ __forceinline__ void item_ring_init(ItemRing& r, uint32_t consumers) {
  for (int s = 0; s < kItemRing; ++s) {
    mbar_init(&r.full[s], 1);
    mbar_init(&r.empty[s], consumers);
  }
  mbar_init(&r.clc_bar, 1);
}

// Cluster launch control (PTX ISA 8.6, sm_100 and later; the grid's clusters
// are single CTAs here): request the cancellation of a not yet launched CTA;
// the response lands in `resp` and completes 16 bytes of `bar`'s transaction.
__device__ __forceinline__ void clc_try_cancel(uint32_t* resp, uint64_t* bar) {
  asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];"
               ::"r"(smem_u32(resp)), "r"(smem_u32(bar)) : "memory");
}
// The x index of the CTA a completed response cancelled, or -1 if the request
// found no CTA left to cancel.
__device__ __forceinline__ int clc_cancelled_x(const uint32_t* resp) {
  const uint32_t w0 = reinterpret_cast<const volatile uint32_t*>(resp)[0];
  const uint32_t w1 = reinterpret_cast<const volatile uint32_t*>(resp)[1];
  const uint32_t w2 = reinterpret_cast<const volatile uint32_t*>(resp)[2];
  const uint32_t w3 = reinterpret_cast<const volatile uint32_t*>(resp)[3];
  const uint64_t lo = ((uint64_t)w1 << 32) | w0, hi = ((uint64_t)w3 << 32) | w2;
  uint32_t cancelled;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
      "mov.b128 r, {%1, %2};\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(cancelled) : "l"(lo), "l"(hi));
  if (!cancelled) return -1;
  uint32_t x;
  asm volatile(
      "{\n\t.reg .b128 r;\n\t"
      "mov.b128 r, {%1, %2};\n\t"
      "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %0, r;\n\t}"
      : "=r"(x) : "l"(lo), "l"(hi));
  return (int)x;
}

// Producer warp (all lanes): fetch the n-th item of this CTA; -1 when none is
// left.  clc: by cluster launch control (the grid has a CTA per item), else
// from the global counter.  After a -1 the producer asks for nothing more.
// withhold_first (a test hook, a kernel parameter): the first item is never
// published, so every consumer's wait for it runs out.
__device__ __forceinline__ int item_publish(ItemRing& r, uint32_t n, uint32_t* counter, int n_work, int lane,
                                            volatile int* abort_flag, WsHeader* hdr, uint32_t where, bool& ok,
                                            int withhold_first, int clc) {
  const int s = (int)(n % kItemRing);
  if (!(ok = mbar_wait_warp(&r.empty[s], ((n / kItemRing) & 1) ^ 1, abort_flag, hdr, where))) return -1;
  // nothing has been issued yet when the first item is withheld, so the CTA
  // exits cleanly after its consumers' waits run out
  if (n == 0 && withhold_first) return -1;
  int w = 0, fail = 0;
  if (lane == 0) {
    if (!clc) {
      w = (int)atomicAdd(counter, 1u);
    } else if (n == 0) {
      w = (int)blockIdx.x;
    } else {  // request n - 1 of this CTA: phase (n - 1) & 1
      mbar_arrive_expect_tx(&r.clc_bar, 16);
      clc_try_cancel(r.clc_resp, &r.clc_bar);
      if (mbar_wait(&r.clc_bar, (n - 1) & 1, abort_flag, hdr, where | 0x80)) {
        w = clc_cancelled_x(r.clc_resp);
      } else {
        w = -1;
        fail = 1;
      }
    }
    if (w >= n_work) w = -1;
    r.item[s] = w;
    mbar_arrive(&r.full[s]);
  }
  if (__shfl_sync(0xffffffffu, fail, 0)) ok = false;
  return __shfl_sync(0xffffffffu, w, 0);
}

// Consumer, one thread: the n-th item (its slot released at once).
__device__ __forceinline__ int item_get(ItemRing& r, uint32_t n, volatile int* abort_flag, WsHeader* hdr,
                                        uint32_t where, bool& ok) {
  const int s = (int)(n % kItemRing);
  if (!(ok = mbar_wait(&r.full[s], (n / kItemRing) & 1, abort_flag, hdr, where))) return -1;
  const int w = *reinterpret_cast<volatile int*>(&r.item[s]);
  mbar_arrive(&r.empty[s]);
  return w;
}

// Consumer, whole warp: the n-th item (lane 0 releases the slot).
__device__ __forceinline__ int item_get_warp(ItemRing& r, uint32_t n, int lane, volatile int* abort_flag,
                                             WsHeader* hdr, uint32_t where, bool& ok) {
  const int s = (int)(n % kItemRing);
  if (!(ok = mbar_wait_warp(&r.full[s], (n / kItemRing) & 1, abort_flag, hdr, where))) return -1;
  const int w = *reinterpret_cast<volatile int*>(&r.item[s]);
  __syncwarp();
  if (lane == 0) mbar_arrive(&r.empty[s]);
  return w;
}

// After an abort, give TMA copies already issued by this CTA time to land
// before the CTA exits (bounded: about 50 microseconds).
__device__ __forceinline__ void drain_after_abort(volatile int* abort_flag) {
  if (*abort_flag) {
    for (int i = 0; i < 100; ++i) __nanosleep(500);
  }
}

__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
        "r"(smem_u32(bar))
      : "memory");
}
// Element-wise add of a shared-memory box into global memory through a tensor
// map (the element type is the map's; the reduction happens in L2, rows past
// the tensor's end are clipped); completion is tracked by bulk groups.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, const void* smem_src, int c0, int c1,
                                                  int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until the shared-memory sources of every committed bulk group have been read.
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk group has completed.
__device__ __forceinline__ void bulk_wait_group0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// All but the N most recent bulk groups of this thread have completed.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Generic-proxy shared-memory writes -> visible to the async proxy (MMA, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Per-warpgroup register budget (all four warps of a warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, loads/stores.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols) : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive (once) on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Shared-memory matrix descriptor (tcgen05 form): start >> 4 in bits 0-13,
// leading-dimension byte offset >> 4 in 16-29, stride-dimension byte offset
// >> 4 in 32-45, the fixed version value 1 in bits 46-47, base offset 0,
// swizzle mode in bits 61-63 (2 = 128B, 4 = 64B, 6 = 32B, 0 = none).
__host__ __device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swz) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1u << 46;
  d |= (uint64_t)(swz & 7u) << 61;
  return d;
}
constexpr uint32_t kSwz128 = 2, kSwz64 = 4, kSwz32 = 6;

// Instruction descriptor, kind::f8f6f4 (E4M3 x E4M3 -> fp32):
// c_format(4-5)=1 (F32), a_format(7-9)=0 (E4M3), b_format(10-12)=0,
// a_major(15), b_major(16) (0 K-major, 1 MN-major), N>>3 in 17-22, M>>4 in 24-28.
__host__ __device__ constexpr uint32_t idesc_f8(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
// Instruction descriptor, kind::mxf8f6f4 block-scaled (E4M3, UE8M0 scales):
// b_sf_id in 4-5, a/b formats 0, majors 15/16, N>>3 in 17-22, scale_format
// (bit 23) = 1 (UE8M0), M>>4 in 24-28, a_sf_id in 29-30.
__host__ __device__ constexpr uint32_t idesc_mxf8(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn,
                                                  uint32_t a_sf_id, uint32_t b_sf_id) {
  return (b_sf_id << 4) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24) |
         (a_sf_id << 29);
}

// Instruction descriptor, kind::mxf4nvf4 block-scaled (E2M1 A and B packed
// two to a byte, UE4M3 scales, one per 16 K-elements, scale_vec::4X):
// a_format (7-9) = b_format (10-12) = 1 (E2M1), K-major A and B, N>>3 in
// 17-22, scale_format (bit 23) = 0 (UE4M3), M>>4 in 24-28, scale ids 0.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(uint32_t M, uint32_t N) {
  return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem], E4M3 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate) : "memory");
}
// Block-scaled form: one UE8M0 scale per 32 K-elements for each row of A
// (scale-A in tensor memory) and each column of B (scale-B in tensor memory).
__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// NVFP4 form: 64 K-elements per instruction; scale words (four UE4M3 bytes,
// byte k for K-elements 16k..16k+15) in tensor memory: row m of A at lane m,
// column sfa + m / 32; column n of B, for the output rows of lane quarter q,
// at lane 32 q + n % 32, column sfb + n / 32 (as copy_scales_x4 lays them out).
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// Shared memory -> tensor memory, 32 rows x 16 bytes (512 contiguous bytes,
// row r at 16 r) copied to lanes r, 32 + r, 64 + r, 96 + r, columns
// col..col+3 (the same words in every lane quarter).  Issued by the MMA
// thread; ordered with its MMAs and tracked by its commits.
__device__ __forceinline__ void copy_scales_x4(uint32_t col_tmem, const void* src) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(col_tmem),
               "l"(smem_desc(smem_u32(src), 128, 128, 0)) : "memory");
}

// 32 lanes x 32 columns of 32-bit: thread t of the warp gets lane (quarter*32+t).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// The wait, with the loaded registers passed through it so that no use of
// them can be scheduled before the loads have landed.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&a)[32], uint32_t (&b)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
        "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]),
        "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]),
        "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31]),
        "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]),
        "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]),
        "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]),
        "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&a)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
        "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]),
        "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]),
        "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31])
      :
      : "memory");
}
// 32 lanes x 16 columns of 32-bit.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&a)[16]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]),
        "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t a) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(a) : "memory");
}
__device__ __forceinline__ void tmem_st2(uint32_t taddr, uint32_t a, uint32_t b) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
               "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Tensor-memory address of (lane, column).
__device__ __forceinline__ uint32_t taddr(uint32_t base, uint32_t lane, uint32_t col) {
  return base + (lane << 16) + col;
}

__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}" : "=r"(pred));
  return pred;
}

// Offset of 16-byte chunk `c` of row `r` in a 128B-swizzled tile (rows of
// 128 bytes, 8-row atoms of 1024 bytes, tile base 1024-aligned).
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c) { return r * 128u + ((c ^ (r & 7u)) << 4); }

}  // namespace flamia
