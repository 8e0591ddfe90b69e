// plan.cu — document tables and the longest-first work lists, built on the
// GPU once per microbatch with no host read-back.
//
// FLAMIA (paper summary), §3.6.2 Load-Balanced Scheduling and the close
// reading 4.4 (GPU-side scheduling): the schedule is built on the GPU with a
// fixed number of merge-sort passes and handed to a persistent grid in
// descending cost.  Here a work item is a (document, 128-token tile); its cost
// is the number of tiles the kernel visits for it: key tiles for a forward
// query tile, query tiles for a backward key tile.  Sort keys are
// (cost descending, item index ascending), unique, so the order is
// deterministic.  The pass count depends only on a host-side bound of the item
// count (ceil(T/128) + n_seq), so the whole plan can be captured in a graph.
#include <mutex>

#include "common.cuh"

namespace flamia {

// One CTA of 1024 threads: the per-document 128-tile and 32-block counts of
// cu_seqlens, exclusive scans into tile_out / blk_out (n_seq + 1 entries
// each; blk_out may be null), chunks of 1024 documents through a
// Hillis-Steele scan in shared memory with a running carry.  Every thread
// returns the totals and whether cu_seqlens is inconsistent (first entry not
// 0, last not T, or a negative length).
__device__ void scan_documents(const int32_t* __restrict__ cu, int n_seq, int T, int32_t* tile_out,
                               int32_t* blk_out, int& total_t, int& total_b, int& bad_out) {
  __shared__ int32_t s_t[1024], s_b[1024];
  __shared__ int32_t carry_t, carry_b, bad;
  const int tid = threadIdx.x;
  if (tid == 0) {
    carry_t = 0;
    carry_b = 0;
    bad = (__ldg(cu) != 0 || __ldg(cu + n_seq) != T) ? 1 : 0;
  }
  __syncthreads();
  for (int base = 0; base < n_seq; base += 1024) {
    const int i = base + tid;
    int nt = 0, nb = 0;
    if (i < n_seq) {
      const int len = __ldg(cu + i + 1) - __ldg(cu + i);
      if (len < 0) bad = 1;
      const int l = len < 0 ? 0 : len;
      nt = (l + 127) / 128;
      nb = (l + 31) / 32;
    }
    s_t[tid] = nt;
    s_b[tid] = nb;
    __syncthreads();
    for (int off = 1; off < 1024; off <<= 1) {  // Hillis-Steele inclusive scan
      int at = tid >= off ? s_t[tid - off] : 0;
      int ab = tid >= off ? s_b[tid - off] : 0;
      __syncthreads();
      s_t[tid] += at;
      s_b[tid] += ab;
      __syncthreads();
    }
    if (i < n_seq) {
      tile_out[i] = carry_t + s_t[tid] - nt;
      if (blk_out != nullptr) blk_out[i] = carry_b + s_b[tid] - nb;
    }
    __syncthreads();
    if (tid == 1023) {
      carry_t += s_t[1023];
      carry_b += s_b[1023];
    }
    __syncthreads();
  }
  if (tid == 0) {
    tile_out[n_seq] = carry_t;
    if (blk_out != nullptr) blk_out[n_seq] = carry_b;
  }
  __syncthreads();
  total_t = carry_t;
  total_b = carry_b;
  bad_out = bad;
}

// Header fields a plan resets (one thread), before the scan.
__device__ __forceinline__ void plan_reset_header(WsHeader* hdr) {
  hdr->fwd_counter = 0;
  hdr->bwd_counter = 0;
  hdr->status = 0;         // the status word covers one call, plan through backward
  hdr->status_where = 0;
  hdr->dbg_phat = nullptr;  // test hooks off unless set after the plan
  hdr->dbg_eb = nullptr;
}
// Header totals of a plan (one thread), after the scan.
__device__ __forceinline__ void plan_set_totals(WsHeader* hdr, int total_t, int total_b, int bad) {
  hdr->n_items = bad ? 0 : total_t;
  hdr->n_blk32 = bad ? 0 : total_b;
  if (bad) report(hdr, FLAMIA_ERR_BAD_SEQLENS, 0x100u);
}

// One CTA: validate cu_seqlens, per-document 128-tile and 32-block counts,
// exclusive scans into tile_prefix / blk32_prefix, totals into the header.
__global__ void __launch_bounds__(1024) plan_prefix_kernel(const int32_t* __restrict__ cu, int n_seq, int T,
                                                           int32_t* tile_prefix, int32_t* blk32_prefix,
                                                           WsHeader* hdr) {
  if (threadIdx.x == 0) plan_reset_header(hdr);
  int tt, tb, bad;
  scan_documents(cu, n_seq, T, tile_prefix, blk32_prefix, tt, tb, bad);
  if (threadIdx.x == 0) plan_set_totals(hdr, tt, tb, bad);
}

// A prefix-table entry: through the read-only cache (a table in global
// memory written by an earlier kernel) or a plain load (shared memory).
template <bool RO>
__device__ __forceinline__ int32_t prefix_at(const int32_t* t, int i) {
  if constexpr (RO) return __ldg(t + i);
  else return t[i];
}

template <bool RO = true>
__device__ __forceinline__ int doc_of_tile(const int32_t* tile_prefix, int n_seq, int g) {
  int lo = 0, hi = n_seq;  // tile_prefix[lo] <= g < tile_prefix[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (prefix_at<RO>(tile_prefix, mid) <= g) lo = mid; else hi = mid;
  }
  return lo;
}

// Sort key of slot g of list `lst` (0: forward, 1: backward).
// A real item's cost is at least 1, so its key's high word is at most
// 0xFFFFFFFE; a padding slot g gets the high word 0xFFFFFFFF and its own
// index below, so padding keys are unique too and sort after every real key
// in slot order.  (Equal padding keys would collide in the merge passes.)
template <bool RO = true>
__device__ __forceinline__ uint64_t plan_key(const int32_t* tile_prefix, int n_seq, int causal, int n_items, int lst,
                                             int g) {
  if (g >= n_items) return (0xFFFFFFFFull << 32) | (uint32_t)g;
  const int doc = doc_of_tile<RO>(tile_prefix, n_seq, g);
  const int p0 = prefix_at<RO>(tile_prefix, doc);
  const int tile = g - p0;
  const int nt = prefix_at<RO>(tile_prefix, doc + 1) - p0;
  const uint32_t cost = causal ? (uint32_t)(lst == 0 ? tile + 1 : nt - tile) : (uint32_t)nt;
  return ((uint64_t)(0xFFFFFFFFu - cost) << 32) | (uint32_t)g;
}

// Bitonic sort (ascending) of the kSortBlock keys in s (1024 threads).  Keys
// past the real items are padding, larger than every real key and ascending
// with the slot, so a block whose real keys fit in the first P = 2^k slots
// only runs the network up to size P: the padding above stays in place and
// the block ends sorted.
__device__ void sort_block_keys(uint64_t* s, int n_real) {
  const int tid = threadIdx.x;
  int P = 2;
  while (P < n_real) P <<= 1;
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const int i = 2 * tid - (tid & (stride - 1));  // lower index of the pair
      const int j = i + stride;
      if (j < P) {
        const bool up = ((i & size) == 0);
        const uint64_t a = s[i], b = s[j];
        if ((a > b) == up) { s[i] = b; s[j] = a; }
      }
      __syncthreads();
    }
  }
}

// Builds and sorts kSortBlock keys per CTA: keys[0 .. sort_n) hold the
// forward list, keys[sort_n .. 2 sort_n) the backward list.
__global__ void __launch_bounds__(1024) block_sort_kernel(const int32_t* __restrict__ tile_prefix, int n_seq,
                                                          int causal, uint64_t* keys, int sort_n,
                                                          const WsHeader* hdr) {
  __shared__ uint64_t s[kSortBlock];
  uint64_t* k = keys + (size_t)blockIdx.x * kSortBlock;
  const int tid = threadIdx.x;
  const int per_list = sort_n / kSortBlock;
  const int lst = (int)blockIdx.x / per_list, g0 = ((int)blockIdx.x % per_list) * kSortBlock;
  const int n_items = hdr->n_items;
  s[tid] = plan_key(tile_prefix, n_seq, causal, n_items, lst, g0 + tid);
  s[tid + 1024] = plan_key(tile_prefix, n_seq, causal, n_items, lst, g0 + tid + 1024);
  __syncthreads();
  sort_block_keys(s, min(kSortBlock, max(0, n_items - g0)));
  k[tid] = s[tid];
  k[tid + 1024] = s[tid + 1024];
}

// The whole plan in one launch when each list fits one sort block
// (ceil(T/128) + n_seq <= 2048, so n_seq <= 2048): CTA l (0: forward list, 1:
// backward list) scans the documents into its own shared copy of the tile
// prefix (CTA 0 also writes the tables and the header, as plan_prefix_kernel
// does), builds its list's keys from that copy, sorts them and writes the
// list's work items.  Nothing is read back from global memory within the
// launch.
__global__ void __launch_bounds__(1024) plan_single_block_kernel(const int32_t* __restrict__ cu, int n_seq, int T,
                                                                 int causal, int32_t* tile_prefix,
                                                                 int32_t* blk32_prefix, WsHeader* hdr,
                                                                 int2* fwd_items, int2* bwd_items) {
  __shared__ int32_t sp[kSortBlock + 1];
  __shared__ uint64_t s[kSortBlock];
  const int tid = threadIdx.x, lst = (int)blockIdx.x;
  if (lst == 0 && tid == 0) plan_reset_header(hdr);
  int tt, tb, bad;
  scan_documents(cu, n_seq, T, sp, lst == 0 ? blk32_prefix : nullptr, tt, tb, bad);
  const int n_items = bad ? 0 : tt;
  if (lst == 0) {
    for (int i = tid; i <= n_seq; i += 1024) tile_prefix[i] = sp[i];
    if (tid == 0) plan_set_totals(hdr, tt, tb, bad);
  }
  s[tid] = plan_key<false>(sp, n_seq, causal, n_items, lst, tid);
  s[tid + 1024] = plan_key<false>(sp, n_seq, causal, n_items, lst, tid + 1024);
  __syncthreads();
  sort_block_keys(s, min(kSortBlock, n_items));
  int2* items = lst == 0 ? fwd_items : bwd_items;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = tid + 1024 * h;
    if (i < n_items) {
      const int g = (int)(uint32_t)(s[i] & 0xFFFFFFFFull);
      const int doc = doc_of_tile<false>(sp, n_seq, g);
      items[i] = make_int2(doc, g - sp[doc]);
    }
  }
}

// One merge pass: sorted runs of `width` keys are merged pairwise.  Each key
// finds its output slot as (own rank) + (number of smaller keys in the
// sibling run), by binary search.  Keys are unique (padding included), so the
// slots of a pass are a permutation: every destination word is written, and
// no pass reads a word that an earlier pass did not write.  Two lists of
// sort_n keys.
__global__ void merge_pass_kernel(const uint64_t* __restrict__ src, uint64_t* __restrict__ dst, int sort_n,
                                  int width) {
  const int gi = blockIdx.x * blockDim.x + threadIdx.x;
  if (gi >= 2 * sort_n) return;
  const int seg = gi / sort_n, i = gi - seg * sort_n;
  const uint64_t* s = src + (size_t)seg * sort_n;
  uint64_t* d = dst + (size_t)seg * sort_n;
  const int pair = i / (2 * width);
  const int a0 = pair * 2 * width;
  const int b0 = a0 + width;
  const int a_len = min(width, sort_n - a0);
  const int b_len = max(0, min(width, sort_n - b0));
  const uint64_t key = s[i];
  const bool in_a = i < b0;
  const int own = in_a ? i - a0 : i - b0;
  const uint64_t* other = in_a ? s + b0 : s + a0;
  int lo = 0, hi = in_a ? b_len : a_len;  // count of keys in `other` smaller than key
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (other[mid] < key) lo = mid + 1; else hi = mid;
  }
  d[a0 + own + lo] = key;
  (void)a_len;
}

__global__ void plan_items_kernel(const uint64_t* __restrict__ keys, const int32_t* __restrict__ tile_prefix,
                                  int n_seq, int sort_n, const WsHeader* hdr, int2* fwd_items, int2* bwd_items) {
  const int gi = blockIdx.x * blockDim.x + threadIdx.x;
  const int n_items = hdr->n_items;
  if (gi >= 2 * sort_n) return;
  const int seg = gi / sort_n, r = gi - seg * sort_n;
  if (r >= n_items) return;
  const int g = (int)(uint32_t)(keys[gi] & 0xFFFFFFFFull);
  const int doc = doc_of_tile(tile_prefix, n_seq, g);
  const int2 it = make_int2(doc, g - __ldg(tile_prefix + doc));
  (seg == 0 ? fwd_items : bwd_items)[r] = it;
}

cudaError_t launch_plan(const flamia_problem_t& p, const WsLayout& L, uint8_t* ws, cudaStream_t st) {
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws + L.header);
  int32_t* tile_prefix = reinterpret_cast<int32_t*>(ws + L.tile_prefix);
  int32_t* blk_prefix = reinterpret_cast<int32_t*>(ws + L.blk32_prefix);
  uint64_t* ka = reinterpret_cast<uint64_t*>(ws + L.keys_a);
  uint64_t* kb = reinterpret_cast<uint64_t*>(ws + L.keys_b);
  const int n = L.sort_n;
  int2* fwd_items = reinterpret_cast<int2*>(ws + L.fwd_items);
  int2* bwd_items = reinterpret_cast<int2*>(ws + L.bwd_items);
  if (n == kSortBlock) {  // each list one sort block: the whole plan in one launch
    plan_single_block_kernel<<<2, 1024, 0, st>>>(p.cu_seqlens, p.n_seq, p.T, p.causal, tile_prefix, blk_prefix, hdr,
                                                  fwd_items, bwd_items);
    return cudaGetLastError();
  }
  plan_prefix_kernel<<<1, 1024, 0, st>>>(p.cu_seqlens, p.n_seq, p.T, tile_prefix, blk_prefix, hdr);
  block_sort_kernel<<<2 * n / kSortBlock, 1024, 0, st>>>(tile_prefix, p.n_seq, p.causal, ka, n, hdr);
  uint64_t *src = ka, *dst = kb;
  for (int w = kSortBlock; w < n; w *= 2) {
    merge_pass_kernel<<<(2 * n + 255) / 256, 256, 0, st>>>(src, dst, n, w);
    uint64_t* t = src; src = dst; dst = t;
  }
  plan_items_kernel<<<(2 * n + 255) / 256, 256, 0, st>>>(src, tile_prefix, p.n_seq, n, hdr, fwd_items, bwd_items);
  return cudaGetLastError();
}

}  // namespace flamia

// ===========================================================================
// Allocation-free work-list builder.
//
// For callers that cannot allocate device memory themselves: code running
// inside a CUDA graph that is being captured (cudaMalloc is not a stream
// operation and cannot be captured), allocator-less embeddings of the library,
// or a framework that forbids allocations outside its own caching allocator.
// flamia_plan_noalloc keeps the planner's scratch (prefix tables, sort keys)
// in the file-scope array below instead of the caller's workspace, and writes
// only the two sorted work lists and the item count to caller-owned buffers.
// Every GPU that loads this library holds the array (about 2.5 MiB) until the
// process exits.  All calls share it: calls whose kernels overlap on the GPU
// (different streams, or different threads) race and must be serialised by
// the caller.
// ===========================================================================
namespace flamia {
namespace {

constexpr int kNoAllocMaxItems = 65536;  // limit on ceil(T/128) + n_seq
constexpr int kNoAllocMaxSeq = 65536;    // limit on n_seq

struct NoAllocScratch {
  WsHeader hdr;
  int32_t tile_prefix[kNoAllocMaxSeq + 1];
  int32_t blk_prefix[kNoAllocMaxSeq + 1];
  uint64_t keys_a[2 * kNoAllocMaxItems];
  uint64_t keys_b[2 * kNoAllocMaxItems];
};

__device__ __align__(256) NoAllocScratch g_noalloc_scratch;

// Device address of g_noalloc_scratch for the current device, looked up once
// per device (the host-side symbol is a stand-in, not a device address).
NoAllocScratch* noalloc_scratch_for_current_device() {
  static std::mutex mu;
  static NoAllocScratch* addr[256] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<NoAllocScratch*>(p);
  }
  return addr[dev];
}

}  // namespace

}  // namespace flamia

extern "C" flamia_status_t flamia_plan_noalloc(const flamia_problem_t* p, int2* fwd_items, int2* bwd_items,
                                               int32_t* n_items, cudaStream_t stream) {
  using namespace flamia;
  if (flamia_workspace_size(p) == 0) return FLAMIA_ERR_INVALID_ARG;
  if (!fwd_items || !bwd_items || !n_items) return FLAMIA_ERR_INVALID_ARG;
  const int max_items = (p->T + 127) / 128 + p->n_seq;
  if (max_items > kNoAllocMaxItems || p->n_seq > kNoAllocMaxSeq) return FLAMIA_ERR_UNSUPPORTED;
  NoAllocScratch* sc = noalloc_scratch_for_current_device();
  if (sc == nullptr) return FLAMIA_ERR_CUDA;
  const int n = ((max_items + kSortBlock - 1) / kSortBlock) * kSortBlock;
  // every scratch word a kernel reads is written earlier in this sequence:
  // the prefix kernel writes the header and both tables, the sort kernel all
  // 2n keys (unique, padding included), and each merge pass writes a
  // permutation of its source; the single-block plan reads nothing it has
  // not written itself; so nothing needs clearing between calls
  if (n == kSortBlock) {  // each list one sort block: the whole plan in one launch
    plan_single_block_kernel<<<2, 1024, 0, stream>>>(p->cu_seqlens, p->n_seq, p->T, p->causal, sc->tile_prefix,
                                                      sc->blk_prefix, &sc->hdr, fwd_items, bwd_items);
  } else {
    plan_prefix_kernel<<<1, 1024, 0, stream>>>(p->cu_seqlens, p->n_seq, p->T, sc->tile_prefix, sc->blk_prefix,
                                              &sc->hdr);
    block_sort_kernel<<<2 * n / kSortBlock, 1024, 0, stream>>>(sc->tile_prefix, p->n_seq, p->causal, sc->keys_a, n,
                                                               &sc->hdr);
    uint64_t *src = sc->keys_a, *dst = sc->keys_b;
    for (int w = kSortBlock; w < n; w *= 2) {
      merge_pass_kernel<<<(2 * n + 255) / 256, 256, 0, stream>>>(src, dst, n, w);
      uint64_t* t = src;
      src = dst;
      dst = t;
    }
    plan_items_kernel<<<(2 * n + 255) / 256, 256, 0, stream>>>(src, sc->tile_prefix, p->n_seq, n, &sc->hdr,
                                                               fwd_items, bwd_items);
  }
  if (cudaMemcpyAsync(n_items, &sc->hdr.n_items, sizeof(int32_t), cudaMemcpyDeviceToDevice, stream) != cudaSuccess)
    return FLAMIA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? FLAMIA_OK : FLAMIA_ERR_CUDA;
}

