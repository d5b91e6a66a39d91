// moe_align_block_size: stable counting sort of token->expert assignments.
//
// Buffers: [Router] "코드 분석" arg_plan (sorted_token_ids, expert_ids,
// num_tokens_post_padded, expert_counts, expert_offsets; the per-expert
// scatter cursors are re-initialised on entry as in "커널 내부 로직 변경").
//
// Each CTA owns a chunk of 4096 consecutive assignments; each of its 16
// warps owns 256 consecutive ones, walked in 8 steps of 32.  Within a step,
// __match_any_sync groups lanes with the same expert, the lowest lane of the
// group advances the warp's counter for that expert, and each lane's rank is
// the counter's old value plus the number of earlier lanes in its group.  An
// exclusive prefix over warps then turns per-warp ranks into chunk ranks that
// preserve the flat-index order.  One chunk: one launch does everything.
// More chunks: phase 1 writes chunk ranks and per-chunk counts to the
// workspace, phase 2 adds the prefix over chunks and scatters.
#include "common.cuh"
#include "kernels.h"

namespace chord {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = 8;
constexpr int kChunk = kThreads * kPerThread;  // 4096 assignments per CTA

struct AlignArgs {
  const int32_t* ids;
  int n, sentinel, begin, E, bm;
  int32_t *sorted, *expert_ids, *ntpp, *counts, *offsets, *positions;
  int32_t *ws_rank, *ws_counts;  // multi-chunk only
  int G;
};

// smem layout (ints): wcnt[kWarps][E] | tot[E] | base[E] | off[E+1]
__device__ __forceinline__ int* sm_wcnt(int* s) { return s; }
__device__ __forceinline__ int* sm_tot(int* s, int E) { return s + kWarps * E; }
__device__ __forceinline__ int* sm_base(int* s, int E) { return s + (kWarps + 1) * E; }
__device__ __forceinline__ int* sm_off(int* s, int E) { return s + (kWarps + 2) * E; }

__device__ __forceinline__ int elem_index(int g, int warp, int step, int lane) {
  return g * kChunk + warp * (32 * kPerThread) + step * 32 + lane;
}

// Per-chunk stable ranks; loc[] = local expert or -1; tot[e] = chunk count.
__device__ void chunk_rank(const AlignArgs& a, int g, int* s, int (&loc)[kPerThread],
                           int (&rank)[kPerThread]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  int* wcnt = sm_wcnt(s);
  for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int step = 0; step < kPerThread; ++step) {
    const int idx = elem_index(g, warp, step, lane);
    int e = -1;
    if (idx < a.n) {
      e = a.ids[idx] - a.begin;
      if (e < 0 || e >= E) e = -1;
    }
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (e >= 0 && lane == leader) {
      base = wcnt[warp * E + e];
      wcnt[warp * E + e] = base + __popc(peers);
    }
    base = __shfl_sync(0xffffffffu, base, leader);
    loc[step] = e;
    rank[step] = base + __popc(peers & lt);
  }
  __syncthreads();
  int* tot = sm_tot(s, E);
  for (int e = tid; e < E; e += kThreads) {
    int run = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
    tot[e] = run;
  }
  __syncthreads();
#pragma unroll
  for (int step = 0; step < kPerThread; ++step)
    if (loc[step] >= 0) rank[step] += wcnt[warp * E + loc[step]];
}

// Exclusive scan of in[0..n) into out[0..n] (out[n] = total); n <= 2*kThreads.
__device__ void block_exclusive_scan(const int* in, int* out, int n, int* scratch /*kWarps+1*/) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = 2 * tid;
  const int v0 = i0 < n ? in[i0] : 0;
  const int v1 = i0 + 1 < n ? in[i0 + 1] : 0;
  int sum = v0 + v1, inc = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? scratch[lane] : 0, wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < kWarps) scratch[lane] = wi - w;  // exclusive warp offsets
    if (lane == kWarps - 1) scratch[kWarps] = wi;
  }
  __syncthreads();
  const int ex = scratch[warp] + inc - sum;
  if (i0 < n) out[i0] = ex;
  if (i0 + 1 < n) out[i0 + 1] = ex + v0;
  if (tid == 0) out[n] = scratch[kWarps];
  __syncthreads();
}

// Given tot (all-chunk counts) and base (this chunk's start per expert):
// offsets, scatter, metadata.
__device__ void scatter_chunk(const AlignArgs& a, int g, int* s, const int (&loc)[kPerThread],
                              const int (&rank)[kPerThread], int* scan_scratch) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, bm = a.bm;
  int* tot = sm_tot(s, E);
  int* base = sm_base(s, E);
  int* off = sm_off(s, E);
  // padded counts into wcnt's space (no longer needed), then scan into off
  int* pad = sm_wcnt(s);
  for (int e = tid; e < E; e += kThreads) pad[e] = (tot[e] + bm - 1) / bm * bm;
  __syncthreads();
  block_exclusive_scan(pad, off, E, scan_scratch);
#pragma unroll
  for (int step = 0; step < kPerThread; ++step) {
    const int idx = elem_index(g, warp, step, lane);
    if (idx >= a.n) continue;
    const int e = loc[step];
    if (e >= 0) {
      const int pos = off[e] + base[e] + rank[step];
      a.sorted[pos] = idx;
      if (a.positions) a.positions[idx] = pos;
    } else if (a.positions) {
      a.positions[idx] = -1;
    }
  }
  // metadata, spread over the chunks' CTAs
  for (int e = tid; e < E; e += kThreads) {
    if (e % a.G != g) continue;
    a.counts[e] = tot[e];
    a.offsets[e] = off[e];
    for (int p = off[e] + tot[e]; p < off[e + 1]; ++p) a.sorted[p] = a.sentinel;
  }
  const int total = off[E];
  const int nblk = total / bm;
  for (int b = g * kThreads + tid; b < nblk; b += a.G * kThreads) {
    const int row = b * bm;
    int lo = 0, hi = E - 1;  // largest e with off[e] <= row
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (off[mid] <= row) lo = mid; else hi = mid - 1;
    }
    a.expert_ids[b] = lo;
  }
  if (g == 0 && tid == 0) {
    a.offsets[E] = total;
    a.ntpp[0] = total;
  }
}

__global__ void __launch_bounds__(kThreads) align_single_kernel(AlignArgs a) {
  extern __shared__ int s[];
  __shared__ int scan_scratch[kWarps + 1];
  int loc[kPerThread], rank[kPerThread];
  chunk_rank(a, 0, s, loc, rank);
  int* base = sm_base(s, a.E);
  for (int e = threadIdx.x; e < a.E; e += kThreads) base[e] = 0;
  __syncthreads();
  scatter_chunk(a, 0, s, loc, rank, scan_scratch);
}

__global__ void __launch_bounds__(kThreads) align_rank_kernel(AlignArgs a) {
  extern __shared__ int s[];
  const int g = blockIdx.x;
  int loc[kPerThread], rank[kPerThread];
  chunk_rank(a, g, s, loc, rank);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int step = 0; step < kPerThread; ++step) {
    const int idx = elem_index(g, warp, step, lane);
    if (idx < a.n) a.ws_rank[idx] = rank[step];
  }
  int* tot = sm_tot(s, a.E);
  for (int e = threadIdx.x; e < a.E; e += kThreads) a.ws_counts[g * a.E + e] = tot[e];
}

__global__ void __launch_bounds__(kThreads) align_scatter_kernel(AlignArgs a) {
  extern __shared__ int s[];
  __shared__ int scan_scratch[kWarps + 1];
  const int g = blockIdx.x, E = a.E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* tot = sm_tot(s, E);
  int* base = sm_base(s, E);
  for (int e = threadIdx.x; e < E; e += kThreads) {
    int t = 0, b = 0;
    for (int gg = 0; gg < a.G; ++gg) {
      const int c = a.ws_counts[gg * E + e];
      if (gg < g) b += c;
      t += c;
    }
    tot[e] = t;
    base[e] = b;
  }
  int loc[kPerThread], rank[kPerThread];
#pragma unroll
  for (int step = 0; step < kPerThread; ++step) {
    const int idx = elem_index(g, warp, step, lane);
    loc[step] = -1;
    rank[step] = 0;
    if (idx < a.n) {
      int e = a.ids[idx] - a.begin;
      if (e >= 0 && e < E) {
        loc[step] = e;
        rank[step] = a.ws_rank[idx];
      }
    }
  }
  __syncthreads();
  scatter_chunk(a, g, s, loc, rank, scan_scratch);
}

size_t align_smem_bytes(int E) { return static_cast<size_t>((kWarps + 3) * E + 1) * sizeof(int); }

}  // namespace

int align_num_chunks(long long n) { return n <= kChunk ? 1 : static_cast<int>((n + kChunk - 1) / kChunk); }

size_t align_workspace_bytes(long long n, int E_local) {
  const int G = align_num_chunks(n);
  if (G == 1) return 0;
  return static_cast<size_t>(n + static_cast<long long>(G) * E_local) * sizeof(int32_t);
}

cudaError_t align_launch(const int32_t* ids, int M, int topk, int begin, int E_local, int bm,
                         int32_t* sorted, int32_t* expert_ids, int32_t* ntpp, int32_t* counts,
                         int32_t* offsets, int32_t* positions, void* ws, cudaStream_t st) {
  AlignArgs a;
  a.ids = ids;
  a.n = M * topk;
  a.sentinel = M * topk;
  a.begin = begin;
  a.E = E_local;
  a.bm = bm;
  a.sorted = sorted;
  a.expert_ids = expert_ids;
  a.ntpp = ntpp;
  a.counts = counts;
  a.offsets = offsets;
  a.positions = positions;
  a.G = align_num_chunks(a.n);
  a.ws_rank = static_cast<int32_t*>(ws);
  a.ws_counts = a.ws_rank ? a.ws_rank + a.n : nullptr;
  const size_t smem = align_smem_bytes(E_local);
  const int max_smem = static_cast<int>(align_smem_bytes(1024));
  cudaError_t err = ensure_smem_limit<align_single_kernel>(max_smem);
  if (err == cudaSuccess) err = ensure_smem_limit<align_rank_kernel>(max_smem);
  if (err == cudaSuccess) err = ensure_smem_limit<align_scatter_kernel>(max_smem);
  if (err != cudaSuccess) return err;
  if (a.G == 1) {
    align_single_kernel<<<1, kThreads, smem, st>>>(a);
    return cudaGetLastError();
  }
  align_rank_kernel<<<a.G, kThreads, smem, st>>>(a);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  align_scatter_kernel<<<a.G, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace chord

// ---------------------------------------------------------------------------
// Allocation-free align: the scratch of the multi-chunk path (per-assignment
// chunk ranks, then per-chunk expert counts) lives in this file-scope device
// array instead of a caller-provided workspace.  Every GPU that loads the
// library holds it (320 KiB) until the process exits.
namespace chord {

constexpr long long kNoAllocMaxAssignments = CHORD_ALIGN_NOALLOC_MAX_ASSIGNMENTS;
constexpr int kNoAllocMaxExperts = CHORD_ALIGN_NOALLOC_MAX_EXPERTS;
constexpr long long kNoAllocScratchInts =
    kNoAllocMaxAssignments +
    ((kNoAllocMaxAssignments + kChunk - 1) / kChunk) * static_cast<long long>(kNoAllocMaxExperts);

static __device__ __align__(256) int32_t g_align_scratch[kNoAllocScratchInts];

namespace {
// Device address of g_align_scratch, looked up once per device.  In host code
// the symbol name is only a host-side stand-in, so it is never passed to a
// kernel directly.
void* g_scratch_ptr[64] = {nullptr};
}  // namespace

cudaError_t align_noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_align_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = p;
  }
  *ptr = g_scratch_ptr[dev];
  return cudaSuccess;
}

size_t align_noalloc_scratch_bytes() { return static_cast<size_t>(kNoAllocScratchInts) * sizeof(int32_t); }

}  // namespace chord
