// moe_align_block_size device code shared by the align kernels and the
// fused route+align kernel: a stable counting sort of token->expert
// assignments.
//
// Buffers: [Router] "코드 분석" arg_plan (sorted_token_ids, expert_ids,
// num_tokens_post_padded, expert_counts, expert_offsets; the per-expert
// scatter cursors are re-initialised on entry as in "커널 내부 로직 변경").
//
// Each CTA owns a chunk of 512 * PER consecutive assignments; each of its 16
// warps owns 32 * PER consecutive ones, walked in PER steps of 32.  One CTA
// aligns up to 4096 assignments alone (PER = 1, 2 or 8 for at most 512,
// 1024 or 4096); above that the assignments are split into chunks of 1024
// (PER = 2), one CTA each, in two phases.  Within a step,
// __match_any_sync groups lanes with the same expert, the lowest lane of the
// group advances the warp's counter for that expert, and each lane's rank is
// the counter's old value plus the number of earlier lanes in its group.  An
// exclusive prefix over warps then turns per-warp ranks into chunk ranks that
// preserve the flat-index order.
#pragma once

#include "common.cuh"

namespace chord {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = 8;
constexpr int kChunk = kThreads * kPerThread;  // 4096: the most one CTA aligns alone
// Above kChunk assignments the align runs in chunks of kThreads * kMultiPer
// (1024) over as many CTAs: more CTAs, each with fewer serial steps.
constexpr int kMultiPer = 2;
constexpr int kMultiChunk = kThreads * kMultiPer;

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

template <int PER = kPerThread>
__device__ __forceinline__ int elem_index(int g, int warp, int step, int lane) {
  return g * (kThreads * PER) + warp * (32 * PER) + step * 32 + lane;
}

// Elements per thread of a one-chunk align of n assignments.
__host__ __device__ constexpr int align_per_thread(long long n) {
  return n <= kThreads ? 1 : (n <= 2 * kThreads ? 2 : kPerThread);
}

// Per-chunk stable ranks; loc[] = local expert or -1; tot[e] = chunk count.
template <int PER = kPerThread>
__device__ void chunk_rank(const AlignArgs& a, int g, int* s, int (&loc)[PER], int (&rank)[PER]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  int* wcnt = sm_wcnt(s);
  for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  // All of this thread's ids are loaded before any is ranked, so the loads
  // are in flight together (ordered L2 loads: the ids may come from the
  // preceding kernel).
  int eid[PER];
#pragma unroll
  for (int step = 0; step < PER; ++step) {
    const int idx = elem_index<PER>(g, warp, step, lane);
    eid[step] = idx < a.n ? ld_cg(a.ids + idx) : a.begin - 1;
  }
#pragma unroll
  for (int step = 0; step < PER; ++step) {
    int e = eid[step] - a.begin;
    if (e < 0 || e >= E) e = -1;
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
  if (E <= 4 * kWarps) {
    // few experts: one warp per expert column, the 16 warp counts scanned
    // across lanes (five shuffles) instead of a 16-step loop per thread
    for (int e = warp; e < E; e += kWarps) {
      const int c = lane < kWarps ? wcnt[lane * E + e] : 0;
      int inc = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (lane < kWarps) wcnt[lane * E + e] = inc - c;
      if (lane == 31) tot[e] = inc;
    }
  } else {
    for (int e = tid; e < E; e += kThreads) {
      int run = 0;
      for (int w = 0; w < kWarps; ++w) {
        const int c = wcnt[w * E + e];
        wcnt[w * E + e] = run;
        run += c;
      }
      tot[e] = run;
    }
  }
  __syncthreads();
#pragma unroll
  for (int step = 0; step < PER; ++step)
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
template <int PER = kPerThread>
__device__ void scatter_chunk(const AlignArgs& a, int g, int* s, const int (&loc)[PER],
                              const int (&rank)[PER], int* scan_scratch) {
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
  for (int step = 0; step < PER; ++step) {
    const int idx = elem_index<PER>(g, warp, step, lane);
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
  // expert e's metadata and padding by chunk e % G
  for (int e = g + a.G * tid; e < E; e += a.G * kThreads) {
    a.counts[e] = tot[e];
    a.offsets[e] = off[e];
    if (bm <= 32)   // short padding: one thread per expert
      for (int p = off[e] + tot[e]; p < off[e + 1]; ++p) a.sorted[p] = a.sentinel;
  }
  if (bm > 32) {
    // up to 127 slots: one warp per expert, lanes on consecutive slots, so
    // the sentinel stores coalesce.  The experts that have padding (at most
    // one per assignment) are listed first, so the warps do not walk the
    // ones without (384 experts cost 24 steps a warp otherwise).
    __shared__ int s_npad;
    int* list = sm_wcnt(s) + E;   // after the padded counts, in the per-warp counts' space
    if (tid == 0) s_npad = 0;
    __syncthreads();
    for (int e = g + a.G * tid; e < E; e += a.G * kThreads)
      if (off[e] + tot[e] < off[e + 1]) list[atomicAdd(&s_npad, 1)] = e;
    __syncthreads();
    const int np = s_npad;
    for (int k = warp; k < np; k += kWarps) {
      const int e = list[k];
      for (int p = off[e] + tot[e] + lane; p < off[e + 1]; p += 32) a.sorted[p] = a.sentinel;
    }
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

// Dynamic shared memory of a one-chunk align over E experts.
inline size_t align_smem_bytes(int E) { return static_cast<size_t>((kWarps + 3) * E + 1) * sizeof(int); }

}  // namespace
}  // namespace chord
