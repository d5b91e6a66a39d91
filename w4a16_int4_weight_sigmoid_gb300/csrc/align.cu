// moe_align_block_size: stable counting sort of token->expert assignments
// (device code in align_impl.cuh).  One chunk of up to 4096 assignments: one
// launch does everything.  More chunks: phase 1 writes chunk ranks and
// per-chunk counts to the workspace, phase 2 adds the prefix over chunks and
// scatters.
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "align_impl.cuh"

namespace chord {
namespace {

template <int PER>
__global__ void __launch_bounds__(kThreads) align_single_kernel(AlignArgs a) {
  extern __shared__ int s[];
  __shared__ int scan_scratch[kWarps + 1];
  int loc[PER], rank[PER];
  grid_dep_wait();     // topk_ids come from the router kernel
  grid_dep_launch();
  chunk_rank<PER>(a, 0, s, loc, rank);
  int* base = sm_base(s, a.E);
  for (int e = threadIdx.x; e < a.E; e += kThreads) base[e] = 0;
  __syncthreads();
  scatter_chunk<PER>(a, 0, s, loc, rank, scan_scratch);
}

template <int PER>
__global__ void __launch_bounds__(kThreads) align_rank_kernel(AlignArgs a) {
  extern __shared__ int s[];
  const int g = blockIdx.x;
  int loc[PER], rank[PER];
  grid_dep_wait();
  grid_dep_launch();
  chunk_rank<PER>(a, g, s, loc, rank);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
  for (int step = 0; step < PER; ++step) {
    const int idx = elem_index<PER>(g, warp, step, lane);
    if (idx < a.n) a.ws_rank[idx] = rank[step];
  }
  int* tot = sm_tot(s, a.E);
  for (int e = threadIdx.x; e < a.E; e += kThreads) a.ws_counts[g * a.E + e] = tot[e];
}

template <int PER>
__global__ void __launch_bounds__(kThreads) align_scatter_kernel(AlignArgs a) {
  extern __shared__ int s[];
  __shared__ int scan_scratch[kWarps + 1];
  const int g = blockIdx.x, E = a.E;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  grid_dep_wait();
  grid_dep_launch();
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
  int loc[PER], rank[PER];
#pragma unroll
  for (int step = 0; step < PER; ++step) {
    const int idx = elem_index<PER>(g, warp, step, lane);
    loc[step] = -1;
    rank[step] = 0;
    if (idx < a.n) {
      int e = ld_cg(a.ids + idx) - a.begin;
      if (e >= 0 && e < E) {
        loc[step] = e;
        rank[step] = a.ws_rank[idx];
      }
    }
  }
  __syncthreads();
  scatter_chunk<PER>(a, g, s, loc, rank, scan_scratch);
}


}  // namespace

int align_num_chunks(long long n) {
  return n <= kChunk ? 1 : static_cast<int>((n + kMultiChunk - 1) / kMultiChunk);
}

size_t align_workspace_bytes(long long n, int E_local) {
  const int G = align_num_chunks(n);
  if (G == 1) return 0;
  return static_cast<size_t>(n + static_cast<long long>(G) * E_local) * sizeof(int32_t);
}

cudaError_t align_launch(const int32_t* ids, int M, int topk, int begin, int E_local, int bm,
                         int32_t* sorted, int32_t* expert_ids, int32_t* ntpp, int32_t* counts,
                         int32_t* offsets, int32_t* positions, void* ws, cudaStream_t st, bool pdl) {
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
  cudaError_t err = ensure_smem_limit<align_single_kernel<1>>(max_smem);
  if (err == cudaSuccess) err = ensure_smem_limit<align_single_kernel<2>>(max_smem);
  if (err == cudaSuccess) err = ensure_smem_limit<align_single_kernel<kPerThread>>(max_smem);
  if (err == cudaSuccess) err = ensure_smem_limit<align_rank_kernel<kMultiPer>>(max_smem);
  if (err == cudaSuccess) err = ensure_smem_limit<align_scatter_kernel<kMultiPer>>(max_smem);
  if (err != cudaSuccess) return err;
  if (a.G == 1) {
    switch (align_per_thread(a.n)) {
      case 1: return launch_kernel(align_single_kernel<1>, dim3(1), dim3(kThreads), smem, st, pdl, a);
      case 2: return launch_kernel(align_single_kernel<2>, dim3(1), dim3(kThreads), smem, st, pdl, a);
      default: return launch_kernel(align_single_kernel<kPerThread>, dim3(1), dim3(kThreads), smem, st, pdl, a);
    }
  }
  err = launch_kernel(align_rank_kernel<kMultiPer>, dim3(a.G), dim3(kThreads), smem, st, pdl, a);
  if (err != cudaSuccess) return err;
  align_scatter_kernel<kMultiPer><<<a.G, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace chord

// ---------------------------------------------------------------------------
// Allocation-free align: the scratch of the multi-chunk path (per-assignment
// chunk ranks, then per-chunk expert counts) lives in this file-scope device
// array instead of a caller-provided workspace.  Every GPU that loads the
// library holds it (512 KiB) until the process exits.
namespace chord {

constexpr long long kNoAllocMaxAssignments = CHORD_ALIGN_NOALLOC_MAX_ASSIGNMENTS;
constexpr int kNoAllocMaxExperts = CHORD_ALIGN_NOALLOC_MAX_EXPERTS;
constexpr long long kNoAllocScratchInts =
    kNoAllocMaxAssignments +
    ((kNoAllocMaxAssignments + kMultiChunk - 1) / kMultiChunk) * static_cast<long long>(kNoAllocMaxExperts);

static __device__ __align__(256) int32_t g_align_scratch[kNoAllocScratchInts];

namespace {
// Device address of g_align_scratch, looked up once per device.  In host code
// the symbol name is only a host-side stand-in, so it is never passed to a
// kernel directly.  Atomic: host threads making their first call on a device
// at the same time may both look it up; they store the same address.
std::atomic<void*> g_scratch_ptr[64];
}  // namespace

cudaError_t align_noalloc_scratch(void** ptr) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    // With lazy module loading this lookup may be what loads the module and
    // reserves the array on this device.
    err = cudaGetSymbolAddress(&p, g_align_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *ptr = p;
  return cudaSuccess;
}

size_t align_noalloc_scratch_bytes() { return static_cast<size_t>(kNoAllocScratchInts) * sizeof(int32_t); }

}  // namespace chord
