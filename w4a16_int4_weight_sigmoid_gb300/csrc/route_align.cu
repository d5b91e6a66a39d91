// Fused router + align for the smallest batches (up to 16 tokens): one CTA
// routes every token (one warp per token, the router's own code), then,
// after a block barrier that
// makes its topk_ids writes visible to all its threads, runs the one-chunk
// stable counting sort over them.  One launch instead of two: [Router]
// "코드 분석" and "커널 내부 로직 변경" fuse routing and align (with counters
// re-initialised at entry) for the same reason -- at decode sizes both
// kernels are launch- and latency-bound.  Outputs are bit-identical to
// chord_moe_route followed by chord_moe_align.
#include "common.cuh"
#include "kernels.h"
#include "align_impl.cuh"
#include "route_impl.cuh"

namespace chord {
namespace {

struct RouteIn {
  const float* logits;
  const float* bias;
  int M, E, topk;
  float* w;
  int32_t* ids;
};

template <int EPL>
__global__ void __launch_bounds__(kThreads) route_align_kernel(RouteIn r, AlignArgs a) {
  extern __shared__ int s[];
  __shared__ int scan_scratch[kWarps + 1];
  const int warp = threadIdx.x >> 5;
  grid_dep_wait();
  grid_dep_launch();
  for (int t = warp; t < r.M; t += kWarps) route_token<EPL>(r.logits, r.bias, t, r.E, r.topk, r.w, r.ids);
  __syncthreads();   // this CTA's topk_ids stores are visible to all its threads
  int loc[kPerThread], rank[kPerThread];
  chunk_rank(a, 0, s, loc, rank);
  int* base = sm_base(s, a.E);
  for (int e = threadIdx.x; e < a.E; e += kThreads) base[e] = 0;
  __syncthreads();
  scatter_chunk(a, 0, s, loc, rank, scan_scratch);
}

template <int EPL>
cudaError_t launch_fused(const RouteIn& r, const AlignArgs& a, cudaStream_t st) {
  const size_t smem = align_smem_bytes(a.E);
  cudaError_t err = ensure_smem_limit<route_align_kernel<EPL>>(static_cast<int>(align_smem_bytes(1024)));
  if (err != cudaSuccess) return err;
  route_align_kernel<EPL><<<1, kThreads, smem, st>>>(r, a);
  return cudaGetLastError();
}

}  // namespace

// One CTA routes one token per warp: beyond kWarps tokens a warp would route
// several in turn and the separate router grid is faster.
bool route_align_fits(int M, long long assignments, int E_local) {
  return M <= kWarps && assignments <= kChunk && E_local >= 1 && E_local <= 1024;
}

cudaError_t route_align_launch(const float* logits, const float* bias, int M, int E_total, int topk,
                               int begin, int E_local, int bm, float* w, int32_t* ids, int32_t* sorted,
                               int32_t* expert_ids, int32_t* ntpp, int32_t* counts, int32_t* offsets,
                               int32_t* positions, cudaStream_t st) {
  if (!route_align_fits(M, static_cast<long long>(M) * topk, E_local)) return cudaErrorInvalidValue;
  RouteIn r{logits, bias, M, E_total, topk, w, ids};
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
  a.G = 1;
  a.ws_rank = nullptr;
  a.ws_counts = nullptr;
  const int epl = (E_total + 31) / 32;
  if (epl <= 1) return launch_fused<1>(r, a, st);
  if (epl <= 2) return launch_fused<2>(r, a, st);
  if (epl <= 4) return launch_fused<4>(r, a, st);
  if (epl <= 8) return launch_fused<8>(r, a, st);
  if (epl <= 12) return launch_fused<12>(r, a, st);
  if (epl <= 16) return launch_fused<16>(r, a, st);
  return launch_fused<32>(r, a, st);
}

}  // namespace chord
