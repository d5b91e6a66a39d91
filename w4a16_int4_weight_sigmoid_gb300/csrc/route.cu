// Sigmoid + bias top-k router: up to 512 tokens at top-k <= 8 a CTA of four
// warps per token, otherwise one warp per token; selection by warp
// reductions (the per-token code is in route_impl.cuh).
#include <cfloat>

#include "common.cuh"
#include "kernels.h"
#include "route_impl.cuh"

namespace chord {
namespace {

// Up to this many tokens the router is a programmatic launch (its launch
// overlaps the kernel before it; logits read with ordered loads after the
// wait): M = 1 3.38 -> 3.19 us, M = 128 3.87 -> 3.41 us per chained call on
// GB300 (one warp per token).  Above it, a plain launch with __ldg loads streams the logits
// faster (M = 4096: 10.4 us against 11.0 us with ordered loads).
constexpr int kChainedMaxM = 512;

template <int EPL, bool CHAINED>
__global__ void __launch_bounds__(128) route_kernel(const float* __restrict__ logits,
                                                    const float* __restrict__ bias, int M, int E,
                                                    int topk, float* __restrict__ w_out,
                                                    int32_t* __restrict__ id_out, int* zero, int n_zero) {
  grid_dep_wait();     // logits may come from the previous kernel (a no-op in a plain launch)
  grid_dep_launch();
  zero_ints(zero, n_zero);
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= M) return;
  route_token<EPL, CHAINED>(logits, bias, t, E, topk, w_out, id_out);
}

// Chained sizes with topk <= kCoopMaxTopk: one token per CTA, routed by its
// four warps together (one token by one warp spent ~5100 cycles on GB300:
// ~2000 computing the sigmoids of its 12 experts per lane with the loads,
// ~2450 in the top-8 rounds, ~570 on the weights).
template <int EPW>
__global__ void __launch_bounds__(kCoopWarps * 32) route_coop_kernel(const float* __restrict__ logits,
                                                                   const float* __restrict__ bias, int M, int E,
                                                                   int topk, float* __restrict__ w_out,
                                                                   int32_t* __restrict__ id_out, int* zero,
                                                                   int n_zero) {
  __shared__ CoopScratch cs;
  grid_dep_wait();     // logits may come from the previous kernel
  grid_dep_launch();
  zero_ints(zero, n_zero);
  route_token_coop<EPW>(logits, bias, blockIdx.x, E, topk, w_out, id_out, cs, threadIdx.x >> 5, 1);
}

template <int EPW>
cudaError_t launch_coop(const float* logits, const float* bias, int M, int E, int topk, float* w, int32_t* ids,
                        cudaStream_t st, int* zero, int n_zero) {
  return launch_kernel(route_coop_kernel<EPW>, dim3(M), dim3(kCoopWarps * 32), 0, st, true, logits, bias, M, E,
                       topk, w, ids, zero, n_zero);
}

template <int EPL>
cudaError_t launch_route(const float* logits, const float* bias, int M, int E, int topk,
                         float* w, int32_t* ids, cudaStream_t st, int* zero, int n_zero) {
  const int warps = 4;
  const int grid = (M + warps - 1) / warps;
  if (M <= kChainedMaxM)
    return launch_kernel(route_kernel<EPL, true>, dim3(grid), dim3(warps * 32), 0, st, true, logits, bias, M, E,
                         topk, w, ids, zero, n_zero);
  return launch_kernel(route_kernel<EPL, false>, dim3(grid), dim3(warps * 32), 0, st, false, logits, bias, M, E,
                       topk, w, ids, zero, n_zero);
}

}  // namespace

cudaError_t route_launch(const float* logits, const float* bias, int M, int E, int topk, float* w,
                         int32_t* ids, cudaStream_t st, int* zero, int n_zero) {
  if (M == 0) return cudaSuccess;
  if (M <= kChainedMaxM && topk <= kCoopMaxTopk) {
    const int epw = (E + 32 * kCoopWarps - 1) / (32 * kCoopWarps);
    if (epw <= 1) return launch_coop<1>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
    if (epw <= 2) return launch_coop<2>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
    if (epw <= 3) return launch_coop<3>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
    if (epw <= 4) return launch_coop<4>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
    return launch_coop<8>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
  }
  const int epl = (E + 31) / 32;
  if (epl <= 1) return launch_route<1>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
  if (epl <= 2) return launch_route<2>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
  if (epl <= 4) return launch_route<4>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
  if (epl <= 8) return launch_route<8>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
  if (epl <= 12) return launch_route<12>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
  if (epl <= 16) return launch_route<16>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
  return launch_route<32>(logits, bias, M, E, topk, w, ids, st, zero, n_zero);
}

}  // namespace chord
