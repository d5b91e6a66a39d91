// Sigmoid + bias top-k router: one warp per token, shuffle-based selection
// (the per-token code is in route_impl.cuh).
#include <cfloat>

#include "common.cuh"
#include "kernels.h"
#include "route_impl.cuh"

namespace chord {
namespace {

template <int EPL>
__global__ void __launch_bounds__(128) route_kernel(const float* __restrict__ logits,
                                                    const float* __restrict__ bias, int M, int E,
                                                    int topk, float* __restrict__ w_out,
                                                    int32_t* __restrict__ id_out, int* zero, int n_zero) {
  grid_dep_wait();     // logits may come from the previous kernel
  grid_dep_launch();
  zero_ints(zero, n_zero);
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= M) return;
  route_token<EPL>(logits, bias, t, E, topk, w_out, id_out);
}

template <int EPL>
cudaError_t launch_route(const float* logits, const float* bias, int M, int E, int topk,
                         float* w, int32_t* ids, cudaStream_t st, int* zero, int n_zero) {
  const int warps = 4;
  const int grid = (M + warps - 1) / warps;
  return launch_kernel(route_kernel<EPL>, dim3(grid), dim3(warps * 32), 0, st, true, logits, bias, M, E, topk,
                       w, ids, zero, n_zero);
}

}  // namespace

cudaError_t route_launch(const float* logits, const float* bias, int M, int E, int topk, float* w,
                         int32_t* ids, cudaStream_t st, int* zero, int n_zero) {
  if (M == 0) return cudaSuccess;
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
