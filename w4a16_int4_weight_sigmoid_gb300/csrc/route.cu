// Sigmoid + bias top-k router: one warp per token, shuffle-based selection.
//
// Buffers: [Router] "코드 분석" (arg_plan: logits, bias, topk_weights,
// topk_ids).  The sigmoid is the fixed binary32 op sequence documented in
// chord_moe.h, written with explicitly rounded intrinsics (no contraction
// into FMA), so every implementation of the sequence returns the same bits.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace chord {
namespace {

// Constants derived from the mathematics: log2(e); ln 2 split into a head
// with 16 fractional bits (n * head is exact for |n| <= 126) and a tail;
// Taylor coefficients 1/j!.
__device__ __forceinline__ float sigmoid_spec(float x) {
  const float kLog2e = (float)(1.0 / 0.6931471805599453);
  const float kLn2Hi = 45426.0f / 65536.0f;
  const float kLn2Lo = (float)(0.6931471805599453 - 45426.0 / 65536.0);
  const float c0 = 1.0f, c1 = 1.0f, c2 = (float)(1.0 / 2.0), c3 = (float)(1.0 / 6.0),
              c4 = (float)(1.0 / 24.0), c5 = (float)(1.0 / 120.0), c6 = (float)(1.0 / 720.0),
              c7 = (float)(1.0 / 5040.0);
  float y = fminf(fmaxf(-x, -87.0f), 87.0f);
  float n = rintf(__fmul_rn(y, kLog2e));
  float r = __fsub_rn(y, __fmul_rn(n, kLn2Hi));
  r = __fsub_rn(r, __fmul_rn(n, kLn2Lo));
  float p = c7;
  p = __fadd_rn(__fmul_rn(p, r), c6);
  p = __fadd_rn(__fmul_rn(p, r), c5);
  p = __fadd_rn(__fmul_rn(p, r), c4);
  p = __fadd_rn(__fmul_rn(p, r), c3);
  p = __fadd_rn(__fmul_rn(p, r), c2);
  p = __fadd_rn(__fmul_rn(p, r), c1);
  p = __fadd_rn(__fmul_rn(p, r), c0);
  float e = __fmul_rn(p, __int_as_float((static_cast<int>(n) + 127) << 23));
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

// (key, id) order: larger key first; equal keys -> smaller id first.
__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

template <int EPL>
__global__ void __launch_bounds__(128) route_kernel(const float* __restrict__ logits,
                                                    const float* __restrict__ bias, int M, int E,
                                                    int topk, float* __restrict__ w_out,
                                                    int32_t* __restrict__ id_out) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= M) return;
  const float* row = logits + static_cast<size_t>(t) * E;
  float key[EPL], sc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      sc[i] = sigmoid_spec(__ldg(row + e));
      key[i] = __fadd_rn(sc[i], __ldg(bias + e));
    } else {
      sc[i] = 0.f;
      key[i] = -FLT_MAX;
    }
  }
  uint32_t taken = 0;
  int my_id = 0;
  float my_s = 0.f;
  for (int r = 0; r < topk; ++r) {
    float bk = -INFINITY;
    int bi = INT32_MAX;
    float bs = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u) && better(key[i], e, bk, bi)) {
        bk = key[i];
        bi = e;
        bs = sc[i];
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, bk, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      const float os = __shfl_xor_sync(0xffffffffu, bs, off);
      if (better(ok, oi, bk, bi)) {
        bk = ok;
        bi = oi;
        bs = os;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == r) {
      my_id = bi;
      my_s = bs;
    }
  }
  // S = s_0 + s_1 + ... in rank order, binary32.
  float S = __shfl_sync(0xffffffffu, my_s, 0);
  for (int r = 1; r < topk; ++r) S = __fadd_rn(S, __shfl_sync(0xffffffffu, my_s, r));
  if (lane < topk) {
    const size_t o = static_cast<size_t>(t) * topk + lane;
    id_out[o] = my_id;
    w_out[o] = __fdiv_rn(my_s, S);
  }
}

template <int EPL>
cudaError_t launch_route(const float* logits, const float* bias, int M, int E, int topk,
                         float* w, int32_t* ids, cudaStream_t st) {
  const int warps = 4;
  const int grid = (M + warps - 1) / warps;
  route_kernel<EPL><<<grid, warps * 32, 0, st>>>(logits, bias, M, E, topk, w, ids);
  return cudaGetLastError();
}

}  // namespace

cudaError_t route_launch(const float* logits, const float* bias, int M, int E, int topk, float* w,
                         int32_t* ids, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const int epl = (E + 31) / 32;
  if (epl <= 1) return launch_route<1>(logits, bias, M, E, topk, w, ids, st);
  if (epl <= 2) return launch_route<2>(logits, bias, M, E, topk, w, ids, st);
  if (epl <= 4) return launch_route<4>(logits, bias, M, E, topk, w, ids, st);
  if (epl <= 8) return launch_route<8>(logits, bias, M, E, topk, w, ids, st);
  if (epl <= 12) return launch_route<12>(logits, bias, M, E, topk, w, ids, st);
  if (epl <= 16) return launch_route<16>(logits, bias, M, E, topk, w, ids, st);
  return launch_route<32>(logits, bias, M, E, topk, w, ids, st);
}

}  // namespace chord
