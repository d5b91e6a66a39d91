// Sigmoid + bias top-k routing of one token by one warp, or by a group of
// four warps (device code shared by the router kernel and the fused
// route+align kernel).
//
// Buffers: [Router] "코드 분석" (arg_plan: logits, bias, topk_weights,
// topk_ids).  The sigmoid is the fixed binary32 op sequence documented in
// chord_moe.h, written with explicitly rounded intrinsics (no contraction
// into FMA), so every implementation of the sequence returns the same bits.
#pragma once

#include "common.cuh"

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

// (key, id) as one integer whose order is the selection order: the key's
// bits mapped to an order-preserving unsigned (keys are never -0.0: s > 0 and
// s + b rounds x + (-x) to +0), then the complement of the id, so among equal
// keys the smaller id compares larger.
__device__ __forceinline__ uint64_t pack_key(float key, int id) {
  const uint32_t b = __float_as_uint(key);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(id));
}

// Route token t with the calling (whole, converged) warp: EPL experts per
// lane (e = lane + 32 i); writes topk_ids / topk_weights row t and returns,
// in lanes 0 .. topk-1, the id of that rank.  ORDERED: the caller is a
// programmatic launch (see grid_dep_wait), so logits and bias are read with
// ordered loads after its wait instead of __ldg.
template <int EPL, bool ORDERED>
__device__ __forceinline__ int route_token(const float* __restrict__ logits, const float* __restrict__ bias,
                                            int t, int E, int topk, float* __restrict__ w_out,
                                            int32_t* __restrict__ id_out) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + static_cast<size_t>(t) * E;
  // All loads first (clamped in-range addresses, no branches), so they are in
  // flight together instead of one round trip per expert (ordered: the bias,
  // which every warp reads, through L1).
  float lg[EPL], bs[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = min(lane + 32 * i, E - 1);
    lg[i] = ORDERED ? ld_cg(row + e) : __ldg(row + e);
    bs[i] = ORDERED ? ld_ca(bias + e) : __ldg(bias + e);
  }
  uint64_t cand[EPL];
  float sc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    sc[i] = sigmoid_spec(lg[i]);
    cand[i] = e < E ? pack_key(__fadd_rn(sc[i], bs[i]), e) : 0;  // 0: below every candidate
  }
  int my_id = 0;
  float my_s = 0.f;
  for (int r = 0; r < topk; ++r) {
    uint64_t best = cand[0];
#pragma unroll
    for (int i = 1; i < EPL; ++i) best = cand[i] > best ? cand[i] : best;
    // warp maximum of the 64-bit keys in two 32-bit reductions: the largest
    // key word, then the largest id word among the lanes holding that key
    // (the id word is never 0, so 0 stands for "not a holder")
    const uint32_t hi = static_cast<uint32_t>(best >> 32);
    const uint32_t top_hi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t top_lo =
        __reduce_max_sync(0xffffffffu, hi == top_hi ? static_cast<uint32_t>(best) : 0u);
    const int id = static_cast<int>(0xFFFFFFFFu - top_lo);
    const int owner = id & 31, slot = id >> 5;
    float s_mine = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      if (i == slot) {
        s_mine = sc[i];
        if (lane == owner) cand[i] = 0;
      }
    }
    const float s_win = __shfl_sync(0xffffffffu, s_mine, owner);
    if (lane == r) {
      my_id = id;
      my_s = s_win;
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
  return my_id;
}

// One token routed by a group of kCoopWarps warps (kCoopWarps * 32 threads):
// warp gw of the group holds experts e = 32 gw + lane + 128 i (EPW per lane,
// 128 EPW >= E), takes the top-k of its own experts by the same rounds as
// route_token (any of the token's top-k is in its warp's top-k), and writes
// them to shared memory; after a barrier the group's warp 0 ranks the
// kCoopWarps * topk candidates, one per lane, by counting the larger keys
// of the other lanes (keys of real
// experts are distinct; key 0 marks no candidate).  Same outputs, bit for
// bit, as route_token; a quarter of the sigmoids and shorter maxima per
// warp.  topk <= kCoopMaxTopk.  bar: named barrier of the group (128
// threads).  Returns, in lanes 0 .. topk-1 of the group's warp 0, the id of
// that rank (other warps: -1).  Ordered loads: the callers are programmatic
// launches (see grid_dep_wait).
constexpr int kCoopWarps = 4, kCoopMaxTopk = 8;
struct CoopScratch {
  unsigned long long key[kCoopWarps * kCoopMaxTopk];
  float s[kCoopWarps * kCoopMaxTopk];
  int id[kCoopMaxTopk];
  float ws[kCoopMaxTopk];
};
template <int EPW>
__device__ __forceinline__ int route_token_coop(const float* __restrict__ logits, const float* __restrict__ bias,
                                                 int t, int E, int topk, float* __restrict__ w_out,
                                                 int32_t* __restrict__ id_out, CoopScratch& cs, int gw, int bar) {
  const int lane = threadIdx.x & 31;
  const float* row = logits + static_cast<size_t>(t) * E;
  float lg[EPW], bs[EPW];
#pragma unroll
  for (int i = 0; i < EPW; ++i) {
    const int e = min(32 * gw + lane + 128 * i, E - 1);
    lg[i] = ld_cg(row + e);
    bs[i] = ld_ca(bias + e);
  }
  uint64_t cand[EPW];
  float sc[EPW];
#pragma unroll
  for (int i = 0; i < EPW; ++i) {
    const int e = 32 * gw + lane + 128 * i;
    sc[i] = sigmoid_spec(lg[i]);
    cand[i] = e < E ? pack_key(__fadd_rn(sc[i], bs[i]), e) : 0;
  }
  for (int r = 0; r < topk; ++r) {
    uint64_t best = cand[0];
#pragma unroll
    for (int i = 1; i < EPW; ++i) best = cand[i] > best ? cand[i] : best;
    const uint32_t hi = static_cast<uint32_t>(best >> 32);
    const uint32_t top_hi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t top_lo =
        __reduce_max_sync(0xffffffffu, hi == top_hi ? static_cast<uint32_t>(best) : 0u);
    const int id = static_cast<int>(0xFFFFFFFFu - top_lo);
    const int owner = id & 31, slot = id >> 7;   // e = 32 gw + owner + 128 slot
    float s_mine = 0.f;
#pragma unroll
    for (int i = 0; i < EPW; ++i) {
      if (i == slot) {
        s_mine = sc[i];
        if (lane == owner) cand[i] = 0;
      }
    }
    const float s_win = __shfl_sync(0xffffffffu, s_mine, owner);
    if (lane == 0) {
      cs.key[gw * topk + r] = (static_cast<uint64_t>(top_hi) << 32) | top_lo;
      cs.s[gw * topk + r] = s_win;
    }
  }
  asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kCoopWarps * 32) : "memory");
  if (gw != 0) return -1;
  const int nc = kCoopWarps * topk;
  const uint64_t mine = lane < nc ? cs.key[lane] : 0;
  int rank = 0;   // from registers: independent shuffles (a loop over shared memory took ~740 cycles)
#pragma unroll
  for (int m = 0; m < kCoopWarps * kCoopMaxTopk; ++m) {
    const uint64_t other = __shfl_sync(0xffffffffu, mine, m);   // 0 past the candidates
    rank += other > mine ? 1 : 0;
  }
  if (lane < nc && mine != 0 && rank < topk) {
    cs.id[rank] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(mine));
    cs.ws[rank] = cs.s[lane];
  }
  __syncwarp();
  // S = s_0 + s_1 + ... in rank order, binary32
  float S = cs.ws[0];
  for (int r = 1; r < topk; ++r) S = __fadd_rn(S, cs.ws[r]);
  int my_id = 0;
  if (lane < topk) {
    my_id = cs.id[lane];
    const size_t o = static_cast<size_t>(t) * topk + lane;
    id_out[o] = my_id;
    w_out[o] = __fdiv_rn(cs.ws[lane], S);
  }
  return my_id;
}

}  // namespace
}  // namespace chord
