// Fused router + align for small batches (up to 4 tokens at top-k <= 8, up to
// 16 above): one CTA routes every token (four warps a token, or one warp a
// token above top-8, the router's own code), then, after a block barrier
// that makes its topk_ids writes visible to all its threads, runs the
// one-chunk stable sort over them.  One launch instead of two: [Router]
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
  int* zero;     // ints to clear for the kernels after this one (or NULL)
  int n_zero;
};

template <int EPL, int PER>
__global__ void __launch_bounds__(kThreads) route_align_kernel(RouteIn r, AlignArgs a) {
  extern __shared__ int s[];
  __shared__ int scan_scratch[kWarps + 1];
  const int warp = threadIdx.x >> 5;
  grid_dep_wait();
  grid_dep_launch();
  zero_ints(r.zero, r.n_zero);
  for (int t = warp; t < r.M; t += kWarps) route_token<EPL, true>(r.logits, r.bias, t, r.E, r.topk, r.w, r.ids);
  __syncthreads();   // this CTA's topk_ids stores are visible to all its threads
  int loc[PER], rank[PER];
  chunk_rank<PER>(a, 0, s, loc, rank);
  int* base = sm_base(s, a.E);
  for (int e = threadIdx.x; e < a.E; e += kThreads) base[e] = 0;
  __syncthreads();
  scatter_chunk<PER>(a, 0, s, loc, rank, scan_scratch);
}

// The smallest batches (M * topk <= 32 assignments, e.g. one decode token at
// top-8): one small CTA without the general align's per-warp tables.  Up to
// kTinyCoopTokens tokens at topk <= kCoopMaxTopk, four warps route each token
// together (EPW > 0: route_token_coop); otherwise warp t routes token t.  The
// ids are kept in shared memory as well as written out; warp 0 then holds
// assignment f in lane f and ranks the assignments by ballots of the expert
// ids' bits (no shared-memory table walk: __match_any_sync and a 32-step
// loop took ~1400 cycles on GB300), writing the present experts' table; the
// whole CTA then fills padding, block map, counts and offsets in one pass
// over that table (a binary search per expert took ~2500 cycles).  Outputs
// are those of the general kernels.
constexpr int kTinyWarps = 4, kTinyMaxWarps = 8, kTinyCoopTokens = 4;
template <int EPL, int EPW>
__global__ void __launch_bounds__(EPW > 0 ? 32 * kCoopWarps * kTinyCoopTokens : 32 * kTinyMaxWarps)
route_align_tiny_kernel(RouteIn r, AlignArgs a) {
  __shared__ int s_id[32];                          // routed expert of assignment f
  __shared__ int t_e[32], t_end[32], t_cnt[32];     // present experts in id order
  __shared__ int s_nlead;
  __shared__ CoopScratch s_coop[EPW > 0 ? kTinyCoopTokens : 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  grid_dep_wait();
  grid_dep_launch();
  zero_ints(r.zero, r.n_zero);
  if (EPW > 0) {   // blockDim = 32 kCoopWarps M: group g of four warps routes token g
    const int g = warp / kCoopWarps, gw = warp % kCoopWarps;
    const int id = route_token_coop<(EPW > 0 ? EPW : 1)>(r.logits, r.bias, g, r.E, r.topk, r.w, r.ids, s_coop[g],
                                                      gw, 1 + g);
    if (gw == 0 && lane < r.topk) s_id[g * r.topk + lane] = id;
  } else {
    for (int t = warp; t < r.M; t += nw) {
      const int id = route_token<EPL, true>(r.logits, r.bias, t, r.E, r.topk, r.w, r.ids);
      if (lane < r.topk) s_id[t * r.topk + lane] = id;
    }
  }
  __syncthreads();
  const int n = a.n, bm = a.bm, E = a.E;
  if (warp == 0) {
    // Assignment f in lane f.  From ballots of the expert id's bits, high to
    // low (E <= 1024): eq = the lanes holding my expert, lt = the lanes
    // holding a smaller one (stable rank = my place among eq).
    int e = lane < n ? s_id[lane] - a.begin : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = 0;
    uint32_t lt = 0, eq = __ballot_sync(0xffffffffu, valid);
#pragma unroll
    for (int b = 9; b >= 0; --b) {
      const bool bit = (e >> b) & 1;
      const uint32_t ones = __ballot_sync(0xffffffffu, valid && bit);
      if (bit) {
        lt |= eq & ~ones;
        eq &= ones;
      } else {
        eq &= ~ones;
      }
    }
    const int cnt = __popc(eq);
    const bool lead = valid && lane == __ffs(eq) - 1;
    const int nb = lead ? (cnt + bm - 1) / bm : 0;   // blocks of my expert (<= 4: n <= 32, bm >= 8)
    const uint32_t leaders = __ballot_sync(0xffffffffu, lead);
    // blocks of the experts below mine, and of all, summed from their bits
    int below_blocks = 0, all_blocks = 0;
#pragma unroll
    for (int b = 0; b < 3; ++b) {
      const uint32_t bits = __ballot_sync(0xffffffffu, (nb >> b) & 1);
      below_blocks += __popc(bits & lt) << b;
      all_blocks += __popc(bits) << b;
    }
    const int off = below_blocks * bm;
    if (lane < n) {
      if (valid) {
        const int pos = off + __popc(eq & ((1u << lane) - 1u));
        a.sorted[pos] = lane;
        if (a.positions) a.positions[lane] = pos;
      } else if (a.positions) {
        a.positions[lane] = -1;
      }
    }
    if (lead) {   // the present experts in id order
      const int k = __popc(lt & leaders);
      t_e[k] = e;
      t_end[k] = off + nb * bm;
      t_cnt[k] = cnt;
    }
    if (lane == 0) {
      s_nlead = __popc(leaders);
      a.ntpp[0] = all_blocks * bm;
    }
  }
  __syncthreads();
  // The whole CTA, one pass over the present experts: each one's padding
  // rows and blocks (at most 127 and 4, blockDim >= 128), and for the
  // thread's experts x the count and the padded rows below x.
  const int nlead = s_nlead, bd = blockDim.x, tid = threadIdx.x;
  constexpr int kMaxX = (1024 + 1 + 127) / 128;   // experts per thread at E <= 1024, blockDim >= 128
  int xoff[kMaxX], xcnt[kMaxX];
#pragma unroll
  for (int j = 0; j < kMaxX; ++j) xoff[j] = xcnt[j] = 0;
  int start = 0;
  for (int k = 0; k < nlead; ++k) {
    const int ek = t_e[k], endk = t_end[k], ck = t_cnt[k];
#pragma unroll
    for (int j = 0; j < kMaxX; ++j) {
      const int x = tid + j * bd;
      if (ek < x) xoff[j] = endk;
      if (ek == x) xcnt[j] = ck;
    }
    if (start + ck + tid < endk) a.sorted[start + ck + tid] = a.sentinel;
    if (start / bm + tid < endk / bm) a.expert_ids[start / bm + tid] = ek;
    start = endk;
  }
#pragma unroll
  for (int j = 0; j < kMaxX; ++j) {
    const int x = tid + j * bd;
    if (x <= E) a.offsets[x] = xoff[j];
    if (x < E) a.counts[x] = xcnt[j];
  }
}

template <int EPL>
cudaError_t launch_tiny(const RouteIn& r, const AlignArgs& a, cudaStream_t st) {
  const int warps = r.M > kTinyWarps ? (r.M < kTinyMaxWarps ? r.M : kTinyMaxWarps) : kTinyWarps;
  return launch_kernel(route_align_tiny_kernel<EPL, 0>, dim3(1), dim3(32 * warps), 0, st, true, r, a);
}
template <int EPW>
cudaError_t launch_tiny_coop(const RouteIn& r, const AlignArgs& a, cudaStream_t st) {
  return launch_kernel(route_align_tiny_kernel<1, EPW>, dim3(1), dim3(32 * kCoopWarps * r.M), 0, st, true, r, a);
}

template <int EPL, int PER>
cudaError_t launch_fused_per(const RouteIn& r, const AlignArgs& a, cudaStream_t st) {
  const size_t smem = align_smem_bytes(a.E);
  cudaError_t err = ensure_smem_limit<route_align_kernel<EPL, PER>>(static_cast<int>(align_smem_bytes(1024)));
  if (err != cudaSuccess) return err;
  return launch_kernel(route_align_kernel<EPL, PER>, dim3(1), dim3(kThreads), smem, st, true, r, a);
}
template <int EPL>
cudaError_t launch_fused(const RouteIn& r, const AlignArgs& a, cudaStream_t st) {
  switch (align_per_thread(a.n)) {
    case 1: return launch_fused_per<EPL, 1>(r, a, st);
    case 2: return launch_fused_per<EPL, 2>(r, a, st);
    default: return launch_fused_per<EPL, kPerThread>(r, a, st);
  }
}

}  // namespace

// At top-k <= kCoopMaxTopk, one launch only up to kTinyCoopTokens tokens
// (four warps route each token): beyond that the router grid, four warps a
// token, and the align kernel are faster (M = 8, 384 experts: 5.96 against
// 6.98 us for the one-CTA form).  Otherwise one CTA routes one token per
// warp: beyond kWarps tokens a warp would route several in turn and the
// separate router grid is faster; up to 32 assignments the one-warp kernel
// takes any number of tokens.
bool route_align_fits(int M, int topk, long long assignments, int E_local) {
  if (assignments > kChunk || E_local < 1 || E_local > 1024) return false;
  if (topk <= kCoopMaxTopk) return M <= kTinyCoopTokens;
  return M <= kWarps || assignments <= 32;
}

cudaError_t route_align_launch(const float* logits, const float* bias, int M, int E_total, int topk,
                               int begin, int E_local, int bm, float* w, int32_t* ids, int32_t* sorted,
                               int32_t* expert_ids, int32_t* ntpp, int32_t* counts, int32_t* offsets,
                               int32_t* positions, cudaStream_t st, int* zero, int n_zero) {
  if (!route_align_fits(M, topk, static_cast<long long>(M) * topk, E_local)) return cudaErrorInvalidValue;
  RouteIn r{logits, bias, M, E_total, topk, w, ids, zero, n_zero};
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
  if (a.n <= 32 && M >= 1 && M <= kTinyCoopTokens && topk <= kCoopMaxTopk) {
    const int epw = (E_total + 32 * kCoopWarps - 1) / (32 * kCoopWarps);
    if (epw <= 1) return launch_tiny_coop<1>(r, a, st);
    if (epw <= 2) return launch_tiny_coop<2>(r, a, st);
    if (epw <= 3) return launch_tiny_coop<3>(r, a, st);
    if (epw <= 4) return launch_tiny_coop<4>(r, a, st);
    return launch_tiny_coop<8>(r, a, st);
  }
  if (a.n <= 32) {
    if (epl <= 1) return launch_tiny<1>(r, a, st);
    if (epl <= 2) return launch_tiny<2>(r, a, st);
    if (epl <= 4) return launch_tiny<4>(r, a, st);
    if (epl <= 8) return launch_tiny<8>(r, a, st);
    if (epl <= 12) return launch_tiny<12>(r, a, st);
    if (epl <= 16) return launch_tiny<16>(r, a, st);
    return launch_tiny<32>(r, a, st);
  }
  if (epl <= 1) return launch_fused<1>(r, a, st);
  if (epl <= 2) return launch_fused<2>(r, a, st);
  if (epl <= 4) return launch_fused<4>(r, a, st);
  if (epl <= 8) return launch_fused<8>(r, a, st);
  if (epl <= 12) return launch_fused<12>(r, a, st);
  if (epl <= 16) return launch_fused<16>(r, a, st);
  return launch_fused<32>(r, a, st);
}

}  // namespace chord
