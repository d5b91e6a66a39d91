// Grouped layouts of the W4A16 GEMM ([Chord] "그룹 SM90 커널 기법"): the
// activation rows are already grouped by expert, so there is no routing and
// no gather.
//   contiguous (prefill): expert e's rows follow expert e-1's, each expert's
//     group padded to a 128-row boundary;
//   masked (decode): a fixed budget of max_m rows per expert, A is
//     [E, max_m, K], and only the first group_rows[e] rows of expert e count.
// One CTA turns the per-expert row counts into the block map the indexed
// GEMM reads (expert counts, offsets, padded total, per-block expert id), so
// the same kernels serve these layouts and the call captures into a CUDA
// graph.
#include "common.cuh"
#include "kernels.h"

namespace chord {
namespace {

constexpr int kSetupThreads = 1024;   // one thread per expert (E <= 1024)

__global__ void __launch_bounds__(kSetupThreads) grouped_setup_kernel(
    const int32_t* __restrict__ group_rows, int E, int masked, int max_m, int bm, long long capacity,
    int32_t* counts, int32_t* offsets, int32_t* ntpp, int32_t* expert_ids, int* status) {
  // 64-bit sizes and sums: a count is at most the rows of A (< 2^31), so
  // no padded size or partial sum can wrap before it is checked
  __shared__ long long s_off[kSetupThreads + 1];
  __shared__ long long s_warp[kSetupThreads / 32];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) s_bad = 0;
  __syncthreads();
  long long c = 0, p = 0;
  if (tid < E) {
    c = group_rows[tid];
    const long long limit = masked ? max_m : capacity;
    if (c < 0 || c > limit) {
      s_bad = 1;
      c = 0;
    }
    p = masked ? max_m : (c + 127) / 128 * 128;
  }
  // exclusive scan of the padded group sizes over the experts
  long long v = p;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const long long o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  if (lane == 31) s_warp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    long long w = s_warp[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const long long o = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += o;
    }
    s_warp[lane] = w;   // inclusive over warps
  }
  __syncthreads();
  const long long excl = v - p + (warp > 0 ? s_warp[warp - 1] : 0);
  if (tid < E) s_off[tid] = excl;
  if (tid == E - 1) s_off[E] = excl + p;
  __syncthreads();
  const long long total = s_off[E];
  if (total > capacity) s_bad = 1;
  __syncthreads();
  const bool bad = s_bad != 0;
  if (tid < E) {   // capacity < 2^31, so every value written fits an int
    counts[tid] = bad ? 0 : static_cast<int>(c);
    offsets[tid] = bad ? 0 : static_cast<int>(s_off[tid]);
  }
  const int used = bad ? 0 : static_cast<int>(total);
  if (tid == 0) {
    offsets[E] = used;
    ntpp[0] = used;
    if (bad) set_status(status, CHORD_ERR_INVALID_ARG);
  }
  // expert of each BLOCK_M block: the largest e with offset <= first row
  // (every padded group size is a multiple of bm)
  const int nblk = used / bm;
  for (int b = tid; b < nblk; b += kSetupThreads) {
    const long long row = static_cast<long long>(b) * bm;
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_off[mid] <= row) lo = mid; else hi = mid - 1;
    }
    expert_ids[b] = lo;
  }
}

}  // namespace

cudaError_t grouped_setup_launch(const int32_t* group_rows, int E, bool masked, int max_m, int bm,
                                 long long capacity, int32_t* counts, int32_t* offsets, int32_t* ntpp,
                                 int32_t* expert_ids, int* status, cudaStream_t st) {
  grouped_setup_kernel<<<1, kSetupThreads, 0, st>>>(group_rows, E, masked ? 1 : 0, max_m, bm, capacity, counts,
                                                    offsets, ntpp, expert_ids, status);
  return cudaGetLastError();
}

}  // namespace chord
