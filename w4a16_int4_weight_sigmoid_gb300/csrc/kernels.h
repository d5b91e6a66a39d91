// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace chord {

struct PackHeader;

// zero, n_zero: ints the kernel clears (for the kernels after it; may be NULL)
cudaError_t route_launch(const float* logits, const float* bias, int M, int E, int topk, float* w,
                         int32_t* ids, cudaStream_t st, int* zero = nullptr, int n_zero = 0);

int align_num_chunks(long long n);
size_t align_workspace_bytes(long long n, int E_local);
// Fused router + one-chunk align (one CTA): only when route_align_fits().
bool route_align_fits(int M, int topk, long long assignments, int E_local);
cudaError_t route_align_launch(const float* logits, const float* bias, int M, int E_total, int topk,
                               int begin, int E_local, int bm, float* w, int32_t* ids, int32_t* sorted,
                               int32_t* expert_ids, int32_t* ntpp, int32_t* counts, int32_t* offsets,
                               int32_t* positions, cudaStream_t st, int* zero = nullptr, int n_zero = 0);
cudaError_t align_launch(const int32_t* ids, int M, int topk, int begin, int E_local, int bm,
                         int32_t* sorted, int32_t* expert_ids, int32_t* ntpp, int32_t* counts,
                         int32_t* offsets, int32_t* positions, void* ws, cudaStream_t st,
                         bool pdl = false);

cudaError_t align_noalloc_scratch(void** ptr);
size_t align_noalloc_scratch_bytes();

PackHeader make_pack_header(int E, int N, int K, bool gate_up);
size_t prepack_bytes(int E, int N, int K);
cudaError_t prepack_launch(const uint8_t* q, const uint16_t* s, int E, int N, int K, bool gate_up,
                           uint8_t* out, cudaStream_t st);

struct GemmLaunch {
  const uint16_t* A;
  bool gather;
  const void* packed;
  int E_local, N, K, M, topk;
  const int32_t* sorted;
  const int32_t* expert_ids;
  const int32_t* ntpp;
  const int32_t* counts;
  const int32_t* offsets;
  int block_m;
  int* work;        // small-M path: 2 ints, zero before the first launch (kept zero)
  int epilogue;
  uint16_t* C;             // BF16 output (STORE, SILU_MUL)
  float* Cf = nullptr;     // FP32 [M, N] accumulator (WEIGHTED_ADD)
  const float* topk_w = nullptr;   // routing weights [M, topk] (WEIGHTED_ADD)
  int* status;
  // Programmatic launch (small-M path only): 0 ordinary; 1 the kernel may
  // start before the previous kernel ends and waits for it before reading
  // anything; 2 as 1, and the expert map (ntpp, expert_ids, counts, offsets)
  // is already complete at launch, so the first weight stages are fetched
  // before the wait (the previous kernel is a GEMM launched with mode 1).
  int pdl = 0;
  int max_blocks = 0;   // BLOCK_M blocks the aligned buffers hold (capacity / block_m)
  // Split-K workspace of the small-M path (kSplitPartialBytes of partials,
  // kSplitCntBytes of counters that are zero between launches); NULL: the
  // kernel never splits K.
  float* split_partial = nullptr;
  int* split_cnt = nullptr;
  // Test of the timeout path (chord_debug_force_timeout): the small-M
  // kernel's producer issues no copy and hands out no item, and the
  // consumers give up their wait for an item after kTestWaitPolls probes.
  int test_timeout = 0;
};
// Dense GEMM: one-expert block map (counts, offsets, ntpp, expert_ids) for M rows.
cudaError_t dense_setup_launch(int M, int bm, int32_t* counts, int32_t* offsets, int32_t* ntpp,
                               int32_t* expert_ids, cudaStream_t st);
// Grouped layouts: block map from per-expert row counts (one CTA, E <= 1024).
// masked: group g at rows [g*max_m, g*max_m + rows); contiguous: groups in
// order, each padded to 128 rows.  A bad count or a total above capacity
// records CHORD_ERR_INVALID_ARG and leaves an empty map.
cudaError_t grouped_setup_launch(const int32_t* group_rows, int E, bool masked, int max_m, int bm,
                                 long long capacity, int32_t* counts, int32_t* offsets, int32_t* ntpp,
                                 int32_t* expert_ids, int* status, cudaStream_t st);
cudaError_t gemm_small_launch(const GemmLaunch& g, int rows_per_pass, cudaStream_t st);
size_t gemm_large_smem_bytes();
cudaError_t gemm_large_launch(const GemmLaunch& g, const uint16_t* B, size_t b_rows, cudaStream_t st);
cudaError_t gather_rows_launch(const uint16_t* x, const int32_t* sorted, const int32_t* ntpp, int topk,
                               int sentinel, int K, size_t capacity, uint16_t* out, cudaStream_t st);

cudaError_t moe_sum_launch(const uint16_t* y, const float* w, const int32_t* pos, int M, int topk,
                           int H, uint16_t* out, cudaStream_t st, bool pdl = false,
                           int y_rows = 0x7fffffff);

}  // namespace chord
