// C ABI of the chord_moe library: argument checks, workspace carving, path
// selection and launches.  No entry point allocates memory or synchronises.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "chord_moe.h"
#include "common.cuh"
#include "kernels.h"

namespace {

thread_local char g_err[512] = "";
// Test hook (chord_debug_force_timeout): later small-M GEMM launches
// withhold their work items from the consumer warps.
std::atomic<int> g_force_timeout{0};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(CHORD_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool valid_block_m(int bm) { return bm == 8 || bm == 16 || bm == 32 || bm == 64 || bm == 128; }

int check_tuning(const chord_tuning* t) {
  if (!t) return CHORD_OK;
  if (t->use_f16_accum)
    return fail(CHORD_ERR_UNSUPPORTED, "FP16 accumulation is not implemented (FP32 only)");
  if (t->batch_invariant)
    return fail(CHORD_ERR_UNSUPPORTED, "batch-invariant mode is not implemented");
  if (t->path < CHORD_PATH_AUTO || t->path > CHORD_PATH_LARGE_M)
    return fail(CHORD_ERR_INVALID_ARG, "unknown path %d", t->path);
  if (t->rows_per_pass != 0 && t->rows_per_pass != 8 && t->rows_per_pass != 16 && t->rows_per_pass != 32)
    return fail(CHORD_ERR_INVALID_ARG, "rows_per_pass=%d not in {0, 8, 16, 32}", t->rows_per_pass);
  return CHORD_OK;
}

// Token rows streamed per weight pass on the small-M path, from the expected
// rows per expert.
int rows_per_pass_for(double tok_e) {
  if (tok_e <= 6.0) return 8;
  if (tok_e <= 14.0) return 16;
  return 32;
}

// chord_w4a16_moe_gemm's automatic path: expected rows per local expert,
// counting every assignment as local (the call does not know E_total), at
// or above which the tensor-core (tcgen05) path is used; [Chord] "인덱스 커널
// 기법" switches schedules around 80 rows per expert.
constexpr double kLargeTokE = 64.0;
// The grouped and dense entry points know the rows per expert themselves
// (expected_m, or M): measured on GB300 with the masked layout at 32 rows
// per expert over 48 Kimi EP8 experts, the tcgen05 path took 305 / 162 us
// (gate/up / down) against 358 / 192 us on the register path.
constexpr double kGroupedLargeTokE = 16.0;
// chord_moe_layer's policy: expected rows per expert M*topk/E_total at or
// above which the tcgen05 path is used.  Measured on GB300 at Kimi EP8
// shapes (whole layer, both paths forced, split-K decode GEMM and two
// dequant groups on the tcgen05 path): M = 256 -> register path 231 us vs
// 333 us; M = 512 -> 317 vs 366 us; M = 1024 -> 655 vs 398 us, so the
// paths cross near M = 590, 12 rows per expert.
constexpr double kLayerLargeTokE = 12.0;
constexpr size_t kWorkBytes = 256;   // work-queue counters at the start of a GEMM workspace
// split-K area of a GEMM workspace: arrival counters, then partial accumulators
constexpr size_t kSplitCnt = chord::kSplitCntBytes;
constexpr size_t kSplitBytes = chord::kSplitCntBytes + chord::kSplitPartialBytes;

// Where one GEMM launch keeps its state on the device.
struct GemmWs {
  int* work = nullptr;              // 2 work-queue counters, zero between launches
  int* split_cnt = nullptr;         // split-K counters, zero between launches (NULL: no split-K)
  float* split_partial = nullptr;   // split-K partial accumulators
  uint16_t* gather = nullptr;       // tcgen05 path with gathered rows: [capacity, K] BF16
  size_t gather_bytes = 0;
};

// [work counters | split counters | split partials] at the start of p.
GemmWs carve_gemm_ws(char* p) {
  GemmWs w;
  w.work = reinterpret_cast<int*>(p);
  w.split_cnt = reinterpret_cast<int*>(p + kWorkBytes);
  w.split_partial = reinterpret_cast<float*>(p + kWorkBytes + kSplitCnt);
  return w;
}

// BLOCK_M the layer aligns with: one small-M pass per block, or 16 (the
// tcgen05 path pads each expert's rows to 16 only).
int layer_block_m(const chord_tuning& plan) {
  return plan.path == CHORD_PATH_LARGE_M ? 16 : plan.rows_per_pass;
}

struct LayerWs {
  size_t work, partial, tw, ids, sorted, eids, ntpp, counts, offsets, pos, align_ws, h, y, total;
  size_t cap;
  int bm;
};

LayerWs layer_ws(int M, int H, int I, int E_local, int topk, int bm) {
  LayerWs w{};
  const size_t mk = static_cast<size_t>(M) * topk;
  w.bm = bm;
  w.cap = chord_moe_align_capacity(M, topk, E_local, bm);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = round_up(o + bytes, 256);
    return at;
  };
  w.tw = take(mk * sizeof(float));
  w.ids = take(mk * sizeof(int32_t));
  w.sorted = take(w.cap * sizeof(int32_t));
  w.eids = take(w.cap / bm * sizeof(int32_t));
  w.ntpp = take(sizeof(int32_t));
  w.counts = take(static_cast<size_t>(E_local) * sizeof(int32_t));
  w.offsets = take(static_cast<size_t>(E_local + 1) * sizeof(int32_t));
  w.pos = take(mk * sizeof(int32_t));
  w.align_ws = take(chord::align_workspace_bytes(static_cast<long long>(mk), E_local));
  w.h = take(w.cap * static_cast<size_t>(I) * 2);
  // Counters, cleared by the router kernel on every call: [down work | gate/up work |
  // down split-K | gate/up split-K]; then the split-K partials, shared by
  // the two GEMMs (the down GEMM writes them only after the gate/up GEMM
  // has completed); then y, whose region holds the gathered x rows of the
  // tcgen05 gate/up path until the down GEMM writes y.
  w.work = take(2 * kWorkBytes + 2 * kSplitCnt);
  w.partial = take(chord::kSplitPartialBytes);
  w.y = take(w.cap * static_cast<size_t>(H) * 2);
  w.total = o;
  return w;
}

// The largest layout over the BLOCK_M values a plan can pick.
size_t layer_ws_max(int M, int H, int I, int E_local, int topk) {
  size_t m = 0;
  for (int bm : {8, 16, 32}) {
    const size_t t = layer_ws(M, H, I, E_local, topk, bm).total;
    m = t > m ? t : m;
  }
  return m;
}

int check_gemm_shapes(int N, int K, int epilogue) {
  if (K <= 0 || K % 64 != 0) return fail(CHORD_ERR_INVALID_ARG, "K=%d must be a positive multiple of 64", K);
  if (N <= 0 || N % 16 != 0) return fail(CHORD_ERR_INVALID_ARG, "N=%d must be a positive multiple of 16", N);
  if (epilogue != CHORD_EPI_STORE && epilogue != CHORD_EPI_SILU_MUL && epilogue != CHORD_EPI_WEIGHTED_ADD)
    return fail(CHORD_ERR_INVALID_ARG, "unknown epilogue %d", epilogue);
  if (epilogue == CHORD_EPI_SILU_MUL && N % 64 != 0)
    return fail(CHORD_ERR_INVALID_ARG, "SiLU*mul needs N=2I with I %% 32 == 0 (N=%d)", N);
  return CHORD_OK;
}

}  // namespace

extern "C" {

const char* chord_last_error_string(void) { return g_err; }

int chord_debug_force_timeout(int enable) {
  g_force_timeout.store(enable ? 1 : 0, std::memory_order_relaxed);
  return CHORD_OK;
}

int chord_version(void) { return 100; }

int chord_moe_route(const float* logits, const float* bias, int M, int E_total, int topk,
                    float* topk_weights, int32_t* topk_ids, void* stream) {
  if (M < 0) return fail(CHORD_ERR_INVALID_ARG, "M=%d < 0", M);
  if (E_total < 1 || E_total > 1024) return fail(CHORD_ERR_INVALID_ARG, "E_total=%d not in [1, 1024]", E_total);
  if (topk < 1 || topk > E_total || topk > 32)
    return fail(CHORD_ERR_INVALID_ARG, "topk=%d not in [1, min(E_total, 32)]", topk);
  if (M > 0 && (!logits || !bias || !topk_weights || !topk_ids))
    return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  cudaError_t e = chord::route_launch(logits, bias, M, E_total, topk, topk_weights, topk_ids,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CHORD_OK : cuda_fail(e, "route launch");
}

size_t chord_moe_align_capacity(int M, int topk, int E_local, int block_m) {
  if (M < 0 || topk < 1 || E_local < 1 || !valid_block_m(block_m)) return 0;
  const size_t R = static_cast<size_t>(M) * topk;
  const size_t cap = R + (R < static_cast<size_t>(E_local) ? R : E_local) * (block_m - 1);
  return round_up(cap, block_m);
}

size_t chord_moe_align_workspace_bytes(int M, int topk, int E_local) {
  if (M < 0 || topk < 1 || E_local < 1) return 0;
  return chord::align_workspace_bytes(static_cast<long long>(M) * topk, E_local);
}

}  // extern "C"

namespace {

// chord_moe_align with a choice of programmatic launch (pdl: the align may
// start before the router kernel ends and waits for it).
int align_impl(const int32_t* topk_ids, int M, int topk, int expert_begin, int E_local, int block_m,
               size_t capacity, int32_t* sorted_token_ids, int32_t* expert_ids,
               int32_t* num_tokens_post_padded, int32_t* expert_counts, int32_t* expert_offsets,
               int32_t* sorted_positions, void* workspace, size_t ws_bytes, void* stream, bool pdl) {
  if (M < 0 || topk < 1 || topk > 32) return fail(CHORD_ERR_INVALID_ARG, "bad M=%d or topk=%d", M, topk);
  if (E_local < 1 || E_local > 1024) return fail(CHORD_ERR_INVALID_ARG, "E_local=%d not in [1, 1024]", E_local);
  if (expert_begin < 0) return fail(CHORD_ERR_INVALID_ARG, "expert_begin=%d < 0", expert_begin);
  if (!valid_block_m(block_m)) return fail(CHORD_ERR_INVALID_ARG, "block_m=%d not in {8,16,32,64,128}", block_m);
  if (static_cast<long long>(M) * topk > (1LL << 30)) return fail(CHORD_ERR_INVALID_ARG, "M*topk too large");
  const size_t need = chord_moe_align_capacity(M, topk, E_local, block_m);
  if (capacity < need) return fail(CHORD_ERR_INVALID_ARG, "capacity %zu < required %zu", capacity, need);
  if (!expert_ids || !num_tokens_post_padded || !expert_counts || !expert_offsets || !sorted_token_ids ||
      (M > 0 && !topk_ids))
    return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  const size_t wneed = chord_moe_align_workspace_bytes(M, topk, E_local);
  if (ws_bytes < wneed || (wneed > 0 && !workspace))
    return fail(CHORD_ERR_WORKSPACE_TOO_SMALL, "align workspace %zu < required %zu", ws_bytes, wneed);
  cudaError_t e = chord::align_launch(topk_ids, M, topk, expert_begin, E_local, block_m,
                                      sorted_token_ids, expert_ids, num_tokens_post_padded,
                                      expert_counts, expert_offsets, sorted_positions, workspace,
                                      static_cast<cudaStream_t>(stream), pdl);
  return e == cudaSuccess ? CHORD_OK : cuda_fail(e, "align launch");
}

// chord_moe_route_align with a programmatic launch of the align kernel
// after the router kernel (pdl) when the two are separate launches.
int route_align_impl(const float* logits, const float* bias, int M, int E_total, int topk,
                     int expert_begin, int E_local, int block_m, size_t capacity, float* topk_weights,
                     int32_t* topk_ids, int32_t* sorted_token_ids, int32_t* expert_ids,
                     int32_t* num_tokens_post_padded, int32_t* expert_counts, int32_t* expert_offsets,
                     int32_t* sorted_positions, void* workspace, size_t ws_bytes, void* stream, bool pdl,
                     int* zero = nullptr, int n_zero = 0);

}  // namespace

extern "C" {

int chord_moe_align(const int32_t* topk_ids, int M, int topk, int expert_begin, int E_local,
                    int block_m, size_t capacity, int32_t* sorted_token_ids, int32_t* expert_ids,
                    int32_t* num_tokens_post_padded, int32_t* expert_counts,
                    int32_t* expert_offsets, int32_t* sorted_positions, void* workspace,
                    size_t ws_bytes, void* stream) {
  return align_impl(topk_ids, M, topk, expert_begin, E_local, block_m, capacity, sorted_token_ids,
                    expert_ids, num_tokens_post_padded, expert_counts, expert_offsets, sorted_positions,
                    workspace, ws_bytes, stream, false);
}

int chord_moe_route_align(const float* logits, const float* bias, int M, int E_total, int topk,
                          int expert_begin, int E_local, int block_m, size_t capacity,
                          float* topk_weights, int32_t* topk_ids, int32_t* sorted_token_ids,
                          int32_t* expert_ids, int32_t* num_tokens_post_padded, int32_t* expert_counts,
                          int32_t* expert_offsets, int32_t* sorted_positions, void* workspace,
                          size_t ws_bytes, void* stream) {
  return route_align_impl(logits, bias, M, E_total, topk, expert_begin, E_local, block_m, capacity,
                          topk_weights, topk_ids, sorted_token_ids, expert_ids, num_tokens_post_padded,
                          expert_counts, expert_offsets, sorted_positions, workspace, ws_bytes, stream,
                          false);
}

}  // extern "C"

namespace {

int route_align_impl(const float* logits, const float* bias, int M, int E_total, int topk,
                     int expert_begin, int E_local, int block_m, size_t capacity, float* topk_weights,
                     int32_t* topk_ids, int32_t* sorted_token_ids, int32_t* expert_ids,
                     int32_t* num_tokens_post_padded, int32_t* expert_counts, int32_t* expert_offsets,
                     int32_t* sorted_positions, void* workspace, size_t ws_bytes, void* stream, bool pdl,
                     int* zero, int n_zero) {
  if (M < 0) return fail(CHORD_ERR_INVALID_ARG, "M=%d < 0", M);
  if (E_total < 1 || E_total > 1024) return fail(CHORD_ERR_INVALID_ARG, "E_total=%d not in [1, 1024]", E_total);
  if (topk < 1 || topk > E_total || topk > 32)
    return fail(CHORD_ERR_INVALID_ARG, "topk=%d not in [1, min(E_total, 32)]", topk);
  if (E_local < 1 || E_local > 1024) return fail(CHORD_ERR_INVALID_ARG, "E_local=%d not in [1, 1024]", E_local);
  if (expert_begin < 0 || expert_begin + E_local > E_total)
    return fail(CHORD_ERR_INVALID_ARG, "local experts [%d, %d) not within E_total=%d", expert_begin,
                expert_begin + E_local, E_total);
  if (!valid_block_m(block_m)) return fail(CHORD_ERR_INVALID_ARG, "block_m=%d not in {8,16,32,64,128}", block_m);
  const size_t need = chord_moe_align_capacity(M, topk, E_local, block_m);
  if (capacity < need) return fail(CHORD_ERR_INVALID_ARG, "capacity %zu < required %zu", capacity, need);
  if (!expert_ids || !num_tokens_post_padded || !expert_counts || !expert_offsets || !sorted_token_ids ||
      (M > 0 && (!logits || !bias || !topk_weights || !topk_ids)))
    return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  const long long n = static_cast<long long>(M) * topk;
  if (!chord::route_align_fits(M, topk, n, E_local)) {
    // more than one chunk: the two separate launches
    cudaError_t er = chord::route_launch(logits, bias, M, E_total, topk, topk_weights, topk_ids,
                                         static_cast<cudaStream_t>(stream), zero, n_zero);
    if (er != cudaSuccess) return cuda_fail(er, "route launch");
    return align_impl(topk_ids, M, topk, expert_begin, E_local, block_m, capacity, sorted_token_ids,
                      expert_ids, num_tokens_post_padded, expert_counts, expert_offsets, sorted_positions,
                      workspace, ws_bytes, stream, pdl);
  }
  cudaError_t e = chord::route_align_launch(logits, bias, M, E_total, topk, expert_begin, E_local, block_m,
                                            topk_weights, topk_ids, sorted_token_ids, expert_ids,
                                            num_tokens_post_padded, expert_counts, expert_offsets,
                                            sorted_positions, static_cast<cudaStream_t>(stream), zero, n_zero);
  return e == cudaSuccess ? CHORD_OK : cuda_fail(e, "route+align launch");
}

}  // namespace

extern "C" {

int chord_moe_align_noalloc(const int32_t* topk_ids, int M, int topk, int expert_begin, int E_local,
                            int block_m, size_t capacity, int32_t* sorted_token_ids,
                            int32_t* expert_ids, int32_t* num_tokens_post_padded,
                            int32_t* expert_counts, int32_t* expert_offsets,
                            int32_t* sorted_positions, void* stream) {
  if (M < 0 || topk < 1 || static_cast<long long>(M) * topk > CHORD_ALIGN_NOALLOC_MAX_ASSIGNMENTS)
    return fail(CHORD_ERR_INVALID_ARG, "allocation-free align takes M*topk <= %d (got M=%d, topk=%d)",
                CHORD_ALIGN_NOALLOC_MAX_ASSIGNMENTS, M, topk);
  if (E_local < 1 || E_local > CHORD_ALIGN_NOALLOC_MAX_EXPERTS)
    return fail(CHORD_ERR_INVALID_ARG, "allocation-free align takes 1 <= E_local <= %d (got %d)",
                CHORD_ALIGN_NOALLOC_MAX_EXPERTS, E_local);
  const size_t wneed = chord_moe_align_workspace_bytes(M, topk, E_local);
  void* scratch = nullptr;
  if (wneed > 0) {
    if (wneed > chord::align_noalloc_scratch_bytes())
      return fail(CHORD_ERR_INVALID_ARG, "scratch need %zu exceeds the static array", wneed);
    cudaError_t e = chord::align_noalloc_scratch(&scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the align scratch");
  }
  return chord_moe_align(topk_ids, M, topk, expert_begin, E_local, block_m, capacity,
                         sorted_token_ids, expert_ids, num_tokens_post_padded, expert_counts,
                         expert_offsets, sorted_positions, scratch, wneed, stream);
}

size_t chord_w4a16_prepack_bytes(int E, int N, int K, int group) {
  if (E < 1 || N < 1 || K < 64 || K % 64 != 0 || group != 32) return 0;
  return chord::prepack_bytes(E, N, K);
}

int chord_w4a16_prepack(const uint8_t* qweight, const chord_bf16* scales, int E, int N, int K,
                        int group, int gate_up, void* packed, size_t packed_bytes, void* stream) {
  if (group != 32) return fail(CHORD_ERR_UNSUPPORTED, "group=%d: only group-32 scales are implemented", group);
  if (E < 1) return fail(CHORD_ERR_INVALID_ARG, "E=%d < 1", E);
  if (K <= 0 || K % 64 != 0) return fail(CHORD_ERR_INVALID_ARG, "K=%d must be a positive multiple of 64", K);
  if (N <= 0 || N % 16 != 0) return fail(CHORD_ERR_INVALID_ARG, "N=%d must be a positive multiple of 16", N);
  if (gate_up && N % 64 != 0) return fail(CHORD_ERR_INVALID_ARG, "gate_up needs N %% 64 == 0 (N=%d)", N);
  if (!qweight || !scales || !packed) return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(packed)) return fail(CHORD_ERR_INVALID_ARG, "packed must be 16-byte aligned");
  const size_t need = chord_w4a16_prepack_bytes(E, N, K, group);
  if (packed_bytes < need) return fail(CHORD_ERR_INVALID_ARG, "packed_bytes %zu < required %zu", packed_bytes, need);
  cudaError_t e = chord::prepack_launch(qweight, scales, E, N, K, gate_up != 0,
                                        static_cast<uint8_t*>(packed), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? CHORD_OK : cuda_fail(e, "prepack launch");
}

static int gemm_impl(const chord_bf16* A, int a_gather, const void* packed_w, int E_local, int N,
                     int K, int M, int topk, const int32_t* sorted_token_ids,
                     const int32_t* expert_ids, const int32_t* ntpp, const int32_t* expert_counts,
                     const int32_t* expert_offsets, int block_m, size_t capacity, int epilogue,
                     void* C, const chord_tuning* tuning, double tok_e, const GemmWs& ws,
                     int* dev_status, void* stream, int pdl = 0, const float* topk_weights = nullptr) {
  int rc = check_tuning(tuning);
  if (rc) return rc;
  rc = check_gemm_shapes(N, K, epilogue);
  if (rc) return rc;
  if (E_local < 1 || M < 0 || topk < 1) return fail(CHORD_ERR_INVALID_ARG, "bad E_local/M/topk");
  if (!valid_block_m(block_m)) return fail(CHORD_ERR_INVALID_ARG, "block_m=%d not in {8,16,32,64,128}", block_m);
  if (!A || !packed_w || !C || !expert_counts || !expert_offsets || !expert_ids || !ntpp ||
      (a_gather && !sorted_token_ids))
    return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(A) || !aligned16(packed_w) || !aligned16(C))
    return fail(CHORD_ERR_INVALID_ARG, "A, packed_w and C must be 16-byte aligned");
  if (!ws.work) return fail(CHORD_ERR_WORKSPACE_TOO_SMALL, "no GEMM workspace");
  if (epilogue == CHORD_EPI_WEIGHTED_ADD) {
    if (a_gather) return fail(CHORD_ERR_UNSUPPORTED, "the weighted-add epilogue reads rows in sorted order (a_gather = 0)");
    if (!topk_weights || !sorted_token_ids)
      return fail(CHORD_ERR_INVALID_ARG, "the weighted-add epilogue needs topk_weights and sorted_token_ids");
  }
  if (M == 0) return CHORD_OK;
  int path = tuning && tuning->path ? tuning->path : CHORD_PATH_AUTO;
  if (path == CHORD_PATH_AUTO)
    path = (tok_e >= kLargeTokE && N % 128 == 0 && E_local <= 1024) ? CHORD_PATH_LARGE_M : CHORD_PATH_SMALL_M;
  if (path == CHORD_PATH_LARGE_M && (N % 128 != 0 || E_local > 1024))
    return fail(CHORD_ERR_UNSUPPORTED, "tcgen05 path needs N %% 128 == 0 and E_local <= 1024");
  chord::GemmLaunch g;
  g.A = A;
  g.gather = a_gather != 0;
  g.packed = packed_w;
  g.E_local = E_local;
  g.N = N;
  g.K = K;
  g.M = M;
  g.topk = topk;
  g.sorted = sorted_token_ids;
  g.expert_ids = expert_ids;
  g.ntpp = ntpp;
  g.counts = expert_counts;
  g.offsets = expert_offsets;
  g.block_m = block_m;
  g.work = ws.work;
  g.split_cnt = ws.split_cnt;
  g.split_partial = ws.split_partial;
  g.test_timeout = g_force_timeout.load(std::memory_order_relaxed) ? 1 : 0;
  g.epilogue = epilogue;
  g.C = epilogue == CHORD_EPI_WEIGHTED_ADD ? nullptr : static_cast<uint16_t*>(C);
  g.Cf = epilogue == CHORD_EPI_WEIGHTED_ADD ? static_cast<float*>(C) : nullptr;
  g.topk_w = topk_weights;
  g.status = dev_status;
  g.pdl = pdl;
  const size_t max_blocks = (capacity + block_m - 1) / block_m;
  g.max_blocks = max_blocks > 0x7fffffff ? 0x7fffffff : static_cast<int>(max_blocks);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (path == CHORD_PATH_LARGE_M) {
    const uint16_t* B = A;
    if (a_gather) {
      const size_t need = capacity * static_cast<size_t>(K) * 2;
      if (!ws.gather || ws.gather_bytes < need)
        return fail(CHORD_ERR_WORKSPACE_TOO_SMALL, "GEMM workspace: gathered rows need %zu bytes", need);
      uint16_t* xs = ws.gather;
      e = chord::gather_rows_launch(A, sorted_token_ids, ntpp, topk, M * topk, K, capacity, xs, st);
      if (e != cudaSuccess) return cuda_fail(e, "gather launch");
      B = xs;
    }
    e = chord::gemm_large_launch(g, B, capacity, st);
    return e == cudaSuccess ? CHORD_OK : cuda_fail(e, "tcgen05 gemm launch");
  }
  const int rpp = tuning && tuning->rows_per_pass ? tuning->rows_per_pass : rows_per_pass_for(tok_e);
  e = chord::gemm_small_launch(g, rpp, st);
  return e == cudaSuccess ? CHORD_OK : cuda_fail(e, "gemm launch");
}

}  // extern "C"

namespace {

// Grouped-layout GEMM: the block map from the per-expert row counts, then
// the indexed GEMM on direct rows.  capacity = rows of A and C.
int grouped_impl(const chord_bf16* A, size_t capacity, const int32_t* group_rows, int E, bool masked,
                 int max_m, double tok_e, const void* packed_w, int N, int K, int epilogue, chord_bf16* C,
                 const chord_tuning* tuning, void* workspace, size_t ws_bytes, int* dev_status, void* stream) {
  int rc = check_tuning(tuning);
  if (rc) return rc;
  rc = check_gemm_shapes(N, K, epilogue);
  if (rc) return rc;
  if (E < 1 || E > 1024) return fail(CHORD_ERR_INVALID_ARG, "E=%d not in [1, 1024]", E);
  if (epilogue == CHORD_EPI_WEIGHTED_ADD)
    return fail(CHORD_ERR_INVALID_ARG, "the weighted-add epilogue needs routing (chord_w4a16_moe_gemm)");
  if (capacity > 0x7fffffffu) return fail(CHORD_ERR_INVALID_ARG, "%zu rows: too many", capacity);
  if (capacity == 0) return CHORD_OK;
  if (!A || !group_rows || !packed_w || !C) return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(A) || !aligned16(packed_w) || !aligned16(C))
    return fail(CHORD_ERR_INVALID_ARG, "A, packed_w and C must be 16-byte aligned");
  if (!workspace || !aligned16(workspace)) return fail(CHORD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  const size_t need = chord_w4a16_grouped_workspace_bytes(E, capacity);
  if (ws_bytes < need) return fail(CHORD_ERR_WORKSPACE_TOO_SMALL, "grouped GEMM workspace %zu < %zu", ws_bytes, need);
  chord_tuning plan{};
  if (tuning) plan = *tuning;
  if (!plan.path) plan.path = (tok_e >= kGroupedLargeTokE && N % 128 == 0) ? CHORD_PATH_LARGE_M : CHORD_PATH_SMALL_M;
  if (!plan.rows_per_pass) plan.rows_per_pass = rows_per_pass_for(tok_e);
  if (plan.path == CHORD_PATH_LARGE_M && N % 128 != 0)   // checked before anything is launched
    return fail(CHORD_ERR_UNSUPPORTED, "tcgen05 path needs N %% 128 == 0");
  // BLOCK_M: 16 on the tcgen05 path; else one pass per block where the
  // group size allows (every padded group is a multiple of BLOCK_M)
  const int seg = masked ? max_m : 128;
  int bm = 16;
  if (plan.path != CHORD_PATH_LARGE_M) bm = seg % plan.rows_per_pass == 0 ? plan.rows_per_pass : (seg % 16 == 0 ? 16 : 8);
  char* ws = static_cast<char*>(workspace);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + kWorkBytes);
  int32_t *counts = meta, *offsets = meta + E, *ntpp = meta + 2 * E + 1;
  int32_t* eids = reinterpret_cast<int32_t*>(ws + kWorkBytes + round_up((2 * static_cast<size_t>(E) + 2) * 4, 256));
  GemmWs gws = carve_gemm_ws(ws + need - kSplitBytes - kWorkBytes);
  gws.work = reinterpret_cast<int*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = chord::grouped_setup_launch(group_rows, E, masked, max_m, bm, static_cast<long long>(capacity),
                                              counts, offsets, ntpp, eids, dev_status, st);
  if (e != cudaSuccess) return cuda_fail(e, "grouped setup launch");
  return gemm_impl(A, 0, packed_w, E, N, K, static_cast<int>(capacity), 1, nullptr, eids, ntpp, counts, offsets, bm,
                   capacity, epilogue, C, &plan, tok_e, gws, dev_status, stream);
}

}  // namespace

extern "C" {

// [256 B work counters | counts, offsets, ntpp | expert_ids for up to rows/8
// blocks | split-K counters | split-K partials]
size_t chord_w4a16_grouped_workspace_bytes(int E, size_t rows) {
  if (E < 1 || E > 1024) return 0;
  return kWorkBytes + round_up((2 * static_cast<size_t>(E) + 2) * 4, 256) + round_up((rows / 8 + 1) * 4, 256) +
         kSplitBytes;
}

int chord_w4a16_grouped_gemm_contiguous(const chord_bf16* A, size_t a_rows, const int32_t* group_rows, int E,
                                        int expected_m, const void* packed_w, int N, int K, int epilogue,
                                        chord_bf16* C, const chord_tuning* tuning, void* workspace,
                                        size_t ws_bytes, int* dev_status, void* stream) {
  const double tok_e = expected_m > 0 ? expected_m : (E > 0 ? static_cast<double>(a_rows) / E : 0.0);
  return grouped_impl(A, a_rows, group_rows, E, false, 0, tok_e, packed_w, N, K, epilogue, C, tuning, workspace,
                      ws_bytes, dev_status, stream);
}

int chord_w4a16_grouped_gemm_masked(const chord_bf16* A, const int32_t* group_rows, int E, int max_m,
                                    int expected_m, const void* packed_w, int N, int K, int epilogue,
                                    chord_bf16* C, const chord_tuning* tuning, void* workspace, size_t ws_bytes,
                                    int* dev_status, void* stream) {
  if (max_m <= 0 || max_m % 16 != 0) return fail(CHORD_ERR_INVALID_ARG, "max_m=%d must be a positive multiple of 16", max_m);
  if (E < 1 || E > 1024) return fail(CHORD_ERR_INVALID_ARG, "E=%d not in [1, 1024]", E);
  const double tok_e = expected_m > 0 ? expected_m : max_m;
  return grouped_impl(A, static_cast<size_t>(E) * max_m, group_rows, E, true, max_m, tok_e, packed_w, N, K,
                      epilogue, C, tuning, workspace, ws_bytes, dev_status, stream);
}

// [256 B work counters | split-K counters | split-K partials | gathered rows]
size_t chord_w4a16_moe_gemm_workspace_bytes(size_t capacity, int K, int a_gather) {
  return kWorkBytes + kSplitBytes + (a_gather ? capacity * static_cast<size_t>(K > 0 ? K : 0) * 2 : 0);
}

int chord_w4a16_moe_gemm(const chord_bf16* A, int a_gather, const void* packed_w, int E_local,
                         int N, int K, int M, int topk, const int32_t* sorted_token_ids,
                         const int32_t* expert_ids, const int32_t* num_tokens_post_padded,
                         const int32_t* expert_counts, const int32_t* expert_offsets, int block_m,
                         size_t capacity, int epilogue, const float* topk_weights, void* C,
                         const chord_tuning* tuning, void* workspace, size_t ws_bytes, int* dev_status,
                         void* stream) {
  const double tok_e = E_local > 0 ? static_cast<double>(M) * topk / E_local : 0.0;
  int rc = check_tuning(tuning);   // argument errors take precedence over the workspace size
  if (rc) return rc;
  rc = check_gemm_shapes(N, K, epilogue);
  if (rc) return rc;
  if (!workspace || !aligned16(workspace) || ws_bytes < kWorkBytes + kSplitBytes)
    return fail(CHORD_ERR_WORKSPACE_TOO_SMALL, "GEMM workspace must hold at least %zu aligned bytes",
                kWorkBytes + kSplitBytes);
  GemmWs gws = carve_gemm_ws(static_cast<char*>(workspace));
  gws.gather = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + kWorkBytes + kSplitBytes);
  gws.gather_bytes = ws_bytes - kWorkBytes - kSplitBytes;
  return gemm_impl(A, a_gather, packed_w, E_local, N, K, M, topk, sorted_token_ids, expert_ids,
                   num_tokens_post_padded, expert_counts, expert_offsets, block_m, capacity, epilogue,
                   C, tuning, tok_e, gws, dev_status, stream, 0, topk_weights);
}

// [256 B work counters | counts, offsets, ntpp (256 B) | expert_ids |
// split-K counters | split-K partials]
size_t chord_w4a16_gemm_workspace_bytes(int M) {
  if (M < 0) return 0;
  return 2 * kWorkBytes + round_up((static_cast<size_t>(M) / 8 + 1) * sizeof(int32_t), 256) + kSplitBytes;
}

int chord_w4a16_gemm(const chord_bf16* A, const void* packed_w, int N, int K, int M, int epilogue,
                     chord_bf16* C, const chord_tuning* tuning, void* workspace, size_t ws_bytes,
                     int* dev_status, void* stream) {
  int rc = check_tuning(tuning);
  if (rc) return rc;
  rc = check_gemm_shapes(N, K, epilogue);
  if (rc) return rc;
  if (M < 0) return fail(CHORD_ERR_INVALID_ARG, "M=%d < 0", M);
  if (epilogue == CHORD_EPI_WEIGHTED_ADD)
    return fail(CHORD_ERR_INVALID_ARG, "the weighted-add epilogue needs routing (chord_w4a16_moe_gemm)");
  if (M == 0) return CHORD_OK;
  if (!A || !packed_w || !C) return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  if (!workspace || !aligned16(workspace)) return fail(CHORD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  const size_t need = chord_w4a16_gemm_workspace_bytes(M);
  if (ws_bytes < need) return fail(CHORD_ERR_WORKSPACE_TOO_SMALL, "dense GEMM workspace %zu < %zu", ws_bytes, need);
  // every row is a row of the single expert: rows per expert = M
  const double tok_e = static_cast<double>(M);
  chord_tuning plan{};
  if (tuning) plan = *tuning;
  if (!plan.path)
    plan.path = (tok_e >= kGroupedLargeTokE && N % 128 == 0) ? CHORD_PATH_LARGE_M : CHORD_PATH_SMALL_M;
  if (!plan.rows_per_pass) plan.rows_per_pass = rows_per_pass_for(tok_e);
  if (plan.path == CHORD_PATH_LARGE_M && N % 128 != 0)   // checked before anything is launched
    return fail(CHORD_ERR_UNSUPPORTED, "tcgen05 path needs N %% 128 == 0");
  const int bm = plan.path == CHORD_PATH_LARGE_M ? 16 : plan.rows_per_pass;
  char* ws = static_cast<char*>(workspace);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + kWorkBytes);
  int32_t *counts = meta, *offsets = meta + 4, *ntpp = meta + 8;
  int32_t* eids = reinterpret_cast<int32_t*>(ws + 2 * kWorkBytes);
  GemmWs gws = carve_gemm_ws(ws + need - kSplitBytes - kWorkBytes);
  gws.work = reinterpret_cast<int*>(ws);
  cudaError_t e = chord::dense_setup_launch(M, bm, counts, offsets, ntpp, eids, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "dense setup launch");
  // direct rows: A is [M, K]; the tensor-core path's activation map covers
  // exactly those M rows (reads past them return zeros)
  return gemm_impl(A, 0, packed_w, 1, N, K, M, 1, nullptr, eids, ntpp, counts, offsets, bm,
                   static_cast<size_t>(M), epilogue, C, &plan, tok_e, gws, dev_status, stream);
}

}  // extern "C"

namespace {

// chord_moe_sum with a choice of programmatic launch (pdl: may start before
// the down GEMM ends and waits for it).
int moe_sum_impl(const chord_bf16* y, const float* topk_weights, const int32_t* sorted_positions, int M,
                 int topk, int H, chord_bf16* out, void* stream, bool pdl, int y_rows = 0x7fffffff) {
  if (M < 0 || topk < 1 || topk > 32 || H <= 0 || H % 8 != 0)
    return fail(CHORD_ERR_INVALID_ARG, "bad M/topk/H (1 <= topk <= 32, H %% 8 == 0)");
  if (M > 0 && (!y || !topk_weights || !sorted_positions || !out)) return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(y) || !aligned16(out)) return fail(CHORD_ERR_INVALID_ARG, "y and out must be 16-byte aligned");
  cudaError_t e = chord::moe_sum_launch(y, topk_weights, sorted_positions, M, topk, H, out,
                                        static_cast<cudaStream_t>(stream), pdl, y_rows);
  return e == cudaSuccess ? CHORD_OK : cuda_fail(e, "moe_sum launch");
}

}  // namespace

extern "C" {

int chord_moe_sum(const chord_bf16* y, const float* topk_weights, const int32_t* sorted_positions,
                  int M, int topk, int H, chord_bf16* out, void* stream) {
  return moe_sum_impl(y, topk_weights, sorted_positions, M, topk, H, out, stream, false);
}

int chord_moe_layer_plan(int M, int E_total, int topk, chord_tuning* plan) {
  if (!plan || M < 0 || E_total < 1 || topk < 1) return fail(CHORD_ERR_INVALID_ARG, "bad plan arguments");
  const double tok_e = static_cast<double>(M) * topk / E_total;
  plan->path = tok_e >= kLayerLargeTokE ? CHORD_PATH_LARGE_M : CHORD_PATH_SMALL_M;
  plan->rows_per_pass = rows_per_pass_for(tok_e);
  plan->use_f16_accum = 0;
  plan->batch_invariant = 0;
  return CHORD_OK;
}

size_t chord_moe_layer_workspace_bytes(int M, int H, int I, int E_local, int topk) {
  if (M < 0 || H <= 0 || I <= 0 || E_local < 1 || topk < 1) return 0;
  return layer_ws_max(M, H, I, E_local, topk);
}

int chord_moe_layer(const chord_bf16* x, const float* logits, const float* bias,
                    const void* w13_packed, const void* w2_packed, int M, int H, int I,
                    int E_total, int expert_begin, int E_local, int topk, chord_bf16* out,
                    float* topk_weights_out, int32_t* topk_ids_out, void* workspace,
                    size_t ws_bytes, const chord_tuning* tuning, int* dev_status, void* stream) {
  int rc = check_tuning(tuning);
  if (rc) return rc;
  if (M < 0) return fail(CHORD_ERR_INVALID_ARG, "M=%d < 0", M);
  if (H <= 0 || H % 64 != 0) return fail(CHORD_ERR_INVALID_ARG, "H=%d must be a positive multiple of 64", H);
  if (I <= 0 || I % 64 != 0) return fail(CHORD_ERR_INVALID_ARG, "I=%d must be a positive multiple of 64", I);
  if (E_local < 1 || expert_begin < 0 || expert_begin + E_local > E_total)
    return fail(CHORD_ERR_INVALID_ARG, "local experts [%d, %d) not within E_total=%d", expert_begin,
                expert_begin + E_local, E_total);
  if (M == 0) return CHORD_OK;
  if (!x || !logits || !bias || !w13_packed || !w2_packed || !out || !workspace)
    return fail(CHORD_ERR_INVALID_ARG, "null pointer");
  chord_tuning plan;
  chord_moe_layer_plan(M, E_total, topk, &plan);
  if (tuning) {
    if (tuning->path) plan.path = tuning->path;
    if (tuning->rows_per_pass) plan.rows_per_pass = tuning->rows_per_pass;
  }
  if (plan.path == CHORD_PATH_LARGE_M && ((2 * I) % 128 != 0 || H % 128 != 0 || E_local > 1024))
    plan.path = CHORD_PATH_SMALL_M;
  const LayerWs w = layer_ws(M, H, I, E_local, topk, layer_block_m(plan));
  if (ws_bytes < w.total)
    return fail(CHORD_ERR_WORKSPACE_TOO_SMALL, "layer workspace %zu < required %zu", ws_bytes,
                layer_ws_max(M, H, I, E_local, topk));
  if (!aligned16(workspace)) return fail(CHORD_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  char* ws = static_cast<char*>(workspace);
  float* tw = topk_weights_out ? topk_weights_out : reinterpret_cast<float*>(ws + w.tw);
  int32_t* ids = topk_ids_out ? topk_ids_out : reinterpret_cast<int32_t*>(ws + w.ids);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + w.sorted);
  int32_t* eids = reinterpret_cast<int32_t*>(ws + w.eids);
  int32_t* ntpp = reinterpret_cast<int32_t*>(ws + w.ntpp);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + w.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + w.offsets);
  int32_t* pos = reinterpret_cast<int32_t*>(ws + w.pos);
  void* aws = ws + w.align_ws;
  chord_bf16* h = reinterpret_cast<chord_bf16*>(ws + w.h);
  chord_bf16* y = reinterpret_cast<chord_bf16*>(ws + w.y);

  // The router is a programmatic launch up to 512 tokens (it touches nothing
  // before the work ahead of the call has completed).  Register-MMA path:
  // every later kernel is one too, so its launch and prologue overlap the
  // end of the kernel before it, and the down GEMM streams its first weight
  // stages while the gate/up GEMM finishes.  The tcgen05 path launches its
  // later kernels in plain stream order.
  const bool pdl = plan.path != CHORD_PATH_LARGE_M;
  // one launch when the assignments fit one align chunk, else two
  // The router kernel (the layer's first) clears both GEMMs' work-queue and
  // split counters; the GEMMs start after it has completed (stream order, or
  // the launch chain: each kernel waits for the one before it, which waited
  // for the router), so they always find them zero, also after a call that
  // stopped on a timeout.
  rc = route_align_impl(logits, bias, M, E_total, topk, expert_begin, E_local, w.bm, w.cap, tw, ids, sorted,
                        eids, ntpp, counts, offsets, pos, aws, chord_moe_align_workspace_bytes(M, topk, E_local),
                        stream, pdl, reinterpret_cast<int*>(ws + w.work),
                        static_cast<int>((2 * kWorkBytes + 2 * kSplitCnt) / sizeof(int)));
  if (rc) return rc;
  const double tok_e = static_cast<double>(M) * topk / E_total;
  GemmWs ws_gu, ws_dn;
  ws_dn.work = reinterpret_cast<int*>(ws + w.work);
  ws_gu.work = reinterpret_cast<int*>(ws + w.work + kWorkBytes);
  ws_dn.split_cnt = reinterpret_cast<int*>(ws + w.work + 2 * kWorkBytes);
  ws_gu.split_cnt = reinterpret_cast<int*>(ws + w.work + 2 * kWorkBytes + kSplitCnt);
  ws_dn.split_partial = ws_gu.split_partial = reinterpret_cast<float*>(ws + w.partial);
  ws_gu.gather = y;   // the gathered x rows live in y's region until the down GEMM writes y
  ws_gu.gather_bytes = w.cap * static_cast<size_t>(H) * 2;
  rc = gemm_impl(x, 1, w13_packed, E_local, 2 * I, H, M, topk, sorted, eids, ntpp, counts, offsets,
                 w.bm, w.cap, CHORD_EPI_SILU_MUL, h, &plan, tok_e, ws_gu, dev_status, stream, pdl ? 1 : 0);
  if (rc) return rc;
  rc = gemm_impl(h, 0, w2_packed, E_local, H, I, M, topk, sorted, eids, ntpp, counts, offsets, w.bm,
                 w.cap, CHORD_EPI_STORE, y, &plan, tok_e, ws_dn, dev_status, stream,
                 pdl ? 2 : 0);
  if (rc) return rc;
  return moe_sum_impl(y, tw, pos, M, topk, H, out, stream, pdl, static_cast<int>(w.cap));
}

}  // extern "C"
