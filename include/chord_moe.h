/*
 * chord_moe.h -- C ABI of the GB300 (sm_103a) W4A16 INT4-weight MoE layer.
 *
 * The layer: sigmoid+bias top-k routing -> moe_align_block_size -> grouped
 * gate/up GEMM (INT4 group-32 weights, BF16 scales, BF16 activations,
 * dequantised in-kernel) with fused SiLU*mul -> grouped down GEMM -> top-k
 * weighted sum back to tokens.
 *
 * Sources, cited by page title and section:
 *   [Chord]   "vLLM 및 Novita AI, Kimi K2.x용 더 빠른 INT4 MoE 커널 출시: Chord"
 *   [HumPR]   "[vllm] vLLM에 고성능 JIT 양자화 커널 'Humming' 도입하기"
 *   [Router]  "[flashinfer] FlashInfer, B200 GPU에서 Kimi-K3 MoE 라우터 성능 최적화"
 *   [Humming] "Humming: vLLM과 Ant Group, 양자화 추론을 위한 범용 커널 라이브러리
 *              오픈소스 공개"
 *
 * Conventions for every entry point:
 *   - Pointers named in the signature are DEVICE pointers unless a comment
 *     says otherwise; the caller owns all memory.  No entry point allocates
 *     device memory or synchronises the stream; `stream` is a cudaStream_t
 *     passed as void* (NULL = legacy default stream).
 *   - BF16 tensors are passed as chord_bf16 (the raw 16-bit pattern).
 *   - Tensors are dense, row-major, and 16-byte aligned.
 *   - Return value: CHORD_OK or a negative CHORD_ERR_* code from host-side
 *     checks or the launch; nothing is launched when a check fails.
 *     chord_last_error_string() describes the last failure on this thread.
 *   - Errors found on the device (packed-weight header mismatch, a bounded
 *     wait that ran out, invalid routing) are written with an atomic
 *     compare-and-swap into the caller's `dev_status` int (first error wins;
 *     the caller zeroes it and reads it when convenient, which keeps every
 *     call capturable in a CUDA graph: [Chord] "런타임 고려사항" notes graph
 *     capture is possible when routing validation is off).
 */
#ifndef CHORD_MOE_H
#define CHORD_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t chord_bf16;

enum chord_status {
  CHORD_OK = 0,
  CHORD_ERR_INVALID_ARG = -1,       /* null pointer, bad shape, misalignment */
  CHORD_ERR_UNSUPPORTED = -2,       /* a compute option this library does not implement */
  CHORD_ERR_CUDA = -3,              /* a CUDA runtime call or launch failed */
  CHORD_ERR_WORKSPACE_TOO_SMALL = -4,
  CHORD_ERR_PREPACK_MISMATCH = -5,  /* packed-weight header does not match the call */
  CHORD_ERR_TIMEOUT = -6,           /* a bounded device wait ran out (device status) */
  CHORD_ERR_ROUTING_INVALID = -7    /* an expert id out of range (device status) */
};

/* GEMM epilogues. */
enum chord_epilogue {
  CHORD_EPI_STORE = 0,        /* C[r, n] = bf16(acc[r, n]) */
  CHORD_EPI_SILU_MUL = 1,     /* C[r, i] = bf16(silu(acc[r, i]) * acc[r, I + i]), I = N/2 */
  CHORD_EPI_WEIGHTED_ADD = 2  /* FP32 C[t, n] += topk_weights[f] * acc[r, n], f = sorted_token_ids[r],
                                 t = f / topk (indexed GEMM only; see chord_w4a16_moe_gemm) */
};

/* GEMM execution paths. */
enum chord_path {
  CHORD_PATH_AUTO = 0,    /* choose from the expected tokens per expert */
  CHORD_PATH_SMALL_M = 1, /* register-MMA weight-streaming path (decode) */
  CHORD_PATH_LARGE_M = 2  /* tcgen05 / TMEM path (prefill) */
};

/* Optional tuning overrides; pass NULL for the built-in heuristics.  The two
 * compute options mirror Humming's compute config ([HumPR] "코드 분석" 2,
 * use_batch_invariant / use_f16_accum); like the backends on [Chord]
 * "런타임 고려사항", this library does not implement them and returns
 * CHORD_ERR_UNSUPPORTED when either is set. */
typedef struct chord_tuning {
  int path;             /* chord_path */
  int rows_per_pass;    /* small-M path: token rows per weight pass, 8/16/32; 0 = heuristic */
  int use_f16_accum;    /* must be 0 */
  int batch_invariant;  /* must be 0 */
} chord_tuning;

/* Description of the last failure on the calling thread ("" if none). */
const char* chord_last_error_string(void);
/* Test hook for the device timeout path, not needed in normal use: while
 * enabled, every later launch of the register-MMA GEMM in this process
 * withholds its work items from its consumer warps (the producer issues no
 * copy and hands out no item), so the consumers' barrier waits run out after
 * a short limit: the kernel records CHORD_ERR_TIMEOUT in dev_status and
 * returns, with no copy in flight and the work-queue counters left zero.
 * Nothing is computed.  enable = 0 turns it off.  Returns CHORD_OK. */
int chord_debug_force_timeout(int enable);
/* Library version, major*10000 + minor*100 + patch. */
int chord_version(void);

/* ---------------------------------------------------------------- routing
 * Sigmoid + bias top-k router.  Buffers follow the fused router's argument
 * plan ([Router] "코드 분석": logits, bias, topk_weights, topk_ids).
 *   logits       FP32 [M, E_total]   router logits (finite values)
 *   bias         FP32 [E_total]      expert score-correction bias
 *   topk_weights FP32 [M, topk]      out: s_j / sum of the selected s
 *   topk_ids     INT32 [M, topk]     out: selected experts, largest key first
 * Per token: s_e = sigmoid(logit_e) in a fixed binary32 op sequence (range
 * reduction n = rint(y*log2e), r = (y - n*ln2_hi) - n*ln2_lo with
 * y = clamp(-x, -87, 87); degree-7 Taylor polynomial in Horner form with
 * separately rounded multiply and add; times 2^n; s = 1/(1+e)), so results
 * are bit-identical across implementations of the same sequence; key_e =
 * s_e + bias_e; the topk largest keys win, equal keys going to the lower id.
 * Requires 1 <= topk <= min(E_total, 32), 1 <= E_total <= 1024, M >= 0.
 * Up to 512 tokens the router kernel is a programmatic dependent launch
 * that touches no memory before the kernel ahead of it in the stream has
 * completed, so stream order holds while its launch overlaps that kernel
 * (the logits' producer, or the previous call); above that it is an
 * ordinary launch.
 */
int chord_moe_route(const float* logits, const float* bias, int M, int E_total, int topk,
                    float* topk_weights, int32_t* topk_ids, void* stream);

/* ------------------------------------------------------------------ align
 * moe_align_block_size: group the M*topk assignments by local expert and pad
 * each group to a multiple of block_m ([Router] "코드 분석" arg_plan:
 * sorted_token_ids, expert_ids, num_tokens_post_padded, expert_counts,
 * expert_offsets; [Chord] "런타임 고려사항": over-allocated buffers).
 *   topk_ids          INT32 [M, topk]  expert of assignment f = t*topk + j
 *   expert_begin, E_local              local experts [begin, begin+E_local);
 *                                      other assignments are dropped
 *   block_m           8, 16, 32, 64 or 128
 *   capacity          rows of sorted_token_ids; must be >= chord_moe_align_capacity()
 *   sorted_token_ids  INT32 [capacity] out: expert e's flat indices f in
 *                     ascending order at rows expert_offsets[e] ..; padding
 *                     rows hold the sentinel M*topk; rows past
 *                     num_tokens_post_padded are not written
 *   expert_ids        INT32 [capacity/block_m] out: local expert of each block
 *   num_tokens_post_padded INT32 [1] out: total padded rows
 *   expert_counts     INT32 [E_local]   out: assignments per local expert
 *   expert_offsets    INT32 [E_local+1] out: exclusive prefix of padded counts
 *   sorted_positions  INT32 [M*topk] out (may be NULL): row of assignment f,
 *                     or -1 if its expert is not local
 *   workspace         device scratch of chord_moe_align_workspace_bytes()
 *                     bytes (may be NULL when that is 0)
 * The per-expert cursors the page calls expert_scatter_offsets live in the
 * workspace and are re-initialised by every call.
 */
size_t chord_moe_align_capacity(int M, int topk, int E_local, int block_m);
size_t chord_moe_align_workspace_bytes(int M, int topk, int E_local);
int chord_moe_align(const int32_t* topk_ids, int M, int topk, int expert_begin, int E_local,
                    int block_m, size_t capacity, int32_t* sorted_token_ids, int32_t* expert_ids,
                    int32_t* num_tokens_post_padded, int32_t* expert_counts,
                    int32_t* expert_offsets, int32_t* sorted_positions, void* workspace,
                    size_t ws_bytes, void* stream);

/* ---------------------------------------------------------- route + align
 * chord_moe_route followed by chord_moe_align in one call, with their
 * arguments and bit-identical outputs ([Router] "코드 분석" and "커널 내부
 * 로직 변경": the fused router kernel also produces the align buffers and
 * re-initialises its counters at entry).  Small calls are one launch of one
 * CTA, which saves a launch and a round trip through the topk_ids buffer: at
 * topk <= 8 up to 4 tokens (four warps route each token, then a ballot-based
 * stable sort of the at most 32 assignments); at larger topk up to 16 tokens
 * or 32 assignments (one warp routes each token, then the stable counting
 * sort).  Larger calls run the two kernels, whose router grid spreads the
 * tokens over many CTAs.
 *   logits, bias, E_total, topk, topk_weights, topk_ids   as chord_moe_route
 *   expert_begin .. sorted_positions, workspace, ws_bytes as chord_moe_align
 *                  (the workspace is needed only when M*topk > 4096)
 * Errors as the two calls; local experts must lie within [0, E_total).
 * The first kernel is launched as chord_moe_route's is.
 */
int chord_moe_route_align(const float* logits, const float* bias, int M, int E_total, int topk,
                          int expert_begin, int E_local, int block_m, size_t capacity,
                          float* topk_weights, int32_t* topk_ids, int32_t* sorted_token_ids,
                          int32_t* expert_ids, int32_t* num_tokens_post_padded, int32_t* expert_counts,
                          int32_t* expert_offsets, int32_t* sorted_positions, void* workspace,
                          size_t ws_bytes, void* stream);

/* Allocation-free variant of chord_moe_align.  The pages have no counterpart;
 * it exists for callers that cannot allocate device memory at all: code
 * running under an engine or plugin that owns every device allocation and
 * hands out no scratch, or a hot path where cudaMalloc is not allowed (it can
 * synchronise the device and is forbidden while a stream is being captured).
 * Arguments, outputs and results are those of chord_moe_align; the only
 * difference is where the scratch lives: when M*topk > 4096 the align needs
 * per-assignment ranks and per-chunk counts, and this entry point keeps them
 * in one static device array inside the library (512 KiB, held by every GPU
 * that loads the library until the process exits) instead of a workspace.
 *   Limits: M*topk <= CHORD_ALIGN_NOALLOC_MAX_ASSIGNMENTS and
 *   E_local <= CHORD_ALIGN_NOALLOC_MAX_EXPERTS; larger calls return
 *   CHORD_ERR_INVALID_ARG and launch nothing.
 *   Set-up: the first call on each device looks up the array's device
 *   address (cudaGetSymbolAddress) with that device current; under lazy
 *   module loading that lookup may be what loads the library's module and
 *   reserves the array.  Make that first call before any stream capture.  It
 *   allocates nothing and calls no cudaMalloc/cudaFree.
 *   Sharing: all calls use the same array and it keeps the last call's
 *   contents (every call rewrites what it reads, so nothing needs clearing);
 *   calls whose executions overlap on the GPU (other streams, other threads)
 *   race on it and must be serialised by the caller.
 */
#define CHORD_ALIGN_NOALLOC_MAX_ASSIGNMENTS 65536
#define CHORD_ALIGN_NOALLOC_MAX_EXPERTS 1024
int chord_moe_align_noalloc(const int32_t* topk_ids, int M, int topk, int expert_begin, int E_local,
                            int block_m, size_t capacity, int32_t* sorted_token_ids,
                            int32_t* expert_ids, int32_t* num_tokens_post_padded,
                            int32_t* expert_counts, int32_t* expert_offsets,
                            int32_t* sorted_positions, void* stream);

/* ---------------------------------------------------------------- prepack
 * Repack INT4 weights and scales into this library's kernel layout
 * ([Humming] "워크로드별 튜닝 및 JIT 컴파일": preprocessing validates
 * parameters, pads dimensions and repacks into the target kernel's layout;
 * [HumPR] "왜 이게 좋은가" 2: automatic padding of shape_n).
 *   qweight  uint8 [E, N, K/2]  two's-complement nibbles, low nibble = even k
 *   scales   BF16  [E, N, K/32] W[e,n,k] = q[e,n,k] * scales[e,n,k/32]
 *   group    must be 32
 *   gate_up  1: rows 0..N/2-1 are the gate projection and N/2..N-1 the up
 *            projection (required for CHORD_EPI_SILU_MUL); 0 otherwise
 *   packed   out, chord_w4a16_prepack_bytes() bytes, 16-byte aligned
 * Requires K % 64 == 0; N % 16 == 0 (gate_up: N % 64 == 0).  N is padded
 * to a multiple of 64 rows with zero weights.  The blob starts with a
 * 256-byte header (magic, version, shapes, flags) that every GEMM launch
 * checks on the device.
 */
size_t chord_w4a16_prepack_bytes(int E, int N, int K, int group);
int chord_w4a16_prepack(const uint8_t* qweight, const chord_bf16* scales, int E, int N, int K,
                        int group, int gate_up, void* packed, size_t packed_bytes, void* stream);

/* ------------------------------------------------------- grouped W4A16 GEMM
 * Indexed MoE GEMM ([Chord] "핵심 기여", "인덱스 커널 기법") over the align
 * buffers ([Router] "코드 분석": sorted_token_ids, expert_ids,
 * num_tokens_post_padded; expert counts and offsets): for every row r of a
 * block b < num_tokens_post_padded / block_m with expert e = expert_ids[b]
 * and r < expert_offsets[e] + expert_counts[e]:
 *   acc[r, n] = sum_k A[row(r), k] * q[e, n, k] * s[e, n, k/32]   (FP32 accumulate)
 * with row(r) = sorted_token_ids[r] / topk when a_gather = 1 (A = the
 * token activations [M, K]) and row(r) = r when a_gather = 0 (A = rows in
 * sorted order [capacity, K], e.g. the gate/up output).
 *   block_m  the BLOCK_M the align buffers were built with
 *   align buffers  as chord_moe_align writes them for this M, topk and
 *            block_m: expert_offsets[e] + expert_counts[e] <= capacity, and
 *            sorted_token_ids below M*topk on every counted row.  The kernels
 *            range-check the block count and the expert ids (recording
 *            CHORD_ERR_INVALID_ARG / CHORD_ERR_ROUTING_INVALID) but do not
 *            re-check every row index against these buffers.
 *   C        BF16 [capacity, N] (STORE) or [capacity, N/2] (SILU_MUL); padding
 *            rows are not written.  CHORD_EPI_WEIGHTED_ADD ([HumPR] "왜 이게
 *            좋은가" 3, moe_fused_mul_sum: the weight multiply and the sum
 *            fused into the GEMM): C is an FP32 [M, N] token-major
 *            accumulator that the caller initialises (zeros, or a partial
 *            sum to add to); every valid row r adds topk_weights[f] *
 *            acc[r, :] to C[f / topk, :] with FP32 atomic adds, f =
 *            sorted_token_ids[r].  The additions of a token's rows happen in
 *            no fixed order, so the low bits of the sum may differ from call
 *            to call; chord_moe_sum is the deterministic alternative.
 *            Needs a_gather = 0 and topk_weights.
 *   topk_weights  FP32 [M, topk] routing weights (CHORD_EPI_WEIGHTED_ADD
 *            only; may be NULL otherwise)
 *   workspace  chord_w4a16_moe_gemm_workspace_bytes() bytes, 16-byte aligned;
 *            zero it once when it is allocated.  Layout: 256 bytes of
 *            work-queue counters, then the split-K area (arrival counters
 *            and partial accumulators, about 4 MB), then, with a_gather = 1
 *            on the tensor-core path, the gathered rows.  Every call leaves
 *            the counters zero (the last CTA of a launch resets the queue,
 *            also after a device timeout; the last split of an item resets
 *            its counter).  After a call that recorded CHORD_ERR_TIMEOUT a
 *            split item may have lost its last split: zero the workspace
 *            again before reusing it.
 *   dev_status  device int for errors found on the device (may be NULL)
 * Two paths ([Humming] "워크로드별 튜닝 및 JIT 컴파일": async-copy + MMA at
 * small batch, TMA + UMMA at large batch), chosen from the expected rows per
 * expert M*topk/E_local unless tuning->path says otherwise: a weight-
 * streaming register-MMA path, and a tcgen05/TMEM path (needs N % 128 == 0).
 * Split-K, gated on grid saturation ([Chord] "인덱스 커널 기법": stream-K
 * only where the grid is not already full): on the register-MMA path, when
 * the launch has at most half as many work items (64 weight rows x one
 * BLOCK_M block) as resident CTAs and block_m <= the rows per pass, the
 * kernel splits K into up to 8 ranges of 512 and the last range of each
 * item to finish adds the FP32 partials in range order, so results are
 * deterministic; it is decided on the device from num_tokens_post_padded.
 * Everything is read on the device, so the call never waits for the host.
 */
size_t chord_w4a16_moe_gemm_workspace_bytes(size_t capacity, int K, int a_gather);
int chord_w4a16_moe_gemm(const chord_bf16* A, int a_gather, const void* packed_w, int E_local,
                         int N, int K, int M, int topk, const int32_t* sorted_token_ids,
                         const int32_t* expert_ids, const int32_t* num_tokens_post_padded,
                         const int32_t* expert_counts, const int32_t* expert_offsets, int block_m,
                         size_t capacity, int epilogue, const float* topk_weights, void* C,
                         const chord_tuning* tuning, void* workspace, size_t ws_bytes, int* dev_status,
                         void* stream);

/* ------------------------------------------------------- dense W4A16 GEMM
 * C = A * (q*s)^T for one weight matrix, no routing: the indexed GEMM above
 * with every row belonging to a single expert ([Humming] "통합 양자화 표현":
 * one weight format serves dense and MoE layers).  packed_w is a
 * chord_w4a16_prepack blob with E = 1.
 *   A          BF16 [M, K] (16-byte aligned)
 *   C          BF16 [M, N] (STORE) or [M, N/2] (SILU_MUL)
 *   workspace  chord_w4a16_gemm_workspace_bytes(M) bytes, 16-byte aligned;
 *              zero it once when allocated (its work-queue and split-K
 *              counters are left zero by every call); each call writes the
 *              one-expert block map into it on the device
 * Path and rows per pass as chord_w4a16_moe_gemm with M rows per expert,
 * unless tuning says otherwise.  Errors as chord_w4a16_moe_gemm.
 */
size_t chord_w4a16_gemm_workspace_bytes(int M);
int chord_w4a16_gemm(const chord_bf16* A, const void* packed_w, int N, int K, int M, int epilogue,
                     chord_bf16* C, const chord_tuning* tuning, void* workspace, size_t ws_bytes,
                     int* dev_status, void* stream);

/* ------------------------------------------------------- grouped layouts
 * The grouped kernels' activation layouts ([Chord] "그룹 SM90 커널 기법":
 * contiguous prefill pads each expert to a 128-row boundary; masked decode
 * reserves a fixed row budget per expert and picks BLOCK_M from the expected
 * token count).  The rows are already grouped by expert: no routing, no
 * gather.  For each expert e and each of its group_rows[e] rows r:
 *   C[r, :] = A[r, :] (q_e s_e)^T          (epilogue CHORD_EPI_STORE), or
 *   C[r, :] = SiLU(gate) * up              (CHORD_EPI_SILU_MUL, N = 2I)
 * with packed_w the prepacked [E, N, K] blob (gate_up = 1 for SiLU*mul).
 *   contiguous: A BF16 [a_rows, K]; expert e's rows start at
 *     sum_{e' < e} ceil(group_rows[e'] / 128) * 128 and run for
 *     group_rows[e]; the padded total must be <= a_rows.
 *   masked: A BF16 [E, max_m, K] (max_m a multiple of 16); expert e's rows
 *     are its first group_rows[e] <= max_m rows.
 *   group_rows   device INT32 [E], 1 <= E <= 1024
 *   expected_m   rows per expert the plan assumes (<= 0: a_rows / E for
 *                contiguous, max_m for masked): picks the register-MMA or
 *                tcgen05 path and BLOCK_M, as chord_w4a16_moe_gemm does
 *   C            BF16, the same row layout as A, N (STORE) or N/2 columns;
 *                rows past an expert's group_rows are not written
 *   workspace    chord_w4a16_grouped_workspace_bytes(E, rows of A) bytes,
 *                16-byte aligned, zeroed once when allocated (its counters
 *                are left zero by every call)
 * Host-side errors return CHORD_ERR_* and launch nothing; a count outside
 * [0, max_m] (masked) or a padded total above the rows of A (contiguous) is
 * recorded in *dev_status as CHORD_ERR_INVALID_ARG and nothing is computed.
 */
size_t chord_w4a16_grouped_workspace_bytes(int E, size_t rows);
int chord_w4a16_grouped_gemm_contiguous(const chord_bf16* A, size_t a_rows, const int32_t* group_rows, int E,
                                        int expected_m, const void* packed_w, int N, int K, int epilogue,
                                        chord_bf16* C, const chord_tuning* tuning, void* workspace,
                                        size_t ws_bytes, int* dev_status, void* stream);
int chord_w4a16_grouped_gemm_masked(const chord_bf16* A, const int32_t* group_rows, int E, int max_m,
                                    int expected_m, const void* packed_w, int N, int K, int epilogue,
                                    chord_bf16* C, const chord_tuning* tuning, void* workspace, size_t ws_bytes,
                                    int* dev_status, void* stream);

/* --------------------------------------------------------- top-k weighted sum
 * moe_fused_mul_sum ([HumPR] "왜 이게 좋은가" 3: weight multiply and sum):
 *   out[t, :] = sum over j = 0..topk-1 with sorted_positions[t*topk+j] >= 0 of
 *               topk_weights[t, j] * y[sorted_positions[t*topk+j], :]
 * accumulated in FP32 in increasing j, rounded once to BF16.  A token with
 * no local assignment gets zeros.  Requires H % 8 == 0 and topk <= 32.
 */
int chord_moe_sum(const chord_bf16* y, const float* topk_weights, const int32_t* sorted_positions,
                  int M, int topk, int H, chord_bf16* out, void* stream);

/* ------------------------------------------------------------- whole layer
 * One MoE layer on this GPU's expert shard: route, align, gate/up GEMM with
 * fused SiLU*mul, down GEMM, top-k weighted sum ([Chord] "핵심 기여").
 *   x            BF16 [M, H]
 *   logits, bias as chord_moe_route (E_total experts)
 *   w13_packed   prepacked gate|up weights [E_local, 2I, H] (gate_up = 1)
 *   w2_packed    prepacked down weights [E_local, H, I]
 *   out          BF16 [M, H]
 *   topk_weights_out FP32 [M, topk], topk_ids_out INT32 [M, topk]: optional
 *                copies of the routing (may be NULL)
 *   workspace    chord_moe_layer_workspace_bytes() bytes, 16-byte aligned,
 *                any contents (every call's first kernel clears the
 *                counters the later kernels use); it holds the routing,
 *                the align buffers, h, y,
 *                and the GEMMs' work-queue and split-K state
 * The expert-parallel shard is implied by E_local < E_total ([Chord]
 * "런타임 고려사항": the profile is inferred from the shapes, no shard
 * argument).  Weights are normalised over all topk experts, local or not.
 * Launch order: the first kernel (the router) is launched as
 * chord_moe_route's is, so it touches no memory before all earlier work in
 * the stream has completed.  On the register-MMA path every later kernel of
 * the call is a programmatic dependent launch: it may start before the previous kernel of the call ends and waits
 * for it before reading its outputs (captured into a CUDA graph, these
 * become programmatic edges).  Work enqueued after the call starts after
 * its last kernel ends.
 */
size_t chord_moe_layer_workspace_bytes(int M, int H, int I, int E_local, int topk);
/* Host-only: the tuning chord_moe_layer uses for these shapes (tokens-per-
 * expert policy, [Chord] "인덱스 커널 기법": the schedule follows the tokens
 * delivered per expert, tok_e = M*topk/E_total; the tcgen05 path from
 * tok_e >= 12, where the two paths measured even on GB300, the register-MMA
 * path below it with 8, 16 or 32 rows per pass).  Writes *plan; returns
 * CHORD_OK or CHORD_ERR_INVALID_ARG.  Passing the plan to
 * chord_w4a16_moe_gemm reproduces the layer's launches exactly. */
int chord_moe_layer_plan(int M, int E_total, int topk, chord_tuning* plan);
int chord_moe_layer(const chord_bf16* x, const float* logits, const float* bias,
                    const void* w13_packed, const void* w2_packed, int M, int H, int I,
                    int E_total, int expert_begin, int E_local, int topk, chord_bf16* out,
                    float* topk_weights_out, int32_t* topk_ids_out, void* workspace,
                    size_t ws_bytes, const chord_tuning* tuning, int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* CHORD_MOE_H */
