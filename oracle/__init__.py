"""CPU oracle for the W4A16 INT4-weight MoE layer with sigmoid+bias routing.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
CPU-baseline leg of the benchmark may import this package.  The product
(the CUDA library and its Python binding) never imports, links or runs it,
and this package never imports the product: the two share no code.

What it is: a plain, slow, obviously correct restatement of what the layer
computes, in numpy.  Routing decisions are taken in binary32 with an op
sequence written out step by step (so a GPU kernel can take the very same
decisions); everything after routing is FP64 with exact dequantisation.
Library primitives used as single steps: numpy's stable argsort and FP64
matmul.  Nothing is blocked, fused or reordered beyond the definitions.

Sources, cited by page title and section:
  [Chord]   "vLLM 및 Novita AI, Kimi K2.x용 더 빠른 INT4 MoE 커널 출시: Chord"
  [HumPR]   "[vllm] vLLM에 고성능 JIT 양자화 커널 'Humming' 도입하기"
  [Router]  "[flashinfer] FlashInfer, B200 GPU에서 Kimi-K3 MoE 라우터 성능 최적화"
  [Humming] "Humming: vLLM과 Ant Group, 양자화 추론을 위한 범용 커널 라이브러리
             오픈소스 공개"
The pages name the buffers of the path (logits, bias, topk_weights/ids,
sorted_token_ids, expert_ids, num_tokens_post_padded, expert counts/offsets:
[Router] "코드 분석", arg_plan) and the W4A16 format (INT4 weights with
group-32 BF16 scales, BF16 activations: [Chord] "TL;DR", "런타임 고려사항";
[Humming] "통합 양자화 표현").  They do not print the routing rule or the
expert MLP; those follow the Kimi-K2 layer definition (sigmoid scores,
top-k on score + bias with ties to the lower id, weights = selected scores
normalised to sum 1, SiLU-gated expert MLP), and every reading taken where
the pages are silent is listed in the module that takes it.

Parity status: every function here is pinned by tests in tests/test_oracle_*.py
(closed forms, brute force, invariants, hand-worked cases); none is unpinned.
"""
from .routing import sigmoid_binary32, exp_binary32, route
from .align import align_capacity, moe_align
from .quant import bf16_to_f64, unpack_int4, dequant, dequant_expert
from .layer import (silu, expert_rows_gemm, silu_mul, moe_sum, moe_layer,
                    moe_layer_tokens)
from .grouped import group_starts, grouped_gemm

__all__ = [
    "sigmoid_binary32", "exp_binary32", "route", "align_capacity", "moe_align",
    "bf16_to_f64", "unpack_int4", "dequant", "dequant_expert", "silu",
    "expert_rows_gemm", "silu_mul", "moe_sum", "moe_layer", "moe_layer_tokens",
    "group_starts", "grouped_gemm",
]
