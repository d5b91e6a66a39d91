"""Align oracle: moe_align_block_size (sort and pad token->expert assignments).

Buffers follow [Router] "코드 분석" (arg_plan: sorted_token_ids, expert_ids,
num_tokens_post_padded, expert_counts, expert_offsets) and [Chord]
"런타임 고려사항" (kernels run on over-allocated align buffers; entries past
num_tokens_post_padded are never read).  Readings where the pages are silent:

  * assignment (t, j) has flat index f = t*k + j; its expert is topk_ids[t, j];
    only experts in [expert_begin, expert_begin + E_local) are kept (an
    expert-parallel shard); the others are dropped;
  * cnt_e = number of kept assignments of local expert e;
    pad_e = ceil(cnt_e / BLOCK_M) * BLOCK_M (an empty expert gets no block);
  * off_e = sum of pad over experts before e; ntpp = off_{E_local};
  * sorted_token_ids[off_e + i] = the i-th flat index (ascending) of expert e
    (a stable sort); slots off_e + cnt_e .. off_e + pad_e - 1 hold the
    sentinel M*k;
  * expert_ids[b] = the local expert owning rows b*BLOCK_M .. (b+1)*BLOCK_M-1;
  * sorted_positions[f] = the row of flat index f, or -1 if dropped (the
    inverse map the top-k weighted sum reads).
"""
from __future__ import annotations

import numpy as np


def align_capacity(M: int, topk: int, E_local: int, block_m: int) -> int:
    """Rows the align buffers need: sum_e ceil(cnt_e/BM)*BM can reach at most
    R + min(E_local, R) * (BM - 1) with R = M*k, rounded up to BM."""
    R = M * topk
    cap = R + min(E_local, R) * (block_m - 1)
    return ((cap + block_m - 1) // block_m) * block_m


def moe_align(topk_ids, expert_begin: int, E_local: int, block_m: int):
    topk_ids = np.asarray(topk_ids)
    M, k = topk_ids.shape
    flat = topk_ids.reshape(-1).astype(np.int64)
    local = flat - expert_begin
    keep = (local >= 0) & (local < E_local)
    counts = np.bincount(local[keep], minlength=E_local).astype(np.int64)
    padded = ((counts + block_m - 1) // block_m) * block_m
    offsets = np.zeros(E_local + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    ntpp = int(offsets[-1])
    sentinel = M * k
    sorted_ids = np.full(ntpp, sentinel, dtype=np.int64)
    positions = np.full(M * k, -1, dtype=np.int64)
    for e in range(E_local):
        f = np.nonzero(keep & (local == e))[0]           # ascending flat indices
        rows = offsets[e] + np.arange(f.size)
        sorted_ids[rows] = f
        positions[f] = rows
    expert_ids = np.repeat(np.arange(E_local, dtype=np.int64), padded // block_m)
    return dict(
        sorted_token_ids=sorted_ids.astype(np.int32),
        expert_ids=expert_ids.astype(np.int32),
        num_tokens_post_padded=ntpp,
        expert_counts=counts.astype(np.int32),
        expert_offsets=offsets.astype(np.int32),
        sorted_positions=positions.astype(np.int32),
    )
