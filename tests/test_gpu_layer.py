"""GPU parity: the whole layer (chord_moe_layer) against the FP64 oracle.

Small shapes are compared on every output element; the Kimi-K2 workloads are
run at full size in the same call the benchmark times, and compared on a
seeded sample of tokens that the oracle computes one by one."""
import numpy as np
import pytest
import torch

import oracle
from w4a16_int4_weight_sigmoid_gb300 import chord
from w4a16_int4_weight_sigmoid_gb300 import workload as wl
from w4a16_int4_weight_sigmoid_gb300.layer import W4A16MoELayer

from gpu_util import assert_close_to_oracle, bf16_to_np, ensure_lib, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def run_layer(shape, d, **kw):
    layer = W4A16MoELayer(d["w13_q"], d["w13_s"], d["w2_q"], d["w2_s"], shape.E_total,
                          shape.expert_begin, shape.topk)
    M = shape.M
    tw = torch.empty((M, shape.topk), dtype=torch.float32, device="cuda")
    ti = torch.empty((M, shape.topk), dtype=torch.int32, device="cuda")
    out = layer.forward(to_device(d["x"]), to_device(d["logits"]), to_device(d["bias"]),
                        topk_weights_out=tw, topk_ids_out=ti, **kw)
    torch.cuda.synchronize()
    assert layer.dev_status.item() == 0
    return layer, bf16_to_np(out), tw.cpu().numpy(), ti.cpu().numpy()


def small(name, M, H, I, E_total, E_local, begin, topk, seed, zipf=0.0):
    return wl.LayerShape(name, M, H, I, E_total, E_local, begin, topk, seed, zipf)


SMALL = [
    wl.TINY,
    small("ep_shard_ragged", 40, 512, 256, 16, 6, 5, 4, 21),
    small("tp_zipf", 48, 256, 192, 32, 32, 0, 6, 22, zipf=1.1),
    small("single_token", 1, 384, 128, 12, 12, 0, 3, 23),
    small("top1_one_expert", 9, 128, 64, 1, 1, 0, 1, 24),
    small("many_rows_per_expert", 256, 256, 128, 4, 4, 0, 2, 25),
]


def test_layer_fresh_workspace_every_call():
    """The register-MMA path chains its kernels with programmatic launches:
    each kernel must read the previous kernel's outputs only after waiting
    for it.  A fresh workspace per call, filled with a pattern that cannot
    be a valid block map (0x7F bytes, 0xFF bytes: counters of 2^31 - 1 - ...
    and -1) or with zeros, exposes any read that comes too early, as a device
    status or as a wrong output; the work-queue counters in it are cleared by
    the router kernel, on both GEMM paths."""
    shape = small("tp_zipf_fresh_ws", 48, 256, 192, 32, 32, 0, 6, 22, zipf=1.1)
    d = wl.layer_inputs(shape)
    ref, _, _ = oracle.moe_layer(d["x"], d["logits"], d["bias"], d["w13_q"], d["w13_s"],
                                 d["w2_q"], d["w2_s"], shape.topk, shape.expert_begin)
    layer = W4A16MoELayer(d["w13_q"], d["w13_s"], d["w2_q"], d["w2_s"], shape.E_total,
                          shape.expert_begin, shape.topk)
    x, lg, b = to_device(d["x"]), to_device(d["logits"]), to_device(d["bias"])
    n = layer.workspace(shape.M).numel()
    large = chord.chord_tuning(chord.CHORD_PATH_LARGE_M, 0, 0, 0)
    for i in range(48):
        layer._ws = torch.full((n,), (0, 0x7F, 0xFF)[i % 3], dtype=torch.uint8, device="cuda")
        out = layer.forward(x, lg, b, tuning=large if i >= 24 else None)
        torch.cuda.synchronize()
        assert layer.dev_status.item() == 0, f"call {i}: device status {layer.dev_status.item()}"
        got = bf16_to_np(out)
        if i in (0, 24):   # each path against the oracle, then against itself
            assert_close_to_oracle(got, ref, shape.name)
            first = got
        else:
            assert np.array_equal(got, first), f"call {i} differs"


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: s.name)
def test_layer_small_full_parity(shape):
    d = wl.layer_inputs(shape)
    ref, w, ids = oracle.moe_layer(d["x"], d["logits"], d["bias"], d["w13_q"], d["w13_s"],
                                   d["w2_q"], d["w2_s"], shape.topk, shape.expert_begin)
    for _ in range(2):
        _, got, gw, gids = run_layer(shape, d)
        assert np.array_equal(gids, ids)
        assert np.array_equal(gw.view(np.uint32), w.view(np.uint32))
        assert_close_to_oracle(got, ref, shape.name)


def test_layer_tokens_without_local_experts_are_zero():
    shape = small("shard_far", 24, 256, 128, 64, 4, 60, 2, 26)
    d = wl.layer_inputs(shape)
    _, got, _, gids = run_layer(shape, d)
    none_local = ~np.any((gids >= 60) & (gids < 64), axis=1)
    assert none_local.any()
    assert np.all(got[none_local] == 0)


@pytest.mark.parametrize("shape", [wl.EP8_DECODE, wl.TP8_DECODE, wl.EP8_PREFILL],
                         ids=lambda s: s.name)
def test_layer_kimi_workloads_sampled(shape):
    d = wl.layer_inputs(shape)
    _, got, gw, gids = run_layer(shape, d)
    w, ids, _ = oracle.route(d["logits"], d["bias"], shape.topk)
    assert np.array_equal(gids, ids)
    assert np.array_equal(gw.view(np.uint32), w.view(np.uint32))
    rng = np.random.default_rng(shape.seed)
    local = np.any((ids >= shape.expert_begin) & (ids < shape.expert_begin + shape.E_local), axis=1)
    cand = np.nonzero(local)[0]
    # every touched local expert contributes the tokens of its first and last
    # assignment (its first and last sorted rows, so the first and the last
    # pass of an expert whose rows take several passes), plus a seeded sample
    flat = ids.ravel()
    chosen = set(rng.choice(cand, size=min(6, cand.size), replace=False).tolist())
    for e in range(shape.expert_begin, shape.expert_begin + shape.E_local):
        f = np.nonzero(flat == e)[0]
        if f.size:
            chosen.update((int(f[0]) // shape.topk, int(f[-1]) // shape.topk))
    tokens = np.array(sorted(chosen), dtype=np.int64)
    ref = oracle.moe_layer_tokens(tokens, d["x"], d["logits"], d["bias"], d["w13_q"], d["w13_s"],
                                  d["w2_q"], d["w2_s"], shape.topk, shape.expert_begin)
    assert_close_to_oracle(got[tokens], ref, shape.name)
    assert np.all(np.isfinite(got))


# Few tokens with K of several 512-wide stages: the decode GEMM sees far fewer
# work items than resident CTAs and splits K (split-K gated on the grid);
# every output element against the oracle, and repeated calls bit-identical
# (the split partials are added in split order whatever CTA finishes last).
SPLIT_K = [
    small("split_k_two_tokens", 2, 2048, 512, 32, 8, 0, 4, 27),
    small("split_k_one_token_both_gemms", 1, 1024, 1024, 8, 4, 0, 2, 28),
    small("split_k_ragged_shard", 3, 1536, 768, 24, 6, 3, 5, 29),
]


@pytest.mark.parametrize("shape", SPLIT_K, ids=lambda s: s.name)
def test_layer_split_k_full_parity(shape):
    d = wl.layer_inputs(shape)
    ref, w, ids = oracle.moe_layer(d["x"], d["logits"], d["bias"], d["w13_q"], d["w13_s"],
                                   d["w2_q"], d["w2_s"], shape.topk, shape.expert_begin)
    first = None
    for _ in range(3):
        _, got, gw, gids = run_layer(shape, d)
        assert np.array_equal(gids, ids)
        assert_close_to_oracle(got, ref, shape.name)
        if first is None:
            first = got
        else:
            assert np.array_equal(got, first), "split-K result changed between calls"


@pytest.mark.parametrize("M", [1, 4])
def test_layer_kimi_ep8_few_tokens(M):
    """Kimi-K2 EP8 shapes at 1 and 4 tokens: the split-K decode path on both
    GEMMs (64 and 112 weight tiles against 608 resident CTAs), every token
    against the oracle."""
    base = wl.EP8_DECODE
    shape = wl.LayerShape(f"kimi_ep8_m{M}", M, base.H, base.I, base.E_total, base.E_local, 0,
                          base.topk, 31 + M)
    d = wl.layer_inputs(shape)
    _, got, gw, gids = run_layer(shape, d)
    w, ids, _ = oracle.route(d["logits"], d["bias"], shape.topk)
    assert np.array_equal(gids, ids)
    ref = oracle.moe_layer_tokens(np.arange(M), d["x"], d["logits"], d["bias"], d["w13_q"], d["w13_s"],
                                  d["w2_q"], d["w2_s"], shape.topk, shape.expert_begin)
    assert_close_to_oracle(got, ref, shape.name)
