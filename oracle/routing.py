"""Router oracle: sigmoid scores, score+bias top-k, normalised weights.

The router's buffers (logits FP32 [M, E], bias FP32 [E] in; topk_weights,
topk_ids out) are those of the fused router's argument plan in [Router]
"코드 분석".  The page does not print the rule; the rule implemented is the
Kimi-K2 one:

  s_e   = sigmoid(logit_e)                      (binary32, op sequence below)
  key_e = fl32(s_e + bias_e)
  ids   = the k experts with the largest key; equal keys -> lower id first;
          emitted in rank order (largest key first)
  S     = s_ids[0] + s_ids[1] + ... + s_ids[k-1]  (binary32, left to right)
  w_j   = fl32(s_ids[j] / S)                      (un-biased scores, scale 1.0)

[Router] "리뷰 피드백 반영" states that routing outputs are compared bit for
bit.  To make bit-exact GPU/CPU agreement possible, the sigmoid is specified
as an explicit binary32 op sequence (every step rounds to nearest even, no
fused multiply-add), written here from the mathematics:

  y  = clamp(-x, -87, 87)
  n  = rint(y * LOG2E)                  (ties to even)
  r  = (y - n*LN2_HI) - n*LN2_LO        (Cody-Waite reduction, |r| <~ ln2/2;
                                         LN2_HI = ln2 rounded down to 16
                                         fractional bits, so n*LN2_HI is exact)
  p  = Horner over the degree-7 Taylor series of e^r, coefficients 1/j!
       rounded to binary32, each step a rounded multiply then a rounded add
  e  = p * 2^n                          (exact power-of-two scaling)
  s  = 1 / (1 + e)

The clamp only changes results for |x| > 87, where s already rounds to 1.0
or is below 2e-38 and cannot change a key fl32(s + bias) unless bias == 0.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32
LOG2E = F32(1.0 / math.log(2.0))
LN2_HI = F32(math.floor(math.log(2.0) * 65536.0) / 65536.0)     # 0.693145751953125
LN2_LO = F32(math.log(2.0) - float(LN2_HI))
TAYLOR = [F32(1.0 / math.factorial(j)) for j in range(8)]       # 1/0! .. 1/7!
CLAMP = F32(87.0)


def exp_binary32(y) -> np.ndarray:
    """e^y in binary32 by the op sequence above; requires |y| <= 87."""
    y = np.asarray(y, dtype=F32)
    n = np.rint(y * LOG2E)
    r = y - n * LN2_HI
    r = r - n * LN2_LO
    p = np.full_like(r, TAYLOR[7])
    for c in TAYLOR[6::-1]:
        p = p * r
        p = p + c
    two_n = ((n.astype(np.int32) + 127) << 23).astype(np.int32).view(F32)
    return p * two_n


def sigmoid_binary32(x) -> np.ndarray:
    """1 / (1 + e^-x) with the specified binary32 op sequence."""
    x = np.asarray(x, dtype=F32)
    y = np.clip(-x, -CLAMP, CLAMP)
    e = exp_binary32(y)
    return F32(1.0) / (F32(1.0) + e)


def route(logits, bias, topk: int):
    """Return (topk_weights FP32 [M, k], topk_ids INT32 [M, k], scores FP32 [M, E])."""
    logits = np.asarray(logits, dtype=F32)
    bias = np.asarray(bias, dtype=F32)
    M, E = logits.shape
    if not (1 <= topk <= E):
        raise ValueError("topk must be in [1, E]")
    s = sigmoid_binary32(logits)
    key = s + bias[None, :]
    # stable ascending sort of -key == key descending with ties kept in id order
    order = np.argsort(-key, axis=1, kind="stable")
    ids = order[:, :topk]
    s_sel = np.take_along_axis(s, ids, axis=1)
    S = s_sel[:, 0].copy()
    for j in range(1, topk):
        S = S + s_sel[:, j]
    w = s_sel / S[:, None]
    return w.astype(F32), ids.astype(np.int32), s
