"""Gradients of the attention forward (dQ, dK, dV) from the definition, fp64 CPU.

TEST INFRASTRUCTURE ONLY. This file is part of the oracle that the CUDA path is
checked against. Only the tests, the package's smoke entry and the benchmark's
CPU baseline leg may import it; the library never does, and it shares no code
with the CUDA kernels.

What it computes, for one (batch, query head) with S = scale Q K^T (+ mask),
P = softmax(S) by rows and O = P V, given the output gradient dO:

    dV = P^T dO
    dP = dO V^T
    D_i = sum_j P_ij dP_ij  ( = sum_c dO_ic O_ic )
    dS = P * (dP - D)                  (elementwise; each row of dS sums to zero)
    dQ = scale dS K
    dK = scale dS^T Q

With grouped query heads, the dK and dV of a kv head are the sums over its
query heads. P is recomputed from the definition; nothing from a forward run
is reused.

Sources:
  * "flash-attention-3" (ai.thesatyajit.com), "Five schedulers": the backward
    pass and its longest-first scheduler for causal masking; and the overview
    table: FP16 / BF16 backward.
  * "FlashAttention-3 Deep Dive" (mojostudio.in) table of contents, sections on
    backward recomputation, the preprocess (D and the base-2 LSE), dQ
    accumulation, and the GQA path for dK and dV: the section titles only; the
    formulas above are the derivative of the forward's definition (the softmax
    Jacobian diag(P_i) - P_i P_i^T applied row by row), written out here.

Parity pins live in tests/test_oracle_backward.py.
"""
from __future__ import annotations

import numpy as np

from .attention import kv_head, scores, softmax_two_pass


def attention_backward_head(q_bh, k_bh, v_bh, do_bh, scale: float, causal: bool, causal_offset: int = 0):
    """(dQ [Nq, d], dK [Nk, d], dV [Nk, d], D [Nq]) for one (batch, head)."""
    q = np.asarray(q_bh, dtype=np.float64)
    k = np.asarray(k_bh, dtype=np.float64)
    v = np.asarray(v_bh, dtype=np.float64)
    do = np.asarray(do_bh, dtype=np.float64)
    s = scores(q, k, scale, causal, causal_offset=causal_offset)
    p, _, _ = softmax_two_pass(s)
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    d_row = (do * o).sum(axis=1)
    ds = p * (dp - d_row[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv, d_row


def attention_backward(q, k, v, do, scale: float, causal: bool):
    """Gradients over [B, N, H, d] q / dO and [B, N, Hkv, d] k, v: (dQ, dK, dV, D [B, H, N])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    dd = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            kh = kv_head(h, H, Hkv)
            gq, gk, gv, drow = attention_backward_head(q[b, :, h], k[b, :, kh], v[b, :, kh], do[b, :, h], scale, causal)
            dq[b, :, h] = gq
            dk[b, :, kh] += gk
            dv[b, :, kh] += gv
            dd[b, h] = drow
    return dq, dk, dv, dd
