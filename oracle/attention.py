"""Plain fp64 two-pass attention forward: the definition, written out.

TEST INFRASTRUCTURE ONLY. This file is the oracle that the CUDA path is checked
against. Only the tests, the package's smoke entry and the benchmark's CPU
baseline leg may import it; the library never does, and it shares no code with
the CUDA kernels.

What it computes (for every batch b and query head h):

    S = scale * Q_bh K_bh^T                      (N x N, fp64, fully materialised)
    S[i, j] = -inf for j > i                     (causal only, top-left aligned)
    m_i = max_j S[i, j]                          (pass 1)
    P[i, j] = exp(S[i, j] - m_i),  l_i = sum_j P[i, j]          (pass 2)
    O_i = (P[i] / l_i) V_bh,       LSE_i = m_i + ln(l_i)

Sources:
  * "FlashAttention-3 Deep Dive" (mojostudio.in), introduction: the attention
    formula softmax(Q K^T / sqrt(d_k)) V, and section 3: P_ij = exp(S_ij - m_i).
  * "flash-attention-3" (ai.thesatyajit.com), opening paragraph: the fused kernel
    reaches this same result without writing the N x N scores to memory.
  * "Hopper" tag page (l1-ca0.github.io), section titles 3.2 "Safe softmax and
    its streaming state" and 4.6 "rescaling, correction, and LSE" name the
    subtract-the-max softmax and the per-row log-sum-exp; the formulas of that
    page did not survive, so LSE is read as the natural-log log-sum-exp of the
    scaled scores.
  * "flash-attention-3", "What is actually in the box": GQA is supported; the
    mapping is read as contiguous groups, kv head = h // (H / Hkv).

Rows whose scores are all masked cannot occur with top-left causal masking and
equal query/key lengths; if one ever did, it is defined as O = 0, LSE = -inf.

Parity pins live in tests/test_oracle.py; every function here is pinned.
"""
from __future__ import annotations

import numpy as np


def kv_head(h: int, H: int, Hkv: int) -> int:
    """GQA: query head h reads kv head h // (H / Hkv) (contiguous groups)."""
    if H % Hkv != 0:
        raise ValueError("H must be a multiple of Hkv")
    return h // (H // Hkv)


def scores(q_bh: np.ndarray, k_bh: np.ndarray, scale: float, causal: bool,
           rows: np.ndarray | None = None, causal_offset: int = 0) -> np.ndarray:
    """Scaled, masked score rows S[i, :] for query rows ``rows`` (default: all).

    q_bh: [Nq, d], k_bh: [Nk, d]. Causal masks keys j > i + causal_offset (offset 0: top-left
    alignment; offset Nk - Nq: bottom-right alignment, used for ragged batches).
    """
    q_bh = np.asarray(q_bh, dtype=np.float64)
    k_bh = np.asarray(k_bh, dtype=np.float64)
    if rows is None:
        rows = np.arange(q_bh.shape[0])
    s = np.float64(scale) * (q_bh[rows] @ k_bh.T)
    if causal:
        j = np.arange(k_bh.shape[0])[None, :]
        s = np.where(j > np.asarray(rows)[:, None] + causal_offset, -np.inf, s)
    return s


def softmax_two_pass(s: np.ndarray):
    """Row softmax of ``s`` in two passes. Returns (P, m, l) with P rows summing to 1."""
    m = s.max(axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 for masked entries
    l = e.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        p = np.where(l[:, None] > 0, e / l[:, None], 0.0)
    return p, m, l


def attention_head(q_bh, k_bh, v_bh, scale: float, causal: bool,
                   rows: np.ndarray | None = None, row_chunk: int = 1024, causal_offset: int = 0):
    """O and LSE for one (batch, head): q_bh [Nq, d], k_bh/v_bh [Nk, d].

    Rows are processed in chunks of ``row_chunk`` only to bound memory; every
    score row is still materialised in full. A row whose keys are all masked
    (or with no keys at all) has O = 0 and LSE = -inf.
    """
    q_bh = np.asarray(q_bh, dtype=np.float64)
    k_bh = np.asarray(k_bh, dtype=np.float64)
    v_bh = np.asarray(v_bh, dtype=np.float64)
    if rows is None:
        rows = np.arange(q_bh.shape[0])
    rows = np.asarray(rows)
    o = np.zeros((rows.size, v_bh.shape[1]), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    for c0 in range(0, rows.size, row_chunk):
        r = rows[c0:c0 + row_chunk]
        s = scores(q_bh, k_bh, scale, causal, rows=r, causal_offset=causal_offset)
        p, m, l = softmax_two_pass(s)
        o[c0:c0 + r.size] = p @ v_bh
        with np.errstate(divide="ignore"):
            lse[c0:c0 + r.size] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse


def attention_forward(q, k, v, scale: float, causal: bool, heads=None, rows=None):
    """Attention forward over [B, N, H, d] q and [B, N, Hkv, d] k, v (fp64).

    Returns (O [B, N, H, d], LSE [B, H, N]) for all heads, or, when ``heads`` is
    a list of (b, h) pairs, a dict {(b, h): (O_bh [len(rows), d], LSE_bh)} for
    those heads and the query rows ``rows`` (default all).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if heads is not None:
        out = {}
        for (b, h) in heads:
            kh = kv_head(h, H, Hkv)
            out[(b, h)] = attention_head(q[b, :, h, :], k[b, :, kh, :], v[b, :, kh, :],
                                         scale, causal, rows=rows)
        return out
    o = np.empty((B, N, H, v.shape[3]), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            kh = kv_head(h, H, Hkv)
            o_bh, lse_bh = attention_head(q[b, :, h, :], k[b, :, kh, :], v[b, :, kh, :], scale, causal)
            o[b, :, h, :] = o_bh
            lse[b, h, :] = lse_bh
    return o, lse


def probabilities(q, k, scale: float, causal: bool):
    """Full softmax matrix P [B, H, N, N] (small inputs only)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    B, N, H, _ = q.shape
    Hkv = k.shape[2]
    p = np.empty((B, H, N, k.shape[1]))
    for b in range(B):
        for h in range(H):
            kh = kv_head(h, H, Hkv)
            p[b, h] = softmax_two_pass(scores(q[b, :, h, :], k[b, :, kh, :], scale, causal))[0]
    return p
