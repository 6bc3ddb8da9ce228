"""Tiled online-softmax attention in fp64: the streaming recurrence, for tiny inputs.

TEST INFRASTRUCTURE ONLY (see oracle/attention.py). Written separately from the
two-pass definition so the two can check each other; neither imports the other.

The recurrence (per query block of Br rows, walking key blocks of Bc columns):

    S_j    = scale * Q_i K_j^T, causal entries j > i set to -inf
    m_new  = max(m, rowmax(S_j))
    P_j    = exp(S_j - m_new)
    l      = l * exp(m - m_new) + rowsum(P_j)
    O_acc  = O_acc * exp(m - m_new) + P_j V_j
    m      = m_new
  and, after the last key block, O = O_acc / l, LSE = m + ln(l).

Sources:
  * "flash-attention-3" (ai.thesatyajit.com), opening paragraph: tile the
    computation and keep a running softmax so the N x N scores never reach memory.
  * "FlashAttention-3 Deep Dive" (mojostudio.in), section 3: P_ij = exp(S_ij - m_i)
    computed per tile, overlapped with the two GEMMs.
  * "Lecture 9 — Hopper / FlashAttention-3 / FlashAttention-4", "Warp
    specialisation in FA3": the consumer does rescale, exp, rowmax/rowsum
    between WGMMA(Q, K^T) and WGMMA(P, V).
  * "Hopper" tag page (l1-ca0.github.io), section titles 3.2.1 "The block-combine
    interpretation", 3.4.1 "Fewer non-matrix operations" (normalise once at the
    end) and 4.2 "Online-softmax state and invariant".

Pure-Python loops over blocks; meant for N <= a few hundred.
"""
from __future__ import annotations

import numpy as np


def attention_online(q, k, v, scale: float, causal: bool, Br: int, Bc: int):
    """Online-softmax forward with block sizes (Br, Bc); same I/O as the two-pass oracle."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, N, H, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    group = H // Hkv
    o = np.zeros((B, N, H, v.shape[3]))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            kh = h // group
            for i0 in range(0, N, Br):
                i1 = min(N, i0 + Br)
                qi = q[b, i0:i1, h, :]
                m = np.full(i1 - i0, -np.inf)
                l = np.zeros(i1 - i0)
                acc = np.zeros((i1 - i0, v.shape[3]))
                for j0 in range(0, Nk, Bc):
                    j1 = min(Nk, j0 + Bc)
                    s = np.float64(scale) * (qi @ k[b, j0:j1, kh, :].T)
                    if causal:
                        ii = np.arange(i0, i1)[:, None]
                        jj = np.arange(j0, j1)[None, :]
                        s = np.where(jj > ii, -np.inf, s)
                    m_new = np.maximum(m, s.max(axis=1))
                    # Rows with nothing unmasked yet keep m = -inf; use 0 as the shift there.
                    shift = np.where(np.isfinite(m_new), m_new, 0.0)
                    alpha = np.exp(np.where(np.isfinite(m), m, -np.inf) - shift)
                    p = np.exp(s - shift[:, None])
                    l = l * alpha + p.sum(axis=1)
                    acc = acc * alpha[:, None] + p @ v[b, j0:j1, kh, :]
                    m = m_new
                with np.errstate(invalid="ignore", divide="ignore"):
                    o[b, i0:i1, h, :] = np.where(l[:, None] > 0, acc / l[:, None], 0.0)
                    lse[b, h, i0:i1] = np.where(l > 0, m + np.log(np.where(l > 0, l, 1.0)), -np.inf)
    return o, lse
