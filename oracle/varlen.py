"""Attention forward over a ragged batch (packed sequences with cumulative offsets), fp64 CPU.

TEST INFRASTRUCTURE ONLY. This file is part of the oracle that the CUDA path is
checked against. Only the tests, the package's smoke entry and the benchmark's
CPU baseline leg may import it; the library never does, and it shares no code
with the CUDA kernels.

What it computes. Sequence b owns query rows cu_q[b] .. cu_q[b+1]-1 of the packed
q [total_q, H, d] and key rows cu_k[b] .. cu_k[b+1]-1 of k, v [total_k, Hkv, d].
Each sequence is an independent attention problem (the definition of
oracle.attention, per head, kv head h // (H / Hkv)). Outputs: O [total_q, H, d]
and LSE [H, total_q].

Sources:
  * "flash-attention-3" (ai.thesatyajit.com), "What is actually in the box" and
    "Five schedulers": the forward takes variable-length batches and a varlen
    scheduler exists because serving traffic is ragged.
  * "FlashAttention-3 Deep Dive" (mojostudio.in), FAQ on variable-length
    sequences: ragged batches are described by cumulative sequence length
    offsets (cu_seqlens), with no padding tokens.

Readings where the pages are silent:
  * query and key lengths of a sequence may differ (separate cu_seqlens for q
    and k);
  * causal masking is bottom-right aligned: query i of a sequence with Nq
    queries and Nk keys sees keys j <= i + (Nk - Nq), so the last query sees
    every key. With Nq = Nk this is the usual top-left mask;
  * rows that see no key (Nk = 0, or i + Nk - Nq < 0 when causal) have O = 0
    and LSE = -inf.

Parity pins live in tests/test_oracle_varlen.py.
"""
from __future__ import annotations

import numpy as np

from .attention import attention_head, kv_head


def attention_varlen(q, k, v, cu_q, cu_k, scale: float, causal: bool):
    """O [total_q, H, d] and LSE [H, total_q] of the ragged batch."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_k = np.asarray(cu_k, dtype=np.int64)
    total_q, H, _ = q.shape
    Hkv = k.shape[1]
    o = np.zeros((total_q, H, v.shape[2]), dtype=np.float64)
    lse = np.full((H, total_q), -np.inf, dtype=np.float64)
    for b in range(cu_q.size - 1):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        k0, k1 = int(cu_k[b]), int(cu_k[b + 1])
        if q1 == q0 or k1 == k0:
            continue          # no queries, or no keys: O = 0, LSE = -inf (already set)
        off = (k1 - k0) - (q1 - q0)
        for h in range(H):
            kh = kv_head(h, H, Hkv)
            o_bh, lse_bh = attention_head(q[q0:q1, h, :], k[k0:k1, kh, :], v[k0:k1, kh, :], scale, causal,
                                          causal_offset=off)
            o[q0:q1, h, :] = o_bh
            lse[h, q0:q1] = lse_bh
    return o, lse
