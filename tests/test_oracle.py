"""Pins for the fp64 oracle: checks against what the pages and the mathematics fix.

None of these re-types the oracle's formula. They use hand-worked values, closed
forms, invariances, an independent pure-Python brute force, an independently
written online-softmax recurrence and a library routine (torch's SDPA math path
in fp64). ``test_planted_mistakes_are_caught`` plants plausible bugs into copies
of the oracle and checks that at least one pin fails for each.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as oracle_attention

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def rand_qkv(B, N, H, Hkv, d, seed, scale_q=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, N, H, d)) * scale_q
    k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    return q, k, v


# ----------------------------------------------------------------------------------------------
# Pins, written against an ``attn(q, k, v, scale, causal) -> (O [B,N,H,d], LSE [B,H,N])`` callable
# ----------------------------------------------------------------------------------------------

def pin_hand_worked(attn):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        o, lse = attn(np.array(c["q"]), np.array(c["k"]), np.array(c["v"]), c["scale"], c["causal"])
        np.testing.assert_allclose(o, np.array(c["o"]), rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse, np.array(c["lse"]), rtol=0, atol=1e-12, err_msg=c["name"])


def pin_brute_force(attn):
    """Pure-Python loops with math.exp / math.fsum on tiny inputs (no numpy arithmetic), for a
    positive and a negative scale (the definition holds for any finite nonzero scale)."""
    for causal, scale in ((False, 0.7), (True, 0.7), (False, -0.55), (True, -0.55)):
        B, N, H, Hkv, d = 1, 5, 4, 2, 3
        q, k, v = rand_qkv(B, N, H, Hkv, d, seed=7 + causal)
        o, lse = attn(q, k, v, scale, causal)
        for h in range(H):
            kh = h // (H // Hkv)
            for i in range(N):
                keys = [j for j in range(N) if (not causal or j <= i)]
                s = [scale * math.fsum(q[0, i, h, t] * k[0, j, kh, t] for t in range(d)) for j in keys]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = math.fsum(w)
                ref_lse = mx + math.log(tot)
                assert abs(lse[0, h, i] - ref_lse) < 1e-12
                for t in range(d):
                    ref_o = math.fsum(w[a] * v[0, keys[a], kh, t] for a in range(len(keys))) / tot
                    assert abs(o[0, i, h, t] - ref_o) < 1e-12


def pin_constant_v(attn):
    for causal in (False, True):
        q, k, v = rand_qkv(2, 37, 4, 2, 8, seed=11, scale_q=3.0)
        c = np.linspace(-2.5, 4.0, 8)
        v[:] = c
        o, _ = attn(q, k, v, 1.0 / math.sqrt(8), causal)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-13)


def pin_permutation(attn):
    q, k, v = rand_qkv(1, 29, 2, 2, 16, seed=12)
    perm = np.random.default_rng(3).permutation(29)
    o1, l1 = attn(q, k, v, 0.25, False)
    o2, l2 = attn(q, k[:, perm], v[:, perm], 0.25, False)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def pin_closed_forms(attn):
    # Q = 0: uniform weights. O_i = mean of the visible V rows, LSE_i = ln(#visible).
    B, N, H, d = 1, 13, 2, 4
    _, k, v = rand_qkv(B, N, H, H, d, seed=13)
    q = np.zeros((B, N, H, d))
    o, lse = attn(q, k, v, 0.5, False)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-13)
    np.testing.assert_allclose(lse, np.full(lse.shape, math.log(N)), atol=1e-13)
    o, lse = attn(q, k, v, 0.5, True)
    csum = np.cumsum(v, axis=1) / np.arange(1, N + 1)[None, :, None, None]
    np.testing.assert_allclose(o, csum, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, N + 1)), atol=1e-13)
    # Causal row 0 sees only key 0: O_0 = V_0, LSE_0 = scale * q_0 . k_0.
    q, k, v = rand_qkv(1, 9, 3, 3, 5, seed=14)
    o, lse = attn(q, k, v, 0.3, True)
    np.testing.assert_allclose(o[0, 0], v[0, 0], atol=1e-13)
    np.testing.assert_allclose(lse[0, :, 0], 0.3 * np.einsum("hd,hd->h", q[0, 0], k[0, 0]), atol=1e-13)
    # N = 1: O = V, LSE = scale * q . k (both masks).
    q, k, v = rand_qkv(2, 1, 2, 1, 6, seed=15)
    for causal in (False, True):
        o, lse = attn(q, k, v, 0.9, causal)
        np.testing.assert_allclose(o, np.repeat(v, 2, axis=2), atol=1e-13)
        np.testing.assert_allclose(lse, 0.9 * np.einsum("bnhd,bnd->bhn", q, k[:, :, 0, :]), atol=1e-13)


def pin_shift_invariance(attn):
    for causal in (False, True):
        q, k, v = rand_qkv(1, 21, 2, 2, 8, seed=16)
        c = np.random.default_rng(5).standard_normal(8)
        o1, l1 = attn(q, k, v, 0.4, causal)
        o2, l2 = attn(q, k + c, v, 0.4, causal)
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l2 - l1, 0.4 * np.einsum("bnhd,d->bhn", q, c), rtol=0, atol=1e-12)


def pin_gqa_mapping(attn):
    B, N, H, Hkv, d = 2, 11, 4, 2, 3
    q, k, _ = rand_qkv(B, N, H, Hkv, d, seed=17)
    v = np.empty((B, N, Hkv, d))
    for kh in range(Hkv):
        v[:, :, kh, :] = kh + 1.0
    for causal in (False, True):
        o, _ = attn(q, k, v, 0.6, causal)
        for h in range(H):
            np.testing.assert_allclose(o[:, :, h, :], h // (H // Hkv) + 1.0, rtol=0, atol=1e-13)


def pin_torch_sdpa(attn):
    """Library cross-check: torch's SDPA in fp64 on CPU (with GQA expanded by repeat_interleave)."""
    for causal in (False, True):
        B, N, H, Hkv, d = 2, 64, 4, 2, 16
        q, k, v = rand_qkv(B, N, H, Hkv, d, seed=18 + causal, scale_q=2.0)
        scale = 1.0 / math.sqrt(d)
        o, lse = attn(q, k, v, scale, causal)
        tq = torch.from_numpy(q).permute(0, 2, 1, 3)
        tk = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(H // Hkv, dim=1)
        tv = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(H // Hkv, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
        np.testing.assert_allclose(o, ref.permute(0, 2, 1, 3).numpy(), rtol=0, atol=1e-12)
        s = torch.einsum("bhid,bhjd->bhij", tq, tk) * scale
        if causal:
            s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=0, atol=1e-12)


def pin_online_recurrence(attn):
    """The separately written tiled online softmax equals ``attn`` to 1e-12 (N <= 64)."""
    for causal in (False, True):
        for (N, Br, Bc) in [(64, 16, 16), (61, 7, 5), (33, 64, 3), (50, 1, 64), (17, 4, 17)]:
            q, k, v = rand_qkv(1, N, 4, 2, 8, seed=N + Br + Bc, scale_q=2.0)
            o1, l1 = attn(q, k, v, 0.35, causal)
            o2, l2 = oracle.attention_online(q, k, v, 0.35, causal, Br, Bc)
            np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
            np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


ALL_PINS = [pin_hand_worked, pin_brute_force, pin_constant_v, pin_permutation, pin_closed_forms,
            pin_shift_invariance, pin_gqa_mapping, pin_torch_sdpa, pin_online_recurrence]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.attention_forward)


# ----------------------------------------------------------------------------------------------
# Pins on the oracle's pieces
# ----------------------------------------------------------------------------------------------

def test_probability_rows_sum_to_one():
    for causal in (False, True):
        q, k, _ = rand_qkv(2, 48, 4, 2, 8, seed=19, scale_q=4.0)
        p = oracle.probabilities(q, k, 0.5, causal)
        assert np.all(p >= 0)
        np.testing.assert_allclose(p.sum(axis=-1), 1.0, rtol=0, atol=1e-15 * 48)
        if causal:
            assert np.all(np.triu(np.ones((48, 48)), 1)[None, None] * p == 0)


def test_lse_is_brute_force_logsumexp():
    q, k, v = rand_qkv(1, 24, 2, 2, 4, seed=20, scale_q=5.0)
    for causal in (False, True):
        _, lse = oracle.attention_forward(q, k, v, 0.8, causal)
        for h in range(2):
            s = oracle.scores(q[0, :, h], k[0, :, h], 0.8, causal)
            for i in range(24):
                row = [x for x in s[i] if np.isfinite(x)]
                mx = max(row)
                ref = mx + math.log(math.fsum(math.exp(x - mx) for x in row))
                assert abs(lse[0, h, i] - ref) < 1e-12


def test_rows_and_heads_selection_matches_full():
    q, k, v = rand_qkv(2, 40, 4, 2, 8, seed=21)
    for causal in (False, True):
        o, lse = oracle.attention_forward(q, k, v, 0.3, causal)
        rows = np.array([0, 5, 17, 39])
        sub = oracle.attention_forward(q, k, v, 0.3, causal, heads=[(1, 3), (0, 0)], rows=rows)
        for (b, h), (ob, lb) in sub.items():
            np.testing.assert_array_equal(ob, o[b, rows, h])
            np.testing.assert_array_equal(lb, lse[b, h, rows])


def test_row_chunking_does_not_change_results():
    q, k, v = rand_qkv(1, 50, 1, 1, 8, seed=22)
    a = oracle.attention_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], 0.5, True, row_chunk=7)
    b = oracle.attention_head(q[0, :, 0], k[0, :, 0], v[0, :, 0], 0.5, True, row_chunk=1024)
    np.testing.assert_allclose(a[0], b[0], atol=1e-14)
    np.testing.assert_allclose(a[1], b[1], atol=1e-14)


def test_large_scores_do_not_overflow():
    """Scores near 1e3 would overflow a plain exp; the subtracted max keeps O finite and exact."""
    q, k, v = rand_qkv(1, 16, 1, 1, 4, seed=23)
    q *= 300.0
    o, lse = oracle.attention_forward(q, k, v, 1.0, False)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    ref, ref_lse = oracle.attention_online(q, k, v, 1.0, False, 4, 4)
    np.testing.assert_allclose(o, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-15)


def test_hand_worked_through_online_recurrence():
    """The hand-worked fixture also pins the online recurrence directly."""
    for br, bc in [(1, 1), (2, 1), (1, 2)]:
        pin_hand_worked(lambda q, k, v, s, c: oracle.attention_online(q, k, v, s, c, br, bc))


# ----------------------------------------------------------------------------------------------
# Planted mistakes: each plausible bug in a copy of the oracle must fail at least one pin
# ----------------------------------------------------------------------------------------------

def _mutant(kind):
    def attn(q, k, v, scale, causal):
        q = np.asarray(q, float)
        k = np.asarray(k, float)
        v = np.asarray(v, float)
        B, N, H, d = q.shape
        Hkv = k.shape[2]
        o = np.zeros((B, N, H, v.shape[3]))
        lse = np.zeros((B, H, N))
        for b in range(B):
            for h in range(H):
                kh = (h % Hkv) if kind == "gqa_modulo" else h // (H // Hkv)
                sc = 1.0 if kind == "scale_dropped" else scale
                kk = v[b, :, kh] if kind == "k_is_v" else k[b, :, kh]
                s = sc * (q[b, :, h] @ kk.T)
                if kind == "scores_transposed":
                    s = s.T
                if causal:
                    i = np.arange(N)[:, None]
                    j = np.arange(N)[None, :]
                    bad = {"mask_reversed": j < i, "mask_diagonal": j >= i}.get(kind, j > i)
                    s = np.where(bad, -np.inf, s)
                m = s.max(axis=1)
                m = np.where(np.isfinite(m), m, 0)
                e = np.exp(s - m[:, None])
                if kind == "mask_after_softmax" and causal:
                    e = np.exp(sc * (q[b, :, h] @ kk.T) - m[:, None])
                    p = e / e.sum(axis=1, keepdims=True)
                    p = np.where(np.arange(N)[None, :] > np.arange(N)[:, None], 0, p)
                    l = e.sum(axis=1)
                else:
                    l = e.sum(axis=1)
                    p = e / l[:, None]
                if kind == "no_normalise":
                    p = e
                o[b, :, h] = p @ v[b, :, kh]
                if kind == "lse_log2":
                    lse[b, h] = (m + np.log(l)) / math.log(2)
                elif kind == "lse_without_max":
                    lse[b, h] = np.log(l)
                else:
                    lse[b, h] = m + np.log(l)
        return o, lse
    return attn


MUTANTS = ["gqa_modulo", "scale_dropped", "k_is_v", "scores_transposed", "mask_reversed",
           "mask_diagonal", "mask_after_softmax", "no_normalise", "lse_log2", "lse_without_max"]


def test_unmutated_copy_passes_all_pins():
    good = _mutant("none")
    for pin in ALL_PINS:
        pin(good)


@pytest.mark.parametrize("kind", MUTANTS)
def test_planted_mistakes_are_caught(kind):
    bad = _mutant(kind)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(bad)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {kind!r}"


# ----------------------------------------------------------------------------------------------
# Decode shape: fewer queries than keys, every query sees every key (no mask)
# ----------------------------------------------------------------------------------------------

def test_oracle_more_keys_than_queries_brute_force():
    """Nq != Nk (decode / split-KV shape): pure-Python brute force, no numpy arithmetic."""
    rng = np.random.default_rng(31)
    B, Nq, Nk, H, Hkv, d = 2, 3, 11, 4, 2, 5
    q = rng.standard_normal((B, Nq, H, d))
    k = rng.standard_normal((B, Nk, Hkv, d))
    v = rng.standard_normal((B, Nk, Hkv, d))
    o, lse = oracle.attention_forward(q, k, v, 0.45, False)
    assert o.shape == (B, Nq, H, d) and lse.shape == (B, H, Nq)
    for b in range(B):
        for h in range(H):
            kh = h // (H // Hkv)
            for i in range(Nq):
                s = [0.45 * math.fsum(q[b, i, h, t] * k[b, j, kh, t] for t in range(d)) for j in range(Nk)]
                mx = max(s)
                w = [math.exp(x - mx) for x in s]
                tot = math.fsum(w)
                assert abs(lse[b, h, i] - (mx + math.log(tot))) < 1e-12
                for t in range(d):
                    ref = math.fsum(w[j] * v[b, j, kh, t] for j in range(Nk)) / tot
                    assert abs(o[b, i, h, t] - ref) < 1e-12


def test_oracle_key_partition_merge_identity():
    """Splitting the keys into ranges and merging the per-range (O, LSE) by exp(LSE_s - LSE)
    reproduces the full result: LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s. This
    is a property of the definition (the split-KV combine), checked here on the oracle itself."""
    rng = np.random.default_rng(32)
    B, Nq, Nk, H, d = 1, 4, 23, 2, 6
    q = rng.standard_normal((B, Nq, H, d)) * 2
    k = rng.standard_normal((B, Nk, H, d))
    v = rng.standard_normal((B, Nk, H, d))
    o, lse = oracle.attention_forward(q, k, v, 0.5, False)
    cuts = [0, 5, 6, 17, 23]
    parts = [oracle.attention_forward(q, k[:, a:b], v[:, a:b], 0.5, False) for a, b in zip(cuts, cuts[1:])]
    lse_all = np.logaddexp.reduce(np.stack([p[1] for p in parts]), axis=0)
    np.testing.assert_allclose(lse_all, lse, rtol=0, atol=1e-12)
    w = [np.exp(p[1] - lse_all) for p in parts]          # [B, H, Nq]
    o_m = sum(np.transpose(wi, (0, 2, 1))[..., None] * p[0] for wi, p in zip(w, parts))
    np.testing.assert_allclose(o_m, o, rtol=0, atol=1e-12)
