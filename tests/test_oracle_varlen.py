"""Pins of the ragged-batch oracle (oracle/varlen.py): reductions to the batched definition, brute
force of the bottom-right causal mask, the prefix-cache identity, and the empty / fully masked
cases. Each would catch a plausible slip (a wrong offset sign, top-left alignment, rows of one
sequence reading another's keys, a dropped sequence)."""
import itertools

import numpy as np
import pytest

import oracle


def packed(lengths, H, d, seed):
    rng = np.random.default_rng(seed)
    total = int(sum(lengths))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return rng.standard_normal((total, H, d)), cu


def test_equal_lengths_match_batched_definition():
    B, N, H, Hkv, d = 3, 40, 4, 2, 16
    rng = np.random.default_rng(1)
    q = rng.standard_normal((B, N, H, d))
    k = rng.standard_normal((B, N, Hkv, d))
    v = rng.standard_normal((B, N, Hkv, d))
    cu = np.arange(B + 1) * N
    for causal in (False, True):
        o_ref, lse_ref = oracle.attention_forward(q, k, v, 0.3, causal)
        o, lse = oracle.attention_varlen(q.reshape(B * N, H, d), k.reshape(B * N, Hkv, d),
                                         v.reshape(B * N, Hkv, d), cu, cu, 0.3, causal)
        assert np.allclose(o, o_ref.reshape(B * N, H, d), rtol=0, atol=1e-13)
        assert np.allclose(lse, np.transpose(lse_ref, (1, 0, 2)).reshape(H, B * N), rtol=0, atol=1e-13)


def brute(q, k, v, scale, allowed):
    """Softmax over allowed keys, written with explicit loops."""
    Nq, Nk = q.shape[0], k.shape[0]
    o = np.zeros((Nq, v.shape[1]))
    lse = np.full(Nq, -np.inf)
    for i in range(Nq):
        js = [j for j in range(Nk) if allowed(i, j)]
        if not js:
            continue
        s = np.array([scale * float(q[i] @ k[j]) for j in js])
        m = s.max()
        w = np.exp(s - m)
        o[i] = sum(wj * v[j] for wj, j in zip(w, js)) / w.sum()
        lse[i] = m + np.log(w.sum())
    return o, lse


@pytest.mark.parametrize("lq,lk", [([3, 5, 1], [7, 5, 4]), ([6, 2], [2, 9]), ([4, 0, 3], [4, 3, 0])])
def test_bottom_right_causal_brute_force(lq, lk):
    H, d = 2, 8
    q, cu_q = packed(lq, H, d, 2)
    k, cu_k = packed(lk, 1, d, 3)
    v, _ = packed(lk, 1, d, 4)
    o, lse = oracle.attention_varlen(q, k, v, cu_q, cu_k, 0.5, True)
    for b in range(len(lq)):
        Nq, Nk = lq[b], lk[b]
        for h in range(H):
            qs, ks, vs = q[cu_q[b]:cu_q[b + 1], h], k[cu_k[b]:cu_k[b + 1], 0], v[cu_k[b]:cu_k[b + 1], 0]
            ob, lb = brute(qs, ks, vs, 0.5, lambda i, j: j <= i + Nk - Nq)
            assert np.allclose(o[cu_q[b]:cu_q[b + 1], h], ob, atol=1e-12)
            assert np.array_equal(np.isinf(lse[h, cu_q[b]:cu_q[b + 1]]), np.isinf(lb))
            fin = np.isfinite(lb)
            assert np.allclose(lse[h, cu_q[b]:cu_q[b + 1]][fin], lb[fin], atol=1e-12)


def test_prefix_cache_identity():
    """Nq queries after Nk - Nq cached keys: the rows equal the last Nq rows of the causal
    attention of the whole Nk-long sequence."""
    Nk, Nq, H, d = 50, 13, 2, 8
    rng = np.random.default_rng(5)
    q_full = rng.standard_normal((Nk, H, d))
    k = rng.standard_normal((Nk, H, d))
    v = rng.standard_normal((Nk, H, d))
    o_full, lse_full = oracle.attention_varlen(q_full, k, v, [0, Nk], [0, Nk], 0.4, True)
    o, lse = oracle.attention_varlen(q_full[Nk - Nq:], k, v, [0, Nq], [0, Nk], 0.4, True)
    assert np.allclose(o, o_full[Nk - Nq:], atol=1e-13)
    assert np.allclose(lse, lse_full[:, Nk - Nq:], atol=1e-13)


def test_fully_masked_and_empty_rows():
    H, d = 1, 4
    # sequence 0: 5 queries, 2 keys, causal -> rows 0..2 see nothing; sequence 1: no keys
    q, cu_q = packed([5, 3], H, d, 6)
    k, cu_k = packed([2, 0], H, d, 7)
    v, _ = packed([2, 0], H, d, 8)
    o, lse = oracle.attention_varlen(q, k, v, cu_q, cu_k, 1.0, True)
    assert np.all(o[:3] == 0) and np.all(np.isneginf(lse[0, :3]))
    assert np.all(np.isfinite(lse[0, 3:5]))
    assert np.all(o[5:] == 0) and np.all(np.isneginf(lse[0, 5:]))
    # the last query of sequence 0 sees both keys: a plain softmax over them
    s = np.array([q[4, 0] @ k[0, 0], q[4, 0] @ k[1, 0]])
    w = np.exp(s - s.max())
    assert np.allclose(o[4, 0], (w[0] * v[0, 0] + w[1] * v[1, 0]) / w.sum(), atol=1e-13)


def test_sequences_are_independent_under_permutation():
    lq, lk = [4, 7, 2], [6, 7, 3]
    H, Hkv, d = 4, 2, 8
    q, cu_q = packed(lq, H, d, 9)
    k, cu_k = packed(lk, Hkv, d, 10)
    v, _ = packed(lk, Hkv, d, 11)
    o, lse = oracle.attention_varlen(q, k, v, cu_q, cu_k, 0.7, True)
    for perm in itertools.permutations(range(3)):
        qs = np.concatenate([q[cu_q[b]:cu_q[b + 1]] for b in perm])
        ks = np.concatenate([k[cu_k[b]:cu_k[b + 1]] for b in perm])
        vs = np.concatenate([v[cu_k[b]:cu_k[b + 1]] for b in perm])
        pq = np.concatenate([[0], np.cumsum([lq[b] for b in perm])])
        pk = np.concatenate([[0], np.cumsum([lk[b] for b in perm])])
        o2, lse2 = oracle.attention_varlen(qs, ks, vs, pq, pk, 0.7, True)
        for i, b in enumerate(perm):
            assert np.allclose(o2[pq[i]:pq[i + 1]], o[cu_q[b]:cu_q[b + 1]], atol=1e-13)
            assert np.allclose(lse2[:, pq[i]:pq[i + 1]], lse[:, cu_q[b]:cu_q[b + 1]], atol=1e-13)


def test_planted_top_left_alignment_is_caught():
    """A top-left mask (offset 0) for Nq < Nk differs from the pinned bottom-right reading."""
    q, cu_q = packed([3], 1, 4, 12)
    k, cu_k = packed([6], 1, 4, 13)
    v, _ = packed([6], 1, 4, 14)
    o, _ = oracle.attention_varlen(q, k, v, cu_q, cu_k, 1.0, True)
    o_tl, _ = oracle.attention_head(q[:, 0], k[:, 0], v[:, 0], 1.0, True)     # top-left
    assert not np.allclose(o[:, 0], o_tl)
