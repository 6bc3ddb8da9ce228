"""Pins of the backward oracle (oracle/backward.py): torch autograd of an independent formulation,
central finite differences, and identities of the softmax gradient. Planted mistakes (a dropped
D term, a missing scale, a transposed dS, top-left GQA sums) are shown to fail them."""
import numpy as np
import pytest
import torch

import oracle
from oracle import backward as bw


def rand(B, N, H, Hkv, d, seed):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, N, H, d)), rng.standard_normal((B, N, Hkv, d)),
            rng.standard_normal((B, N, Hkv, d)), rng.standard_normal((B, N, H, d)))


def autograd(q, k, v, do, scale, causal):
    """torch's own softmax and matmul in fp64, differentiated by autograd."""
    B, N, H, d = q.shape
    G = H // k.shape[2]
    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    kk = tk.repeat_interleave(G, dim=2)
    vv = tv.repeat_interleave(G, dim=2)
    s = torch.einsum("bihc,bjhc->bhij", tq, kk) * scale
    if causal:
        mask = torch.ones(N, N, dtype=torch.bool).triu(1)
        s = s.masked_fill(mask, float("-inf"))
    o = torch.einsum("bhij,bjhc->bihc", torch.softmax(s, dim=-1), vv)
    o.backward(torch.tensor(do, dtype=torch.float64))
    return tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,Hkv", [(2, 2), (4, 1)])
def test_matches_autograd(causal, H, Hkv):
    q, k, v, do = rand(2, 37, H, Hkv, 16, 3 + H + int(causal))
    dq, dk, dv, _ = bw.attention_backward(q, k, v, do, 0.3, causal)
    aq, ak, av = autograd(q, k, v, do, 0.3, causal)
    assert np.abs(dq - aq).max() < 1e-12
    assert np.abs(dk - ak).max() < 1e-12
    assert np.abs(dv - av).max() < 1e-12


def test_central_differences():
    q, k, v, do = rand(1, 6, 1, 1, 4, 7)
    scale = 0.7

    def loss(q_, k_, v_):
        o, _ = oracle.attention_head(q_[0, :, 0], k_[0, :, 0], v_[0, :, 0], scale, True)
        return float((o * do[0, :, 0]).sum())

    dq, dk, dv, _ = bw.attention_backward(q, k, v, do, scale, True)
    h = 1e-6
    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        for idx in [(0, 0, 0, 0), (0, 3, 0, 2), (0, 5, 0, 3)]:
            a = arr.copy()
            a[idx] += h
            up = loss(*(a if arr is x else x for x in (q, k, v)))
            a[idx] -= 2 * h
            dn = loss(*(a if arr is x else x for x in (q, k, v)))
            assert abs((up - dn) / (2 * h) - grad[idx]) < 1e-7


def test_softmax_gradient_identities():
    q, k, v, do = rand(2, 50, 4, 2, 8, 11)
    for causal in (False, True):
        dq, dk, dv, dd = bw.attention_backward(q, k, v, do, 0.5, causal)
        # a common shift of every key changes each score row by a constant: no gradient along it
        assert np.abs(dk.sum(axis=1)).max() < 1e-10
        # rows of P sum to one: the dV rows sum to the dO rows of the heads that read them
        G = 2
        want = do.reshape(2, 50, 2, G, 8).sum(axis=3).sum(axis=1)
        assert np.abs(dv.sum(axis=1) - want).max() < 1e-10
        # D = rowsum(dO * O)
        o, _ = oracle.attention_forward(q, k, v, 0.5, causal)
        assert np.abs(dd - np.einsum("bihc,bihc->bhi", do, o)).max() < 1e-12


def test_causal_last_key_sees_only_last_query():
    q, k, v, do = rand(1, 9, 1, 1, 4, 13)
    _, dk, dv, _ = bw.attention_backward(q, k, v, do, 1.0, True)
    p = oracle.probabilities(q, k, 1.0, True)[0, 0]
    # key 8 is visible only to query 8: dV_8 = P_88 dO_8
    assert np.allclose(dv[0, 8, 0], p[8, 8] * do[0, 8, 0], atol=1e-14)


def _mutant(kind):
    def f(q, k, v, do, scale, causal):
        s = oracle.scores(q, k, scale, causal)
        p = oracle.softmax_two_pass(s)[0]
        o = p @ v
        dp = do @ v.T
        d_row = (do * o).sum(1)
        if kind == "no_D":
            ds = p * dp
        elif kind == "transposed_dS":
            ds = (p * (dp - d_row[:, None])).T
        else:
            ds = p * (dp - d_row[:, None])
        dq = (1.0 if kind == "no_scale" else scale) * ds @ k
        dk = scale * ds.T @ q
        return dq, dk, p.T @ do
    return f


@pytest.mark.parametrize("kind", ["no_D", "transposed_dS", "no_scale"])
def test_planted_mistakes_fail_autograd(kind):
    q, k, v, do = rand(1, 12, 1, 1, 8, 17)
    aq, ak, av = autograd(q, k, v, do, 0.4, True)
    mq, mk, mv = _mutant(kind)(q[0, :, 0], k[0, :, 0], v[0, :, 0], do[0, :, 0], 0.4, True)
    bad = max(np.abs(mq - aq[0, :, 0]).max(), np.abs(mk - ak[0, :, 0]).max())
    assert bad > 1e-3
