"""GPU parity with a negative score scale.

The definition S = scale * Q K^T holds for any finite nonzero scale. With scale < 0 the kernels
compute S = -(Q K^T) (the MMA negates Q through its instruction descriptor) and scale by |scale|,
so the online softmax's running maximum is still taken over the scaled scores. Every entry point
that runs the forward kernel is checked against the fp64 oracle at the same negative scale, on
every element, at the bf16 / fp8 bars the other parity tests use; the backward pass, whose scale
enters only as a factor, is checked the same way.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_72_gb300 import binding, inputs
from parity_util import all_heads, compare_heads, oracle_heads, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)


def small(name, **kw):
    base = dict(B=1, H=2, Hkv=2, N=256, d=64, causal=False, seed=4100)
    base.update(kw)
    return inputs.Workload(name, **base)


CASES = [
    small("neg_d64_noncausal", N=300),
    small("neg_d128_causal_gqa", B=2, H=4, Hkv=2, N=640, d=128, causal=True, seed=4101),
    small("neg_d128_noncausal_outliers", H=4, Hkv=1, N=512, d=128, seed=4102, k_outlier_frac=0.005),
    small("neg_d256_causal", H=2, Hkv=1, N=384, d=256, causal=True, seed=4103),
    small("neg_fp8_causal", H=2, Hkv=1, N=640, d=128, causal=True, dtype="fp8_e4m3", seed=4104),
    # 64 work tiles of 16 key tiles: the last wave is halved across two launches
    small("neg_halved_wave", H=8, Hkv=2, N=2048, d=128, seed=4105),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_negative_scale_matches_oracle(w):
    x = inputs.make_inputs(w)
    scale = -0.7 * w.scale
    o, lse = run_cuda(w, x, scale=scale)
    compare_heads(w, o, lse, oracle_heads(w, x, all_heads(w), scale=scale))


def test_negative_scale_is_not_the_positive_one():
    """The sign reaches the kernel: +scale and -scale give different outputs."""
    w = CASES[1]
    x = inputs.make_inputs(w)
    o_pos, _ = run_cuda(w, x, scale=w.scale)
    o_neg, _ = run_cuda(w, x, scale=-w.scale)
    assert float((o_pos.float() - o_neg.float()).abs().max()) > 0.1


def test_negative_scale_split_kv():
    w = inputs.Workload("neg_split", B=2, H=8, Hkv=2, N=3, d=128, causal=False, seed=4106, Nk=1500, splits=4)
    x = inputs.make_inputs(w)
    scale = -w.scale
    o, lse = binding.attn_fwd_splitkv(x.q.cuda(), x.k.cuda(), x.v.cuda(), w.splits, scale=scale)
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    compare_heads(w, o, lse, oracle_heads(w, x, all_heads(w), scale=scale))


def test_negative_scale_varlen():
    w = inputs.VarlenWorkload("neg_varlen", H=4, Hkv=2, d=128, causal=True, lengths_q=(1, 129, 300, 0, 257),
                              lengths_k=None, dtype="bf16", seed=4107)
    x = inputs.make_varlen_inputs(w)
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    plan = binding.attn_varlen_plan(cu_q, cu_k, w.H, w.total_q, w.total_k, w.d, w.causal)
    scale = -0.5
    o, lse = binding.attn_fwd_varlen(x.q.cuda(), x.k.cuda(), x.v.cuda(), cu_q, cu_k, plan, w.causal, scale=scale)
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    f = lambda t: t.float().double().numpy()
    o_ref, lse_ref = oracle.attention_varlen(f(x.q), f(x.k), f(x.v), w.cu_q, w.cu_k, scale, w.causal)
    og = o.float().cpu().double().numpy()
    lg = lse.cpu().double().numpy()
    assert np.isfinite(og).all()
    assert float(np.abs(og - o_ref).max()) <= 2e-2
    assert float(np.linalg.norm(og - o_ref) / np.linalg.norm(o_ref)) <= 1e-2
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin)
    assert float(np.abs(lg[fin] - lse_ref[fin]).max()) <= 1e-3


@pytest.mark.parametrize("causal", [False, True])
def test_negative_scale_backward(causal):
    B, N, H, Hkv, d = 1, 384, 4, 2, 128
    g = torch.Generator().manual_seed(4108 + int(causal))
    mk = lambda *s: torch.randn(s, generator=g).to(torch.bfloat16)
    q, k, v, do = mk(B, N, H, d), mk(B, N, Hkv, d), mk(B, N, Hkv, d), mk(B, N, H, d)
    scale = -d ** -0.5
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = binding.attn_fwd(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = binding.attn_bwd(qc, kc, vc, o, lse, doc, causal, scale=scale)
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    f = lambda t: t.double().numpy()
    refs = oracle.attention_backward(f(q), f(k), f(v), f(do), scale, causal)[:3]
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        gg = got.float().cpu().double().numpy()
        rel = float(np.linalg.norm(gg - ref) / np.linalg.norm(ref))
        mx = float(np.abs(gg - ref).max() / np.abs(ref).max())
        assert rel <= 1e-2 and mx <= 2e-2, (name, rel, mx)
