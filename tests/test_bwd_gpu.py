"""GPU parity of the backward pass (attn_bwd) against the fp64 backward oracle.

The backward is fed the oracle's own O (rounded to bf16) and LSE, so it is checked alone; a
second test runs the GPU forward then the GPU backward. Expected values come from the oracle
only. Tolerances: the kernel rounds P and dS to bf16 before the tensor-core products (relative
2^-9 per element) and accumulates in fp32; relative L2 error <= 1e-2 per gradient and the
largest elementwise error <= 2e-2 of the gradient's largest entry leave room for that.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_72_gb300 import binding

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_REL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)


def draw(B, N, H, Hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    mk = lambda *s: torch.randn(s, generator=g).to(torch.bfloat16)
    return mk(B, N, H, d), mk(B, N, Hkv, d), mk(B, N, Hkv, d), mk(B, N, H, d)


def compare(name, got, ref):
    g = got.float().cpu().double().numpy()
    assert np.isfinite(g).all(), name
    err = g - ref
    # a floor of 1e-3 per entry for gradients that vanish (N = 1: dS = P (dP - D) = 0 exactly)
    rel = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-3 * np.sqrt(ref.size)))
    mx = float(np.abs(err).max() / max(np.abs(ref).max(), 1e-3))
    assert rel <= REL_L2 and mx <= MAX_REL, (name, rel, mx)
    return rel, mx


CASES = [
    (1, 256, 2, 2, 128, False),
    (1, 256, 2, 2, 128, True),
    (2, 300, 4, 2, 128, True),
    (1, 129, 4, 1, 128, False),
    (2, 640, 2, 1, 64, True),
    (1, 100, 2, 2, 64, False),
    (1, 1, 2, 1, 128, True),
    (1, 513, 8, 2, 64, True),
    # 160 dK/dV and 320 dQ tiles on a 152-SM grid: partial zig-zag turns in both kernels
    (1, 1024, 40, 20, 128, True),
]


@pytest.mark.parametrize("B,N,H,Hkv,d,causal", CASES, ids=lambda v: str(v))
def test_backward_alone(B, N, H, Hkv, d, causal):
    q, k, v, do = draw(B, N, H, Hkv, d, 9000 + N + d + H)
    scale = d ** -0.5
    f = lambda t: t.double().numpy()
    o_ref, lse_ref = oracle.attention_forward(f(q), f(k), f(v), scale, causal)
    dq_ref, dk_ref, dv_ref, _ = oracle.attention_backward(f(q), f(k), f(v), f(do), scale, causal)
    o = torch.tensor(o_ref, dtype=torch.float32).to(torch.bfloat16)
    lse = torch.tensor(lse_ref, dtype=torch.float32)
    dq, dk, dv = binding.attn_bwd(q.cuda(), k.cuda(), v.cuda(), o.cuda(), lse.cuda(), do.cuda(), causal, scale=scale)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, hex(detail)
    compare("dq", dq, dq_ref)
    compare("dk", dk, dk_ref)
    compare("dv", dv, dv_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_forward_then_backward(causal):
    B, N, H, Hkv, d = 2, 384, 4, 2, 128
    q, k, v, do = draw(B, N, H, Hkv, d, 9100 + int(causal))
    scale = d ** -0.5
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = binding.attn_fwd(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = binding.attn_bwd(qc, kc, vc, o, lse, doc, causal, scale=scale)
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    f = lambda t: t.double().numpy()
    dq_ref, dk_ref, dv_ref, _ = oracle.attention_backward(f(q), f(k), f(v), f(do), scale, causal)
    compare("dq", dq, dq_ref)
    compare("dk", dk, dk_ref)
    compare("dv", dv, dv_ref)


def test_backward_is_deterministic():
    B, N, H, Hkv, d = 1, 512, 4, 1, 128
    q, k, v, do = draw(B, N, H, Hkv, d, 9200)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = binding.attn_fwd(qc, kc, vc, causal=True)
    a = binding.attn_bwd(qc, kc, vc, o, lse, doc, True)
    b = binding.attn_bwd(qc, kc, vc, o, lse, doc, True)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


LONG = [
    # 32 key tiles x 4 query heads per kv head: long dQ rings and many zig-zag turns (causal)
    (1, 4096, 8, 2, 128, True),
    # 64 key tiles per query tile, every one visited (non-causal)
    (1, 8192, 2, 1, 128, False),
]


@pytest.mark.parametrize("B,N,H,Hkv,d,causal", LONG, ids=lambda v: str(v))
def test_backward_long_sequences(B, N, H, Hkv, d, causal):
    """Every element of dQ, dK and dV at N >= 4096 against the oracle (every head: a kv head's dK
    and dV sum over all of its query heads)."""
    q, k, v, do = draw(B, N, H, Hkv, d, 9300 + N + int(causal))
    scale = d ** -0.5
    f = lambda t: t.double().numpy()
    o_ref, lse_ref = oracle.attention_forward(f(q), f(k), f(v), scale, causal)
    o = torch.tensor(o_ref, dtype=torch.float32).to(torch.bfloat16)
    lse = torch.tensor(lse_ref, dtype=torch.float32)
    dq, dk, dv = binding.attn_bwd(q.cuda(), k.cuda(), v.cuda(), o.cuda(), lse.cuda(), do.cuda(), causal, scale=scale)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, hex(detail)
    dq_ref, dk_ref, dv_ref, _ = oracle.attention_backward(f(q), f(k), f(v), f(do), scale, causal)
    print("dq", compare("dq", dq, dq_ref), "dk", compare("dk", dk, dk_ref), "dv", compare("dv", dv, dv_ref))
