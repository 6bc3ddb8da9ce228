"""GPU parity of the e4m3 forward with descale factors per (batch, head).

The inputs give each head its own magnitude (factors spread over up to four and a half orders),
quantise each (batch, head) slice of q, k and v with its own amax, and compare the CUDA output
with the fp64 oracle run on exactly the dequantised values. A second check shows why the per-head form
exists: against attention of the unquantised fp32 draw, per-head descales give a smaller error
than one descale per tensor, because quiet heads keep their mantissa bits.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_72_gb300 import binding, inputs
from parity_util import FP8_MAX_LSE, FP8_REL_L2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)


def spread_draw(B, N, H, Hkv, d, seed):
    """fp32 q [B,N,H,d], k/v [B,N,Hkv,d]; head h (and batch b) scaled by its own factor."""
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((B, N, H, d), generator=g)
    k = torch.randn((B, N, Hkv, d), generator=g)
    v = torch.randn((B, N, Hkv, d), generator=g)
    fq = torch.logspace(-2.5, 0.5, B * H).reshape(B, H)
    fk = torch.logspace(0.5, -2.0, B * Hkv).reshape(B, Hkv)
    fv = torch.logspace(-3.5, 1.0, B * Hkv).reshape(B, Hkv)
    return q * fq[:, None, :, None], k * fk[:, None, :, None], v * fv[:, None, :, None]


def deq(x8, desc, b, h):
    """Dequantised (b, h) slice in fp64: the exact values the kernel multiplies."""
    return x8[b, :, h, :].float().double().numpy() * np.float64(desc[b, h].item())


def oracle_all(q8, k8, v8, dq, dk, dv, scale, causal):
    B, N, H, d = q8.shape
    G = H // k8.shape[2]
    o = np.zeros((B, N, H, d))
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, :, h, :], lse[b, h, :] = oracle.attention_head(deq(q8, dq, b, h), deq(k8, dk, b, h // G),
                                                                deq(v8, dv, b, h // G), scale, causal)
    return o, lse


def rel_l2(a, ref):
    return float(np.linalg.norm((a - ref).ravel()) / np.linalg.norm(ref.ravel()))


CASES = [
    dict(B=1, H=4, Hkv=2, N=384, causal=True, seed=4101),
    dict(B=2, H=4, Hkv=4, N=300, causal=False, seed=4102),
    dict(B=2, H=8, Hkv=2, N=640, causal=True, seed=4103),
    dict(B=1, H=8, Hkv=4, N=2048, causal=False, seed=4104),   # every tile's keys halved
]


@pytest.mark.parametrize("c", CASES, ids=lambda c: f"B{c['B']}H{c['H']}Hkv{c['Hkv']}N{c['N']}c{int(c['causal'])}")
def test_per_head_descale_parity(c):
    B, H, Hkv, N, d = c["B"], c["H"], c["Hkv"], c["N"], 128
    q, k, v = spread_draw(B, N, H, Hkv, d, c["seed"])
    q8, dq = inputs.quantize_e4m3_per_head(q)
    k8, dk = inputs.quantize_e4m3_per_head(k)
    v8, dv = inputs.quantize_e4m3_per_head(v)
    scale = 1.0 / np.sqrt(d)
    o, lse = binding.attn_fwd_fp8_scaled(q8.cuda(), k8.cuda(), v8.cuda(), c["causal"], dq.cuda(), dk.cuda(),
                                         dv.cuda(), scale=scale)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, (st, detail)
    o_ref, lse_ref = oracle_all(q8, k8, v8, dq, dk, dv, scale, c["causal"])
    og = o.float().cpu().double().numpy()
    lg = lse.cpu().double().numpy()
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    # per head, so a quiet head's error is not hidden by a loud one
    for b in range(B):
        for h in range(H):
            r = rel_l2(og[b, :, h, :], o_ref[b, :, h, :])
            assert r <= FP8_REL_L2, (b, h, r)
    assert float(np.abs(lg - lse_ref).max()) <= FP8_MAX_LSE


def test_zero_strides_match_per_tensor_entry():
    """Descales broadcast with stride 0 reproduce attn_fwd's per-tensor output bit for bit."""
    w = inputs.Workload("fp8_eq", B=2, H=4, Hkv=2, N=512, d=128, causal=True, dtype="fp8_e4m3", seed=4104)
    x = inputs.make_inputs(w)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    dq, dk, dv = (torch.tensor([s], dtype=torch.float32, device="cuda") for s in (x.descale_q, x.descale_k,
                                                                                   x.descale_v))
    o1, l1 = binding.attn_fwd(q, k, v, causal=True, scale=w.scale, descale_q=dq, descale_k=dk, descale_v=dv)
    o2, l2 = binding.attn_fwd_fp8_scaled(q, k, v, True, dq.view(1, 1), dk.view(1, 1), dv.view(1, 1), scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_batch_only_descale():
    """Strides (1, 0): one descale per batch element, shared by its heads."""
    B, H, Hkv, N, d = 3, 4, 2, 256, 128
    q, k, v = spread_draw(B, N, H, Hkv, d, 4105)
    q = q * torch.tensor([0.05, 1.0, 20.0])[:, None, None, None]
    dq = torch.stack([inputs.quantize_e4m3(q[b])[1] * torch.ones(()) for b in range(B)]).float()
    q8 = torch.stack([inputs.quantize_e4m3(q[b])[0] for b in range(B)])
    k8, dk = inputs.quantize_e4m3_per_head(k)
    v8, dv = inputs.quantize_e4m3_per_head(v)
    scale = 1.0 / np.sqrt(d)
    o, lse = binding.attn_fwd_fp8_scaled(q8.cuda(), k8.cuda(), v8.cuda(), False, dq.cuda().view(B, 1), dk.cuda(),
                                         dv.cuda(), scale=scale)
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    o_ref, lse_ref = oracle_all(q8, k8, v8, dq.view(B, 1).expand(B, H), dk, dv, scale, False)
    assert rel_l2(o.float().cpu().double().numpy(), o_ref) <= FP8_REL_L2
    assert float(np.abs(lse.cpu().double().numpy() - lse_ref).max()) <= FP8_MAX_LSE


def test_per_head_beats_per_tensor_on_spread_heads():
    # with one descale per tensor the quietest v head (factor 10^-3.5) falls into e4m3's
    # subnormal range; its own descale keeps it at full relative precision
    B, H, Hkv, N, d = 1, 8, 4, 512, 128
    q, k, v = spread_draw(B, N, H, Hkv, d, 4106)
    scale = 1.0 / np.sqrt(d)
    # attention of the unquantised draw (fp64 oracle), the target both encodings approximate
    G = H // Hkv
    o_true = np.zeros((B, N, H, d))
    for h in range(H):
        o_true[0, :, h, :] = oracle.attention_head(q[0, :, h, :].double().numpy(), k[0, :, h // G, :].double().numpy(),
                                                   v[0, :, h // G, :].double().numpy(), scale, True)[0]
    q8h, dqh = inputs.quantize_e4m3_per_head(q)
    k8h, dkh = inputs.quantize_e4m3_per_head(k)
    v8h, dvh = inputs.quantize_e4m3_per_head(v)
    oh, _ = binding.attn_fwd_fp8_scaled(q8h.cuda(), k8h.cuda(), v8h.cuda(), True, dqh.cuda(), dkh.cuda(), dvh.cuda(),
                                        scale=scale)
    q8t, sq = inputs.quantize_e4m3(q)
    k8t, sk = inputs.quantize_e4m3(k)
    v8t, sv = inputs.quantize_e4m3(v)
    dev = [torch.tensor([s], dtype=torch.float32, device="cuda") for s in (sq, sk, sv)]
    ot, _ = binding.attn_fwd(q8t.cuda(), k8t.cuda(), v8t.cuda(), causal=True, scale=scale, descale_q=dev[0],
                             descale_k=dev[1], descale_v=dev[2])
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    oh = oh.float().cpu().double().numpy()
    ot = ot.float().cpu().double().numpy()
    err_h = [rel_l2(oh[0, :, h, :], o_true[0, :, h, :]) for h in range(H)]
    err_t = [rel_l2(ot[0, :, h, :], o_true[0, :, h, :]) for h in range(H)]
    # the worst head is much better with per-head scales, and no head is worse by much
    assert max(err_h) < 0.5 * max(err_t), (err_h, err_t)
    assert all(eh <= 1.25 * et + 1e-3 for eh, et in zip(err_h, err_t)), (err_h, err_t)
