"""GPU parity of the e4m3 block quantiser and the block-scaled e4m3 forward.

* attn_quantize_e4m3 against oracle.fp8_quant: codes and descales bit for bit without a rotation;
  with the Hadamard rotation (fp32 butterflies on the GPU, exact sums in the oracle) descales
  within 1e-6 and codes equal except at near-ties of the rounding, where either neighbour is right.
* attn_fwd_fp8_blockscaled on codes and descales made by the oracle, against the fp64 oracle
  attention of the same dequantised values.
* The whole chain (GPU quantiser + block-scaled forward) against attention of the bf16 inputs,
  and its error against the per-tensor e4m3 path on inputs with outliers.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_quant as fq
from exact_attention_72_gb300 import binding, inputs
from parity_util import FP8_MAX_LSE, FP8_REL_L2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)


def bf16_draw(shape, seed, outlier_frac=0.0, outlier_mag=10.0):
    """N(0, 1) entries; a fraction of them multiplied by outlier_mag; rounded to bf16."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g)
    if outlier_frac:
        m = torch.rand(shape, generator=g) < outlier_frac
        x[m] *= outlier_mag
    return x.to(torch.bfloat16)


def gpu_quantize(x, block_rows, signs=None):
    x8, ds = binding.quantize_e4m3(x.cuda(), block_rows, None if signs is None else signs.cuda())
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    return x8.cpu().float().double().numpy(), ds.cpu().numpy()


QCASES = [
    # (B, N, Hx, d, block_rows)
    (2, 300, 3, 128, 128),
    (2, 300, 3, 128, 64),
    (1, 257, 2, 64, 128),
    (1, 200, 2, 256, 64),
    (1, 77, 1, 128, 1),          # one row per block
    (2, 300, 2, 128, 200),       # blocks longer than one CTA's 128 rows
    (1, 1000, 2, 128, 1000),     # one block per (batch, head)
    (1, 515, 2, 256, 515),
    (1, 130, 2, 128, 8),         # sixteen blocks per 128-row chunk
    (1, 640, 1, 128, 32),
    (1, 100, 1, 128, 100),       # a block size that does not divide 128
    (1, 35, 2, 64, 5),
]


@pytest.mark.parametrize("B,N,Hx,d,R", QCASES, ids=lambda v: str(v))
def test_quantizer_bit_exact(B, N, Hx, d, R):
    x = bf16_draw((B, N, Hx, d), 5000 + N + d + R, outlier_frac=0.002)
    codes, ds = gpu_quantize(x, R)
    c_ref, d_ref = fq.quantize_blocks(x.double().numpy(), R)
    assert ds.shape == d_ref.shape
    assert np.array_equal(ds, d_ref)
    assert np.array_equal(codes, c_ref)


def test_quantizer_zero_block():
    x = torch.zeros((1, 130, 2, 128), dtype=torch.bfloat16)
    x[0, 64:, 1] = 1.5
    codes, ds = gpu_quantize(x, 64)
    c_ref, d_ref = fq.quantize_blocks(x.double().numpy(), 64)
    assert np.array_equal(ds, d_ref) and ds[0, 0, 0] == 1.0 and np.array_equal(codes, c_ref)


def near_tie(y, rel=1e-5):
    """True where y is within rel of a rounding boundary between two e4m3 values."""
    lo = fq.e4m3_round(y * (1 - rel))
    hi = fq.e4m3_round(y * (1 + rel))
    return lo != hi


@pytest.mark.parametrize("B,N,Hx,d,R", [(2, 300, 3, 128, 128), (1, 200, 2, 128, 64), (1, 256, 2, 64, 64),
                                        (1, 130, 2, 256, 128), (1, 600, 1, 128, 600), (1, 300, 2, 128, 16),
                                        (1, 300, 1, 256, 300)], ids=lambda v: str(v))
def test_quantizer_rotated(B, N, Hx, d, R):
    x = bf16_draw((B, N, Hx, d), 6000 + N + d, outlier_frac=0.002)
    s = inputs.hadamard_signs(d, 77 + d)
    codes, ds = gpu_quantize(x, R, s)
    c_ref, d_ref = fq.quantize_blocks(x.double().numpy(), R, s.double().numpy())
    assert np.allclose(ds, d_ref, rtol=1e-6, atol=0)
    # the oracle's fp32 quotient u / descale_u, from its exact rotation
    u = (x.double().numpy() * s.double().numpy()) @ fq.sylvester_hadamard(d)
    rows = np.arange(N) // R
    ds_u = np.transpose(d_ref.astype(np.float64)[:, :, rows], (0, 2, 1))[:, :, :, None] * np.sqrt(d)
    y = u / ds_u
    diff = codes != c_ref
    assert not np.any(diff & ~near_tie(y)), int((diff & ~near_tie(y)).sum())
    # where they differ, the GPU code is the other neighbour of the tie
    assert np.all(np.abs(codes[diff] - c_ref[diff]) <= np.abs(c_ref[diff]) * 2.0 ** -3 + 2.0 ** -9)
    assert diff.mean() < 1e-3


def to_e4m3(codes):
    return torch.tensor(codes, dtype=torch.float32).to(torch.float8_e4m3fn)


def oracle_blockscaled(qd, kd, vd, scale, causal):
    """fp64 attention of dequantised q [B,N,H,d], k/v [B,N,Hkv,d]: (O [B,N,H,d], LSE [B,H,N])."""
    B, N, H, d = qd.shape
    G = H // kd.shape[2]
    o = np.zeros(qd.shape)
    lse = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            o[b, :, h], lse[b, h] = oracle.attention_head(qd[b, :, h], kd[b, :, h // G], vd[b, :, h // G], scale,
                                                          causal)
    return o, lse


def rel_l2(a, ref):
    return float(np.linalg.norm((a - ref).ravel()) / np.linalg.norm(ref.ravel()))


BCASES = [
    dict(B=1, H=4, Hkv=2, N=384, causal=True, rot=False, seed=7001),
    dict(B=2, H=2, Hkv=2, N=300, causal=False, rot=False, seed=7002),
    dict(B=1, H=4, Hkv=1, N=640, causal=True, rot=True, seed=7003),
    dict(B=1, H=2, Hkv=2, N=200, causal=False, rot=True, seed=7004),
    # 17 key tiles, 36 work tiles: the last wave's keys are halved across two launches
    dict(B=1, H=4, Hkv=2, N=2100, causal=False, rot=False, seed=7005),
    # head dim 256 (one Q tile per work tile)
    dict(B=1, H=2, Hkv=1, N=300, causal=True, rot=True, seed=7006, d=256),
    # head dim 64 (64-byte rows)
    dict(B=1, H=4, Hkv=2, N=640, causal=True, rot=True, seed=7007, d=64),
    dict(B=1, H=4, Hkv=2, N=2100, causal=False, rot=False, seed=7008, d=64),
]


@pytest.mark.parametrize("c", BCASES, ids=lambda c: f"B{c['B']}H{c['H']}N{c['N']}c{int(c['causal'])}r{int(c['rot'])}")
def test_blockscaled_forward_parity(c):
    B, H, Hkv, N, d = c["B"], c["H"], c["Hkv"], c["N"], c.get("d", 128)
    q = bf16_draw((B, N, H, d), c["seed"], 0.002).double().numpy()
    k = bf16_draw((B, N, Hkv, d), c["seed"] + 1, 0.002).double().numpy()
    v = bf16_draw((B, N, Hkv, d), c["seed"] + 2, 0.002).double().numpy()
    s = inputs.hadamard_signs(d, c["seed"]).double().numpy() if c["rot"] else None
    cq, dq = fq.quantize_blocks(q, 128, s)
    ck, dk = fq.quantize_blocks(k, 64, s)
    cv, dv = fq.quantize_blocks(v, N)
    scale = d ** -0.5
    o, lse = binding.attn_fwd_fp8_blockscaled(to_e4m3(cq).cuda(), to_e4m3(ck).cuda(), to_e4m3(cv).cuda(),
                                              c["causal"], torch.tensor(dq).cuda(), torch.tensor(dk).cuda(),
                                              torch.tensor(dv[:, :, 0]).contiguous().cuda(), scale=scale)
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    o_ref, lse_ref = oracle_blockscaled(fq.dequantize_blocks(cq, dq, 128), fq.dequantize_blocks(ck, dk, 64),
                                        fq.dequantize_blocks(cv, dv, N), scale, c["causal"])
    og, lg = o.float().cpu().double().numpy(), lse.cpu().double().numpy()
    assert np.isfinite(og).all() and np.isfinite(lg).all()
    for b in range(B):
        for h in range(H):
            assert rel_l2(og[b, :, h], o_ref[b, :, h]) <= FP8_REL_L2, (b, h)
    assert float(np.abs(lg - lse_ref).max()) <= FP8_MAX_LSE


def test_k_block_scale_reaches_each_half_tile():
    """k blocks of very different magnitude inside one 128-key tile: each 64-key half must use its
    own descale (a kernel that applied one scale per tile would be off by the ratio)."""
    B, H, Hkv, N, d = 1, 2, 1, 256, 128
    q = bf16_draw((B, N, H, d), 7100).double().numpy()
    k = bf16_draw((B, N, Hkv, d), 7101).double().numpy()
    k[:, 64:128] *= 40.0
    k[:, 192:] *= 0.02
    v = bf16_draw((B, N, Hkv, d), 7102).double().numpy()
    cq, dq = fq.quantize_blocks(q, 128)
    ck, dk = fq.quantize_blocks(k, 64)
    cv, dv = fq.quantize_blocks(v, N)
    scale = 0.02
    o, lse = binding.attn_fwd_fp8_blockscaled(to_e4m3(cq).cuda(), to_e4m3(ck).cuda(), to_e4m3(cv).cuda(), False,
                                              torch.tensor(dq).cuda(), torch.tensor(dk).cuda(),
                                              torch.tensor(dv[:, :, 0]).contiguous().cuda(), scale=scale)
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    o_ref, lse_ref = oracle_blockscaled(fq.dequantize_blocks(cq, dq, 128), fq.dequantize_blocks(ck, dk, 64),
                                        fq.dequantize_blocks(cv, dv, N), scale, False)
    assert rel_l2(o.float().cpu().double().numpy(), o_ref) <= FP8_REL_L2
    assert float(np.abs(lse.cpu().double().numpy() - lse_ref).max()) <= FP8_MAX_LSE


def test_uniform_block_descales_match_per_tensor_entry():
    """Block descales that all hold the same value give attn_fwd's per-tensor output bit for bit."""
    w = inputs.Workload("fp8_eq", B=1, H=4, Hkv=2, N=384, d=128, causal=True, dtype="fp8_e4m3", seed=7200)
    x = inputs.make_inputs(w)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    one = lambda s: torch.tensor([s], dtype=torch.float32, device="cuda")
    o1, l1 = binding.attn_fwd(q, k, v, causal=True, scale=w.scale, descale_q=one(x.descale_q),
                              descale_k=one(x.descale_k), descale_v=one(x.descale_v))
    dq = torch.full((1, 4, 3), x.descale_q, dtype=torch.float32, device="cuda")
    dk = torch.full((1, 2, 6), x.descale_k, dtype=torch.float32, device="cuda")
    dv = torch.full((1, 2), x.descale_v, dtype=torch.float32, device="cuda")
    o2, l2 = binding.attn_fwd_fp8_blockscaled(q, k, v, True, dq, dk, dv, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def chain(qb, kb, vb, causal, signs):
    """GPU quantiser (q blocks of 128, k blocks of 64, v per head) then the block-scaled forward."""
    N = qb.shape[1]
    sg = None if signs is None else signs.cuda()
    q8, dq = binding.quantize_e4m3(qb.cuda(), 128, sg)
    k8, dk = binding.quantize_e4m3(kb.cuda(), 64, sg)
    v8, dv = binding.quantize_e4m3(vb.cuda(), N)
    o, _ = binding.attn_fwd_fp8_blockscaled(q8, k8, v8, causal, dq, dk, dv.view(dv.shape[0], dv.shape[1]))
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    return o.float().cpu().double().numpy()


def test_chain_error_against_bf16_attention_and_per_tensor():
    B, N, H, d = 1, 1024, 2, 128
    qb = bf16_draw((B, N, H, d), 7300, 0.001, 10.0)
    kb = bf16_draw((B, N, H, d), 7301, 0.001, 10.0)
    vb = bf16_draw((B, N, H, d), 7302, 0.001, 10.0)
    o_true, _ = oracle_blockscaled(qb.double().numpy(), kb.double().numpy(), vb.double().numpy(), d ** -0.5, True)
    err = lambda o: float(np.sqrt(np.mean((o - o_true) ** 2)))
    e_rot = err(chain(qb, kb, vb, True, inputs.hadamard_signs(d, 7303)))
    e_blk = err(chain(qb, kb, vb, True, None))
    q8, sq = inputs.quantize_e4m3(qb)
    k8, sk = inputs.quantize_e4m3(kb)
    v8, sv = inputs.quantize_e4m3(vb)
    one = lambda s: torch.tensor([s], dtype=torch.float32, device="cuda")
    ot, _ = binding.attn_fwd(q8.cuda(), k8.cuda(), v8.cuda(), causal=True, descale_q=one(sq), descale_k=one(sk),
                             descale_v=one(sv))
    e_tensor = err(ot.float().cpu().double().numpy())
    assert rel_l2(chain(qb, kb, vb, True, inputs.hadamard_signs(d, 7303)), o_true) <= FP8_REL_L2
    assert e_rot < e_blk < e_tensor, (e_rot, e_blk, e_tensor)
    assert e_tensor / e_rot > 1.2, (e_rot, e_blk, e_tensor)
