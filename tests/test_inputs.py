"""Checks of the seeded input recipe (shapes, reproducibility, outliers, e4m3 quantisation)."""
import numpy as np
import torch

from exact_attention_72_gb300 import inputs


def test_workload_table_shapes_and_flops():
    w = inputs.WORKLOADS[inputs.HEADLINE]
    assert (w.B, w.H, w.Hkv, w.N, w.d, w.causal) == (2, 32, 8, 8192, 128, True)
    assert abs(w.flops - 1.0995e12) / 1.0995e12 < 1e-4
    assert inputs.WORKLOADS["fp8_noncausal_n8192_d128"].dtype == "fp8_e4m3"
    assert [x.seed for x in inputs.WORKLOADS.values()] == [1000, 1001, 1002, 1003, 1004, 1005]


def test_inputs_are_reproducible_and_bf16():
    w = inputs.WORKLOADS["tiny_bf16_d64"]
    a = inputs.make_inputs(w)
    b = inputs.make_inputs(w)
    assert a.q.dtype == torch.bfloat16 and a.q.shape == (1, 256, 2, 64)
    assert torch.equal(a.q, b.q) and torch.equal(a.k, b.k) and torch.equal(a.v, b.v)
    q64, _, _ = a.as_f64()
    assert q64.dtype == np.float64
    assert np.array_equal(q64, a.q.float().double().numpy())


def test_k_outliers():
    w = inputs.Workload("t", B=1, H=4, Hkv=2, N=100, d=32, causal=True, k_outlier_frac=0.005)
    x = inputs.make_inputs(w)
    n = int(round(0.005 * x.k.numel()))
    assert int((x.k.float().abs() == 8.0).sum()) == n      # N(0,1) never rounds to exactly 8
    assert int((x.k.float() == 8.0).sum()) > 0 and int((x.k.float() == -8.0).sum()) > 0


def test_e4m3_quantisation():
    w = inputs.WORKLOADS["fp8_noncausal_n8192_d128"].replace(N=512)
    x = inputs.make_inputs(w)
    assert x.q.dtype == torch.float8_e4m3fn
    g = torch.Generator().manual_seed(w.seed)
    q32 = torch.randn((w.B, w.N, w.H, w.d), generator=g)
    assert np.float32(x.descale_q) == np.float32(float(q32.abs().max()) / 448.0)
    q8 = x.q.float()
    assert float(q8.abs().max()) == 448.0
    assert torch.isfinite(q8).all()
    # every stored code is an e4m3 value; re-casting is the identity
    assert torch.equal(q8.to(torch.float8_e4m3fn).float(), q8)
    # the dequantised values are close to the fp32 draw (e4m3 has a 3-bit mantissa)
    deq = q8 * x.descale_q
    assert float(((deq - q32).abs() / q32.abs().clamp_min(1e-2)).median()) < 0.07
