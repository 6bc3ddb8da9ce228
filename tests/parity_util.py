"""Helpers shared by the GPU parity tests: run the CUDA path, run the oracle, compare.

Tolerances (from the stated acceptance bar for this path):
  bf16: max|dO| <= 2e-2, ||dO||_2 / ||O||_2 <= 1e-2, max|dLSE| <= 1e-3
  fp8 : ||dO||_2 / ||O||_2 <= 6e-2 (LSE error reported, bounded loosely)
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_attention_72_gb300 import binding, inputs

BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 1e-2
BF16_MAX_LSE = 1e-3
FP8_REL_L2 = 6e-2
FP8_MAX_LSE = 5e-2   # not part of the stated bar; catches gross LSE errors on the fp8 path


def to_device(x: inputs.AttnInputs, device="cuda"):
    q, k, v = x.q.to(device), x.k.to(device), x.v.to(device)
    desc = None
    if x.q.dtype == torch.float8_e4m3fn:
        desc = [torch.tensor([s], dtype=torch.float32, device=device) for s in (x.descale_q, x.descale_k, x.descale_v)]
    return q, k, v, desc


def run_cuda(w: inputs.Workload, x: inputs.AttnInputs, scale=None):
    q, k, v, desc = to_device(x)
    kw = {}
    if desc is not None:
        kw = dict(descale_q=desc[0], descale_k=desc[1], descale_v=desc[2])
    o, lse = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale if scale is None else scale, **kw)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, f"device status {st} detail {detail:#x}"
    return o, lse


def head_f64(t: torch.Tensor, b: int, h: int, descale: float) -> np.ndarray:
    a = t[b, :, h, :].to(torch.float32).to(torch.float64).numpy()
    if t.dtype == torch.float8_e4m3fn:
        a = a * np.float64(np.float32(descale))
    return a


def oracle_heads(w: inputs.Workload, x: inputs.AttnInputs, heads, rows=None, scale=None):
    """Oracle O/LSE for the listed (b, h) heads; returns {(b, h): (O [rows, d], LSE [rows])}.

    ``scale`` defaults to the workload's 1/sqrt(d)."""
    out = {}
    g = w.H // w.Hkv
    sc = w.scale if scale is None else scale
    for (b, h) in heads:
        kh = h // g
        out[(b, h)] = oracle.attention_head(head_f64(x.q, b, h, x.descale_q), head_f64(x.k, b, kh, x.descale_k),
                                            head_f64(x.v, b, kh, x.descale_v), sc, w.causal, rows=rows)
    return out


def compare_heads(w: inputs.Workload, o_gpu: torch.Tensor, lse_gpu: torch.Tensor, ref: dict, rows=None):
    """Checks the tolerance bar over the listed heads (all of them together for the L2 norm)."""
    o_cpu = o_gpu.float().cpu()
    lse_cpu = lse_gpu.cpu()
    num = den = 0.0
    max_abs = max_lse = 0.0
    for (b, h), (o_ref, lse_ref) in ref.items():
        og = o_cpu[b, :, h, :].double().numpy()
        lg = lse_cpu[b, h, :].double().numpy()
        if rows is not None:
            og, lg = og[rows], lg[rows]
        assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg)), f"non-finite output at head {(b, h)}"
        d = og - o_ref
        num += float((d * d).sum())
        den += float((o_ref * o_ref).sum())
        max_abs = max(max_abs, float(np.abs(d).max()))
        max_lse = max(max_lse, float(np.abs(lg - lse_ref).max()))
    rel = (num / den) ** 0.5 if den > 0 else num ** 0.5
    stats = dict(rel_l2=rel, max_abs=max_abs, max_lse=max_lse)
    if w.dtype == "fp8_e4m3":
        assert rel <= FP8_REL_L2, stats
        assert max_lse <= FP8_MAX_LSE, stats
    else:
        assert max_abs <= BF16_MAX_ABS, stats
        assert rel <= BF16_REL_L2, stats
        assert max_lse <= BF16_MAX_LSE, stats
    return stats


def all_heads(w: inputs.Workload):
    return [(b, h) for b in range(w.B) for h in range(w.H)]


def check_convex_hull(w: inputs.Workload, x: inputs.AttnInputs, o_gpu: torch.Tensor):
    """Property at any size: each O row is a convex combination of V rows of its kv head, so per
    (b, h, column) it lies within [min V, max V] (plus bf16 output rounding)."""
    o = o_gpu.float()
    v = x.v.to(o.device).float()
    if x.v.dtype == torch.float8_e4m3fn:
        v = v * x.descale_v
    g = w.H // w.Hkv
    vmin = v.amin(dim=1).repeat_interleave(g, dim=1)   # [B, H, d]
    vmax = v.amax(dim=1).repeat_interleave(g, dim=1)
    slack = 1e-2 * torch.maximum(vmax.abs(), vmin.abs()) + 1e-3
    assert torch.isfinite(o).all()
    assert (o >= (vmin - slack)[:, None]).all() and (o <= (vmax + slack)[:, None]).all()
