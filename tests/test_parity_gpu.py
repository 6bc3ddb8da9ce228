"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs.

Small shapes are compared on every output element; they span several KV tiles, ragged tails
and all head dims. The full-size workloads are compared on whole sampled heads (every row),
plus a convex-hull property on every element of every head.
"""
import numpy as np
import pytest
import torch

from exact_attention_72_gb300 import binding, inputs
from parity_util import (all_heads, check_convex_hull, compare_heads, oracle_heads, run_cuda, to_device)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import binding, build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)   # a correct launch never waits this long


def small(name, **kw):
    base = dict(B=1, H=2, Hkv=2, N=256, d=64, causal=False, seed=77)
    base.update(kw)
    return inputs.Workload(name, **base)


SMALL = [
    inputs.WORKLOADS["tiny_bf16_d64"],
    small("causal_d128_gqa", B=2, H=4, Hkv=2, N=640, d=128, causal=True),
    small("noncausal_d128", B=1, H=3, Hkv=3, N=512, d=128),
    small("causal_d64", B=1, H=2, Hkv=1, N=768, d=64, causal=True),
    small("noncausal_d256", B=1, H=2, Hkv=2, N=384, d=256),
    small("causal_d256", B=1, H=2, Hkv=1, N=512, d=256, causal=True),
    small("outliers_causal", B=1, H=4, Hkv=1, N=512, d=128, causal=True, k_outlier_frac=0.005),
    small("fp8_noncausal", B=1, H=2, Hkv=2, N=512, d=128, dtype="fp8_e4m3"),
    small("fp8_causal", B=1, H=2, Hkv=1, N=640, d=128, causal=True, dtype="fp8_e4m3"),
    small("fp8_d256_noncausal", B=1, H=2, Hkv=2, N=384, d=256, dtype="fp8_e4m3"),
    small("fp8_d256_causal_gqa", B=2, H=4, Hkv=2, N=640, d=256, causal=True, dtype="fp8_e4m3"),
    # e4m3 at d = 64: 64-byte rows in the 64-byte swizzle
    small("fp8_d64_noncausal", B=1, H=2, Hkv=2, N=512, d=64, dtype="fp8_e4m3"),
    small("fp8_d64_causal_gqa", B=2, H=4, Hkv=2, N=640, d=64, causal=True, dtype="fp8_e4m3"),
    # 160 causal work tiles on a 152-SM grid: a second, partial turn dealt in reverse (zig-zag)
    small("causal_gqa_two_turns", B=1, H=40, Hkv=20, N=1024, d=128, causal=True, seed=78),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_full_parity(w):
    x = inputs.make_inputs(w)
    o, lse = run_cuda(w, x)
    compare_heads(w, o, lse, oracle_heads(w, x, all_heads(w)))


RAGGED_N = [1, 7, 100, 127, 128, 129, 255, 257, 300, 513]


@pytest.mark.parametrize("N", RAGGED_N)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_ragged_lengths(N, causal, d):
    w = small(f"ragged_{N}_{d}_{int(causal)}", B=2, H=2, Hkv=1, N=N, d=d, causal=causal, seed=N * 7 + d)
    x = inputs.make_inputs(w)
    o, lse = run_cuda(w, x)
    compare_heads(w, o, lse, oracle_heads(w, x, all_heads(w)))


@pytest.mark.parametrize("N", [1, 129, 300])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_ragged_lengths_fp8(N, causal, d):
    w = small(f"ragged_fp8_{N}_{d}", B=1, H=2, Hkv=2, N=N, d=d, causal=causal, dtype="fp8_e4m3", seed=N + d)
    x = inputs.make_inputs(w)
    o, lse = run_cuda(w, x)
    compare_heads(w, o, lse, oracle_heads(w, x, all_heads(w)))


def test_many_tiles_persistent_loop():
    """More work tiles than SMs, so each CTA walks several tiles (phase bookkeeping)."""
    w = small("persistent", B=3, H=40, Hkv=10, N=512, d=128, causal=True, seed=5)
    x = inputs.make_inputs(w)
    o, lse = run_cuda(w, x)
    heads = [(0, 0), (1, 17), (2, 39), (2, 3), (0, 38)]
    compare_heads(w, o, lse, oracle_heads(w, x, heads))
    check_convex_hull(w, x, o)


def test_repeatable_bitwise():
    w = SMALL[1]
    x = inputs.make_inputs(w)
    o1, l1 = run_cuda(w, x)
    o2, l2 = run_cuda(w, x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


FULL = list(inputs.WORKLOADS.values()) + list(inputs.EXTRA_FWD_WORKLOADS.values())


def sample_heads(w):
    hs = {(0, 0), (w.B - 1, w.H - 1), (0, w.H // 2), (w.B - 1, min(w.H - 1, w.H // w.Hkv))}
    return sorted(hs)


@pytest.mark.parametrize("w", FULL, ids=lambda w: w.name)
def test_full_size_sampled_heads(w):
    x = inputs.make_inputs(w)
    o, lse = run_cuda(w, x)
    heads = sample_heads(w)
    stats = compare_heads(w, o, lse, oracle_heads(w, x, heads))
    check_convex_hull(w, x, o)
    print(w.name, stats)


def _shifted_out(shape):
    """A bf16 output view that is 16- but not 32-byte aligned."""
    n = int(np.prod(shape))
    buf = torch.empty(n + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(shape)
    assert out.data_ptr() % 32 == 16
    return out


ALIGN_CASES = [SMALL[0], SMALL[1], SMALL[4], SMALL[7], SMALL[9],
               # non-causal, one sparse wave: the halved last wave's merge reads and rewrites o
               small("halved_gqa", B=1, H=8, Hkv=2, N=2048, d=128, seed=79)]


@pytest.mark.parametrize("w", ALIGN_CASES, ids=lambda w: w.name)
def test_output_alignment_paths_agree(w):
    """An o that is only 16-byte aligned takes 16-byte stores instead of 32-byte ones: same bits."""
    from exact_attention_72_gb300 import binding
    from parity_util import to_device
    x = inputs.make_inputs(w)
    q, k, v, desc = to_device(x)
    kw = {} if desc is None else dict(descale_q=desc[0], descale_k=desc[1], descale_v=desc[2])
    o_a, l_a = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, **kw)
    assert o_a.data_ptr() % 32 == 0
    o_b, l_b = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale, out=_shifted_out(o_a.shape), **kw)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, (st, hex(detail))
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)


@pytest.mark.parametrize("d,dtype,causal", [(64, "bf16", True), (128, "bf16", False), (256, "bf16", True),
                                            (64, "fp8_e4m3", False), (128, "fp8_e4m3", True),
                                            (256, "fp8_e4m3", False)])
def test_many_launches_bitwise(d, dtype, causal):
    """200 launches of one seeded call give the same bits every time, with every status OK, on a
    shape with more work tiles than SMs (a second, partial turn) and a ragged last tile: the
    pipelines' barrier phases and buffer rotations do not race, whatever the timing."""
    w = small(f"many_{d}_{dtype}_{int(causal)}", B=2, H=40, Hkv=10, N=700, d=d, causal=causal, dtype=dtype,
              seed=90 + d)
    x = inputs.make_inputs(w)
    o0, l0 = run_cuda(w, x)
    compare_heads(w, o0, l0, oracle_heads(w, x, [(0, 0), (1, 39)]))
    q, k, v, desc = to_device(x)
    kw = {} if desc is None else dict(descale_q=desc[0], descale_k=desc[1], descale_v=desc[2])
    o = torch.empty_like(o0)
    lse = torch.empty_like(l0)
    for _ in range(200):
        binding.attn_fwd(q, k, v, causal=causal, scale=w.scale, out=o, lse=lse, **kw)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, f"device status {st} detail {detail:#x}"
    assert torch.equal(o, o0) and torch.equal(lse, l0)
