"""GPU parity of the non-causal tiles whose keys are cut across two launches.

When the last wave of work tiles would leave SMs idle, attn_fwd cuts some tiles' keys in two: the
first launch covers a tile's first key tiles and writes O and LSE, a dependent launch covers the
rest and merges. One partial wave filling at most half of the SMs is halved; more than one wave is
dealt in equal shares of key tiles, cutting the tiles the share boundaries fall in. Every case
below makes the library cut some tiles (asserted through attn_fwd_tail_units) and compares every
row of the cut heads, and of a head that was not cut, with the fp64 oracle.
"""
import numpy as np
import pytest
import torch

from exact_attention_72_gb300 import binding, inputs
from parity_util import all_heads, check_convex_hull, compare_heads, oracle_heads, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)   # a correct launch never waits this long


def case(name, **kw):
    base = dict(B=1, H=8, Hkv=2, N=2048, d=128, causal=False, seed=91)
    base.update(kw)
    return inputs.Workload(name, **base)


CASES = [
    # one wave of 64 tiles, every tile cut at key tile 8 of 16 (GQA)
    case("one_wave_gqa"),
    # ragged keys: 16 key tiles, the last one 80 keys long, in the second part
    case("ragged_n2000", H=4, Hkv=4, N=2000, seed=92),
    case("d64", H=4, Hkv=1, N=4096, d=64, seed=93),
    # d = 256 (128-row tiles): 17 key tiles, parts of 8 and 9, ragged query and key tails
    case("d256_ragged", H=3, Hkv=3, N=2100, d=256, seed=94),
    case("fp8_per_tensor", H=4, Hkv=2, N=2304, dtype="fp8_e4m3", seed=95),
    case("fp8_d64", H=4, Hkv=2, N=4096, d=64, dtype="fp8_e4m3", seed=97),
    case("outliers", H=4, Hkv=1, N=2048, seed=96, k_outlier_frac=0.005),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_halved_tiles_match_oracle(w):
    assert binding.attn_fwd_halved_tail_tiles(w.B, w.H, w.N, w.d, w.causal) > 0
    x = inputs.make_inputs(w)
    o, lse = run_cuda(w, x)
    compare_heads(w, o, lse, oracle_heads(w, x, all_heads(w)))


def cut_heads(w):
    """(batch, head) pairs holding a cut tile, from the library's list of cut tiles."""
    rpt = 256 if w.d <= 128 else 128
    n_mb = -(-w.N // rpt)
    return sorted({divmod(t // n_mb, w.H) for t, _ in binding.attn_fwd_tail_units(w.B, w.H, w.N, w.d, w.causal)})


SHARE_CASES = [
    # 160 tiles of 16 key tiles on 152 SMs: shares of 16.8 key tiles over all tiles
    case("shares_160", H=20, Hkv=4, N=2048, seed=97),
    # 320 tiles: one whole round, then 168 tiles in shares (GQA)
    case("shares_after_a_round", H=20, Hkv=5, N=4096, seed=101),
    # d = 64: 160 tiles of 64 key tiles
    case("shares_d64", H=5, Hkv=1, N=8192, d=64, seed=102),
    # ragged: 162 tiles of 17 key tiles, the last one 52 keys long, the last query block 52 rows
    case("shares_ragged", H=18, Hkv=6, N=2100, seed=103),
    # shares of about 8 key tiles, every tile 8 key tiles: most tiles cut
    case("shares_short", B=3, H=13, Hkv=13, N=1024, seed=104),
    case("shares_outliers", H=20, Hkv=4, N=2048, seed=105, k_outlier_frac=0.005),
]


@pytest.mark.parametrize("w", SHARE_CASES, ids=lambda w: w.name)
def test_shared_tail_matches_oracle(w):
    units = binding.attn_fwd_tail_units(w.B, w.H, w.N, w.d, w.causal)
    assert len(units) > 0 and any(j != (-(-w.N // 128)) // 2 for _, j in units)
    heads = cut_heads(w)
    x = inputs.make_inputs(w)
    o, lse = run_cuda(w, x)
    whole = [(0, 0)] if (0, 0) not in heads else []
    compare_heads(w, o, lse, oracle_heads(w, x, heads + whole))
    check_convex_hull(w, x, o)


def test_shared_tail_repeatable_bitwise():
    w = SHARE_CASES[1]
    x = inputs.make_inputs(w)
    o1, l1 = run_cuda(w, x)
    o2, l2 = run_cuda(w, x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_halved_repeatable_bitwise():
    w = CASES[0]
    x = inputs.make_inputs(w)
    o1, l1 = run_cuda(w, x)
    o2, l2 = run_cuda(w, x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_halved_matches_whole_tiles_within_rounding():
    """The same heads computed as whole tiles (19 heads: 152 tiles, one full wave, no halving) and
    as halved tiles (the first 8 heads alone: 64 tiles) agree to within the extra bf16 rounding."""
    whole = case("whole", H=19, Hkv=19, N=2048, seed=98)            # 152 tiles: no halving
    assert binding.attn_fwd_halved_tail_tiles(whole.B, whole.H, whole.N, whole.d, False) == 0
    x = inputs.make_inputs(whole)
    o_w, l_w = run_cuda(whole, x)
    # the first 8 heads alone: 64 tiles, all halved
    sub = case("sub", H=8, Hkv=8, N=2048, seed=98)
    assert binding.attn_fwd_halved_tail_tiles(sub.B, sub.H, sub.N, sub.d, False) == 64
    q, k, v = (t[:, :, :8].contiguous().cuda() for t in (x.q, x.k, x.v))
    o_h, l_h = binding.attn_fwd(q, k, v, causal=False, scale=sub.scale)
    assert binding.attn_get_status()[0] == binding.ATTN_OK
    torch.cuda.synchronize()
    a, b = o_w[:, :, :8].float(), o_h.float()
    # a bf16 rounding (relative error <= 2^-8) of O_a, plus the final rounding on each side
    bound = 4 * 2.0 ** -8 * max(float(a.abs().max()), float(b.abs().max()))
    assert float((a - b).abs().max()) <= bound
    assert float((l_w[:, :8] - l_h).abs().max()) <= 1e-4


@pytest.mark.parametrize("name", ["noncausal_bf16_n4096_d256", "fp8_noncausal_n8192_d128"])
def test_halved_rows_error_against_whole_rows(name):
    """The rows of halved tiles carry one more bf16 rounding (of the first part's O). On the full
    d = 256 and e4m3 workloads, their error against the oracle is measured beside that of rows
    computed whole: both within the bar, and the halved rows' worst error within 2x the whole
    rows' (the figures are printed)."""
    w = inputs.WORKLOADS[name]
    units = binding.attn_fwd_tail_units(w.B, w.H, w.N, w.d, w.causal, fp8=w.dtype != "bf16")
    nh = len(units)
    assert nh > 0
    rpt = 256 if w.d <= 128 else 128
    n_mb = -(-w.N // rpt)
    halved = {}
    for t, _ in units:   # non-causal tiles: head-major, query blocks in order
        b, h = divmod(t // n_mb, w.H)
        mb = t % n_mb
        halved.setdefault((b, h), []).extend(range(mb * rpt, min(w.N, (mb + 1) * rpt)))
    whole_heads = [(0, 0), (0, 1)]
    assert not set(whole_heads) & set(halved)
    x = inputs.make_inputs(w)
    o, lse = run_cuda(w, x)
    stats = {}
    for label, heads in (("whole", {hd: None for hd in whole_heads}), ("halved", halved)):
        num = den = mx = 0.0
        for (b, h), rows in heads.items():
            r = None if rows is None else np.asarray(sorted(rows))
            ref = oracle_heads(w, x, [(b, h)], rows=r)
            stats_h = compare_heads(w, o, lse, ref, rows=r)
            o_ref = ref[(b, h)][0]
            og = o[b, :, h, :].float().cpu().double().numpy()
            og = og if r is None else og[r]
            num += float(((og - o_ref) ** 2).sum())
            den += float((o_ref ** 2).sum())
            mx = max(mx, stats_h["max_abs"])
        stats[label] = dict(max_abs=mx, rel_l2=(num / den) ** 0.5)
    print(name, "halved tiles", nh, stats)
    assert stats["halved"]["max_abs"] <= 2.0 * stats["whole"]["max_abs"], stats
