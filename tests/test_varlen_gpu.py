"""GPU parity of the ragged-batch (varlen) forward and its tile plan.

* Equal lengths: the varlen path gives attn_fwd's output bit for bit (same tiles, same arithmetic).
* Ragged batches against oracle.attention_varlen on every element: lengths around the 128-row
  tile and 256-row work-tile edges, empty query or key sequences, more queries than keys (rows
  that see nothing under the bottom-right causal mask) and more keys than queries, GQA, every
  head dim, e4m3.
* Sequences that end in the first half of a work tile, over hundreds of launches: every launch
  finishes and gives the same bits.
* The plan read back: a permutation of all (sequence, head, query block) tiles, costs never
  increasing. A plan built for other arguments, or from bad offsets, is refused on the GPU: the
  forward writes nothing and the status word reports it.
"""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_72_gb300 import binding, inputs
from parity_util import BF16_MAX_ABS, BF16_MAX_LSE, BF16_REL_L2, FP8_MAX_LSE, FP8_REL_L2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)


def run_varlen(w, x, plan=None):
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    if plan is None:
        plan = binding.attn_varlen_plan(cu_q, cu_k, w.H, w.total_q, w.total_k, w.d, w.causal)
    kw = {}
    if x.q.dtype == torch.float8_e4m3fn:
        kw = {n: torch.tensor([s], dtype=torch.float32, device="cuda")
              for n, s in (("descale_q", x.descale_q), ("descale_k", x.descale_k), ("descale_v", x.descale_v))}
    o, lse = binding.attn_fwd_varlen(x.q.cuda(), x.k.cuda(), x.v.cuda(), cu_q, cu_k, plan, w.causal, scale=w.scale,
                                     **kw)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, (st, hex(detail))
    return o, lse, plan


def f64(t, s):
    a = t.float().double().numpy()
    return a * np.float64(np.float32(s)) if t.dtype == torch.float8_e4m3fn else a


def check(w, x, o, lse):
    o_ref, lse_ref = oracle.attention_varlen(f64(x.q, x.descale_q), f64(x.k, x.descale_k), f64(x.v, x.descale_v),
                                             w.cu_q, w.cu_k, w.scale, w.causal)
    og = o.float().cpu().double().numpy()
    lg = lse.cpu().double().numpy()
    assert np.isfinite(og).all()
    # rows that see no key: exactly 0 and -inf
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lg), empty), int((np.isneginf(lg) != empty).sum())
    assert np.all(og[empty.T] == 0.0)
    fin = ~empty
    d = og - o_ref
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(o_ref), 1e-30))
    max_lse = float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    if w.dtype == "bf16":
        assert float(np.abs(d).max()) <= BF16_MAX_ABS and rel <= BF16_REL_L2 and max_lse <= BF16_MAX_LSE, \
            (float(np.abs(d).max()), rel, max_lse)
    else:
        assert rel <= FP8_REL_L2 and max_lse <= FP8_MAX_LSE, (rel, max_lse)


def vw(name, lq, lk=None, H=4, Hkv=2, d=128, causal=True, dtype="bf16", seed=8000):
    return inputs.VarlenWorkload(name, H=H, Hkv=Hkv, d=d, causal=causal, lengths_q=tuple(lq),
                                 lengths_k=None if lk is None else tuple(lk), dtype=dtype, seed=seed)


CASES = [
    vw("edges_causal", [1, 127, 128, 129, 255, 256, 257, 300]),
    vw("edges_noncausal", [1, 127, 128, 129, 255, 256, 257, 300], causal=False),
    vw("empty_seqs", [0, 200, 0, 77], [5, 200, 0, 0]),
    vw("more_keys", [16, 1, 130, 64], [700, 33, 400, 64]),
    vw("more_keys_noncausal", [16, 1, 130, 64], [700, 33, 400, 64], causal=False),
    vw("more_queries", [300, 129, 40], [100, 129, 3]),
    vw("d64_gqa", [333, 64, 517], H=8, Hkv=2, d=64),
    # d = 64 (three rotating S buffers): work tiles whose first Q tile sees no key while the
    # second does (bottom-right mask, more queries than keys), empty sequences, sequences with
    # one Q tile, and many short sequences
    vw("d64_more_queries", [300, 129, 40], [100, 129, 3], d=64, seed=8010),
    vw("d64_empty_and_more_keys", [0, 200, 0, 77, 16, 130], [5, 200, 0, 0, 700, 400], d=64, seed=8011),
    vw("d64_many_short_noncausal", inputs.varlen_lengths(40, 1, 90, 8012), H=2, Hkv=1, d=64, causal=False,
       seed=8012),
    vw("d256", [333, 64, 200], H=2, Hkv=1, d=256),
    vw("d256_more_queries", [260, 5], [130, 300], H=2, Hkv=2, d=256),
    vw("fp8_causal", [250, 600, 90], dtype="fp8_e4m3"),
    vw("fp8_noncausal", [250, 600, 90], [100, 600, 300], causal=False, dtype="fp8_e4m3"),
    vw("fp8_d256_causal", [300, 129, 40], H=2, Hkv=1, d=256, dtype="fp8_e4m3"),
    vw("fp8_d64_causal", [333, 64, 517], H=8, Hkv=2, d=64, dtype="fp8_e4m3", seed=8020),
    vw("fp8_d64_noncausal", [0, 200, 77, 130], [5, 200, 700, 400], d=64, causal=False, dtype="fp8_e4m3",
       seed=8021),
    vw("many_short", inputs.varlen_lengths(40, 1, 90, 8001), H=2, Hkv=1),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_varlen_parity(w):
    x = inputs.make_varlen_inputs(w)
    o, lse, _ = run_varlen(w, x)
    check(w, x, o, lse)


@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_ragged_ends_over_many_launches(dtype):
    # Every sequence ends in the first half of a 256-row work tile, so its last work tile has a
    # second Q tile with no keys while the first one walks up to 17 key tiles. The issuer of that
    # idle tile then only paces itself on the K/V ring, the case that needs the ring's even stage
    # count. Hundreds of launches back to back must all finish (no bounded wait gives up) and
    # give the same bits; the first is checked against the oracle.
    w = vw("ragged_ends_" + dtype, [256 * k + 100 for k in range(1, 9)], H=4, Hkv=2, dtype=dtype, seed=8200)
    x = inputs.make_varlen_inputs(w)
    o, lse, plan = run_varlen(w, x)
    check(w, x, o, lse)
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    kw = {}
    if dtype == "fp8_e4m3":
        kw = {n: torch.tensor([s], dtype=torch.float32, device="cuda")
              for n, s in (("descale_q", x.descale_q), ("descale_k", x.descale_k), ("descale_v", x.descale_v))}
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o2, lse2 = torch.empty_like(o), torch.empty_like(lse)
    for _ in range(400):
        binding.attn_fwd_varlen(q, k, v, cu_q, cu_k, plan, w.causal, scale=w.scale, out=o2, lse=lse2, **kw)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, (st, hex(detail))
    assert torch.equal(o2, o) and torch.equal(lse2, lse)


@pytest.mark.parametrize("d,causal", [(64, True), (128, True), (128, False), (256, True)])
def test_equal_lengths_match_uniform_entry_bit_for_bit(d, causal):
    B, N, H, Hkv = 3, 640, 4, 2
    w = vw("eq", [N] * B, H=H, Hkv=Hkv, d=d, causal=causal, seed=8100 + d)
    x = inputs.make_varlen_inputs(w)
    o_v, lse_v, _ = run_varlen(w, x)
    o_u, lse_u = binding.attn_fwd(x.q.view(B, N, H, d).cuda(), x.k.view(B, N, Hkv, d).cuda(),
                                  x.v.view(B, N, Hkv, d).cuda(), causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o_v.view(B, N, H, d), o_u)
    assert torch.equal(lse_v.view(H, B, N).permute(1, 0, 2), lse_u)


def test_plan_is_a_longest_first_permutation():
    w = vw("plan", [1000, 3, 0, 513, 256, 2000], [1000, 3, 10, 900, 256, 100], H=3, Hkv=1)
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    plan = binding.attn_varlen_plan(cu_q, cu_k, w.H, w.total_q, w.total_k, w.d, True)
    words = plan.view(torch.int32).cpu().numpy()
    n, B, H, R, causal, off, tq, tk = words[:8]
    assert (B, H, R, causal, tq, tk) == (w.B, 3, 256, 1, w.total_q, w.total_k)
    tiles = words[off:off + 2 * n].reshape(n, 2)
    got = sorted((int(b), int(e) >> 16, int(e) & 0xFFFF) for b, e in tiles)
    want = sorted((b, h, m) for b in range(w.B) for h in range(H) for m in range(-(-w.lengths_q[b] // 256)))
    assert got == want
    # cost of a tile: 128-key tiles its longest Q tile visits (bottom-right causal)

    def cost(b, m):
        nq, nk = w.lengths_q[b], w.lk[b]
        best = 0
        for pos0 in (m * 256, m * 256 + 128):
            if pos0 >= nq or nk == 0:
                continue
            last = min(pos0 + 127, nq - 1) + nk - nq
            if last >= 0:
                best = max(best, min(-(-nk // 128), last // 128 + 1))
        return best
    costs = [cost(int(b), int(e) & 0xFFFF) for b, e in tiles]
    assert all(a >= b for a, b in zip(costs, costs[1:]))


def test_mismatched_plan_is_refused():
    w = vw("mismatch", [300, 200])
    x = inputs.make_varlen_inputs(w)
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    plan = binding.attn_varlen_plan(cu_q, cu_k, w.H, w.total_q, w.total_k, w.d, False)   # non-causal plan
    o = torch.full((w.total_q, w.H, w.d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.H, w.total_q), 7.0, dtype=torch.float32, device="cuda")
    binding.attn_fwd_varlen(x.q.cuda(), x.k.cuda(), x.v.cuda(), cu_q, cu_k, plan, True, out=o, lse=lse)
    st, detail = binding.attn_get_status()
    binding.attn_clear_status()
    assert st == binding.ATTN_ERR_INVALID_ARG and detail == 0x2000000C
    assert bool((o == 7.0).all()) and bool((lse == 7.0).all())


def test_bad_offsets_give_an_invalid_plan():
    w = vw("bad", [300, 200])
    x = inputs.make_varlen_inputs(w)
    cu_q = torch.tensor([0, 300, 600], dtype=torch.int32, device="cuda")     # past total_q = 500
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    plan = binding.attn_varlen_plan(cu_q, cu_k, w.H, w.total_q, w.total_k, w.d, True)
    assert int(plan.view(torch.int32)[1]) == -1
    o = torch.full((w.total_q, w.H, w.d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.H, w.total_q), 7.0, dtype=torch.float32, device="cuda")
    binding.attn_fwd_varlen(x.q.cuda(), x.k.cuda(), x.v.cuda(), cu_q, cu_k, plan, True, out=o, lse=lse)
    st, _ = binding.attn_get_status()
    binding.attn_clear_status()
    assert st == binding.ATTN_ERR_INVALID_ARG
    assert bool((o == 7.0).all())


def test_plan_reused_across_calls():
    w = vw("reuse", [500, 17, 260])
    x1 = inputs.make_varlen_inputs(w)
    x2 = inputs.make_varlen_inputs(w.__class__(**{**w.__dict__, "seed": 8201}))
    o1, lse1, plan = run_varlen(w, x1)
    o2, lse2, _ = run_varlen(w, x2, plan=plan)
    check(w, x1, o1, lse1)
    check(w, x2, o2, lse2)


@pytest.mark.parametrize("w", [CASES[2], CASES[6], CASES[10]], ids=lambda w: w.name)
def test_output_alignment_paths_agree(w):
    """An o that is only 16-byte aligned takes 16-byte stores instead of 32-byte ones: same bits
    (empty rows included)."""
    x = inputs.make_varlen_inputs(w)
    o_a, l_a, plan = run_varlen(w, x)
    assert o_a.data_ptr() % 32 == 0
    buf = torch.empty(o_a.numel() + 8, dtype=torch.bfloat16, device="cuda")
    out = buf[8:].view(o_a.shape)
    assert out.data_ptr() % 32 == 16
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    o_b, l_b = binding.attn_fwd_varlen(x.q.cuda(), x.k.cuda(), x.v.cuda(), cu_q, cu_k, plan, w.causal,
                                       scale=w.scale, out=out)
    st, detail = binding.attn_get_status()
    assert st == binding.ATTN_OK, (st, hex(detail))
    assert torch.equal(o_a, o_b) and torch.equal(l_a, l_b)
