"""attn_fwd_splitkv_static, the split-KV entry point that allocates nothing.

It exists for callers that cannot call cudaMalloc (a plugin whose framework owns every device
allocation, a server with a committed memory budget, a latency-critical path that must not risk
an allocation's device synchronization); its partial results live in the library's fixed 16 MiB
device scratch. This file is collected last so a run that stops at the first failure has run
every other test before it. It must pass alone in a fresh process and after the other tests.

Each call goes through the C ABI (ctypes). Its output must equal, bit for bit, that of
attn_fwd_splitkv, the entry point with a caller workspace: both run the same split and combine
kernels with the same split count, so any difference (a partial overwrite of the scratch, stale
contents read back) shows. Each call is also compared with the fp64 oracle at the bf16 bars the
other parity tests use. Two calls in a row use different shapes and split counts, so stale
scratch contents from the first call would show up in the second.
"""
import ctypes
import math

import pytest
import torch

from exact_attention_72_gb300 import binding, inputs
from parity_util import all_heads, compare_heads, oracle_heads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)


def call_static_through_c_abi(q, k, v, num_splits, scale):
    lib = binding.lib()
    B, Nq, H, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    o = torch.full((B, Nq, H, d), float("nan"), dtype=torch.bfloat16, device=q.device)
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device=q.device)
    fn = lib.attn_fwd_splitkv_static
    st = fn(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
            ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()), B, H, Hkv, Nq, Nk, d, ctypes.c_float(scale),
            num_splits, binding.ATTN_DTYPE_BF16, None, None, None,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == binding.ATTN_OK, binding.attn_status_string(st)
    torch.cuda.synchronize()
    return o, lse


def check_against_workspace_entry_point(w, splits_static=None, oracle_heads_list=None):
    x = inputs.make_inputs(w)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o_s, lse_s = call_static_through_c_abi(q, k, v, w.splits if splits_static is None else splits_static, w.scale)
    o_w, lse_w = binding.attn_fwd_splitkv(q, k, v, w.splits, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(o_s.float()).all() and torch.isfinite(lse_s).all()
    assert torch.equal(o_s, o_w) and torch.equal(lse_s, lse_w)
    heads = all_heads(w) if oracle_heads_list is None else oracle_heads_list
    compare_heads(w, o_s, lse_s, oracle_heads(w, x, heads))


def test_static_scratch_matches_workspace_entry_point_on_two_calls_in_a_row():
    first = inputs.Workload("no_alloc_1", B=2, H=8, Hkv=2, N=4, d=128, causal=False, seed=301, Nk=1500, splits=4)
    second = inputs.Workload("no_alloc_2", B=1, H=16, Hkv=4, N=9, d=128, causal=False, seed=302, Nk=3000, splits=7)
    check_against_workspace_entry_point(first)
    check_against_workspace_entry_point(second)


def test_static_scratch_counts_only_the_splits_that_run():
    """128 requested splits over 200 keys run as 2 (one per 128-key tile). Their partial results
    (64 x 64 query rows x 2 splits) fit the scratch, although 128 splits' worth would not."""
    w = inputs.Workload("no_alloc_clamp", B=64, H=64, Hkv=8, N=1, d=128, causal=False, seed=303, Nk=200, splits=2)
    assert binding.attn_fwd_splitkv_workspace_bytes(64, 64, 1, 128, 128) > 16 * 1024 * 1024
    assert binding.attn_fwd_splitkv_workspace_bytes(64, 64, 1, 128, 2) <= 16 * 1024 * 1024
    check_against_workspace_entry_point(w, splits_static=128, oracle_heads_list=[(0, 0), (17, 33), (63, 63)])


def test_static_scratch_refuses_oversized_requests():
    # 2 splits (256 keys: both run) x 128 heads x 128 queries x (128 + 1) floats is just over 16 MiB.
    need = binding.attn_fwd_splitkv_workspace_bytes(1, 128, 128, 128, 2)
    assert need > 16 * 1024 * 1024
    lib = binding.lib()
    q = torch.zeros((1, 128, 128, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 256, 8, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 128, 128), dtype=torch.float32, device="cuda")
    st = lib.attn_fwd_splitkv_static(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kv.data_ptr()),
                                     ctypes.c_void_p(kv.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                                     ctypes.c_void_p(lse.data_ptr()), 1, 128, 8, 128, 256, 128,
                                     ctypes.c_float(1 / math.sqrt(128)), 2, binding.ATTN_DTYPE_BF16, None, None, None,
                                     None)
    assert st == binding.ATTN_ERR_UNSUPPORTED
