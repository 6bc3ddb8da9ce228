"""attn_fwd_splitkv_static, the split-KV entry point that allocates nothing.

It exists for callers that cannot call cudaMalloc (a plugin whose framework owns every device
allocation, a server with a committed memory budget, a latency-critical path that must not risk
an allocation's device synchronization); its partial results live in the library's fixed 16 MiB
device scratch. This file is collected last so a run that stops at the first failure has run
every other test before it. It must pass alone in a fresh process and after the other tests.

Each call goes through the C ABI (ctypes) and is checked against attn_fwd_splitkv, the entry point
with a caller workspace, within the bf16 tolerances the other parity tests use. Two calls in a row
use different shapes and split counts, so stale scratch contents from the first call would show
up in the second.
"""
import ctypes
import math

import pytest
import torch

from exact_attention_72_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

MAX_ABS_O = 2e-2     # bf16 bar used by the parity tests
MAX_ABS_LSE = 1e-3


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


def check_against_workspace_entry_point(w):
    x = inputs.make_inputs(w)
    q, k, v = x.q.cuda(), x.k.cuda(), x.v.cuda()
    o_s, lse_s = call_static_through_c_abi(q, k, v, w.splits, w.scale)
    o_w, lse_w = binding.attn_fwd_splitkv(q, k, v, w.splits, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(o_s.float()).all() and torch.isfinite(lse_s).all()
    assert float((o_s.float() - o_w.float()).abs().max()) <= MAX_ABS_O
    assert float((lse_s - lse_w).abs().max()) <= MAX_ABS_LSE


def test_static_scratch_matches_workspace_entry_point_on_two_calls_in_a_row():
    first = inputs.Workload("no_alloc_1", B=2, H=8, Hkv=2, N=4, d=128, causal=False, seed=301, Nk=1500, splits=4)
    second = inputs.Workload("no_alloc_2", B=1, H=16, Hkv=4, N=9, d=128, causal=False, seed=302, Nk=3000, splits=7)
    check_against_workspace_entry_point(first)
    check_against_workspace_entry_point(second)


def test_static_scratch_refuses_oversized_requests():
    # 128 splits x 64 batches x 64 heads x 1 query x (128 + 1) floats is far beyond 16 MiB.
    need = binding.attn_fwd_splitkv_workspace_bytes(64, 64, 1, 128, 128)
    assert need > 16 * 1024 * 1024
    lib = binding.lib()
    q = torch.zeros((64, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((64, 128, 8, 128), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((64, 64, 1), dtype=torch.float32, device="cuda")
    st = lib.attn_fwd_splitkv_static(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kv.data_ptr()),
                                     ctypes.c_void_p(kv.data_ptr()), ctypes.c_void_p(o.data_ptr()),
                                     ctypes.c_void_p(lse.data_ptr()), 64, 64, 8, 1, 128, 128,
                                     ctypes.c_float(1 / math.sqrt(128)), 128, binding.ATTN_DTYPE_BF16, None, None, None,
                                     None)
    assert st == binding.ATTN_ERR_UNSUPPORTED
