"""Failure handling on the GPU without a GPU fault: a K/V copy is skipped on purpose so a
bounded wait runs out; the kernel must unwind, report ATTN_ERR_TIMEOUT through the status word,
and leave the context usable for a correct follow-up call. Also checks the host-buffer entry
point against the device one."""
import pytest
import torch

from exact_attention_72_gb300 import binding, inputs
from parity_util import all_heads, compare_heads, oracle_heads, run_cuda, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    from exact_attention_72_gb300 import binding, build
    build.build()
    binding.attn_debug_set(timeout_ns=1_000_000_000)   # a correct launch never waits this long


# The fourth case has its keys halved across two launches; CTA 0 of each skips a copy. The e4m3
# cases cover the 8-bit instances, at d = 64 with the 64-byte swizzle.
@pytest.mark.parametrize("d,causal,N,dtype", [(128, True, 512, "bf16"), (256, False, 512, "bf16"),
                                              (64, False, 512, "bf16"), (128, False, 2048, "bf16"),
                                              (128, True, 512, "fp8_e4m3"), (128, False, 2048, "fp8_e4m3"),
                                              (64, True, 512, "fp8_e4m3")])
def test_skipped_copy_times_out_and_context_survives(d, causal, N, dtype):
    w = inputs.Workload("fault", B=1, H=4, Hkv=2, N=N, d=d, causal=causal, seed=3, dtype=dtype)
    x = inputs.make_inputs(w)
    q, k, v, desc = to_device(x)
    kw = {} if desc is None else dict(descale_q=desc[0], descale_k=desc[1], descale_v=desc[2])
    binding.attn_clear_status()
    binding.attn_debug_set(timeout_ns=50_000_000, skip_load=True)
    try:
        binding.attn_fwd(q, k, v, causal=causal, **kw)
        st, detail = binding.attn_get_status()
    finally:
        binding.attn_debug_set(1_000_000_000, False)
    assert st == binding.ATTN_ERR_TIMEOUT
    assert detail & 0x40000000
    binding.attn_clear_status()
    o, lse = run_cuda(w, x)           # asserts the status is OK again
    compare_heads(w, o, lse, oracle_heads(w, x, all_heads(w)))


HOST_SHAPES = [
    dict(B=1, H=4, Hkv=2, N=384, d=128, causal=True),      # one batch, two KV-head chunks
    dict(B=2, H=8, Hkv=4, N=300, d=128, causal=False),     # two batches x two KV-head chunks, ragged N
    dict(B=5, H=2, Hkv=1, N=256, d=64, causal=True),       # uneven batch chunks
    dict(B=1, H=6, Hkv=3, N=200, d=256, causal=False),     # three KV-head chunks
    # keys of every tile halved across two launches, in the device call and in each of the four
    # chunks (two launches per chunk on the host path's two compute streams)
    dict(B=1, H=8, Hkv=4, N=2048, d=128, causal=False),
]


@pytest.mark.parametrize("shape", HOST_SHAPES, ids=lambda s: "B{B}_H{H}_Hkv{Hkv}_N{N}_d{d}".format(**s))
@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_host_entry_point_matches_device_entry_point(dtype, shape):
    w = inputs.Workload("host", dtype=dtype, seed=9, **shape)
    x = inputs.make_inputs(w)
    o_dev, lse_dev = run_cuda(w, x)
    code = binding.ATTN_DTYPE_FP8_E4M3 if dtype == "fp8_e4m3" else binding.ATTN_DTYPE_BF16
    ws = torch.empty(binding.attn_fwd_host_workspace_bytes(w.B, w.H, w.Hkv, w.N, w.d, code), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty((w.B, w.N, w.H, w.d), dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory()
    binding.attn_fwd_host(x.q.pin_memory(), x.k.pin_memory(), x.v.pin_memory(), o, lse, w.causal, ws,
                          descale_q=x.descale_q, descale_k=x.descale_k, descale_v=x.descale_v)
    assert torch.equal(o, o_dev.cpu()) and torch.equal(lse, lse_dev.cpu())
