"""bench.py's kernel-launch accounting (the `gpu_launches` key) against the library's own launch
rules, on the CPU: a non-causal forward that cuts tiles' keys across launches makes two, split-KV
decode two (forward + combine), the block-scaled chain five quantiser launches plus the forward."""
import bench
from exact_attention_72_gb300 import binding, inputs


def test_forward_launch_counts_follow_the_cutting_rule():
    for w in inputs.WORKLOADS.values():
        cut = len(binding.attn_fwd_tail_units(w.B, w.H, w.N, w.d, w.causal, fp8=w.dtype != "bf16")) > 0
        assert bench.launches_per_step(w) == (2 if cut else 1), w.name
    assert bench.launches_per_step(inputs.WORKLOADS["noncausal_bf16_n4096_d256"]) == 2
    assert bench.launches_per_step(inputs.WORKLOADS["fp8_noncausal_n8192_d128"]) == 2
    assert bench.launches_per_step(inputs.WORKLOADS["causal_gqa_bf16_n8192_d128"]) == 1
    # 1024 tiles on 152 SMs: the last 264 dealt in equal shares of key tiles
    assert bench.launches_per_step(inputs.WORKLOADS["noncausal_bf16_n16384_d64"]) == 2


def test_decode_and_block_scaled_counts():
    for w in inputs.DECODE_WORKLOADS.values():
        assert bench.launches_per_step(w) == 2
    w = inputs.FP8_BLOCK_WORKLOADS["fp8_block_hadamard_noncausal_n8192_d128"]
    # q and k quantised in one launch each, v in three (maxima, codes, descales), forward in two
    assert bench.launches_per_step(w) == 1 + 1 + 3 + 2
