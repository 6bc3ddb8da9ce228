"""Seeded synthetic inputs for the attention forward workloads.

This module is shared by the CUDA path's tests and benchmark and by the oracle's
tests. It holds no attention arithmetic: it only draws random tensors, rounds
them to the storage type the kernel reads (bf16, or e4m3 with a per-tensor
descale) and hands out an fp64 copy of exactly those stored values.

Workload shapes follow the pages' benchmark and configurations:
  * "Lecture 9 — Hopper / FlashAttention-3 / FlashAttention-4", "Benchmark task":
    q, k, v of shape (B, N, H, D) drawn with randn, bf16, causal.
  * "flash-attention-3" (ai.thesatyajit.com), "FP8 is a different kernel":
    FP8 inputs with per-tensor descale factors.

Readings taken where the pages are silent (each one is listed in the design
notes of the repository):
  * seeds: ``torch.Generator('cpu').manual_seed(1000 + index)``; draw order Q, K,
    V (fp32 randn), then outlier positions, then outlier signs;
  * outliers: ``round(frac * K.numel())`` flat positions drawn without
    replacement, each set to +-magnitude with probability 1/2 per sign, before
    the bf16 rounding (8 is exact in bf16);
  * FP8: ``descale = amax(|x|) / 448`` in fp32 and
    ``x8 = e4m3(round-to-nearest-even, saturate to +-448)(x / descale)``; the
    value the kernel sees is ``x8 * descale``.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention-forward problem: shapes, mask, storage type and input recipe."""

    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    causal: bool
    dtype: str = "bf16"            # "bf16", "fp8_e4m3" (storage type of q, k, v), or "fp8_block":
                                   # stored bf16, quantised on the GPU into e4m3 blocks each step
    seed: int = 1000
    k_outlier_frac: float = 0.0    # fraction of K entries replaced by +-k_outlier_mag
    k_outlier_mag: float = 8.0
    Nk: Optional[int] = None       # keys per sequence when it differs from N (decode shapes)
    splits: int = 1                # split-KV ranges (decode shapes); 0: the library's choice

    @property
    def n_keys(self) -> int:
        return self.N if self.Nk is None else self.Nk

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """4*B*H*Nq*Nk*d, halved for causal (the benchmark's counting convention)."""
        f = 4.0 * self.B * self.H * self.N * self.n_keys * self.d
        return f / 2.0 if self.causal else f

    @property
    def elt_bytes(self) -> int:
        return 1 if self.dtype == "fp8_e4m3" else 2

    @property
    def algorithmic_bytes(self) -> int:
        """Read q, k, v once; write o (bf16) and lse (fp32) once."""
        q = self.B * self.N * self.H * self.d * self.elt_bytes
        kv = 2 * self.B * self.n_keys * self.Hkv * self.d * self.elt_bytes
        o = self.B * self.N * self.H * self.d * 2
        lse = self.B * self.H * self.N * 4
        return q + kv + o + lse

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five configurations (the fourth has two shapes). Index i uses seed 1000+i.
WORKLOADS = {
    "tiny_bf16_d64": Workload("tiny_bf16_d64", B=1, H=2, Hkv=2, N=256, d=64, causal=False, seed=1000),
    "causal_bf16_n2048_d128": Workload("causal_bf16_n2048_d128", B=4, H=16, Hkv=16, N=2048, d=128,
                                       causal=True, seed=1001),
    "causal_gqa_bf16_n8192_d128": Workload("causal_gqa_bf16_n8192_d128", B=2, H=32, Hkv=8, N=8192, d=128,
                                           causal=True, seed=1002, k_outlier_frac=0.005),
    "noncausal_bf16_n16384_d64": Workload("noncausal_bf16_n16384_d64", B=1, H=16, Hkv=16, N=16384, d=64,
                                          causal=False, seed=1003),
    "noncausal_bf16_n4096_d256": Workload("noncausal_bf16_n4096_d256", B=2, H=8, Hkv=8, N=4096, d=256,
                                          causal=False, seed=1004),
    "fp8_noncausal_n8192_d128": Workload("fp8_noncausal_n8192_d128", B=1, H=16, Hkv=16, N=8192, d=128,
                                         causal=False, dtype="fp8_e4m3", seed=1005),
}

# Forward workloads beyond the five configurations: e4m3 at d = 64, in the shape of the d = 64
# configuration.
EXTRA_FWD_WORKLOADS = {
    "fp8_noncausal_n16384_d64": Workload("fp8_noncausal_n16384_d64", B=1, H=16, Hkv=16, N=16384, d=64,
                                         causal=False, dtype="fp8_e4m3", seed=1006),
}

# The headline workload the benchmark times.
HEADLINE = "causal_gqa_bf16_n8192_d128"

# Decode-shaped workloads for the split-KV path (few queries, long KV sequence, no mask).
DECODE_WORKLOADS = {
    "decode_gqa_bf16_nq1_nk16384_d128": Workload("decode_gqa_bf16_nq1_nk16384_d128", B=8, H=32, Hkv=8, N=1,
                                                 d=128, causal=False, seed=1101, Nk=16384, splits=0),
    "decode_gqa_bf16_nq16_nk8192_d128": Workload("decode_gqa_bf16_nq16_nk8192_d128", B=4, H=32, Hkv=8, N=16,
                                                 d=128, causal=False, seed=1102, Nk=8192, splits=0),
}


# Block-scaled e4m3 workload: bf16 inputs (K with outliers) quantised on the GPU every step (q in
# blocks of 128 rows and k in blocks of 64 rows, both after the random Hadamard rotation; v with
# one descale per head), then the block-scaled e4m3 forward. Same shape as the fp8 configuration.
FP8_BLOCK_WORKLOADS = {
    "fp8_block_hadamard_noncausal_n8192_d128": Workload("fp8_block_hadamard_noncausal_n8192_d128", B=1, H=16,
                                                        Hkv=16, N=8192, d=128, causal=False, dtype="fp8_block",
                                                        seed=1201, k_outlier_frac=0.005),
}


# Backward pass on the GQA configuration's shape: q, k, v and the output gradient dO drawn in that
# order (fp32 randn, rounded to bf16); O and LSE come from the forward.
BWD_WORKLOADS = {
    "bwd_causal_gqa_bf16_n8192_d128": Workload("bwd_causal_gqa_bf16_n8192_d128", B=2, H=32, Hkv=8, N=8192, d=128,
                                               causal=True, seed=1401),
}


def make_grad_output(w: Workload, seed: Optional[int] = None) -> torch.Tensor:
    """Seeded output gradient dO [B, N, H, d] in bf16 (drawn after q, k, v from its own seed)."""
    g = torch.Generator(device="cpu")
    g.manual_seed((w.seed if seed is None else seed) + 100000)
    return torch.randn((w.B, w.N, w.H, w.d), generator=g, dtype=torch.float32).to(torch.bfloat16)


@dataclasses.dataclass(frozen=True)
class VarlenWorkload:
    """A ragged batch: sequence b has lengths_q[b] queries and lengths_k[b] keys, packed by rows."""

    name: str
    H: int
    Hkv: int
    d: int
    causal: bool
    lengths_q: tuple
    lengths_k: Optional[tuple] = None   # None: same as lengths_q
    dtype: str = "bf16"
    seed: int = 1300

    @property
    def lk(self) -> tuple:
        return self.lengths_q if self.lengths_k is None else self.lengths_k

    @property
    def B(self) -> int:
        return len(self.lengths_q)

    @property
    def total_q(self) -> int:
        return int(sum(self.lengths_q))

    @property
    def total_k(self) -> int:
        return int(sum(self.lk))

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lengths_q)]).astype(np.int32)

    @property
    def cu_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lk)]).astype(np.int32)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Sum over sequences of 4*H*Nq*Nk*d, halved for causal (the benchmark's convention)."""
        f = sum(4.0 * self.H * nq * nk * self.d for nq, nk in zip(self.lengths_q, self.lk))
        return f / 2.0 if self.causal else f


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    """n sequence lengths drawn uniformly from [lo, hi] (numpy PCG64 seeded with ``seed``)."""
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


# Ragged batch of the GQA configuration's heads: 16 sequences of 256 .. 8192 tokens, causal.
VARLEN_WORKLOADS = {
    "varlen_causal_gqa_bf16_16seq_d128": VarlenWorkload("varlen_causal_gqa_bf16_16seq_d128", H=32, Hkv=8, d=128,
                                                        causal=True, lengths_q=varlen_lengths(16, 256, 8192, 1301),
                                                        seed=1301),
}


def make_varlen_inputs(w: VarlenWorkload):
    """Seeded packed q [total_q, H, d], k, v [total_k, Hkv, d] as AttnInputs (bf16 or e4m3)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = torch.randn((w.total_q, w.H, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.total_k, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.total_k, w.Hkv, w.d), generator=g, dtype=torch.float32)
    if w.dtype == "bf16":
        return AttnInputs(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16))
    q8, sq = quantize_e4m3(q)
    k8, sk = quantize_e4m3(k)
    v8, sv = quantize_e4m3(v)
    return AttnInputs(q8, k8, v8, sq, sk, sv)


@dataclasses.dataclass
class AttnInputs:
    """Stored inputs (what the kernel reads) plus their exact fp64 values."""

    q: torch.Tensor            # [B, N, H, d]   bf16 or float8_e4m3fn, CPU
    k: torch.Tensor            # [B, N, Hkv, d]
    v: torch.Tensor            # [B, N, Hkv, d]
    descale_q: float = 1.0     # fp32 value; 1.0 for bf16
    descale_k: float = 1.0
    descale_v: float = 1.0

    def as_f64(self):
        """fp64 numpy copies of the values the kernel sees (x8 * descale for e4m3)."""
        def up(t, s):
            a = t.to(torch.float32).to(torch.float64).numpy()
            if t.dtype == torch.float8_e4m3fn:
                a = a * np.float64(np.float32(s))
            return a
        return up(self.q, self.descale_q), up(self.k, self.descale_k), up(self.v, self.descale_v)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor e4m3 quantisation: returns (x8, descale) with x ~= x8 * descale."""
    x = x.to(torch.float32)
    amax = float(x.abs().max())
    descale = np.float32(amax / E4M3_MAX) if amax > 0 else np.float32(1.0)
    y = (x / torch.tensor(descale, dtype=torch.float32)).clamp_(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn), float(descale)


def quantize_e4m3_per_head(x: torch.Tensor):
    """Per-(batch, head) e4m3 quantisation of x [B, N, H, d]: returns (x8, descale [B, H]) with
    x[b, :, h, :] ~= x8[b, :, h, :] * descale[b, h]."""
    x = x.to(torch.float32)
    amax = x.abs().amax(dim=(1, 3))                                   # [B, H]
    descale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax)).to(torch.float32)
    y = (x / descale[:, None, :, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    return y.to(torch.float8_e4m3fn), descale


def hadamard_signs(d: int, seed: int) -> torch.Tensor:
    """The d random signs (+-1, float32) of a random Hadamard rotation, drawn from ``seed``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.randint(0, 2, (d,), generator=g).to(torch.float32) * 2.0 - 1.0


def make_inputs(w: Workload, seed: Optional[int] = None) -> AttnInputs:
    """Draw the seeded inputs of workload ``w`` on the CPU."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    q = torch.randn((w.B, w.N, w.H, w.d), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.n_keys, w.Hkv, w.d), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.n_keys, w.Hkv, w.d), generator=g, dtype=torch.float32)
    if w.k_outlier_frac > 0:
        n_out = int(round(w.k_outlier_frac * k.numel()))
        idx = torch.randperm(k.numel(), generator=g)[:n_out]
        sign = torch.randint(0, 2, (n_out,), generator=g).to(torch.float32) * 2.0 - 1.0
        k.view(-1)[idx] = sign * w.k_outlier_mag
    if w.dtype in ("bf16", "fp8_block"):
        return AttnInputs(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16))
    if w.dtype == "fp8_e4m3":
        q8, sq = quantize_e4m3(q)
        k8, sk = quantize_e4m3(k)
        v8, sv = quantize_e4m3(v)
        return AttnInputs(q8, k8, v8, sq, sk, sv)
    raise ValueError(f"unknown dtype {w.dtype!r}")
