"""FP8 (e4m3) block quantisation and Hadamard incoherence processing, on the CPU.

TEST INFRASTRUCTURE ONLY. This file is part of the oracle that the CUDA path is
checked against. Only the tests, the package's smoke entry and the benchmark's
CPU baseline leg may import it; the library never does, and it shares no code
with the CUDA kernels.

What it computes, for a tensor x laid out [B, N, Hx, d] (Hx heads of d values):

  * Hadamard rotation (optional), per row of d values:
        x' = x R,   R = diag(sigma) H_d / sqrt(d)
    H_d is the Sylvester Hadamard matrix (entries +-1, H_d H_d^T = d I) and sigma
    a vector of d random signs, drawn by the caller and passed in. R is
    orthogonal, so rotating both Q and K by the same R leaves Q K^T unchanged.
  * Block quantisation: rows [i*R0, (i+1)*R0) of one (b, head) form block i
    (the last block may be short). Per block, in fp32:
        descale = amax(|x'|) / 448            (1 when the block is all zero)
        code    = e4m3(x' / descale)          (round to nearest even, saturate to +-448)
    and code * descale approximates x'.

Where floating point decides a code, it is decided in fp32, the precision the
kernel uses: the rotated values are computed exactly (fp64 sums of bf16 inputs)
and rounded once to fp32, then divided in fp32. With a rotation the stored
descale is the fp32 rounding of descale_u / sqrt(d), where descale_u is the
descale of the unnormalised rotation x diag(sigma) H_d; the codes do not depend
on the 1/sqrt(d) factor, since it cancels in x' / descale.

Sources:
  * "FlashAttention-3 Deep Dive" (mojostudio.in), section 4 "FP8 Block
    Quantization & Numerical Incoherence Elimination": a separate fp32 scale
    per tile, x~ = clip(x / s, -448, 448); Q' = Q H, K' = K H with a random
    orthogonal Hadamard matrix, and the invariance (QH)(KH)^T = QK^T.
  * Same page, the FP8 question of its FAQ: block scales per 128 x 64 tile plus
    a randomised Hadamard transform reduce the error against the standard FP8
    path. The tile is read as 128 query rows by 64 keys of the score matrix,
    so Q blocks hold 128 rows and K blocks 64 rows (of one batch and head).
  * The e4m3 format (OCP 8-bit floating point): 1 sign bit, 4 exponent bits
    with bias 7, 3 mantissa bits, largest finite value 448, subnormal step 2^-9.

Parity pins live in tests/test_oracle_fp8.py; every function here is pinned.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_round(y) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at +-448; fp64 out.

    A magnitude a in binade [2^e, 2^(e+1)) with e >= -6 has step 2^(e-3) (three
    mantissa bits); below 2^-6 the subnormal step is 2^-9.
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, e = np.frexp(a)                     # a = f 2^e with f in [0.5, 1): binade 2^(e-1)
    step = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    q = np.minimum(np.round(a / step) * step, E4M3_MAX)   # np.round: half to even
    return np.copysign(q, y)


def sylvester_hadamard(d: int) -> np.ndarray:
    """H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]]; d a power of two."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation(signs) -> np.ndarray:
    """The random orthogonal Hadamard matrix R = diag(sigma) H_d / sqrt(d)."""
    s = np.asarray(signs, dtype=np.float64)
    if not np.all(np.abs(s) == 1.0):
        raise ValueError("signs must be +-1")
    d = s.shape[0]
    return (s[:, None] * sylvester_hadamard(d)) / np.sqrt(d)


def quantize_blocks(x, block_rows: int, signs=None):
    """Block-quantise x [B, N, Hx, d] (values exact in fp64, e.g. bf16 upcast).

    Returns (codes, descale): codes [B, N, Hx, d] as the fp64 value of each e4m3
    code, descale fp32 [B, Hx, ceil(N / block_rows)].
    """
    x = np.asarray(x, dtype=np.float64)
    B, N, Hx, d = x.shape
    if block_rows < 1:
        raise ValueError("block_rows must be positive")
    if signs is not None:
        u = (x * np.asarray(signs, dtype=np.float64)) @ sylvester_hadamard(d)   # exact: sums of bf16 values
    else:
        u = x
    u32 = u.astype(np.float32)
    nblk = -(-N // block_rows)
    codes = np.zeros(x.shape, dtype=np.float64)
    descale = np.zeros((B, Hx, nblk), dtype=np.float32)
    for b in range(B):
        for h in range(Hx):
            for i in range(nblk):
                blk = u32[b, i * block_rows:(i + 1) * block_rows, h, :]
                amax = np.float32(np.abs(blk).max())
                ds = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
                codes[b, i * block_rows:(i + 1) * block_rows, h, :] = e4m3_round(blk / ds)   # fp32 division
                if signs is not None:
                    ds = np.float32(np.float64(ds) / np.sqrt(np.float64(d)))
                descale[b, h, i] = ds
    return codes, descale


def dequantize_blocks(codes, descale, block_rows: int) -> np.ndarray:
    """code * descale of its block, fp64 [B, N, Hx, d]."""
    codes = np.asarray(codes, dtype=np.float64)
    N = codes.shape[1]
    rows = np.arange(N) // block_rows                           # block of each row
    ds = np.asarray(descale, dtype=np.float64)[:, :, rows]     # [B, Hx, N]
    return codes * np.transpose(ds, (0, 2, 1))[:, :, :, None]
