"""Pins of the fp8 quantisation oracle (oracle/fp8_quant.py) against the e4m3 format, a library
Hadamard routine, closed forms and brute force; each would catch a plausible slip in it."""
import numpy as np
import pytest
import torch

from oracle import fp8_quant as fq

scipy_linalg = pytest.importorskip("scipy.linalg")


# ---------------------------------------------------------------- e4m3 rounding

def test_e4m3_hand_values():
    # values fixed by the format: 3 mantissa bits, bias 7, max 448, subnormal step 2^-9
    cases = {
        448.0: 448.0, 416.0: 416.0, 440.0: 448.0,      # step 32 in [256, 512)
        432.0: 448.0, 400.0: 384.0,                    # ties between 13*32 | 14*32 and 12*32 | 13*32 -> even
        460.0: 448.0, 464.0: 448.0, 1.0e6: 448.0,      # saturation
        1.0: 1.0, 1.0625: 1.0, 1.0625 + 1e-9: 1.125,   # 1.0625 is the tie between 1 and 1.125 -> even (1.0)
        1.1875: 1.25,                                  # tie between 1.125 and 1.25 -> even mantissa (1.25)
        2.0 ** -6: 2.0 ** -6,                          # smallest normal
        2.0 ** -9: 2.0 ** -9,                          # smallest subnormal
        2.0 ** -10: 0.0,                               # half a subnormal step: tie -> 0 (even)
        3 * 2.0 ** -10: 2.0 ** -8,                     # 1.5 steps: tie -> 2 steps
        7 * 2.0 ** -9: 7 * 2.0 ** -9,                  # largest subnormal
        0.0: 0.0,
    }
    for y, want in cases.items():
        assert fq.e4m3_round(y) == want, (y, fq.e4m3_round(y), want)
        assert fq.e4m3_round(-y) == -want


def test_e4m3_matches_library_cast():
    # torch's float8_e4m3fn cast (round to nearest even) on every code, every midpoint and
    # random values inside the finite range (the library cast does not saturate: stay below 464)
    codes = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().double().numpy()
    codes = np.unique(codes[np.isfinite(codes)])
    mids = (codes[1:] + codes[:-1]) / 2
    rng = np.random.default_rng(3)
    rand = rng.uniform(-460, 460, 20000) * 2.0 ** rng.integers(-14, 1, 20000)
    y = np.concatenate([codes, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf), rand])
    y = y[np.abs(y) < 464].astype(np.float32).astype(np.float64)
    lib = torch.tensor(y, dtype=torch.float32).to(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(fq.e4m3_round(y), lib)


# ---------------------------------------------------------------- Hadamard rotation

@pytest.mark.parametrize("d", [1, 2, 4, 64, 128, 256])
def test_sylvester_matches_scipy(d):
    assert np.array_equal(fq.sylvester_hadamard(d), scipy_linalg.hadamard(d))


def test_rotation_is_orthogonal_and_keeps_inner_products():
    rng = np.random.default_rng(1)
    s = rng.choice([-1.0, 1.0], 128)
    R = fq.rotation(s)
    assert np.abs(R @ R.T - np.eye(128)).max() < 1e-14
    q, k = rng.standard_normal((50, 128)), rng.standard_normal((70, 128))
    assert np.abs((q @ R) @ (k @ R).T - q @ k.T).max() < 1e-11


def test_rotation_closed_forms():
    s = np.array([1.0, -1.0, -1.0, 1.0])
    R = fq.rotation(s)
    # e_0 R = sigma_0 (row 0 of H) / 2 = [1, 1, 1, 1] / 2; e_1 R = -[1, -1, 1, -1] / 2
    assert np.allclose(np.eye(4)[0] @ R, [0.5, 0.5, 0.5, 0.5], atol=0, rtol=0)
    assert np.allclose(np.eye(4)[1] @ R, [-0.5, 0.5, -0.5, 0.5], atol=0, rtol=0)
    # one outlier spreads evenly: amax of a 1-hot row drops by sqrt(d)
    x = np.zeros(128)
    x[37] = 100.0
    s = np.random.default_rng(2).choice([-1.0, 1.0], 128)
    assert np.allclose(np.abs(x @ fq.rotation(s)), 100.0 / np.sqrt(128.0), rtol=1e-15, atol=0)
    with pytest.raises(ValueError):
        fq.rotation(np.array([1.0, 0.5]))


# ---------------------------------------------------------------- block quantisation

def bf16_draw(shape, seed, outliers=0.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(shape, generator=g)
    if outliers:
        m = torch.rand(shape, generator=g) < outliers
        x[m] *= 20.0
    return x.to(torch.bfloat16).double().numpy()


def test_block_descales_by_brute_force():
    x = bf16_draw((2, 200, 3, 64), 4)      # N = 200: blocks of 64 leave a short last block (8 rows)
    codes, ds = fq.quantize_blocks(x, 64)
    assert ds.shape == (2, 3, 4) and ds.dtype == np.float32
    for b in range(2):
        for h in range(3):
            for i in range(4):
                blk = x[b, i * 64:(i + 1) * 64, h, :]
                assert ds[b, h, i] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))
                # the block's largest value maps to 448 exactly
                assert np.abs(codes[b, i * 64:(i + 1) * 64, h, :]).max() == 448.0


def test_codes_match_library_cast_of_fp32_quotient():
    x = bf16_draw((1, 256, 2, 128), 5, outliers=0.002)
    codes, ds = fq.quantize_blocks(x, 128)
    for h in range(2):
        for i in range(2):
            blk = x[0, i * 128:(i + 1) * 128, h, :].astype(np.float32)
            want = torch.tensor(blk / ds[0, h, i]).to(torch.float8_e4m3fn).double().numpy()
            assert np.array_equal(codes[0, i * 128:(i + 1) * 128, h, :], want)


def test_dequantised_error_within_format_bound():
    x = bf16_draw((1, 300, 2, 128), 6, outliers=0.001)
    codes, ds = fq.quantize_blocks(x, 128)
    deq = fq.dequantize_blocks(codes, ds, 128)
    rows = np.arange(300) // 128
    dsr = np.transpose(ds.astype(np.float64)[:, :, rows], (0, 2, 1))[:, :, :, None]
    # half a step: 2^-4 relative for normal codes, 2^-10 * descale absolute in the subnormal range,
    # plus the fp32 rounding of the quotient
    bound = np.maximum(np.abs(x) * 2.0 ** -4, dsr * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)


def test_zero_block_and_single_block():
    x = np.zeros((1, 10, 1, 64))
    codes, ds = fq.quantize_blocks(x, 4)
    assert np.all(codes == 0) and np.all(ds == 1.0) and ds.shape == (1, 1, 3)
    x = bf16_draw((1, 10, 2, 64), 7)
    c1, d1 = fq.quantize_blocks(x, 10)
    c2, d2 = fq.quantize_blocks(x, 1000)      # one block per (b, head) either way
    assert np.array_equal(c1, c2) and np.array_equal(d1, d2) and d1.shape == (1, 2, 1)


def test_rotated_quantisation_reconstructs_the_rotation():
    rng = np.random.default_rng(8)
    s = rng.choice([-1.0, 1.0], 128)
    x = bf16_draw((1, 256, 2, 128), 9, outliers=0.002)
    codes, ds = fq.quantize_blocks(x, 64, s)
    xr = x @ fq.rotation(s)
    deq = fq.dequantize_blocks(codes, ds, 64)
    assert np.abs(deq - xr).max() <= np.abs(xr).max() * 2.0 ** -4 * 1.01
    # the codes do not depend on the 1/sqrt(d) normalisation; the descale carries it
    c_u, d_u = fq.quantize_blocks(x @ (s[:, None] * fq.sylvester_hadamard(128)), 64)
    assert np.array_equal(codes, c_u)
    assert np.allclose(ds, d_u / np.sqrt(128.0), rtol=2 ** -23, atol=0)
    # the rotation spreads the outliers: a smaller amax per block
    _, ds_plain = fq.quantize_blocks(x, 64)
    assert np.median(ds_plain / ds) > 1.5


def test_block_mapping_is_per_batch_and_head():
    # give every (b, head, block) its own magnitude; each descale must see only its own rows
    x = np.ones((2, 6, 3, 64))
    mag = np.arange(1, 2 * 3 * 3 + 1, dtype=np.float64).reshape(2, 3, 3)     # [b, h, block]
    for b in range(2):
        for h in range(3):
            for i in range(3):
                x[b, 2 * i:2 * i + 2, h, :] *= mag[b, h, i]
    _, ds = fq.quantize_blocks(x, 2)
    assert np.array_equal(ds, (mag.astype(np.float32) / np.float32(448.0)).astype(np.float32))
    deq = fq.dequantize_blocks(np.full(x.shape, 448.0), ds, 2)
    assert np.allclose(deq, x, rtol=1e-6)


def test_block_scales_and_rotation_reduce_attention_error():
    """The pages' claim, on the oracle: with outliers in q, k and v (0.1% of entries x10), block
    scales plus the rotation give a smaller attention error than one scale per tensor. The pages
    quote 2.6x on their data; this seeded recipe gives about 1.5x, and the test asks for 1.3x."""
    import oracle
    rng = np.random.default_rng(5)
    B, N, H, d = 1, 1024, 2, 128

    def draw():
        x = rng.standard_normal((B, N, H, d))
        m = rng.random(x.shape) < 0.001
        x[m] = rng.standard_normal(int(m.sum())) * 10.0
        return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).double().numpy()

    q, k, v = draw(), draw(), draw()
    s = rng.choice([-1.0, 1.0], d)

    def att(q, k, v):
        return np.stack([oracle.attention_head(q[0, :, h], k[0, :, h], v[0, :, h], d ** -0.5, True)[0]
                         for h in range(H)])

    def per_tensor(x):     # one block spanning every row of every head
        c, ds = fq.quantize_blocks(x.reshape(B, N * H, 1, d), N * H)
        return fq.dequantize_blocks(c, ds, N * H).reshape(x.shape)

    def per_block(x, rows, signs=None):
        c, ds = fq.quantize_blocks(x, rows, signs)
        return fq.dequantize_blocks(c, ds, rows)

    ref = att(q, k, v)
    err = lambda o: float(np.sqrt(np.mean((o - ref) ** 2)))
    e_tensor = err(att(per_tensor(q), per_tensor(k), per_tensor(v)))
    vq = per_block(v, N)   # v: one scale per (batch, head) in both blocked variants
    e_block = err(att(per_block(q, 128), per_block(k, 64), vq))
    R = fq.rotation(s)
    # scores of the rotated, quantised q and k: (q' R^T)(k' R^T)^T = q' k'^T
    e_rot = err(att(per_block(q, 128, s) @ R.T, per_block(k, 64, s) @ R.T, vq))
    assert e_block < e_tensor and e_rot < e_block
    assert e_tensor / e_rot > 1.3, (e_tensor, e_block, e_rot)
