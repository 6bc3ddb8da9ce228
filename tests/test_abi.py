"""C-ABI checks that need no GPU: the library builds, loads, exports every declared entry point,
and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from exact_attention_72_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("attn_fwd", "attn_fwd_host", "attn_get_status", "attn_get_status_detail", "attn_status_string"):
        assert n in names


def test_get_status_has_the_one_argument_form():
    """attn_get_status takes the stream alone; the raw word comes from attn_get_status_detail."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    assert re.search(r"attn_status_t\s+attn_get_status\s*\(\s*cudaStream_t\s+stream\s*\)\s*;", text)
    assert re.search(r"attn_status_t\s+attn_get_status_detail\s*\(\s*cudaStream_t\s+stream\s*,\s*uint32_t\s*\*\s*detail\s*\)",
                     text)


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared in attn.h but not exported: {missing}"


def test_status_strings_and_version(lib):
    assert binding.attn_status_string(binding.ATTN_OK) == "ok"
    assert binding.attn_status_string(binding.ATTN_ERR_TIMEOUT) == "kernel wait timed out"
    assert binding.attn_status_string(99) == "unknown status"
    assert binding.attn_version() >= 100


def _call(lib, q=4096, k=8192, v=12288, o=16384, lse=1 << 20, B=1, H=2, Hkv=2, N=128, d=128, scale=0.1,
          causal=0, dtype=0, dq=None, dk=None, dv=None):
    # Fake, non-dereferenced addresses: every call here must fail validation before any CUDA call.
    return lib.attn_fwd(q, k, v, o, lse, B, H, Hkv, N, d, scale, causal, dtype, dq, dk, dv, None)


def test_validation_rejects_bad_arguments(lib):
    INV, UNS = binding.ATTN_ERR_INVALID_ARG, binding.ATTN_ERR_UNSUPPORTED
    assert _call(lib, q=0) == INV                         # null pointer
    assert _call(lib, lse=0) == INV
    assert _call(lib, B=0) == INV                         # empty batch
    assert _call(lib, N=0) == INV                         # empty sequence
    assert _call(lib, H=3, Hkv=2) == INV                  # H not a multiple of Hkv
    assert _call(lib, scale=float("nan")) == INV
    assert _call(lib, scale=float("inf")) == INV
    assert _call(lib, dtype=7) == INV
    assert _call(lib, d=96) == UNS                        # head dim without an instance
    assert _call(lib, d=96, dtype=1, dq=1 << 24, dk=1 << 24, dv=1 << 24) == UNS   # e4m3: d = 64, 128, 256
    assert _call(lib, scale=0.0) == UNS                  # 0 * (-inf) for masked scores
    assert _call(lib, dtype=1) == INV                     # fp8 without descales
    assert _call(lib, q=4097) == INV                      # misaligned (TMA needs 16 bytes)
    assert _call(lib, o=16392) == INV
    assert _call(lib, lse=(1 << 20) + 2) == INV
    # o overlapping q (q spans 1*128*2*128*2 = 64 KiB from 4096)
    assert _call(lib, q=1 << 16, k=1 << 24, v=1 << 25, o=(1 << 16) + 4096, lse=1 << 26) == INV
    # lse overlapping v
    assert _call(lib, q=1 << 16, k=1 << 24, v=1 << 25, o=1 << 27, lse=(1 << 25) + 64) == INV


def test_host_workspace_size(lib):
    n = binding.attn_fwd_host_workspace_bytes(2, 32, 8, 8192, 128, binding.ATTN_DTYPE_BF16)
    q = 2 * 8192 * 32 * 128 * 2
    kv = 2 * 8192 * 8 * 128 * 2
    assert n >= q + 2 * kv + q + 2 * 32 * 8192 * 4
    assert binding.attn_fwd_host_workspace_bytes(0, 1, 1, 1, 128, 0) == 0
    assert binding.attn_fwd_host_workspace_bytes(1, 1, 1, 1, 96, 0) == 0


def test_splitkv_validation(lib):
    INV, UNS = binding.ATTN_ERR_INVALID_ARG, binding.ATTN_ERR_UNSUPPORTED

    def call(Nq=1, Nk=512, B=1, H=8, Hkv=2, d=128, splits=4, ws=1 << 28, ws_bytes=1 << 20, scale=0.1, dtype=0,
             q=1 << 16, k=1 << 20, v=1 << 24, o=1 << 26, lse=1 << 27):
        return lib.attn_fwd_splitkv(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, scale, splits, dtype, None, None, None,
                                    ws, ws_bytes, None)

    assert call(Nq=0) == INV
    assert call(Nk=0) == INV
    assert call(splits=0) == INV
    assert call(splits=129) == INV
    assert call(H=6, Hkv=2) == UNS                 # group of 3 heads cannot tile 128 rows
    assert call(d=96) == UNS
    assert call(ws_bytes=16) == INV                 # workspace too small
    assert call(ws=(1 << 28) + 8) == INV            # workspace misaligned
    assert call(ws=(1 << 16)) == INV                # workspace overlaps q
    need = binding.attn_fwd_splitkv_workspace_bytes(2, 32, 1, 128, 16)
    assert need >= 16 * 2 * 32 * 1 * (128 + 1) * 4
    assert binding.attn_fwd_splitkv_workspace_bytes(1, 1, 1, 128, 0) == 0


def test_fp8_scaled_validation(lib):
    INV, UNS = binding.ATTN_ERR_INVALID_ARG, binding.ATTN_ERR_UNSUPPORTED

    def call(B=1, H=4, Hkv=2, N=256, d=128, sqb=0, sqh=1, skb=0, skh=1, dq=1 << 12, dk=1 << 13, dv=1 << 14):
        return lib.attn_fwd_fp8_scaled(1 << 16, 1 << 20, 1 << 24, 1 << 26, 1 << 27, B, H, Hkv, N, d, 0.1, 1,
                                       dq, sqb, sqh, dk, dv, skb, skh, None)

    assert call(sqh=-1) == INV
    assert call(skb=-4) == INV
    assert call(dq=0) == INV                         # descale pointers are required
    assert call(dv=0) == INV
    assert call(N=0) == INV
    assert call(d=96) == UNS                         # e4m3 is built for d = 64, 128 and 256


def test_quantize_and_blockscaled_validation(lib):
    INV, UNS = binding.ATTN_ERR_INVALID_ARG, binding.ATTN_ERR_UNSUPPORTED

    def q(x=1 << 20, x8=1 << 26, ds=1 << 28, B=1, N=256, Hx=2, d=128, R=64, signs=None):
        return lib.attn_quantize_e4m3(x, x8, ds, B, N, Hx, d, R, signs, None)

    assert q(x=0) == INV and q(x8=0) == INV and q(ds=0) == INV
    assert q(R=0) == INV and q(N=0) == INV and q(Hx=0) == INV
    assert q(d=96) == UNS and q(d=32) == UNS
    assert q(x=(1 << 20) + 8) == INV                    # x not 16-byte aligned
    assert q(ds=(1 << 28) + 2) == INV                   # descale not 4-byte aligned
    assert q(x8=(1 << 20) + 1024) == INV                # codes overlap x
    assert q(ds=(1 << 26) + 64) == INV                  # descales overlap the codes
    assert binding.attn_quantize_e4m3_descale_count(2, 300, 3, 128) == 2 * 3 * 3
    assert binding.attn_quantize_e4m3_descale_count(1, 300, 1, 0) == 0

    def f(N=256, d=128, H=4, Hkv=2):
        return lib.attn_fwd_fp8_blockscaled(1 << 16, 1 << 20, 1 << 24, 1 << 26, 1 << 27, 1, H, Hkv, N, d, 0.1, 1,
                                            1 << 12, 1 << 13, 1 << 14, None)

    assert f(N=0) == INV and f(H=0) == INV
    assert f(d=96) == UNS


def test_varlen_validation(lib):
    INV, UNS = binding.ATTN_ERR_INVALID_ARG, binding.ATTN_ERR_UNSUPPORTED
    need = binding.attn_varlen_plan_bytes(3, 4, 1000, 128)
    # header (8 words), 4 prefix words, padding to 8 bytes, then 4 heads x (ceil(1000/256) + 3) tiles
    assert need == ((8 + 3 + 2) & ~1) * 4 + 4 * (4 + 3) * 8
    assert binding.attn_varlen_plan_bytes(0, 4, 1000, 128) == 0
    assert binding.attn_varlen_plan_bytes(3, 4, 1000, 96) == 0

    def plan(cu_q=1 << 12, cu_k=1 << 13, B=3, H=4, tq=1000, tk=1000, d=128, p=1 << 20, nbytes=1 << 16):
        return lib.attn_varlen_plan(cu_q, cu_k, B, H, tq, tk, d, 1, p, nbytes, None)

    assert plan(cu_q=0) == INV and plan(p=0) == INV
    assert plan(B=0) == INV and plan(tq=-1) == INV
    assert plan(d=96) == UNS
    assert plan(p=(1 << 20) + 8) == INV          # plan not 16-byte aligned
    assert plan(nbytes=need - 1) == INV           # plan buffer too small

    def fwd(q=1 << 16, plan=1 << 28, plan_bytes=1 << 16, B=3, H=4, Hkv=2, tq=1000, tk=900, d=128, scale=0.1,
            dtype=0):
        return lib.attn_fwd_varlen(q, 1 << 20, 1 << 24, 1 << 26, 1 << 27, 1 << 12, 1 << 13, plan, plan_bytes, B, H,
                                   Hkv, tq, tk, d, scale, 1, dtype, None, None, None, None)

    assert fwd(q=0) == INV and fwd(plan=0) == INV
    assert fwd(plan_bytes=16) == INV              # shorter than the plan header
    assert fwd(B=0) == INV and fwd(tq=-1) == INV and fwd(H=3, Hkv=2) == INV
    assert fwd(d=96) == UNS and fwd(scale=0.0) == UNS
    assert fwd(tq=0) == binding.ATTN_OK           # no query rows: nothing to do


def test_split_heuristic_bounds(lib):
    # clamped to [1, ceil(Nk / 128)] (152 SMs when no device can be queried)
    for args in [(8, 32, 8, 1, 16384, 128), (4, 32, 8, 16, 8192, 128), (1, 1, 1, 1, 100, 64), (64, 64, 8, 1, 512, 128)]:
        s = binding.attn_splitkv_num_splits(*args)
        assert 1 <= s <= -(-args[4] // 128)
    assert binding.attn_splitkv_num_splits(0, 1, 1, 1, 1, 128) == 1
    # one wave on 152 SMs: 64 units (B8 x Hkv8, one query block each) -> 2 splits; 32 units -> 4;
    # more units than SMs -> no split; a single unit -> one split per key tile, up to 128
    assert binding.attn_splitkv_num_splits(8, 32, 8, 1, 16384, 128) == 2
    assert binding.attn_splitkv_num_splits(4, 32, 8, 16, 8192, 128) == 4
    assert binding.attn_splitkv_num_splits(64, 64, 8, 1, 512, 128) == 1
    assert binding.attn_splitkv_num_splits(1, 8, 1, 1, 16384, 128) == 128


def test_halved_tail_rule(lib):
    """Non-causal bf16 calls at d <= 128 with more than one wave that is not a whole number of
    waves deal the tiles after the last whole round but one in 152 equal shares of key tiles (at
    least 8 key tiles per tile), each share boundary inside a tile cutting that tile; otherwise a
    last wave filling at most half of the 152 SMs is halved when its tiles have at least 16 key
    tiles."""
    f = binding.attn_fwd_halved_tail_tiles
    # 512 tiles: whole rounds 0..303, then 208 tiles of 64 key tiles in 152 shares; the boundaries
    # floor(c W / 152) that are not multiples of 64
    assert f(1, 16, 8192, 128, False) == 144
    # d = 256 keeps the halved last wave: 512 tiles, three waves of 152, then 56
    assert f(2, 8, 4096, 256, False) == 56
    assert f(1, 16, 16384, 64, False) == 144    # 1024 tiles of 128 key tiles
    assert f(2, 32, 8192, 128, True) == 0       # causal: longest-first deal instead
    assert f(1, 19, 8192, 128, False) == 0      # 608 tiles: four whole waves
    assert f(1, 8, 2048, 128, False) == 64      # one wave of 64 tiles, halved
    assert f(1, 8, 1920, 128, False) == 0       # 15 key tiles: halves too short
    assert f(1, 2, 256, 64, False) == 0
    assert f(0, 8, 4096, 128, False) == 0
    assert f(1, 8, 4096, 96, False) == 0
    # the half-the-SMs boundary (d = 256: 128-row tiles): 4 heads x 19 blocks = 76 tiles are
    # halved, 4 x 20 = 80 are not; 16 key tiles is the shortest range that is halved
    assert f(1, 4, 2432, 256, False) == 76
    assert f(1, 4, 2560, 256, False) == 0
    assert f(1, 4, 2048, 256, False) == 64
    assert f(1, 4, 1920, 256, False) == 0
    # a second wave of exactly 76 tiles (152 + 76 = 228 = 12 heads x 19 blocks) is halved
    assert f(1, 12, 2432, 256, False) == 76
    # 156 tiles (39 heads x 4 blocks): 8 key tiles per tile is the shortest that is cut (shares of
    # 8.2 key tiles), 7 is not
    assert f(1, 39, 1024, 128, False) == 132
    assert f(1, 39, 896, 128, False) == 0


def test_tail_units(lib):
    """The cut tiles in the second launch's order: halved tiles all at the middle; shares: every
    unit in the tiles after the whole rounds, each tile once, longest second part first."""
    units = binding.attn_fwd_tail_units(1, 8, 2048, 128, False)
    assert units == [(t, 8) for t in range(64)]
    # e4m3 keeps the halved last wave: 512 tiles, the last 56 cut at key tile 32
    assert binding.attn_fwd_tail_units(1, 16, 8192, 128, False, fp8=True) == [(t, 32) for t in range(456, 512)]
    units = binding.attn_fwd_tail_units(1, 16, 8192, 128, False)   # 512 tiles, 64 key tiles
    assert len(units) == binding.attn_fwd_halved_tail_tiles(1, 16, 8192, 128, False) == 144
    tiles = [t for t, _ in units]
    kv0 = [j for _, j in units]
    assert len(set(tiles)) == len(tiles)
    assert all(304 <= t < 512 for t in tiles) and all(0 < j < 64 for j in kv0)
    assert kv0 == sorted(kv0)
    # each share of 13312 / 152 = 87.6 key tiles ends inside at most one tile, so a unit's
    # tile is the one its boundary falls in: boundary = (t - 304) * 64 + j
    bounds = sorted((t - 304) * 64 + j for t, j in units)
    assert bounds == [s for s in (c * 13312 // 152 for c in range(1, 152)) if s % 64]
    assert binding.attn_fwd_tail_units(2, 32, 8192, 128, True) == []