"""ctypes binding of libattn_gb300.so (argument marshalling only; all compute runs in the library).

The Python names mirror the C ABI in include/attn.h. ``attn_fwd`` takes torch CUDA tensors
(PyTorch is used for device memory and streams only) and raises ``AttnError`` on any non-OK
status. There is no fallback: if the library is missing the call fails.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

from . import build as _build

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_CUDA, ATTN_ERR_TIMEOUT = range(5)
ATTN_DTYPE_BF16, ATTN_DTYPE_FP8_E4M3 = 0, 1
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
                4: "ATTN_ERR_TIMEOUT"}

_LIB = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


def lib_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """Loads the library (it must have been built: ``exact_attention_72_gb300.build.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{os.path.basename(path)} is not built; call exact_attention_72_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.restype = i
    L.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, vp, vp, vp]
    L.attn_fwd_fp8_scaled.restype = i
    L.attn_fwd_fp8_scaled.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, i, vp, vp, i, i, vp]
    L.attn_fwd_fp8_blockscaled.restype = i
    L.attn_fwd_fp8_blockscaled.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, vp]
    L.attn_quantize_e4m3.restype = i
    L.attn_quantize_e4m3.argtypes = [vp, vp, vp, i, i, i, i, i, vp, vp]
    L.attn_quantize_e4m3_descale_count.restype = sz
    L.attn_quantize_e4m3_descale_count.argtypes = [i, i, i, i]
    L.attn_varlen_plan_bytes.restype = sz
    L.attn_varlen_plan_bytes.argtypes = [i, i, i, i]
    L.attn_varlen_plan.restype = i
    L.attn_varlen_plan.argtypes = [vp, vp, i, i, i, i, i, i, vp, sz, vp]
    L.attn_fwd_varlen.restype = i
    L.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, i, i, vp, vp, vp, vp]
    L.attn_bwd_workspace_bytes.restype = sz
    L.attn_bwd_workspace_bytes.argtypes = [i, i, i]
    L.attn_bwd.restype = i
    L.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, sz, vp]
    L.attn_splitkv_num_splits.restype = i
    L.attn_splitkv_num_splits.argtypes = [i, i, i, i, i, i]
    L.attn_fwd_halved_tail_tiles.restype = i
    L.attn_fwd_halved_tail_tiles.argtypes = [i, i, i, i, i]
    L.attn_fwd_tail_units.restype = i
    L.attn_fwd_tail_units.argtypes = [i, i, i, i, i, i, vp, vp, i]
    L.attn_fwd_host.restype = i
    L.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, vp, vp, vp, sz, vp]
    L.attn_fwd_splitkv.restype = i
    L.attn_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, vp, vp, vp, sz, vp]
    L.attn_fwd_splitkv_static.restype = i
    L.attn_fwd_splitkv_static.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, vp, vp, vp]
    L.attn_fwd_splitkv_workspace_bytes.restype = sz
    L.attn_fwd_splitkv_workspace_bytes.argtypes = [i, i, i, i, i]
    L.attn_fwd_host_workspace_bytes.restype = sz
    L.attn_fwd_host_workspace_bytes.argtypes = [i, i, i, i, i, i]
    L.attn_get_status.restype = i
    L.attn_get_status.argtypes = [vp]
    L.attn_get_status_detail.restype = i
    L.attn_get_status_detail.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    L.attn_clear_status.restype = i
    L.attn_clear_status.argtypes = []
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_status_string.argtypes = [i]
    L.attn_debug_set.restype = None
    L.attn_debug_set.argtypes = [ctypes.c_ulonglong, i]
    L.attn_version.restype = i
    L.attn_version.argtypes = []
    _LIB = L
    return L


def _check(status: int, what: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, what)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return ATTN_DTYPE_BF16
    if t.dtype == torch.float8_e4m3fn:
        return ATTN_DTYPE_FP8_E4M3
    raise TypeError(f"q/k/v must be bfloat16 or float8_e4m3fn, got {t.dtype}")


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def attn_fwd(q, k, v, causal: bool, scale: Optional[float] = None, descale_q=None, descale_k=None,
             descale_v=None, out=None, lse=None, stream=None):
    """O, LSE = attention forward of q [B,N,H,d], k/v [B,N,Hkv,d] (CUDA tensors, bf16 or e4m3).

    ``descale_*`` (fp8 only) are one-element float32 CUDA tensors. ``out`` (bf16 [B,N,H,d]) and
    ``lse`` (float32 [B,H,N]) are allocated if not given. Returns (out, lse).
    """
    import torch
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must be [B, N, Hkv, d] with q's dtype")
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    ptrs = [0, 0, 0]
    if code == ATTN_DTYPE_FP8_E4M3:
        for idx, t in enumerate((descale_q, descale_k, descale_v)):
            if t is None or t.dtype != torch.float32 or not t.is_cuda:
                raise ValueError("fp8 needs descale_q/k/v as float32 CUDA tensors")
            ptrs[idx] = t.data_ptr()
    st = lib().attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Hkv, N, d,
                        float(scale), int(bool(causal)), code, ptrs[0], ptrs[1], ptrs[2], _stream_handle(stream))
    _check(st, "attn_fwd")
    return out, lse


def attn_fwd_fp8_scaled(q, k, v, causal: bool, descale_q, descale_k, descale_v, scale: Optional[float] = None,
                        out=None, lse=None, stream=None):
    """attn_fwd for e4m3 q/k/v with descale factors per (batch, head).

    ``descale_q`` is a float32 CUDA tensor of shape [B, H] (or any shape broadcastable to it by
    strides, e.g. [1, H] expanded); ``descale_k`` and ``descale_v`` are [B, Hkv] with the SAME
    strides as each other. Strides are taken from the tensors (a stride of 0 repeats a value).
    """
    import torch
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float8_e4m3fn:
            raise ValueError(f"{name} must be a contiguous float8_e4m3fn CUDA tensor")
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, N, Hkv, d]")
    dq = descale_q.expand(B, H)
    dk = descale_k.expand(B, Hkv)
    dv = descale_v.expand(B, Hkv)
    for name, t in (("descale_q", dq), ("descale_k", dk), ("descale_v", dv)):
        if t.dtype != torch.float32 or not t.is_cuda:
            raise ValueError(f"{name} must be a float32 CUDA tensor")
    if dk.stride() != dv.stride():
        raise ValueError("descale_k and descale_v must share strides")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = lib().attn_fwd_fp8_scaled(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H,
                                   Hkv, N, d, float(scale), int(bool(causal)), dq.data_ptr(), dq.stride(0),
                                   dq.stride(1), dk.data_ptr(), dv.data_ptr(), dk.stride(0), dk.stride(1),
                                   _stream_handle(stream))
    _check(st, "attn_fwd_fp8_scaled")
    return out, lse


def attn_varlen_plan_bytes(B: int, H: int, total_q: int, d: int) -> int:
    return int(lib().attn_varlen_plan_bytes(B, H, total_q, d))


def _check_offsets(name, cu):
    import torch
    if not cu.is_cuda or cu.dtype != torch.int32 or cu.dim() != 1 or not cu.is_contiguous() or cu.numel() < 2:
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor of B + 1 offsets")


def attn_varlen_plan(cu_seqlens_q, cu_seqlens_k, H: int, total_q: int, total_k: int, d: int, causal: bool,
                     plan=None, stream=None):
    """Work-tile plan of a ragged batch (uint8 CUDA tensor), reusable across forward calls."""
    import torch
    _check_offsets("cu_seqlens_q", cu_seqlens_q)
    _check_offsets("cu_seqlens_k", cu_seqlens_k)
    B = cu_seqlens_q.numel() - 1
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    need = attn_varlen_plan_bytes(B, H, total_q, d)
    if plan is None:
        plan = torch.empty(max(need, 16), dtype=torch.uint8, device=cu_seqlens_q.device)
    st = lib().attn_varlen_plan(cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), B, H, total_q, total_k, d,
                                int(bool(causal)), plan.data_ptr(), plan.numel() * plan.element_size(),
                                _stream_handle(stream))
    _check(st, "attn_varlen_plan")
    return plan


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, plan, causal: bool, scale: Optional[float] = None,
                    descale_q=None, descale_k=None, descale_v=None, out=None, lse=None, stream=None):
    """Ragged-batch forward: q [total_q, H, d], k/v [total_k, Hkv, d] packed along rows.

    Returns (out bf16 [total_q, H, d], lse float32 [H, total_q]). ``plan`` comes from
    attn_varlen_plan with the same offsets, H, d, causal and totals.
    """
    import torch
    total_q, H, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError(f"{name} must be a contiguous 3-D CUDA tensor")
    if k.shape != (total_k, Hkv, d) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must be [total_k, Hkv, d] with q's dtype")
    _check_offsets("cu_seqlens_q", cu_seqlens_q)
    _check_offsets("cu_seqlens_k", cu_seqlens_k)
    B = cu_seqlens_q.numel() - 1
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((total_q, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    ptrs = [0, 0, 0]
    if code == ATTN_DTYPE_FP8_E4M3:
        for idx, t in enumerate((descale_q, descale_k, descale_v)):
            if t is None or t.dtype != torch.float32 or not t.is_cuda:
                raise ValueError("fp8 needs descale_q/k/v as float32 CUDA tensors")
            ptrs[idx] = t.data_ptr()
    st = lib().attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(), plan.data_ptr(),
                               plan.numel() * plan.element_size(), B, H, Hkv,
                               total_q, total_k, d, float(scale), int(bool(causal)), code, ptrs[0] or None,
                               ptrs[1] or None, ptrs[2] or None, _stream_handle(stream))
    _check(st, "attn_fwd_varlen")
    return out, lse


def attn_bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(lib().attn_bwd_workspace_bytes(B, H, N))


def attn_bwd(q, k, v, o, lse, dout, causal: bool, scale: Optional[float] = None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd for bf16 q/o/dout [B,N,H,d], k/v [B,N,Hkv,d], lse [B,H,N]."""
    import torch
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape or o.shape != q.shape or dout.shape != q.shape:
        raise ValueError("shapes: q, o, dout [B, N, H, d]; k, v [B, N, Hkv, d]")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 CUDA tensor [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = attn_bwd_workspace_bytes(B, H, N)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Hkv, N, d, float(scale),
                        int(bool(causal)), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        _stream_handle(stream))
    _check(st, "attn_bwd")
    return dq, dk, dv


ATTN_FP8_Q_BLOCK = 128   # query rows per q descale block (attn_fwd_fp8_blockscaled)
ATTN_FP8_K_BLOCK = 64    # keys per k descale block


def attn_fwd_fp8_blockscaled(q, k, v, causal: bool, descale_q, descale_k, descale_v, scale: Optional[float] = None,
                             out=None, lse=None, stream=None):
    """attn_fwd for e4m3 q/k/v with block descales: descale_q [B, H, ceil(N/128)], descale_k
    [B, Hkv, ceil(N/64)], descale_v [B, Hkv] (contiguous float32 CUDA tensors)."""
    import torch
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.float8_e4m3fn:
            raise ValueError(f"{name} must be a contiguous float8_e4m3fn CUDA tensor")
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be [B, N, Hkv, d]")
    want = {"descale_q": (B, H, -(-N // ATTN_FP8_Q_BLOCK)), "descale_k": (B, Hkv, -(-N // ATTN_FP8_K_BLOCK)),
            "descale_v": (B, Hkv)}
    for (name, shape), t in zip(want.items(), (descale_q, descale_k, descale_v)):
        if tuple(t.shape) != shape or t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of shape {shape}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = lib().attn_fwd_fp8_blockscaled(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B,
                                        H, Hkv, N, d, float(scale), int(bool(causal)), descale_q.data_ptr(),
                                        descale_k.data_ptr(), descale_v.data_ptr(), _stream_handle(stream))
    _check(st, "attn_fwd_fp8_blockscaled")
    return out, lse


def quantize_e4m3(x, block_rows: int, signs=None, out=None, descale=None, stream=None):
    """e4m3 codes of bf16 x [B, N, Hx, d] with a descale per block of ``block_rows`` rows of one
    (batch, head), optionally after the rotation diag(signs) H_d / sqrt(d). Returns (x8, descale)
    with descale float32 [B, Hx, ceil(N / block_rows)]."""
    import torch
    if not x.is_cuda or not x.is_contiguous() or x.dtype != torch.bfloat16 or x.dim() != 4:
        raise ValueError("x must be a contiguous bfloat16 CUDA tensor [B, N, Hx, d]")
    B, N, Hx, d = x.shape
    nblk = -(-N // block_rows) if block_rows > 0 else 0
    if out is None:
        out = torch.empty((B, N, Hx, d), dtype=torch.float8_e4m3fn, device=x.device)
    if descale is None:
        descale = torch.empty((B, Hx, nblk), dtype=torch.float32, device=x.device)
    sp = 0
    if signs is not None:
        if not signs.is_cuda or signs.dtype != torch.float32 or signs.numel() != d or not signs.is_contiguous():
            raise ValueError("signs must be a contiguous float32 CUDA tensor of d values")
        sp = signs.data_ptr()
    st = lib().attn_quantize_e4m3(x.data_ptr(), out.data_ptr(), descale.data_ptr(), B, N, Hx, d, int(block_rows),
                                  sp or None, _stream_handle(stream))
    _check(st, "attn_quantize_e4m3")
    return out, descale


def attn_quantize_e4m3_descale_count(B: int, N: int, Hx: int, block_rows: int) -> int:
    return int(lib().attn_quantize_e4m3_descale_count(B, N, Hx, block_rows))


def attn_fwd_halved_tail_tiles(B: int, H: int, N: int, d: int, causal: bool) -> int:
    """Work tiles of an attn_fwd call whose key range the library cuts across two launches."""
    return int(lib().attn_fwd_halved_tail_tiles(B, H, N, d, int(bool(causal))))


def attn_fwd_tail_units(B: int, H: int, N: int, d: int, causal: bool, fp8: bool = False):
    """The cut tiles of an attn_fwd call (bf16, or e4m3 with fp8 set), in the second launch's
    order: [(work tile, first key tile of the second part), ...]."""
    code = ATTN_DTYPE_FP8_E4M3 if fp8 else ATTN_DTYPE_BF16
    n = int(lib().attn_fwd_tail_units(B, H, N, d, int(bool(causal)), code, None, None, 0))
    if n == 0:
        return []
    t = (ctypes.c_int * n)()
    k = (ctypes.c_int * n)()
    got = lib().attn_fwd_tail_units(B, H, N, d, int(bool(causal)), code, t, k, n)
    assert got == n
    return list(zip(t, k))


def attn_splitkv_num_splits(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    """The library's split count for a decode shape on the current device (about one wave)."""
    return int(lib().attn_splitkv_num_splits(B, H, Hkv, Nq, Nk, d))


def attn_fwd_splitkv(q, k, v, num_splits: int, scale: Optional[float] = None, descale_q=None, descale_k=None,
                     descale_v=None, workspace=None, out=None, lse=None, stream=None):
    """Split-KV decode forward: q [B,Nq,H,d] attends to all keys of k/v [B,Nk,Hkv,d] (no mask).

    ``workspace`` (CUDA uint8, at least attn_fwd_splitkv_workspace_bytes(...) bytes) is allocated
    here with torch if not given. Returns (out [B,Nq,H,d] bf16, lse [B,H,Nq] fp32).
    """
    import torch
    B, Nq, H, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if k.shape != (B, Nk, Hkv, d) or v.shape != k.shape or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must be [B, Nk, Hkv, d] with q's dtype")
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty((B, Nq, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ptrs = [0, 0, 0]
    if code == ATTN_DTYPE_FP8_E4M3:
        for idx, t in enumerate((descale_q, descale_k, descale_v)):
            if t is None or t.dtype != torch.float32 or not t.is_cuda:
                raise ValueError("fp8 needs descale_q/k/v as float32 CUDA tensors")
            ptrs[idx] = t.data_ptr()
    st = lib().attn_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Hkv,
                                Nq, Nk, d, float(scale), int(num_splits), code, ptrs[0], ptrs[1], ptrs[2],
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                _stream_handle(stream))
    _check(st, "attn_fwd_splitkv")
    return out, lse


def attn_fwd_splitkv_static(q, k, v, num_splits: int, scale: Optional[float] = None, out=None, lse=None,
                            stream=None):
    """attn_fwd_splitkv without a workspace: the library's fixed 16 MiB device scratch holds the
    partial results (for callers that cannot allocate device memory). bf16 inputs; calls that
    overlap on the GPU share that scratch and must be serialized."""
    import torch
    B, Nq, H, d = q.shape
    Nk, Hkv = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Nq, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    st = lib().attn_fwd_splitkv_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B,
                                       H, Hkv, Nq, Nk, d, float(scale), int(num_splits), _dtype_code(q), None, None,
                                       None, _stream_handle(stream))
    _check(st, "attn_fwd_splitkv_static")
    return out, lse


def attn_fwd_splitkv_workspace_bytes(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    return int(lib().attn_fwd_splitkv_workspace_bytes(B, H, Nq, d, num_splits))


def attn_fwd_host(q, k, v, out, lse, causal: bool, workspace, scale: Optional[float] = None,
                  descale_q: float = 1.0, descale_k: float = 1.0, descale_v: float = 1.0, stream=None):
    """The same forward on HOST (CPU, ideally pinned) tensors through attn_fwd_host.

    ``workspace`` is a CUDA uint8 tensor of at least attn_fwd_host_workspace_bytes(...) bytes.
    The call returns once o and lse are back in host memory.
    """
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    code = _dtype_code(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    for t in (q, k, v, out, lse):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("attn_fwd_host takes contiguous host tensors")
    dq, dk, dv = (ctypes.c_float(descale_q), ctypes.c_float(descale_k), ctypes.c_float(descale_v))
    fp8 = code == ATTN_DTYPE_FP8_E4M3
    st = lib().attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, Hkv, N,
                             d, float(scale), int(bool(causal)), code,
                             ctypes.addressof(dq) if fp8 else None, ctypes.addressof(dk) if fp8 else None,
                             ctypes.addressof(dv) if fp8 else None, workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, "attn_fwd_host")
    return out, lse


def attn_fwd_host_workspace_bytes(B: int, H: int, Hkv: int, N: int, d: int, dtype_code: int) -> int:
    return int(lib().attn_fwd_host_workspace_bytes(B, H, Hkv, N, d, dtype_code))


def attn_get_status(stream=None) -> tuple[int, int]:
    """(status, raw status word) after synchronizing ``stream`` (C: attn_get_status_detail)."""
    detail = ctypes.c_uint32(0)
    st = lib().attn_get_status_detail(_stream_handle(stream), ctypes.byref(detail))
    return st, detail.value


def attn_clear_status() -> None:
    _check(lib().attn_clear_status(), "attn_clear_status")


def attn_status_string(status: int) -> str:
    return lib().attn_status_string(status).decode()


def attn_debug_set(timeout_ns: int = 0, skip_load: bool = False) -> None:
    lib().attn_debug_set(int(timeout_ns), int(bool(skip_load)))


def attn_version() -> int:
    return int(lib().attn_version())
