"""Sparse-graph attention for GB300 (sm_103a): thin ctypes binding over libsa.so.

Every function here only marshals arguments (torch tensors -> device pointers, the
current CUDA stream) and calls the C ABI declared in ``include/sa_api.h``; all the
work of the hot path runs in the library's CUDA kernels. There is no CPU fallback:
if the library is missing or the device is not an sm_103 GPU, calls raise.

Names follow the C ABI: ``sa_build_mask``, ``sa_attn_fwd``, ``sa_attn_fwd_heads``,
``sa_offset_attn_fwd``, ``sa_offset_attn_fwd_list``, ``sa_fib_offsets``, ``sa_pow2_offsets``, ``sa_layer_alpha``, ``sa_block_ratios``, ``sa_mask_nnz_bound``, ``sa_device_status``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB, build as build_library

MASK_TOPK, MASK_BIGBIRD, MASK_FULL, MASK_LITERAL_MEAN = 0, 1, 2, 3
LITERAL_LOCAL, LITERAL_PAIRS = 1, 2          # parts of the LITERAL_MEAN mask (0 = both)
_MODES = {"topk": MASK_TOPK, "bigbird": MASK_BIGBIRD, "full": MASK_FULL, "literal_mean": MASK_LITERAL_MEAN}

STATUS = {0: "SA_OK", -1: "SA_ERR_INVALID_ARG", -2: "SA_ERR_UNSUPPORTED", -3: "SA_ERR_CAPACITY",
          -4: "SA_ERR_CUDA", -5: "SA_ERR_TIMEOUT", -6: "SA_ERR_DEVICE"}


class SAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


class MaskParams(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("block", ctypes.c_int32), ("n_tokens", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("causal", ctypes.c_int32), ("window_blocks", ctypes.c_int32),
                ("global_blocks", ctypes.c_int32), ("topk", ctypes.c_int32), ("random_blocks", ctypes.c_int32),
                ("components", ctypes.c_int32), ("seed", ctypes.c_uint64)]


_lib = None
_I64x3 = ctypes.c_int64 * 3
_P = ctypes.c_void_p


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libsa.so (built in-tree by ``build_library``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with content_adaptive_sparse_gb300.build_library()")
    lib = ctypes.CDLL(path)
    lib.sa_version.restype = ctypes.c_int
    lib.sa_status_string.restype = ctypes.c_char_p
    lib.sa_status_string.argtypes = [ctypes.c_int]
    lib.sa_mask_nnz_bound.argtypes = [ctypes.POINTER(MaskParams), ctypes.POINTER(ctypes.c_int64)]
    lib.sa_build_mask.argtypes = [ctypes.POINTER(MaskParams), _P, _P, _P, ctypes.c_int64, _P]
    lib.sa_attn_fwd.argtypes = [_P, _P, _P, _I64x3, _I64x3, _I64x3, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                _P, _P, ctypes.c_int32, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
    lib.sa_attn_fwd_heads.argtypes = [_P, _P, _P, _I64x3, _I64x3, _I64x3, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, _P, _P, _P, ctypes.c_int32, ctypes.c_float,
                                      _P, _P, _P, ctypes.c_size_t, _P]
    lib.sa_attn_fwd_workspace_size.argtypes = [ctypes.c_int32] * 7 + [_P]
    lib.sa_attn_bwd_workspace_size.argtypes = [ctypes.c_int32] * 5 + [ctypes.c_int64, _P]
    lib.sa_attn_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _I64x3, _I64x3, _I64x3] + [ctypes.c_int32] * 7 + \
        [_P, _P, ctypes.c_int32, ctypes.c_float, _P, _P, _P, _P, ctypes.c_size_t, _P]
    lib.sa_attn_bwd_heads.argtypes = [_P, _P, _P, _P, _P, _P, _I64x3, _I64x3, _I64x3] + [ctypes.c_int32] * 8 + \
        [_P, _P, _P, _P, ctypes.c_int32, ctypes.c_float, _P, _P, _P, _P, ctypes.c_size_t, _P]
    lib.sa_attn_bwd_noalloc.argtypes = [_P, _P, _P, _P, _P, _P, _I64x3, _I64x3, _I64x3] + \
        [ctypes.c_int32] * 7 + [_P, _P, ctypes.c_int64, ctypes.c_int32, ctypes.c_float, _P, _P, _P, _P]
    lib.sa_offset_attn_fwd.argtypes = [_P, _P, _P, _I64x3, _I64x3, _I64x3] + [ctypes.c_int32] * 9 + \
        [ctypes.c_float, _P, _P, _P]
    lib.sa_offset_attn_fwd_list.argtypes = [_P, _P, _P, _I64x3, _I64x3, _I64x3, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P,
                                            ctypes.c_int32, ctypes.c_float, _P, _P, _P]
    lib.sa_offset_attn_interp_fwd.argtypes = [_P, _P, _P, _I64x3, _I64x3, _I64x3] + [ctypes.c_int32] * 6 + \
        [ctypes.c_double, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _P, _P, _P]
    lib.sa_fib_offsets.argtypes = [ctypes.c_int32] * 5 + [_P, ctypes.c_int32, _P]
    lib.sa_pow2_offsets.argtypes = [ctypes.c_int32] * 5 + [_P, ctypes.c_int32, _P]
    lib.sa_layer_alpha.argtypes = [ctypes.c_int32] * 7 + [_P, _P]
    lib.sa_block_ratios.argtypes = [_P, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _P,
                                    ctypes.c_int32]
    lib.sa_build_mask_from_bytes.argtypes = [ctypes.POINTER(MaskParams), _P, ctypes.c_int32, ctypes.c_int32, _P, _P,
                                             _P, _P, ctypes.c_int64, _P]
    lib.sa_device_status.argtypes = [_P]
    lib.sa_selftest_bounded_wait.argtypes = [_P]
    for name in ("sa_mask_nnz_bound", "sa_build_mask", "sa_attn_fwd", "sa_attn_fwd_heads", "sa_attn_fwd_workspace_size",
                 "sa_attn_bwd",
                 "sa_attn_bwd_noalloc", "sa_attn_bwd_heads", "sa_attn_bwd_workspace_size", "sa_offset_attn_fwd", "sa_offset_attn_fwd_list",
                 "sa_offset_attn_interp_fwd", "sa_fib_offsets", "sa_pow2_offsets", "sa_layer_alpha", "sa_block_ratios",
                 "sa_device_status", "sa_selftest_bounded_wait", "sa_build_mask_from_bytes"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(fn: str, code: int):
    if code != 0:
        raise SAError(fn, code)


def _stream_ptr(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _strides(t) -> _I64x3:
    st = t.stride()
    if t.dim() != 4 or st[3] != 1:
        raise ValueError("expected a [batch, tokens, heads, head_dim] tensor with contiguous head_dim")
    return _I64x3(st[0], st[1], st[2])


def mask_params(mode, block, n_tokens, batch, causal=1, window_blocks=0, global_blocks=0, topk=0,
                random_blocks=0, seed=0, components=0) -> MaskParams:
    return MaskParams(_MODES.get(mode, mode) if isinstance(mode, str) else mode, block, n_tokens, batch, causal,
                      window_blocks, global_blocks, topk, random_blocks, components, seed)


# ------------------------------------------------------------------ C ABI, same names

def sa_mask_nnz_bound(params: MaskParams) -> int:
    out = ctypes.c_int64(0)
    _check("sa_mask_nnz_bound", load_library().sa_mask_nnz_bound(ctypes.byref(params), ctypes.byref(out)))
    return int(out.value)


def sa_build_mask(params: MaskParams, ratio, row_ptr, col_idx, stream=None) -> None:
    """Writes ``row_ptr`` (int32 [batch, nb+1]) and ``col_idx`` (int32 [capacity]) on the GPU."""
    rp = 0 if ratio is None else ratio.data_ptr()
    _check("sa_build_mask", load_library().sa_build_mask(ctypes.byref(params), rp, row_ptr.data_ptr(),
                                                          col_idx.data_ptr(), col_idx.numel(), _stream_ptr(stream)))


def sa_attn_fwd_workspace_size(batch: int, n_tokens: int, heads: int, head_dim: int, block: int,
                               csr_batches: int, n_masks: int = 1) -> int:
    out = ctypes.c_size_t(0)
    _check("sa_attn_fwd_workspace_size", load_library().sa_attn_fwd_workspace_size(
        batch, n_tokens, heads, head_dim, block, csr_batches, n_masks, ctypes.byref(out)))
    return int(out.value)


def fwd_workspace(q, block: int, csr_shared: bool = False, n_masks: int = 1):
    """A device workspace of sa_attn_fwd_workspace_size bytes for q's shape (uint8 tensor)."""
    import torch
    b, n, h, d = q.shape
    nbytes = sa_attn_fwd_workspace_size(b, n, h, d, block, 1 if csr_shared else b, n_masks)
    return torch.empty((nbytes,), dtype=torch.uint8, device=q.device)


def sa_attn_fwd(q, k, v, row_ptr, col_idx, block: int, causal: int, o, lse, csr_shared: bool = False,
                softmax_scale: float | None = None, stream=None, workspace=None) -> None:
    """``workspace``: a uint8 device tensor (see fwd_workspace); one is allocated on the current
    stream when omitted."""
    b, n, h, d = q.shape
    hkv = k.shape[2]
    scale = 1.0 / float(np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    ws = fwd_workspace(q, block, csr_shared) if workspace is None else workspace
    _check("sa_attn_fwd", load_library().sa_attn_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides(q), _strides(k), _strides(o), b, n, h, hkv, d, block,
        int(causal), row_ptr.data_ptr(), col_idx.data_ptr(), int(bool(csr_shared)), scale, o.data_ptr(),
        lse.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(), _stream_ptr(stream)))


def sa_attn_fwd_heads(q, k, v, csrs, head_mask, block: int, causal: int, o, lse, csr_shared: bool = False,
                      softmax_scale: float | None = None, stream=None, workspace=None) -> None:
    """``csrs``: list of (row_ptr, col_idx) device tensors; query head h uses
    ``csrs[head_mask[h]]``."""
    b, n, h, d = q.shape
    hkv = k.shape[2]
    nm = len(csrs)
    rps = (ctypes.c_void_p * nm)(*[rp.data_ptr() for rp, _ in csrs])
    cis = (ctypes.c_void_p * nm)(*[ci.data_ptr() for _, ci in csrs])
    hm = np.ascontiguousarray(np.asarray(head_mask, dtype=np.int32))
    if hm.shape != (h,):
        raise ValueError("head_mask needs one CSR index per query head")
    scale = 1.0 / float(np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    ws = fwd_workspace(q, block, csr_shared, nm) if workspace is None else workspace
    _check("sa_attn_fwd_heads", load_library().sa_attn_fwd_heads(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides(q), _strides(k), _strides(o), b, n, h, hkv, d, block,
        int(causal), nm, ctypes.cast(rps, _P), ctypes.cast(cis, _P), hm.ctypes.data, int(bool(csr_shared)), scale,
        o.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(), _stream_ptr(stream)))


def sa_attn_bwd_workspace_size(batch: int, n_tokens: int, heads: int, block: int, csr_batches: int,
                               col_capacity: int) -> int:
    out = ctypes.c_size_t(0)
    _check("sa_attn_bwd_workspace_size", load_library().sa_attn_bwd_workspace_size(
        batch, n_tokens, heads, block, csr_batches, col_capacity, ctypes.byref(out)))
    return int(out.value)


def sa_attn_bwd(q, k, v, o, d_o, lse, row_ptr, col_idx, block: int, causal: int, dq, dk, dv, workspace,
                csr_shared: bool = False, softmax_scale: float | None = None, stream=None) -> None:
    b, n, h, d = q.shape
    hkv = k.shape[2]
    scale = 1.0 / float(np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    if _strides(d_o)[:] != _strides(o)[:] or _strides(dq)[:] != _strides(q)[:] or \
            _strides(dk)[:] != _strides(k)[:] or _strides(dv)[:] != _strides(v)[:]:
        raise ValueError("d_o / dq / dk / dv must have the strides of o / q / k / v")
    _check("sa_attn_bwd", load_library().sa_attn_bwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), d_o.data_ptr(), lse.data_ptr(), _strides(q),
        _strides(k), _strides(o), b, n, h, hkv, d, block, int(causal), row_ptr.data_ptr(), col_idx.data_ptr(),
        int(bool(csr_shared)), scale, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream_ptr(stream)))


def sa_attn_bwd_heads(q, k, v, o, d_o, lse, csrs, head_mask, block: int, causal: int, dq, dk, dv, workspace,
                      csr_shared: bool = False, softmax_scale: float | None = None, stream=None) -> None:
    """``csrs``: list of (row_ptr, col_idx) device tensors; query head h uses
    ``csrs[head_mask[h]]``; each col_idx's size is its capacity."""
    b, n, h, d = q.shape
    hkv = k.shape[2]
    nm = len(csrs)
    rps = (ctypes.c_void_p * nm)(*[rp.data_ptr() for rp, _ in csrs])
    cis = (ctypes.c_void_p * nm)(*[ci.data_ptr() for _, ci in csrs])
    caps = (ctypes.c_int64 * nm)(*[ci.numel() for _, ci in csrs])
    hm = np.ascontiguousarray(np.asarray(head_mask, dtype=np.int32))
    if hm.shape != (h,):
        raise ValueError("head_mask needs one CSR index per query head")
    scale = 1.0 / float(np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    _check("sa_attn_bwd_heads", load_library().sa_attn_bwd_heads(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), d_o.data_ptr(), lse.data_ptr(), _strides(q),
        _strides(k), _strides(o), b, n, h, hkv, d, block, int(causal), nm, ctypes.cast(rps, _P), ctypes.cast(cis, _P),
        ctypes.cast(caps, _P), hm.ctypes.data, int(bool(csr_shared)), scale, dq.data_ptr(), dk.data_ptr(),
        dv.data_ptr(), workspace.data_ptr(), workspace.numel() * workspace.element_size(), _stream_ptr(stream)))


def attn_bwd_heads(q, k, v, o, lse, d_o, csrs, head_mask, block: int, causal: int, csr_shared: bool = False,
                   softmax_scale: float | None = None):
    """Allocate dq / dk / dv and the workspace, run the head-group backward."""
    import torch
    b, n, h, d = q.shape
    cap = sum(ci.numel() for _, ci in csrs)
    ws_bytes = sa_attn_bwd_workspace_size(b, n, h, block, (1 if csr_shared else b) * len(csrs), cap)
    ws = torch.empty((ws_bytes,), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sa_attn_bwd_heads(q, k, v, o, d_o, lse, csrs, head_mask, block, causal, dq, dk, dv, ws, csr_shared,
                      softmax_scale)
    return dq, dk, dv


def sa_attn_bwd_noalloc(q, k, v, o, d_o, lse, row_ptr, col_idx, block: int, causal: int, dq, dk, dv,
                        csr_shared: bool = False, softmax_scale: float | None = None, stream=None,
                        col_capacity: int | None = None) -> None:
    """sa_attn_bwd for callers that cannot allocate: the scratch is the library's own
    (no workspace argument). ``col_capacity`` defaults to the size of ``col_idx``."""
    b, n, h, d = q.shape
    hkv = k.shape[2]
    scale = 1.0 / float(np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    cap = col_idx.numel() if col_capacity is None else int(col_capacity)
    _check("sa_attn_bwd_noalloc", load_library().sa_attn_bwd_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), d_o.data_ptr(), lse.data_ptr(), _strides(q),
        _strides(k), _strides(o), b, n, h, hkv, d, block, int(causal), row_ptr.data_ptr(), col_idx.data_ptr(),
        cap, int(bool(csr_shared)), scale, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), _stream_ptr(stream)))


def sa_offset_attn_fwd(q, k, v, window: int, alpha_num: int, alpha_den: int, n_rungs: int, o, lse,
                       softmax_scale: float | None = None, stream=None) -> None:
    """Window plus the Fibonacci offsets round_half_even(alpha * f_k), alpha = num / den."""
    b, n, h, d = q.shape
    hkv = k.shape[2]
    scale = 1.0 / float(np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    _check("sa_offset_attn_fwd", load_library().sa_offset_attn_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides(q), _strides(k), _strides(o), b, n, h, hkv, d, window,
        int(alpha_num), int(alpha_den), int(n_rungs), scale, o.data_ptr(), lse.data_ptr(), _stream_ptr(stream)))


def sa_offset_attn_fwd_list(q, k, v, window: int, offsets, o, lse, softmax_scale: float | None = None,
                            stream=None) -> None:
    b, n, h, d = q.shape
    hkv = k.shape[2]
    offs = np.ascontiguousarray(np.asarray(offsets, dtype=np.int32))
    scale = 1.0 / float(np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    _check("sa_offset_attn_fwd_list", load_library().sa_offset_attn_fwd_list(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides(q), _strides(k), _strides(o), b, n, h, hkv, d, window,
        offs.ctypes.data if offs.size else None, int(offs.size), scale, o.data_ptr(), lse.data_ptr(),
        _stream_ptr(stream)))


def _ladder(fn: str, alpha_num: int, alpha_den: int, n_rungs: int, window: int, n_tokens: int) -> list[int]:
    buf = (ctypes.c_int32 * 128)()
    cnt = ctypes.c_int32(0)
    _check(fn, getattr(load_library(), fn)(alpha_num, alpha_den, n_rungs, window, n_tokens, ctypes.cast(buf, _P), 128,
                                           ctypes.byref(cnt)))
    return [int(buf[i]) for i in range(cnt.value)]


def sa_offset_attn_interp_fwd(q, k, v, window: int, alpha: float, o, lse, n_rungs: int = 15, ladder: int = 0,
                              softmax_scale: float | None = None, stream=None) -> None:
    b, n, h, d = q.shape
    hkv = k.shape[2]
    scale = 1.0 / float(np.sqrt(d)) if softmax_scale is None else float(softmax_scale)
    _check("sa_offset_attn_interp_fwd", load_library().sa_offset_attn_interp_fwd(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), _strides(q), _strides(k), _strides(o), b, n, h, hkv, d, window,
        float(alpha), n_rungs, ladder, scale, o.data_ptr(), lse.data_ptr(), _stream_ptr(stream)))


def offset_attn_interp_fwd(q, k, v, window: int, alpha: float, n_rungs: int = 15, ladder: int = 0,
                           softmax_scale: float | None = None):
    import torch
    b, n, h, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    sa_offset_attn_interp_fwd(q, k, v, window, alpha, o, lse, n_rungs, ladder, softmax_scale)
    return o, lse


def sa_fib_offsets(alpha_num: int, alpha_den: int, n_rungs: int, window: int, n_tokens: int) -> list[int]:
    return _ladder("sa_fib_offsets", alpha_num, alpha_den, n_rungs, window, n_tokens)


def sa_pow2_offsets(alpha_num: int, alpha_den: int, n_rungs: int, window: int, n_tokens: int) -> list[int]:
    return _ladder("sa_pow2_offsets", alpha_num, alpha_den, n_rungs, window, n_tokens)


def sa_layer_alpha(layer: int, layers: int, lo=(1, 2), hi=(3, 2), stride: int = 1) -> tuple[int, int]:
    """(numerator, denominator) of the layer's alpha (linear ramp, coprime ``stride``)."""
    num, den = ctypes.c_int32(0), ctypes.c_int32(0)
    _check("sa_layer_alpha", load_library().sa_layer_alpha(layer, layers, lo[0], lo[1], hi[0], hi[1], stride,
                                                            ctypes.byref(num), ctypes.byref(den)))
    return int(num.value), int(den.value)


def sa_block_ratios(data: np.ndarray, block: int, level: int = 6, n_threads: int = 0) -> np.ndarray:
    """Host zlib ratios of ``uint8 [batch, n_tokens]``; returns float32 [batch, nb]."""
    arr = np.ascontiguousarray(np.asarray(data, dtype=np.uint8))
    if arr.ndim == 1:
        arr = arr[None, :]
    out = np.empty((arr.shape[0], arr.shape[1] // block), dtype=np.float32)
    _check("sa_block_ratios", load_library().sa_block_ratios(arr.ctypes.data, arr.shape[0], arr.shape[1], block,
                                                              level, out.ctypes.data, n_threads))
    return out


def sa_build_mask_from_bytes(params: MaskParams, data, h_ratio, d_ratio, row_ptr, col_idx, level: int = 6,
                             n_threads: int = 0, stream=None) -> None:
    """Host ratios of ``data`` (uint8 [batch, n_tokens], host) into ``h_ratio`` (float32 host
    tensor, pinned for an asynchronous upload), then their upload into ``d_ratio`` and the
    mask build, enqueued on the stream."""
    arr = np.ascontiguousarray(np.asarray(data, dtype=np.uint8))
    _check("sa_build_mask_from_bytes", load_library().sa_build_mask_from_bytes(
        ctypes.byref(params), arr.ctypes.data, level, n_threads, h_ratio.data_ptr(), d_ratio.data_ptr(),
        row_ptr.data_ptr(), col_idx.data_ptr(), col_idx.numel(), _stream_ptr(stream)))


def sa_selftest_bounded_wait(stream=None) -> None:
    """Launch the failure-path self-test (a wait that times out after 1 s)."""
    _check("sa_selftest_bounded_wait", load_library().sa_selftest_bounded_wait(_stream_ptr(stream)))


def sa_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status code."""
    return int(load_library().sa_device_status(_stream_ptr(stream)))


# ------------------------------------------------------------------ conveniences (allocation + one call)

def build_mask(params: MaskParams, ratio=None, device="cuda"):
    """Allocate CSR buffers of the exact size bound and build the mask."""
    import torch
    nb = params.n_tokens // params.block
    cap = sa_mask_nnz_bound(params)
    row_ptr = torch.empty((params.batch, nb + 1), dtype=torch.int32, device=device)
    col_idx = torch.empty((max(cap, 1),), dtype=torch.int32, device=device)
    sa_build_mask(params, ratio, row_ptr, col_idx)
    return row_ptr, col_idx


def attn_fwd(q, k, v, row_ptr, col_idx, block: int, causal: int, csr_shared: bool = False,
             softmax_scale: float | None = None):
    import torch
    b, n, h, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    sa_attn_fwd(q, k, v, row_ptr, col_idx, block, causal, o, lse, csr_shared, softmax_scale)
    return o, lse


def attn_fwd_heads(q, k, v, csrs, head_mask, block: int, causal: int, csr_shared: bool = False,
                   softmax_scale: float | None = None):
    import torch
    b, n, h, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    sa_attn_fwd_heads(q, k, v, csrs, head_mask, block, causal, o, lse, csr_shared, softmax_scale)
    return o, lse


def attn_bwd(q, k, v, o, lse, d_o, row_ptr, col_idx, block: int, causal: int, csr_shared: bool = False,
             softmax_scale: float | None = None):
    """Allocate dq / dk / dv and the workspace, run the backward; returns (dq, dk, dv)."""
    import torch
    b, n, h, d = q.shape
    ws_bytes = sa_attn_bwd_workspace_size(b, n, h, block, 1 if csr_shared else b, col_idx.numel())
    ws = torch.empty((ws_bytes,), dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    sa_attn_bwd(q, k, v, o, d_o, lse, row_ptr, col_idx, block, causal, dq, dk, dv, ws, csr_shared, softmax_scale)
    return dq, dk, dv


def offset_attn_fwd(q, k, v, window: int, offsets, softmax_scale: float | None = None):
    import torch
    b, n, h, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    sa_offset_attn_fwd_list(q, k, v, window, offsets, o, lse, softmax_scale)
    return o, lse


def fib_offset_attn_fwd(q, k, v, window: int, alpha_num: int, alpha_den: int, n_rungs: int = 15,
                        softmax_scale: float | None = None):
    """Allocate O / LSE and run sa_offset_attn_fwd (Fibonacci offsets of alpha = num / den)."""
    import torch
    b, n, h, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    sa_offset_attn_fwd(q, k, v, window, alpha_num, alpha_den, n_rungs, o, lse, softmax_scale)
    return o, lse


__all__ = [
    "build_library", "load_library", "SAError", "MaskParams", "mask_params",
    # C ABI
    "sa_mask_nnz_bound", "sa_build_mask", "sa_attn_fwd", "sa_attn_fwd_heads", "sa_attn_bwd",
    "sa_attn_bwd_workspace_size", "sa_attn_bwd_noalloc", "sa_attn_bwd_heads", "sa_offset_attn_fwd", "sa_offset_attn_interp_fwd",
    "sa_fib_offsets", "sa_pow2_offsets", "sa_layer_alpha", "sa_block_ratios", "sa_device_status",
    "sa_selftest_bounded_wait",
    # allocating conveniences
    "build_mask", "attn_fwd", "attn_fwd_heads", "attn_bwd", "attn_bwd_heads", "offset_attn_fwd", "offset_attn_interp_fwd",
    # constants
    "MASK_TOPK", "MASK_BIGBIRD", "MASK_FULL", "MASK_LITERAL_MEAN", "LITERAL_LOCAL", "LITERAL_PAIRS",
]
