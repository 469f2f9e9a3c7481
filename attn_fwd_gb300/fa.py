"""Thin Python binding of libfa.so (the C ABI in include/fa.h).

Functions named like the C entry points take PyTorch CUDA tensors and
marshal pointers, sizes and the current stream; every step of the attention
path runs in the library's kernels.  ``forward`` and ``backward`` are small
conveniences that allocate the outputs and the workspace.  If the library is
missing or fails to load, every call raises: there is no fallback.
"""
from __future__ import annotations

import ctypes
import functools
import os
import threading

import torch

from . import build as _build

FA_OK = 0
FA_ERR_INVALID = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_ARCH = -3
FA_ERR_LAUNCH = -4
FA_ERR_TIMEOUT = -5
FA_ERR_CUDA = -6
FA_ERR_SCRATCH = -7

MASK_NONE, MASK_CAUSAL, MASK_BLOCK, MASK_BLOCK_CAUSAL = 0, 1, 2, 3

_lib = None
_lock = threading.Lock()

_vp, _i, _f, _sz, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint64
_SIGS = {
    "fa_version": (_i, []),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_fwd_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp] * 10 + [_i, _i, _i, _i, _f, _i, _vp]),
    "fa_bwd_blocksparse": (_i, [_vp] * 11 + [_i, _i, _i, _i, _f, _i, _vp]),
    "fa_bwd_preprocess": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "fa_bwd_main": (_i, [_vp] * 8 + [_i, _i, _i, _i, _f, _i, _f, _u64, _vp]),
    "fa_fwd_dropout": (_i, [_vp] * 6 + [_i, _i, _i, _i, _f, _i, _f, _u64, _vp]),
    "fa_dropout_effective_p": (_f, [_f]),
    "fa_bwd_dropout": (_i, [_vp] * 11 + [_i, _i, _i, _i, _f, _i, _f, _u64, _vp]),
    "fa_bwd_dq_convert": (_i, [_vp, _vp, _i, _i, _i, _i, _f, _vp]),
    "fa_bwd_noalloc": (_i, [_vp] * 9 + [_i, _i, _i, _i, _f, _i, _vp]),
    "fa_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "fa_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "fa_fwd_fp8_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fa_fwd_fp8": (_i, [_vp] * 8 + [_i, _i, _i, _i, _f, _i, _vp, _vp]),
    "fa_block_mask_window": (_i, [_vp, _i, _i, _i]),
    "fa_block_mask_dilated": (_i, [_vp, _i, _i, _i, _i]),
    "fa_get_device_error": (_i, [_vp]),
    "fa_set_wait_timeout_ns": (_i, [_u64]),
    "fa_debug_wait_timeout": (_i, [_u64, _vp]),
    "fa_fwd_bwd_host_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fa_fwd_bwd_host": (_i, [_vp] * 11 + [_sz, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_fwd_host_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fa_fwd_host": (_i, [_vp] * 7 + [_sz, _i, _i, _i, _i, _f, _i, _vp]),
}


class FAError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} returned {code}: {status_string(code) if _lib else code}")


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libfa.so (once).  Raises if it is absent: build it with
    ``__graft_entry__.build()``."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or _build.LIB
            if not os.path.exists(p):
                raise RuntimeError(f"libfa.so not found at {p}; run __graft_entry__.build() first")
            lib = ctypes.CDLL(p)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().fa_status_string(code).decode()


def _check(fn: str, rc: int):
    if rc != FA_OK:
        raise FAError(fn, rc)


def _on_device(pick):
    """Run the wrapped entry point with the device of its tensors current: the
    library launches on the current device (its status word, its SM count,
    the scratch array of fa_bwd_noalloc) and the default stream is that
    device's current stream.  `pick` chooses the tensor from the arguments."""
    def wrap(fn):
        @functools.wraps(fn)
        def run(*args, **kwargs):
            t = pick(*args, **kwargs)
            if isinstance(t, torch.Tensor) and t.is_cuda:
                with torch.cuda.device(t.device):
                    return fn(*args, **kwargs)
            return fn(*args, **kwargs)
        return run
    return wrap


_first = _on_device(lambda *a, **k: a[0] if a else None)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _bf16(t: torch.Tensor, name: str):
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous() and t.dim() == 4):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor [B, H, N, d]")
    return ctypes.c_void_p(t.data_ptr())


def _f32(t: torch.Tensor, name: str):
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _mask_ptr(block_mask):
    if block_mask is None:
        return ctypes.c_void_p(0)
    if not (block_mask.is_cuda and block_mask.dtype == torch.uint8 and block_mask.is_contiguous()):
        raise ValueError("block_mask must be a contiguous uint8 CUDA tensor [N/128, N/128]")
    return ctypes.c_void_p(block_mask.data_ptr())


def _ptr_or_null(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


# --------------------------------------------------------------------------- #
# C entry points (same names)
# --------------------------------------------------------------------------- #
def fa_version() -> int:
    return load().fa_version()


@_first
def fa_fwd(q, k, v, o, lse, scale, causal=False, stream=None):
    B, H, N, d = q.shape
    rc = load().fa_fwd(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _f32(lse, "lse"),
                       B, H, N, d, float(scale), int(bool(causal)), _stream(stream))
    _check("fa_fwd", rc)


@_first
def fa_fwd_blocksparse(q, k, v, o, lse, block_mask, scale, causal=False, stream=None):
    B, H, N, d = q.shape
    rc = load().fa_fwd_blocksparse(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"),
                                   _f32(lse, "lse"), _mask_ptr(block_mask), B, H, N, d, float(scale),
                                   int(bool(causal)), _stream(stream))
    _check("fa_fwd_blocksparse", rc)


def fa_bwd_workspace_bytes(B, H, N, d) -> int:
    return load().fa_bwd_workspace_bytes(B, H, N, d)


@_first
def fa_bwd(q, k, v, o, do, lse, dq, dk, dv, workspace, scale, causal=False, stream=None):
    B, H, N, d = q.shape
    rc = load().fa_bwd(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _bf16(do, "do"),
                       _f32(lse, "lse"), _bf16(dq, "dq"), _bf16(dk, "dk"), _bf16(dv, "dv"),
                       ctypes.c_void_p(workspace.data_ptr()), B, H, N, d, float(scale),
                       int(bool(causal)), _stream(stream))
    _check("fa_bwd", rc)


@_first
def fa_bwd_blocksparse(q, k, v, o, do, lse, block_mask, dq, dk, dv, workspace, scale, causal=False, stream=None):
    B, H, N, d = q.shape
    rc = load().fa_bwd_blocksparse(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"),
                                   _bf16(do, "do"), _f32(lse, "lse"), _mask_ptr(block_mask),
                                   _bf16(dq, "dq"), _bf16(dk, "dk"), _bf16(dv, "dv"),
                                   ctypes.c_void_p(workspace.data_ptr()), B, H, N, d, float(scale),
                                   int(bool(causal)), _stream(stream))
    _check("fa_bwd_blocksparse", rc)


@_first
def fa_bwd_preprocess(o, do, lse, workspace, stream=None):
    B, H, N, d = o.shape
    rc = load().fa_bwd_preprocess(_bf16(o, "o"), _bf16(do, "do"), _f32(lse, "lse"),
                                  ctypes.c_void_p(workspace.data_ptr()), B, H, N, d, _stream(stream))
    _check("fa_bwd_preprocess", rc)


@_first
def fa_bwd_main(q, k, v, do, block_mask, dk, dv, workspace, scale, mask_kind, dropout_p=0.0, seed=0,
                stream=None):
    B, H, N, d = q.shape
    rc = load().fa_bwd_main(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(do, "do"),
                            _mask_ptr(block_mask), _bf16(dk, "dk"), _bf16(dv, "dv"),
                            ctypes.c_void_p(workspace.data_ptr()), B, H, N, d, float(scale), int(mask_kind),
                            float(dropout_p), int(seed) & (2 ** 64 - 1), _stream(stream))
    _check("fa_bwd_main", rc)


def fa_dropout_effective_p(dropout_p) -> float:
    """The drop probability the dropout calls apply: dropout_p rounded to a
    multiple of 1/256 (see include/fa.h)."""
    v = load().fa_dropout_effective_p(float(dropout_p))
    if v < 0:
        raise ValueError("dropout_p must be in [0, 1)")
    return v


@_first
def fa_fwd_dropout(q, k, v, o, lse, block_mask, scale, causal, dropout_p, seed, stream=None):
    B, H, N, d = q.shape
    rc = load().fa_fwd_dropout(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _f32(lse, "lse"),
                               _mask_ptr(block_mask), B, H, N, d, float(scale), int(bool(causal)),
                               float(dropout_p), int(seed) & (2 ** 64 - 1), _stream(stream))
    _check("fa_fwd_dropout", rc)


@_first
def fa_bwd_dropout(q, k, v, o, do, lse, block_mask, dq, dk, dv, workspace, scale, causal, dropout_p, seed,
                   stream=None):
    B, H, N, d = q.shape
    rc = load().fa_bwd_dropout(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _bf16(do, "do"),
                               _f32(lse, "lse"), _mask_ptr(block_mask), _bf16(dq, "dq"), _bf16(dk, "dk"),
                               _bf16(dv, "dv"), ctypes.c_void_p(workspace.data_ptr()), B, H, N, d, float(scale),
                               int(bool(causal)), float(dropout_p), int(seed) & (2 ** 64 - 1), _stream(stream))
    _check("fa_bwd_dropout", rc)


@_first
def fa_bwd_dq_convert(workspace, dq, scale, stream=None):
    B, H, N, d = dq.shape
    rc = load().fa_bwd_dq_convert(ctypes.c_void_p(workspace.data_ptr()), _bf16(dq, "dq"), B, H, N, d,
                                  float(scale), _stream(stream))
    _check("fa_bwd_dq_convert", rc)


@_first
def fa_bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, scale, causal=False, stream=None):
    """fa_bwd without a workspace argument: the library uses its own static
    device scratch (see include/fa.h), so this call allocates nothing."""
    B, H, N, d = q.shape
    rc = load().fa_bwd_noalloc(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _bf16(do, "do"),
                               _f32(lse, "lse"), _bf16(dq, "dq"), _bf16(dk, "dk"), _bf16(dv, "dv"),
                               B, H, N, d, float(scale), int(bool(causal)), _stream(stream))
    _check("fa_bwd_noalloc", rc)


def _host(t: torch.Tensor, name: str, dtype=torch.bfloat16, dim=4):
    if t.is_cuda or t.dtype != dtype or not t.is_contiguous() or t.dim() != dim:
        raise ValueError(f"{name} must be a contiguous {dtype} host tensor with {dim} dimensions")
    return ctypes.c_void_p(t.data_ptr())


def fa_fwd_bwd_host_workspace_bytes(B, H, N, d) -> int:
    return load().fa_fwd_bwd_host_workspace_bytes(B, H, N, d)


@_on_device(lambda *a, **k: k.get("workspace", a[10] if len(a) > 10 else None))
def fa_fwd_bwd_host(q, k, v, do, o, lse, dq, dk, dv, block_mask, workspace, scale, causal=False, stream=None):
    """Forward and backward of host tensors (pinned for overlap), streamed
    through the device in chunks of heads; see include/fa.h."""
    B, H, N, d = q.shape
    if not (workspace.is_cuda and workspace.dtype == torch.uint8):
        raise ValueError("workspace must be a uint8 CUDA tensor")
    rc = load().fa_fwd_bwd_host(_host(q, "q"), _host(k, "k"), _host(v, "v"), _host(do, "do"), _host(o, "o"),
                                _host(lse, "lse", torch.float32, 3), _host(dq, "dq"), _host(dk, "dk"),
                                _host(dv, "dv"), _mask_ptr(block_mask), ctypes.c_void_p(workspace.data_ptr()),
                                workspace.numel(), B, H, N, d, float(scale), int(bool(causal)), _stream(stream))
    _check("fa_fwd_bwd_host", rc)


def fa_fwd_host_workspace_bytes(B, H, N, d) -> int:
    return load().fa_fwd_host_workspace_bytes(B, H, N, d)


@_on_device(lambda *a, **k: k.get("workspace", a[6] if len(a) > 6 else None))
def fa_fwd_host(q, k, v, o, lse, block_mask, workspace, scale, causal=False, stream=None):
    """The forward of host tensors (pinned for overlap), streamed through the
    device in chunks of heads; see include/fa.h."""
    B, H, N, d = q.shape
    if not (workspace.is_cuda and workspace.dtype == torch.uint8):
        raise ValueError("workspace must be a uint8 CUDA tensor")
    rc = load().fa_fwd_host(_host(q, "q"), _host(k, "k"), _host(v, "v"), _host(o, "o"),
                            _host(lse, "lse", torch.float32, 3), _mask_ptr(block_mask),
                            ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), B, H, N, d, float(scale),
                            int(bool(causal)), _stream(stream))
    _check("fa_fwd_host", rc)


def fa_decode_workspace_bytes(B, H, Nq, Nk, d) -> int:
    return load().fa_decode_workspace_bytes(B, H, Nq, Nk, d)


@_first
def fa_decode(q, k, v, o, lse, seqlens_k, scale, causal=False, workspace=None, stream=None):
    """q, o [B,H,Nq,d]; k, v [B,H,Nk,d]; lse [B,H,Nq]; seqlens_k int32 [B] or None."""
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != (B, H, Nk, d):
        raise ValueError("k and v must be [B, H, Nk, d] like q")
    if seqlens_k is not None:
        if seqlens_k.dtype != torch.int32 or not seqlens_k.is_cuda or seqlens_k.numel() != B:
            raise ValueError("seqlens_k must be a CUDA int32 tensor of B entries")
        sl = ctypes.c_void_p(seqlens_k.data_ptr())
    else:
        sl = ctypes.c_void_p(0)
    ws = ctypes.c_void_p(workspace.data_ptr()) if workspace is not None else ctypes.c_void_p(0)
    rc = load().fa_decode(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _f32(lse, "lse"), sl,
                          B, H, Nq, Nk, d, float(scale), int(bool(causal)), ws, _stream(stream))
    _check("fa_decode", rc)


def fa_fwd_fp8_workspace_bytes(B, H, N, d) -> int:
    return load().fa_fwd_fp8_workspace_bytes(B, H, N, d)


def _fp8(t, name):
    if not (t.is_cuda and t.dtype == torch.float8_e4m3fn and t.is_contiguous() and t.dim() == 4):
        raise ValueError(f"{name} must be a contiguous float8_e4m3fn CUDA tensor [B, H, N, d]")
    return ctypes.c_void_p(t.data_ptr())


def _descale(t, name, n):
    if t is None:
        return ctypes.c_void_p(0)
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous() and t.numel() == n):
        raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor of B*H entries")
    return ctypes.c_void_p(t.data_ptr())


@_first
def fa_fwd_fp8(q, k, v, o, lse, q_descale, k_descale, v_descale, scale, causal, workspace, stream=None):
    B, H, N, d = q.shape
    rc = load().fa_fwd_fp8(_fp8(q, "q"), _fp8(k, "k"), _fp8(v, "v"), _bf16(o, "o"), _f32(lse, "lse"),
                           _descale(q_descale, "q_descale", B * H), _descale(k_descale, "k_descale", B * H),
                           _descale(v_descale, "v_descale", B * H), B, H, N, d, float(scale), int(bool(causal)),
                           ctypes.c_void_p(workspace.data_ptr()), _stream(stream))
    _check("fa_fwd_fp8", rc)


def forward_fp8(q, k, v, q_descale=None, k_descale=None, v_descale=None, causal=False, scale=None, stream=None):
    """8-bit forward: returns (O bf16 [B,H,N,d], LSE fp32 [B,H,N])."""
    B, H, N, d = q.shape
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    n = fa_fwd_fp8_workspace_bytes(B, H, N, d)
    if n == 0:
        raise ValueError("unsupported sizes for the 8-bit forward (d must be 128)")
    ws = torch.empty(n, dtype=torch.uint8, device=q.device)
    fa_fwd_fp8(q, k, v, o, lse, q_descale, k_descale, v_descale, scale, causal, ws, stream)
    return o, lse


def fa_block_mask_window(N, left, right) -> torch.Tensor:
    """Sliding-window block mask, uint8 [nb, nb] on the host (see include/fa.h)."""
    nb = (N + 127) // 128
    m = torch.empty((max(nb, 1), max(nb, 1)), dtype=torch.uint8)
    _check("fa_block_mask_window", load().fa_block_mask_window(ctypes.c_void_p(m.data_ptr()), N, left, right))
    return m


def fa_block_mask_dilated(N, window, dilation, causal=False) -> torch.Tensor:
    """Dilated-window block mask, uint8 [nb, nb] on the host (see include/fa.h)."""
    nb = (N + 127) // 128
    m = torch.empty((max(nb, 1), max(nb, 1)), dtype=torch.uint8)
    _check("fa_block_mask_dilated", load().fa_block_mask_dilated(ctypes.c_void_p(m.data_ptr()), N, window,
                                                                 dilation, int(bool(causal))))
    return m


def fa_get_device_error(stream=None) -> int:
    return load().fa_get_device_error(_stream(stream))


def fa_set_wait_timeout_ns(ns: int):
    _check("fa_set_wait_timeout_ns", load().fa_set_wait_timeout_ns(int(ns)))


def fa_debug_wait_timeout(ns: int, stream=None) -> int:
    return load().fa_debug_wait_timeout(int(ns), _stream(stream))


# --------------------------------------------------------------------------- #
# conveniences that allocate outputs
# --------------------------------------------------------------------------- #
def forward(q, k, v, causal=False, scale=None, block_mask=None, dropout_p=0.0, seed=0, stream=None):
    """Returns (O bf16 [B,H,N,d], LSE fp32 [B,H,N])."""
    B, H, N, d = q.shape
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if dropout_p:
        fa_fwd_dropout(q, k, v, o, lse, block_mask, scale, causal, dropout_p, seed, stream)
    elif block_mask is not None:
        fa_fwd_blocksparse(q, k, v, o, lse, block_mask, scale, causal, stream)
    else:
        fa_fwd(q, k, v, o, lse, scale, causal, stream)
    return o, lse


def decode(q, k, v, seqlens_k=None, causal=False, scale=None, ws=None, stream=None):
    """Returns (O bf16 [B,H,Nq,d], LSE fp32 [B,H,Nq]) of q against the cache k, v."""
    B, H, Nq, d = q.shape
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if ws is None:
        n = fa_decode_workspace_bytes(B, H, Nq, k.shape[2], d)
        ws = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    fa_decode(q, k, v, o, lse, seqlens_k, scale, causal, ws, stream)
    return o, lse


def workspace(B, H, N, d, device) -> torch.Tensor:
    n = fa_bwd_workspace_bytes(B, H, N, d)
    if n == 0:
        raise ValueError("invalid sizes for the backward workspace")
    return torch.empty(n, dtype=torch.uint8, device=device)


def backward(q, k, v, o, lse, do, causal=False, scale=None, block_mask=None, ws=None, dropout_p=0.0, seed=0,
             stream=None):
    """Returns (dQ, dK, dV), bf16 [B,H,N,d]."""
    B, H, N, d = q.shape
    scale = (1.0 / d ** 0.5) if scale is None else scale
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = workspace(B, H, N, d, q.device) if ws is None else ws
    if dropout_p:
        fa_bwd_dropout(q, k, v, o, do, lse, block_mask, dq, dk, dv, ws, scale, causal, dropout_p, seed, stream)
    elif block_mask is not None:
        fa_bwd_blocksparse(q, k, v, o, do, lse, block_mask, dq, dk, dv, ws, scale, causal, stream)
    else:
        fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, scale, causal, stream)
    return dq, dk, dv


def forward_backward_host(q, k, v, do, causal=False, scale=None, block_mask=None, ws=None, stream=None):
    """Forward and backward of host tensors; returns pinned host (O, LSE, dQ,
    dK, dV).  ``ws``: a device workspace of fa_fwd_bwd_host_workspace_bytes
    bytes (allocated when omitted)."""
    B, H, N, d = q.shape
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o, dq, dk, dv = (torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(4))
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    if ws is None:
        ws = torch.empty(fa_fwd_bwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa_fwd_bwd_host(q, k, v, do, o, lse, dq, dk, dv, block_mask, ws, scale, causal, stream)
    return o, lse, dq, dk, dv


def forward_host(q, k, v, causal=False, scale=None, block_mask=None, ws=None, stream=None):
    """The forward of host tensors; returns pinned host (O, LSE).  ``ws``: a
    device workspace of fa_fwd_host_workspace_bytes bytes (allocated when
    omitted)."""
    B, H, N, d = q.shape
    scale = (1.0 / d ** 0.5) if scale is None else scale
    o = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    if ws is None:
        ws = torch.empty(fa_fwd_host_workspace_bytes(B, H, N, d), dtype=torch.uint8, device="cuda")
    fa_fwd_host(q, k, v, o, lse, block_mask, ws, scale, causal, stream)
    return o, lse


def fa_status_string(code: int) -> str:
    return status_string(code)
