"""Python binding of libsdpa_gb300.so (scaled dot-product attention on GB300).

Argument marshalling only: shapes and device pointers of torch tensors are
passed to the C ABI declared in include/sdpa.h, outputs and workspaces are
allocated with torch on the inputs' device, and work is enqueued on torch's
current CUDA stream of that device.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback.  Importing works without a GPU;
calling needs the built library (``build()``) and a CUDA device, and raises
otherwise.

The C ABI receives plain pointers and one shape, so it cannot see a tensor whose
extents disagree with that shape.  The binding therefore checks every tensor's
shape, dtype, device and contiguity against the shape derived from q, k and v
(ValueError) before it loads the library or launches anything.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional

from .build import LIB_PATH, build  # noqa: F401

__all__ = [
    "SdpaError", "load_library", "exported_symbols", "sdpa_forward", "sdpa_backward", "sdpa_decode",
    "forward_workspace_bytes", "backward_workspace_bytes", "decode_workspace_bytes",
    "decode_num_splits", "last_device_status", "Shape", "Options", "Band", "Dropout", "PagedKV",
    "sdpa_decode_paged", "selftest_wait_timeout",
    "build", "LIB_PATH",
]

SDPA_F32, SDPA_BF16 = 0, 1
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "timeout"}

# Every symbol include/sdpa.h declares.
EXPORTS = (
    "sdpa_forward", "sdpa_forward_workspace_bytes", "sdpa_backward", "sdpa_backward_workspace_bytes",
    "sdpa_decode", "sdpa_decode_workspace_bytes", "sdpa_decode_num_splits", "sdpa_status_string",
    "sdpa_last_device_status", "sdpa_decode_noalloc", "sdpa_forward_opts", "sdpa_backward_opts",
    "sdpa_decode_opts", "sdpa_decode_paged", "sdpa_selftest_wait_timeout",
)


class SdpaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} (status {status})")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("Hq", ctypes.c_int64), ("Hkv", ctypes.c_int64),
                ("L", ctypes.c_int64), ("S", ctypes.c_int64), ("E", ctypes.c_int64),
                ("Ev", ctypes.c_int64), ("dtype", ctypes.c_int32), ("mask_b", ctypes.c_int32),
                ("mask_h", ctypes.c_int32)]


class Options(ctypes.Structure):
    """sdpa_options: padding lengths (device int32 [B] or NULL), diagonal alignment, band bounds."""
    _fields_ = [("seq_len_q", ctypes.c_void_p), ("seq_len_kv", ctypes.c_void_p),
                ("diagonal_alignment", ctypes.c_int32), ("right_bound", ctypes.c_int32),
                ("left_bound", ctypes.c_int32), ("dropout_p", ctypes.c_double), ("dropout_seed", ctypes.c_uint64),
                ("dropout_offset", ctypes.c_uint64)]


class Band:
    """Padding and diagonal band of a call (see sdpa_options in include/sdpa.h).

    seq_len_q, seq_len_kv: None or CUDA int32 tensors of B lengths; alignment:
    "top_left" or "bottom_right"; right_bound: None or >= 0 (0 = causal);
    left_bound: None or >= 1 (sliding window).
    """

    def __init__(self, seq_len_q=None, seq_len_kv=None, alignment="top_left", right_bound=None, left_bound=None):
        self.seq_len_q, self.seq_len_kv = seq_len_q, seq_len_kv
        self.alignment, self.right_bound, self.left_bound = alignment, right_bound, left_bound

    def options(self, dropout=None, batch: Optional[int] = None) -> Options:
        """The sdpa_options struct; batch, when given, is the call's B, which each length tensor must match."""
        import torch
        for t in (self.seq_len_q, self.seq_len_kv):
            if t is not None and batch is not None and (t.dim() != 1 or t.numel() != batch):
                raise ValueError(f"seq_len tensors must hold B = {batch} lengths, got shape {tuple(t.shape)}")
            if t is not None and (not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous()):
                raise ValueError("seq_len tensors must be contiguous CUDA int32")
        align = {"top_left": 0, "bottom_right": 1}.get(self.alignment)
        if align is None:
            raise ValueError("alignment is top_left or bottom_right")
        dp, ds, do = (0.0, 0, 0) if dropout is None else (float(dropout.p), int(dropout.seed), int(dropout.offset))
        return Options(_ptr(self.seq_len_q), _ptr(self.seq_len_kv), align,
                       -1 if self.right_bound is None else int(self.right_bound),
                       0 if self.left_bound is None else int(self.left_bound), dp, ds & (2 ** 64 - 1),
                       do & (2 ** 64 - 1))


class Dropout:
    """Attention dropout of a prefill forward/backward pair: probability p in [0, 1), 64-bit seed, offset in
    [0, 2^32) (the library checks both and answers INVALID_ARG)."""

    def __init__(self, p: float, seed: int, offset: int = 0):
        self.p, self.seed, self.offset = float(p), int(seed), int(offset)


class PagedKV(ctypes.Structure):
    """sdpa_paged_kv: page tables (device int32 [B * max_blocks]), block sizes, table width, container sizes."""
    _fields_ = [("page_table_k", ctypes.c_void_p), ("page_table_v", ctypes.c_void_p),
                ("block_size_k", ctypes.c_int32), ("block_size_v", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("num_blocks_k", ctypes.c_int64), ("num_blocks_v", ctypes.c_int64)]


_lib = None
_P = ctypes.c_void_p


def load_library(path: Optional[str] = None):
    """Load libsdpa_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} is missing; run scaled_dot_product_sm_gb300.build()")
    lib = ctypes.CDLL(path)
    SP = ctypes.POINTER(Shape)
    lib.sdpa_forward.argtypes = [SP, _P, _P, _P, _P, ctypes.c_double, ctypes.c_int, ctypes.c_int, _P, _P, _P,
                                 ctypes.c_size_t, _P]
    lib.sdpa_forward.restype = ctypes.c_int
    lib.sdpa_backward.argtypes = [SP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                  _P, _P, _P, _P, ctypes.c_size_t, _P]
    lib.sdpa_backward.restype = ctypes.c_int
    lib.sdpa_decode.argtypes = [SP, _P, _P, _P, _P, ctypes.c_double, ctypes.c_int, ctypes.c_int, _P, _P, _P,
                                ctypes.c_size_t, _P]
    lib.sdpa_decode.restype = ctypes.c_int
    lib.sdpa_decode_noalloc.argtypes = [SP, _P, _P, _P, _P, ctypes.c_double, ctypes.c_int, ctypes.c_int, _P, _P,
                                        _P]
    lib.sdpa_decode_noalloc.restype = ctypes.c_int
    OP = ctypes.POINTER(Options)
    lib.sdpa_forward_opts.argtypes = [SP, OP, _P, _P, _P, _P, ctypes.c_double, ctypes.c_int, _P, _P, _P,
                                      ctypes.c_size_t, _P]
    lib.sdpa_forward_opts.restype = ctypes.c_int
    lib.sdpa_backward_opts.argtypes = [SP, OP, _P, _P, _P, _P, _P, _P, _P, ctypes.c_double, ctypes.c_int,
                                       _P, _P, _P, _P, ctypes.c_size_t, _P]
    lib.sdpa_backward_opts.restype = ctypes.c_int
    lib.sdpa_decode_opts.argtypes = [SP, OP, _P, _P, _P, _P, ctypes.c_double, ctypes.c_int, ctypes.c_int, _P, _P,
                                     _P, ctypes.c_size_t, _P]
    lib.sdpa_decode_opts.restype = ctypes.c_int
    lib.sdpa_decode_paged.argtypes = [SP, OP, ctypes.POINTER(PagedKV), _P, _P, _P, _P, ctypes.c_double, ctypes.c_int,
                                      ctypes.c_int, _P, _P, _P, ctypes.c_size_t, _P]
    lib.sdpa_decode_paged.restype = ctypes.c_int
    for fn in ("sdpa_forward_workspace_bytes", "sdpa_backward_workspace_bytes"):
        getattr(lib, fn).argtypes = [SP]
        getattr(lib, fn).restype = ctypes.c_size_t
    lib.sdpa_decode_workspace_bytes.argtypes = [SP, ctypes.c_int]
    lib.sdpa_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.sdpa_decode_num_splits.argtypes = [SP]
    lib.sdpa_decode_num_splits.restype = ctypes.c_int
    lib.sdpa_status_string.argtypes = [ctypes.c_int]
    lib.sdpa_status_string.restype = ctypes.c_char_p
    lib.sdpa_last_device_status.argtypes = [ctypes.c_void_p]
    lib.sdpa_last_device_status.restype = ctypes.c_int
    lib.sdpa_selftest_wait_timeout.argtypes = [ctypes.c_void_p]
    lib.sdpa_selftest_wait_timeout.restype = ctypes.c_int
    if path == LIB_PATH:
        _lib = lib
    return lib


def exported_symbols(path: Optional[str] = None):
    """Names of EXPORTS that the library resolves (loads it, calls nothing)."""
    lib = load_library(path)
    found = []
    for name in EXPORTS:
        try:
            getattr(lib, name)
            found.append(name)
        except AttributeError:
            pass
    return found


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return SDPA_F32
    if t.dtype == torch.bfloat16:
        return SDPA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _expect(t, name, shape, dtype):
    """Raises ValueError unless t (if given) has exactly this shape and dtype."""
    if t is None:
        return
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(int(x) for x in shape)}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _check_mask(mask, L, S):
    """The additive mask is fp32 [mask_b, mask_h, L, S]; the library checks mask_b and mask_h."""
    import torch
    if mask is None:
        return
    if mask.dim() != 4:
        raise ValueError("mask must be 4-D [B|1, Hq|1, L, S]")
    _expect(mask, "mask", (mask.shape[0], mask.shape[1], L, S), torch.float32)


def _check_qkv(q, k, v, mask):
    """q [B,Hq,L,E], k [B,Hkv,S,E], v [B,Hkv,S,Ev] of one dtype, and the mask."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, T, D]")
    B, Hq, L, E = q.shape
    _, Hkv, S, _ = k.shape
    _expect(k, "k", (B, Hkv, S, E), q.dtype)
    _expect(v, "v", (B, Hkv, S, v.shape[3]), q.dtype)
    _check_mask(mask, L, S)


def _shape(q, k, v, mask) -> Shape:
    _check_qkv(q, k, v, mask)
    B, Hq, L, E = q.shape
    _, Hkv, S, _ = k.shape
    Ev = v.shape[3]
    mb, mh = (1, 1) if mask is None else (mask.shape[0], mask.shape[1])
    return Shape(B, Hq, Hkv, L, S, E, Ev, _dtype_code(q), mb, mh)


def _check_tensors(*ts):
    """Every tensor given is contiguous and on the first one's CUDA device."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous (BHSD)")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors must be on one device: {dev} and {t.device}")


def _band_tensors(band):
    return (None, None) if band is None else (band.seq_len_q, band.seq_len_kv)


def _on_device(t):
    """Makes t's device current for the call, so the library launches there and on its stream
    (no switch when it is current already)."""
    import torch
    if not t.is_cuda or t.device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(t.device)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _scale(scale):
    return float("nan") if scale is None else float(scale)


def _raise(status, where):
    if status != 0:
        raise SdpaError(status, where)


def _workspace(nbytes, device):
    import torch
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def forward_workspace_bytes(q, k, v, mask=None) -> int:
    return int(load_library().sdpa_forward_workspace_bytes(ctypes.byref(_shape(q, k, v, mask))))


def backward_workspace_bytes(q, k, v, mask=None) -> int:
    return int(load_library().sdpa_backward_workspace_bytes(ctypes.byref(_shape(q, k, v, mask))))


def decode_workspace_bytes(q, k, v, num_splits=0) -> int:
    return int(load_library().sdpa_decode_workspace_bytes(ctypes.byref(_shape(q, k, v, None)), int(num_splits)))


def decode_num_splits(q, k, v) -> int:
    return int(load_library().sdpa_decode_num_splits(ctypes.byref(_shape(q, k, v, None))))


def sdpa_forward(q, k, v, mask=None, scale=None, is_causal=False, enable_gqa=False,
                 out=None, lse=None, workspace=None, stream=None, band=None, dropout=None):
    """O [B,Hq,L,Ev] (dtype of q) and LSE [B,Hq,L] fp32 of softmax(scale*q k^T + mask) v.

    band: None, or a Band (padding lengths, diagonal alignment, bounds) used in
    place of is_causal (sdpa_forward_opts).  dropout: None or a Dropout (the
    backward must get the same one).
    """
    import torch
    shp = _shape(q, k, v, mask)
    B, Hq, L, _ = q.shape
    _expect(out, "out", (B, Hq, L, v.shape[3]), q.dtype)
    _expect(lse, "lse", (B, Hq, L), torch.float32)
    _check_tensors(q, k, v, mask, out, lse, workspace, *_band_tensors(band))
    with _on_device(q):
        return _forward(shp, q, k, v, mask, scale, is_causal, enable_gqa, out, lse, workspace, stream, band, dropout)


def _forward(shp, q, k, v, mask, scale, is_causal, enable_gqa, out, lse, workspace, stream, band, dropout):
    import torch
    lib = load_library()
    B, Hq, L, _ = q.shape
    if out is None:
        out = torch.empty(B, Hq, L, v.shape[3], dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, L, dtype=torch.float32, device=q.device)
    # the workspace holds the decode route's split partials (one query row) or the unit
    # counter of calls with padding lengths; other calls run without one
    if workspace is None and (L == 1 or (band is not None and (band.seq_len_q is not None
                                                             or band.seq_len_kv is not None))):
        need = int(lib.sdpa_forward_workspace_bytes(ctypes.byref(shp)))
        if need:
            workspace = _workspace(need, q.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if band is None and dropout is not None:
        band = Band(right_bound=0 if is_causal else None)
    if band is not None:
        opts = band.options(dropout, batch=B)
        st = lib.sdpa_forward_opts(ctypes.byref(shp), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v), _ptr(mask),
                                   _scale(scale), int(bool(enable_gqa)), _ptr(out), _ptr(lse), _ptr(workspace), wsb,
                                   _stream(stream))
        _raise(st, "sdpa_forward_opts")
        return out, lse
    st = lib.sdpa_forward(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(mask), _scale(scale),
                          int(bool(is_causal)), int(bool(enable_gqa)), _ptr(out), _ptr(lse), _ptr(workspace),
                          wsb, _stream(stream))
    _raise(st, "sdpa_forward")
    return out, lse


def sdpa_backward(q, k, v, o, dO, lse, mask=None, scale=None, is_causal=False, enable_gqa=False,
                  dq=None, dk=None, dv=None, workspace=None, stream=None, band=None, dropout=None):
    """dQ, dK, dV of sum(O * dO); o and lse are the forward's outputs (same band)."""
    import torch
    shp = _shape(q, k, v, mask)
    B, Hq, L, _ = q.shape
    _expect(o, "o", (B, Hq, L, v.shape[3]), q.dtype)
    _expect(dO, "dO", (B, Hq, L, v.shape[3]), q.dtype)
    _expect(lse, "lse", (B, Hq, L), torch.float32)
    _expect(dq, "dq", q.shape, q.dtype)
    _expect(dk, "dk", k.shape, q.dtype)
    _expect(dv, "dv", v.shape, q.dtype)
    _check_tensors(q, k, v, o, dO, lse, mask, dq, dk, dv, workspace, *_band_tensors(band))
    with _on_device(q):
        return _backward(shp, q, k, v, o, dO, lse, mask, scale, is_causal, enable_gqa, dq, dk, dv, workspace,
                         stream, band, dropout)


def _backward(shp, q, k, v, o, dO, lse, mask, scale, is_causal, enable_gqa, dq, dk, dv, workspace, stream, band,
              dropout):
    import torch
    lib = load_library()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        workspace = _workspace(lib.sdpa_backward_workspace_bytes(ctypes.byref(shp)), q.device)
    wsb = workspace.numel() * workspace.element_size()
    if band is None and dropout is not None:
        band = Band(right_bound=0 if is_causal else None)
    if band is not None:
        opts = band.options(dropout, batch=q.shape[0])
        st = lib.sdpa_backward_opts(ctypes.byref(shp), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                    _ptr(dO), _ptr(lse), _ptr(mask), _scale(scale), int(bool(enable_gqa)), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(workspace), wsb, _stream(stream))
        _raise(st, "sdpa_backward_opts")
        return dq, dk, dv
    st = lib.sdpa_backward(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dO), _ptr(lse),
                           _ptr(mask), _scale(scale), int(bool(is_causal)), int(bool(enable_gqa)), _ptr(dq),
                           _ptr(dk), _ptr(dv), _ptr(workspace), wsb, _stream(stream))
    _raise(st, "sdpa_backward")
    return dq, dk, dv


def sdpa_decode(q, k, v, mask=None, scale=None, enable_gqa=False, num_splits=0,
                out=None, lse=None, workspace=None, stream=None, band=None):
    """Split-KV decode forward (bf16): same outputs as sdpa_forward (band: sdpa_decode_opts)."""
    import torch
    shp = _shape(q, k, v, mask)
    B, Hq, L, _ = q.shape
    _expect(out, "out", (B, Hq, L, v.shape[3]), q.dtype)
    _expect(lse, "lse", (B, Hq, L), torch.float32)
    _check_tensors(q, k, v, mask, out, lse, workspace, *_band_tensors(band))
    with _on_device(q):
        return _decode(shp, q, k, v, mask, scale, enable_gqa, num_splits, out, lse, workspace, stream, band)


def _decode(shp, q, k, v, mask, scale, enable_gqa, num_splits, out, lse, workspace, stream, band):
    import torch
    lib = load_library()
    B, Hq, L, _ = q.shape
    if out is None:
        out = torch.empty(B, Hq, L, v.shape[3], dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty(B, Hq, L, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = _workspace(lib.sdpa_decode_workspace_bytes(ctypes.byref(shp), int(num_splits)), q.device)
    wsb = workspace.numel() * workspace.element_size()
    if band is not None:
        opts = band.options(batch=B)
        st = lib.sdpa_decode_opts(ctypes.byref(shp), ctypes.byref(opts), _ptr(q), _ptr(k), _ptr(v), _ptr(mask),
                                  _scale(scale), int(bool(enable_gqa)), int(num_splits), _ptr(out), _ptr(lse),
                                  _ptr(workspace), wsb, _stream(stream))
        _raise(st, "sdpa_decode_opts")
        return out, lse
    st = lib.sdpa_decode(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(mask), _scale(scale),
                         int(bool(enable_gqa)), int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace), wsb,
                         _stream(stream))
    _raise(st, "sdpa_decode")
    return out, lse


def sdpa_decode_paged(q, k_container, v_container, page_table_k, page_table_v, S, mask=None, scale=None,
                      enable_gqa=False, num_splits=0, band=None, out=None, lse=None, workspace=None, stream=None):
    """Split-KV decode over paged caches (bf16).

    k_container [num_blocks_k, Hkv, bs_k, E], v_container [num_blocks_v, Hkv, bs_v, Ev];
    page tables CUDA int32 [B, max_blocks]; S = the longest cache; band usually
    carries seq_len_kv (each sequence's cache length).
    """
    import torch
    if q.dim() != 4 or k_container.dim() != 4 or v_container.dim() != 4:
        raise ValueError("q and the containers must be 4-D")
    B, Hq, L, E = q.shape
    Hkv, Ev = k_container.shape[1], v_container.shape[3]
    _expect(k_container, "k_container", (k_container.shape[0], Hkv, k_container.shape[2], E), q.dtype)
    _expect(v_container, "v_container", (v_container.shape[0], Hkv, v_container.shape[2], Ev), q.dtype)
    for t in (page_table_k, page_table_v):
        if t.dtype != torch.int32 or t.dim() != 2 or t.shape[0] != B:
            raise ValueError("page tables must be int32 [B, max_blocks]")
    if page_table_k.shape != page_table_v.shape:
        raise ValueError("page tables must have the same shape")
    _check_mask(mask, L, int(S))
    _expect(out, "out", (B, Hq, L, Ev), q.dtype)
    _expect(lse, "lse", (B, Hq, L), torch.float32)
    _check_tensors(q, k_container, v_container, mask, page_table_k, page_table_v, out, lse, workspace,
                   *_band_tensors(band))
    mb, mh = (1, 1) if mask is None else (mask.shape[0], mask.shape[1])
    shp = Shape(B, Hq, Hkv, L, int(S), E, Ev, _dtype_code(q), mb, mh)
    paged = PagedKV(_ptr(page_table_k), _ptr(page_table_v), k_container.shape[2], v_container.shape[2],
                    page_table_k.shape[1], k_container.shape[0], v_container.shape[0])
    opts = (band or Band()).options(batch=B)
    with _on_device(q):
        lib = load_library()
        if out is None:
            out = torch.empty(B, Hq, L, Ev, dtype=q.dtype, device=q.device)
        if lse is None:
            lse = torch.empty(B, Hq, L, dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = _workspace(lib.sdpa_decode_workspace_bytes(ctypes.byref(shp), int(num_splits)), q.device)
        st = lib.sdpa_decode_paged(ctypes.byref(shp), ctypes.byref(opts), ctypes.byref(paged), _ptr(q),
                                   _ptr(k_container), _ptr(v_container), _ptr(mask), _scale(scale),
                                   int(bool(enable_gqa)), int(num_splits), _ptr(out), _ptr(lse), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(st, "sdpa_decode_paged")
    return out, lse


def last_device_status(stream=None) -> int:
    """Reads and clears the device status word after the work on `stream` (default: torch's
    current stream), synchronising that stream only."""
    return int(load_library().sdpa_last_device_status(_stream(stream)))


def selftest_wait_timeout(stream=None) -> None:
    """Runs the failure-path self-test kernel (a bounded wait that nothing satisfies: it gives
    up after about a second and records a timeout); read last_device_status() afterwards."""
    _raise(load_library().sdpa_selftest_wait_timeout(_stream(stream)), "sdpa_selftest_wait_timeout")

