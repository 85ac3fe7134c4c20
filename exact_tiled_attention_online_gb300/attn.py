"""Python binding of the C ABI in ``include/attn.h`` (ctypes).

Argument marshalling only: this module checks tensor shapes and dtypes,
allocates outputs and workspace through PyTorch's caching allocator, and passes
raw device pointers and the current CUDA stream to the library.  Every step of
the attention itself runs in the library's CUDA kernels; there is no other
implementation behind these functions, and they raise if the library is
missing.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from . import build as _build

MASK_NONE = 0
CAUSAL_TOP_LEFT = 1
CAUSAL_BOTTOM_RIGHT = 2
DTYPE_BF16 = 0
DTYPE_FP32 = 1

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "workspace too small",
          4: "CUDA error", 5: "device wait timed out", 6: "cu_seqlens out of bounds",
          7: "needs more than the static scratch holds",
          8: "a backward input holds an infinity or NaN"}


class AttnStrides(ctypes.Structure):
    """``attn_strides``: {token stride, head stride} in elements per tensor."""
    _fields_ = [(n, ctypes.c_int64 * 2) for n in ("q", "k", "v", "o", "dout", "dq", "dk", "dv")]


class AttnBiasTensor(ctypes.Structure):
    """``attn_bias_tensor``: fp32 data and its sequence, head and row strides."""
    _fields_ = [("data", ctypes.c_void_p), ("seq_stride", ctypes.c_int64),
                ("head_stride", ctypes.c_int64), ("row_stride", ctypes.c_int64)]


class AttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: status {status} ({STATUS.get(status, '?')})")
        self.status = status


_lib: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB_PATH


def library() -> ctypes.CDLL:
    """Load the in-tree CUDA library (built by ``build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA attention library not built: {path} is missing "
                           "(run exact_tiled_attention_online_gb300.build.build())")
    L = ctypes.CDLL(path)
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.attn_fwd.argtypes = [P, P, P, P, P, P, P, P] + [I] * 8 + [F, I, I, P, I, P, SZ, P]
    L.attn_fwd.restype = I
    L.attn_bwd.argtypes = [P] * 12 + [I] * 8 + [F, I, I, P, I, P, SZ, P]
    L.attn_bwd.restype = I
    ex = [ctypes.POINTER(AttnStrides), ctypes.POINTER(AttnBiasTensor)]
    L.attn_fwd_ex.argtypes = ex + L.attn_fwd.argtypes
    L.attn_fwd_ex.restype = I
    L.attn_bwd_ex.argtypes = ex + L.attn_bwd.argtypes
    L.attn_bwd_ex.restype = I
    L.attn_fwd_workspace_size.argtypes = [I] * 9
    L.attn_fwd_workspace_size.restype = SZ
    L.attn_bwd_workspace_size.argtypes = [I] * 9
    L.attn_bwd_workspace_size.restype = SZ
    L.attn_mask_probe.argtypes = [P, P] + [I] * 8 + [P, P]
    L.attn_mask_probe.restype = I
    L.attn_get_device_error.argtypes = [P]
    L.attn_get_device_error.restype = I
    L.attn_status_string.argtypes = [I]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_last_plan.argtypes = []
    L.attn_last_plan.restype = ctypes.c_char_p
    L.attn_version.argtypes = []
    L.attn_version.restype = I
    L.attn_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.attn_set_wait_limit_ns.restype = None
    L.attn_set_deterministic.argtypes = [ctypes.c_int]
    L.attn_set_deterministic.restype = None
    L.attn_get_deterministic.argtypes = []
    L.attn_get_deterministic.restype = ctypes.c_int
    _lib = L
    return L


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype == torch.float32:
        return DTYPE_FP32
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp32 expected")


def _check(t: torch.Tensor, name: str, dims: int, strided: bool = False):
    """``strided``: a [tokens, heads, d] tensor whose features are contiguous
    and whose token and head strides the library takes as they are."""
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions")
    if strided:
        if t.stride(-1) != 1:
            raise ValueError(f"{name}: the last dimension must be contiguous")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _strides(**tensors) -> AttnStrides:
    s = AttnStrides()
    for name, t in tensors.items():
        if t is not None:
            getattr(s, name)[0] = t.stride(0)
            getattr(s, name)[1] = t.stride(1)
    return s


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _slopes_ptr(slopes: Optional[torch.Tensor], hq: int) -> Optional[int]:
    if slopes is None:
        return None
    _check(slopes, "bias_slopes", 1)
    if slopes.dtype != torch.float32 or slopes.numel() != hq:
        raise ValueError("bias_slopes must be fp32 with one slope per query head")
    return slopes.data_ptr()


def _btab(bias: Optional[torch.Tensor], batch: int, hq: int, max_q: int, max_k: int):
    """``attn_bias_tensor`` for a 4-D fp32 CUDA tensor [1 or B, 1 or Hq,
    >= max_seqlen_q, >= max_seqlen_k] with unit key stride (broadcast views
    from ``expand`` are fine), or None."""
    if bias is None:
        return None
    if not getattr(bias, "is_cuda", False) or bias.dtype != torch.float32:
        raise ValueError("bias must be an fp32 CUDA tensor")
    if bias.dim() != 4 or bias.shape[0] not in (1, batch) or bias.shape[1] not in (1, hq):
        raise ValueError("bias must be [1 or B, 1 or Hq, rows, keys]")
    if bias.shape[2] < max_q or bias.shape[3] < max_k or (bias.shape[3] > 1 and bias.stride(3) != 1):
        raise ValueError("bias must cover max_seqlen_q rows and max_seqlen_k keys, keys contiguous")
    st = [0 if bias.shape[i] == 1 else bias.stride(i) for i in range(3)]
    return AttnBiasTensor(bias.data_ptr(), st[0], st[1], st[2])


def fwd_workspace_size(batch, max_q, max_k, total_q, hq, hkv, d, dtype_code, window=0) -> int:
    n = library().attn_fwd_workspace_size(batch, max_q, max_k, total_q, hq, hkv, d, int(window),
                                          dtype_code)
    if n == ctypes.c_size_t(-1).value:
        raise AttnError("attn_fwd_workspace_size", 1)
    return n


def bwd_workspace_size(batch, max_q, max_k, total_q, total_k, hq, hkv, d, dtype_code) -> int:
    n = library().attn_bwd_workspace_size(batch, max_q, max_k, total_q, total_k, hq, hkv, d,
                                          dtype_code)
    if n == ctypes.c_size_t(-1).value:
        raise AttnError("attn_bwd_workspace_size", 1)
    return n


def fwd(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int,
        mask: int = CAUSAL_TOP_LEFT, scale: Optional[float] = None,
        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
        workspace: Optional[torch.Tensor] = None, stream=None, want_lse: bool = True,
        o_f32: Optional[torch.Tensor] = None, want_o_f32: bool = False, window: int = 0,
        bias_slopes: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None):
    """Attention forward on packed ragged tensors (layouts in include/attn.h).

    ``window`` > 0 (causal masks only) bounds every row to the ``window`` key
    positions that end at its causal bound.  ``bias_slopes`` (fp32 CUDA
    tensor, one slope per query head) adds the linear positional bias
    -slope_h * |i + off - j|.  ``bias`` (fp32 CUDA tensor [1 or B, 1 or Hq,
    rows, keys], entry [s, h, i, j] for in-sequence row i and key j) is added
    to the scaled logits; -inf entries mask pairs.

    Returns (o, lse), or (o, lse, o_f32) when ``want_o_f32`` is set or an
    ``o_f32`` buffer is given.  lse is [n_heads_q, total_q] fp32 (None when
    ``want_lse`` is False and no ``lse`` buffer is given); o_f32 is the fp32
    output before rounding, which ``bwd`` uses for the D term.
    """
    _check(q, "q", 3, True), _check(k, "k", 3, True), _check(v, "v", 3, True)
    _check(cu_seqlens_q, "cu_seqlens_q", 1), _check(cu_seqlens_k, "cu_seqlens_k", 1)
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share a dtype")
    total_q, hq, d = q.shape
    total_k, hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, device=q.device)
    _check(out, "out", 3, True)
    if lse is None and want_lse:
        lse = torch.empty((hq, total_q), dtype=torch.float32, device=q.device)
    ret_f32 = want_o_f32 or o_f32 is not None
    if o_f32 is None and want_o_f32:
        o_f32 = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    ws_bytes = fwd_workspace_size(batch, max_seqlen_q, max_seqlen_k, total_q, hq, hkv, d, dt,
                                  window)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    strides = _strides(q=q, k=k, v=v, o=out)
    bt = _btab(bias, batch, hq, max_seqlen_q, max_seqlen_k)
    st = library().attn_fwd_ex(
        ctypes.byref(strides), None if bt is None else ctypes.byref(bt),
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(o_f32), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_k),
        batch, max_seqlen_q, max_seqlen_k, total_q, total_k, hq, hkv, d, float(scale),
        int(mask), int(window), _slopes_ptr(bias_slopes, hq), dt, _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream))
    if st != 0:
        raise AttnError("attn_fwd", st)
    return (out, lse, o_f32) if ret_f32 else (out, lse)


def bwd(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
        max_seqlen_k: int, mask: int = CAUSAL_TOP_LEFT, scale: Optional[float] = None,
        dq=None, dk=None, dv=None, workspace=None, stream=None,
        o_f32: Optional[torch.Tensor] = None, window: int = 0,
        bias_slopes: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None):
    """Attention backward; returns (dq, dk, dv) with dk/dv summed over each
    KV head's group of query heads.  Pass the forward's ``o_f32`` when it was
    kept: D_i = dO_i . O_i then comes from it; without it the library
    recomputes the fp32 output for D (one extra forward pass).  Pass the
    forward's mask, ``window``, ``bias_slopes`` and ``bias``."""
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _check(t, n, 3, True)
    _check(lse, "lse", 2)
    dt = _dtype_code(q)
    total_q, hq, d = q.shape
    total_k, hkv, _ = k.shape
    batch = cu_seqlens_q.numel() - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty(q.shape, dtype=q.dtype, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=k.dtype, device=k.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=v.dtype, device=v.device) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, 3, True)
    ws_bytes = bwd_workspace_size(batch, max_seqlen_q, max_seqlen_k, total_q, total_k, hq, hkv,
                                  d, dt)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    strides = _strides(q=q, k=k, v=v, o=o, dout=dout, dq=dq, dk=dk, dv=dv)
    bt = _btab(bias, batch, hq, max_seqlen_q, max_seqlen_k)
    st = library().attn_bwd_ex(
        ctypes.byref(strides), None if bt is None else ctypes.byref(bt),
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(o_f32), _ptr(dout), _ptr(dq),
        _ptr(dk), _ptr(dv),
        _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), batch, max_seqlen_q, max_seqlen_k, total_q,
        total_k, hq, hkv, d, float(scale), int(mask), int(window),
        _slopes_ptr(bias_slopes, hq), dt, _ptr(workspace),
        0 if workspace is None else workspace.numel(), _stream(stream))
    if st != 0:
        raise AttnError("attn_bwd", st)
    return dq, dk, dv


def mask_probe(cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, total_q, total_k,
               mask, tile_rows=128, stream=None, window: int = 0) -> torch.Tensor:
    out = torch.empty((total_q, total_k), dtype=torch.uint8, device=cu_seqlens_q.device)
    st = library().attn_mask_probe(_ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
                                   cu_seqlens_q.numel() - 1, max_seqlen_q, max_seqlen_k,
                                   total_q, total_k, int(mask), int(window), int(tile_rows),
                                   _ptr(out), _stream(stream))
    if st != 0:
        raise AttnError("attn_mask_probe", st)
    return out


def get_device_error(stream=None) -> int:
    return library().attn_get_device_error(_stream(stream))


def set_wait_limit_ns(ns: int) -> None:
    """Bound of every wait inside the kernels for the following calls (0:
    the 2 s default); see ``attn_set_wait_limit_ns`` in include/attn.h."""
    library().attn_set_wait_limit_ns(int(ns))


def set_deterministic(on: bool) -> None:
    """Backward form for the following bf16 calls: True keeps the
    two-kernel backward (every gradient reproducible bit for bit), False
    (the default) the fused one (dQ summed with reductions); see
    ``attn_set_deterministic`` in include/attn.h."""
    library().attn_set_deterministic(1 if on else 0)


def get_deterministic() -> bool:
    return bool(library().attn_get_deterministic())


def last_plan() -> str:
    return library().attn_last_plan().decode()


def status_string(code: int) -> str:
    return library().attn_status_string(code).decode()
