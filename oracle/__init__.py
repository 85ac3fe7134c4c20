"""fp64 CPU oracle for exact scaled-dot-product attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never import it, and it imports nothing from them: the two sides share only
the seeded input generators, which hold none of the method's arithmetic.

The arithmetic lives in ``attn_oracle.c`` (plain C, fp64, OpenMP over
independent rows); this module compiles it with gcc on first use and marshals
numpy arrays through ctypes.  Every function here states the passage it
follows:

* allowed pairs: per-token sequence id and in-sequence position, top-left
  ``j <= i`` or bottom-right ``j <= i + Nk - Nq`` ("causal-mask-and-ragged-
  sequence-layouts", first and third paragraphs), optionally bounded to the
  last ``window`` keys up to that causal bound (``window > 0``; the bounded
  window of "attention-algorithm-error-and-complexity-tests", fifth
  paragraph), optionally a linear positional bias -slope_h |i + off - j|
  on every allowed logit (``slopes``), and optionally an explicit bias
  tensor ``bias`` [B or 1, Hq or 1, rows, keys] added to the allowed logits,
  whose -inf entries remove pairs (same page, third paragraph: bias and mask
  terms enter the logits before the softmax);
* forward: two-pass stable softmax over the allowed set, empty rows give
  O = 0 and lse = -inf (same page, fourth paragraph; "formal-correctness",
  "The FlashAttention Proof", online recurrence equals recomputed softmax);
* backward: recompute form with K/V repeated per query head and gradients
  summed over each group ("attention-algorithm-error-and-complexity-tests",
  third and fourth paragraphs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MASK_NONE = 0
MASK_TOP_LEFT = 1
MASK_BOTTOM_RIGHT = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "libattn_oracle.so")
_lock = threading.Lock()

_I32 = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.POINTER(ctypes.c_int64)
_F64 = ctypes.POINTER(ctypes.c_double)
_U8 = ctypes.POINTER(ctypes.c_uint8)


def compile_library(src: str = _SRC, out: str = _LIB) -> str:
    """Compile the C oracle with gcc (strict IEEE fp64: no fast-math, no FMA
    contraction, so x86 and Arm builds round identically)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """Build the oracle library if it is missing or older than its source."""
    with _lock:
        if (not os.path.exists(_LIB)
                or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)):
            compile_library()
    return _LIB


def _ptr(a: np.ndarray, typ):
    return a.ctypes.data_as(typ)


def _f64(x) -> np.ndarray:
    """Any float array (fp32 / bf16 values held as fp32, fp64) -> contiguous
    fp64.  bf16 and fp32 values are exact in fp64."""
    if hasattr(x, "detach"):  # a torch tensor on the CPU
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


_keep = []  # slope arrays handed to the C library stay alive until process exit


def _slopes(slopes, hq: int):
    """NULL, or a pointer to ``hq`` fp64 slopes."""
    if slopes is None:
        return None
    a = _f64(slopes).reshape(-1)
    if a.shape[0] != hq:
        raise ValueError("one slope per query head")
    _keep.append(a)
    if len(_keep) > 64:
        del _keep[:32]
    return _ptr(a, _F64)


def _btab(bias, batch: int, hq: int):
    """(NULL, NULL), or pointers to a bias tensor [Bb, Hb, Mq, Mk] (Bb in
    {1, batch}, Hb in {1, hq}; a dimension of 1 broadcasts) and its sequence,
    head and row strides."""
    if bias is None:
        return None, None
    a = _f64(bias)
    if a.ndim != 4 or a.shape[0] not in (1, batch) or a.shape[1] not in (1, hq):
        raise ValueError("bias tensor must be [1 or B, 1 or Hq, rows, keys]")
    _, hb, mq, mk = a.shape
    st = np.array([0 if a.shape[0] == 1 else hb * mq * mk, 0 if hb == 1 else mq * mk, mk],
                  np.int64)
    _keep.extend([a, st])
    if len(_keep) > 64:
        del _keep[:32]
    return _ptr(a, _F64), _ptr(st, _I64)


class Oracle:
    """ctypes front end to one compiled copy of ``attn_oracle.c``.

    ``Oracle()`` uses the package's own build; tests that plant a mistake in a
    copy of the source load that copy through ``Oracle(path)``.
    """

    def __init__(self, lib_path: str | None = None):
        self.lib = ctypes.CDLL(lib_path or build())
        L = self.lib
        L.oracle_token_meta.argtypes = [_I32, ctypes.c_int, ctypes.c_int, _I32, _I32]
        L.oracle_token_meta.restype = ctypes.c_int
        L.oracle_mask.argtypes = [_I32, _I32, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, _U8]
        L.oracle_mask.restype = ctypes.c_int
        common = [_F64, _F64, _F64]
        sizes = ([_I32, _I32] + [ctypes.c_int] * 6
                 + [ctypes.c_double, ctypes.c_int, ctypes.c_int, _F64, _F64, _I64])
        L.oracle_fwd.argtypes = common + sizes + [_I64, ctypes.c_int64, _F64, _F64]
        L.oracle_fwd.restype = ctypes.c_int
        L.oracle_bwd.argtypes = common + [_F64] + sizes + [_F64] * 5
        L.oracle_bwd.restype = ctypes.c_int
        L.oracle_bwd_sampled.argtypes = (common + [_F64] + sizes
                                         + [_I64, ctypes.c_int64, _F64,
                                            _I64, ctypes.c_int64, _F64, _F64])
        L.oracle_bwd_sampled.restype = ctypes.c_int

    # -- mask ---------------------------------------------------------------
    def token_meta(self, cu_seqlens, total: int):
        """(seq_id, pos) of every packed token; tokens map to the segment that
        contains them and positions restart at 0 in each segment."""
        cu = _i32(cu_seqlens)
        sid = np.empty(max(total, 1), np.int32)
        pos = np.empty(max(total, 1), np.int32)
        rc = self.lib.oracle_token_meta(_ptr(cu, _I32), len(cu) - 1, total,
                                        _ptr(sid, _I32), _ptr(pos, _I32))
        if rc != 0:
            raise ValueError("invalid cu_seqlens")
        return sid[:total], pos[:total]

    def mask(self, cu_q, cu_k, total_q: int, total_k: int, mask_kind: int,
             window: int = 0):
        """The materialised packed mask, uint8 [total_q, total_k]."""
        cq, ck = _i32(cu_q), _i32(cu_k)
        m = np.zeros((total_q, total_k), np.uint8)
        rc = self.lib.oracle_mask(_ptr(cq, _I32), _ptr(ck, _I32), len(cq) - 1,
                                  total_q, total_k, mask_kind, int(window),
                                  _ptr(m, _U8))
        if rc != 0:
            raise ValueError("invalid mask arguments")
        return m[:total_q, :total_k]

    # -- forward ------------------------------------------------------------
    def fwd(self, q, k, v, cu_q, cu_k, scale: float, mask_kind: int, rows=None,
            window: int = 0, slopes=None, bias=None):
        """Forward.  q [Tq, Hq, d], k/v [Tk, Hkv, d].

        rows None -> (o [Tq, Hq, d], lse [Hq, Tq]); rows = int array [n, 2] of
        (token, head) -> (o [n, d], lse [n]).
        """
        q, k, v = _f64(q), _f64(k), _f64(v)
        cq, ck = _i32(cu_q), _i32(cu_k)
        tq, hq, d = q.shape
        tk, hkv, _ = k.shape
        if rows is None:
            o = np.zeros((tq, hq, d))
            lse = np.zeros((hq, tq))
            rp, n = None, 0
        else:
            rows = np.ascontiguousarray(np.asarray(rows, np.int64).reshape(-1, 2))
            n = rows.shape[0]
            o = np.zeros((max(n, 1), d))
            lse = np.zeros(max(n, 1))
            rp = _ptr(rows, _I64)
        rc = self.lib.oracle_fwd(_ptr(q, _F64), _ptr(k, _F64), _ptr(v, _F64),
                                 _ptr(cq, _I32), _ptr(ck, _I32), len(cq) - 1,
                                 tq, tk, hq, hkv, d, float(scale), mask_kind,
                                 int(window), _slopes(slopes, hq), *_btab(bias, len(cq) - 1, hq),
                                 rp, n, _ptr(o, _F64),
                                 _ptr(lse, _F64))
        if rc != 0:
            raise ValueError("invalid oracle_fwd arguments")
        if rows is not None:
            return o[:n], lse[:n]
        return o, lse

    # -- backward -----------------------------------------------------------
    def bwd(self, q, k, v, dout, cu_q, cu_k, scale: float, mask_kind: int,
            window: int = 0, slopes=None, bias=None):
        """Full backward -> (dq, dk, dv, o, lse), fp64."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        cq, ck = _i32(cu_q), _i32(cu_k)
        tq, hq, d = q.shape
        tk, hkv, _ = k.shape
        dq = np.zeros((tq, hq, d))
        dk = np.zeros((tk, hkv, d))
        dv = np.zeros((tk, hkv, d))
        o = np.zeros((tq, hq, d))
        lse = np.zeros((hq, tq))
        rc = self.lib.oracle_bwd(_ptr(q, _F64), _ptr(k, _F64), _ptr(v, _F64),
                                 _ptr(dout, _F64), _ptr(cq, _I32), _ptr(ck, _I32),
                                 len(cq) - 1, tq, tk, hq, hkv, d, float(scale),
                                 mask_kind, int(window), _slopes(slopes, hq),
                                 *_btab(bias, len(cq) - 1, hq), _ptr(dq, _F64),
                                 _ptr(dk, _F64),
                                 _ptr(dv, _F64), _ptr(o, _F64), _ptr(lse, _F64))
        if rc != 0:
            raise ValueError("invalid oracle_bwd arguments")
        return dq, dk, dv, o, lse

    def bwd_sampled(self, q, k, v, dout, cu_q, cu_k, scale: float,
                    mask_kind: int, q_rows, k_rows, window: int = 0, slopes=None,
                    bias=None):
        """dQ at sampled (token, head) rows and dK, dV at sampled
        (key token, kv head) rows -> (dq [nq, d], dk [nk, d], dv [nk, d])."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        cq, ck = _i32(cu_q), _i32(cu_k)
        tq, hq, d = q.shape
        tk, hkv, _ = k.shape
        qr = np.ascontiguousarray(np.asarray(q_rows, np.int64).reshape(-1, 2))
        kr = np.ascontiguousarray(np.asarray(k_rows, np.int64).reshape(-1, 2))
        dq = np.zeros((max(len(qr), 1), d))
        dk = np.zeros((max(len(kr), 1), d))
        dv = np.zeros((max(len(kr), 1), d))
        rc = self.lib.oracle_bwd_sampled(
            _ptr(q, _F64), _ptr(k, _F64), _ptr(v, _F64), _ptr(dout, _F64),
            _ptr(cq, _I32), _ptr(ck, _I32), len(cq) - 1, tq, tk, hq, hkv, d,
            float(scale), mask_kind, int(window), _slopes(slopes, hq),
            *_btab(bias, len(cq) - 1, hq), _ptr(qr, _I64), len(qr),
            _ptr(dq, _F64),
            _ptr(kr, _I64), len(kr), _ptr(dk, _F64), _ptr(dv, _F64))
        if rc != 0:
            raise ValueError("invalid oracle_bwd_sampled arguments")
        return dq[:len(qr)], dk[:len(kr)], dv[:len(kr)]


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def fwd(*a, **kw):
    return default().fwd(*a, **kw)


def bwd(*a, **kw):
    return default().bwd(*a, **kw)


def bwd_sampled(*a, **kw):
    return default().bwd_sampled(*a, **kw)


def mask(*a, **kw):
    return default().mask(*a, **kw)


def token_meta(*a, **kw):
    return default().token_meta(*a, **kw)
