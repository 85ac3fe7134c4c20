"""attn_fwd_static_scratch: the forward for callers that cannot allocate.

Some callers cannot give the library a workspace: plug-ins inside a host
runtime that owns a fixed device-memory plan and exposes no allocator, and
serving loops where a cudaMalloc (which may synchronise the device or fail
under memory pressure) is not allowed once they run.  For them the library
keeps the split-KV decode's partial outputs in a static device array of its
own.  This test calls that entry point through the C ABI and checks it
against attn_fwd with a caller workspace, twice in a row (the array keeps
the previous call's contents), and checks that a problem too large for the
array is refused before anything runs.

The file name makes pytest collect it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT_STATUS = 7


def _entry():
    lib = attn.library()
    f = lib.attn_fwd_static_scratch
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P] * 8 + [I] * 8 + [F, I, I, P, I, P]
    f.restype = I
    return f


def _call_static(x, w, o, lse, o32):
    f = _entry()
    return f(x["q"].data_ptr(), x["k"].data_ptr(), x["v"].data_ptr(), o.data_ptr(),
             lse.data_ptr(), o32.data_ptr(), x["cu_seqlens_q"].data_ptr(),
             x["cu_seqlens_k"].data_ptr(), w.batch, w.max_q, w.max_k, w.total_q, w.total_k,
             w.hq, w.hkv, w.d, w.scale, w.mask, w.window, None, attn.DTYPE_BF16,
             torch.cuda.current_stream().cuda_stream)


CASES = [  # decode-like shapes that take the split-KV plan
    ("q1", (1,) * 8, (4096, 3000, 129, 4096, 1, 777, 4096, 2048)),
    ("q16", (16,) * 4, (8192, 5000, 16, 300)),
]


@pytest.mark.parametrize("name,lq,lk", CASES, ids=[c[0] for c in CASES])
def test_static_scratch_matches_workspace_forward(name, lq, lk):
    w = inputs.custom(name, lq, lk, 32, 8, 128, "bf16", inputs.MASK_BOTTOM_RIGHT, seed=21)
    x = inputs.make_inputs(w, device="cuda")
    ref_o, ref_lse, ref_o32 = attn.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                                       x["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale,
                                       want_o_f32=True)
    assert "splits=" in attn.last_plan() and "+combine" in attn.last_plan()
    for call in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        o32 = torch.full_like(ref_o32, float("nan"))
        assert _call_static(x, w, o, lse, o32) == 0, f"call {call}"
        torch.cuda.synchronize()
        assert attn.get_device_error() == 0
        assert "static scratch" in attn.last_plan()
        compare.check_close(f"o call {call}", o, ref_o)
        compare.check_close(f"o_f32 call {call}", o32, ref_o32)
        compare.check_lse(f"lse call {call}", lse, ref_lse)


FALLTHROUGH = [  # shapes whose plan keeps nothing in the array: (name, lq, lk, mask)
    ("no_query_rows", (0, 0), (2048, 4096), inputs.MASK_BOTTOM_RIGHT),
    ("no_keys", (5, 3), (0, 0), inputs.MASK_BOTTOM_RIGHT),
    ("q_longer_than_k", (64, 64), (32, 32), inputs.MASK_BOTTOM_RIGHT),
    ("prefill", (300, 129), (300, 129), inputs.MASK_TOP_LEFT),
]


@pytest.mark.parametrize("name,lq,lk,mask", FALLTHROUGH, ids=[c[0] for c in FALLTHROUGH])
def test_static_scratch_without_split(name, lq, lk, mask):
    """Calls that do not take the split plan (no query rows, no keys, a
    non-split prefill, Nq > Nk bottom-right) give attn_fwd's results; rows
    with no allowed key get exact zeros and lse = -inf."""
    w = inputs.custom(name, lq, lk, 32, 8, 128, "bf16", mask, seed=23)
    x = inputs.make_inputs(w, device="cuda")
    ref_o, ref_lse, ref_o32 = attn.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                                       x["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale,
                                       want_o_f32=True)
    assert "splits=" not in attn.last_plan() or "splits=1" in attn.last_plan()
    for call in range(2):
        o = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        o32 = torch.full_like(ref_o32, float("nan"))
        assert _call_static(x, w, o, lse, o32) == 0, f"call {call}"
        torch.cuda.synchronize()
        assert attn.get_device_error() == 0
        compare.check_close(f"o call {call}", o, ref_o)
        compare.check_close(f"o_f32 call {call}", o32, ref_o32)
        compare.check_lse(f"lse call {call}", lse, ref_lse)
        empty = torch.isneginf(lse)
        if name in ("no_keys", "q_longer_than_k"):
            assert empty.any()
        if empty.any():
            rows = empty.t().nonzero()  # (token, head) of every empty row
            assert torch.count_nonzero(o[rows[:, 0], rows[:, 1]]) == 0
            assert torch.count_nonzero(o32[rows[:, 0], rows[:, 1]]) == 0


def test_static_scratch_refuses_oversize_problem():
    # 64 sequences x 8 queries x 128 query heads against 64k keys: the split
    # plan's partial outputs would need about 100 MB, over the 64 MiB array.
    lq, lk = (8,) * 64, (65536,) * 64
    w = inputs.custom("big", lq, lk, 128, 8, 128, "bf16", inputs.MASK_BOTTOM_RIGHT, seed=2)
    ws = attn.fwd_workspace_size(w.batch, w.max_q, w.max_k, w.total_q, w.hq, w.hkv, w.d,
                                 attn.DTYPE_BF16)
    if ws <= (64 << 20):
        pytest.skip("this GPU's plan for the shape fits the static array")
    q = torch.zeros((w.total_q, w.hq, w.d), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, w.hkv, w.d), dtype=torch.bfloat16, device="cuda")
    x = {"q": q, "k": kv, "v": kv,
         "cu_seqlens_q": inputs.cu_seqlens(lq).cuda(), "cu_seqlens_k": inputs.cu_seqlens(lk).cuda()}
    o = torch.empty_like(q)
    lse = torch.empty((w.hq, w.total_q), dtype=torch.float32, device="cuda")
    o32 = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    # sizes only: the call must refuse before touching any buffer
    assert _call_static(x, w, o, lse, o32) == SCRATCH_LIMIT_STATUS
    assert attn.status_string(SCRATCH_LIMIT_STATUS)
