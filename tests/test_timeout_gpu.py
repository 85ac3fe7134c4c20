"""Bounded device waits that run out, on every tensor-core kernel.

Every wait inside the kernels is bounded; attn_set_wait_limit_ns lowers the
bound for the calls after it.  Below 1000 ns a wait gives up as soon as its
condition is not already met, so each call below times out in its first
block that waits for anything, with nothing broken: every copy and product
the kernels issue is valid and completes.  The blocks that gave up drain
their copies and products in flight before they free their tensor memory,
the device flag reads ATTN_ERR_DEVICE_TIMEOUT, and the same process then
computes correct results with the default bound.  (The pages say nothing on
failure handling; this is the library's own contract.)
"""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import backward_form

pytestmark = pytest.mark.gpu
TL, BR = inputs.MASK_TOP_LEFT, inputs.MASK_BOTTOM_RIGHT
TIMEOUT = 5

CALLS = [  # (name, lq, lk, hq, hkv, mask, backward, plan substring)
    ("prefill", (300, 129), (300, 129), 8, 2, TL, False, "fwd_tc2"),
    ("decode_split", (1,) * 4, (9000, 4097, 300, 6000), 32, 8, BR, False, "splits="),
    ("backward", (300, 129), (300, 129), 8, 2, TL, True, "bwd_fused_tc"),
    ("backward_two_kernel", (300, 129), (300, 129), 8, 2, TL, "two_kernel", "bwd_dkdv_tc"),
    ("backward_plain", (300, 129), (300, 129), 8, 2, TL, "plain", "fwd_tc2_delta"),
]


def _call(x, backward):
    with backward_form(backward == "two_kernel"):
        return _call_form(x, backward)


def _call_form(x, backward):
    w = x["workload"]
    d = x
    keep = backward is True or backward == "two_kernel"
    res = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                   w.max_k, w.mask, w.scale, want_o_f32=keep)
    grads = None
    if backward:
        grads = attn.bwd(d["q"], d["k"], d["v"], res[0], res[1], d["dout"], d["cu_seqlens_q"],
                         d["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale,
                         o_f32=res[2] if keep else None)
    return res, grads, attn.last_plan()


@pytest.mark.parametrize("case", CALLS, ids=[c[0] for c in CALLS])
def test_expired_wait_reports_and_recovers(case):
    name, lq, lk, hq, hkv, mask, backward, plan_part = case
    w = inputs.custom(name, lq, lk, hq, hkv, 128, "bf16", mask, seed=81,
                      backward=bool(backward), v_shift_per_seq=2.0)
    x = inputs.make_inputs(w, device="cuda")
    assert attn.get_device_error() == 0
    attn.set_wait_limit_ns(1)
    try:
        _, _, plan = _call(x, backward)
        assert plan_part in plan, plan
        assert attn.get_device_error() == TIMEOUT
    finally:
        attn.set_wait_limit_ns(0)  # the default bound again
    # same process, default bound: clean flag and results within the contract
    (o, lse, *_), grads, _ = _call(x, backward)
    assert attn.get_device_error() == 0
    host = {k: (t.cpu() if hasattr(t, "cpu") else t) for k, t in x.items()}
    if backward:
        rdq, rdk, rdv, ro, rlse = oracle.bwd(host["q"], host["k"], host["v"], host["dout"],
                                             host["cu_seqlens_q"], host["cu_seqlens_k"],
                                             w.scale, mask)
        for nm, got, ref in zip(("dq", "dk", "dv"), grads, (rdq, rdk, rdv)):
            compare.check_close(nm, got, ref)
    else:
        ro, rlse = oracle.fwd(host["q"], host["k"], host["v"], host["cu_seqlens_q"],
                              host["cu_seqlens_k"], w.scale, mask)
    compare.check_close("o", o, ro)
    compare.check_lse("lse", lse, rlse)


def test_many_expired_calls_leave_the_device_usable():
    """Repeated timeouts in a row (every block of a large grid giving up and
    draining) followed by a normal call: the device still computes the right
    answer, so no block freed tensor memory or exited with work in flight
    that a later block could see."""
    w = inputs.custom("many", (2048,) * 4, (2048,) * 4, 16, 4, 128, "bf16", TL, seed=82)
    x = inputs.make_inputs(w, device="cuda")
    attn.set_wait_limit_ns(1)
    try:
        for _ in range(5):
            _call(x, False)
        assert attn.get_device_error() == TIMEOUT
    finally:
        attn.set_wait_limit_ns(0)
    (o, lse, *_), _, _ = _call(x, False)
    assert attn.get_device_error() == 0
    rows = np.array([(0, 0), (2047, 3), (4096 + 1000, 15), (8191, 7)], np.int64)
    host = {k: (t.cpu() if hasattr(t, "cpu") else t) for k, t in x.items()}
    ro, rlse = oracle.fwd(host["q"], host["k"], host["v"], host["cu_seqlens_q"],
                          host["cu_seqlens_k"], w.scale, w.mask, rows=rows)
    on, ln = compare.to_np(o), compare.to_np(lse)
    compare.check_close("o", on[rows[:, 0], rows[:, 1]], ro)
    compare.check_lse("lse", ln[rows[:, 1], rows[:, 0]], rlse)


def test_expired_wait_staged_bias_reports_and_recovers():
    """The prefill with a head-shared bias tensor streamed through shared
    memory (warp 2 copying each key tile's entries): the same expiry, drain
    (the entries' copies included) and recovery."""
    w = inputs.custom("tmo_bias", (300, 129), (300, 129), 8, 2, 128, "bf16", TL, seed=82)
    x = inputs.make_inputs(w, device="cuda")
    bias = inputs.bias_tensor(w.batch, 1, w.max_q, w.max_k, seed=83).cuda()
    args = (x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.max_q, w.max_k, TL,
            w.scale)
    assert attn.get_device_error() == 0
    attn.set_wait_limit_ns(1)
    try:
        attn.fwd(*args, bias=bias)
        assert "_btab_smem" in attn.last_plan(), attn.last_plan()
        assert attn.get_device_error() == TIMEOUT
    finally:
        attn.set_wait_limit_ns(0)
    o, lse = attn.fwd(*args, bias=bias)
    assert attn.get_device_error() == 0
    host = {k: (t.cpu() if hasattr(t, "cpu") else t) for k, t in x.items()}
    ro, rlse = oracle.fwd(host["q"], host["k"], host["v"], host["cu_seqlens_q"],
                          host["cu_seqlens_k"], w.scale, TL, bias=bias.cpu())
    compare.check_close("o", o, ro)
    compare.check_lse("lse", lse, rlse)
