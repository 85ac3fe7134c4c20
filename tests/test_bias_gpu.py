"""Linear positional bias -slope_h |i + off - j| on the GPU against the fp64
oracle, forward and backward, on every kernel plan ("attention-algorithm-
error-and-complexity-tests", third paragraph; "causal-mask-and-ragged-
sequence-layouts", sixth paragraph: the backward rebuilds the same bias)."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import sample_rows

pytestmark = pytest.mark.gpu
TL, BR, NONE = inputs.MASK_TOP_LEFT, inputs.MASK_BOTTOM_RIGHT, inputs.MASK_NONE


def geometric_slopes(hq):
    return inputs.bias_slopes(hq)


def run(x, slopes, backward=False):
    w = x["workload"]
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    sl = slopes.cuda()
    o, lse, o32 = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                           w.max_k, w.mask, w.scale, want_o_f32=True, window=w.window,
                           bias_slopes=sl)
    plan = attn.last_plan()
    grads = None
    if backward:
        grads = attn.bwd(d["q"], d["k"], d["v"], o, lse, d["dout"], d["cu_seqlens_q"],
                         d["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale, o_f32=o32,
                         window=w.window, bias_slopes=sl)
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    return o, lse, grads, plan


FWD = [  # (name, lq, lk, hq, hkv, d, dtype, mask, window, plan substring)
    ("prefill_tl", (300, 1, 129, 700), None, 8, 2, 128, "bf16", TL, 0, "fwd_tc2"),
    ("prefill_br", (300, 50), (700, 40), 4, 2, 128, "bf16", BR, 0, "fwd_tc2"),
    ("prefill_none_d64", (200, 77), (150, 300), 4, 4, 64, "bf16", NONE, 0, "fwd_tc2"),
    ("prefill_tl_window", (640, 100), None, 4, 1, 128, "bf16", TL, 200, "fwd_tc2"),
    ("decode_split", (1,) * 6, (9000, 129, 1, 3000, 12000, 5000), 32, 8, 128, "bf16", BR, 0, "splits="),
    ("decode_q16", (16,) * 3, (4000, 16, 600), 32, 8, 128, "bf16", BR, 0, "fwd_tc_"),
    ("fp32", (90, 33), (90, 40), 4, 2, 64, "fp32", BR, 0, "fwd_simt"),
]


@pytest.mark.parametrize("case", FWD, ids=[c[0] for c in FWD])
def test_bias_forward_full(case):
    name, lq, lk, hq, hkv, d, dt, mask, window, plan = case
    w = inputs.custom(name, lq, lk or lq, hq, hkv, d, dt, mask, seed=51, v_shift_per_seq=3.0,
                      window=window)
    x = inputs.make_inputs(w)
    sl = geometric_slopes(hq)
    o, lse, _, got_plan = run(x, sl)
    assert plan in got_plan, got_plan
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.scale,
                        mask, window=window, slopes=sl.double().numpy())
    tol = {} if dt == "bf16" else {"atol": 1e-4, "rtol": 1e-4}
    compare.check_close("o", o, ro, **tol)
    compare.check_lse("lse", lse, rl)


BWD = [  # (name, lq, lk, hq, hkv, d, dtype, mask, window)
    ("tc_tl", (300, 129), (300, 129), 4, 2, 128, "bf16", TL, 0),
    ("tc_br", (300, 50), (700, 40), 4, 1, 128, "bf16", BR, 0),
    ("tc_none_d64", (200, 77), (150, 300), 4, 4, 64, "bf16", NONE, 0),
    ("tc_tl_window", (320, 65), (320, 65), 8, 2, 128, "bf16", TL, 100),
    ("simt_fp32", (40, 70), (50, 70), 4, 2, 64, "fp32", BR, 0),
]


@pytest.mark.parametrize("case", BWD, ids=[c[0] for c in BWD])
def test_bias_backward_full(case):
    name, lq, lk, hq, hkv, d, dt, mask, window = case
    w = inputs.custom(name, lq, lk, hq, hkv, d, dt, mask, seed=53, backward=True,
                      v_shift_per_seq=2.0, window=window)
    x = inputs.make_inputs(w)
    sl = geometric_slopes(hq)
    o, lse, (dq, dk, dv), _ = run(x, sl, backward=True)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, mask, window=window,
                                         slopes=sl.double().numpy())
    tol = {} if dt == "bf16" else {"atol": 1e-4, "rtol": 1e-4}
    compare.check_close("o", o, ro, **tol)
    compare.check_lse("lse", lse, rlse)
    compare.check_close("dq", dq, rdq, **tol)
    compare.check_close("dk", dk, rdk, **tol)
    compare.check_close("dv", dv, rdv, **tol)


def test_bias_prefill_full_size_sampled():
    """The prefill benchmark's shape (4 x 4096 tokens, 32 / 8 heads) with
    geometric slopes, on sampled rows."""
    base = inputs.WORKLOADS["gqa_prefill"]
    w = inputs.custom("gqa_prefill_bias", base.seqlens_q, base.seqlens_k, base.hq, base.hkv,
                      base.d, "bf16", TL, seed=base.seed)
    x = inputs.make_inputs(w)
    sl = geometric_slopes(w.hq)
    o, lse, _, _ = run(x, sl)
    rows = sample_rows(w, 48, seed=6)
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.scale,
                        TL, rows=rows, slopes=sl.double().numpy())
    on, ln = compare.to_np(o), compare.to_np(lse)
    compare.check_close("o", on[rows[:, 0], rows[:, 1]], ro)
    compare.check_lse("lse", ln[rows[:, 1], rows[:, 0]], rl)


def test_zero_slopes_match_no_bias():
    """All-zero slopes take the bias kernels and agree with the plain ones
    within the bf16 contract."""
    w = inputs.custom("zero_slopes", (300, 129), (300, 129), 4, 2, 128, "bf16", TL, seed=55,
                      backward=True)
    x = inputs.make_inputs(w)
    o0, lse0, g0, _ = run(x, torch.zeros(w.hq), backward=True)
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    o1, lse1, o32 = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                             w.max_q, w.max_k, w.mask, w.scale, want_o_f32=True)
    g1 = attn.bwd(d["q"], d["k"], d["v"], o1, lse1, d["dout"], d["cu_seqlens_q"],
                  d["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale, o_f32=o32)
    compare.check_close("o", o0, compare.to_np(o1))
    compare.check_lse("lse", lse0, compare.to_np(lse1))
    for a, b in zip(g0, g1):
        compare.check_close("grad", a, compare.to_np(b))
