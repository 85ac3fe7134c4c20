"""The backward as most callers make it, against the fp64 oracle:

* without the forward's fp32 output (``o_f32`` NULL), on value rows with
  large common offsets per sequence, so that a D term formed from the
  bf16-rounded O would miss the contract ("attention-algorithm-error-and-
  complexity-tests", fourth paragraph: gradient checks that catch a missing
  or wrong denominator term in the backward), with every mask kind, a
  window, the linear positional bias and an explicit bias tensor, and on the
  full-size training workload at sampled rows;
* on inputs scaled far from unit magnitude (exact powers of two in bf16),
  with the gradients compared after scaling them back by the matching power
  of two, so that the absolute part of the tolerance cannot hide a loss of
  precision in the backward's fp16 operands (same page, second paragraph:
  a tolerance must not hide errors).
"""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import sample_rows, tc_backward

pytestmark = pytest.mark.gpu
TL, BR, NONE = inputs.MASK_TOP_LEFT, inputs.MASK_BOTTOM_RIGHT, inputs.MASK_NONE


def run(x, keep_o32, slopes=None, bias=None):
    w = x["workload"]
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    sl = None if slopes is None else slopes.cuda()
    b = None if bias is None else bias.cuda()
    res = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                   w.max_k, w.mask, w.scale, want_o_f32=keep_o32, window=w.window,
                   bias_slopes=sl, bias=b)
    o, lse = res[0], res[1]
    o32 = res[2] if keep_o32 else None
    dq, dk, dv = attn.bwd(d["q"], d["k"], d["v"], o, lse, d["dout"], d["cu_seqlens_q"],
                          d["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale, o_f32=o32,
                          window=w.window, bias_slopes=sl, bias=b)
    plan = attn.last_plan()
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    return (o, lse, dq, dk, dv), plan


CASES = [  # (name, lq, lk, hq, hkv, d, mask, v shift per sequence, window, bias kind)
    ("packed_shift10", (1, 63, 64, 65, 127, 128, 129, 255, 256, 257), None, 8, 8, 128, TL, 10.0,
     0, None),
    ("ragged_gqa4_shift2", (63, 129, 1, 200), None, 8, 2, 128, TL, 2.0, 0, None),
    ("ragged_gqa4_shift10", (63, 129, 1, 200), None, 8, 2, 128, TL, 10.0, 0, None),
    ("br_empty_rows_shift10", (64, 10), (32, 300), 4, 1, 128, BR, 10.0, 0, None),
    ("noncausal_d64_shift10", (100, 37), (50, 260), 4, 4, 64, NONE, 10.0, 0, None),
    ("window_shift10", (300, 129), None, 8, 2, 128, TL, 10.0, 64, None),
    ("slopes_shift10", (300, 50), (700, 40), 4, 2, 128, BR, 10.0, 0, "slopes"),
    ("bias_tensor_shift10", (63, 129, 1, 200), None, 8, 2, 128, TL, 10.0, 0, "tensor"),
    # one set of entries per sequence shared by the heads: staged through
    # shared memory in the recomputing forward
    ("bias_shared_shift10", (63, 129, 1, 200), None, 8, 2, 128, TL, 10.0, 0, "shared"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_without_o_f32(case):
    """attn_bwd with o_f32 = NULL: the library recomputes D from the fp32
    output (plan names fwd_tc2_delta); every gradient meets the contract."""
    name, lq, lk, hq, hkv, d, mask, shift, window, kind = case
    w = inputs.custom(name, lq, lk or lq, hq, hkv, d, "bf16", mask, seed=71, backward=True,
                      v_shift_per_seq=shift, window=window)
    x = inputs.make_inputs(w)
    slopes = inputs.bias_slopes(hq) if kind == "slopes" else None
    bias = inputs.bias_tensor(w.batch, 1 if kind == "shared" else hq, w.max_q, w.max_k, seed=72,
                              dead_rows=2) if kind in ("tensor", "shared") else None
    (o, lse, dq, dk, dv), plan = run(x, False, slopes, bias)
    assert "fwd_tc2_delta" in plan and tc_backward(plan), plan
    rdq, rdk, rdv, ro, rlse = oracle.bwd(
        x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.scale, mask,
        window=window, slopes=None if slopes is None else slopes.double().numpy(), bias=bias)
    stats = {}
    compare.check_close("o", o, ro, stats=stats)
    compare.check_lse("lse", lse, rlse, stats=stats)
    compare.check_close("dq", dq, rdq, stats=stats)
    compare.check_close("dk", dk, rdk, stats=stats)
    compare.check_close("dv", dv, rdv, stats=stats)
    for h, t in np.argwhere(np.isneginf(rlse)):
        assert np.all(compare.to_np(dq)[t, h] == 0.0)


def test_without_o_f32_equals_with_it_closely():
    """Both D routes form D from an fp32 output normalised by the rounded
    probability sum (only the fp32 summation order differs), so their
    gradients agree to one bf16 rounding step, far inside the contract."""
    w = inputs.custom("d_routes", (200, 77, 300), (200, 77, 300), 8, 2, 128, "bf16", TL, seed=73,
                      backward=True, v_shift_per_seq=10.0)
    x = inputs.make_inputs(w)
    (_, _, dq0, dk0, dv0), p0 = run(x, False)
    (_, _, dq1, dk1, dv1), p1 = run(x, True)
    assert "fwd_tc2_delta" in p0 and "fwd_tc2_delta" not in p1
    for a, b in ((dq0, dq1), (dk0, dk1), (dv0, dv1)):
        compare.check_close("routes", a, b, atol=1e-3, rtol=2.0 ** -7)  # one bf16 step


def test_train_full_size_sampled_without_o_f32():
    w = inputs.WORKLOADS["train_fwd_bwd"]
    x = inputs.make_inputs(w)
    (o, lse, dq, dk, dv), plan = run(x, False)
    assert "fwd_tc2_delta" in plan
    qrows = sample_rows(w, 24, seed=18)
    rng = np.random.default_rng(19)
    krows = [(0, 0), (3, 2), (8191, 1), (8192, 3), (8192 + 7000, 0)]
    krows += [(int(rng.integers(16384 - 300, 16384)), int(rng.integers(4))) for _ in range(6)]
    krows = np.array(krows, np.int64)
    rdq, rdk, rdv = oracle.bwd_sampled(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                       x["cu_seqlens_k"], w.scale, w.mask, qrows, krows)
    dqn, dkn, dvn = compare.to_np(dq), compare.to_np(dk), compare.to_np(dv)
    compare.check_close("dq", dqn[qrows[:, 0], qrows[:, 1]], rdq)
    compare.check_close("dk", dkn[krows[:, 0], krows[:, 1]], rdk)
    compare.check_close("dv", dvn[krows[:, 0], krows[:, 1]], rdv)


MAGNITUDES = [-26, -18, 6]  # log2 of the common input scale


@pytest.mark.parametrize("keep_o32", [True, False], ids=["o_f32", "no_o_f32"])
@pytest.mark.parametrize("e", MAGNITUDES, ids=[f"2^{e}" for e in MAGNITUDES])
def test_backward_input_magnitude(e, keep_o32):
    """Q, K, V and dO all scaled by 2^e (exact in bf16).  O and dV scale like
    V and dO (2^e), dQ and dK like dS times Q or K (2^3e); each is compared
    with the oracle after multiplying both sides by the inverse power of two,
    so the contract is applied at unit magnitude.  Unscaled fp16 copies
    would make these inputs subnormal or zero (2^-18 keeps about 6 of the 8
    significant bits, 2^-26 none)."""
    w = inputs.custom("mag", (63, 129, 200), (63, 129, 200), 8, 2, 128, "bf16", TL, seed=74, backward=True,
                      v_shift_per_seq=1.0)
    x = inputs.make_inputs(w)
    f = 2.0 ** e
    for name in ("q", "k", "v", "dout"):
        x[name] = (x[name].double() * f).to(torch.bfloat16)
    (o, lse, dq, dk, dv), plan = run(x, keep_o32)
    assert tc_backward(plan), plan
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, w.mask)
    u1, u3 = 2.0 ** -e, 2.0 ** (-3 * e)
    compare.check_close("o", compare.to_np(o) * u1, ro * u1)
    compare.check_lse("lse", lse, rlse)
    compare.check_close("dv", compare.to_np(dv) * u1, rdv * u1)
    compare.check_close("dq", compare.to_np(dq) * u3, rdq * u3)
    compare.check_close("dk", compare.to_np(dk) * u3, rdk * u3)


def test_nonfinite_backward_input_is_reported():
    """An infinity in dO is outside the contract; the backward reports it
    through the device flag (ATTN_ERR_DEVICE_RANGE) instead of returning
    silently wrong gradients."""
    w = inputs.custom("inf", (70,), (70,), 4, 2, 128, "bf16", TL, seed=75, backward=True)
    x = inputs.make_inputs(w)
    x["dout"][5, 1, 7] = float("inf")
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    o, lse = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                      w.max_k, w.mask, w.scale)
    assert attn.get_device_error() == 0
    attn.bwd(d["q"], d["k"], d["v"], o, lse, d["dout"], d["cu_seqlens_q"], d["cu_seqlens_k"],
             w.max_q, w.max_k, w.mask, w.scale)
    assert attn.get_device_error() == 8
    assert attn.get_device_error() == 0  # cleared by the read
