"""CUDA backward against the fp64 oracle's gradients (dQ, and dK / dV summed
over each KV head's query heads), on small problems in full and on the
full-size training workload at sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import backward_form, sample_rows

pytestmark = pytest.mark.gpu
TL, BR, NONE = inputs.MASK_TOP_LEFT, inputs.MASK_BOTTOM_RIGHT, inputs.MASK_NONE


def run_fwd_bwd(x):
    w = x["workload"]
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    o, lse, o32 = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"],
                           w.max_q, w.max_k, w.mask, w.scale, want_o_f32=True, window=w.window)
    dq, dk, dv = attn.bwd(d["q"], d["k"], d["v"], o, lse, d["dout"], d["cu_seqlens_q"],
                          d["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale, o_f32=o32,
                          window=w.window)
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    return o, lse, dq, dk, dv


CASES = [  # (name, lq, lk, hq, hkv, d, dtype, mask)
    ("tiny_fp32", (64,), (64,), 1, 1, 64, "fp32", TL),
    ("ragged_gqa4", (63, 129, 1, 200), (63, 129, 1, 200), 8, 2, 128, "bf16", TL),
    ("br_empty_rows", (64, 10), (32, 300), 4, 1, 128, "bf16", BR),
    ("noncausal_d64", (100, 37), (50, 260), 4, 4, 64, "bf16", NONE),
    ("zero_length", (0, 33, 0), (5, 33, 0), 2, 1, 64, "bf16", TL),
    ("zero_length_d128", (0, 33, 0, 130), (5, 33, 0, 7), 4, 2, 128, "bf16", BR),
]


FORMS = [False, True]  # fused (the default), two-kernel
FORM_IDS = ["fused", "two_kernel"]


@pytest.mark.parametrize("two_kernel", FORMS, ids=FORM_IDS)
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_full(case, two_kernel):
    name, lq, lk, hq, hkv, d, dt, mask = case
    # value ranges differ per sequence so that leakage shows
    w = inputs.custom(name, lq, lk, hq, hkv, d, dt, mask, seed=17, backward=True,
                      v_shift_per_seq=2.0)
    x = inputs.make_inputs(w)
    with backward_form(two_kernel):
        o, lse, dq, dk, dv = run_fwd_bwd(x)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, mask)
    compare.check_close("o", o, ro)
    compare.check_lse("lse", lse, rlse)
    compare.check_close("dq", dq, rdq)
    compare.check_close("dk", dk, rdk)
    compare.check_close("dv", dv, rdv)
    empty = np.isneginf(rlse)
    for h, t in np.argwhere(empty):
        assert np.all(compare.to_np(dq)[t, h] == 0.0)


@pytest.mark.parametrize("two_kernel", FORMS, ids=FORM_IDS)
def test_train_full_size_sampled(two_kernel):
    w = inputs.WORKLOADS["train_fwd_bwd"]
    x = inputs.make_inputs(w)
    with backward_form(two_kernel):
        o, lse, dq, dk, dv = run_fwd_bwd(x)
        assert ("bwd_dq_tc" if two_kernel else "bwd_fused_tc") in attn.last_plan()
    qrows = sample_rows(w, 24, seed=8)
    rng = np.random.default_rng(9)
    # keys near the start of a sequence are reached by every later query row;
    # keys near the end by few: sample both
    krows = [(0, 0), (5, 1), (8191, 3), (8192, 2), (8192 + 8000, 0)]
    krows += [(int(rng.integers(16384 - 300, 16384)), int(rng.integers(4))) for _ in range(6)]
    krows = np.array(krows, np.int64)
    rdq, rdk, rdv = oracle.bwd_sampled(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                       x["cu_seqlens_k"], w.scale, w.mask, qrows, krows)
    dqn, dkn, dvn = compare.to_np(dq), compare.to_np(dk), compare.to_np(dv)
    compare.check_close("dq", dqn[qrows[:, 0], qrows[:, 1]], rdq)
    compare.check_close("dk", dkn[krows[:, 0], krows[:, 1]], rdk)
    compare.check_close("dv", dvn[krows[:, 0], krows[:, 1]], rdv)
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()


def test_backward_deterministic():
    """Two-kernel form: every gradient row has one owner CTA and no atomics,
    so repeated calls give bit-identical dq, dk, dv."""
    w = inputs.custom("det", (300, 129), (300, 129), 8, 2, 128, "bf16", TL, seed=4, backward=True)
    x = inputs.make_inputs(w)
    with backward_form(True):
        first = run_fwd_bwd(x)
        assert "bwd_dq_tc" in attn.last_plan()
        for _ in range(3):
            again = run_fwd_bwd(x)
            for a, b in zip(first, again):
                assert torch.equal(a, b)


AGREE = [  # (name, lq, lk, hq, hkv, mask, window, bias kind)
    ("ragged_gqa4", (63, 129, 1, 200), None, 8, 2, TL, 0, None),
    ("long_gqa8", (1100, 517), None, 16, 2, TL, 0, None),
    ("br_empty_rows", (64, 10), (32, 300), 4, 1, BR, 0, None),
    ("noncausal", (100, 37), (50, 260), 4, 4, NONE, 0, None),
    ("window", (700, 129), None, 8, 2, TL, 100, None),
    ("slopes", (300, 50), (700, 40), 4, 2, BR, 0, "slopes"),
    ("bias_tensor", (63, 129, 1, 200), None, 8, 2, TL, 0, "tensor"),
]


@pytest.mark.parametrize("case", AGREE, ids=[c[0] for c in AGREE])
def test_fused_matches_two_kernel(case):
    """The fused backward computes dK and dV with the same products in the
    same order as the two-kernel one (bit-identical, and identical from call
    to call); only dQ is summed differently (fp32 reductions across key
    tiles), so it agrees to about one bf16 rounding."""
    name, lq, lk, hq, hkv, mask, window, kind = case
    w = inputs.custom(name, lq, lk or lq, hq, hkv, 128, "bf16", mask, seed=19, backward=True,
                      v_shift_per_seq=2.0, window=window)
    x = inputs.make_inputs(w)
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    sl = inputs.bias_slopes(hq).cuda() if kind == "slopes" else None
    bt = inputs.bias_tensor(w.batch, hq, w.max_q, w.max_k, seed=20, dead_rows=2).cuda() \
        if kind == "tensor" else None
    o, lse, o32 = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                           w.max_k, mask, w.scale, want_o_f32=True, window=window,
                           bias_slopes=sl, bias=bt)

    def grads(two_kernel):
        with backward_form(two_kernel):
            g = attn.bwd(d["q"], d["k"], d["v"], o, lse, d["dout"], d["cu_seqlens_q"],
                         d["cu_seqlens_k"], w.max_q, w.max_k, mask, w.scale, o_f32=o32,
                         window=window, bias_slopes=sl, bias=bt)
            plan = attn.last_plan()
        torch.cuda.synchronize()
        assert attn.get_device_error() == 0
        assert ("bwd_dq_tc" if two_kernel else "bwd_fused_tc") in plan, plan
        return g

    dq2, dk2, dv2 = grads(True)
    dqf, dkf, dvf = grads(False)
    assert torch.equal(dkf, dk2) and torch.equal(dvf, dv2)
    compare.check_close("dq fused vs two-kernel", dqf, compare.to_np(dq2).astype(np.float64),
                        atol=1e-3, rtol=2.0 ** -7)
    dqf2, dkf2, dvf2 = grads(False)
    assert torch.equal(dkf2, dkf) and torch.equal(dvf2, dvf)
    compare.check_close("dq fused repeat", dqf2, compare.to_np(dqf).astype(np.float64),
                        atol=1e-3, rtol=2.0 ** -7)


@pytest.mark.parametrize("mask", [TL, BR, NONE])
def test_backward_fp32_path(mask):
    """fp32 inputs take the CUDA-core backward; it meets the same contract."""
    w = inputs.custom("fp32bwd", (37, 70), (50, 70), 4, 2, 64, "fp32", mask, seed=6, backward=True)
    x = inputs.make_inputs(w)
    o, lse, dq, dk, dv = run_fwd_bwd(x)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, mask)
    for name, got, ref in (("o", o, ro), ("dq", dq, rdq), ("dk", dk, rdk), ("dv", dv, rdv)):
        compare.check_close(name, got, ref, atol=1e-4, rtol=1e-4)


@pytest.mark.parametrize("seed", [101, 102, 103, 104, 105, 106, 107, 108])
def test_fused_backward_random_shapes(seed):
    """Random packed batches for the fused backward (head_dim 128): 1-4
    sequences of 0-400 queries, keys as many (top-left) or independent
    (bottom-right, no mask), GQA groups 1, 2 and 4, a bounded window half of
    the time with a causal rule, value offsets per sequence; every gradient
    against the oracle, empty rows giving zero dQ
    ("causal-mask-and-ragged-sequence-layouts", fourth and fifth paragraphs)."""
    rng = np.random.default_rng(seed)
    batch = int(rng.integers(1, 5))
    mask = [TL, BR, NONE][int(rng.integers(3))]
    lq = [int(x) for x in rng.integers(0, 401, size=batch)]
    lk = lq if mask == TL else [int(x) for x in rng.integers(1, 401, size=batch)]
    hkv = int(rng.choice([1, 2, 4]))
    hq = hkv * int(rng.choice([1, 2, 4]))
    window = int(rng.integers(1, 300)) if mask != NONE and rng.random() < 0.5 else 0
    w = inputs.custom(f"rand{seed}", lq, lk, hq, hkv, 128, "bf16", mask, seed=seed, backward=True,
                      v_shift_per_seq=2.0, window=window)
    x = inputs.make_inputs(w)
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    o, lse, o32 = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                           w.max_k, mask, w.scale, want_o_f32=True, window=window)
    dq, dk, dv = attn.bwd(d["q"], d["k"], d["v"], o, lse, d["dout"], d["cu_seqlens_q"],
                          d["cu_seqlens_k"], w.max_q, w.max_k, mask, w.scale, o_f32=o32,
                          window=window)
    plan = attn.last_plan()
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    if w.total_q > 0 and w.total_k > 0:
        assert "bwd_fused_tc" in plan, plan
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, mask, window=window)
    tag = f"seed {seed}: lq {lq} lk {lk} hq {hq} hkv {hkv} mask {mask} window {window}"
    compare.check_close(f"dq ({tag})", dq, rdq)
    compare.check_close(f"dk ({tag})", dk, rdk)
    compare.check_close(f"dv ({tag})", dv, rdv)
    for h, t in np.argwhere(np.isneginf(rlse)):
        assert np.all(compare.to_np(dq)[t, h] == 0.0)
