"""CUDA backward against the fp64 oracle's gradients (dQ, and dK / dV summed
over each KV head's query heads), on small problems in full and on the
full-size training workload at sampled rows."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import sample_rows

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
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_backward_full(case):
    name, lq, lk, hq, hkv, d, dt, mask = case
    # value ranges differ per sequence so that leakage shows
    w = inputs.custom(name, lq, lk, hq, hkv, d, dt, mask, seed=17, backward=True,
                      v_shift_per_seq=2.0)
    x = inputs.make_inputs(w)
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


def test_train_full_size_sampled():
    w = inputs.WORKLOADS["train_fwd_bwd"]
    x = inputs.make_inputs(w)
    o, lse, dq, dk, dv = run_fwd_bwd(x)
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
    """Every gradient row has one owner CTA and no atomics: repeated calls give
    bit-identical dq, dk, dv."""
    w = inputs.custom("det", (300, 129), (300, 129), 8, 2, 128, "bf16", TL, seed=4, backward=True)
    x = inputs.make_inputs(w)
    first = run_fwd_bwd(x)
    for _ in range(3):
        again = run_fwd_bwd(x)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


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
