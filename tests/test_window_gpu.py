"""Bounded causal windows on the GPU against the fp64 oracle: every row sees
at most W keys, the last W positions up to its causal bound
("attention-algorithm-error-and-complexity-tests", fifth paragraph; mask
rules of "causal-mask-and-ragged-sequence-layouts").  Each kernel plan is hit:
the two-tile prefill, packed decode with and without key splits, the
CUDA-core fp32 path, both backward paths, and the mask probe."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import oracle_fwd, run_fwd, sample_rows
from tests.test_backward_gpu import run_fwd_bwd
from tests.test_parity_gpu import check_full, check_rows

pytestmark = pytest.mark.gpu
TL, BR = inputs.MASK_TOP_LEFT, inputs.MASK_BOTTOM_RIGHT

FWD = [  # (name, lq, lk, hq, hkv, d, dtype, mask, window, plan substring)
    ("prefill_w1", (300, 129), None, 4, 2, 128, "bf16", TL, 1, "fwd_tc2"),
    ("prefill_w100", (700, 1, 255, 257), None, 8, 2, 128, "bf16", TL, 100, "fwd_tc2"),
    ("prefill_w128", (513, 384), None, 4, 1, 128, "bf16", TL, 128, "fwd_tc2"),
    ("prefill_w257_d64", (640, 100), None, 4, 4, 64, "bf16", TL, 257, "fwd_tc2"),
    ("prefill_br_w200", (300, 50), (700, 40), 4, 2, 128, "bf16", BR, 200, "fwd_tc2"),
    ("prefill_tl_q_longer_w64", (600,), (200,), 4, 2, 128, "bf16", TL, 64, "fwd_tc2"),
    ("decode_w300_no_split", (1,) * 6, (5000, 129, 1, 300, 4097, 2000), 32, 8, 128, "bf16", BR,
     300, "fwd_tc_"),
    ("decode_w3000_split", (1,) * 6, (9000, 129, 1, 3000, 12000, 5000), 32, 8, 128, "bf16", BR,
     3000, "splits="),
    ("decode_q16_w500", (16,) * 3, (4000, 16, 600), 32, 8, 128, "bf16", BR, 500, "fwd_tc_"),
    ("fp32_w7", (90, 33), (90, 33), 4, 2, 64, "fp32", TL, 7, "fwd_simt"),
]


@pytest.mark.parametrize("case", FWD, ids=[c[0] for c in FWD])
def test_window_forward_full(case):
    name, lq, lk, hq, hkv, d, dt, mask, window, plan = case
    w = inputs.custom(name, lq, lk or lq, hq, hkv, d, dt, mask, seed=31, v_shift_per_seq=3.0,
                      window=window)
    x = inputs.make_inputs(w)
    o, lse, _ = run_fwd(x)
    assert plan in attn.last_plan(), attn.last_plan()
    check_full(x, o, lse)


def test_window_prefill_full_size_sampled():
    """The prefill benchmark's shape (4 x 4096 tokens, 32 / 8 heads) with a
    1024-key window, on sampled rows."""
    base = inputs.WORKLOADS["gqa_prefill"]
    w = inputs.custom("gqa_prefill_w1024", base.seqlens_q, base.seqlens_k, base.hq, base.hkv,
                      base.d, "bf16", TL, seed=base.seed, window=1024)
    x = inputs.make_inputs(w)
    o, lse, _ = run_fwd(x)
    check_rows(x, o, lse, sample_rows(w, 48, seed=5))


BWD = [  # (name, lq, lk, hq, hkv, d, dtype, mask, window)
    ("tc_w1", (300, 129), (300, 129), 4, 2, 128, "bf16", TL, 1),
    ("tc_w100_ragged", (700, 1, 255, 257), (700, 1, 255, 257), 8, 2, 128, "bf16", TL, 100),
    ("tc_br_w200", (300, 50), (700, 40), 4, 1, 128, "bf16", BR, 200),
    ("tc_w64_d64", (320, 65), (320, 65), 4, 4, 64, "bf16", TL, 64),
    ("simt_fp32_w5", (40, 70), (50, 70), 4, 2, 64, "fp32", BR, 5),
]


@pytest.mark.parametrize("case", BWD, ids=[c[0] for c in BWD])
def test_window_backward_full(case):
    name, lq, lk, hq, hkv, d, dt, mask, window = case
    w = inputs.custom(name, lq, lk, hq, hkv, d, dt, mask, seed=37, backward=True,
                      v_shift_per_seq=2.0, window=window)
    x = inputs.make_inputs(w)
    o, lse, dq, dk, dv = run_fwd_bwd(x)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, mask, window=window)
    tol = {} if dt == "bf16" else {"atol": 1e-4, "rtol": 1e-4}
    compare.check_close("o", o, ro, **tol)
    compare.check_lse("lse", lse, rlse)
    compare.check_close("dq", dq, rdq, **tol)
    compare.check_close("dk", dk, rdk, **tol)
    compare.check_close("dv", dv, rdv, **tol)


@pytest.mark.parametrize("window", [1, 63, 128, 129, 300])
@pytest.mark.parametrize("mask", [TL, BR])
@pytest.mark.parametrize("tile_rows", [32, 128])
def test_window_probe_equals_oracle(window, mask, tile_rows):
    lq, lk = (1, 200, 513, 64), (300, 200, 513, 20)
    cq, ck = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    tq, tk = int(cq[-1]), int(ck[-1])
    got = attn.mask_probe(cq.cuda(), ck.cuda(), max(lq), max(lk), tq, tk, mask, tile_rows,
                          window=window)
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    ref = oracle.mask(cq.numpy(), ck.numpy(), tq, tk, mask, window)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_window_rejected_without_causal_rule():
    w = inputs.custom("none_w", (8,), (8,), 2, 1, 64, "bf16", inputs.MASK_NONE, seed=1)
    x = inputs.make_inputs(w, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], 8, 8,
                 inputs.MASK_NONE, window=4)
