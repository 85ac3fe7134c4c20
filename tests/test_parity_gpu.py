"""CUDA path against the fp64 oracle, element by element, on seeded inputs.

Small and mid-size problems are compared in full; the full-size workloads
are compared on sampled rows that the oracle computes one by one, in the same
launch configuration the benchmark times."""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import oracle_fwd, run_fwd, sample_rows

pytestmark = pytest.mark.gpu

TL, BR, NONE = inputs.MASK_TOP_LEFT, inputs.MASK_BOTTOM_RIGHT, inputs.MASK_NONE


def check_full(x, o, lse):
    o_ref, lse_ref = oracle_fwd(x)
    compare.check_close("o", o, o_ref)
    compare.check_lse("lse", lse, lse_ref)
    # empty rows: exact zeros and -inf
    empty = np.isneginf(lse_ref)
    if empty.any():
        on = compare.to_np(o)
        for h, t in np.argwhere(empty):
            assert np.all(on[t, h] == 0.0)


def check_rows(x, o, lse, rows):
    o_ref, lse_ref = oracle_fwd(x, rows=rows)
    on, ln = compare.to_np(o), compare.to_np(lse)
    compare.check_close("o", on[rows[:, 0], rows[:, 1]], o_ref)
    compare.check_lse("lse", ln[rows[:, 1], rows[:, 0]], lse_ref)


def test_tiny_fp32():
    x = inputs.make_inputs(inputs.WORKLOADS["tiny_fp32"])
    o, lse, _ = run_fwd(x)
    check_full(x, o, lse)
    o_ref, _ = oracle_fwd(x)
    # the fp32 path is far inside the bf16 contract
    assert np.abs(compare.to_np(o) - o_ref).max() < 1e-4


def test_varlen_causal_full():
    x = inputs.make_inputs(inputs.WORKLOADS["varlen_causal"])
    o, lse, _ = run_fwd(x)
    check_full(x, o, lse)


EDGE = [  # (name, lq, lk, hq, hkv, d, mask)
    ("ragged_tile_edges_tl", (63, 64, 65, 127, 128, 129, 1), None, 4, 1, 128, TL),
    ("ragged_tile_edges_br", (1, 5, 129), (300, 5, 128), 8, 2, 128, BR),
    ("q_longer_br_empty_rows", (64, 100), (32, 7), 8, 8, 128, BR),
    ("q_longer_tl", (200,), (70,), 4, 2, 64, TL),
    ("noncausal_gqa8", (130, 3), (257, 9), 16, 2, 128, NONE),
    ("zero_length_segments", (0, 40, 0, 17), (0, 40, 5, 17), 2, 1, 64, TL),
    ("d64_gqa4", (256, 190), (256, 190), 8, 2, 64, TL),
    ("single_token_each", (1, 1, 1), (1, 1, 1), 4, 4, 128, TL),
    ("decode_like_q1", (1,) * 5, (1000, 129, 128, 1, 4097), 32, 8, 128, BR),
    ("decode_like_q16", (16,) * 3, (2000, 16, 300), 32, 8, 128, BR),
]


@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
def test_edge_shapes(case):
    name, lq, lk, hq, hkv, d, mask = case
    w = inputs.custom(name, lq, lk if lk else lq, hq, hkv, d, "bf16", mask, seed=11,
                      v_shift_per_seq=3.0)
    x = inputs.make_inputs(w)
    o, lse, _ = run_fwd(x)
    check_full(x, o, lse)


def test_decode_empty_rows_full():
    x = inputs.make_inputs(inputs.WORKLOADS["decode_empty_rows"])
    o, lse, _ = run_fwd(x)
    check_full(x, o, lse)
    ln = compare.to_np(lse)
    # rows 0..31 of every sequence are empty under bottom-right alignment
    for s in range(32):
        assert np.all(np.isneginf(ln[:, s * 64:s * 64 + 32]))
        assert np.all(np.isfinite(ln[:, s * 64 + 32:s * 64 + 64]))


def test_count_probe():
    """Q = 0 makes every allowed logit 0, so exp(lse) is the allowed-set size
    of the row: the allowed sets are checked end to end."""
    w = inputs.custom("count", (5, 130, 64), (300, 129, 64), 4, 2, 128, "bf16", BR, seed=3)
    x = inputs.make_inputs(w)
    x["q"] = torch.zeros_like(x["q"])
    o, lse, _ = run_fwd(x)
    ln = compare.to_np(lse)
    cu = inputs.cu_seqlens(w.seqlens_q).numpy()
    for s, (nq, nk) in enumerate(zip(w.seqlens_q, w.seqlens_k)):
        for i in range(nq):
            n = max(0, min(i + nk - nq + 1, nk))
            got = ln[:, cu[s] + i]
            if n == 0:
                assert np.all(np.isneginf(got))
            else:
                assert np.all(np.abs(got - math.log(n)) <= 1e-4 * max(1.0, math.log(n)))


@pytest.mark.parametrize("name", ["gqa_prefill", "decode_q1", "decode_q16"])
def test_full_size_sampled(name):
    w = inputs.WORKLOADS[name]
    x = inputs.make_inputs(w)
    o, lse, _ = run_fwd(x)
    rows = sample_rows(w, 48, seed=5)
    check_rows(x, o, lse, rows)
    assert np.all(np.isfinite(compare.to_np(o)))


def test_forward_deterministic():
    x = inputs.make_inputs(inputs.WORKLOADS["varlen_causal"])
    o1, l1, dev = run_fwd(x)
    for _ in range(3):
        o2, l2, _ = run_fwd(x)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("lk", [(2048, 2048), (16384, 16384), (0, 0)])
def test_empty_query_batch_is_a_no_op(lk):
    """cu_seqlens_q = [0, 0, 0] against long key ranges: a legal call with no
    query row ("causal-mask-and-ragged-sequence-layouts", fifth paragraph).
    The forward, the backward and the workspace queries return OK and write
    nothing (sentinel buffers stay as they were)."""
    w = inputs.custom("noq", (0, 0), lk, 32, 8, 128, "bf16", BR, seed=2, backward=True)
    x = inputs.make_inputs(w, device="cuda")
    assert attn.fwd_workspace_size(w.batch, 0, w.max_k, 0, w.hq, w.hkv, w.d,
                                   attn.DTYPE_BF16) >= 0
    o = torch.empty((0, w.hq, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.hq, 0), dtype=torch.float32, device="cuda")
    o2, lse2 = attn.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], 0,
                        w.max_k, BR, w.scale, out=o, lse=lse)
    assert o2.numel() == 0 and lse2.numel() == 0
    dk = torch.full_like(x["k"], 7.0)
    dv = torch.full_like(x["v"], 7.0)
    dq, dk, dv = attn.bwd(x["q"], x["k"], x["v"], o, lse, x["dout"], x["cu_seqlens_q"],
                          x["cu_seqlens_k"], 0, w.max_k, BR, w.scale, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    # no query row reaches any key: every key's gradient is zero
    assert dq.numel() == 0
    assert torch.count_nonzero(dk) == 0 and torch.count_nonzero(dv) == 0


def test_bad_cu_seqlens_sets_device_flag():
    """cu_seqlens that run past total_q are caught on the device (no access
    beyond the buffers) and reported through the error flag."""
    w = inputs.custom("bad", (8, 8), (8, 8), 2, 1, 64, "bf16", TL)
    x = inputs.make_inputs(w, device="cuda")
    bad = torch.tensor([0, 8, 20], dtype=torch.int32, device="cuda")
    attn.fwd(x["q"], x["k"], x["v"], bad, x["cu_seqlens_k"], 12, 8, TL)
    assert attn.get_device_error() == 6
    assert attn.get_device_error() == 0  # cleared by the read


@pytest.mark.parametrize("which", ["q", "k"])
def test_uniform_totals_with_bad_cu_seqlens_set_device_flag(which):
    """Totals of batch x max with cu_seqlens in which one sequence runs past
    the max (a broken layout contract the totals alone do not show) are
    caught on the device and reported; a correct call afterwards is clean."""
    w = inputs.custom("unif", (128, 128), (128, 128), 4, 2, 128, "bf16", TL)
    x = inputs.make_inputs(w, device="cuda")
    bad = torch.tensor([0, 60, 256], dtype=torch.int32, device="cuda")
    cu_q = bad if which == "q" else x["cu_seqlens_q"]
    cu_k = bad if which == "k" else x["cu_seqlens_k"]
    attn.fwd(x["q"], x["k"], x["v"], cu_q, cu_k, 128, 128, TL)
    assert "fwd_tc2" in attn.last_plan(), attn.last_plan()
    assert attn.get_device_error() == 6
    attn.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], 128, 128, TL)
    assert attn.get_device_error() == 0


@pytest.mark.parametrize("scale", [-0.07, 0.0])
def test_non_positive_scale(scale):
    """scale <= 0 takes the path that scales scores before the row max."""
    w = inputs.custom("negscale", (130, 7), (200, 7), 4, 2, 128, "bf16", BR, seed=5)
    x = inputs.make_inputs(w)
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    o, lse = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                      w.max_k, w.mask, scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"],
                                scale, w.mask)
    compare.check_close("o", o, o_ref)
    compare.check_lse("lse", lse, lse_ref)
