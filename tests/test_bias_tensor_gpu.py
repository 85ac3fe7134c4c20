"""Explicit bias tensor on the GPU against the fp64 oracle, forward and
backward: entries added to the scaled logits, -inf entries masking pairs,
rows with no finite logit empty ("attention-algorithm-error-and-complexity-
tests", third paragraph; "causal-mask-and-ragged-sequence-layouts", sixth
paragraph: the backward rebuilds the same terms)."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import sample_rows, tc_backward

pytestmark = pytest.mark.gpu
TL, BR, NONE = inputs.MASK_TOP_LEFT, inputs.MASK_BOTTOM_RIGHT, inputs.MASK_NONE


def run(x, bias, slopes=None):
    w = x["workload"]
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    b = bias.cuda()
    sl = None if slopes is None else slopes.cuda()
    o, lse, o32 = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                           w.max_k, w.mask, w.scale, want_o_f32=True, window=w.window,
                           bias_slopes=sl, bias=b)
    fplan = attn.last_plan()
    dq, dk, dv = attn.bwd(d["q"], d["k"], d["v"], o, lse, d["dout"], d["cu_seqlens_q"],
                          d["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale, o_f32=o32,
                          window=w.window, bias_slopes=sl, bias=b)
    bplan = attn.last_plan()
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    return (o, lse, dq, dk, dv), (fplan, bplan)


CASES = [  # (name, lq, lk, hq, hkv, d, dtype, mask, window, bias broadcast, slopes,
    #          forward kernel, backward kernel)
    ("bf16_tl_full", (63, 129, 1, 200), None, 8, 2, 128, "bf16", TL, 0, False, False, "fwd_tc2", "tc"),
    ("bf16_tl_long", (700, 300), None, 4, 2, 128, "bf16", TL, 0, False, False, "fwd_tc2", "tc"),
    ("bf16_br_head_bcast", (40, 9), (100, 300), 4, 1, 64, "bf16", BR, 0, True, False, "fwd_tc2", "tc"),
    ("bf16_none_d64", (200, 77), (150, 300), 4, 4, 64, "bf16", NONE, 0, False, False, "fwd_tc2", "tc"),
    ("bf16_none_slopes", (50, 77), (70, 20), 4, 4, 128, "bf16", NONE, 0, False, True, "fwd_simt", "simt"),
    ("bf16_tl_window", (90, 333), None, 4, 2, 64, "bf16", TL, 9, False, False, "fwd_tc2", "tc"),
    ("fp32_br", (37, 70), (50, 70), 4, 2, 64, "fp32", BR, 0, True, True, "fwd_simt", "simt"),
    # d = 128 with the entries shared by the heads of a CTA: staged through
    # shared memory (key extent a multiple of 4 entries, 16-byte rows)
    ("bf16_tl_bcast_d128", (63, 129, 1, 200), None, 8, 2, 128, "bf16", TL, 0, True, False,
     "_btab_smem", "tc"),
    ("bf16_tl_window_bcast_d128", (90, 332, 260), None, 4, 2, 128, "bf16", TL, 9, True, False,
     "_btab_smem", "tc"),
    ("bf16_none_bcast_d128", (200, 77), (150, 300), 4, 2, 128, "bf16", NONE, 0, True, False,
     "_btab_smem", "tc"),
    ("bf16_br_bcast_d128", (40, 9, 130), (100, 300, 140), 8, 4, 128, "bf16", BR, 0, True, False,
     "_btab_smem", "tc"),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_bias_tensor_fwd_bwd(case):
    name, lq, lk, hq, hkv, d, dt, mask, window, bcast, with_slopes, kernel, bkernel = case
    w = inputs.custom(name, lq, lk or lq, hq, hkv, d, dt, mask, seed=61, backward=True,
                      v_shift_per_seq=2.0, window=window)
    x = inputs.make_inputs(w)
    bias = inputs.bias_tensor(1 if bcast else w.batch, 1 if bcast else hq, w.max_q, w.max_k,
                              seed=62, dead_rows=3)
    slopes = inputs.bias_slopes(hq) if with_slopes else None
    (o, lse, dq, dk, dv), (fplan, bplan) = run(x, bias, slopes)
    assert "_btab" in fplan and "_btab" in bplan and kernel in fplan and \
        (tc_backward(bplan) if bkernel == "tc" else bkernel in bplan), (fplan, bplan)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, mask, window=window,
                                         slopes=None if slopes is None else slopes.double().numpy(),
                                         bias=bias)
    tol = {} if dt == "bf16" else dict(atol=1e-4, rtol=1e-4)
    compare.check_close("o", o, ro, **tol)
    compare.check_lse("lse", lse, rlse)
    compare.check_close("dq", dq, rdq, **tol)
    compare.check_close("dk", dk, rdk, **tol)
    compare.check_close("dv", dv, rdv, **tol)
    # rows without a finite logit: O and dQ exactly zero
    for h, t in np.argwhere(np.isneginf(rlse)):
        assert np.all(compare.to_np(o)[t, h] == 0.0)
        assert np.all(compare.to_np(dq)[t, h] == 0.0)


def test_bias_tensor_broadcast_view_matches_materialised():
    """A stride-0 view from ``expand`` gives bit for bit what the materialised
    tensor gives."""
    w = inputs.custom("bview", (30, 45), (30, 45), 4, 2, 64, "bf16", TL, seed=63, backward=True)
    x = inputs.make_inputs(w)
    small = inputs.bias_tensor(1, 1, w.max_q, w.max_k, seed=64)
    view = small.expand(w.batch, 4, w.max_q, w.max_k)
    got_v, _ = run(x, view)
    got_m, _ = run(x, view.contiguous())
    for a, b in zip(got_v, got_m):
        assert torch.equal(a, b)


def test_zero_bias_tensor_matches_no_bias_oracle():
    """A zero tensor changes nothing: the result meets the oracle without bias."""
    w = inputs.custom("bzero", (70, 3), (70, 20), 2, 1, 128, "bf16", BR, seed=65, backward=True)
    x = inputs.make_inputs(w)
    (o, lse, dq, dk, dv), _ = run(x, torch.zeros((1, 1, w.max_q, w.max_k)))
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, BR)
    compare.check_close("o", o, ro)
    compare.check_lse("lse", lse, rlse)
    compare.check_close("dq", dq, rdq)
    compare.check_close("dk", dk, rdk)
    compare.check_close("dv", dv, rdv)


@pytest.mark.parametrize("keys,staged", [(200, True), (131, False), (70, False)])
def test_bias_tensor_staging_choice(keys, staged):
    """Entries shared by a CTA's two heads go through shared memory when TMA
    can address them (rows a multiple of 16 bytes); otherwise the softmax
    warps load them.  Both routes meet the oracle."""
    w = inputs.custom("bstage", (keys, keys - 50), (keys, keys - 50), 4, 2, 128, "bf16", TL,
                      seed=68, backward=True)
    x = inputs.make_inputs(w)
    bias = inputs.bias_tensor(1, 1, w.max_q, w.max_k, seed=69, dead_rows=1)
    (o, lse, dq, dk, dv), (fplan, _) = run(x, bias)
    assert "_btab" in fplan and ("_btab_smem" in fplan) == staged, fplan
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, TL, bias=bias)
    compare.check_close("o", o, ro)
    compare.check_lse("lse", lse, rlse)
    compare.check_close("dq", dq, rdq)
    compare.check_close("dk", dk, rdk)
    compare.check_close("dv", dv, rdv)


@pytest.mark.parametrize("seed", range(6))
def test_bias_tensor_staged_random_shapes(seed):
    """Random packed batches on the staged forward (head_dim 128, even GQA
    group, entries shared by the heads): 1-4 sequences of 0-300 queries, keys
    as many (top-left) or independent (bottom-right, no mask), a window half
    of the time with a causal rule, a tensor per sequence or one for all, its
    key dimension padded to a multiple of 4 entries (16-byte rows), about a
    fifth of the entries and a few whole rows -inf; forward and backward
    against the oracle."""
    rng = np.random.default_rng(100 + seed)
    batch = int(rng.integers(1, 5))
    mask = [TL, BR, NONE][int(rng.integers(3))]
    lq = [int(x) for x in rng.integers(0, 301, size=batch)]
    lk = lq if mask == TL else [int(x) for x in rng.integers(1, 301, size=batch)]
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([2, 4]))
    window = int(rng.integers(1, 200)) if mask != NONE and rng.random() < 0.5 else 0
    w = inputs.custom(f"bsrand{seed}", lq, lk, hq, hkv, 128, "bf16", mask, seed=110 + seed,
                      backward=True, v_shift_per_seq=2.0, window=window)
    x = inputs.make_inputs(w)
    per_seq = bool(rng.random() < 0.5)
    keys = max(4, (w.max_k + 3) // 4 * 4)
    bias = inputs.bias_tensor(w.batch if per_seq else 1, 1, max(1, w.max_q), keys, seed=120 + seed,
                              dead_rows=2)
    (o, lse, dq, dk, dv), (fplan, _) = run(x, bias)
    if w.max_q > 0:
        assert "_btab_smem" in fplan, fplan
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, mask, window=window,
                                         bias=bias)
    tag = f"seed {seed}: lq {lq} lk {lk} hq {hq} hkv {hkv} mask {mask} window {window}"
    compare.check_close(f"o ({tag})", o, ro)
    compare.check_lse(f"lse ({tag})", lse, rlse)
    compare.check_close(f"dq ({tag})", dq, rdq)
    compare.check_close(f"dk ({tag})", dk, rdk)
    compare.check_close(f"dv ({tag})", dv, rdv)
    for h, t in np.argwhere(np.isneginf(rlse)):
        assert np.all(compare.to_np(o)[t, h] == 0.0)


@pytest.mark.parametrize("shape", ["heads_only", "sequences_only"])
def test_bias_tensor_mixed_broadcast(shape):
    """A tensor with one entry per head shared by every sequence, or one per
    sequence shared by every head, on the tensor-core path forward and
    backward."""
    w = inputs.custom("bmix", (130, 40, 200), (130, 90, 200), 4, 2, 128, "bf16", BR, seed=66,
                      backward=True)
    x = inputs.make_inputs(w)
    b, hb = (1, 4) if shape == "heads_only" else (w.batch, 1)
    bias = inputs.bias_tensor(b, hb, w.max_q, w.max_k, seed=67, dead_rows=2)
    (o, lse, dq, dk, dv), (fplan, bplan) = run(x, bias)
    assert "fwd_tc2" in fplan and tc_backward(bplan), (fplan, bplan)
    rdq, rdk, rdv, ro, rlse = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                         x["cu_seqlens_k"], w.scale, BR, bias=bias)
    compare.check_close("o", o, ro)
    compare.check_lse("lse", lse, rlse)
    compare.check_close("dq", dq, rdq)
    compare.check_close("dk", dk, rdk)
    compare.check_close("dv", dv, rdv)


def test_bias_tensor_prefill_full_size_sampled():
    """The bias-tensor prefill workload at full size: sampled rows against the
    oracle with the same [B, 1, N, N] tensor."""
    w = inputs.WORKLOADS["bias_tensor_prefill"]
    x = inputs.make_inputs(w)
    bias = inputs.bias_tensor(w.batch, 1, w.max_q, w.max_k, w.seed + 1)
    d = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    o, lse = attn.fwd(d["q"], d["k"], d["v"], d["cu_seqlens_q"], d["cu_seqlens_k"], w.max_q,
                      w.max_k, w.mask, w.scale, bias=bias.cuda())
    assert "fwd_tc2" in attn.last_plan() and "_btab_smem" in attn.last_plan()
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    rows = sample_rows(w, 24, seed=71)
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.scale,
                        w.mask, rows=rows, bias=bias)
    on, ln = compare.to_np(o), compare.to_np(lse)
    compare.check_close("o", on[rows[:, 0], rows[:, 1]], ro)
    compare.check_lse("lse", ln[rows[:, 1], rows[:, 0]], rl)


def test_bias_tensor_train_full_size_sampled():
    """The bias-tensor training workload at full size: sampled dQ rows and dK,
    dV key rows against the oracle's sampled backward."""
    w = inputs.WORKLOADS["bias_tensor_train"]
    x = inputs.make_inputs(w)
    bias = inputs.bias_tensor(w.batch, 1, w.max_q, w.max_k, w.seed + 1)
    (o, lse, dq, dk, dv), (fplan, bplan) = run(x, bias)
    assert "fwd_tc2" in fplan and tc_backward(bplan), (fplan, bplan)
    qrows = sample_rows(w, 8, seed=72)
    krows = np.array([(0, 0), (8191, 3), (8192, 1), (16383, 2)], np.int64)
    rdq, rdk, rdv = oracle.bwd_sampled(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                       x["cu_seqlens_k"], w.scale, w.mask, qrows, krows,
                                       bias=bias)
    compare.check_close("dq", compare.to_np(dq)[qrows[:, 0], qrows[:, 1]], rdq)
    compare.check_close("dk", compare.to_np(dk)[krows[:, 0], krows[:, 1]], rdk)
    compare.check_close("dv", compare.to_np(dv)[krows[:, 0], krows[:, 1]], rdv)
