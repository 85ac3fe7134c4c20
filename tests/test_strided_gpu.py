"""Noncontiguous layouts on the GPU ("causal-mask-and-ragged-sequence-layouts",
fifth paragraph: include noncontiguous layouts where supported): q, k and v
as views of one fused [T, Hq + 2 Hkv + 1, d] projection output, the output
in a buffer with a wider feature row, and the gradients written into the
matching fused gradient buffer.  The results equal the contiguous call's bit
for bit (same kernels, same arithmetic) and the oracle within the contract;
the extra head of each fused buffer, which no tensor owns, is left alone."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs
from tests import compare
from tests.gpu_cases import backward_form

pytestmark = pytest.mark.gpu
TL, BR = inputs.MASK_TOP_LEFT, inputs.MASK_BOTTOM_RIGHT
SENTINEL = 7.0


def fused(x, w):
    """Copy q, k, v into one [T, Hq + 2 Hkv + 1, d] tensor (last head: a
    sentinel) and return the views (needs T_q == T_k)."""
    T = w.total_q
    hq, hkv = w.hq, w.hkv
    buf = torch.full((T, hq + 2 * hkv + 1, w.d), SENTINEL, dtype=x["q"].dtype, device="cuda")
    buf[:, :hq] = x["q"].cuda()
    buf[:, hq:hq + hkv] = x["k"].cuda()
    buf[:, hq + hkv:hq + 2 * hkv] = x["v"].cuda()
    return buf, buf[:, :hq], buf[:, hq:hq + hkv], buf[:, hq + hkv:hq + 2 * hkv]


CASES = [  # (name, lengths, hq, hkv, d, dtype, mask)
    ("prefill_gqa", (300, 129, 1, 700), 8, 2, 128, "bf16", TL),
    ("prefill_d64", (200, 77), 4, 4, 64, "bf16", BR),
    ("fp32", (70, 33), 4, 2, 64, "fp32", TL),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_fused_qkv_forward_backward(case):
    name, lens, hq, hkv, d, dt, mask = case
    w = inputs.custom(name, lens, lens, hq, hkv, d, dt, mask, seed=61, backward=True,
                      v_shift_per_seq=2.0)
    x = inputs.make_inputs(w)
    cq, ck = x["cu_seqlens_q"].cuda(), x["cu_seqlens_k"].cuda()
    buf, q, k, v = fused(x, w)
    assert not q.is_contiguous() and not k.is_contiguous()
    # output rows of 2 d features, of which the first d are O
    wide = torch.full((w.total_q, hq, 2 * d), SENTINEL, dtype=q.dtype, device="cuda")
    o = wide[:, :, :d]
    o_s, lse_s, o32_s = attn.fwd(q, k, v, cq, ck, w.max_q, w.max_k, mask, w.scale, out=o,
                                 want_o_f32=True)
    qc, kc, vc = q.contiguous(), k.contiguous(), v.contiguous()
    o_c, lse_c, o32_c = attn.fwd(qc, kc, vc, cq, ck, w.max_q, w.max_k, mask, w.scale,
                                 want_o_f32=True)
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    assert torch.equal(o_s, o_c) and torch.equal(lse_s, lse_c) and torch.equal(o32_s, o32_c)
    assert torch.all(wide[:, :, d:] == SENTINEL)
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.scale, mask)
    tol = {} if dt == "bf16" else {"atol": 1e-4, "rtol": 1e-4}
    compare.check_close("o", o_s, ro, **tol)
    compare.check_lse("lse", lse_s, rl)

    # backward: dout strided too, gradients into a fused buffer
    dwide = torch.zeros((w.total_q, hq, 2 * d), dtype=q.dtype, device="cuda")
    dwide[:, :, :d] = x["dout"].cuda()
    dout = dwide[:, :, :d]
    gbuf = torch.full_like(buf, SENTINEL)
    dq, dk, dv = gbuf[:, :hq], gbuf[:, hq:hq + hkv], gbuf[:, hq + hkv:hq + 2 * hkv]
    for two_kernel in (True, False):
        # the two-kernel form is bit-reproducible: strided equals contiguous
        # exactly; the fused form sums dQ in an order set by the CTAs' timing
        with backward_form(two_kernel):
            attn.bwd(q, k, v, o_s, lse_s, dout, cq, ck, w.max_q, w.max_k, mask, w.scale, dq=dq,
                     dk=dk, dv=dv, o_f32=o32_s)
            g_c = attn.bwd(qc, kc, vc, o_c, lse_c, dout.contiguous(), cq, ck, w.max_q, w.max_k,
                           mask, w.scale, o_f32=o32_c)
        torch.cuda.synchronize()
        assert attn.get_device_error() == 0
        assert torch.equal(dk, g_c[1]) and torch.equal(dv, g_c[2])
        if two_kernel:
            assert torch.equal(dq, g_c[0])
        else:
            compare.check_close("dq strided vs contiguous", dq,
                                compare.to_np(g_c[0]).astype(np.float64), atol=1e-3,
                                rtol=2.0 ** -7)
        assert torch.all(gbuf[:, -1] == SENTINEL)
    rdq, rdk, rdv, _, _ = oracle.bwd(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                     x["cu_seqlens_k"], w.scale, mask)
    compare.check_close("dq", dq, rdq, **tol)
    compare.check_close("dk", dk, rdk, **tol)
    compare.check_close("dv", dv, rdv, **tol)


def test_decode_split_strided():
    """The split-KV decode plan (and its combine) with q, k, v and o strided."""
    lq, lk = (1,) * 4, (9000, 129, 3000, 12000)
    w = inputs.custom("decode_strided", lq, lk, 32, 8, 128, "bf16", BR, seed=62)
    x = inputs.make_inputs(w)
    cq, ck = x["cu_seqlens_q"].cuda(), x["cu_seqlens_k"].cuda()
    kvbuf = torch.empty((w.total_k, 2 * w.hkv, w.d), dtype=torch.bfloat16, device="cuda")
    kvbuf[:, :w.hkv] = x["k"].cuda()
    kvbuf[:, w.hkv:] = x["v"].cuda()
    k, v = kvbuf[:, :w.hkv], kvbuf[:, w.hkv:]
    qwide = torch.zeros((w.total_q, w.hq, 2 * w.d), dtype=torch.bfloat16, device="cuda")
    qwide[:, :, :w.d] = x["q"].cuda()
    q = qwide[:, :, :w.d]
    o_s, lse_s = attn.fwd(q, k, v, cq, ck, w.max_q, w.max_k, BR, w.scale)
    assert "splits=" in attn.last_plan()
    o_c, lse_c = attn.fwd(q.contiguous(), k.contiguous(), v.contiguous(), cq, ck, w.max_q,
                          w.max_k, BR, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o_s, o_c) and torch.equal(lse_s, lse_c)
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.scale, BR)
    compare.check_close("o", o_s, ro)
    compare.check_lse("lse", lse_s, rl)
