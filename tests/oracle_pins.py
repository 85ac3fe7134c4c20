"""Pins that tie the fp64 oracle to facts fixed outside itself.

Every pin takes an ``Oracle`` instance and raises ``AssertionError`` when the
oracle disagrees with a closed form, an invariant, a library special case or a
finite difference.  ``test_oracle.py`` runs them against the real oracle and
``test_oracle_mutants.py`` runs them against copies of the oracle with one
plausible mistake planted each, to show that every such mistake is caught.

None of the expected values here come from the oracle or from the CUDA path:
they are closed forms written with numpy, torch's fp64 CPU reference
attention, or central differences.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

NONE, TOP_LEFT, BOTTOM_RIGHT = 0, 1, 2
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def cu(lengths):
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return np.array(out, np.int32)


def row_range(kind, i, nq, nk, window=0):
    """Closed-form [a, b) of allowed key positions of zero-based query row i:
    the causal bound is i (top-left) or i + nk - nq (bottom-right), and a
    window W > 0 keeps only the W positions ending at that bound."""
    if kind == NONE:
        return 0, nk
    bound = i if kind == TOP_LEFT else i + nk - nq
    b = min(max(bound + 1, 0), nk)
    a = 0 if window <= 0 else min(max(bound + 1 - window, 0), nk)
    return a, b


def row_count(kind, i, nq, nk, window=0):
    """Closed-form number of allowed keys of zero-based query row i."""
    a, b = row_range(kind, i, nq, nk, window)
    return b - a


def allowed_interval(kind, lq, lk, window=0):
    """[(token, key_start, key_end)] for every packed query token: under every
    rule the allowed keys of a row are one interval of its own sequence (a
    prefix without a window)."""
    out = []
    cq, ck = cu(lq), cu(lk)
    for s, (nq, nk) in enumerate(zip(lq, lk)):
        for i in range(nq):
            a, b = row_range(kind, i, nq, nk, window)
            out.append((cq[s] + i, ck[s] + a, ck[s] + b))
    return out


def rand_case(rng, lq, lk, hq, hkv, d):
    tq, tk = sum(lq), sum(lk)
    q = rng.standard_normal((tq, hq, d))
    k = rng.standard_normal((tk, hkv, d))
    v = rng.standard_normal((tk, hkv, d))
    return q, k, v


SHAPES = [  # (lq, lk, hq, hkv, d, kind)
    ((5, 1, 7), (5, 1, 7), 4, 2, 8, TOP_LEFT),
    ((3, 6), (8, 2), 2, 1, 4, BOTTOM_RIGHT),  # Nq<Nk and Nq>Nk (empty rows)
    ((6, 4), (4, 6), 3, 3, 5, TOP_LEFT),      # Nq>Nk top-left
    ((4, 0, 3), (4, 0, 3), 2, 2, 4, NONE),    # a zero-length segment
    ((2, 5), (9, 3), 4, 1, 3, BOTTOM_RIGHT),
]

WINDOWS = (1, 2, 3, 7)  # bounded windows, all shorter than some sequence


# --------------------------------------------------------------------------
# mask
# --------------------------------------------------------------------------
def pin_token_meta(orc):
    sid, pos = orc.token_meta(np.array([0, 3, 3, 7], np.int32), 7)
    assert list(sid) == [0, 0, 0, 2, 2, 2, 2]
    assert list(pos) == [0, 1, 2, 0, 1, 2, 3]


def pin_mask_intervals(orc):
    """The materialised mask equals, bit for bit, the prefix interval that the
    closed form of each rule gives, with nothing across sequences."""
    for lq, lk, _, _, _, kind in SHAPES:
        for k2 in (NONE, TOP_LEFT, BOTTOM_RIGHT):
            for w in (0,) + (WINDOWS if k2 != NONE else ()):
                m = orc.mask(cu(lq), cu(lk), sum(lq), sum(lk), k2, w)
                ref = np.zeros_like(m)
                for t, a, b in allowed_interval(k2, lq, lk, w):
                    ref[t, a:b] = 1
                assert np.array_equal(m, ref), (lq, lk, k2, w)


def pin_window_counts(orc):
    """Hand-counted windowed masks ("attention-algorithm-error-and-complexity-
    tests", fifth paragraph: a bounded window makes the pair count linear in
    the length).  Top-left, N = 6, W = 2: rows see 1, 2, 2, 2, 2, 2 keys (11
    pairs).  Bottom-right, Nq = 3, Nk = 7, W = 3: the bounds are 4, 5, 6, so
    every row sees 3 keys (9 pairs) starting at 2, 3, 4.  Bottom-right,
    Nq = 5, Nk = 2, W = 1: bounds -3..1, rows 3 and 4 see key 0 and key 1."""
    m = orc.mask(cu([6]), cu([6]), 6, 6, TOP_LEFT, 2)
    assert list(m.sum(axis=1)) == [1, 2, 2, 2, 2, 2]
    assert m[5, 4] == 1 and m[5, 3] == 0 and m[5, 5] == 1
    m = orc.mask(cu([3]), cu([7]), 3, 7, BOTTOM_RIGHT, 3)
    assert [list(np.nonzero(r)[0]) for r in m] == [[2, 3, 4], [3, 4, 5], [4, 5, 6]]
    m = orc.mask(cu([5]), cu([2]), 5, 2, BOTTOM_RIGHT, 1)
    assert [list(np.nonzero(r)[0]) for r in m] == [[], [], [], [0], [1]]
    # a window needs a causal rule: without one there is no bound to end at
    try:
        orc.mask(cu([3]), cu([3]), 3, 3, NONE, 2)
    except ValueError:
        pass
    else:
        raise AssertionError("window without a causal rule accepted")


def pin_window_one_key(orc):
    """W = 1: every non-empty row sees exactly the key at its causal bound, so
    O_i = v_bound and lse_i = scale * q_i . k_bound."""
    rng = np.random.default_rng(14)
    for lq, lk, hq, hkv, d, kind in SHAPES:
        if kind == NONE:
            continue
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        o, lse = orc.fwd(q, k, v, cu(lq), cu(lk), 0.55, kind, window=1)
        g = hq // hkv
        for t, a, b in allowed_interval(kind, lq, lk, 1):
            for h in range(hq):
                if b == a:
                    assert np.all(o[t, h] == 0.0) and lse[h, t] == -math.inf
                    continue
                assert b == a + 1
                np.testing.assert_allclose(o[t, h], v[a, h // g], rtol=1e-14, atol=1e-14)
                ref = 0.55 * float(q[t, h] @ k[a, h // g])
                assert abs(lse[h, t] - ref) <= 1e-12 * max(1.0, abs(ref))


def pin_window_covering_is_causal(orc):
    """A window at least as long as every key sequence removes nothing: the
    result equals the unbounded causal one exactly."""
    rng = np.random.default_rng(15)
    for lq, lk, hq, hkv, d, kind in SHAPES:
        if kind == NONE:
            continue
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        do = rng.standard_normal(q.shape)
        a = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.5, kind)
        b = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.5, kind, window=max(lk))
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def pin_golden_mask_counts(orc):
    with open(os.path.join(GOLDEN, "mask_counts.json")) as f:
        cases = json.load(f)["cases"]
    kinds = {"top_left": TOP_LEFT, "bottom_right": BOTTOM_RIGHT, "none": NONE}
    for c in cases:
        lq, lk = c["seqlens_q"], c["seqlens_k"]
        m = orc.mask(cu(lq), cu(lk), sum(lq), sum(lk), kinds[c["mask"]])
        assert int(m.sum(dtype=np.int64)) == c["pairs_per_head"], c["name"]
        assert int((m.sum(axis=1) == 0).sum()) == c["empty_rows_per_head"], c["name"]


# --------------------------------------------------------------------------
# forward: hand cases ("attention-algorithm-error-and-complexity-tests",
# first paragraph)
# --------------------------------------------------------------------------
def pin_uniform_logits(orc):
    """Q = 0: every allowed logit is 0, so O_i is the mean of the allowed V
    rows and lse_i = ln |A_i|; empty rows give exact zeros and -inf."""
    rng = np.random.default_rng(1)
    cases = [(s, 0) for s in SHAPES] + [(s, 3) for s in SHAPES if s[5] != NONE]
    for (lq, lk, hq, hkv, d, kind), w in cases:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        q[:] = 0.0
        o, lse = orc.fwd(q, k, v, cu(lq), cu(lk), 0.37, kind, window=w)
        g = hq // hkv
        for t, a, b in allowed_interval(kind, lq, lk, w):
            for h in range(hq):
                if b == a:
                    assert np.all(o[t, h] == 0.0) and lse[h, t] == -math.inf
                else:
                    ref = v[a:b, h // g].mean(axis=0)
                    np.testing.assert_allclose(o[t, h], ref, rtol=1e-12, atol=1e-12)
                    assert abs(lse[h, t] - math.log(b - a)) < 1e-12


def _dominant_case(n_keys, big, d=4, scale=0.5):
    """One query whose score against key jstar is ``big`` and 0 against the
    others (orthogonal keys)."""
    rng = np.random.default_rng(2)
    q = np.zeros((1, 1, d))
    q[0, 0, 0] = 1.0
    k = rng.standard_normal((n_keys, 1, d))
    k[:, 0, 0] = 0.0
    jstar = n_keys // 2
    k[jstar, 0, 0] = big / scale
    v = rng.standard_normal((n_keys, 1, d))
    return q, k, v, jstar, scale


def pin_single_dominant_score(orc):
    """One score L above the rest: O = (e^L v* + sum_other v) / (e^L + n - 1).
    L = 800 overflows exp in fp64 unless the row max is subtracted first."""
    for big in (3.0, 800.0):
        n = 6
        q, k, v, js, scale = _dominant_case(n, big)
        o, lse = orc.fwd(q, k, v, cu([1]), cu([n]), scale, NONE)
        w = math.exp(-big)  # weights relative to e^L
        others = [j for j in range(n) if j != js]
        ref = (v[js, 0] + w * v[others, 0].sum(axis=0)) / (1.0 + (n - 1) * w)
        np.testing.assert_allclose(o[0, 0], ref, rtol=1e-12, atol=1e-12)
        assert abs(lse[0, 0] - (big + math.log1p((n - 1) * w))) < 1e-12


def pin_masked_dominant_score(orc):
    """A huge score on a masked key (a future key under top-left, or a key of
    another packed sequence) must be excluded before the max and the
    denominator: the row stays the uniform mean of its allowed keys."""
    d, scale = 4, 0.5
    rng = np.random.default_rng(3)
    lq = lk = (4, 5)
    q = np.zeros((9, 1, d))
    q[:, 0, 0] = 1.0
    k = rng.standard_normal((9, 1, d))
    k[:, 0, 0] = 0.0
    v = rng.standard_normal((9, 1, d))
    k[3, 0, 0] = 1000.0 / scale  # last key of sequence 0: future for rows 0..2
    k[8, 0, 0] = 1000.0 / scale  # last key of sequence 1
    o, lse = orc.fwd(q, k, v, cu(lq), cu(lk), scale, TOP_LEFT)
    for t, a, b in allowed_interval(TOP_LEFT, lq, lk):
        if t in (3, 8):
            continue  # these rows do see the dominant key
        np.testing.assert_allclose(o[t, 0], v[a:b, 0].mean(axis=0), rtol=1e-12, atol=1e-12)
        assert abs(lse[0, t] - math.log(b - a)) < 1e-12


# --------------------------------------------------------------------------
# forward: invariants (third paragraph of the same page)
# --------------------------------------------------------------------------
def pin_row_shift(orc):
    """K + 1 w^T adds scale * q_i . w to every logit of row i: O unchanged,
    lse shifted by exactly that amount."""
    rng = np.random.default_rng(4)
    for lq, lk, hq, hkv, d, kind in SHAPES:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        w = rng.standard_normal(d)
        scale = 0.41
        o0, l0 = orc.fwd(q, k, v, cu(lq), cu(lk), scale, kind)
        o1, l1 = orc.fwd(q, k + w, v, cu(lq), cu(lk), scale, kind)
        np.testing.assert_allclose(o1, o0, rtol=1e-9, atol=1e-10)
        shift = scale * np.einsum("thd,d->ht", q, w)
        fin = np.isfinite(l0)
        assert np.array_equal(fin, np.isfinite(l1))
        np.testing.assert_allclose(l1[fin], l0[fin] + shift[fin], rtol=1e-10, atol=1e-10)


def pin_permutation_noncausal(orc):
    """Permuting keys and values together inside each sequence leaves every
    noncausal row unchanged."""
    rng = np.random.default_rng(5)
    lq, lk = (3, 6), (7, 5)
    q, k, v = rand_case(rng, lq, lk, 2, 1, 6)
    ck = cu(lk)
    perm = np.concatenate([ck[s] + rng.permutation(n) for s, n in enumerate(lk)])
    o0, l0 = orc.fwd(q, k, v, cu(lq), ck, 0.3, NONE)
    o1, l1 = orc.fwd(q, k[perm], v[perm], cu(lq), ck, 0.3, NONE)
    np.testing.assert_allclose(o1, o0, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=1e-12, atol=1e-12)


def pin_gqa_vs_repeat(orc):
    """Shared KV heads equal K/V explicitly repeated by the contiguous
    grouping h -> h // (Hq/Hkv), forward and gradients (dK, dV summed over
    each group)."""
    rng = np.random.default_rng(6)
    lq = lk = (5, 3)
    hq, hkv, d = 6, 2, 4
    q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
    do = rng.standard_normal(q.shape)
    g = hq // hkv
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    a = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.5, TOP_LEFT)
    b = orc.bwd(q, kr, vr, do, cu(lq), cu(lk), 0.5, TOP_LEFT)
    np.testing.assert_allclose(a[3], b[3], rtol=1e-12, atol=1e-12)  # O
    np.testing.assert_allclose(a[0], b[0], rtol=1e-10, atol=1e-12)  # dQ
    dk_sum = b[1].reshape(-1, hkv, g, d).sum(axis=2)
    dv_sum = b[2].reshape(-1, hkv, g, d).sum(axis=2)
    np.testing.assert_allclose(a[1], dk_sum, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(a[2], dv_sum, rtol=1e-10, atol=1e-12)


def pin_packed_vs_separate(orc):
    """A packed batch equals each sequence run alone, outputs and gradients
    gathered back to packed storage order ("causal-mask-and-ragged-sequence-
    layouts", second and fifth paragraphs)."""
    rng = np.random.default_rng(7)
    for kind in (TOP_LEFT, BOTTOM_RIGHT):
        lq, lk = (4, 2, 5), (6, 2, 3)
        q, k, v = rand_case(rng, lq, lk, 2, 1, 4)
        do = rng.standard_normal(q.shape)
        packed = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.6, kind)
        cq, ck = cu(lq), cu(lk)
        for s in range(len(lq)):
            qs, ks = slice(cq[s], cq[s + 1]), slice(ck[s], ck[s + 1])
            one = orc.bwd(q[qs], k[ks], v[ks], do[qs], cu([lq[s]]), cu([lk[s]]), 0.6, kind)
            np.testing.assert_allclose(packed[3][qs], one[3], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(packed[4][:, qs], one[4], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(packed[0][qs], one[0], rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(packed[1][ks], one[1], rtol=1e-11, atol=1e-13)
            np.testing.assert_allclose(packed[2][ks], one[2], rtol=1e-11, atol=1e-13)


# --------------------------------------------------------------------------
# library special case: torch's fp64 CPU reference attention with an explicit
# boolean mask ("causal-mask-and-ragged-sequence-layouts", fourth paragraph)
# --------------------------------------------------------------------------
def pin_torch_sdpa_fp64(orc):
    rng = np.random.default_rng(8)
    cases = [(s, 0) for s in SHAPES] + [(s, 2) for s in SHAPES if s[5] != NONE]
    for (lq, lk, hq, hkv, d, kind), w in cases:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        do = rng.standard_normal(q.shape)
        scale = 1.0 / math.sqrt(d)
        dq, dk, dv, o, lse = orc.bwd(q, k, v, do, cu(lq), cu(lk), scale, kind, window=w)
        g = hq // hkv
        cq, ck = cu(lq), cu(lk)
        for s, (nq, nk) in enumerate(zip(lq, lk)):
            if nq == 0:
                continue
            rows = [i for i in range(nq) if row_count(kind, i, nq, nk, w) > 0]
            mask = np.zeros((nq, nk), bool)
            for i in range(nq):
                a, b = row_range(kind, i, nq, nk, w)
                mask[i, a:b] = True
            qs = torch.tensor(q[cq[s]:cq[s + 1]].transpose(1, 0, 2), requires_grad=True)
            ks = torch.tensor(k[ck[s]:ck[s + 1]].transpose(1, 0, 2), requires_grad=True)
            vs = torch.tensor(v[ck[s]:ck[s + 1]].transpose(1, 0, 2), requires_grad=True)
            kr = ks.repeat_interleave(g, dim=0)
            vr = vs.repeat_interleave(g, dim=0)
            if not rows:
                continue
            ri = torch.tensor(rows)
            out = torch.nn.functional.scaled_dot_product_attention(
                qs[:, ri], kr, vr, attn_mask=torch.tensor(mask[rows]), scale=scale)
            dot = torch.tensor(do[cq[s]:cq[s + 1]].transpose(1, 0, 2))[:, ri]
            (out * dot).sum().backward()
            ref_o = out.detach().numpy().transpose(1, 0, 2)
            got_o = o[cq[s]:cq[s + 1]][rows]
            np.testing.assert_allclose(got_o, ref_o, rtol=1e-10, atol=1e-12)
            got_dq = dq[cq[s]:cq[s + 1]][rows]
            ref_dq = qs.grad.numpy().transpose(1, 0, 2)[rows]
            np.testing.assert_allclose(got_dq, ref_dq, rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dk[ck[s]:ck[s + 1]], ks.grad.numpy().transpose(1, 0, 2),
                                       rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dv[ck[s]:ck[s + 1]], vs.grad.numpy().transpose(1, 0, 2),
                                       rtol=1e-9, atol=1e-11)


# --------------------------------------------------------------------------
# backward ("attention-algorithm-error-and-complexity-tests", fourth paragraph)
# --------------------------------------------------------------------------
def pin_finite_differences(orc):
    """Central differences of L = sum O * dO on a tiny smooth case (the mask
    does not depend on the values, so no step crosses a discontinuity)."""
    rng = np.random.default_rng(9)
    lq, lk = (3, 4), (3, 5)
    hq, hkv, d, scale = 2, 1, 3, 0.7
    q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
    do = rng.standard_normal(q.shape)
    for kind, w in ((BOTTOM_RIGHT, 0), (TOP_LEFT, 2)):
        dq, dk, dv, _, _ = orc.bwd(q, k, v, do, cu(lq), cu(lk), scale, kind, window=w)

        def loss(qq, kk, vv):
            o, _ = orc.fwd(qq, kk, vv, cu(lq), cu(lk), scale, kind, window=w)
            return float((o * do).sum())

        h = 1e-5
        for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xs = []
                for sign in (1.0, -1.0):
                    xx = x.copy()
                    xx[idx] += sign * h
                    xs.append({"q": (xx, k, v), "k": (q, xx, v), "v": (q, k, xx)}[name])
                fd[idx] = (loss(*xs[0]) - loss(*xs[1])) / (2 * h)
            np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=(name, w))


def pin_dv_column_sum(orc):
    """Softmax rows sum to one, so sum_j dV_j of a KV head equals the sum of
    dO over every non-empty row of its query heads."""
    rng = np.random.default_rng(10)
    cases = [(s, 0) for s in SHAPES] + [(s, 2) for s in SHAPES if s[5] != NONE]
    for (lq, lk, hq, hkv, d, kind), w in cases:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        do = rng.standard_normal(q.shape)
        dq, dk, dv, o, lse = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.5, kind, window=w)
        g = hq // hkv
        nonempty = np.zeros((sum(lq), hq), bool)
        for t, a, b in allowed_interval(kind, lq, lk, w):
            nonempty[t, :] = b > a
        for hk in range(hkv):
            ref = np.zeros(d)
            for h in range(hk * g, hk * g + g):
                ref += do[nonempty[:, h], h].sum(axis=0)
            np.testing.assert_allclose(dv[:, hk].sum(axis=0), ref, rtol=1e-10, atol=1e-10)


def pin_dq_key_shift(orc):
    """Each row of dS sums to zero (softmax Jacobian), so adding a common
    vector to every key leaves dQ unchanged."""
    rng = np.random.default_rng(11)
    lq, lk, hq, hkv, d, kind = SHAPES[0]
    q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
    do = rng.standard_normal(q.shape)
    w = rng.standard_normal(d)
    a = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.5, kind)
    b = orc.bwd(q, k + w, v, do, cu(lq), cu(lk), 0.5, kind)
    np.testing.assert_allclose(b[0], a[0], rtol=1e-8, atol=1e-10)


def pin_scale_identity(orc):
    """L depends on Q and K only through Q K^T, so d/da L(aQ) = d/da L(aK) at
    a = 1: sum <dQ, Q> = sum <dK, K>."""
    rng = np.random.default_rng(12)
    for lq, lk, hq, hkv, d, kind in SHAPES:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        do = rng.standard_normal(q.shape)
        dq, dk, dv, _, _ = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.45, kind)
        a, b = float((dq * q).sum()), float((dk * k).sum())
        assert abs(a - b) <= 1e-10 * max(1.0, abs(a)), (a, b)


def pin_empty_rows_backward(orc):
    """All-masked rows (bottom-right, Nq > Nk) have zero dQ and add nothing
    to dK/dV: zeroing their dO changes no gradient."""
    rng = np.random.default_rng(13)
    lq, lk = (6,), (2,)
    q, k, v = rand_case(rng, lq, lk, 2, 1, 4)
    do = rng.standard_normal(q.shape)
    dq, dk, dv, o, lse = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.5, BOTTOM_RIGHT)
    empty = [i for i in range(6) if row_count(BOTTOM_RIGHT, i, 6, 2) == 0]
    assert empty == [0, 1, 2, 3]
    assert np.all(dq[empty] == 0.0) and np.all(o[empty] == 0.0)
    assert np.all(lse[:, empty] == -math.inf)
    do2 = do.copy()
    do2[empty] = 0.0
    _, dk2, dv2, _, _ = orc.bwd(q, k, v, do2, cu(lq), cu(lk), 0.5, BOTTOM_RIGHT)
    assert np.array_equal(dk, dk2) and np.array_equal(dv, dv2)


# --------------------------------------------------------------------------
# linear positional bias -slope_h |i + off - j| ("attention-algorithm-error-
# and-complexity-tests", third paragraph; "causal-mask-and-ragged-sequence-
# layouts", sixth paragraph)
# --------------------------------------------------------------------------
def bias_offset(kind, nq, nk):
    return nk - nq if kind == BOTTOM_RIGHT else 0


def slopes_for(hq, seed=40):
    return np.random.default_rng(seed).uniform(0.05, 0.9, hq)


def pin_bias_uniform_logits(orc):
    """Q = 0: the logits are the bias alone, so O_i is the average of the
    allowed V rows weighted by exp(-slope |i + off - j|), a closed form."""
    rng = np.random.default_rng(41)
    for lq, lk, hq, hkv, d, kind in SHAPES:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        q[:] = 0.0
        sl = slopes_for(hq)
        o, lse = orc.fwd(q, k, v, cu(lq), cu(lk), 0.37, kind, slopes=sl)
        g = hq // hkv
        cq, ck = cu(lq), cu(lk)
        for s_, (nq, nk) in enumerate(zip(lq, lk)):
            off = bias_offset(kind, nq, nk)
            for i in range(nq):
                a, b = row_range(kind, i, nq, nk)
                t = cq[s_] + i
                for h in range(hq):
                    if b == a:
                        assert np.all(o[t, h] == 0.0) and lse[h, t] == -math.inf
                        continue
                    js = np.arange(a, b)
                    w = np.exp(-sl[h] * np.abs(i + off - js))
                    ref = (w[:, None] * v[ck[s_] + js, h // g]).sum(0) / w.sum()
                    np.testing.assert_allclose(o[t, h], ref, rtol=1e-12, atol=1e-12)
                    assert abs(lse[h, t] - math.log(w.sum())) < 1e-12


def pin_bias_zero_slopes(orc):
    """Zero slopes give the unbiased result exactly."""
    rng = np.random.default_rng(42)
    for lq, lk, hq, hkv, d, kind in SHAPES:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        do = rng.standard_normal(q.shape)
        a = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.5, kind)
        b = orc.bwd(q, k, v, do, cu(lq), cu(lk), 0.5, kind, slopes=np.zeros(hq))
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def pin_bias_torch_sdpa_fp64(orc):
    """torch's fp64 reference attention with the bias as an additive float
    mask (-inf on disallowed pairs), forward and every gradient; windows and
    the noncausal rule included."""
    rng = np.random.default_rng(43)
    cases = [(s_, 0) for s_ in SHAPES] + [(s_, 3) for s_ in SHAPES if s_[5] != NONE]
    for (lq, lk, hq, hkv, d, kind), w in cases:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        do = rng.standard_normal(q.shape)
        sl = slopes_for(hq, seed=44)
        scale = 1.0 / math.sqrt(d)
        dq, dk, dv, o, lse = orc.bwd(q, k, v, do, cu(lq), cu(lk), scale, kind, window=w, slopes=sl)
        g = hq // hkv
        cq, ck = cu(lq), cu(lk)
        for s_, (nq, nk) in enumerate(zip(lq, lk)):
            rows = [i for i in range(nq) if row_count(kind, i, nq, nk, w) > 0]
            if not rows:
                continue
            off = bias_offset(kind, nq, nk)
            bias = np.full((hq, nq, nk), -np.inf)
            for i in range(nq):
                a, b = row_range(kind, i, nq, nk, w)
                js = np.arange(a, b)
                bias[:, i, a:b] = -sl[:, None] * np.abs(i + off - js)[None, :]
            qs = torch.tensor(q[cq[s_]:cq[s_ + 1]].transpose(1, 0, 2), requires_grad=True)
            ks = torch.tensor(k[ck[s_]:ck[s_ + 1]].transpose(1, 0, 2), requires_grad=True)
            vs = torch.tensor(v[ck[s_]:ck[s_ + 1]].transpose(1, 0, 2), requires_grad=True)
            ri = torch.tensor(rows)
            out = torch.nn.functional.scaled_dot_product_attention(
                qs[:, ri], ks.repeat_interleave(g, dim=0), vs.repeat_interleave(g, dim=0),
                attn_mask=torch.tensor(bias[:, rows]), scale=scale)
            dot = torch.tensor(do[cq[s_]:cq[s_ + 1]].transpose(1, 0, 2))[:, ri]
            (out * dot).sum().backward()
            np.testing.assert_allclose(o[cq[s_]:cq[s_ + 1]][rows], out.detach().numpy().transpose(1, 0, 2),
                                       rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(dq[cq[s_]:cq[s_ + 1]][rows],
                                       qs.grad.numpy().transpose(1, 0, 2)[rows], rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dk[ck[s_]:ck[s_ + 1]], ks.grad.numpy().transpose(1, 0, 2),
                                       rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dv[ck[s_]:ck[s_ + 1]], vs.grad.numpy().transpose(1, 0, 2),
                                       rtol=1e-9, atol=1e-11)


def pin_bias_finite_differences(orc):
    """Central differences of L = sum O * dO with a bias (the bias does not
    depend on Q, K or V, so the gradients keep their form)."""
    rng = np.random.default_rng(45)
    lq, lk = (3, 4), (5, 4)
    hq, hkv, d, scale = 2, 1, 3, 0.7
    q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
    do = rng.standard_normal(q.shape)
    sl = np.array([0.3, 1.1])
    for kind in (BOTTOM_RIGHT, NONE):
        dq, dk, dv, _, _ = orc.bwd(q, k, v, do, cu(lq), cu(lk), scale, kind, slopes=sl)

        def loss(qq, kk, vv):
            o, _ = orc.fwd(qq, kk, vv, cu(lq), cu(lk), scale, kind, slopes=sl)
            return float((o * do).sum())

        h = 1e-5
        for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            fd = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xs = []
                for sign in (1.0, -1.0):
                    xx = x.copy()
                    xx[idx] += sign * h
                    xs.append({"q": (xx, k, v), "k": (q, xx, v), "v": (q, k, xx)}[name])
                fd[idx] = (loss(*xs[0]) - loss(*xs[1])) / (2 * h)
            np.testing.assert_allclose(grad, fd, rtol=1e-6, atol=1e-8, err_msg=(name, kind))


def rand_btab(rng, lq, lk, hq, p_minf=0.2):
    """A random explicit bias tensor [B, Hq, max Nq, max Nk]: N(0, 1) entries,
    about ``p_minf`` of them -inf (masked pairs)."""
    b = rng.standard_normal((len(lq), hq, max(max(lq), 1), max(max(lk), 1)))
    b[rng.random(b.shape) < p_minf] = -np.inf
    return b


def pin_tab_torch_sdpa_fp64(orc):
    """torch's fp64 reference attention with the causal rule and the explicit
    bias tensor together as one additive float mask, forward, lse and every
    gradient, on the rows that keep at least one finite logit."""
    rng = np.random.default_rng(46)
    for (lq, lk, hq, hkv, d, kind) in SHAPES:
        q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
        do = rng.standard_normal(q.shape)
        bt = rand_btab(rng, lq, lk, hq)
        scale = 1.0 / math.sqrt(d)
        dq, dk, dv, o, lse = orc.bwd(q, k, v, do, cu(lq), cu(lk), scale, kind, bias=bt)
        g = hq // hkv
        cq, ck = cu(lq), cu(lk)
        for s_, (nq, nk) in enumerate(zip(lq, lk)):
            full = np.full((hq, nq, nk), -np.inf)
            for i in range(nq):
                a, b = row_range(kind, i, nq, nk)
                full[:, i, a:b] = bt[s_, :, i, a:b]
            live = np.isfinite(full).any(axis=2)  # [hq, nq]
            for h in range(hq):
                for i in range(nq):
                    t = cq[s_] + i
                    if not live[h, i]:
                        assert np.isneginf(lse[h, t]) and np.all(o[t, h] == 0) and np.all(dq[t, h] == 0)
            qs = torch.tensor(q[cq[s_]:cq[s_ + 1]].transpose(1, 0, 2), requires_grad=True)
            ks = torch.tensor(k[ck[s_]:ck[s_ + 1]].transpose(1, 0, 2), requires_grad=True)
            vs = torch.tensor(v[ck[s_]:ck[s_ + 1]].transpose(1, 0, 2), requires_grad=True)
            if not live.any():
                continue
            # dead rows get a harmless finite mask in torch and no upstream gradient
            safe = np.where(live[:, :, None], full, 0.0)
            wgt = torch.tensor(live[:, :, None].astype(np.float64))
            kr, vr = ks.repeat_interleave(g, dim=0), vs.repeat_interleave(g, dim=0)
            out = torch.nn.functional.scaled_dot_product_attention(
                qs, kr, vr, attn_mask=torch.tensor(safe), scale=scale)
            dot = torch.tensor(do[cq[s_]:cq[s_ + 1]].transpose(1, 0, 2))
            (out * dot * wgt).sum().backward()
            ref_lse = torch.logsumexp(qs.detach() @ kr.detach().transpose(1, 2) * scale
                                      + torch.tensor(full), dim=2).numpy()
            ot = out.detach().numpy().transpose(1, 0, 2)
            for h in range(hq):
                rows = np.nonzero(live[h])[0]
                np.testing.assert_allclose(o[cq[s_] + rows, h], ot[rows, h], rtol=1e-10, atol=1e-12)
                np.testing.assert_allclose(lse[h, cq[s_] + rows], ref_lse[h, rows], rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(dq[cq[s_] + rows, h],
                                           qs.grad.numpy().transpose(1, 0, 2)[rows, h], rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dk[ck[s_]:ck[s_ + 1]], ks.grad.numpy().transpose(1, 0, 2),
                                       rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(dv[ck[s_]:ck[s_ + 1]], vs.grad.numpy().transpose(1, 0, 2),
                                       rtol=1e-9, atol=1e-11)


def pin_tab_zero_and_broadcast(orc):
    """A zero bias tensor changes nothing (bit for bit), and a tensor of one
    sequence or one head gives exactly what its explicit expansion gives."""
    rng = np.random.default_rng(47)
    lq, lk, hq, hkv, d = (4, 6), (7, 6), 4, 2, 5
    q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
    for kind in (NONE, TOP_LEFT, BOTTOM_RIGHT):
        o0, l0 = orc.fwd(q, k, v, cu(lq), cu(lk), 0.4, kind)
        o1, l1 = orc.fwd(q, k, v, cu(lq), cu(lk), 0.4, kind, bias=np.zeros((1, 1, 6, 7)))
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
        for shape in ((1, hq, 6, 7), (2, 1, 6, 7), (1, 1, 6, 7)):
            b = rng.standard_normal(shape)
            ob, lb = orc.fwd(q, k, v, cu(lq), cu(lk), 0.4, kind, bias=b)
            oe, le = orc.fwd(q, k, v, cu(lq), cu(lk), 0.4, kind,
                             bias=np.ascontiguousarray(np.broadcast_to(b, (2, hq, 6, 7))))
            assert np.array_equal(ob, oe) and np.array_equal(lb, le)


def pin_tab_row_constant(orc):
    """A bias that is constant along a row's keys leaves O unchanged and adds
    the constant to lse (softmax is shift-invariant)."""
    rng = np.random.default_rng(48)
    lq, lk, hq, hkv, d = (5, 3), (5, 8), 2, 1, 4
    q, k, v = rand_case(rng, lq, lk, hq, hkv, d)
    c = rng.uniform(-3, 3, (2, hq, 5))
    b = np.repeat(c[:, :, :, None], 8, axis=3)
    for kind in (TOP_LEFT, BOTTOM_RIGHT):
        o0, l0 = orc.fwd(q, k, v, cu(lq), cu(lk), 0.6, kind)
        o1, l1 = orc.fwd(q, k, v, cu(lq), cu(lk), 0.6, kind, bias=b)
        np.testing.assert_allclose(o1, o0, rtol=1e-12, atol=1e-14)
        cq = cu(lq)
        for s_, nq in enumerate(lq):
            for i in range(nq):
                t = cq[s_] + i
                for h in range(hq):
                    if np.isfinite(l0[h, t]):
                        np.testing.assert_allclose(l1[h, t], l0[h, t] + c[s_, h, i], rtol=1e-12, atol=1e-12)


ALL_PINS = [
    pin_token_meta, pin_mask_intervals, pin_golden_mask_counts,
    pin_window_counts, pin_window_one_key, pin_window_covering_is_causal,
    pin_uniform_logits, pin_single_dominant_score, pin_masked_dominant_score,
    pin_row_shift, pin_permutation_noncausal, pin_gqa_vs_repeat,
    pin_packed_vs_separate, pin_torch_sdpa_fp64, pin_finite_differences,
    pin_dv_column_sum, pin_dq_key_shift, pin_scale_identity,
    pin_empty_rows_backward, pin_bias_uniform_logits, pin_bias_zero_slopes,
    pin_bias_torch_sdpa_fp64, pin_bias_finite_differences,
    pin_tab_torch_sdpa_fp64, pin_tab_zero_and_broadcast, pin_tab_row_constant,
]
