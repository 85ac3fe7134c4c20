"""A CPU model, in fp64, of the tiled online-softmax recurrence that the CUDA
forward runs, checked against the oracle ("formal-correctness", "The
FlashAttention Proof": running max, rescale of the denominator and the
accumulator when the max moves, new exponentiated terms, final divide; and the
invariant that the online denominator equals the recomputed denominator at the
current max).

The model works on one query row at a time over key tiles of ``bc`` lanes; a
tile that runs past the sequence end has out-of-range lanes, which are masked
before the max ("causal-mask-and-ragged-sequence-layouts", second paragraph).
It also models the lazy-rescale variant the GPU kernels use: the reference max
only moves when the new max exceeds it by more than ``tau`` (in log2 units),
which is exact because O and l always share the same reference.

Mutants of the recurrence (the bug classes the "formal-correctness" page
lists) must disagree with the oracle on the pinned inputs.
"""
import math

import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins

LOG2E = 1.0 / math.log(2.0)


def online_row(s_row, allowed, v_rows, bc, tau=0.0, mutant=None, check=None):
    """Online softmax of one row.  s_row: scaled logits over the sequence's
    keys, allowed: bool per key, v_rows: [nk, d].  Returns (o, lse)."""
    nk, d = v_rows.shape
    m = -math.inf   # reference max, log2 units
    l = 0.0
    acc = np.zeros(d)
    n_tiles = (nk + bc - 1) // bc
    for t in range(n_tiles):
        lanes = range(t * bc, (t + 1) * bc)
        x = np.full(bc, -math.inf)
        for c, j in enumerate(lanes):
            in_range = j < nk
            if mutant == "out_of_range_counted" and not in_range:
                x[c] = 0.0
            elif in_range and (allowed[j] or mutant == "mask_after_max"):
                x[c] = s_row[j] * LOG2E
        tile_max = x.max()
        if mutant == "mask_after_max":
            for c, j in enumerate(lanes):
                if j < nk and not allowed[j]:
                    x[c] = -math.inf
        m_new = m
        if tile_max > m + tau or m == -math.inf:
            m_new = max(m, tile_max)
        alpha = 1.0 if m_new == -math.inf else 2.0 ** (m - m_new)
        p = np.where(np.isneginf(x), 0.0,
                     np.exp2(np.where(np.isneginf(x), 0.0, x - (m_new if m_new > -math.inf else 0.0))))
        if mutant != "no_l_rescale":
            l = alpha * l
        l += p.sum()
        if mutant != "no_o_rescale":
            acc = alpha * acc
        for c, j in enumerate(lanes):
            if j < nk and p[c] != 0.0:
                acc += p[c] * v_rows[j]
        m = m_new
        if check is not None:
            check(t, m, l, lanes)
    if l == 0.0:
        return np.zeros(d), -math.inf
    return acc / l, (m + math.log2(l)) / LOG2E


def model_fwd(q, k, v, lq, lk, hq, hkv, scale, kind, bc, tau=0.0, mutant=None,
              invariant=False):
    g = hq // hkv
    cq, ck = pins.cu(lq), pins.cu(lk)
    o = np.zeros(q.shape)
    lse = np.zeros((hq, q.shape[0]))
    for s, (nq, nk) in enumerate(zip(lq, lk)):
        off = 0 if kind == pins.TOP_LEFT else nk - nq
        for i in range(nq):
            t = cq[s] + i
            allowed = np.array([kind == pins.NONE or j <= i + off for j in range(nk)])
            if mutant == "global_position":
                allowed = np.array([kind == pins.NONE or ck[s] + j <= i + off
                                    for j in range(nk)])
            for h in range(hq):
                kv = h // g
                s_row = scale * (k[ck[s]:ck[s + 1], kv] @ q[t, h])
                check = None
                if invariant:
                    def check(tile, m, l, lanes, s_row=s_row, allowed=allowed):
                        seen = [j for j in range(min(lanes[-1] + 1, nk)) if allowed[j]]
                        ref = sum(2.0 ** (s_row[j] * LOG2E - m) for j in seen)
                        assert abs(l - ref) <= 1e-12 * max(1.0, ref), (tile, l, ref)
                o[t, h], lse[h, t] = online_row(s_row, allowed, v[ck[s]:ck[s + 1], kv],
                                                bc, tau, mutant, check)
    return o, lse


CASES = [
    ((5, 1, 9), (5, 1, 9), 2, 1, 4, pins.TOP_LEFT),
    ((3, 7), (9, 4), 2, 2, 3, pins.BOTTOM_RIGHT),
    ((6,), (6,), 1, 1, 4, pins.NONE),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("tau", [0.0, 8.0])
def test_tile_model_equals_oracle(case, tau):
    lq, lk, hq, hkv, d, kind = CASES[case]
    rng = np.random.default_rng(30 + case)
    q, k, v = pins.rand_case(rng, lq, lk, hq, hkv, d)
    q *= 3.0  # spread the logits so the max moves between tiles
    o_ref, l_ref = oracle.fwd(q, k, v, pins.cu(lq), pins.cu(lk), 0.5, kind)
    o, l = model_fwd(q, k, v, lq, lk, hq, hkv, 0.5, kind, bc=2, tau=tau, invariant=True)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    fin = np.isfinite(l_ref)
    assert np.array_equal(fin, np.isfinite(l))
    np.testing.assert_allclose(l[fin], l_ref[fin], rtol=1e-12, atol=1e-12)


def _rising_case():
    """Scores that rise along the keys, so the running max moves in every
    tile, plus a masked dominant key."""
    lq = lk = (6, 5)
    d = 2
    q = np.zeros((11, 1, d))
    q[:, 0, 0] = 1.0
    k = np.zeros((11, 1, d))
    k[:, 0, 0] = np.array([0, 1, 2, 3, 4, 1000, 0, 1, 2, 3, 4], float)
    rng = np.random.default_rng(31)
    v = rng.standard_normal((11, 1, d))
    return q, k, v, lq, lk


@pytest.mark.parametrize("mutant", ["no_l_rescale", "no_o_rescale", "mask_after_max",
                                    "out_of_range_counted", "global_position"])
def test_recurrence_mutants_disagree(mutant):
    q, k, v, lq, lk = _rising_case()
    o_ref, l_ref = oracle.fwd(q, k, v, pins.cu(lq), pins.cu(lk), 1.0, pins.TOP_LEFT)
    o, l = model_fwd(q, k, v, lq, lk, 1, 1, 1.0, pins.TOP_LEFT, bc=4, mutant=mutant)
    bad = ~np.isclose(o, o_ref, rtol=1e-6, atol=1e-6).all() or \
        ~np.isclose(l, l_ref, rtol=1e-6, atol=1e-6).all()
    assert bad, f"mutant {mutant} not detected"
