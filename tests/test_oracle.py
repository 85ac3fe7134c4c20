"""The fp64 oracle against its pins (CPU only)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(orc, pin):
    pin(orc)


def test_sampled_backward_equals_full(orc):
    rng = np.random.default_rng(20)
    lq, lk = (5, 7), (6, 7)
    q, k, v = pins.rand_case(rng, lq, lk, 4, 2, 5)
    do = rng.standard_normal(q.shape)
    cq, ck = pins.cu(lq), pins.cu(lk)
    for kind in (pins.TOP_LEFT, pins.BOTTOM_RIGHT, pins.NONE):
        dq, dk, dv, o, lse = orc.bwd(q, k, v, do, cq, ck, 0.5, kind)
        qr = [(t, h) for t in range(12) for h in range(4)]
        kr = [(u, h) for u in range(13) for h in range(2)]
        sq, sk, sv = orc.bwd_sampled(q, k, v, do, cq, ck, 0.5, kind, qr, kr)
        np.testing.assert_allclose(sq, np.array([dq[t, h] for t, h in qr]), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(sk, np.array([dk[u, h] for u, h in kr]), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(sv, np.array([dv[u, h] for u, h in kr]), rtol=1e-12, atol=1e-14)


def test_row_subset_equals_full(orc):
    rng = np.random.default_rng(21)
    lq, lk = (3, 9), (3, 9)
    q, k, v = pins.rand_case(rng, lq, lk, 2, 1, 4)
    o, lse = orc.fwd(q, k, v, pins.cu(lq), pins.cu(lk), 0.5, pins.TOP_LEFT)
    rows = [(11, 1), (0, 0), (3, 1)]
    o2, l2 = orc.fwd(q, k, v, pins.cu(lq), pins.cu(lk), 0.5, pins.TOP_LEFT, rows=rows)
    for r, (t, h) in enumerate(rows):
        assert np.array_equal(o2[r], o[t, h]) and l2[r] == lse[h, t]


@pytest.mark.parametrize("cu_bad", [[1, 3], [0, 4, 2], [0, 2]])
def test_invalid_cu_seqlens_rejected(orc, cu_bad):
    total = 3
    q = np.zeros((total, 1, 2))
    with pytest.raises(ValueError):
        orc.fwd(q, q, q, np.array(cu_bad), np.array(cu_bad), 1.0, 1)
