"""The tile planner and lane predicate the kernels use, dumped by the mask
probe, equal the oracle's materialised mask bit for bit
("causal-mask-and-ragged-sequence-layouts", first to fourth paragraphs)."""
import numpy as np
import pytest
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs

pytestmark = pytest.mark.gpu

SHAPES = [
    ((63, 64, 65, 127, 128, 129, 255, 256, 257), None),
    ((1, 16, 64), (300, 16, 32)),      # Nq < Nk and Nq > Nk
    ((0, 5, 0, 130), (7, 5, 0, 130)),  # zero-length segments
    ((200,), (70,)),
    ((1,) * 4, (129, 128, 1, 257)),
]


@pytest.mark.parametrize("shape", range(len(SHAPES)))
@pytest.mark.parametrize("mask", [0, 1, 2])
@pytest.mark.parametrize("tile_rows", [16, 32, 128])
def test_probe_equals_oracle_mask(shape, mask, tile_rows):
    lq, lk = SHAPES[shape]
    lk = lk or lq
    cq, ck = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    tq, tk = int(cq[-1]), int(ck[-1])
    got = attn.mask_probe(cq.cuda(), ck.cuda(), max(lq), max(lk), tq, tk, mask, tile_rows)
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    ref = oracle.mask(cq.numpy(), ck.numpy(), tq, tk, mask)
    g = got.cpu().numpy()
    if not np.array_equal(g, ref):
        bad = np.argwhere(g != ref)[:10]
        raise AssertionError(f"mask differs at {bad.tolist()}")


def test_probe_config_sizes():
    """The decode and empty-row configurations' geometry (one sequence)."""
    for lq, lk, mask in (((1,), (32768,), 2), ((16,), (32768,), 2), ((64, 64), (32, 32), 2),
                         ((4096,), (4096,), 1)):
        cq, ck = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
        tq, tk = int(cq[-1]), int(ck[-1])
        for tr in (32, 128):
            got = attn.mask_probe(cq.cuda(), ck.cuda(), max(lq), max(lk), tq, tk, mask, tr)
            ref = oracle.mask(cq.numpy(), ck.numpy(), tq, tk, mask)
            assert np.array_equal(got.cpu().numpy(), ref)
