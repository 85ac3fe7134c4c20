"""Shared helpers for the GPU parity tests: run the CUDA path through the
binding and the oracle on the same seeded inputs."""
import contextlib

import numpy as np
import torch

import oracle
from exact_tiled_attention_online_gb300 import attn, inputs


def run_fwd(x, mask=None):
    w = x["workload"]
    dev = {k: (t.cuda() if hasattr(t, "cuda") else t) for k, t in x.items()}
    o, lse = attn.fwd(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"], dev["cu_seqlens_k"],
                      w.max_q, w.max_k, w.mask if mask is None else mask, w.scale,
                      window=w.window)
    torch.cuda.synchronize()
    assert attn.get_device_error() == 0
    return o, lse, dev


def oracle_fwd(x, rows=None):
    w = x["workload"]
    return oracle.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.scale,
                      w.mask, rows=rows, window=w.window)


@contextlib.contextmanager
def backward_form(deterministic):
    """Run the enclosed calls with the two-kernel (True) or the fused (False)
    bf16 backward, then restore the previous setting."""
    prev = attn.get_deterministic()
    attn.set_deterministic(deterministic)
    try:
        yield
    finally:
        attn.set_deterministic(prev)


def tc_backward(plan):
    """The plan ran a tensor-core backward (fused or two-kernel)."""
    return "bwd_dq_tc" in plan or "bwd_fused_tc" in plan


def sample_rows(w, n, seed):
    """(token, head) rows for sampled checks: the first and last row of
    every sequence plus uniform random rows."""
    rng = np.random.default_rng(seed)
    cu = inputs.cu_seqlens(w.seqlens_q).numpy()
    rows = []
    for s in range(w.batch):
        if cu[s + 1] > cu[s]:
            rows.append((cu[s], rng.integers(w.hq)))
            rows.append((cu[s + 1] - 1, rng.integers(w.hq)))
    for _ in range(n):
        rows.append((rng.integers(w.total_q), rng.integers(w.hq)))
    return np.array(rows, np.int64)
