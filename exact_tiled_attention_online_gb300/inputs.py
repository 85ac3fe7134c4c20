"""Seeded synthetic inputs for the attention workloads.

This module draws random tensors and packs cumulative sequence lengths; it
holds none of the attention arithmetic, so both the CUDA path and the fp64
oracle can be fed from it without sharing any of the method.

Recipe (the pages fix no generator, so this is a stated choice):
  * a ``torch.Generator`` on the CPU (or on the target device for inputs too
    large to round-trip through host memory) seeded with ``1000 + index``;
  * Q, K, V and, when a backward is wanted, dO are drawn in that order as
    fp32 N(0, 1) and then cast to the workload dtype (round to nearest even);
  * for the packed ragged workload, the value rows of sequence ``s`` are
    shifted by ``10 * s`` before the cast, so that any leakage between packed
    sequences is visible in the output ("causal-mask-and-ragged-sequence-
    layouts", fifth paragraph);
  * every ragged batch is packed back to back and addressed by int32
    cumulative lengths ``cu_seqlens = [0, L0, L0 + L1, ...]``.
  * an explicit bias tensor is drawn by its own generator (seed + 1) as
    fp32 N(0, 1) entries with about a fifth of them set to -inf.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

MASK_NONE = 0
MASK_TOP_LEFT = 1
MASK_BOTTOM_RIGHT = 2


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem shape: ragged lengths, heads, width, dtype."""

    name: str
    seqlens_q: tuple
    seqlens_k: tuple
    hq: int
    hkv: int
    d: int
    dtype: str  # "bf16" or "fp32"
    mask: int
    seed: int
    backward: bool = False
    v_shift_per_seq: float = 0.0
    window: int = 0  # > 0: bounded causal window of that many keys per row
    bias: bool = False  # linear positional bias with slopes bias_slopes(hq)
    bias_tensor: bool = False  # explicit bias tensor bias_tensor(B, 1, max_q, max_k, seed + 1)

    @property
    def batch(self) -> int:
        return len(self.seqlens_q)

    @property
    def total_q(self) -> int:
        return int(sum(self.seqlens_q))

    @property
    def total_k(self) -> int:
        return int(sum(self.seqlens_k))

    @property
    def max_q(self) -> int:
        return int(max(self.seqlens_q)) if self.seqlens_q else 0

    @property
    def max_k(self) -> int:
        return int(max(self.seqlens_k)) if self.seqlens_k else 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


VARLEN_LENGTHS = (1, 63, 64, 65, 127, 128, 129, 255, 256, 257, 1000, 2048)

# The five workloads the attention pages' methodology calls for, by name.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", (64,), (64,), 1, 1, 64, "fp32",
                          MASK_TOP_LEFT, 1000),
    "varlen_causal": Workload("varlen_causal", VARLEN_LENGTHS, VARLEN_LENGTHS,
                              16, 16, 128, "bf16", MASK_TOP_LEFT, 1001,
                              v_shift_per_seq=10.0),
    "gqa_prefill": Workload("gqa_prefill", (4096,) * 4, (4096,) * 4, 32, 8, 128,
                            "bf16", MASK_TOP_LEFT, 1002),
    "decode_q1": Workload("decode_q1", (1,) * 32, (32768,) * 32, 32, 8, 128,
                          "bf16", MASK_BOTTOM_RIGHT, 1003),
    "decode_q16": Workload("decode_q16", (16,) * 32, (32768,) * 32, 32, 8, 128,
                           "bf16", MASK_BOTTOM_RIGHT, 1003),
    "decode_empty_rows": Workload("decode_empty_rows", (64,) * 32, (32,) * 32,
                                  32, 8, 128, "bf16", MASK_BOTTOM_RIGHT, 1003),
    "train_fwd_bwd": Workload("train_fwd_bwd", (8192,) * 2, (8192,) * 2, 16, 4,
                              128, "bf16", MASK_TOP_LEFT, 1004, backward=True),
    # the prefill shape under a bounded causal window (linear pair work)
    "window_prefill": Workload("window_prefill", (4096,) * 4, (4096,) * 4, 32, 8,
                               128, "bf16", MASK_TOP_LEFT, 1002, window=1024),
    # the prefill shape with a linear positional bias on every logit
    "bias_prefill": Workload("bias_prefill", (4096,) * 4, (4096,) * 4, 32, 8,
                             128, "bf16", MASK_TOP_LEFT, 1002, bias=True),
    # the prefill shape with an explicit [B, 1, N, N] bias tensor shared by the
    # heads (a fifth of its entries -inf)
    "bias_tensor_prefill": Workload("bias_tensor_prefill", (4096,) * 4, (4096,) * 4, 32, 8,
                                    128, "bf16", MASK_TOP_LEFT, 1002, bias_tensor=True),
    # the training shape with an explicit [B, 1, N, N] bias tensor, forward + backward
    "bias_tensor_train": Workload("bias_tensor_train", (8192,) * 2, (8192,) * 2, 16, 4,
                                  128, "bf16", MASK_TOP_LEFT, 1004, backward=True,
                                  bias_tensor=True),
}


def bias_slopes(hq: int) -> torch.Tensor:
    """Slopes of the positional-bias workloads: head h gets 2^(-8 (h + 1) / hq),
    a geometric sequence from steep to nearly flat (a stated choice; the pages
    fix no slopes)."""
    return torch.tensor([2.0 ** (-8.0 * (h + 1) / hq) for h in range(hq)], dtype=torch.float32)


def bias_tensor(batch: int, hb: int, rows: int, keys: int, seed: int, p_masked: float = 0.2,
                dead_rows: int = 0) -> torch.Tensor:
    """A seeded explicit bias tensor [batch, hb, rows, keys] (fp32, CPU):
    N(0, 1) entries, about ``p_masked`` of them -inf, and in addition
    ``dead_rows`` random (sequence, head, row) triples masked over every key.
    Use ``batch`` or ``hb`` = 1 for a tensor that broadcasts."""
    g = torch.Generator().manual_seed(seed)
    b = torch.randn((batch, hb, rows, keys), generator=g, dtype=torch.float32)
    b[torch.rand(b.shape, generator=g) < p_masked] = float("-inf")
    for _ in range(dead_rows):
        s = int(torch.randint(batch, (1,), generator=g))
        h = int(torch.randint(hb, (1,), generator=g))
        i = int(torch.randint(rows, (1,), generator=g))
        b[s, h, i, :] = float("-inf")
    return b


def cu_seqlens(lengths: Sequence[int]) -> torch.Tensor:
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp32": torch.float32}[name]


def make_inputs(w: Workload, device: str = "cpu", gen_device: str = "cpu",
                backward: Optional[bool] = None) -> dict:
    """Draw the workload's tensors.  Returns a dict with q, k, v (and dout),
    cu_seqlens_q/k (int32, on ``device``) and the Workload itself.

    ``gen_device`` picks where the generator runs: "cpu" gives the reference
    stream that tests reproduce exactly; a CUDA device gives a different but
    identically distributed stream without a host round trip.
    """
    want_bwd = w.backward if backward is None else backward
    g = torch.Generator(device=gen_device)
    g.manual_seed(w.seed)
    dt = torch_dtype(w.dtype)

    def draw(rows: int, heads: int) -> torch.Tensor:
        return torch.randn((rows, heads, w.d), generator=g, device=gen_device,
                           dtype=torch.float32)

    q = draw(w.total_q, w.hq)
    k = draw(w.total_k, w.hkv)
    v = draw(w.total_k, w.hkv)
    if w.v_shift_per_seq:
        start = 0
        for s, n in enumerate(w.seqlens_k):
            v[start:start + n] += w.v_shift_per_seq * s
            start += n
    out = {"q": q.to(dt), "k": k.to(dt), "v": v.to(dt)}
    if want_bwd:
        out["dout"] = draw(w.total_q, w.hq).to(dt)
    out = {name: t.to(device) for name, t in out.items()}
    out["cu_seqlens_q"] = cu_seqlens(w.seqlens_q).to(device)
    out["cu_seqlens_k"] = cu_seqlens(w.seqlens_k).to(device)
    out["workload"] = w
    return out


def custom(name: str, seqlens_q, seqlens_k, hq: int, hkv: int, d: int,
           dtype: str = "bf16", mask: int = MASK_TOP_LEFT, seed: int = 7,
           backward: bool = False, v_shift_per_seq: float = 0.0,
           window: int = 0) -> Workload:
    """A Workload for tests (small ragged shapes, edge cases)."""
    return Workload(name, tuple(int(x) for x in seqlens_q),
                    tuple(int(x) for x in seqlens_k), hq, hkv, d, dtype, mask,
                    seed, backward, v_shift_per_seq, int(window))
