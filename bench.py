"""Benchmark of the exact tiled attention hot path on one or more GB300s.

One step runs every workload of the hot path once on seeded synthetic inputs
that are already resident in HBM:

  gqa_prefill     causal GQA prefill forward, B=4, N=4096, 32/8 heads, d=128
                  (the headline: ``value`` is its TFLOP/s);
  decode_q1/q16   split-KV decode, B=32, Nk=32768, Nq=1 / 16, bottom-right;
  train_fwd_bwd   forward + backward, B=2, N=8192, 16/4 heads, d=128;
  varlen_causal   packed ragged forward, 12 sequences, 16 heads, d=128;
  window_prefill  the gqa_prefill shape under a bounded 1024-key causal window;
  bias_prefill    the gqa_prefill shape with a linear positional bias;
  bias_tensor_prefill  the gqa_prefill shape with an explicit [B, 1, N, N]
                  bias tensor shared by the heads;
  bias_tensor_train    the train_fwd_bwd shape with such a tensor, forward +
                  backward;
  train_fwd_bwd_plain  train_fwd_bwd without keeping the forward's fp32
                  output, so the backward recomputes it for its D term;
  train_fwd_bwd_det    train_fwd_bwd with the two-kernel backward, whose
                  gradients are reproducible bit for bit (the default
                  fused backward sums dQ with reductions).

Every workload is timed with CUDA events on the launching stream after an L2
flush (a 256 MiB write), W warm-up steps first, K timed steps, medians and
tails reported ("attention-kernel-portability-and-benchmarking", fourth
paragraph).  Work counts only allowed (query, key) pairs: 4 d flops per pair
forward, 10 d backward; decode bytes are one read of the K/V cache plus Q, O
and lse.

Output: one JSON line on stdout (the summary: headline, roofline, e2e,
clocks, CPU baselines, then every workload's value, unit, median time and
roofline fraction at the end of the line) and one JSON line on stderr with
the details (kernel plans, p90 and max times, memory).

``--impl reference`` times the fp64 CPU oracle instead, on bounded samples of
the same workload, on the host cores.

Under torchrun every rank runs its own replica of the workloads (the work
shards by sequence and head with no exchange), timings take the max over
ranks and ``value`` sums the ranks' work.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_tiled_attention_online_gb300 import inputs  # noqa: E402

HEADLINE = "gqa_prefill"
METRIC = "attention TFLOP/s (fwd, fwd+bwd) and decode HBM GB/s, % of GB300 roofline"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------------
# work accounting (closed-form pair counts of the alignment rules)
# --------------------------------------------------------------------------
def row_keys(mask, i, nq, nk, window=0):
    """Allowed keys of in-sequence row i (closed form)."""
    if mask == inputs.MASK_NONE:
        return nk
    off = 0 if mask == inputs.MASK_TOP_LEFT else nk - nq
    end = max(0, min(i + off + 1, nk))
    begin = max(0, min(i + off + 1 - window, nk)) if window > 0 else 0
    return end - begin


def allowed_pairs(w) -> int:
    """Allowed (query, key) pairs over all sequences and query heads: row i
    sees the keys in [clip(b + 1 - W), clip(b + 1)) with causal bound b
    (W unbounded without a window)."""
    total = 0
    for nq, nk in zip(w.seqlens_q, w.seqlens_k):
        i = np.arange(nq, dtype=np.int64)
        if w.mask == inputs.MASK_NONE:
            total += nq * nk
        else:
            off = 0 if w.mask == inputs.MASK_TOP_LEFT else nk - nq
            end = np.clip(i + off + 1, 0, nk)
            begin = np.clip(i + off + 1 - w.window, 0, nk) if w.window > 0 else 0
            total += int((end - begin).sum())
    return total * w.hq


def fwd_flops(w) -> float:
    return 4.0 * w.d * allowed_pairs(w)


def bwd_flops(w) -> float:
    return 10.0 * w.d * allowed_pairs(w)


def decode_bytes(w) -> float:
    kv = 2 * w.total_k * w.hkv * w.d * 2
    q_o = 2 * w.total_q * w.hq * w.d * 2
    return float(kv + q_o + w.total_q * w.hq * 4)


def alu_peak_tflops(peaks) -> float:
    """fp32 FMA peak of the whole GPU: SMs x 128 lanes x 2 flops x clock."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() \
        else 152
    return sms * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def count_kernels(plan: str) -> int:
    """Our kernels in one call, from the plan string ('+'-joined names)."""
    head = plan.split(" ")[0]
    n = len([p for p in head.split("+") if p])
    if "+combine" in plan and "+combine" not in head:
        n += 1
    return n


# --------------------------------------------------------------------------
# clocks sampling
# --------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:8]):
                if flag.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
class Runner:
    """Inputs, outputs and workspaces of one workload, allocated once."""

    def __init__(self, name, device, gen_device, batch_div=1):
        from exact_tiled_attention_online_gb300 import attn
        self.attn = attn
        self.name = name
        base = name
        for suffix in ("_plain", "_det"):
            if base.endswith(suffix):
                base = base[:-len(suffix)]
        self.w = inputs.WORKLOADS[base]
        self.two_kernel = name.endswith("_det")
        if batch_div > 1:  # a smaller case of the same kernels, for profiler captures
            w = self.w
            b = max(1, w.batch // batch_div)
            self.w = dataclasses.replace(w, seqlens_q=w.seqlens_q[:b], seqlens_k=w.seqlens_k[:b])
        x = inputs.make_inputs(self.w, device=device, gen_device=gen_device)
        self.x = x
        w = self.w
        self.o = torch.empty_like(x["q"])
        self.lse = torch.empty((w.hq, w.total_q), dtype=torch.float32, device=device)
        self.keep_o32 = w.backward and not name.endswith("_plain")
        self.o32 = torch.empty(x["q"].shape, dtype=torch.float32, device=device) \
            if self.keep_o32 else None
        ws = attn.fwd_workspace_size(w.batch, w.max_q, w.max_k, w.total_q, w.hq, w.hkv, w.d,
                                     attn.DTYPE_BF16, w.window)
        self.ws = torch.empty(max(ws, 1), dtype=torch.uint8, device=device)
        if w.backward:
            self.dq = torch.empty_like(x["q"])
            self.dk = torch.empty_like(x["k"])
            self.dv = torch.empty_like(x["v"])
            bws = attn.bwd_workspace_size(w.batch, w.max_q, w.max_k, w.total_q, w.total_k, w.hq,
                                          w.hkv, w.d, attn.DTYPE_BF16)
            self.bws = torch.empty(max(bws, 1), dtype=torch.uint8, device=device)
        self.slopes = inputs.bias_slopes(w.hq).to(device) if w.bias else None
        self.btab_cpu = inputs.bias_tensor(w.batch, 1, w.max_q, w.max_k, w.seed + 1) \
            if w.bias_tensor else None
        self.btab = None if self.btab_cpu is None else self.btab_cpu.to(device)
        self.plans = []
        self.ws_bytes = self.ws.numel() + (self.bws.numel() if w.backward else 0)

    def run(self):
        a, w, x = self.attn, self.w, self.x
        a.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.max_q, w.max_k,
              w.mask, w.scale, out=self.o, lse=self.lse, workspace=self.ws, o_f32=self.o32,
              window=w.window, bias_slopes=self.slopes, bias=self.btab)
        plans = [a.last_plan()]
        if w.backward:
            a.set_deterministic(self.two_kernel)
            try:
                a.bwd(x["q"], x["k"], x["v"], self.o, self.lse, x["dout"], x["cu_seqlens_q"],
                      x["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale, dq=self.dq,
                      dk=self.dk, dv=self.dv, workspace=self.bws, o_f32=self.o32,
                      window=w.window, bias_slopes=self.slopes, bias=self.btab)
                plans.append(a.last_plan())
            finally:
                a.set_deterministic(False)
        self.plans = plans

    def kernels_per_run(self):
        return sum(count_kernels(p) for p in self.plans)

    def work(self):
        w = self.w
        if self.name.startswith("decode"):
            return decode_bytes(w), "GB/s"
        f = fwd_flops(w) + (bwd_flops(w) if w.backward else 0.0)
        return f, "TFLOP/s"


def validate(r: Runner, n_rows=24):
    """Sampled rows against the oracle before any timing ("attention-kernel-
    portability-and-benchmarking", fifth paragraph)."""
    import oracle
    w = r.w
    rng = np.random.default_rng(123)
    rows = np.stack([rng.integers(w.total_q, size=n_rows), rng.integers(w.hq, size=n_rows)], 1)
    host = {k: (t.cpu() if hasattr(t, "cpu") else t) for k, t in r.x.items()}
    o_ref, l_ref = oracle.fwd(host["q"], host["k"], host["v"], host["cu_seqlens_q"],
                              host["cu_seqlens_k"], w.scale, w.mask, rows=rows, window=w.window,
                              slopes=inputs.bias_slopes(w.hq).double().numpy() if w.bias else None,
                              bias=r.btab_cpu)
    on = r.o.double().cpu().numpy()[rows[:, 0], rows[:, 1]]
    ln = r.lse.double().cpu().numpy()[rows[:, 1], rows[:, 0]]
    err = np.abs(on - o_ref)
    ok_o = bool(np.all(err <= 1e-2 + 1e-2 * np.abs(o_ref)))
    fin = np.isfinite(l_ref)
    ok_l = bool(np.array_equal(np.isfinite(ln), fin)) and bool(
        np.all(np.abs(ln[fin] - l_ref[fin]) <= 1e-4 * np.maximum(1, np.abs(l_ref[fin]))))
    return {"rows": int(n_rows), "max_abs_err_o": float(err.max()), "ok": ok_o and ok_l}


def time_gpu(args, rank, world, device):
    from exact_tiled_attention_online_gb300 import attn
    attn.library()
    torch.cuda.set_device(device)
    names = [n.strip() for n in args.workloads.split(",") if n.strip()]
    runners = {}
    memory = {}
    for n in names:  # each workload's buffers, then its first run, with its memory figures
        big = n.startswith("decode") or n.startswith("train_fwd_bwd") or n == "bias_tensor_train"
        torch.cuda.synchronize()
        before = torch.cuda.memory_allocated(device)
        torch.cuda.reset_peak_memory_stats(device)
        runners[n] = Runner(n, device, device if big else "cpu", args.batch_div)
        runners[n].run()
        torch.cuda.synchronize()
        memory[n] = {"workspace_bytes": int(runners[n].ws_bytes),
                     "buffers_bytes": int(torch.cuda.memory_allocated(device) - before),
                     "peak_allocated_bytes": int(torch.cuda.max_memory_allocated(device) - before),
                     "reserved_bytes": int(torch.cuda.memory_reserved(device))}
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    if attn.get_device_error() != 0:
        raise RuntimeError("device error flag set during the first run")
    validated = {}
    if rank == 0 and not args.skip_validate:
        for n in ("gqa_prefill", "varlen_causal", "bias_tensor_prefill"):
            if n in runners:
                validated[n] = validate(runners[n])

    for _ in range(args.warmup):
        for r in runners.values():
            flush.zero_()
            r.run()
    torch.cuda.synchronize()

    events = {n: [] for n in names}
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        t0 = time.perf_counter()
        for _ in range(args.steps):
            for n, r in runners.items():
                flush.zero_()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                r.run()
                e1.record(stream)
                events[n].append((e0, e1))
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    if attn.get_device_error() != 0:
        raise RuntimeError("device error flag set during the timed steps")

    # the headline again with L2 warm: back-to-back launches, no flush
    warm = {}
    if HEADLINE in runners:
        r = runners[HEADLINE]
        ev = []
        for _ in range(args.steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            r.run()
            e1.record(stream)
            ev.append((e0, e1))
        torch.cuda.synchronize()
        warm[HEADLINE] = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)

    per = {}
    for n, r in runners.items():
        ms = sorted(e0.elapsed_time(e1) for e0, e1 in events[n])
        work, unit = r.work()
        per[n] = {"ms_median": statistics.median(ms), "ms_p90": ms[int(0.9 * (len(ms) - 1))],
                  "ms_max": ms[-1], "work": work, "unit": unit, "plan": r.plans,
                  "kernels": r.kernels_per_run(), "memory": memory[n]}
        if n in warm:
            per[n]["ms_median_l2_warm"] = warm[n]
    per_total = {"max_memory_allocated": int(torch.cuda.max_memory_allocated(device)),
                 "max_memory_reserved": int(torch.cuda.max_memory_reserved(device))}
    return runners, per, wall, clocks.summary(), validated, per_total


def reduce_max(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def rate(work, unit, ms):
    if unit == "GB/s":
        return work / (ms * 1e-3) / 1e9
    return work / (ms * 1e-3) / 1e12


def e2e_headline(args, r: Runner, device):
    """The headline workload through the public API with host buffers: every
    step copies Q, K, V (and cu_seqlens) from pinned host memory, runs the
    forward, and reads O and lse back into pinned host memory.  Steps are
    pipelined the way a serving loop would run them: copies in, the kernel
    and copies out go on three streams with two device buffer sets, so step
    i + 1's inputs travel while step i computes and step i - 1's outputs come
    back; events order every reuse of a buffer.  (Splitting the copies over
    more streams measured no faster: the host link is the limit.)"""
    x, w = r.x, r.w
    names = ("q", "k", "v", "cu_seqlens_q", "cu_seqlens_k")
    host = {k: x[k].cpu().pin_memory() for k in names}
    o_h = [torch.empty(r.o.shape, dtype=r.o.dtype).pin_memory() for _ in range(2)]
    l_h = [torch.empty(r.lse.shape, dtype=r.lse.dtype).pin_memory() for _ in range(2)]
    dev = [{k: torch.empty_like(v, device=device) for k, v in host.items()} for _ in range(2)]
    outs = [(torch.empty_like(r.o), torch.empty_like(r.lse), torch.empty_like(r.ws))
            for _ in range(2)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(device=device) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):  # every buffer starts free
        for ev in (ev_cmp[b], ev_out[b]):
            ev.record(s_cmp)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_h[0].numel() * o_h[0].element_size() + l_h[0].numel() * l_h[0].element_size()

    def step(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_cmp[b])  # the kernel that read this input set is done
            for k in names:
                dev[b][k].copy_(host[k], non_blocking=True)
            ev_in[b].record(s_in)
        o, lse, ws = outs[b]
        s_cmp.wait_event(ev_in[b])
        s_cmp.wait_event(ev_out[b])  # this output set has been read back
        r.attn.fwd(dev[b]["q"], dev[b]["k"], dev[b]["v"], dev[b]["cu_seqlens_q"],
                   dev[b]["cu_seqlens_k"], w.max_q, w.max_k, w.mask, w.scale, out=o, lse=lse,
                   workspace=ws, window=w.window, stream=s_cmp)
        ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            o_h[b].copy_(o, non_blocking=True)
            l_h[b].copy_(lse, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_cmp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    for i in range(args.steps):
        step(i)
    s_cmp.wait_stream(s_in)
    s_cmp.wait_stream(s_out)
    e1.record(s_cmp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    # the last step's result is the one a caller would read: check it landed
    last = (args.steps - 1) & 1
    torch.testing.assert_close(o_h[last], outs[last][0].cpu(), rtol=0, atol=0)
    torch.testing.assert_close(l_h[last], outs[last][1].cpu(), rtol=0, atol=0)
    return ms, h2d, d2h


def set_oracle_threads(n):
    """OpenMP thread count for the oracle's next parallel regions (those
    started from this thread); None leaves the default (all cores)."""
    import ctypes
    try:
        gomp = ctypes.CDLL("libgomp.so.1")
    except OSError:
        return False
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    gomp.omp_set_num_threads(int(n) if n else int(os.environ.get("OMP_NUM_THREADS", cores)))
    return True


def cpu_baseline(workload: str, budget_s: float = 12.0, threads=None, repeats: int = 1):
    """The oracle, as it stands, on a bounded sample of the workload: random
    (token, head) rows of the forward (every row when the sample would cover
    the workload), timed on the host cores; the median of ``repeats`` runs.
    ``threads``: OpenMP threads (None: all cores)."""
    import oracle
    w = inputs.WORKLOADS[workload]
    x = inputs.make_inputs(w)
    rng = np.random.default_rng(7)
    q = x["q"].double().numpy()
    k = x["k"].double().numpy()
    v = x["v"].double().numpy()
    cq, ck = x["cu_seqlens_q"].numpy(), x["cu_seqlens_k"].numpy()
    orc = oracle.default()
    set_oracle_threads(threads)
    all_rows = w.total_q * w.hq

    def sample(n):
        if n >= all_rows:  # the whole workload
            rows = np.stack(np.meshgrid(np.arange(w.total_q), np.arange(w.hq), indexing="ij"),
                            -1).reshape(-1, 2)
        else:
            rows = np.stack([rng.integers(w.total_q, size=n), rng.integers(w.hq, size=n)], 1)
        t0 = time.perf_counter()
        orc.fwd(q, k, v, cq, ck, w.scale, w.mask, rows=rows, window=w.window)
        dt = time.perf_counter() - t0
        # allowed pairs of the sampled rows, by the closed form
        seq = np.searchsorted(cq, rows[:, 0], side="right") - 1
        pairs = 0
        for t, s in zip(rows[:, 0], seq):
            nq, nk = cq[s + 1] - cq[s], ck[s + 1] - ck[s]
            pairs += row_keys(w.mask, int(t - cq[s]), int(nq), int(nk), w.window)
        return dt, 4.0 * w.d * pairs

    dt, fl = sample(min(64, all_rows))
    n = int(min(200000, all_rows, max(64, 64 * budget_s / max(dt, 1e-3))))
    runs = [sample(n) for _ in range(max(1, repeats))]
    rates = sorted(f / d / 1e12 for d, f in runs)
    secs = sorted(d for d, _ in runs)
    set_oracle_threads(None)
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    used = int(threads) if threads else min(cores, int(os.environ.get("OMP_NUM_THREADS", cores)))
    what = "every (token, head) row" if n >= all_rows else f"{n} random (token, head) rows"
    return {"value": statistics.median(rates), "unit": "TFLOP/s", "cores": used,
            "kind": "oracle", "seconds": statistics.median(secs), "repeats": len(runs),
            "sample": f"{what} of {workload}, forward, fp64"}


def cpu_baseline_legs(budget_s: float = 1.5):
    """The oracle on the three forward workloads the CPU can take in part
    (tiny fp32, packed ragged, GQA prefill), single-core and on all cores,
    median of 3 runs each ("attention-kernel-portability-and-benchmarking",
    fourth and fifth paragraphs: medians, the inputs and the conditions)."""
    legs = {}
    for name in ("tiny_fp32", "varlen_causal", "gqa_prefill"):
        for threads in (1, None):
            r = cpu_baseline(name, budget_s=budget_s, threads=threads, repeats=3)
            legs[f"{name}@{r['cores']}c"] = {"tflops": r["value"], "s": r["seconds"],
                                             "sample": r["sample"]}
    return legs


def run_sweep(args):
    """Prefill forward over a range of sequence lengths with batch, heads,
    head width, dtype and mask family fixed ("attention-algorithm-error-and-
    complexity-tests", fifth paragraph): one JSON line per length with the
    parameters beside the time, then the fitted exponent of time against N
    (dense causal attention keeps quadratic pair work, so about 2 once the
    GPU is full)."""
    from exact_tiled_attention_online_gb300 import attn
    attn.library()
    device = torch.device("cuda", 0)
    lengths = [int(x) for x in args.sweep.split(",")]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    points = []
    win = args.sweep_window
    mask_name = f"causal_top_left_window_{win}" if win > 0 else "causal_top_left"
    for n in lengths:
        w = inputs.custom(f"sweep_{n}", (n,) * args.sweep_batch, (n,) * args.sweep_batch, 32, 8,
                          128, "bf16", inputs.MASK_TOP_LEFT, seed=2000 + n, window=win)
        x = inputs.make_inputs(w, device=device, gen_device=device)
        o = torch.empty_like(x["q"])
        lse = torch.empty((w.hq, w.total_q), dtype=torch.float32, device=device)

        def run():
            attn.fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_k"], w.max_q,
                     w.max_k, w.mask, w.scale, out=o, lse=lse, window=win)
        for _ in range(args.warmup):
            run()
        ms = []
        for _ in range(args.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            run()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        med = statistics.median(ms)
        fl = fwd_flops(w)
        points.append((n, med))
        print(json.dumps({"sweep": "prefill_fwd", "seq_len": n, "batch": w.batch, "heads_q": w.hq,
                          "heads_kv": w.hkv, "head_dim": w.d, "dtype": "bf16",
                          "mask": mask_name, "allowed_pairs": allowed_pairs(w),
                          "ms_median": med, "tflops": fl / (med * 1e-3) / 1e12,
                          "plan": attn.last_plan()}))
    if len(points) >= 2:
        lx = np.log([p[0] for p in points])
        ly = np.log([p[1] for p in points])
        slope = float(np.polyfit(lx[-3:], ly[-3:], 1)[0]) if len(points) >= 3 else \
            float((ly[-1] - ly[0]) / (lx[-1] - lx[0]))
        print(json.dumps({"sweep": "prefill_fwd", "fit": "time ~ N^a over the three longest",
                          "a": slope, "batch": args.sweep_batch, "heads_q": 32, "heads_kv": 8,
                          "head_dim": 128, "mask": mask_name}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workloads",
                    default="gqa_prefill,decode_q1,decode_q16,train_fwd_bwd,varlen_causal,"
                            "window_prefill,bias_prefill,bias_tensor_prefill,bias_tensor_train,"
                            "train_fwd_bwd_plain,train_fwd_bwd_det")
    ap.add_argument("--skip-validate", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--batch-div", type=int, default=1,
                    help="divide every workload's batch (smaller cases for profiler captures; "
                         "not a benchmark setting)")
    ap.add_argument("--sweep", default="",
                    help="comma-separated sequence lengths: prefill-forward length sweep "
                         "(one JSON line per length) instead of the benchmark")
    ap.add_argument("--sweep-batch", type=int, default=1)
    ap.add_argument("--sweep-window", type=int, default=0,
                    help="bounded causal window for the sweep (0: unbounded causal); a bounded "
                         "window has linear pair work, so the fitted exponent tends to 1")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.sweep:
        run_sweep(args)
        return

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    peaks, peak_kind = load_peaks()

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    device = torch.device("cuda", local)
    runners, per, wall, clocks, validated, mem_total = time_gpu(args, rank, world, device)

    head = per[HEADLINE] if HEADLINE in per else next(iter(per.values()))
    head_name = HEADLINE if HEADLINE in per else next(iter(per))
    head_ms = reduce_max(head["ms_median"], world, device)
    value = rate(head["work"] * world, head["unit"], head_ms)
    step_ms = reduce_max(wall * 1e3 / args.steps, world, device)

    workloads = {}
    for n, d in per.items():
        ms = reduce_max(d["ms_median"], world, device)
        v = rate(d["work"] * world, d["unit"], ms)
        if d["unit"] == "GB/s":
            peak = peaks["hbm_gbs"]
            roof = {"bound": "hbm", "achieved": rate(d["work"], "GB/s", ms), "peak": peak,
                    "unit": "GB/s"}
        elif "_simt" in " ".join(d["plan"]):
            # CUDA-core kernels: the fp32 FMA rate, 128 lanes x 2 flops per SM
            # and cycle at the maximum SM clock
            peak = alu_peak_tflops(peaks)
            roof = {"bound": "alu", "achieved": rate(d["work"], "TFLOP/s", ms), "peak": peak,
                    "unit": "TFLOP/s"}
        else:
            peak = peaks["bf16_tflops"]
            roof = {"bound": "tensor", "achieved": rate(d["work"], "TFLOP/s", ms), "peak": peak,
                    "unit": "TFLOP/s"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        workloads[n] = {"value": v, "unit": d["unit"], "ms_median": ms, "ms_p90": d["ms_p90"],
                        "ms_max": d["ms_max"], "roofline": roof, "plan": d["plan"],
                        "memory": d["memory"]}
        if "ms_median_l2_warm" in d:
            workloads[n]["ms_median_l2_warm"] = d["ms_median_l2_warm"]

    out = {"metric": METRIC, "value": value, "unit": head["unit"], "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded N(0,1); shapes of the five attention workloads)",
           "config": {"workload": head_name, "batch": runners[head_name].w.batch,
                      "seq_len_q": runners[head_name].w.max_q,
                      "seq_len_k": runners[head_name].w.max_k,
                      "heads_q": runners[head_name].w.hq, "heads_kv": runners[head_name].w.hkv,
                      "head_dim": runners[head_name].w.d, "mask": "causal_top_left",
                      "l2": "flushed before every timed workload (256 MiB write)",
                      "parallelism": f"replicas x{world}, no collective"},
           "gpu_launches": sum(d["kernels"] for d in per.values()) * args.steps,
           "clocks": clocks,
           "validated": {n: v["ok"] for n, v in validated.items()}}

    hw = workloads[head_name]
    roof = dict(hw["roofline"])
    roof["peak_source"] = f"{peak_kind} bf16_tflops (burst)" if roof["unit"] == "TFLOP/s" \
        else f"{peak_kind} hbm_gbs"
    roof["traffic"] = traffic_for(head_name)
    out["roofline"] = roof

    if not args.no_e2e:
        ms, h2d, d2h = e2e_headline(args, runners[head_name], device)
        ms = reduce_max(ms, world, device)
        out["e2e"] = {"value": rate(per[head_name]["work"] * world, head["unit"], ms),
                      "unit": head["unit"], "ms_per_step": ms, "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": d2h,
                      "schedule": "pipelined: copies in, kernel, copies out on three streams, "
                                  "two buffer sets"}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(head_name, repeats=3)
        out["cpu_baseline_legs"] = {k: round(v["tflops"], 6)
                                    for k, v in cpu_baseline_legs().items()}
    out["memory"] = {"max_allocated_mb": round(mem_total["max_memory_allocated"] / 2**20, 1),
                     "max_reserved_mb": round(mem_total["max_memory_reserved"] / 2**20, 1)}
    if HEADLINE in workloads and "ms_median_l2_warm" in workloads[HEADLINE]:
        out["l2_warm"] = {"workload": HEADLINE,
                          "ms_median": workloads[HEADLINE]["ms_median_l2_warm"],
                          "value": rate(per[HEADLINE]["work"] * world, per[HEADLINE]["unit"],
                                        workloads[HEADLINE]["ms_median_l2_warm"])}
    # every workload, compact, at the end of the line: value, unit, median ms,
    # roofline fraction, workspace MiB (the details go to stderr)
    out["workloads"] = {n: [round(wv["value"], 1), "GB/s" if wv["unit"] == "GB/s" else "TF",
                            round(wv["ms_median"], 4), round(wv["roofline"]["frac"], 3),
                            round(wv["memory"]["workspace_bytes"] / 2**20, 1)]
                        for n, wv in workloads.items()}
    out["workloads_fields"] = "value, unit, ms_median, roofline frac, workspace MiB"
    if rank == 0:
        detail = {"detail": True, "workloads": workloads, "validated": validated,
                  "memory_total": mem_total}
        print(json.dumps(detail), file=sys.stderr)
        print(json.dumps(out))
    if world > 1:
        torch.distributed.destroy_process_group()


def traffic_for(workload: str):
    """DRAM bytes per launch of the headline's dominant kernel from the
    committed ncu summary, when it was taken on the kernel source as it is
    now; otherwise null."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(workload)
    if not d:
        return None
    src = os.path.join(ROOT, "exact_tiled_attention_online_gb300", "csrc", d["source"])
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return d["dram_bytes_per_launch"] if sha == d.get("source_sha") else None


def run_reference(args, rank, world):
    """The oracle on the host cores, same metric and workload, each step a
    bounded sample; under torchrun only rank 0 works."""
    if rank != 0:
        return
    per_step = []
    info = None
    budget = max(2.0, min(12.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        info = cpu_baseline(HEADLINE, budget_s=budget)
        if i >= args.warmup:
            per_step.append(info)
    value = statistics.median(p["value"] for p in per_step)
    secs = statistics.median(p["seconds"] for p in per_step)
    out = {"metric": METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1))",
           "config": {"workload": HEADLINE, "sample": info["sample"]},
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": info["cores"],
                            "kind": "oracle", "sample": info["sample"]},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


if __name__ == "__main__":
    main()
