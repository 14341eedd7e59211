#!/usr/bin/env python
"""Benchmark of the paged-KV attention step on GB300.

One step = one pass of the whole hot path over one batch: q/k RMSNorm + RoPE +
slot scatter (pkv_qknorm_rope_store), then paged attention — varlen prefill
(pkv_attn_prefill) for the headline workload, single-token decode
(pkv_attn_decode) for the decode workloads reported alongside it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line on rank 0.  Headline: the varlen causal prefill workload
(8 prompts, lengths U[1,2048] from the seed, empty cache), metric prefill
attention TFLOP/s over the whole step.  Decode KV GB/s is reported for the
batched-decode workload (B=256, contexts U[512,4096]) and the long-context
workload (contexts 40960, B = 1, 8, 32) under "decode".

Timing: CUDA events on the launching stream around every step (medians over
the steps; the step total in a pass of its own, since an event between the
store and the attention would keep the attention kernel from starting its
set-up during the store's tail), with the L2 flushed between steps, outside the events: a 256 MiB
write (twice the L2), then a 256 MiB read, so that the write's own dirty lines
are written back before the timed step rather than inside it (the decode
figures with the write alone are reported beside the others as "dirty_l2").
Decode workloads whose K/V exceed the L2 (all but the tiny one) are timed as
launches back to back between one pair of events instead, as a stream of
decode steps runs them (inputs larger than the L2 need no flush); the
one-at-a-time figures are kept beside them as "isolated".
End to end ("e2e"): the same step from pinned host buffers, each step's H2D of
its inputs and D2H of its output inside the timed region; two buffer sets let
neighbouring steps' copies overlap the kernels (the serial figure is reported
beside it).
Multi-GPU (torchrun): every rank runs an independent batch (weak scaling, no
collective on the data path); times are max-reduced over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged GQA decode KV GB/s (% HBM peak); prefill attn TFLOP/s (% bf16 peak)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HEAD_DIM, NQ, NKV = 128, 32, 8


# ------------------------------------------------------------------ work accounting
def causal_flops(wl) -> int:
    """2 FLOP per multiply-add, QK^T and PV, over the visible (query, key) pairs only."""
    tot = 0
    for lq, lk in zip(wl.new_lens.tolist(), wl.seq_lens_k.tolist()):
        tot += lq * (lk - lq) + lq * (lq + 1) // 2
    return 4 * HEAD_DIM * NQ * tot


def decode_bytes(wl) -> int:
    """Algorithmic HBM bytes of one decode launch: every K/V byte of the contexts, q and out."""
    return int(wl.context_lens.astype(np.int64).sum()) * 2 * NKV * HEAD_DIM * 2 + wl.num_seqs * 2 * NQ * HEAD_DIM * 2


def store_bytes(wl) -> int:
    """Algorithmic HBM bytes of one store launch: q read + write, k and v read, K/V rows written,
    two int32 indices and the 512-byte cos/sin row per token."""
    stored = int((wl.slot_mapping >= 0).sum())
    T = wl.num_tokens
    return T * (2 * NQ * HEAD_DIM * 2 + 8 + 512) + stored * 4 * NKV * HEAD_DIM * 2


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def profiled_traffic(kernel: str, source: str):
    """DRAM bytes per launch measured by ncu, if taken on the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        table = json.load(f)
    e = table.get(kernel)
    if not e:
        return None
    with open(os.path.join(ROOT, "paged_kv_cache_rmsnorm_gb300", "csrc", source), "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()[:16]
    if e.get("source_sha256_16") != h:
        return None
    return e.get("bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(prefix="pkv_clocks_", suffix=".csv")
        self.proc = None
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(gpu_index)], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"samples": 0, "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        busy = [s for s in sm if mx and s >= 0.5 * max(mx)]
        return {"sm_mhz": statistics.median(busy or sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ device inputs
def dev_u16(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def dev_i32(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


class DeviceStep:
    """A workload resident in HBM, run through the C ABI."""

    def __init__(self, wl, torch, fast_cache: bool = False, seed: int = 0):
        import paged_kv_cache_rmsnorm_gb300 as pkv

        self.pkv, self.torch, self.wl = pkv, torch, wl
        self.q = dev_u16(wl.q, torch)
        self.k = dev_u16(wl.k, torch)
        self.v = dev_u16(wl.v, torch)
        self.pos = dev_i32(wl.positions, torch)
        self.slots = dev_i32(wl.slot_mapping, torch)
        self.wq = dev_u16(wl.q_norm_w, torch)
        self.wk = dev_u16(wl.k_norm_w, torch)
        shape = (wl.num_blocks, 256, NKV, HEAD_DIM)
        if fast_cache:
            # timing only: N(0,1) history drawn on the device instead of per block on the host
            g = torch.Generator(device="cuda")
            g.manual_seed(seed)
            self.kc = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
            self.vc = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
        else:
            kc, vc = wl.materialize_cache()
            self.kc, self.vc = dev_u16(kc, torch), dev_u16(vc, torch)
        self.bt = dev_i32(wl.block_table, torch)
        self.ctx = dev_i32(wl.context_lens, torch)
        self.cu_q = dev_i32(wl.cu_seqlens_q, torch)
        self.cu_k = dev_i32(wl.cu_seqlens_k, torch)
        self.out = torch.empty_like(self.q)
        self.ws = pkv.decode_workspace(wl.num_seqs, wl.max_seqlen_k) if wl.mode == "decode" else None
        # the call's scalar arguments, computed once (each workload property is a NumPy reduction)
        self._decode = wl.mode == "decode"
        self._max_q, self._max_k, self._scale = int(wl.max_seqlen_q), int(wl.max_seqlen_k), float(wl.scale)

    def store(self):
        self.pkv.qknorm_rope_store(self.q, self.k, self.v, self.pos, self.slots, self.wq, self.wk, self.kc, self.vc)

    def attend(self):
        if self._decode:
            self.pkv.attn_decode(self.q, self.kc, self.vc, self.ctx, self.bt, self._max_k, self._scale,
                                 out=self.out, workspace=self.ws)
        else:
            self.pkv.attn_prefill(self.q, self.kc, self.vc, self.cu_q, self.cu_k, self.bt, self._max_q,
                                  self._max_k, self._scale, out=self.out)


class L2Flush:
    """Evicts the L2 (129 MB) between timed steps.  ``__call__`` writes a 256 MiB buffer (twice
    the L2) and then reads another 256 MiB: after the write alone the L2 is full of dirty lines,
    and the next kernel would pay their write-back to HBM (up to 129 MB, about 19 us at the copy
    rate) as if it were its own traffic; after the read the L2 holds clean lines, which cost nothing
    to evict.  ``dirty`` does the write alone."""

    def __init__(self, torch):
        self.torch = torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")

    def dirty(self, i: int) -> None:
        self.w.fill_(i & 0x7F)

    def __call__(self, i: int) -> None:
        self.w.fill_(i & 0x7F)
        self.torch.sum(self.r, dim=0, out=self.sink)


def time_device(step: DeviceStep, K: int, W: int, flush, torch, dist=None):
    """Median ms of [store, attention, whole step] over K steps; ``flush(i)`` runs before step i.

    The whole step is timed in a pass of its own, with events only around it: an event recorded between
    the store and the attention (as the breakdown pass does) separates the two kernels in the stream, so
    the attention kernel could not start its set-up during the store's tail as it does in a step."""
    for _ in range(W):
        step.store()
        step.attend()
    stream = torch.cuda.current_stream()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    _barrier(dist)
    torch.cuda.synchronize()
    for i in range(K):
        flush(i)
        ev[i][0].record(stream)
        step.store()
        ev[i][1].record(stream)
        step.attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    st = [e[0].elapsed_time(e[1]) for e in ev]
    at = [e[1].elapsed_time(e[2]) for e in ev]
    for i in range(K):
        flush(i)
        ev[i][0].record(stream)
        step.store()
        step.attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    _barrier(dist)
    tot = [e[0].elapsed_time(e[2]) for e in ev]
    return _max_ranks([statistics.median(st), statistics.median(at), statistics.median(tot)], dist, torch)


L2_BYTES = 129e6  # GB300 L2


def time_back_to_back(step: DeviceStep, K: int, W: int, torch, dist=None):
    """ms per launch of [attention alone, store + attention] over K launches back to back between one pair of
    CUDA events: the launch overhead is amortised as in a stream of decode steps.  Only for inputs larger than the
    L2, so that no launch finds the previous one's data in it (a cyclic pass over more than the L2 misses)."""
    stream = torch.cuda.current_stream()
    for _ in range(W):
        step.attend()
    res = []
    for fn in (step.attend, lambda: (step.store(), step.attend())):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(dist)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(K):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        _barrier(dist)
        res.append(e0.elapsed_time(e1) / K)
    return _max_ranks(res, dist, torch)


def time_e2e(step: DeviceStep, K: int, W: int, torch, dist=None):
    """Whole steps through the public API from pinned host buffers: every step copies its own inputs
    host -> device, runs store + attention and copies its output device -> host, all inside the
    timed region.  Two sets of input/output buffers let step i+1's H2D (one copy stream) and step
    i-1's D2H (another) run while step i's kernels run on the compute stream; events keep a buffer
    set from being refilled before the kernels that read it, or drained, are done.  Returns
    (pipelined ms per step, serial ms per step, H2D bytes, D2H bytes)."""
    import copy

    wl = step.wl
    host = {
        "q": torch.from_numpy(wl.q.view(np.int16)).view(torch.bfloat16).pin_memory(),
        "k": torch.from_numpy(wl.k.view(np.int16)).view(torch.bfloat16).pin_memory(),
        "v": torch.from_numpy(wl.v.view(np.int16)).view(torch.bfloat16).pin_memory(),
        "pos": torch.from_numpy(wl.positions).pin_memory(),
        "slots": torch.from_numpy(wl.slot_mapping).pin_memory(),
        "bt": torch.from_numpy(wl.block_table).pin_memory(),
        "ctx": torch.from_numpy(wl.context_lens).pin_memory(),
        "cu_q": torch.from_numpy(wl.cu_seqlens_q).pin_memory(),
        "cu_k": torch.from_numpy(wl.cu_seqlens_k).pin_memory(),
    }
    # buffer set 0 is the step's own device tensors; set 1 has its own inputs and output (same cache)
    sets = [step, copy.copy(step)]
    for name in ("q", "k", "v", "pos", "slots", "bt", "ctx", "cu_q", "cu_k", "out"):
        setattr(sets[1], name, torch.empty_like(getattr(step, name)))
    out_host = [torch.empty(step.out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_host[0].numel() * out_host[0].element_size()

    def upload(b):
        for name, t in host.items():
            getattr(sets[b], name).copy_(t, non_blocking=True)

    def serial(b):
        upload(b)
        sets[b].store()
        sets[b].attend()
        out_host[b].copy_(sets[b].out, non_blocking=True)

    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "cmp", "out")}
    for k in ev:
        for e in ev[k]:
            e.record(main)

    def pipelined(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev["cmp"][b])  # step i-2's kernels are done with set b (q is rewritten in place)
            upload(b)
            ev["in"][b].record(s_in)
        main.wait_event(ev["in"][b])
        main.wait_event(ev["out"][b])  # step i-2's output has left set b
        sets[b].store()
        sets[b].attend()
        ev["cmp"][b].record(main)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev["cmp"][b])
            out_host[b].copy_(sets[b].out, non_blocking=True)
            ev["out"][b].record(s_out)

    def timed(fn):
        for i in range(W):
            fn(i)
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _barrier(dist)
        torch.cuda.synchronize()
        a.record(main)
        for i in range(K):
            fn(i)
        for e in ev["out"]:
            main.wait_event(e)
        z.record(main)
        torch.cuda.synchronize()
        _barrier(dist)
        return a.elapsed_time(z) / K

    ms_serial = timed(lambda i: serial(0))
    ms_pipe = timed(pipelined)
    ms_pipe, ms_serial = _max_ranks([ms_pipe, ms_serial], dist, torch)
    return ms_pipe, ms_serial, h2d, d2h


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def build_library(pkv, dist=None, local_rank: int = 0) -> None:
    """Compile libpkv.so if stale.  Under torchrun the ranks of a node share one source tree, so
    only local rank 0 compiles; the others wait at a barrier and then find the library fresh."""
    if dist is None:
        pkv.build()
        return
    if local_rank == 0:
        try:
            pkv.build()
        finally:
            dist.barrier()
    else:
        dist.barrier()
        if not pkv.library_is_fresh():
            raise RuntimeError("local rank 0 did not leave a fresh libpkv.so (its build failed)")
        pkv.build()


def _max_ranks(vals, dist, torch, device="cuda"):
    """Element-wise max over ranks (timing only; the data path has no collective)."""
    if dist is None:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def rank_seed(base: int, rank: int) -> int:
    """Each rank runs an independent batch of the same workload: weak scaling."""
    return base + 1000 * rank


def whole_job_value(units_per_rank: float, world: int, seconds: float) -> float:
    """Units processed by all ranks divided by the max-over-ranks time."""
    return units_per_rank * world / seconds


# ------------------------------------------------------------------ CPU oracle baseline
def oracle_sample(wl, budget_pairs: float):
    """The first sequences of the workload whose visible (query, key) pairs fit the budget (at least one)."""
    pairs = [lq * (lk - lq) + lq * (lq + 1) // 2 for lq, lk in zip(wl.new_lens.tolist(), wl.seq_lens_k.tolist())]
    n, acc = 0, 0
    for p in pairs:
        if n and acc + p > budget_pairs:
            break
        acc += p
        n += 1
    return wl.subset(np.arange(n)), n


def time_oracle(wl, steps: int, warmup: int, seconds_per_step: float):
    import oracle

    # calibrate the sample so one step costs about `seconds_per_step`
    probe, _ = oracle_sample(wl, 2e6)
    kc, vc = probe.materialize_cache()
    t0 = time.perf_counter()
    oracle.run_step(probe, kc, vc)
    rate = causal_flops(probe) / max(time.perf_counter() - t0, 1e-3)
    budget = seconds_per_step * rate / (4 * HEAD_DIM * NQ)
    sample, nseq = oracle_sample(wl, budget)
    kc, vc = sample.materialize_cache()
    for _ in range(warmup):
        oracle.run_step(sample, kc, vc)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.run_step(sample, kc, vc)
    dt = (time.perf_counter() - t0) / steps
    return causal_flops(sample) / dt / 1e12, dt, nseq, sample


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ------------------------------------------------------------------ main
def chosen_decode(args) -> set:
    return {w for w in args.decode_workloads.split(",") if w and w != "none"}


def bench_add_rmsnorm(torch, pkv, flush, K, W, peaks, T):
    """pkv_add_rmsnorm on a [T, 4096] bf16 batch (T = the headline batch's token count)."""
    g = torch.Generator(device="cuda").manual_seed(4096)
    x = torch.randn(T, pkv.HIDDEN, device="cuda", generator=g).to(torch.bfloat16)
    r = torch.randn(T, pkv.HIDDEN, device="cuda", generator=g).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(pkv.HIDDEN, device="cuda", generator=g)).to(torch.bfloat16)
    out = torch.empty_like(x)
    ts = []
    for i in range(W + K):
        r.copy_(x)  # the residual starts from the same values every step
        flush(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkv.add_rmsnorm(x, r, w, out)
        e1.record()
        torch.cuda.synchronize()
        if i >= W:
            ts.append(e0.elapsed_time(e1))
    ms = sorted(ts)[len(ts) // 2]
    nbytes = 4 * 2 * pkv.HIDDEN * T  # read x and r, write out and the new residual (4 rows of 8 KiB per token)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"residual add + RMSNorm, [{T}, {pkv.HIDDEN}] bf16", "tokens": T, "kernel_us": ms * 1e3,
            "bytes_per_launch": nbytes, "gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
            "traffic": profiled_traffic("add_rmsnorm_10780", "add_rmsnorm.cu"),
            "timing": "median of per-launch CUDA events, L2 flushed (write, then read) before each launch"}


def bench_decode_graph(torch, pkv, cfg, K, W, rank):
    """Store + decode per step, eager launches against one CUDA-graph replay (steps back to back)."""
    from paged_kv_cache_rmsnorm_gb300.graphs import DecodeGraph
    from workloads import config_workload

    wl = config_workload(cfg, seed=rank_seed(20260 + cfg, rank))
    ds = DeviceStep(wl, torch, fast_cache=True, seed=cfg + 1000 * rank)
    g = DecodeGraph(ds.q, ds.k, ds.v, ds.pos, ds.slots, ds.wq, ds.wk, ds.kc, ds.vc, ds.ctx, ds.bt, wl.max_seqlen_k,
                    wl.scale).capture()

    def per_step_us(fn):
        for _ in range(W):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / K

    eager_us = per_step_us(g.eager)
    graph_us = per_step_us(g.replay)
    return {"workload": wl.name, "batch": wl.num_seqs, "eager_step_us": eager_us, "graph_step_us": graph_us,
            "speedup": eager_us / graph_us, "launches_per_step": 2,
            "timing": f"{K} steps back to back after {W}, CUDA events around the run (no L2 flush)"}


def bench_qkv(torch, pkv, K, W, peaks, T):
    """pkv_qkv_rope_store on the headline batch's T tokens: [T, 4096] x [6144, 4096]^T plus norm/RoPE/store."""
    g = torch.Generator(device="cuda").manual_seed(6144)
    x = torch.randn(T, pkv.HIDDEN, device="cuda", generator=g).to(torch.bfloat16)
    w = (torch.randn(pkv.QKV_OUT, pkv.HIDDEN, device="cuda", generator=g) / 64).to(torch.bfloat16)
    wq = (1 + 0.1 * torch.randn(128, device="cuda", generator=g)).to(torch.bfloat16)
    wk = (1 + 0.1 * torch.randn(128, device="cuda", generator=g)).to(torch.bfloat16)
    pos = torch.randint(0, 40960, (T,), device="cuda", generator=g, dtype=torch.int32)
    nb = (T + 255) // 256 + 16
    slots = torch.randperm(nb * 256, device="cuda", generator=g)[:T].to(torch.int32)
    kc = torch.zeros(nb, 256, 8, 128, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    q = torch.empty(T, 32, 128, dtype=torch.bfloat16, device="cuda")
    ts = []
    for i in range(W + K):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        pkv.qkv_rope_store(x, w, pos, slots, wq, wk, kc, vc, q_out=q)
        e1.record()
        torch.cuda.synchronize()
        if i >= W:
            ts.append(e0.elapsed_time(e1))
    ms = sorted(ts)[len(ts) // 2]
    flops = 2.0 * T * pkv.HIDDEN * pkv.QKV_OUT
    tf = flops / (ms * 1e-3) / 1e12
    return {"workload": f"QKV projection + norm/RoPE/store, [{T}, 4096] x [6144, 4096]^T bf16", "tokens": T,
            "kernel_us": ms * 1e3, "tflops": tf, "frac_of_bf16_peak": tf / peaks["bf16_tflops"],
            "flops_per_launch": flops, "traffic": profiled_traffic("qkv_10780", "qkv.cu"), "timing": "median of per-launch CUDA events (weights stay in L2: 50 MB)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--decode-workloads", default="tiny,batched,long1,long8,long32",
                    help="comma list of tiny,batched,long1,long8,long32, or none")
    ap.add_argument("--prefill-workloads", default="chunked",
                    help="prefill workloads besides the headline one: chunked, or none")
    ap.add_argument("--next", default="add_rmsnorm,decode_graph,qkv",
                    help="comma list of work next to the step to time (add_rmsnorm, decode_graph, qkv), or none")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    from workloads import config_workload

    wl = config_workload(2, seed=rank_seed(20262, rank))
    config = {"workload": "varlen causal prefill: 8 prompts, lengths U[1,2048] (seeded), empty cache, "
                          "32/8 heads, d=128, 256-token blocks, permuted block ids",
              "tokens": wl.num_tokens, "prompt_lengths": wl.new_lens.tolist(), "causal_flops": causal_flops(wl),
              "l2": ("flushed between timed steps: a 256 MiB write, then a 256 MiB read (clean L2); decode "
                     "workloads whose K/V exceed the L2 use inputs larger than the L2 instead (launches back to back)"),
              "parallelism": f"replicas x{world}"}

    if args.impl == "reference":
        # the reference arm: the CPU oracle as it stands, rank 0 only
        if rank != 0:
            return 0
        steps, warm = max(1, args.steps), args.warmup
        per_step = max(0.5, 150.0 / (steps + warm))
        tflops, dt, nseq, sample = time_oracle(wl, steps, warm, per_step)
        desc = f"first {nseq} of 8 prompts ({sample.num_tokens} tokens, {causal_flops(sample):.3g} causal FLOP)"
        line = {"impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": 0,
                "steps": steps, "warmup": warm, "ms_per_step": dt * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                                 "sample": desc},
                "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import torch

    dist = None
    if world > 1:
        import torch.distributed as td

        torch.cuda.set_device(local_rank)
        td.init_process_group("nccl")
        dist = td
    else:
        torch.cuda.set_device(0)
    import paged_kv_cache_rmsnorm_gb300 as pkv

    build_library(pkv, dist, local_rank)
    pkv.init()
    peaks, peak_src = load_peaks()
    flush = L2Flush(torch)
    clocks = ClockSampler(local_rank)

    # ---------------- headline: varlen prefill step
    step = DeviceStep(wl, torch)
    K, W = args.steps, args.warmup
    st_ms, at_ms, tot_ms = time_device(step, K, W, flush, torch, dist)
    assert pkv.check_errors() == [], "kernel error flags during the prefill bench"
    flops = causal_flops(wl)
    value = whole_job_value(flops, world, tot_ms * 1e-3) / 1e12
    e2e = None
    if not args.no_e2e:
        e2e_ms, serial_ms, h2d, d2h = time_e2e(step, max(10, K // 4), W, torch, dist)
        e2e = {"value": flops * world / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "pipeline": "two buffer sets: H2D, kernels and D2H of neighbouring steps overlap on three streams",
               "serial_ms_per_step": serial_ms,
               "serial_value": flops * world / (serial_ms * 1e-3) / 1e12}
    prefill_tflops = flops / (at_ms * 1e-3) / 1e12
    peak_tc = peaks["bf16_tflops"]
    launches = 2 * K

    # ---------------- the other prefill workload: a 512-token chunk after a cached, partly shared prefix
    prefill = {"varlen B=8": {"workload": config["workload"], "tokens": wl.num_tokens, "causal_flops": flops,
                              "store_us": st_ms * 1e3, "prefill_us": at_ms * 1e3, "step_us": tot_ms * 1e3,
                              "tflops": prefill_tflops, "frac_of_bf16_peak": prefill_tflops / peak_tc}}
    if "chunked" in {w for w in args.prefill_workloads.split(",") if w}:
        cwl = config_workload(4, seed=rank_seed(20264, rank))
        cs = DeviceStep(cwl, torch, fast_cache=True, seed=4 + 1000 * rank)
        cs_ms, ca_ms, ct_ms = time_device(cs, K, W, flush, torch, dist)
        assert pkv.check_errors() == [], "kernel error flags during the chunked prefill bench"
        cflops = causal_flops(cwl)
        ctf = cflops / (ca_ms * 1e-3) / 1e12
        prefill["chunked S=16"] = {
            "workload": cwl.name, "tokens": cwl.num_tokens, "prefix_lengths": cwl.hist_lens.tolist(),
            "causal_flops": cflops, "store_us": cs_ms * 1e3, "prefill_us": ca_ms * 1e3, "step_us": ct_ms * 1e3,
            "tflops": ctf, "frac_of_bf16_peak": ctf / peak_tc,
            "step_tflops": whole_job_value(cflops, world, ct_ms * 1e-3) / 1e12}
        del cs
        torch.cuda.empty_cache()

    # ---------------- decode workloads
    decode = {}
    if "tiny" in chosen_decode(args):
        g = bench_decode_graph(torch, pkv, 1, max(20, min(K, 100)), W, rank)
        decode["tiny B=4"] = {"workload": g["workload"], "batch": g["batch"], "eager_step_us": g["eager_step_us"],
                              "graph_step_us": g["graph_step_us"], "launches_per_step": g["launches_per_step"],
                              "timing": g["timing"]}
        assert pkv.check_errors() == [], "kernel error flags during the tiny decode bench"
    chosen = chosen_decode(args)
    for key, name, idx, batch in (("batched", "batched B=256", 3, None), ("long1", "long B=1", 5, 1),
                                  ("long8", "long B=8", 5, 8), ("long32", "long B=32", 5, 32)):
        if key in chosen:
            dwl = config_workload(idx, seed=rank_seed(20260 + idx, rank), batch=batch)
            ds = DeviceStep(dwl, torch, fast_cache=True, seed=idx + 1000 * rank)
            Kd = max(10, min(K, 50))
            s_ms, a_ms, t_ms = time_device(ds, Kd, W, flush, torch, dist)
            _, a_dirty_ms, _ = time_device(ds, Kd, W, flush.dirty, torch, dist)
            assert pkv.check_errors() == [], f"kernel error flags during decode bench {name}"
            kv = decode_bytes(dwl)
            isolated = {"decode_kernel_us": a_ms * 1e3, "store_kernel_us": s_ms * 1e3, "step_us": t_ms * 1e3,
                        "frac_of_hbm": kv / (a_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                        # the decode's share of one isolated step: the step timed whole (its decode starts its
                        # set-up during the store's tail) minus the store timed alone
                        "decode_in_step_us": (t_ms - s_ms) * 1e3,
                        "frac_of_hbm_in_step": (kv / ((t_ms - s_ms) * 1e-3) / 1e9 / peaks["hbm_gbs"]
                                                if t_ms > s_ms else None),
                        "timing": "one step at a time after an L2 flush, CUDA events around the store and "
                                  "around the decode launch (each launch's overhead inside its interval); "
                                  "decode_in_step_us: the whole step, timed without an event between store and "
                                  "decode, minus the store"}
            if kv > L2_BYTES:
                # the K/V read per launch is larger than the L2: launches back to back, one pair of events
                a_ms, t_ms = time_back_to_back(ds, Kd, W, torch, dist)
                timing = (f"{Kd} launches back to back between one pair of CUDA events (K/V of {kv / 1e6:.0f} MB "
                          f"per launch, larger than the {L2_BYTES / 1e6:.0f} MB L2, so no flush)")
            else:
                timing = isolated["timing"]
            gbs = kv / (a_ms * 1e-3) / 1e9
            decode[name] = {
                "workload": dwl.name, "batch": dwl.num_seqs, "kv_bytes": kv,
                "decode_kernel_us": a_ms * 1e3, "store_kernel_us": s_ms * 1e3, "step_us": t_ms * 1e3,
                "kv_gbs": gbs, "frac_of_hbm": gbs / peaks["hbm_gbs"],
                "tokens_per_s_per_layer": dwl.num_seqs * world / (t_ms * 1e-3),
                "timing": timing,
                "isolated": isolated,
                "dirty_l2": {"decode_kernel_us": a_dirty_ms * 1e3,
                             "frac_of_hbm": kv / (a_dirty_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                             "note": "L2 left full of the flush's dirty lines: their write-back lands in the kernel"},
            }
            if key == "batched":
                decode[name]["traffic"] = profiled_traffic("decode_batched256", "decode.cu")
            del ds
            torch.cuda.empty_cache()

    # ---------------- next to the step: residual add + RMSNorm over the hidden size
    nxt = {}
    if "add_rmsnorm" in {w for w in args.next.split(",") if w}:
        nxt["add_rmsnorm"] = bench_add_rmsnorm(torch, pkv, flush, max(10, min(K, 50)), W, peaks, wl.num_tokens)
        assert pkv.check_errors() == [], "kernel error flags during the add_rmsnorm bench"
    if "qkv" in {w for w in args.next.split(",") if w}:
        nxt["qkv_rope_store"] = bench_qkv(torch, pkv, max(10, min(K, 50)), W, peaks, wl.num_tokens)
        assert pkv.check_errors() == [], "kernel error flags during the qkv bench"
        torch.cuda.empty_cache()
    for key, cfg in (("decode_graph_batched", 3),):
        if "decode_graph" in {w for w in args.next.split(",") if w}:
            nxt[key] = bench_decode_graph(torch, pkv, cfg, max(20, min(K, 100)), W, rank)
            assert pkv.check_errors() == [], f"kernel error flags during the {key} bench"
            torch.cuda.empty_cache()

    clk = clocks.stop()

    # ---------------- CPU oracle baseline (rank 0, N=1)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tflops_cpu, dt, nseq, sample = time_oracle(wl, 1, 0, 15.0)
        cpu = {"value": tflops_cpu, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"first {nseq} of 8 prompts ({sample.num_tokens} tokens, "
                         f"{causal_flops(sample):.3g} causal FLOP), norm+RoPE+store+attention, fp64 NumPy",
               "seconds": dt}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": tot_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": config,
            "breakdown_us": {"store": st_ms * 1e3, "prefill": at_ms * 1e3},
            "roofline": {"bound": "tensor", "kernel": "prefill attention", "achieved": prefill_tflops,
                         "peak": peak_tc, "unit": "TFLOP/s", "frac": prefill_tflops / peak_tc,
                         "peak_source": f"{peak_src} bf16_tflops (burst)",
                         "traffic": profiled_traffic("prefill", "prefill_tc.cu"),
                         "algorithmic_flops_per_launch": flops},
            "store_roofline": {"bound": "hbm", "achieved": store_bytes(wl) / (st_ms * 1e-3) / 1e9,
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": store_bytes(wl) / (st_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                               "bytes_per_launch": store_bytes(wl),
                               "traffic": profiled_traffic("store_varlen8", "store.cu")},
            "prefill": prefill,
            "decode": decode,
            "next": nxt,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
