#!/usr/bin/env python
"""KDA prefill tokens/s and decode state GB/s on one GB300, with roofline
fractions, the fp64 CPU oracle timed beside it, and an end-to-end figure.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one ``kda_prefill_varlen`` call on the long-context prefill
workload (B=1, T=2^20, H=16, dk=dv=128, bf16, snapshots every 32768 tokens):
the device-side plan kernel, the chunked prefill kernel, which writes the
outputs, the 32 snapshots and the final state, and the exact-recomputation
launch (which does nothing unless a gate left the chunked algorithm's range).
The same run also times the single-sequence prefill (B=1, T=8192, H=32,
snapshots every 1024), the varlen batch with copy-on-write resume (16
sequences, snapshots every 256) and three 32768-token sequences at H=32 (96
(sequence, head) pairs, between the cooperative mode and a full GPU of
per-state CTAs) and reports them under "prefill", each with its own roofline, and the batched decode (256 sequences x 1 token), the
speculative-verify decode (64 x 8 tokens with per-token states) and the
speculative verify with the previous step's commit folded in (64 x 8 tokens,
kda_decode_spec) under "decode".
Inputs are synthetic (seeded, see hybrid_linear_attention_delta_gb300/inputs.py).
L2 is flushed (a 256 MiB write) between timed steps.  ``--impl reference``
times the fp64 CPU oracle on a bounded sample of the same workload instead.
Under torchrun (N > 1) every rank runs an independent replica (the path has
no exchange step) and the value is the sum of tokens over ranks divided by
the slowest rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s & decode state GB/s on 1 GB300, % of tensor/HBM roofline"
HEADLINE = "prefill_1m"
EXTRA_PREFILL = ("prefill_8k", "varlen_resume", "prefill_3x32k")
FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["source"] = "fallback"
    return d


def prefill_algorithmic(w, lens, n_snaps, n_resumed, es):
    """Algorithmic bytes and flops of one prefill call.

    bytes per token-head: q, k, g (dk each), v (dv), beta (1) in, out (dv):
    (3 dk + 2 dv + 1) * element size = 1282 B for bf16 at dk = dv = 128; plus
    one dk x dv fp32 state per (sequence, head) for the final state, for each
    snapshot and for each resumed initial state.
    flops per token-head at chunk C = 64 (tensor-core products only):
    5 * 2 C d (K+K-^T, Q+K-^T, T K+, T V, M U) + 3 * 2 d^2 (W S, Q+ S, K^T U)."""
    T = sum(lens)
    H, dk, dv = w.H, w.dk, w.dv
    per_tok = (3 * dk + 2 * dv + 1) * es
    state = dk * dv * 4
    B = len(lens)
    nbytes = T * H * per_tok + H * state * (B + n_snaps + n_resumed)
    C = 64
    flops = T * H * (5 * 2 * C * dk + 3 * 2 * dk * dv)
    return nbytes, flops, T * H * per_tok


# the kernel each decode workload runs (kda_decode.cu)
DECODE_KERNEL = {
    "decode_256x1": "decode128_single_kernel (one token per state)",
    "decode_fused_256x1": "decode_fused_kernel (convolution + recurrence + gated RMSNorm)",
    "verify_64x8": "decode128_kernel (staged tokens, per-token states, one CTA per state)",
    "spec_verify_64x8": "decode128_kernel (speculative: replay + commit + verify, one CTA per state)",
}


def spec_algorithmic(w, N, accepted, es):
    """Bytes of one speculative verify with commit: each touched state read
    once, written once when its sequence accepted at least one token, the
    replayed tokens' k, v, g, beta and the verified tokens' q, k, v, g, beta
    and outputs."""
    H, dk, dv = w.H, w.dk, w.dv
    state = dk * dv * 4
    n_write = int((accepted > 0).sum())
    replayed = int(accepted.sum())
    b = N * H * state + n_write * H * state
    b += replayed * H * (2 * dk + dv + 1) * es
    b += N * w.n_tok * H * (3 * dk + 2 * dv + 1) * es
    return b


def fused_decode_algorithmic(w, N, n_tok, es, conv_width=4):
    """Bytes of one fused decode call: each state read and written once, each
    convolution state ((2 dk + dv) x (W-1) raw inputs) read and written once,
    and per token-head the raw q, k, v, g, beta, gate in and the output out:
    (2 dk + dv) + dk + 1 + dv + dv elements (769 at dk = dv = 128)."""
    H, dk, dv = w.H, w.dk, w.dv
    state = dk * dv * 4
    conv = (2 * dk + dv) * (conv_width - 1) * es
    return N * H * (2 * state + 2 * conv + n_tok * ((2 * dk + dv) + dk + 1 + 2 * dv) * es)


def decode_algorithmic(w, N, n_tok, per_tok, es):
    """Bytes of one decode call: each touched state read once and written once
    (64 KiB each at 128 x 128 fp32), per-token states written when asked, and
    the token I/O (3 dk + 2 dv + 1 elements per token-head)."""
    H, dk, dv = w.H, w.dk, w.dv
    state = dk * dv * 4
    b = N * H * (2 * state + n_tok * (3 * dk + 2 * dv + 1) * es)
    if per_tok:
        b += N * H * n_tok * state
    return b


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                if self.uuid and parts[0] != self.uuid:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[4:8]):
                    if val.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def source_hash(names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "hybrid_linear_attention_delta_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, src_files):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_hash") != source_hash(src_files):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ GPU arms

def time_calls(fn, steps, warmup, flush, torch):
    """Per-step CUDA-event times of fn(events) (ms): whole call and main kernel."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn(None)
    torch.cuda.synchronize()
    call_ms, kern_ms = [], []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)   # torch creates the CUDA events lazily; the library re-records them
        k1.record(stream)
        e0.record(stream)
        fn((k0, k1))
        e1.record(stream)
        e1.synchronize()
        call_ms.append(e0.elapsed_time(e1))
        kern_ms.append(k0.elapsed_time(k1))
    return call_ms, kern_ms


def reduce_over_ranks(torch, values, device):
    """Max of each value over all ranks (the slowest rank's time); identity on
    one process.  ``device`` is where the backend's tensors live ("cuda" for
    NCCL, "cpu" for gloo)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_throughput(tokens_per_rank, world, seconds):
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (weak scaling, each rank an independent replica)."""
    return tokens_per_rank * world / seconds


def bench_prefill(args, torch, kda, inputs, world, rank, workload, retain=0, e2e=True,
                  fused=False):
    w = inputs.WORKLOADS[workload]
    if args.tokens and workload == args.workload:
        # a shortened single-sequence workload (profiling captures only)
        b = inputs.make_batch(w, device="cuda", lengths=[args.tokens])
    elif args.seqs and workload == args.workload:
        # the first sequences of a varlen workload (profiling captures only)
        b = inputs.make_batch(w, device="cuda", lengths=inputs.seq_lengths(w)[:args.seqs])
    else:
        b = inputs.make_batch(w, device="cuda")
    dev = {n: getattr(b, n) for n in ("q", "k", "v", "g", "beta")}
    cu = b.cu_seqlens.cuda()
    slots = b.init_slots.cuda()
    pool = b.pool
    T, H = dev["q"].shape[:2]
    out = torch.empty((T, H, w.dv), dtype=dev["q"].dtype, device="cuda")
    n_snaps = kda.kda_snapshot_count(b.cu_seqlens, w.snap_interval)
    ws = kda.workspace_for(len(b.cu_seqlens) - 1, H, pool.shape[0])
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    launches = []
    if retain:
        # a retention map: every retain-th interval snapshot of each
        # sequence kept, straight into a free pool slot; the rest dropped
        smap_h = retention_map(b, w.snap_interval, retain, pool.shape[0])
        smap = smap_h.cuda()
        snaps = None
        n_written = int((smap_h >= 0).sum())

        def prefill(events=None):
            kda.kda_prefill_varlen_retain(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], cu,
                                          slots, pool, out, w.snap_interval, smap, workspace=ws,
                                          events=events)
    elif fused:
        # the layer around the recurrence: dev q, k, v serve as the raw inputs
        snaps = torch.empty((n_snaps, H, w.dk, w.dv), dtype=torch.float32, device="cuda")
        n_written = n_snaps
        ft = inputs.fused_tensors(T, H, w.dk, w.dv, dev["q"].dtype, w.index, pool.shape[0],
                                  device="cuda")
        scratch = torch.empty(kda.kda_fused_scratch_bytes(T, H, w.dk, w.dv, kda.KDA_BF16),
                              dtype=torch.uint8, device="cuda")

        def prefill(events=None):
            kda.kda_prefill_varlen_fused(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                                         ft["gate"], ft["conv_w"], ft["norm_w"], cu, slots, pool,
                                         ft["conv_pool"], out, w.snap_interval, snaps,
                                         workspace=ws, scratch=scratch, events=events)
    else:
        snaps = torch.empty((n_snaps, H, w.dk, w.dv), dtype=torch.float32, device="cuda")
        n_written = n_snaps

        def prefill(events=None):
            kda.kda_prefill_varlen(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], cu, slots,
                                   pool, out, w.snap_interval, snaps, workspace=ws, events=events)

    def call(events):
        prefill(events)
        launches.append(kda.kda_last_launch_count())

    call(None)
    st, bits = kda.kda_device_status(ws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"prefill device check failed: {st} bits={bits}")
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(_uuid(torch))
    clocks.start()
    launches.clear()
    call_ms, kern_ms = time_calls(call, args.steps, args.warmup, flush, torch)
    timed_launches = sum(launches[-args.steps:])
    ck = clocks.stop()

    # end to end through the same public call, host (pinned) buffers in and out
    host = {}
    for n, t in (dev.items() if e2e else ()):
        host[n] = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        host[n].copy_(t)
    host_cu, host_slots = b.cu_seqlens.pin_memory(), b.init_slots.pin_memory()
    host_out = torch.empty(out.shape if e2e else (0,), dtype=out.dtype, pin_memory=True)
    stream = torch.cuda.current_stream()
    h2d = sum(t.numel() * t.element_size() for t in host.values()) + \
        host_cu.numel() * 4 + host_slots.numel() * 4
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step():
        for n in dev:
            dev[n].copy_(host[n], non_blocking=True)
        cu.copy_(host_cu, non_blocking=True)
        slots.copy_(host_slots, non_blocking=True)
        prefill()
        host_out.copy_(out, non_blocking=True)

    e2e_ms = []
    for _ in range(2 if e2e else 0):
        e2e_step()
    torch.cuda.synchronize()
    for _ in range(max(3, args.steps // 2) if e2e else 0):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    st, bits = kda.kda_device_status(ws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"prefill device check failed: {st} bits={bits}")

    cu_h = b.cu_seqlens.tolist()
    lens = [cu_h[i + 1] - cu_h[i] for i in range(len(cu_h) - 1)]
    n_resumed = int((b.init_slots[:, 0] >= 0).sum())
    nbytes, flops, _ = prefill_algorithmic(w, lens, n_written, n_resumed,
                                           dev["q"].element_size())
    return dict(w=w, T=T, B=len(lens), call_ms=call_ms, kern_ms=kern_ms, clocks=ck,
                nbytes=nbytes, flops=flops, launches=timed_launches, e2e_ms=e2e_ms, h2d=h2d,
                d2h=d2h, n_snaps=n_written, n_resumed=n_resumed)


def retention_map(b, interval, every, n_slots):
    """int32 [n_snaps]: snapshot j of each sequence kept when (j + 1) % every
    == 0, each into its own pool slot that no sequence reads or writes; -1
    elsewhere (the scheduler's retention decision, taken before the call)."""
    import torch
    cu = b.cu_seqlens.tolist()
    used = set(int(x) for x in b.init_slots.flatten().tolist() if x >= 0)
    free = [s for s in range(n_slots) if s not in used]
    out = []
    for i in range(len(cu) - 1):
        for j in range((cu[i + 1] - cu[i]) // interval):
            out.append(-1 if (j + 1) % every else (free.pop(0) if free else None))
    if None in out:
        raise ValueError(f"--retain {every}: the workload's pool has {n_slots} slots, too few "
                         "free ones for the kept snapshots (use a workload with a slot pool, "
                         "e.g. --workload varlen_resume)")
    return torch.tensor(out, dtype=torch.int32)


def bench_decode(name, args, torch, kda, inputs):
    fused = name.startswith("decode_fused")
    w = inputs.WORKLOADS["decode_256x1" if fused else name]
    b = inputs.make_batch(w, device="cuda")
    dev = {n: getattr(b, n) for n in ("q", "k", "v", "g", "beta")}
    slot_ids = b.slot_ids.cuda()
    pool = b.pool
    N = slot_ids.numel()
    H = w.H
    out = torch.empty((N * w.n_tok, H, w.dv), dtype=dev["q"].dtype, device="cuda")
    per = (torch.empty((N, w.n_tok, H, w.dk, w.dv), dtype=torch.float32, device="cuda")
           if w.per_tok_states else None)
    ws = kda.workspace_for(N, H, pool.shape[0])
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    if fused:
        ft = inputs.fused_tensors(N * w.n_tok, H, w.dk, w.dv, dev["q"].dtype, w.index, w.n_slots,
                                  device="cuda")

        def call(events):
            kda.kda_decode_fused(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], ft["gate"],
                                 ft["conv_w"], ft["norm_w"], slot_ids, pool, ft["conv_pool"], out,
                                 w.n_tok, workspace=ws, events=events)
    elif w.spec:
        prev = {n: t.cuda() for n, t in b.extra["prev"].items()}
        acc = b.extra["accepted"].cuda()

        def call(events):
            kda.kda_decode_spec(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], slot_ids,
                                pool, out, w.n_tok, prev["k"], prev["v"], prev["g"],
                                prev["beta"], acc, w.n_tok, workspace=ws, events=events)
    else:
        def call(events):
            kda.kda_decode(dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], slot_ids, pool,
                           out, w.n_tok, per, workspace=ws, events=events)

    call_ms, kern_ms = time_calls(call, args.steps, args.warmup, flush, torch)
    st, bits = kda.kda_device_status(ws)
    if st != kda.KDA_OK:
        raise RuntimeError(f"decode device check failed: {st} bits={bits}")
    if fused:
        nbytes = fused_decode_algorithmic(w, N, w.n_tok, dev["q"].element_size())
    elif w.spec:
        nbytes = spec_algorithmic(w, N, b.extra["accepted"], dev["q"].element_size())
    else:
        nbytes = decode_algorithmic(w, N, w.n_tok, w.per_tok_states, dev["q"].element_size())
    return dict(w=w, N=N, call_ms=call_ms, kern_ms=kern_ms, nbytes=nbytes)


def _uuid(torch):
    try:
        u = torch.cuda.get_device_properties(0).uuid
        return "GPU-" + str(u)
    except Exception:
        return None


# ------------------------------------------------------------------ CPU oracle

class OracleSample:
    """The fp64 C oracle timed on whole heads of a prefill workload's first
    sequence (at most 8192 tokens of it, from a zero state: the oracle's cost
    per token-head does not depend on the state).  Inputs are drawn once."""

    def __init__(self, workload):
        import numpy as np
        import oracle
        from hybrid_linear_attention_delta_gb300 import inputs
        self.oracle, self.np = oracle, np
        self.w = w = inputs.WORKLOADS[workload]
        lens = inputs.seq_lengths(w)
        self.T = min(lens[0], 8192)
        tt = inputs.token_tensors(self.T, w.H, w.dk, w.dv, inputs.torch_dtype(w.dtype), w.index,
                                  "cpu")
        self.cores = oracle.host_cores()
        self.arrs = {n: oracle._f64(tt[n]) for n in ("q", "k", "v", "g", "beta")}
        self.cu = np.array([0, self.T], dtype=np.int64)
        self.tok_heads = sum(lens) * w.H    # of the whole workload

    def run_heads(self, n, threads=None):
        sub = {k: self.np.ascontiguousarray(a[:, :n]) for k, a in self.arrs.items()}
        t0 = time.perf_counter()
        self.oracle.run(sub["q"], sub["k"], sub["v"], sub["g"], sub["beta"], self.cu, None,
                        self.w.snap_interval, nthreads=threads or self.cores)
        return time.perf_counter() - t0

    def measure(self, target_s, max_heads=None, one_core=False):
        """Returns a cpu_baseline dict whose value is the workload's tokens/s
        at the sampled token-head rate."""
        w = self.w
        t1 = max(self.run_heads(1), 1e-3)
        n = int(min(max_heads or w.H, w.H, max(1, target_s / t1)))
        reps, t = 0, 0.0
        while reps == 0 or (t < 0.8 * target_s and reps < 64):
            t += self.run_heads(n)
            reps += 1
        t /= reps
        rate = self.T * n / t                       # token-heads per second
        tokens = self.tok_heads / w.H
        value = rate / w.H                          # tokens/s of H-head work
        out = {"value": value, "unit": "tokens/s", "cores": self.cores, "kind": "oracle",
               "sample": f"{n} of {w.H} heads x {self.T} tokens of {w.name} (C fp64, "
                         f"{self.cores} threads over 16-column state blocks), {t:.2f} s "
                         f"per pass, mean of {reps}; "
                         f"value = tokens/s of all {w.H} heads at that rate "
                         f"({tokens:.0f}-token workload)",
               "seconds": t}
        if one_core:  # the same oracle on one thread, one head
            t1c = self.run_heads(1, threads=1)
            out["one_core"] = {"value": self.T / t1c / w.H, "unit": "tokens/s", "cores": 1,
                               "sample": f"1 head x {self.T} tokens, 1 thread, {t1c:.2f} s; "
                                         f"value = tokens/s of all {w.H} heads at that rate"}
        return out


# ------------------------------------------------------------------ main

def prefill_kernel_name(pre):
    if pre["w"].dtype != "bf16":
        return "recurrent_kernel (token-recurrent fp32 prefill)"
    if pre["B"] * pre["w"].H <= 64:
        return "coop_kernel (cooperative chunked prefill)"
    return "chunked_kernel (per-state chunked prefill)"


def prefill_roofline(pre, kern_s, P, traffic_key):
    """Roofline of a prefill call's main kernel: algorithmic bytes (and tensor
    FLOP) over its CUDA-event time, against the measured HBM copy bandwidth
    (and bf16 dense peak)."""
    algo_gbs = pre["nbytes"] / kern_s / 1e9
    algo_tflops = pre["flops"] / kern_s / 1e12
    return {"bound": "hbm", "achieved": algo_gbs, "peak": P["hbm_gbs"], "unit": "GB/s",
            "frac": algo_gbs / P["hbm_gbs"],
            "traffic": None if traffic_key is None else ncu_traffic(
                traffic_key, ["kda_chunked.cu", "kda_sm100.cuh"]),
            "kernel": prefill_kernel_name(pre),
            "kernel_ms": kern_s * 1e3, "algorithmic_bytes": pre["nbytes"],
            "peak_source": P["source"],
            "tensor": None if pre["w"].dtype != "bf16" else {
                "achieved": algo_tflops, "unit": "TFLOP/s", "peak": P.get("bf16_tflops"),
                "frac": algo_tflops / P.get("bf16_tflops", 1900.0),
                "algorithmic_flops": pre["flops"]}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=HEADLINE,
                    choices=["prefill_8k", "varlen_resume", "prefill_1m", "prefill_3x32k",
                             "tiny_f32"],
                    help="prefill workload of a step (default: the 2^20-token single sequence)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="shorten the step's single-sequence workload to this many tokens "
                         "(profiling captures of a smaller case; not a bench number)")
    ap.add_argument("--seqs", type=int, default=0,
                    help="keep only the first N sequences of the step's varlen workload "
                         "(profiling captures of a smaller case; not a bench number)")
    ap.add_argument("--retain", type=int, default=0,
                    help="keep every N-th interval snapshot in pool slots (retention map) "
                         "instead of writing all of them to the snapshot buffer")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other prefill workloads (reported under \"prefill\")")
    ap.add_argument("--no-prefill", action="store_true", help="decode only (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer leg (profiling)")
    ap.add_argument("--fused", action="store_true",
                    help="run the step's prefill through the layer around the recurrence "
                         "(convolution, prefill, gated RMSNorm); profiling captures, no e2e leg")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    import hybrid_linear_attention_delta_gb300 as kda
    from hybrid_linear_attention_delta_gb300 import inputs
    kda.lib()   # raises if the CUDA library has not been built

    P = peaks()
    if not args.no_prefill:
        pre = bench_prefill(args, torch, kda, inputs, world, rank, args.workload,
                            retain=args.retain, e2e=not (args.no_e2e or args.fused),
                            fused=args.fused)
        step_s = statistics.mean(pre["call_ms"]) / 1e3
        kern_s = statistics.mean(pre["kern_ms"]) / 1e3
        e2e_s = statistics.mean(pre["e2e_ms"]) / 1e3 if pre["e2e_ms"] else float("nan")
        step_s, e2e_s, kern_s = reduce_over_ranks(torch, [step_s, e2e_s, kern_s], "cuda")

    extra = {}
    if not (args.no_prefill or args.no_extra or args.tokens or args.seqs):
        for name in EXTRA_PREFILL:
            if name == args.workload:
                continue
            r = bench_prefill(args, torch, kda, inputs, world, rank, name, e2e=False)
            ks = statistics.mean(r["kern_ms"]) / 1e3
            cs = statistics.mean(r["call_ms"]) / 1e3
            extra[name] = {"workload": r["w"].note, "ms_per_call": cs * 1e3,
                           "kernel_ms": ks * 1e3, "tokens_per_s": r["T"] / cs,
                           "snapshots": r["n_snaps"], "resumed": r["n_resumed"],
                           "roofline": prefill_roofline(r, ks, P, "prefill_" + name)}
        # the layer around the recurrence on the 8k-token workload: the whole
        # call (plan, convolution, convolution states, prefill, recomputation
        # check, gated RMSNorm), its bytes those of the layer's inputs and
        # outputs (raw q, k, v, g, beta, gate in; the normed output out)
        r = bench_prefill(args, torch, kda, inputs, world, rank, "prefill_8k", e2e=False,
                          fused=True)
        ks = statistics.mean(r["kern_ms"]) / 1e3
        cs = statistics.mean(r["call_ms"]) / 1e3
        w8 = r["w"]
        fb = r["T"] * w8.H * (3 * w8.dk + 1 + 3 * w8.dv) * 2 + \
            w8.H * w8.dk * w8.dv * 4 * (1 + r["n_snaps"]) + \
            2 * w8.H * (2 * w8.dk + w8.dv) * 3 * 2
        extra["prefill_8k_fused"] = {
            "workload": w8.note + "; with the short convolution and the gated RMSNorm",
            "ms_per_call": cs * 1e3, "prefill_kernel_ms": ks * 1e3,
            "tokens_per_s": r["T"] / cs, "launches": r["launches"] // max(args.steps, 1),
            "call_GBps": fb / cs / 1e9, "algorithmic_bytes": fb,
            "roofline": {"bound": "hbm", "achieved": fb / cs / 1e9, "peak": P["hbm_gbs"],
                         "unit": "GB/s", "frac": fb / cs / 1e9 / P["hbm_gbs"], "traffic": None,
                         "kernel": "whole call (6 kernels)", "peak_source": P["source"]}}

    dec = {}
    if not args.no_decode:
        for name in ("decode_256x1", "verify_64x8", "spec_verify_64x8", "decode_fused_256x1"):
            r = bench_decode(name, args, torch, kda, inputs)
            ks = statistics.mean(r["kern_ms"]) / 1e3
            cs = statistics.mean(r["call_ms"]) / 1e3
            gbs = r["nbytes"] / ks / 1e9
            dec[name] = {"workload": r["w"].note, "ms_per_call": cs * 1e3,
                         "kernel_ms": ks * 1e3, "tokens_per_s": r["N"] * r["w"].n_tok / cs,
                         "state_GBps": gbs, "algorithmic_bytes": r["nbytes"],
                         "roofline": {"bound": "hbm", "achieved": gbs, "peak": P["hbm_gbs"],
                                      "unit": "GB/s", "frac": gbs / P["hbm_gbs"],
                                      "traffic": ncu_traffic(
                                          "decode128_" + name,
                                          ["kda_fused.cu" if name.startswith("decode_fused")
                                           else "kda_decode.cu"]),
                                      "kernel": DECODE_KERNEL[name],
                                      "peak_source": P["source"]}}

    if rank != 0:
        if world > 1:
            torch.distributed.barrier()
        return 0
    if args.no_prefill:
        print(json.dumps({"metric": METRIC, "note": "decode-only run", "decode": dec}), flush=True)
        return 0

    cpu = None
    if not args.no_cpu_baseline:
        cpu = OracleSample(args.workload).measure(target_s=12.0, one_core=True)
        cpu.pop("seconds", None)

    short = (f" shortened to {args.tokens} tokens" if args.tokens else
             f" (first {args.seqs} sequences only)" if args.seqs else "")
    line = {
        "metric": METRIC,
        "value": job_throughput(pre["T"], world, step_s),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": pre["w"].dtype,
        "data": "synthetic (seeded; q,k L2-normalised, g=-exp(N(-3,1)), beta=sigmoid(N(0,1)))",
        "config": {"workload": f'{pre["w"].name}: {pre["w"].note}{short}', "B": pre["B"],
                   "T": pre["T"], "H": pre["w"].H, "dk": pre["w"].dk, "dv": pre["w"].dv,
                   "snapshots": pre["n_snaps"], "resumed": pre["n_resumed"],
                   **({"retention": f"every {args.retain}th interval snapshot kept in a pool "
                                    "slot (kda_prefill_varlen_retain)"} if args.retain else {}),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "flushed between timed steps (256 MiB write); inputs exceed L2"},
        "roofline": prefill_roofline(pre, kern_s, P,
                                     None if (args.retain or args.tokens or args.seqs or args.fused)
                                     else "prefill_" + args.workload),
        "cpu_baseline": cpu,
        "e2e": None if (args.no_e2e or args.fused) else {"value": job_throughput(pre["T"], world, e2e_s),
                                         "unit": "tokens/s",
                                         "h2d_bytes_per_step": pre["h2d"],
                                         "d2h_bytes_per_step": pre["d2h"]},
        "gpu_launches": pre["launches"],
        "clocks": pre["clocks"],
        "prefill": extra,
        "decode": dec,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
    return 0


def reference_arm(args, world, rank):
    """The fp64 CPU oracle as it stands, on bounded samples of the workload
    (each step about 2 s of CPU work on whole heads)."""
    if rank != 0:
        return 0
    sampler = OracleSample(args.workload)
    per = []
    for i in range(args.warmup + args.steps):
        r = sampler.measure(target_s=2.0)
        if i >= args.warmup:
            per.append(r)
    value = statistics.mean(r["value"] for r in per)
    ms = statistics.mean(r["seconds"] for r in per) * 1e3
    cpu = {"value": value, "unit": "tokens/s", "cores": per[-1]["cores"], "kind": "oracle",
           "sample": per[-1]["sample"]}
    w = sampler.w
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": f"{w.name}: {w.note}", "sample": cpu["sample"]},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
