"""Benchmark: one step = the whole hot path on synthetic inputs resident in HBM:

  * prefill  attn_fwd    on the long causal workload  B=1, H=32, N=8192, d=128
                         (1% of K rows x2, seeded), bf16 in / bf16 O + fp32 lse
  * decode   attn_decode on the paged GQA workload     64 sequences, Hq=32, Hkv=8,
                         d=128, 16-token blocks, lengths U[1024, 32768], random table

Prints ONE JSON line (rank 0). ``value`` is prefill TFLOP/s (algorithmic FLOPs:
4 * d per allowed (query, key) pair, i.e. 4 N^2 d per head halved for causal);
``decode`` carries the decode KV-read GB/s. Both inputs exceed the 129 MB L2,
so no flush is needed between steps. ``backward`` times attn_bwd on the prefill
workload in a loop of its own after the step (same warm-up and step counts;
10 * d FLOPs per allowed pair); ``--no-backward`` skips it. ``paged_prefill`` times
attn_prefill_paged on the chunked-prefill workload (16 sequences, 2048 new queries
each over a paged cache) the same way; ``--no-paged-prefill`` skips it. ``blocksparse``
times attn_fwd_blocksparse on a 32k-token global + local block pattern the same way
(4 * d FLOPs per allowed pair of the listed blocks); ``--no-blocksparse`` skips it.
``fp8_prefill`` times attn_fwd_fp8 on the long causal workload quantised per tensor to
E4M3 (same FLOP count; roofline against twice the measured bf16 peak);
``--no-fp8`` skips it.
``decode_graph`` times a 32-layer decode step (8 sequences, each layer its own cache) two
ways: one attn_decode call per layer, and the same calls captured once with
attn_decode_graph_create and replayed with one graph launch per step (KV GB/s over the
step); ``--no-decode-graph`` skips it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (the only other place, with ``cpu_baseline``, where the oracle runs).
Multi-GPU (torchrun, N > 1): independent replicas, one per GPU (the path has no
exchange step); value = all ranks' work / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s & % bf16 peak; decode KV-read GB/s & % HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- accounting
def allowed_pairs(Nq: int, Nk: int, causal: bool, window: int) -> int:
    """Number of (query, key) pairs the mask allows, summed over the rows of one head."""
    i = np.arange(Nq, dtype=np.int64)
    diag = i + (Nk - Nq)
    hi = np.minimum(Nk, diag + 1) if causal else np.full(Nq, Nk, dtype=np.int64)
    lo = np.maximum(0, diag - window) if window >= 0 else np.zeros(Nq, dtype=np.int64)
    return int(np.maximum(hi - lo, 0).sum())


def attention_flops(B, Hq, Nq, Nk, d, causal=False, window=-1) -> int:
    """Algorithmic FLOPs: two matmuls (Q K^T and P V), 2 FLOPs per multiply-add, over the
    allowed pairs -- 4 N^2 d per head without a mask ("Attention kernels", FLOP count)."""
    return 4 * d * allowed_pairs(Nq, Nk, causal, window) * B * Hq


def backward_flops(B, Hq, Nq, Nk, d, causal=False, window=-1) -> int:
    """Algorithmic FLOPs of the backward with the scores recomputed: five matmuls over the
    allowed pairs (S = Q K^T, dP = dO V^T, dV = P^T dO, dK = dS^T Q, dQ = dS K), i.e.
    2.5 times the forward ("Modern attention kernels", "Backward pass recomputes scores")."""
    return 10 * d * allowed_pairs(Nq, Nk, causal, window) * B * Hq


def paged_prefill_flops(q_lens, kv_lens, Hq, d, causal=True, window=-1) -> int:
    """Algorithmic FLOPs of prefill over a paged cache: 4 d per allowed pair, each sequence
    with its own Nq = q_len and Nk = kv_len (bottom-right alignment)."""
    return int(sum(4 * d * allowed_pairs(int(a), int(b), causal, window) * Hq for a, b in zip(q_lens, kv_lens)))


def blocksparse_pairs(pattern, Nq, Nk, causal, window, block=128) -> int:
    """Allowed (query, key) pairs of one head under a block pattern [n_qblk][n_kblk], counted
    exactly per listed block pair with the causal / window mask (bottom-right alignment)."""
    pat = np.asarray(pattern, dtype=bool)
    delta = Nk - Nq
    total = 0
    for r, c in zip(*np.nonzero(pat)):
        i = np.arange(r * block, min((r + 1) * block, Nq), dtype=np.int64)
        lo = np.full(i.shape, c * block, dtype=np.int64)
        hi = np.full(i.shape, min((c + 1) * block, Nk), dtype=np.int64)
        if causal:
            hi = np.minimum(hi, i + delta + 1)
        if window >= 0:
            lo = np.maximum(lo, i + delta - window)
        total += int(np.maximum(hi - lo, 0).sum())
    return total


def score_matrix_bytes(N: int, bytes_per_el: int = 2) -> int:
    """Size of one head's N x N score matrix."""
    return N * N * bytes_per_el


def naive_score_traffic_bytes(N: int, heads: int, layers: int, bytes_per_el: int = 2) -> int:
    """Score-matrix traffic of materialised attention: S written, read, P written, read."""
    return 4 * score_matrix_bytes(N, bytes_per_el) * heads * layers


def decode_kv_bytes(seq_lens, Hkv: int, d: int) -> int:
    """Bytes of K and V the decode step must read: every cached token of every sequence."""
    return int(np.asarray(seq_lens, dtype=np.int64).sum()) * Hkv * d * 2 * 2


def prefill_io_bytes(B, Hq, Hkv, Nq, Nk, d) -> int:
    """Compulsory HBM bytes of prefill: Q, K, V read once; O and lse written once."""
    return 2 * d * (B * Hq * Nq * 2 + B * Hkv * Nk * 2) + 4 * B * Hq * Nq


# ----------------------------------------------------------------------------- multi-rank
def reduce_max(vals, world: int, device):
    """Element-wise maximum of per-rank timings across all ranks (identity for one rank)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def whole_job_rate(units_per_rank: float, world: int, max_ms: float, unit_scale: float) -> float:
    """Replicas: every rank does the same work; the job's rate is all ranks' units over the
    slowest rank's time."""
    return world * units_per_rank / (max_ms * 1e-3) / unit_scale


# ----------------------------------------------------------------------------- environment
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {
    "attn_fwd_sm103": ("fwd_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_decode_sm103": ("decode_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_bwd_sm103": ("bwd_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_fwd_sm103_paged": ("fwd_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_fwd_sm103_sparse": ("fwd_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_fwd_sm103_fp8": ("fwd_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_decode_sm103_c8_step": ("decode_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_fwd_sm103_c1": ("fwd_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_fwd_sm103_c2": ("fwd_kernel.cu", "ptx.cuh", "internal.h"),
    "attn_fwd_sm103_c4": ("fwd_kernel.cu", "ptx.cuh", "internal.h"),
}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the sources a kernel is built from (so stale counters can be detected)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_06_gb300", "csrc")
    for fn in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch (read + write) from the committed ncu summary, or None when
    the kernel's sources changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(kernel)
        if e and e.get("source_hash") == kernel_source_hash(kernel):
            return float(e["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the benchmark runs.
    ``mark()`` brackets the timed step region and ``window(name)`` each further timed loop;
    the summary covers the samples taken inside those windows (the step region's own
    samples are reported separately, since a short step region may hold only a few)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.gpu = gpu_index
        self.interval = interval_ms
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None
        self.windows = []  # (name, start, end) of the timed loops after the step

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            import atexit
            atexit.register(self.__exit__, None, None, None)  # never leave the sampler running
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def window(self, name: str, start: float, end: float):
        self.windows.append((name, start, end))

    def __exit__(self, *exc):
        if self.proc is not None and self.proc.returncode is None and not self.out.closed:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        import datetime
        if self.proc is None or not self.path:
            return None
        try:
            rows = list(csv.reader(io.StringIO(open(self.path).read())))
            os.unlink(self.path)
        except Exception:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        step, timed, everything = [], [], []
        for r in rows:
            if len(r) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rec = (float(r[2]), float(r[3]), [n for n, v in zip(names, r[6:10]) if v.strip().lower() == "active"],
                       float(r[4]) if r[4].strip() not in ("", "[N/A]") else None)
            except ValueError:
                continue
            everything.append(rec)
            in_step = self.t0 is not None and self.t1 is not None and self.t0 <= ts <= self.t1
            if in_step:
                step.append(rec)
            if in_step or any(a <= ts <= b for _, a, b in self.windows):
                timed.append(rec)
        use = timed or everything
        if not use:
            return None
        reasons = sorted({n for rec in use for n in rec[2]})
        power = [rec[3] for rec in use if rec[3] is not None]
        return {"sm_mhz": float(np.median([rec[0] for rec in use])), "sm_max_mhz": float(max(rec[1] for rec in use)),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(step),
                "step_region_sm_mhz": float(np.median([rec[0] for rec in step])) if step else None,
                "timed_loops": len(self.windows), "interval_ms": self.interval,
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------------------- our arm
class Part:
    """One half of the step: its inputs (pinned host + device), outputs and work units."""

    def __init__(self, name, host, outputs, run, units, unit_scale, unit, launches):
        self.name, self.host, self.outputs, self.run = name, host, outputs, run
        self.units, self.unit_scale, self.unit, self.launches = units, unit_scale, unit, launches
        self.dev = None


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import exact_tiled_attention_06_gb300 as eta
    from exact_tiled_attention_06_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    eta.build()
    eta.load_library()
    pc, dc = inputs.C3, inputs.C5
    parts = []

    if args.workload in ("both", "prefill"):
        q_h, k_h, v_h = inputs.prefill_config_inputs(pc, seed=pc.seed + rank)
        host = {n: t.pin_memory() for n, t in (("q", q_h), ("k", k_h), ("v", v_h))}
        o = torch.empty(q_h.shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty((pc.B, pc.Hq, pc.Nq), dtype=torch.float32, device=dev)

        def run_prefill(ins):
            eta.attn_fwd(ins["q"], ins["k"], ins["v"], causal=pc.causal, window=pc.window, scale=pc.scale, out=o,
                         lse=lse)

        flops = attention_flops(pc.B, pc.Hq, pc.Nq, pc.Nk, pc.d, pc.causal, pc.window)
        parts.append(Part("prefill", host, (o, lse), run_prefill, flops, 1e12, "TFLOP/s", 1))

    if args.workload in ("both", "decode"):
        if args.decode_seqs:
            dx = inputs.decode_inputs(args.decode_seqs, dc.Hq, dc.Hkv, dc.d, dc.block_size, len_lo=dc.len_lo,
                                      len_hi=dc.len_hi, seed=dc.seed + rank)
        else:
            dx = inputs.decode_config_inputs(dc, seed=dc.seed + rank)
        S = dx.q.shape[0]
        host = {n: t.pin_memory() for n, t in (("q", dx.q), ("kc", dx.k_cache), ("vc", dx.v_cache),
                                                ("bt", dx.block_table), ("sl", dx.seq_lens))}
        do = torch.empty(dx.q.shape, dtype=torch.bfloat16, device=dev)
        dlse = torch.empty((S, dc.Hq), dtype=torch.float32, device=dev)
        mb = dx.block_table.shape[1]
        ws = torch.empty(eta.attn_decode_workspace_size(S, dc.Hq, dc.Hkv, dc.d, dc.block_size, mb),
                         dtype=torch.uint8, device=dev)

        def run_decode(ins):
            eta.attn_decode(ins["q"], ins["kc"], ins["vc"], ins["bt"], ins["sl"], scale=dc.scale, workspace=ws,
                            out=do, lse=dlse)

        kv_bytes = decode_kv_bytes(dx.seq_lens.numpy(), dc.Hkv, dc.d)
        part = Part("decode", host, (do, dlse), run_decode, kv_bytes, 1e9, "GB/s", 1)
        part.extra = {"num_seqs": S, "sum_seq_len": int(dx.seq_lens.sum()), "workspace_bytes": int(ws.numel()),
                      "workspace": ws, "seq_lens": dx.seq_lens.tolist()}
        parts.append(part)

    for p in parts:
        p.dev = {n: t.to(dev) for n, t in p.host.items()}
    stream = torch.cuda.current_stream()

    # ---- warm-up
    for _ in range(args.warmup):
        for p in parts:
            p.run(p.dev)
    torch.cuda.synchronize()
    err = eta.attn_get_device_error()
    if err != 0:
        raise RuntimeError(f"device error during warm-up: {eta.attn_status_string(err)}")

    # ---- timed region: K steps; CUDA events around each part on the launching stream
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in parts]
          for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank).__enter__()  # runs until every timed loop below is done
    clocks.mark(True)
    torch.cuda.nvtx.range_push("timed step")
    t_start.record(stream)
    for i in range(args.steps):
        for j, p in enumerate(parts):
            ev[i][j][0].record(stream)
            p.run(p.dev)
            ev[i][j][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    clocks.mark(False)
    if world > 1:
        dist.barrier()
    err = eta.attn_get_device_error()
    if err != 0:
        raise RuntimeError(f"device error in the timed region: {eta.attn_status_string(err)}")
    total_ms = t_start.elapsed_time(t_end)
    part_ms = [np.array([ev[i][j][0].elapsed_time(ev[i][j][1]) for i in range(args.steps)])
               for j in range(len(parts))]

    # ---- end to end through the public API with host buffers: every step copies its
    #      inputs host->device, runs, and copies its outputs device->host (pinned memory)
    e2e_ms = [0.0 for _ in parts]
    e2e_steps = 0
    h2d = d2h = 0
    if not args.no_e2e:
        outs_h = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in p.outputs] for p in parts]
        h2d = sum(t.numel() * t.element_size() for p in parts for t in p.host.values())
        d2h = sum(t.numel() * t.element_size() for p in parts for t in p.outputs)
        e2e_steps = max(1, min(args.steps, 5))
        e_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in parts]
                for _ in range(e2e_steps)]

        def e2e_call(j, p):
            # the library's host-buffer entry points: copies in, compute, copies out (prefill
            # pipelines chunks of kv heads over two copy streams and the compute stream)
            oh, lh = outs_h[j]
            if p.name == "prefill":
                eta.attn_fwd_host(p.host["q"], p.host["k"], p.host["v"], oh, lh, p.dev["q"], p.dev["k"], p.dev["v"],
                                  p.outputs[0], p.outputs[1], causal=pc.causal, window=pc.window, scale=pc.scale)
            else:
                eta.attn_decode_host(p.host["q"], p.host["kc"], p.host["vc"], p.host["bt"], p.host["sl"], oh, lh,
                                     p.dev["q"], p.dev["kc"], p.dev["vc"], p.dev["bt"], p.dev["sl"], p.outputs[0],
                                     p.outputs[1], scale=dc.scale, workspace=p.extra["workspace"])

        def e2e_step(i=None):
            for j, p in enumerate(parts):
                if i is not None:
                    e_ev[i][j][0].record(stream)
                e2e_call(j, p)
                if i is not None:
                    e_ev[i][j][1].record(stream)

        # untimed warm-up: the first copies into freshly pinned pages run far below the link rate
        for _ in range(max(1, min(args.warmup, 3))):
            e2e_step()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push("timed e2e step")
        for i in range(e2e_steps):
            e2e_step(i)
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_pop()
        e2e_ms = [float(np.mean([e_ev[i][j][0].elapsed_time(e_ev[i][j][1]) for i in range(e2e_steps)]))
                  for j in range(len(parts))]

    def timed_loop(run, what):
        """W untimed calls, then at least K calls (and at least --min-loop-seconds of them,
        so the clock sampler sees the loop) each bracketed by CUDA events on the launching
        stream, between barriers; the device error word is checked after both."""
        for _ in range(max(args.warmup, 1)):
            run()
        torch.cuda.synchronize()
        err = eta.attn_get_device_error()
        if err != 0:
            raise RuntimeError(f"device error in the {what} warm-up: {eta.attn_status_string(err)}")
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(3):
            run()
        c1.record(stream)
        torch.cuda.synchronize()
        est_ms = max(c0.elapsed_time(c1) / 3, 1e-3)
        reps = int(max(args.steps, min(math.ceil(args.min_loop_seconds * 1e3 / est_ms), 100000)))
        reps = int(reduce_max([reps], world, dev)[0])  # every rank times the same count
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        torch.cuda.nvtx.range_push(f"timed {what}")
        w0 = time.time()
        for e0, e1 in evs:
            e0.record(stream)
            run()
            e1.record(stream)
        torch.cuda.synchronize()
        clocks.window(what, w0, time.time())
        torch.cuda.nvtx.range_pop()
        if world > 1:
            dist.barrier()
        err = eta.attn_get_device_error()
        if err != 0:
            raise RuntimeError(f"device error in the timed {what}: {eta.attn_status_string(err)}")
        return np.array([e0.elapsed_time(e1) for e0, e1 in evs])

    # ---- backward of the prefill workload, in a loop of its own: W untimed launches,
    #      then K launches bracketed by CUDA events on the launching stream (inputs and
    #      the fp32 dQ accumulator exceed L2, so no flush is needed)
    bwd_ms = None
    pre = next((p for p in parts if p.name == "prefill"), None)
    if pre is not None and not args.no_backward:
        do_d = inputs.grad_output(pc.B, pc.Hq, pc.Nq, pc.d, seed=pc.seed + rank).to(dev)
        ws_b = torch.empty(eta.attn_bwd_workspace_size(pc.B, pc.Hq, pc.Nq, pc.d), dtype=torch.uint8, device=dev)
        dq = torch.empty_like(pre.dev["q"])
        dk = torch.empty_like(pre.dev["k"])
        dv = torch.empty_like(pre.dev["v"])
        pre.run(pre.dev)  # o and lse of these inputs

        def run_bwd():
            eta.attn_bwd(pre.dev["q"], pre.dev["k"], pre.dev["v"], o, do_d, lse, causal=pc.causal,
                         window=pc.window, scale=pc.scale, workspace=ws_b, dq=dq, dk=dk, dv=dv)

        bwd_ms = timed_loop(run_bwd, "backward")

    # ---- chunked prefill over a paged cache, in a loop of its own (inputs exceed L2)
    pp_ms = None
    ppc = inputs.C6
    if args.workload in ("both", "prefill") and not args.no_paged_prefill:
        px = inputs.paged_prefill_config_inputs(ppc, seed=ppc.seed + rank)
        pq, pkc, pvc = px.q.to(dev), px.k_cache.to(dev), px.v_cache.to(dev)
        pbt, pql, pkl = px.block_table.to(dev), px.q_lens.to(dev), px.kv_lens.to(dev)
        po = torch.empty_like(pq)
        plse = torch.empty(pq.shape[:3], dtype=torch.float32, device=dev)
        pp_flops = paged_prefill_flops(px.q_lens.tolist(), px.kv_lens.tolist(), ppc.Hq, ppc.d, ppc.causal)

        def run_pp():
            eta.attn_prefill_paged(pq, pkc, pvc, pbt, pql, pkl, causal=ppc.causal, scale=ppc.scale, out=po, lse=plse)

        pp_ms = timed_loop(run_pp, "paged prefill")

    # ---- block-sparse prefill (global + local pattern), in a loop of its own
    bs_ms = None
    spc = inputs.C7
    if args.workload in ("both", "prefill") and not args.no_blocksparse:
        sq, sk, sv, spat = inputs.sparse_config_inputs(spc, seed=spc.seed + rank)
        srp, sci = inputs.block_csr(spat)
        sq, sk, sv, srp, sci = sq.to(dev), sk.to(dev), sv.to(dev), srp.to(dev), sci.to(dev)
        so = torch.empty_like(sq)
        slse = torch.empty(sq.shape[:3], dtype=torch.float32, device=dev)
        bs_flops = 4 * spc.d * spc.B * spc.Hq * blocksparse_pairs(spat.numpy(), spc.N, spc.N, spc.causal, -1)

        def run_bs():
            eta.attn_fwd_blocksparse(sq, sk, sv, srp, sci, causal=spc.causal, scale=spc.scale, out=so, lse=slse)

        bs_ms = timed_loop(run_bs, "block-sparse prefill")

    # ---- FP8 prefill: the long causal workload quantised per tensor to E4M3, in a loop of
    #      its own (inputs 128 MiB + O 64 MiB, above L2)
    f8_ms = None
    if args.workload in ("both", "prefill") and not args.no_fp8:
        fx = inputs.fp8_prefill_inputs(pc.B, pc.Hq, pc.Hkv, pc.Nq, pc.Nk, pc.d, seed=pc.seed + rank,
                                       k_boost_frac=pc.k_boost_frac)
        fq, fk, fvt = fx.q8.to(dev), fx.k8.to(dev), fx.vt8.to(dev)
        fo = torch.empty(fq.shape, dtype=torch.bfloat16, device=dev)
        flse = torch.empty(fq.shape[:3], dtype=torch.float32, device=dev)
        f8_flops = attention_flops(pc.B, pc.Hq, pc.Nq, pc.Nk, pc.d, pc.causal, pc.window)

        def run_f8():
            eta.attn_fwd_fp8(fq, fk, fvt, fx.q_descale, fx.k_descale, fx.v_descale, causal=pc.causal,
                             window=pc.window, scale=pc.scale, out=fo, lse=flse)

        f8_ms = timed_loop(run_f8, "FP8 prefill")

    # ---- a many-layer decode step (every layer its own cache): one attn_decode call per
    #      layer from the host, against the same calls captured once as a CUDA graph and
    #      replayed with one launch per step (the step's KV, ~1 GB, exceeds L2)
    eager_ms = graph_ms = None
    gc = inputs.C8
    if args.workload in ("both", "decode") and not args.no_decode_graph:
        gx = inputs.decode_step_config_inputs(gc, seed=gc.seed + rank)
        gq, gk, gv = ([t.to(dev) for t in ts] for ts in (gx.q, gx.k_cache, gx.v_cache))
        gbt, gsl = gx.block_table.to(dev), gx.seq_lens.to(dev)
        gws = torch.empty(eta.attn_decode_workspace_size(gc.num_seqs, gc.Hq, gc.Hkv, gc.d, gc.block_size,
                                                         gbt.shape[1]), dtype=torch.uint8, device=dev)
        gout = [torch.empty_like(t) for t in gq]
        glse = [torch.empty((gc.num_seqs, gc.Hq), dtype=torch.float32, device=dev) for _ in gq]
        graph = eta.attn_decode_graph_create(gq, gk, gv, gbt, gsl, scale=gc.scale, workspace=gws, outs=gout,
                                             lses=glse)
        g_kv = gc.n_layers * decode_kv_bytes(gx.seq_lens.numpy(), gc.Hkv, gc.d)

        def run_eager():
            for l in range(gc.n_layers):
                eta.attn_decode(gq[l], gk[l], gv[l], gbt, gsl, scale=gc.scale, workspace=gws, out=gout[l],
                                lse=glse[l])

        def run_graph():
            graph.launch(stream)

        eager_ms = timed_loop(run_eager, "per-call decode step")
        graph_ms = timed_loop(run_graph, "graph decode step")
        graph.close()

    # ---- the other prefill workloads (the pages' check shape C1, C2, C4): attn_fwd in a
    #      loop of its own each (C2 and C4 inputs exceed L2; C1 is a latency case of 4
    #      blocks whose inputs stay in L2, reported without a roofline target)
    cfg_ms = {}
    if args.workload in ("both", "prefill") and not args.no_other_prefill:
        for cfg in (inputs.C1, inputs.C2, inputs.C4):
            xq, xk, xv = (t.to(dev) for t in inputs.prefill_config_inputs(cfg, seed=cfg.seed + rank))
            xo = torch.empty(xq.shape, dtype=torch.bfloat16, device=dev)
            xl = torch.empty(xq.shape[:3], dtype=torch.float32, device=dev)

            def run_cfg(cfg=cfg, xq=xq, xk=xk, xv=xv, xo=xo, xl=xl):
                eta.attn_fwd(xq, xk, xv, causal=cfg.causal, window=cfg.window, scale=cfg.scale, out=xo, lse=xl)

            if args.only_config and not cfg.name.startswith(args.only_config):
                continue
            per_call = timed_loop(run_cfg, cfg.name)
            # the same launches replayed from a captured graph (100 per replay): the kernel's
            # own time without the host's per-call cost, which dominates the 4-block C1
            cfg_graph_ms = None
            try:
                if args.no_graph_replay:
                    raise RuntimeError("skipped")
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for _ in range(100):
                        run_cfg()
                g.replay()
                torch.cuda.synchronize()
                g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                reps = 10
                g0.record(stream)
                for _ in range(reps):
                    g.replay()
                g1.record(stream)
                torch.cuda.synchronize()
                cfg_graph_ms = g0.elapsed_time(g1) / (reps * 100)
                del g
            except Exception:
                cfg_graph_ms = None
            err = eta.attn_get_device_error()
            if err != 0:
                raise RuntimeError(f"device error in the {cfg.name} graph replay: {eta.attn_status_string(err)}")
            cfg_ms[cfg.name] = (cfg, per_call, cfg_graph_ms)
            del xq, xk, xv, xo, xl
    clocks.__exit__(None, None, None)

    # ---- max over ranks
    extra = ([float(bwd_ms.mean())] if bwd_ms is not None else []) + ([float(pp_ms.mean())] if pp_ms is not None else [])
    extra += [float(bs_ms.mean())] if bs_ms is not None else []
    extra += [float(eager_ms.mean()), float(graph_ms.mean())] if graph_ms is not None else []
    extra += [float(f8_ms.mean())] if f8_ms is not None else []
    extra += [float(v[1].mean()) for v in cfg_ms.values()]
    vals = reduce_max([total_ms] + [float(m.mean()) for m in part_ms] + e2e_ms + extra, world, dev)
    cfg_means = {}
    for name in reversed(list(cfg_ms)):
        cfg_means[name] = vals.pop()
    f8_mean = vals.pop() if f8_ms is not None else None
    graph_mean = vals.pop() if graph_ms is not None else None
    eager_mean = vals.pop() if graph_ms is not None else None
    bs_mean = vals.pop() if bs_ms is not None else None
    pp_mean = vals.pop() if pp_ms is not None else None
    bwd_mean = vals.pop() if bwd_ms is not None else None
    total_ms, means, e2e_ms = vals[0], vals[1:1 + len(parts)], vals[1 + len(parts):]
    if rank != 0:
        return None

    peaks, peak_kind = load_peaks()

    def roofline(p, mean_ms, ms):
        achieved = p.units / (mean_ms * 1e-3) / p.unit_scale  # one launch on one GPU
        if p.name == "prefill":
            rf = {"kernel": "attn_fwd_sm103<128>", "bound": "tensor", "achieved": round(achieved, 2),
                  "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                  "frac": round(achieved / peaks["bf16_tflops"], 4),
                  "peak_kind": f"{peak_kind} bf16 dense burst",
                  "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                  "traffic": load_traffic("attn_fwd_sm103")}
        else:
            rf = {"kernel": "attn_decode_sm103<128>", "bound": "hbm",
                  "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                  "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_kind": f"{peak_kind} HBM copy",
                  "traffic": load_traffic("attn_decode_sm103")}
        rf["ms_per_launch"] = round(mean_ms, 4)
        rf["ms_p10_p50_p90"] = [round(float(np.percentile(ms, x)), 4) for x in (10, 50, 90)]
        return rf

    main_p, main_ms = parts[0], means[0]
    value = whole_job_rate(main_p.units, world, main_ms, main_p.unit_scale)
    config = {"workload": " + ".join({"prefill": pc.name, "decode": dc.name}[p.name] for p in parts),
              "l2": "inputs larger than L2 (prefill Q/K/V 192 MiB, decode KV ~4 GB); no flush",
              "parallelism": f"replicas x{world}"}
    for p in parts:
        if p.name == "prefill":
            config["prefill"] = {"B": pc.B, "Hq": pc.Hq, "Hkv": pc.Hkv, "Nq": pc.Nq, "Nk": pc.Nk, "d": pc.d,
                                 "causal": pc.causal, "window": pc.window, "k_boost_frac": pc.k_boost_frac,
                                 "flops_per_launch": p.units}
        else:
            config["decode"] = {"num_seqs": p.extra["num_seqs"], "Hq": dc.Hq, "Hkv": dc.Hkv, "d": dc.d,
                                "block_size": dc.block_size, "len_range": [dc.len_lo, dc.len_hi],
                                "sum_seq_len": p.extra["sum_seq_len"], "kv_bytes_per_launch": p.units}
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": main_p.unit,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config,
        "roofline": roofline(main_p, main_ms, part_ms[0]),
    }
    if len(parts) > 1:
        p = parts[1]
        result["decode"] = {"value": round(whole_job_rate(p.units, world, means[1], p.unit_scale), 2), "unit": p.unit,
                            "roofline": roofline(p, means[1], part_ms[1]),
                            "workspace_bytes": p.extra["workspace_bytes"]}
    if not args.no_e2e:
        e2e = {"value": round(whole_job_rate(main_p.units, world, e2e_ms[0], main_p.unit_scale), 3), "unit": main_p.unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(sum(e2e_ms), 3),
               "steps": e2e_steps}
        if len(parts) > 1:
            e2e["decode_value"] = round(whole_job_rate(parts[1].units, world, e2e_ms[1], parts[1].unit_scale), 2)
            e2e["decode_unit"] = parts[1].unit
        result["e2e"] = e2e
    result["gpu_launches"] = sum(p.launches for p in parts) * args.steps
    result["clocks"] = clocks.summary()
    if bwd_ms is not None:
        flops = backward_flops(pc.B, pc.Hq, pc.Nq, pc.Nk, pc.d, pc.causal, pc.window)
        achieved = flops / (bwd_mean * 1e-3) / 1e12
        result["backward"] = {
            "value": round(whole_job_rate(flops, world, bwd_mean, 1e12), 2), "unit": "TFLOP/s",
            "workload": f"attn_bwd on {pc.name}", "flops_per_launch": flops, "steps": args.steps,
            "warmup": args.warmup, "gpu_launches": 3 * args.steps,
            "roofline": {"kernel": "attn_bwd_prep + attn_bwd_sm103<128> + attn_bwd_dq_out", "bound": "tensor",
                         "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "peak_kind": f"{peak_kind} bf16 dense burst",
                         "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                         "traffic": load_traffic("attn_bwd_sm103"),
                         "ms_per_launch": round(bwd_mean, 4),
                         "ms_p10_p50_p90": [round(float(np.percentile(bwd_ms, x)), 4) for x in (10, 50, 90)]},
        }
    if pp_ms is not None:
        achieved = pp_flops / (pp_mean * 1e-3) / 1e12
        result["paged_prefill"] = {
            "value": round(whole_job_rate(pp_flops, world, pp_mean, 1e12), 2), "unit": "TFLOP/s",
            "workload": ppc.name, "flops_per_launch": pp_flops, "steps": args.steps, "warmup": args.warmup,
            "gpu_launches": args.steps,
            "config": {"num_seqs": ppc.num_seqs, "Hq": ppc.Hq, "Hkv": ppc.Hkv, "d": ppc.d,
                       "block_size": ppc.block_size, "q_len": ppc.q_len,
                       "kv_len_sum_min_max": [int(px.kv_lens.sum()), int(px.kv_lens.min()), int(px.kv_lens.max())],
                       "causal": ppc.causal},
            "roofline": {"kernel": "attn_fwd_sm103<128, paged>", "bound": "tensor", "achieved": round(achieved, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "peak_kind": f"{peak_kind} bf16 dense burst",
                         "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                         "traffic": load_traffic("attn_fwd_sm103_paged"),
                         "ms_per_launch": round(pp_mean, 4),
                         "ms_p10_p50_p90": [round(float(np.percentile(pp_ms, x)), 4) for x in (10, 50, 90)]},
        }
    if bs_ms is not None:
        achieved = bs_flops / (bs_mean * 1e-3) / 1e12
        result["blocksparse"] = {
            "value": round(whole_job_rate(bs_flops, world, bs_mean, 1e12), 2), "unit": "TFLOP/s",
            "workload": spc.name, "flops_per_launch": bs_flops, "steps": args.steps, "warmup": args.warmup,
            "gpu_launches": args.steps,
            "config": {"B": spc.B, "Hq": spc.Hq, "Hkv": spc.Hkv, "N": spc.N, "d": spc.d, "causal": spc.causal,
                       "global_blocks": spc.n_global, "local_blocks": spc.n_local,
                       "listed_blocks": int(spat.sum()), "all_blocks": int(spat.numel())},
            "roofline": {"kernel": "attn_fwd_sm103<128, sparse>", "bound": "tensor", "achieved": round(achieved, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "peak_kind": f"{peak_kind} bf16 dense burst",
                         "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                         "traffic": load_traffic("attn_fwd_sm103_sparse"),
                         "ms_per_launch": round(bs_mean, 4),
                         "ms_p10_p50_p90": [round(float(np.percentile(bs_ms, x)), 4) for x in (10, 50, 90)]},
        }
    if f8_ms is not None:
        achieved = f8_flops / (f8_mean * 1e-3) / 1e12
        fp8_peak = 2.0 * peaks["bf16_tflops"]  # measured bf16 dense x the nominal fp8 : bf16 ratio (2)
        result["fp8_prefill"] = {
            "value": round(whole_job_rate(f8_flops, world, f8_mean, 1e12), 2), "unit": "TFLOP/s",
            "workload": pc.name + "_e4m3", "flops_per_launch": f8_flops, "steps": args.steps, "warmup": args.warmup,
            "gpu_launches": args.steps, "dtype": "e4m3 Q/K/V, fp32 accumulation, bf16 O",
            "config": {"B": pc.B, "Hq": pc.Hq, "Hkv": pc.Hkv, "N": pc.Nq, "d": pc.d, "causal": pc.causal,
                       "scales": "per tensor, max|x| / 448"},
            "roofline": {"kernel": "attn_fwd_sm103<128, fp8>", "bound": "tensor", "achieved": round(achieved, 2),
                         "peak": round(fp8_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp8_peak, 4),
                         "peak_kind": f"{peak_kind} bf16 dense burst x 2 (nominal fp8 : bf16)",
                         "frac_of_bf16_peak": round(achieved / peaks["bf16_tflops"], 4),
                         "traffic": load_traffic("attn_fwd_sm103_fp8"),
                         "ms_per_launch": round(f8_mean, 4),
                         "ms_p10_p50_p90": [round(float(np.percentile(f8_ms, x)), 4) for x in (10, 50, 90)]},
        }
    if graph_ms is not None:
        achieved = g_kv / (graph_mean * 1e-3) / 1e9
        result["decode_graph"] = {
            "value": round(whole_job_rate(g_kv, world, graph_mean, 1e9), 2), "unit": "GB/s",
            "workload": gc.name, "kv_bytes_per_step": g_kv, "steps": args.steps, "warmup": args.warmup,
            "gpu_launches": gc.n_layers * args.steps, "graph_nodes_per_step": 2 * gc.n_layers,
            "us_per_step_graph": round(graph_mean * 1e3, 2), "us_per_step_per_call": round(eager_mean * 1e3, 2),
            "per_call_value": round(whole_job_rate(g_kv, world, eager_mean, 1e9), 2),
            "graph_speedup": round(eager_mean / graph_mean, 3),
            "config": {"n_layers": gc.n_layers, "num_seqs": gc.num_seqs, "Hq": gc.Hq, "Hkv": gc.Hkv, "d": gc.d,
                       "block_size": gc.block_size,
                       "seq_len_sum_min_max": [int(gx.seq_lens.sum()), int(gx.seq_lens.min()), int(gx.seq_lens.max())]},
            "roofline": {"kernel": "attn_decode_sm103<128> (x n_layers, one graph)", "bound": "hbm",
                         "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_kind": f"{peak_kind} HBM copy",
                         "traffic": load_traffic("attn_decode_sm103_c8_step"), "traffic_unit": "bytes per step",
                         "ms_per_step": round(graph_mean, 4),
                         "ms_p10_p50_p90": [round(float(np.percentile(graph_ms, x)), 4) for x in (10, 50, 90)]},
        }
    details = {"workloads": "per-sequence lengths of the paged workloads timed in the bench line (seeded draws)"}
    if pp_ms is not None:
        details[ppc.name] = {"kv_lens": px.kv_lens.tolist(), "q_lens": px.q_lens.tolist()}
    if graph_ms is not None:
        details[gc.name] = {"seq_lens": gx.seq_lens.tolist()}
    if len(parts) > 1:
        details[dc.name] = {"seq_lens": parts[1].extra["seq_lens"]}
    result["_details"] = details
    if cfg_ms:
        other = {}
        for name, (cfg, ms, gms) in cfg_ms.items():
            mean = cfg_means[name]
            flops = attention_flops(cfg.B, cfg.Hq, cfg.Nq, cfg.Nk, cfg.d, cfg.causal, cfg.window)
            achieved = flops / (mean * 1e-3) / 1e12
            kernel = f"attn_fwd_sm103<{cfg.d}>"
            other[name] = {
                "value": round(whole_job_rate(flops, world, mean, 1e12), 2), "unit": "TFLOP/s",
                "flops_per_launch": flops, "launches_timed": int(len(ms)),
                "graph_replay": None if gms is None else {
                    "ms_per_launch": round(gms, 5), "value": round(flops / (gms * 1e-3) / 1e12, 2),
                    "frac": round(flops / (gms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)},
                "roofline": {"kernel": kernel, "bound": "tensor", "achieved": round(achieved, 2),
                             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": round(achieved / peaks["bf16_tflops"], 4),
                             "traffic": load_traffic("attn_fwd_sm103_" + name.split("_")[0].lower()),
                             "ms_per_launch": round(mean, 5),
                             "ms_p10_p50_p90": [round(float(np.percentile(ms, x)), 5) for x in (10, 50, 90)]},
            }
        result["prefill_configs"] = other
    return result


# ----------------------------------------------------------------------------- oracle timing
def oracle_sample(heads=32, rows=None, seqs=4):
    """Time the fp64 oracle on a bounded sample of the same workload.

    Prefill: ``heads`` heads of the long causal workload, all rows (or only the last
    ``rows`` rows, the ones with the most keys). Decode: ``seqs`` sequences of the
    longest length of the decode workload, with its heads, block size and layout.
    Returns seconds and work units per part plus a description."""
    import oracle
    from exact_tiled_attention_06_gb300 import inputs

    orc = oracle.default()
    pc, dc = inputs.C3, inputs.C5
    rows = pc.Nq if rows is None else rows
    q, k, v = inputs.prefill_inputs(1, heads, heads, pc.Nq, pc.Nk, pc.d, seed=pc.seed,
                                    k_boost_frac=pc.k_boost_frac)
    q64, k64, v64 = q.double().numpy(), k.double().numpy(), v.double().numpy()
    sel = np.array([[0, h, i] for h in range(heads) for i in range(pc.Nq - rows, pc.Nq)], dtype=np.int64)
    t0 = time.perf_counter()
    orc.attn_fwd_rows(q64, k64, v64, sel, pc.scale, pc.causal, pc.window)
    t_pre = time.perf_counter() - t0
    pre_flops = 4 * pc.d * heads * sum(min(pc.Nk, i + 1) for i in range(pc.Nq - rows, pc.Nq))
    x = inputs.decode_inputs(seqs, dc.Hq, dc.Hkv, dc.d, dc.block_size, seq_lens=[dc.len_hi] * seqs, seed=dc.seed)
    kc, vc = x.k_cache.double().numpy(), x.v_cache.double().numpy()
    t0 = time.perf_counter()
    orc.attn_decode(x.q.double().numpy(), kc, vc, x.block_table.numpy(), x.seq_lens.numpy(), dc.scale)
    t_dec = time.perf_counter() - t0
    dec_bytes = decode_kv_bytes(x.seq_lens.numpy(), dc.Hkv, dc.d)
    desc = (f"prefill: {heads} head(s) x last {rows} query rows of {pc.name}; decode: {seqs} sequence(s) of "
            f"{dc.len_hi} tokens with the decode workload's heads, block size and layout")
    return {"t_pre": t_pre, "pre_flops": pre_flops, "t_dec": t_dec, "dec_bytes": dec_bytes, "desc": desc,
            "cores": orc.num_threads()}


def cpu_baseline_entry(sample):
    return {"value": round(sample["pre_flops"] / sample["t_pre"] / 1e12, 6), "unit": "TFLOP/s",
            "cores": sample["cores"], "kind": "oracle", "sample": sample["desc"],
            "decode_value": round(sample["dec_bytes"] / sample["t_dec"] / 1e9, 4), "decode_unit": "GB/s",
            "seconds": round(sample["t_pre"] + sample["t_dec"], 2)}


def run_reference(args):
    samples = []
    for _ in range(min(args.warmup, 1)):
        oracle_sample(heads=1, rows=128, seqs=1)
    for _ in range(args.steps):
        samples.append(oracle_sample(heads=1, rows=512, seqs=2))
    t_pre = sum(s["t_pre"] for s in samples)
    t_dec = sum(s["t_dec"] for s in samples)
    pre_flops = sum(s["pre_flops"] for s in samples)
    dec_bytes = sum(s["dec_bytes"] for s in samples)
    value = pre_flops / t_pre / 1e12
    from exact_tiled_attention_06_gb300 import inputs
    base = {"value": round(value, 6), "unit": "TFLOP/s", "cores": samples[0]["cores"], "kind": "oracle",
            "sample": samples[0]["desc"]}
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round((t_pre + t_dec) / args.steps * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{inputs.C3.name} + {inputs.C5.name}", "sampled": True},
        "decode": {"value": round(dec_bytes / t_dec / 1e9, 4), "unit": "GB/s"},
        "cpu_baseline": base,
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def summary_of(result):
    """One short entry per timed workload: [value, unit, roofline fraction, DRAM bytes per
    launch (null when no current record)], then the clocks seen."""
    out = {}

    def add(name, block):
        rf = block.get("roofline", {})
        out[name] = [block.get("value"), block.get("unit"), rf.get("frac"), rf.get("traffic")]

    add("prefill C3", result)
    for key, name in (("decode", "decode C5"), ("backward", "backward C3"), ("paged_prefill", "paged prefill C6"),
                      ("blocksparse", "block-sparse C7"), ("fp8_prefill", "FP8 prefill C3"),
                      ("decode_graph", "decode step C8 (graph)")):
        if key in result:
            add(name, result[key])
    for name, block in result.get("prefill_configs", {}).items():
        add("prefill " + name.split("_")[0], block)
        g = block.get("graph_replay")
        if g:
            out["prefill " + name.split("_")[0] + " (graph)"] = [g["value"], block.get("unit"), g["frac"]]
    if "e2e" in result:
        out["e2e"] = [result["e2e"]["value"], result["e2e"]["unit"], result["e2e"].get("decode_value"),
                      result["e2e"].get("decode_unit")]
    c = result.get("clocks") or {}
    out["clocks"] = [c.get("sm_mhz"), c.get("sm_max_mhz"), c.get("reasons"), c.get("samples")]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) leg")
    ap.add_argument("--workload", choices=["both", "prefill", "decode"], default="both",
                    help="profiling aid: run only one half of the step (the JSON line then omits the other)")
    ap.add_argument("--no-backward", action="store_true", help="skip the backward measurement")
    ap.add_argument("--no-paged-prefill", action="store_true", help="skip the chunked paged prefill measurement")
    ap.add_argument("--no-decode-graph", action="store_true",
                    help="skip the many-layer decode step (per-call launches against one CUDA-graph replay)")
    ap.add_argument("--no-blocksparse", action="store_true", help="skip the block-sparse prefill measurement")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 (E4M3) prefill measurement")
    ap.add_argument("--no-other-prefill", action="store_true",
                    help="skip the C1, C2 and C4 prefill measurements")
    ap.add_argument("--min-loop-seconds", type=float, default=0.5,
                    help="each timed loop after the step runs at least this long (and at least --steps calls)")
    ap.add_argument("--only-config", default=None, choices=["C1", "C2", "C4"],
                    help="profiling aid: of the C1 / C2 / C4 prefill loops run only this one")
    ap.add_argument("--no-graph-replay", action="store_true",
                    help="profiling aid: skip the graph-replayed timing of the C1 / C2 / C4 loops")
    ap.add_argument("--details", default=os.path.join(ROOT, "bench_details.json"),
                    help="file for the per-sequence lengths of the paged workloads (kept out of the JSON line)")
    ap.add_argument("--decode-seqs", type=int, default=None,
                    help="profiling aid: fewer decode sequences than the workload's 64")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    # the CPU baseline runs before any GPU work (its pool of threads is OpenMP in the oracle)
    sample = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = oracle_sample()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    result = run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0 and result is not None:
        details = result.pop("_details", None)
        if details is not None and args.details:
            try:
                with open(args.details, "w") as f:
                    json.dump(details, f)
                result["details_file"] = os.path.relpath(args.details, ROOT)
            except OSError:
                pass
        result["cpu_baseline"] = cpu_baseline_entry(sample) if sample else None
        result["summary"] = summary_of(result)  # last key: stays in a record that keeps the line's tail
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
