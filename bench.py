"""Benchmark: one step = the whole hot path on synthetic inputs resident in HBM:

  * prefill  attn_fwd    on the long causal workload  B=1, H=32, N=8192, d=128
                         (1% of K rows x2, seeded), bf16 in / bf16 O + fp32 lse
  * decode   attn_decode on the paged GQA workload     64 sequences, Hq=32, Hkv=8,
                         d=128, 16-token blocks, lengths U[1024, 32768], random table

Prints ONE JSON line (rank 0). ``value`` is prefill TFLOP/s (algorithmic FLOPs:
4 * d per allowed (query, key) pair, i.e. 4 N^2 d per head halved for causal);
``decode`` carries the decode KV-read GB/s. Both inputs exceed the 129 MB L2,
so no flush is needed between steps.

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


# ----------------------------------------------------------------------------- environment
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_06_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the kernel
    sources changed after the counters were taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(kernel)
        if e and e.get("source_hash") == kernel_source_hash():
            return float(e["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        try:
            rows = list(csv.reader(io.StringIO(open(self.path).read())))
            os.unlink(self.path)
        except Exception:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- our arm
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

    # ---- synthetic inputs: pinned host copies (for the end-to-end leg) and HBM-resident copies
    q_h, k_h, v_h = inputs.prefill_config_inputs(pc, seed=pc.seed + rank)
    dx = inputs.decode_config_inputs(dc, seed=dc.seed + rank)
    host = {"q": q_h, "k": k_h, "v": v_h, "dq": dx.q, "kc": dx.k_cache, "vc": dx.v_cache, "bt": dx.block_table,
            "sl": dx.seq_lens}
    host = {n: t.pin_memory() for n, t in host.items()}
    d_in = {n: t.to(dev) for n, t in host.items()}
    o = torch.empty_like(d_in["q"])
    lse = torch.empty((pc.B, pc.Hq, pc.Nq), dtype=torch.float32, device=dev)
    do = torch.empty_like(d_in["dq"])
    dlse = torch.empty((dc.num_seqs, dc.Hq), dtype=torch.float32, device=dev)
    mb = dx.block_table.shape[1]
    ws = torch.empty(eta.attn_decode_workspace_size(dc.num_seqs, dc.Hq, dc.Hkv, dc.d, dc.block_size, mb),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def prefill(ins, out, out_lse):
        eta.attn_fwd(ins["q"], ins["k"], ins["v"], causal=pc.causal, window=pc.window, scale=pc.scale, out=out,
                     lse=out_lse)

    def decode(ins, out, out_lse):
        eta.attn_decode(ins["dq"], ins["kc"], ins["vc"], ins["bt"], ins["sl"], scale=dc.scale, workspace=ws,
                        out=out, lse=out_lse)

    flops = attention_flops(pc.B, pc.Hq, pc.Nq, pc.Nk, pc.d, pc.causal, pc.window)
    kv_bytes = decode_kv_bytes(dx.seq_lens.numpy(), dc.Hkv, dc.d)
    launches_per_step = 1 + 2  # prefill kernel; decode split + combine

    # ---- warm-up
    for _ in range(args.warmup):
        prefill(d_in, o, lse)
        decode(d_in, do, dlse)
    torch.cuda.synchronize()
    err = eta.attn_get_device_error()
    if err != 0:
        raise RuntimeError(f"device error during warm-up: {eta.attn_status_string(err)}")

    # ---- timed region: K steps, events around each kernel on the launching stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        t_start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            prefill(d_in, o, lse)
            ev[i][1].record(stream)
            decode(d_in, do, dlse)
            ev[i][2].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    err = eta.attn_get_device_error()
    if err != 0:
        raise RuntimeError(f"device error in the timed region: {eta.attn_status_string(err)}")
    total_ms = t_start.elapsed_time(t_end)
    pre_ms = np.array([e[0].elapsed_time(e[1]) for e in ev])
    dec_ms = np.array([e[1].elapsed_time(e[2]) for e in ev])

    # ---- end to end through the public API with host buffers (copies inside the timed region)
    h_o = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
    h_lse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    h_do = torch.empty(do.shape, dtype=do.dtype, pin_memory=True)
    h_dlse = torch.empty(dlse.shape, dtype=dlse.dtype, pin_memory=True)
    pre_names, dec_names = ("q", "k", "v"), ("dq", "kc", "vc", "bt", "sl")
    h2d_pre = sum(host[n].numel() * host[n].element_size() for n in pre_names)
    h2d_dec = sum(host[n].numel() * host[n].element_size() for n in dec_names)
    d2h_pre = o.numel() * 2 + lse.numel() * 4
    d2h_dec = do.numel() * 2 + dlse.numel() * 4
    e2e_steps = max(1, min(args.steps, 5))
    e_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(e2e_steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(e2e_steps):
        e_ev[i][0].record(stream)
        for n in pre_names:
            d_in[n].copy_(host[n], non_blocking=True)
        prefill(d_in, o, lse)
        h_o.copy_(o, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)
        e_ev[i][1].record(stream)
        for n in dec_names:
            d_in[n].copy_(host[n], non_blocking=True)
        decode(d_in, do, dlse)
        h_do.copy_(do, non_blocking=True)
        h_dlse.copy_(dlse, non_blocking=True)
        e_ev[i][2].record(stream)
    torch.cuda.synchronize()
    e2e_pre_ms = float(np.mean([e[0].elapsed_time(e[1]) for e in e_ev]))
    e2e_dec_ms = float(np.mean([e[1].elapsed_time(e[2]) for e in e_ev]))

    # ---- max over ranks
    vals = torch.tensor([total_ms, pre_ms.mean(), dec_ms.mean(), e2e_pre_ms, e2e_dec_ms], dtype=torch.float64,
                        device=dev)
    if world > 1:
        dist.all_reduce(vals, op=dist.ReduceOp.MAX)
    total_ms, pre_mean, dec_mean, e2e_pre_ms, e2e_dec_ms = (float(x) for x in vals.cpu())
    if rank != 0:
        return None

    peaks, peak_kind = load_peaks()
    step_ms = total_ms / args.steps
    # whole-job prefill throughput: all ranks' FLOPs over the max-over-ranks prefill time
    pre_tflops = world * flops / (pre_mean * 1e-3) / 1e12
    dec_gbs = world * kv_bytes / (dec_mean * 1e-3) / 1e9
    achieved_pre = flops / (pre_mean * 1e-3) / 1e12  # one launch, one GPU
    achieved_dec = kv_bytes / (dec_mean * 1e-3) / 1e9
    result = {
        "metric": METRIC,
        "value": round(pre_tflops, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{pc.name} + {dc.name}",
            "prefill": {"B": pc.B, "Hq": pc.Hq, "Hkv": pc.Hkv, "Nq": pc.Nq, "Nk": pc.Nk, "d": pc.d,
                        "causal": pc.causal, "window": pc.window, "k_boost_frac": pc.k_boost_frac,
                        "flops_per_launch": flops},
            "decode": {"num_seqs": dc.num_seqs, "Hq": dc.Hq, "Hkv": dc.Hkv, "d": dc.d,
                       "block_size": dc.block_size, "len_range": [dc.len_lo, dc.len_hi],
                       "sum_seq_len": int(dx.seq_lens.sum()), "kv_bytes_per_launch": kv_bytes},
            "l2": "inputs larger than L2 (prefill Q/K/V 192 MiB, decode KV ~4.4 GB); no flush",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "kernel": "attn_fwd_sm103<128>",
            "bound": "tensor",
            "achieved": round(achieved_pre, 2),
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": round(achieved_pre / peaks["bf16_tflops"], 4),
            "peak_kind": f"{peak_kind} bf16 dense burst",
            "frac_of_sustained": round(achieved_pre / peaks["bf16_tflops_sustained"], 4),
            "traffic": load_traffic("attn_fwd_sm103"),
            "ms_per_launch": round(pre_mean, 4),
            "ms_p10_p90": [round(float(np.percentile(pre_ms, 10)), 4), round(float(np.percentile(pre_ms, 90)), 4)],
        },
        "decode": {
            "value": round(dec_gbs, 2),
            "unit": "GB/s",
            "roofline": {
                "kernel": "attn_decode_split_sm103<128> + attn_decode_combine_sm103<128>",
                "bound": "hbm",
                "achieved": round(achieved_dec, 2),
                "peak": peaks["hbm_gbs"],
                "unit": "GB/s",
                "frac": round(achieved_dec / peaks["hbm_gbs"], 4),
                "peak_kind": f"{peak_kind} HBM copy",
                "traffic": load_traffic("attn_decode_split_sm103"),
                "ms_per_launch": round(dec_mean, 4),
                "ms_p10_p90": [round(float(np.percentile(dec_ms, 10)), 4),
                               round(float(np.percentile(dec_ms, 90)), 4)],
            },
            "workspace_bytes": int(ws.numel()),
        },
        "e2e": {
            "value": round(world * flops / (e2e_pre_ms * 1e-3) / 1e12, 3),
            "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d_pre + h2d_dec,
            "d2h_bytes_per_step": d2h_pre + d2h_dec,
            "decode_value": round(world * kv_bytes / (e2e_dec_ms * 1e-3) / 1e9, 2),
            "decode_unit": "GB/s",
            "ms_per_step": round(e2e_pre_ms + e2e_dec_ms, 3),
            "steps": e2e_steps,
        },
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    return result


# ----------------------------------------------------------------------------- oracle timing
def oracle_sample(heads=4, rows=None, seqs=2):
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
        result["cpu_baseline"] = cpu_baseline_entry(sample) if sample else None
        print(json.dumps(result), flush=True)


if __name__ == "__main__":
    main()
