"""Benchmark of the KDA hot path on GB300.

Headline (one JSON line on rank 0): packed-decode state-bytes GB/s on the serving
decode workload (128 sequences x 32 heads, K = V = 128, fp32 state pool of 512 slots,
state indices = column 0 of an int32 [128, 8] block table), lower_bound = -5.0.
A step is one kda_packed_decode call over that batch. Each step addresses one of four
disjoint sets of 128 slots in turn, so the 256 MiB a step reads were last touched
four steps (1 GiB of state traffic) earlier: L2 (129 MB) cannot serve them.

The same line carries the other rows of the path measured on their own workloads
(chunked prefill tokens/s, spec-verify, mixed batch), the decode kernel's roofline
against the measured HBM copy bandwidth, the fp64 oracle's throughput on the host
cores (cpu_baseline), an end-to-end number through the public binding with host
buffers, and the SM clocks seen during the timed region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this path has) on the
same workload and metric.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

NOMINAL_HBM_GBS = 8000.0
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PREFILL_ALG_FLOPS_PER_CHUNK = None  # computed from the lengths below


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK, source="fallback")


def prefill_alg_flops(lengths, H, K, V, C=64):
    """Algorithmic flops of the chunked form: per (chunk of c rows, head)
    6cKV + c^2 (3K + 2V) + c^3 / 3 (triangular products counted at half)."""
    tot = 0
    for L in lengths:
        full, rem = divmod(int(L), C)
        for c in [C] * full + ([rem] if rem else []):
            tot += 6 * c * K * V + c * c * (3 * K + 2 * V) + c ** 3 / 3
    return tot * H


def prefill_min_bytes(w):
    """q, k, v, raw_g in bf16, o out bf16, beta bf16, and each sequence's state R+W."""
    N, H, K, V = w.N, w.H, w.K, w.V
    per_tok = 2 * (2 * H * K + H * V) + 2 * H * K + 2 * H + 2 * H * V
    return N * per_tok + w.num_entries * 2 * 4 * H * K * V


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        if torch.cuda.is_available():
            torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """Largest value over the ranks (the timed region's duration of the slowest rank)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_units(total, world, rank):
    """Units [lo, hi) of `total` independent units owned by `rank` (contiguous blocks)."""
    per, extra = divmod(total, world)
    lo = rank * per + min(rank, extra)
    return lo, lo + per + (1 if rank < extra else 0)


def source_sha(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "linear_attention_state_recurrent_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, sha):
    """dram bytes per launch from the committed ncu summary, if it was taken on this source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d.get(kernel_key)
        if ent and ent.get("source_sha") == sha:
            return float(ent["dram_bytes_per_launch"])
    except (OSError, ValueError):
        pass
    return None


# ---------------------------------------------------------------------------
# reference arm: the fp64 oracle on the host cores
# ---------------------------------------------------------------------------

def decode_config(world):
    """The headline workload's config (both arms report the same)."""
    return {"workload": "serving decode: 128 seqs x H=32 heads, K=V=128, fp32 pool "
                        "512 slots (1 GiB), state_indices = column 0 of an int32 "
                        "[128,8] block table (stride 8), lower_bound=-5.0",
            "l2": "inputs larger than L2: steps rotate over 4 disjoint 128-slot "
                  "sets (256 MiB read per step, 1 GiB between reuses)",
            "parallelism": "1 GPU" if world == 1 else
                           f"heads split over {world} ranks (tensor-parallel layout, each rank its own pool of "
                           "its heads, no collective on the data path)"}


# sequences of the serving decode that one reference step runs (a bounded sample: the
# oracle takes ~0.1-0.4 s for all 128, so a --steps count meant for the GPU arm still
# finishes in a few minutes)
REFERENCE_SAMPLE_SEQS = 2


def run_reference(args, world, rank):
    if rank != 0:
        return
    from linear_attention_state_recurrent_gb300 import workloads as wl
    from oracle import kda_oracle as ko
    w = wl.serving_decode(-5.0)
    sets = wl.serving_decode_index_sets(w)
    cores = ko.max_threads()
    n = REFERENCE_SAMPLE_SEQS
    bounds_all = w.seq_bounds()

    def step(i):
        # sequences n*i .. n*i + n - 1 (mod 128), slots from the rotating sets
        first = (n * i) % w.num_entries
        idx = [(first + k) % w.num_entries for k in range(n)]
        ko.run(w, bounds=[bounds_all[e] for e in idx], slots=sets[i % 4][idx])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    sample_bytes = 2 * 4 * w.K * w.V * w.H * n
    gbs = sample_bytes * args.steps / dt / 1e9
    sample = (f"{n} of the 128 sequences per step (x 32 heads, K=V=128: {sample_bytes} state "
              f"bytes read + written), rotating through all 128; {args.steps} steps")
    line = {"impl": "reference", "metric": "KDA decode state-bytes GB/s", "value": gbs,
            "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": decode_config(world),
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline_decode(w, sets, budget_s=10.0, budget_1t_s=5.0):
    """The fp64 oracle on the host: all cores (OpenMP over (sequence, head)) on full
    serving-decode calls, and one thread on a bounded sample of them."""
    from oracle import kda_oracle as ko
    cores = ko.max_threads()
    ko.run(w, slots=sets[0])
    n, t0 = 0, time.perf_counter()
    while True:
        ko.run(w, slots=sets[n % 4])
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s:
            break
    # single thread: 8 of the 128 sequences per call, rotating through all of them
    bounds_all = w.seq_bounds()
    per = 8
    m, t1 = 0, time.perf_counter()
    while True:
        first = (per * m) % w.num_entries
        idx = [(first + k) % w.num_entries for k in range(per)]
        ko.run(w, bounds=[bounds_all[e] for e in idx], slots=sets[m % 4][idx], nthreads=1)
        m += 1
        dt1 = time.perf_counter() - t1
        if dt1 >= budget_1t_s:
            break
    one = 2 * 4 * w.K * w.V * w.H * per * m / dt1 / 1e9
    return {"value": w.state_bytes_per_call() * n / dt / 1e9, "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{n} full serving-decode calls (128 seqs x 32 heads) in {dt:.1f} s, fp64, OpenMP over (seq, head)",
            "single_thread": {"value": one, "unit": "GB/s", "cores": 1,
                              "sample": f"{m} calls of {per} of the 128 sequences (x 32 heads) in {dt1:.1f} s, one thread"}}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--workload", choices=["decode", "prefill", "spec", "spec_ckpt", "fused_decode", "fused_spec", "mixed"], default="decode",
                    help="decode (default) is the headline line; the others time one row alone")
    ap.add_argument("--prefill-lengths", default=None,
                    help="comma-separated sequence lengths for --workload prefill (H=32, K=V=128; "
                         "default: the seed-1 lengths, 33,494 tokens), e.g. a smaller case for profiling")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    from linear_attention_state_recurrent_gb300 import kda
    from linear_attention_state_recurrent_gb300 import workloads as wl

    dev = f"cuda:{local}"
    stream = torch.cuda.current_stream()
    pk = peaks()
    if args.workload != "decode":
        run_row(args, torch, kda, wl, dev, stream, pk, world, rank, local)
        return

    # ---- headline: serving decode ----
    # Under torchrun the heads are split across the ranks as tensor parallelism does: rank
    # r holds heads shard_units(H, world, r) of every slot (its own pool) and runs the same
    # call on them; nothing crosses ranks on the data path.
    w_full = wl.serving_decode(-5.0)
    w = w_full
    if world > 1:
        lo, hi = shard_units(w_full.H, world, rank)
        w = wl.shard_heads(w_full, lo, hi)
    dw = wl.DeviceWorkload(w, dev)
    sets = wl.serving_decode_index_sets(w)
    idx_dev = [torch.from_numpy(s).to(dev) for s in sets]
    out = torch.empty(w.N, w.H * w.V, dtype=torch.bfloat16, device=dev)
    hd = kda.make_heads(dw.A_log, dw.dt_bias, w.lower_bound, w.K, w.V, w.scale, w.eps)
    states = [kda.make_state(dw.pool_view(), ix) for ix in idx_dev]
    lib = kda.lib
    s_ptr = ctypes.c_void_p(stream.cuda_stream)
    call_args = [(ctypes.c_void_p(dw.mixed_qkv.data_ptr()), dw.mixed_qkv.stride(0),
                  ctypes.c_void_p(dw.raw_g.data_ptr()), dw.raw_g.stride(0),
                  ctypes.c_void_p(dw.raw_beta.data_ptr()), dw.raw_beta.stride(0), w.N,
                  ctypes.byref(hd), ctypes.byref(st), ctypes.c_void_p(out.data_ptr()),
                  out.stride(0), None, s_ptr) for st in states]

    def step(i):
        s = lib.kda_packed_decode(*call_args[i & 3])
        if s:
            raise RuntimeError(kda.last_error())

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms_total = max_over_ranks(ev0.elapsed_time(ev1), world)
    ms_step = ms_total / args.steps
    state_bytes = w.state_bytes_per_call()          # this rank's heads
    total_bytes = w_full.state_bytes_per_call()     # all ranks together
    value = total_bytes * args.steps / (ms_total * 1e-3) / 1e9
    achieved = state_bytes / (ms_step * 1e-3) / 1e9
    sha = source_sha("kda_recurrent.cu", "kda_common.cuh", "kda_pdl.cuh")
    traffic = ncu_traffic("decode_kernel<128,128> serving_decode", sha)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                "peak_source": f"{pk['source']} HBM copy bandwidth (of {pk['source']})",
                "frac_of_nominal_8TBs": achieved / NOMINAL_HBM_GBS,
                "algorithmic_bytes_per_launch": state_bytes,
                "kernel": "kda::decode_kernel<128,128>"}

    # ---- end to end through the public binding with host buffers ----
    e2e = None
    if rank == 0 or world > 1:
        # A step's inputs (mixed_qkv, raw_g, raw_beta, state indices) sit in one pinned host
        # buffer and travel in one copy into one device buffer that the call reads through
        # views (segments 256-byte aligned); one buffer per rotated index set.
        parts = [dw.mixed_qkv, dw.raw_g, dw.raw_beta, idx_dev[0]]
        offs, tot = [], 0
        for t in parts:
            offs.append(tot)
            tot += (t.numel() * t.element_size() + 255) // 256 * 256
        d_all = torch.empty(tot, dtype=torch.uint8, device=dev)

        def seg(buf, k):
            t = parts[k]
            n = t.numel() * t.element_size()
            return buf[offs[k]:offs[k] + n].view(t.dtype).view(t.shape)
        h_all = []
        for sidx in sets:
            hb = torch.empty(tot, dtype=torch.uint8).pin_memory()
            for k, t in enumerate(parts[:3]):
                seg(hb, k).copy_(t.cpu())
            seg(hb, 3).copy_(torch.from_numpy(sidx))
            h_all.append(hb)
        d_qkv, d_g, d_b, d_idx = (seg(d_all, k) for k in range(4))
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        e2e_steps = min(args.steps, 2000)
        h2d = sum(t.numel() * t.element_size() for t in parts)
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step(i):   # one step at a time: copy in, call, copy out, wait
            d_all.copy_(h_all[i & 3], non_blocking=True)
            o, _ = kda.kda_packed_decode(d_qkv, d_g, d_b, dw.A_log, dw.dt_bias,
                                         w.lower_bound, dw.pool_view(), d_idx, scale=w.scale,
                                         l2_eps=w.eps, out=out)
            h_out.copy_(o, non_blocking=True)
            stream.synchronize()

        # Pipelined steps, as a serving loop with asynchronous scheduling runs them: step i's
        # input copy (a copy stream, into one of two device buffers) overlaps step i-1's call;
        # its output is copied to the host on a third stream once its call is done (so the
        # next call follows this one directly), and the host waits for step i-1's output
        # right after issuing step i. Every step's copies are inside the timed region.
        d_in = [d_all, torch.empty(tot, dtype=torch.uint8, device=dev)]
        d_views = [[seg(d, k) for k in range(4)] for d in d_in]
        d_out = [out, torch.empty_like(out)]
        h_outs = [h_out, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
        in_stream, out_stream = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]     # step's input copy done
        ev_call = [torch.cuda.Event() for _ in range(2)]   # step's call done
        ev_done = [torch.cuda.Event() for _ in range(2)]   # step's output copy done (buffers b free)

        def e2e_pipelined_step(i):
            b = i & 1
            with torch.cuda.stream(in_stream):
                in_stream.wait_event(ev_done[b])   # step i-2 has finished with buffers b
                d_in[b].copy_(h_all[i & 3], non_blocking=True)
                ev_in[b].record(in_stream)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_done[b])
            vq, vg, vb, vi = d_views[b]
            o, _ = kda.kda_packed_decode(vq, vg, vb, dw.A_log, dw.dt_bias, w.lower_bound,
                                         dw.pool_view(), vi, scale=w.scale, l2_eps=w.eps,
                                         out=d_out[b])
            ev_call[b].record(stream)
            with torch.cuda.stream(out_stream):
                out_stream.wait_event(ev_call[b])
                h_outs[b].copy_(o, non_blocking=True)
                ev_done[b].record(out_stream)
            if i > 0:
                ev_done[b ^ 1].synchronize()   # the host takes step i-1's result

        def timed(fn):
            for i in range(5):
                fn(i)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for i in range(e2e_steps):
                fn(i)
            torch.cuda.synchronize()
            return max_over_ranks(time.perf_counter() - t0, world)

        dt_sync = timed(e2e_step)
        dt = timed(e2e_pipelined_step)
        e2e = {"value": total_bytes * e2e_steps / dt / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": dt / e2e_steps * 1e3, "steps": e2e_steps,
               "api": "kda.kda_packed_decode, pipelined: step i's pinned host -> device input copy "
                      "(copy stream, two device buffers) overlaps step i-1's call; each step's output "
                      "is copied device -> host on a third stream after its call, and the host waits "
                      "for step i-1's output after issuing step i",
               "one_step_at_a_time": {"value": total_bytes * e2e_steps / dt_sync / 1e9, "unit": "GB/s",
                                      "ms_per_step": dt_sync / e2e_steps * 1e3,
                                      "api": "copy in, call, copy out, stream sync, each step"}}

    # ---- other rows (rank 0 only) ----
    secondary = {}
    if rank == 0 and not args.no_secondary:
        secondary = measure_secondary(torch, kda, wl, dev, stream, pk, local)

    del dw, states, call_args
    torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_decode(w, sets)

    if rank == 0:
        line = {"metric": "KDA decode state-bytes GB/s", "value": value, "unit": "GB/s",
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": ms_step, "higher_is_better": True,
                "scaling": "strong" if world > 1 else "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": decode_config(world),
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": args.steps, "clocks": clk.summary()}
        line.update(secondary)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_row(args, torch, kda, wl, dev, stream, pk, world, rank, local):
    """One non-headline row alone: chunked prefill, spec-verify or mixed batch, timed over
    --steps calls after --warmup calls (the same calls the secondary fields time)."""
    if args.workload == "prefill":
        if args.prefill_lengths:
            w = wl.varlen_case([int(x) for x in args.prefill_lengths.split(",")], 32, 128, 128, seed=1,
                               name="prefill " + args.prefill_lengths)
        else:
            w = wl.chunked_prefill(None)
        metric, unit = "chunk-prefill tokens/s", "tokens/s"
    elif args.workload == "mixed":
        w = wl.mixed_batch()
        metric, unit = "mixed-batch tokens/s", "tokens/s"
    elif args.workload == "spec_ckpt":
        w = wl.spec_checkpoints()
        metric, unit = "spec-verify-checkpoints state-bytes GB/s", "GB/s"
    elif args.workload == "fused_decode":
        w = wl.with_layer_tail(wl.serving_decode(-5.0), seed=99)
        metric, unit = "fused-decode state-bytes GB/s", "GB/s"
    elif args.workload == "fused_spec":
        w = wl.with_layer_tail(wl.spec_verify(), seed=99)
        metric, unit = "fused-spec-verify state-bytes GB/s", "GB/s"
    else:
        w = wl.spec_verify()
        metric, unit = "spec-verify state-bytes GB/s", "GB/s"
    dw = wl.DeviceWorkload(w, dev)
    out = torch.empty(w.N, w.H * w.V, dtype=torch.bfloat16, device=dev)
    if args.workload in ("spec", "spec_ckpt", "fused_decode", "fused_spec"):
        ms = time_spec_graph(torch, kda, w, dw, out, calls=20, replays=max(1, args.steps // 20))
        value = spec_state_bytes(w) * world / (ms * 1e-3) / 1e9
        line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": w.name, "tokens": w.N, "H": w.H, "K": w.K, "V": w.V,
                           "timing": "CUDA graph replays of 20 pre-marshalled C-ABI calls"},
                "frac_hbm": value / pk["hbm_gbs"], "gpu_launches": 20 * max(1, args.steps // 20)}
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    for _ in range(args.warmup):
        wl.run_gpu(dw, kda, out=out)
    torch.cuda.synchronize()
    barrier(world)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            wl.run_gpu(dw, kda, out=out)
        ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(ev0.elapsed_time(ev1), world) / args.steps
    if unit == "tokens/s":
        value = w.N * world / (ms * 1e-3)
    else:
        value = w.state_bytes_per_call() * world / (ms * 1e-3) / 1e9
    line = {"metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "tokens": w.N, "H": w.H, "K": w.K, "V": w.V},
            "clocks": clk.summary(), "gpu_launches": args.steps * {"prefill": 3, "mixed": 4}.get(args.workload, 1)}
    if args.workload == "prefill":
        flops = prefill_alg_flops([b - a for a, b in w.seq_bounds()], w.H, w.K, w.V)
        line["tflops_algorithmic"] = flops / (ms * 1e-3) / 1e12
        line["frac_bf16_peak"] = line["tflops_algorithmic"] / pk["bf16_tflops"]
        line["frac_hbm_min_bytes"] = prefill_min_bytes(w) / (ms * 1e-3) / 1e9 / pk["hbm_gbs"]
    if rank == 0:
        print(json.dumps(line), flush=True)


def spec_call_args(kda, w, dw, out, stream_handle, indices=None):
    """Pre-marshalled C-ABI arguments of one kda_spec_verify call (kda_spec_verify_checkpoints
    for a checkpoint workload, kda_fused_decode / kda_fused_spec_verify for a fused one),
    kept alive with the structs they point to. `indices` (a device int32 tensor) replaces
    the workload's state-index view. Returns (function, args, keep-alive)."""
    hd = kda.make_heads(dw.A_log, dw.dt_bias, w.lower_bound, w.K, w.V, w.scale, w.eps)
    st = kda.make_state(dw.pool_view(), dw.indices_view() if indices is None else indices, w.null_slot)
    head = (ctypes.c_void_p(dw.mixed_qkv.data_ptr()), dw.mixed_qkv.stride(0),
            ctypes.c_void_p(dw.raw_g.data_ptr()), dw.raw_g.stride(0),
            ctypes.c_void_p(dw.raw_beta.data_ptr()), dw.raw_beta.stride(0),
            w.num_entries, w.tokens_per_req)
    tail = (ctypes.byref(hd), ctypes.byref(st), ctypes.c_void_p(out.data_ptr()), out.stride(0),
            None, ctypes.c_void_p(stream_handle))
    if w.fused:
        cv = None if w.conv_weight is None else kda.make_conv(dw.conv_weight, dw.conv_bias, dw.conv_pool)
        nm = None if w.norm_weight is None else kda.make_norm(dw.out_gate, dw.norm_weight, w.norm_eps)
        ext = (None if cv is None else ctypes.byref(cv), None if nm is None else ctypes.byref(nm))
        tail = tail[:2] + ext + tail[2:]
        if w.kind == "decode":
            return kda.lib.kda_fused_decode, head[:7] + tail, (hd, st, cv, nm)
        return kda.lib.kda_fused_spec_verify, head + tail, (hd, st, cv, nm)
    if w.kind == "spec_ckpt":
        acc = None if dw.num_accepted is None else ctypes.c_void_p(dw.num_accepted.data_ptr())
        return kda.lib.kda_spec_verify_checkpoints, head + (acc,) + tail, (hd, st)
    return kda.lib.kda_spec_verify, head + tail, (hd, st)


def spec_index_sets(w, count):
    """`count` disjoint state-index arrays for a spec-verify workload: every real request
    gets fresh slots from 1 .. num_slots - 1 in each set, padding requests keep the null
    slot. Rotating through them between calls keeps a call's state out of L2."""
    import numpy as np
    idx = w.indices()
    real = np.nonzero(idx != w.null_slot)[0]
    avail = np.array([s for s in range(w.num_slots) if s != w.null_slot], dtype=np.int32)
    rng = np.random.default_rng(777)
    rng.shuffle(avail)
    assert count * len(real) <= len(avail)
    sets = []
    for i in range(count):
        a = np.full(w.num_entries, w.null_slot, dtype=np.int32)
        a[real] = avail[i * len(real):(i + 1) * len(real)]
        sets.append(a)
    return sets


def time_spec_graph(torch, kda, w, dw, out, calls=20, replays=50, index_sets=None):
    """Spec-verify calls are a few microseconds of GPU time, far below the host cost of a
    Python call, so they are timed as replays of a CUDA graph of `calls` launches. With
    `index_sets` (device int32 tensors) consecutive calls rotate through them."""
    cap = torch.cuda.Stream()
    marsh = [spec_call_args(kda, w, dw, out, cap.cuda_stream, ix) for ix in (index_sets or [None])]
    keep = marsh
    with torch.cuda.stream(cap):
        for _ in range(3):
            for fn, args, _k in marsh:
                if fn(*args):
                    raise RuntimeError(kda.last_error())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for i in range(calls):
            fn, args, _k = marsh[i % len(marsh)]
            fn(*args)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(replays):
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    del keep
    return ev0.elapsed_time(ev1) / (calls * replays)


def spec_state_bytes(w):
    """State bytes of one spec-verify call: each real request's tile read + written once,
    each padding request's (null-slot) tile read only. With per-token checkpoints a real
    request writes its tile once per token."""
    null = sum(1 for s in w.indices() if s == w.null_slot)
    real = w.num_entries - null
    writes = w.tokens_per_req if w.kind == "spec_ckpt" else 1
    total = (real * (1 + writes) + null) * 4 * w.K * w.V * w.H
    if w.conv_weight is not None:   # the conv state: W-1 bf16 inputs per channel, read + written
        C = 2 * w.H * w.K + w.H * w.V
        total += (real * 2 + null) * (w.conv_width - 1) * C * 2
    return total


def spec_leg(torch, kda, w, dw, out, pk, desc, rotate_sets):
    """A spec-verify-shaped leg: L2-cold (rotating disjoint slot sets across the graph's
    calls, when the workload leaves room for them) and warm (the same slots every call)."""
    sbytes = spec_state_bytes(w)
    res = {"workload": desc}
    if rotate_sets:
        sets = [torch.from_numpy(a).to(dw.mixed_qkv.device) for a in spec_index_sets(w, rotate_sets)]
        ms = time_spec_graph(torch, kda, w, dw, out, index_sets=sets)
        dw.reset_pool()
        res.update({"us_per_call": ms * 1e3, "state_gbs": sbytes / (ms * 1e-3) / 1e9,
                    "frac_hbm": sbytes / (ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                    "timing": f"L2-cold: CUDA graph of 20 calls rotating over {rotate_sets} disjoint slot sets "
                              f"({rotate_sets - 1} calls' state, {(rotate_sets - 1) * sbytes / 1e6:.0f} MB, "
                              "between reuses of a slot), 50 replays"})
    ms_w = time_spec_graph(torch, kda, w, dw, out)
    warm = {"us_per_call": ms_w * 1e3, "state_gbs": sbytes / (ms_w * 1e-3) / 1e9,
            "timing": "L2-warm: CUDA graph of 20 calls on the same slots, 50 replays"}
    if rotate_sets:
        res["warm"] = warm
    else:
        res.update(warm)
        res["frac_hbm"] = warm["state_gbs"] / pk["hbm_gbs"]
    return res


def time_calls_clocked(torch, fn, stream, n, warmup, local):
    """Mean ms per call of `n` calls after `warmup`, CUDA events on `stream`, SM clocks
    sampled during the timed region."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        ev0.record(stream)
        for _ in range(n):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / n, clk.summary()


def prefill_leg(torch, kda, wl, w, dev, stream, pk, lower_bound, local, calls=20):
    dw = wl.DeviceWorkload(w, dev)
    out = torch.empty(w.N, w.H * w.V, dtype=torch.bfloat16, device=dev)
    cu_h = torch.from_numpy(w.cu_seqlens)
    nb = kda.kda_chunk_prefill_workspace_bytes(cu_h, w.H, w.K, w.V)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)

    def pf():
        kda.kda_chunk_prefill(dw.mixed_qkv, dw.raw_g, dw.raw_beta, dw.A_log, dw.dt_bias, lower_bound,
                              dw.pool_view(), dw.indices_view(), dw.cu, cu_seqlens_host=cu_h,
                              scale=w.scale, out=out, workspace=ws)
    ms, clocks = time_calls_clocked(torch, pf, stream, calls, 3, local)
    flops = prefill_alg_flops([b - a for a, b in w.seq_bounds()], w.H, w.K, w.V)
    mb = prefill_min_bytes(w)
    sha = source_sha("kda_chunk.cu", "kda_common.cuh", "kda_tc.cuh", "kda_f32x2.cuh", "kda_pdl.cuh")
    traffic = ncu_traffic("prefill (prep_kernel + chain_kernel) chunked_prefill", sha) \
        if (w.K, w.V) == (128, 128) else None
    achieved = mb / (ms * 1e-3) / 1e9
    res = {"metric": "chunk-prefill tokens/s", "value": w.N / (ms * 1e-3), "unit": "tokens/s",
           "ms_per_call": ms, "calls": calls,
           "workload": f"8 seqs (seed-1 lengths, 33,494 tokens), H=32, K={w.K}, V={w.V}, chunk 64, "
                       f"lower_bound={lower_bound}",
           "tflops_algorithmic": flops / (ms * 1e-3) / 1e12,
           "frac_bf16_peak": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"],
           "hbm_gbs_min_bytes": achieved, "frac_hbm": achieved / pk["hbm_gbs"],
           "flop_count": "6cKV + c^2(3K+2V) + c^3/3 per (chunk of c rows, head)",
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                        "peak_source": f"{pk['source']} HBM copy bandwidth (of {pk['source']})",
                        "algorithmic_bytes_per_call": mb,
                        "kernels": "kda::chunk::prep_kernel (one CTA per (chunk, head)) then kda::chunk::chain_kernel",
                        "tensor_frac": flops / (ms * 1e-3) / 1e12 / pk["bf16_tflops"]},
           "clocks": clocks}
    del dw, ws, out
    return res


def measure_secondary(torch, kda, wl, dev, stream, pk, local=0):
    res = {}
    out = torch.empty(128, 32 * 128, dtype=torch.bfloat16, device=dev)
    # spec verify: 16 requests x 8 tokens, L2-cold over 8 disjoint slot sets
    w = wl.spec_verify()
    dw = wl.DeviceWorkload(w, dev)
    res["spec_verify"] = spec_leg(torch, kda, w, dw, out, pk,
                                  "16 requests x 8 tokens, H=32, K=V=128, 2 padding requests on the null slot", 8)
    del dw
    # spec verify with per-token checkpoints: 16 requests x 8 tokens, 8 writes per request
    # (264 MB of state per call: no call is served from L2)
    w = wl.spec_checkpoints()
    dw = wl.DeviceWorkload(w, dev)
    res["spec_verify_checkpoints"] = spec_leg(
        torch, kda, w, dw, out, pk,
        "16 requests x 8 tokens, H=32, K=V=128, state stored after every token (block-table row of 8 slots), "
        "2 padding requests on the null slot", 0)
    del dw
    # fused layer tail (conv W=4 -> recurrence -> gated RMSNorm): serving decode, spec 16x8
    for key, base, desc, rot in (
            ("fused_decode", wl.serving_decode(-5.0),
             "128 seqs, H=32, K=V=128, conv width 4, gated RMSNorm, index stride 8", 0),
            ("fused_spec_verify", wl.spec_verify(),
             "16 requests x 8 tokens, H=32, K=V=128, conv width 4, gated RMSNorm, 2 padding", 8)):
        w = wl.with_layer_tail(base, seed=99)
        dw = wl.DeviceWorkload(w, dev)
        fo = torch.empty(w.N, w.H * w.V, dtype=torch.bfloat16, device=dev)
        r = spec_leg(torch, kda, w, dw, fo, pk, desc, rot)
        r["bytes"] = "KDA state and conv state, read + written (null slot read only)"
        res[key] = r
        del dw, fo
    # chunked prefill: seed-1 lengths, 33,494 tokens, both gate forms
    w = wl.chunked_prefill(None)
    res["chunk_prefill"] = prefill_leg(torch, kda, wl, w, dev, stream, pk, None, local)
    res["chunk_prefill_lower_bound"] = prefill_leg(torch, kda, wl, wl.chunked_prefill(-5.0), dev, stream, pk,
                                                   -5.0, local)
    # the same lengths with K = V = 64 heads (the tensor-core path on half-filled tiles)
    w64 = wl.varlen_case(wl.PREFILL_LENGTHS_SEED1, 32, 64, 64, seed=1, num_slots=16, name="chunked_prefill_k64")
    res["chunk_prefill_k64"] = prefill_leg(torch, kda, wl, w64, dev, stream, pk, None, local)
    res["mixed_batch"] = mixed_leg(torch, kda, wl, dev, stream, pk, local)
    return res


def mixed_leg(torch, kda, wl, dev, stream, pk, local, calls=20):
    """96 decodes + 4 x 4096 prefill tokens through kda_mixed_batch: `calls` calls after 3
    warm-up calls, CUDA events, clocks sampled."""
    w = wl.mixed_batch()
    dw = wl.DeviceWorkload(w, dev)
    out = torch.empty(w.N, w.H * w.V, dtype=torch.bfloat16, device=dev)
    cu_h = torch.from_numpy(w.cu_seqlens)
    nb = kda.kda_chunk_prefill_workspace_bytes(cu_h[w.num_decodes:], w.H, w.K, w.V)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)

    def mb_call():
        kda.kda_mixed_batch(dw.mixed_qkv, dw.raw_g, dw.raw_beta, dw.A_log, dw.dt_bias, None,
                            dw.pool_view(), dw.indices_view(), dw.cu, w.num_decodes,
                            cu_seqlens_host=cu_h, scale=w.scale, out=out, workspace=ws)
    ms, clocks = time_calls_clocked(torch, mb_call, stream, calls, 3, local)
    del dw, ws
    return {"workload": "96 decodes + 4 x 4096 prefill tokens, H=32, K=V=128, index stride 4",
            "tokens_per_s": w.N / (ms * 1e-3), "ms_per_call": ms, "calls": calls,
            "algorithmic_bytes": 1095505920,
            "hbm_gbs": 1095505920 / (ms * 1e-3) / 1e9,
            "frac_hbm": 1095505920 / (ms * 1e-3) / 1e9 / pk["hbm_gbs"], "clocks": clocks}


if __name__ == "__main__":
    main()
