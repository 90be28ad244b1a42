#!/usr/bin/env python3
"""Decode-attention benchmark of the FastOCR path (and R-SWA) on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one decode step through every layer of the workload (focal layers:
full attention + image scores + top-k; other layers: gather attention over
prompt + selected image tokens + generated tokens, with Cross-Step Fixation
Reuse), captured once in a CUDA graph and replayed. Inputs are synthetic and
seeded (synth module) and resident in HBM. L2 is flushed (512 MB memset,
untimed) before every timed step. Prints one JSON line.

--impl reference times the CPU oracle (fp64 NumPy, one thread) on a bounded
sample of the same workload instead -- the deliberately slow baseline.
Under torchrun (N > 1) every rank runs an independent replica (its own
sequences, seed + rank); value = all ranks' steps / max-over-ranks time.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attention steps/s and µs/step at tau=0.05; achieved HBM GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0
FLUSH_BYTES = 512 << 20
CSRC = os.path.join(ROOT, "dynamic_sparse_kv_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.md")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="qwen7b_b1")
    ap.add_argument("--tau", type=float, default=None)
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                    help="override a workload field, e.g. --set batch=8 (profiling runs)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-compare", action="store_true", help="skip the dense / tau=1 arms")
    ap.add_argument("--rswa-ring", action="store_true",
                    help="R-SWA: keep only prefix + window pages per sequence (ring block table)")
    ap.add_argument("--oracle-leg", default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


# ------------------------------------------------------------------ distributed

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(x: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity when world == 1)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ helpers

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_digest() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (line: `traffic <kernel> <workload> <bytes> <digest>`)."""
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.strip().strip("`").split()
                if len(parts) == 5 and parts[0] == "traffic" and parts[1] == kernel \
                        and parts[2] == workload:
                    return float(parts[3]) if parts[4] == source_digest() else None
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle leg

def oracle_leg(spec: str):
    """Run in a child process with one BLAS thread: time the oracle's steady
    decode steps on a bounded sample of the workload. Prints a JSON dict."""
    import numpy as np

    import oracle.schedule as S
    import synth
    name, tau, budget = spec.split(":")
    wl = synth.workload(name)
    if float(tau) > 0:
        wl = wl.with_(tau=float(tau))
    # the sample: every layer of sequence 0, decode steps after warm-up, until
    # the time budget is used (at least 2 steps)
    wl1 = wl.with_(batch=1)
    if wl1.mode == "rswa":   # the late steps the GPU bench times (window full)
        t_first, max_steps = max(0, wl1.steps - 64), wl1.steps
    else:
        t_first, max_steps = 0, min(wl1.steps, wl1.warmup + 64)
    case = synth.make_case(wl1, device="cpu", step0=t_first, n_steps=max_steps - t_first)
    kvs = {}

    def kv(l, b):
        if l not in kvs:
            K, V = case.logical_kv(l, 0, wl1.max_tokens)
            kvs[l] = (K.double().numpy(), V.double().numpy())
        return kvs[l]

    img = case.img_range.numpy()
    for l in range(wl1.layers):
        kv(l, 0)
    focal, f_last = wl1.focal_layers, [None]
    t = t_first
    if wl1.mode == "fastocr" and focal is None:
        ratio = np.zeros(wl1.layers)
        for t in range(wl1.warmup):
            q = case.q_at(t).double().numpy()
            _, mass, sel = S.warmup_step(q, kv, np.array([wl1.seq_len_at(t)]), img, wl1.tau)
            ratio += mass
        focal = S.choose_focal_layers(ratio, wl1.n_focal)
        f_last = list(sel[max(focal)])
        t = wl1.warmup
    import oracle.attention as A
    done, t0 = 0, time.perf_counter()
    while True:
        q = case.q_at(t).double().numpy()
        n_t = np.array([wl1.seq_len_at(t)])
        if wl1.mode == "rswa":
            for l in range(wl1.layers):
                A.rswa_attend(q[l, 0], *kv(l, 0), int(n_t[0]), wl1.rswa_prefix, wl1.rswa_window)
        else:
            _, _, f_last = S.steady_step(q, kv, n_t, img, wl1.tau, focal, f_last)
        done += 1
        t += 1
        el = time.perf_counter() - t0
        if (el >= float(budget) and done >= 2) or t >= max_steps:
            break
    seq_steps_per_s = done / el
    print(json.dumps({"seq_steps_per_s": seq_steps_per_s, "steps": done, "seconds": el,
                      "batch": wl.batch}))


def run_oracle_leg(workload: str, tau, budget_s: float):
    env = dict(os.environ)
    for v in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "OMP_NUM_THREADS"):
        env[v] = "1"
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-leg",
           f"{workload}:{tau if tau else 0}:{budget_s}"]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        raise RuntimeError(f"oracle leg failed: {r.stderr[-2000:]}")
    d = json.loads(r.stdout.strip().splitlines()[-1])
    # the oracle ran one sequence; a step of the workload covers `batch` sequences
    d["value"] = d["seq_steps_per_s"] / d["batch"]
    return d


# ------------------------------------------------------------------ GPU benchmark

def kv_bytes(wl, kind: str, n_t: int, k_per_seq) -> float:
    """Algorithmic KV bytes one launch of `kind` reads (all sequences)."""
    row = 2 * wl.kv_heads * wl.head_dim * (2 if wl.dtype == "bf16" else 4)  # K + V per token
    tot = 0
    for b in range(wl.batch):
        if kind in ("focal", "full"):
            n = n_t
        elif kind == "sparse":
            n = wl.prompt + int(k_per_seq[b]) + (n_t - wl.prompt - wl.n_img)
        else:  # rswa
            n = min(wl.rswa_prefix, n_t) + max(0, n_t - max(wl.rswa_prefix, n_t - wl.rswa_window))
        tot += n * row
    return float(tot)


def run_gpu(args, rank, world, local_rank):
    import torch

    import synth
    from dynamic_sparse_kv_gb300 import CapturedStep, DecodeAttention
    import dynamic_sparse_kv_gb300._native as N

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = synth.workload(args.workload)
    if args.tau is not None:
        wl = wl.with_(tau=args.tau)
    for item in args.set:
        key, val = item.split("=", 1)
        wl = wl.with_(**{key: type(getattr(wl, key))(val)})
    wl = wl.with_(seed=wl.seed + 1000 * rank)
    K, W = args.steps, args.warmup
    assert W >= 3, "at least 3 warm-up steps"
    if wl.mode == "fastocr":
        t0_steady, step0 = wl.warmup, 0         # the warm-up reads steps [0, warmup)
    else:   # R-SWA: the last steps before T = wl.steps generated tokens (window full)
        t0_steady = step0 = max(0, wl.steps - (W + K))
    span = wl.steps - t0_steady                 # steady steps available in the workload
    n_gen = min(wl.steps, t0_steady + W + K) - step0
    case = synth.make_case(wl, device=dev, step0=step0, n_steps=n_gen)
    storage = "full"
    if wl.mode == "rswa" and args.rswa_ring:
        # bounded memory: pages past the prefix form a ring of ceil(n / page)
        # pages per sequence; the timed kernels are the same
        from dynamic_sparse_kv_gb300 import ring_block_table
        table, per = ring_block_table(wl.batch, wl.rswa_prefix, wl.rswa_window, wl.page_size,
                                      wl.max_tokens)
        n_pages = wl.batch * per
        k_ring = case.k_cache[:, :n_pages].clone()
        v_ring = case.v_cache[:, :n_pages].clone()
        case = dataclasses.replace(case, k_cache=k_ring, v_cache=v_ring,
                                   block_table=table.to(dev))
        torch.cuda.empty_cache()
        storage = "ring"

    def t_of(i):                                # i-th bench step -> decode step index
        return t0_steady + (i % min(span, n_gen - (t0_steady - step0)))

    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def build(tau, kind):
        dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                              img_range=case.img_range, max_img=wl.n_img, tau=tau, mode=wl.mode,
                              rswa_prefix=wl.rswa_prefix, rswa_window=wl.rswa_window)
        focal = None
        if kind == "fastocr":
            if wl.focal_layers is not None:
                dec.set_focal_layers(wl.focal_layers)
                focal = tuple(wl.focal_layers)
            else:
                qw = torch.empty_like(case.q_at(0))
                dec.begin_warmup()
                for t in range(wl.warmup):   # the method's profiling warm-up (untimed)
                    dec.set_seq_len(wl.seq_len_at(t))
                    dec.warmup_step(case.q_at(t).contiguous(), qw)
                focal, _ = dec.finish_warmup(wl.n_focal)
        dec.set_seq_len(wl.seq_len_at(t_of(0)))
        return dec, focal, CapturedStep(dec, kind)

    def stage(dec, cap, i):
        t = t_of(i)
        dec.set_seq_len(wl.seq_len_at(t))
        cap.q.copy_(case.q_at(t))

    def time_graph(dec, cap, n_warm, n_timed, sampler_gpu=None):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
        for i in range(n_warm):
            stage(dec, cap, i)
            flush.zero_()
            cap.replay()
        torch.cuda.synchronize()
        barrier(world)
        sampler = ClockSampler(sampler_gpu) if sampler_gpu else None
        wall0 = time.perf_counter()
        for j in range(n_timed):
            stage(dec, cap, n_warm + j)
            flush.zero_()
            starts[j].record()
            cap.replay()
            ends[j].record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
        clocks = sampler.stop() if sampler else None
        barrier(world)
        per = [s.elapsed_time(e) for s, e in zip(starts, ends)]      # ms
        return per, wall, clocks

    gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    kind = "rswa" if wl.mode == "rswa" else "fastocr"
    dec, focal, cap = build(wl.tau, kind)
    per, wall, clocks = time_graph(dec, cap, W, K, sampler_gpu=gpu_uuid)
    total_ms = reduce_max(sum(per), world, dev)
    status = dec.device_status()
    assert status == 0, f"device status {status}"

    # ---- per-kernel durations (eager launches queued behind a sleep, events between)
    def layer_kind(l):
        if kind == "rswa":
            return "rswa"
        return "focal" if l in dec.sel else "sparse"

    n_kt = min(K, 50)
    kt = {"focal": [], "sparse": [], "rswa": [], "full": []}
    kbytes = {"focal": [], "sparse": [], "rswa": [], "full": []}
    stream = torch.cuda.current_stream()
    for j in range(n_kt):
        stage(dec, cap, W + j)
        flush.zero_()
        torch.cuda._sleep(4_000_000)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(dec.layers + 1)]
        ev[0].record()
        cur = dec.sel[max(dec.focal)] if kind == "fastocr" else None
        for l in range(dec.layers):
            if kind == "rswa":
                N.fastocr_rswa_attend(dec.handle, cap.q[l], dec.kv[l], wl.rswa_prefix,
                                      wl.rswa_window, cap.out[l], stream)
            elif l in dec.sel:
                idx, kk = dec.sel[l]
                N.fastocr_focal_attend(dec.handle, cap.q[l], dec.kv[l], dec.img_range, dec.tau,
                                       cap.out[l], idx, dec.stride, kk, -1, stream)
                cur = (idx, kk)
            else:
                N.fastocr_sparse_attend(dec.handle, cap.q[l], dec.kv[l], dec.img_range, cur[0],
                                        dec.stride, cur[1], cap.out[l], stream)
            ev[l + 1].record()
        torch.cuda.synchronize()
        n_t = wl.seq_len_at(t_of(W + j))
        k_seq = dec.sel[max(dec.focal)][1].tolist() if kind == "fastocr" else None
        for l in range(dec.layers):
            kd = layer_kind(l)
            kt[kd].append(ev[l].elapsed_time(ev[l + 1]) * 1e-3)      # s
            kbytes[kd].append(kv_bytes(wl, kd, n_t, k_seq))
    peak, peak_src = measured_peaks()
    kernels = {}
    for kd in kt:
        if not kt[kd]:
            continue
        launches_per_step = len(kt[kd]) / n_kt
        mean_s = statistics.fmean(kt[kd])
        bpl = statistics.fmean(kbytes[kd])
        kernels[kd] = {"launches_per_step": launches_per_step, "us_per_launch": mean_s * 1e6,
                       "kv_bytes_per_launch": bpl, "gbs": bpl / mean_s / 1e9,
                       "share": launches_per_step * mean_s}
    tot_share = sum(v["share"] for v in kernels.values())
    for v in kernels.values():
        v["share"] = v["share"] / tot_share
    dom = max(kernels, key=lambda k: kernels[k]["share"])
    kname = {"focal": "attend_focal", "sparse": "attend_sparse", "rswa": "attend_rswa",
             "full": "attend_full"}[dom]
    roofline = {"bound": "hbm", "kernel": kname, "achieved": kernels[dom]["gbs"], "peak": peak,
                "unit": "GB/s", "frac": kernels[dom]["gbs"] / peak,
                "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_src == "measured" else "fallback 6.8 TB/s",
                "traffic": recorded_traffic(kname, wl.name)}

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        q_host = torch.empty((n_gen,) + tuple(cap.q.shape), dtype=cap.q.dtype, pin_memory=True)
        q_host.copy_(case.q)
        out_host = torch.empty(tuple(cap.out.shape), dtype=cap.out.dtype, pin_memory=True)
        n_e = min(K, 200)
        s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_e)]
        e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_e)]
        for j in range(W + n_e):
            t = t_of(j)
            flush.zero_()
            if j >= W:
                s_ev[j - W].record()
            dec.set_seq_len(wl.seq_len_at(t))
            cap.q.copy_(q_host[t - case.step0], non_blocking=True)
            cap.replay()
            out_host.copy_(cap.out, non_blocking=True)
            if j >= W:
                e_ev[j - W].record()
        torch.cuda.synchronize()
        e_ms = reduce_max(sum(s.elapsed_time(e) for s, e in zip(s_ev, e_ev)), world, dev)
        qb = cap.q.numel() * cap.q.element_size() + 4 * wl.batch
        e2e = {"value": world * n_e / (e_ms * 1e-3), "unit": "steps/s",
               "h2d_bytes_per_step": qb, "d2h_bytes_per_step": cap.out.numel() * cap.out.element_size(),
               "us_per_step": e_ms * 1e3 / n_e}

    # ---- comparison arms: dense (every layer full) and the tau = 1 FastOCR pipeline
    compare = {}
    if not args.no_compare and kind == "fastocr":
        dcap = CapturedStep(dec, "dense")
        per_d, _, _ = time_graph(dec, dcap, W, min(K, 200))
        compare["dense_us_per_step"] = statistics.fmean(per_d) * 1e3
        dec1, _, cap1 = build(1.0, "fastocr")
        per_1, _, _ = time_graph(dec1, cap1, W, min(K, 200))
        compare["tau1_us_per_step"] = statistics.fmean(per_1) * 1e3
        dec1.close()
        # adaptive layer selection: the cost of one profiling step (full
        # attention, scoring, selection and profile accumulation in every
        # layer) and of capturing the steady step anew after C changes
        pcap = CapturedStep(dec, "profile")
        per_p, _, _ = time_graph(dec, pcap, W, min(K, 200))
        compare["profile_us_per_step"] = statistics.fmean(per_p) * 1e3
        torch.cuda.synchronize()
        c0 = time.perf_counter()
        del pcap
        pcap = CapturedStep(dec, "fastocr")
        torch.cuda.synchronize()
        compare["recapture_ms"] = (time.perf_counter() - c0) * 1e3
        del pcap
        # latency floor of a decode step's launch chain: as many dependent
        # one-element kernels as the step has layers, in one CUDA graph
        tiny = torch.zeros(1, device=dev)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            tiny.add_(1.0)
        torch.cuda.current_stream().wait_stream(side)
        chain = torch.cuda.CUDAGraph()
        with torch.cuda.graph(chain):
            for _ in range(wl.layers):
                tiny.add_(1.0)
        ts = []
        for _ in range(W + 50):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            chain.replay()
            s1.record()
            torch.cuda.synchronize()
            ts.append(s0.elapsed_time(s1) * 1e3)
        compare["launch_chain_floor_us_per_step"] = statistics.median(ts[W:])
        del chain

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        try:
            leg = run_oracle_leg(wl.name, args.tau, 10.0)
            cpu = {"value": leg["value"], "unit": "steps/s", "cores": 1, "kind": "oracle",
                   "sample": f"fp64 NumPy oracle, 1 thread, {leg['steps']} steady decode steps "
                             f"of sequence 0 ({leg['seconds']:.1f} s), scaled to the "
                             f"{wl.batch}-sequence step"}
        except Exception as e:  # report, do not hide
            cpu = {"value": None, "unit": "steps/s", "cores": 1, "kind": "oracle",
                   "sample": f"failed: {e}"[:300]}

    us_per_step = total_ms * 1e3 / K
    step_bytes = sum(kernels[k]["kv_bytes_per_launch"] * kernels[k]["launches_per_step"]
                     for k in kernels)
    value = world * K / (total_ms * 1e-3)
    res = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "batch_per_gpu": wl.batch, "layers": wl.layers,
                   "q_heads": wl.q_heads, "kv_heads": wl.kv_heads, "head_dim": wl.head_dim,
                   "prompt": wl.prompt, "n_img": wl.n_img, "tau": wl.tau,
                   "focal_layers": list(focal) if focal else None, "page_size": wl.page_size,
                   "parallelism": f"replicas{world}",
                   "l2": "flushed before every timed step (512 MB memset, untimed)",
                   "us_per_step": us_per_step, "kv_bytes_per_step": step_bytes,
                   "achieved_step_gbs": step_bytes / (us_per_step * 1e-6) / 1e9,
                   "wall_s_timed_loop": wall, "kernels": kernels, **compare},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": cap.launches * K, "clocks": clocks,
    }
    if wl.mode == "rswa":
        res["config"].update({
            "rswa_prefix": wl.rswa_prefix, "rswa_window": wl.rswa_window,
            "generated_tokens_timed": [t_of(W) + 1, t_of(W + K - 1) + 1], "storage": storage,
            "kv_cache_bytes_per_layer": 2 * case.k_cache[0].numel() * case.k_cache.element_size()})
    if "dense_us_per_step" in compare:
        res["config"]["speedup_vs_dense"] = compare["dense_us_per_step"] / us_per_step
        res["config"]["speedup_vs_tau1"] = compare["tau1_us_per_step"] / us_per_step
    dec.close()
    return res


def run_reference(args):
    import synth
    wl = synth.workload(args.workload)
    t0 = time.perf_counter()
    legs = [run_oracle_leg(args.workload, args.tau, 3.0) for _ in range(max(1, args.steps // 50))]
    el = time.perf_counter() - t0
    v = statistics.fmean(l["value"] for l in legs)
    steps = sum(l["steps"] for l in legs)
    sample = (f"fp64 NumPy oracle, 1 thread, {steps} steady decode steps of sequence 0 "
              f"over {len(legs)} runs, scaled to the {wl.batch}-sequence step")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": 0,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "tau": args.tau or wl.tau,
                       "wall_s": el},
            "cpu_baseline": {"value": v, "unit": "steps/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_leg:
        oracle_leg(args.oracle_leg)
        return 0
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
