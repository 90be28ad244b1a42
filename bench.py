#!/usr/bin/env python3
"""Decode-attention benchmark of the FastOCR path (and R-SWA) on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one decode step through every layer of the workload (focal layers:
full attention + image scores + top-k; other layers: gather attention over
prompt + selected image tokens + generated tokens, with Cross-Step Fixation
Reuse), captured once in a CUDA graph and replayed. Inputs are synthetic and
seeded (synth module) and resident in HBM. L2 is flushed (512 MB memset,
untimed) before every timed step. The K-step timed pass is repeated until the
timed work spans a few seconds (so the clock sampler sees it); the reported
value is the median pass. Prints one JSON line.

The headline workload is `serving_b32` (32 sequences x 8192 image tokens, the
largest single-GPU configuration); the batch-1 `qwen7b_b1` workload is
measured in the same run and reported in the line's `secondary` block.

Inside the line, `config.kernels` gives each layer kind's share of the step:
the step's layers of one kind (focal: attend + selection; sparse: gather
attend) captured alone in a graph, in step order, and replayed like the step,
so the kinds' times add up to about the step (`kinds_sum_over_step`); the
roofline record takes the kind with the largest share. `alone` gives one
launch of each kind timed by itself (its own graph, L2 flushed).

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
import math
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
PROBE_BYTES = 2 << 30
CSRC = os.path.join(ROOT, "dynamic_sparse_kv_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_NAME = {"focal": "attend_focal", "sparse": "attend_sparse", "rswa": "attend_rswa",
               "full": "attend_full"}


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="serving_b32")
    ap.add_argument("--secondary", default="qwen7b_b1",
                    help="second workload reported in the same line ('none' to skip)")
    ap.add_argument("--soak", type=float, default=4.0,
                    help="seconds of timed passes (repeats of the K-step pass)")
    ap.add_argument("--tau", type=float, default=None)
    ap.add_argument("--set", action="append", default=[], metavar="FIELD=VALUE",
                    help="override a workload field, e.g. --set batch=8 (profiling runs)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-compare", action="store_true", help="skip the dense / tau=1 arms")
    ap.add_argument("--no-probe", action="store_true", help="skip the read-only bandwidth probe")
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


# the sources that define the attend and selection kernels and how they are
# launched (split choice, variants); the no-alloc entry point and the
# streaming utilities do not change what an ncu capture of those kernels sees
KERNEL_SOURCES = ("abi.cu", "attend_impl.cuh", "attend_kernels.cuh", "kernels_bf16.cu",
                  "kernels_f32.cu")


def source_digest() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary (profiles/traffic.json),
    if it was taken on the current kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            entries = json.load(f)["entries"]
    except (OSError, ValueError, KeyError):
        return None
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload:
            return float(e["bytes_per_launch"]) if e.get("digest") == source_digest() else None
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
                 "-lms", "50", "-i", gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
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


def kinds_check(kernels: dict, us_per_step: float) -> dict:
    """How the per-kind in-step times add up against the step."""
    tot = sum(v["us_in_step"] for v in kernels.values())
    return {"kinds_sum_us": tot, "kinds_sum_over_step": tot / us_per_step,
            "kinds_exceed_step": tot > 1.10 * us_per_step}


def read_probe(dev, flush, world):
    """Read-only HBM bandwidth: fastocr_read_probe over 2 GiB (16x L2), L2
    flushed before each of 12 timed reads; median and best GB/s."""
    import torch

    import dynamic_sparse_kv_gb300._native as N
    buf = torch.ones(PROBE_BYTES, dtype=torch.uint8, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    times = []
    for r in range(15):
        flush.zero_()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        N.fastocr_read_probe(buf, PROBE_BYTES, sink)
        e.record()
        torch.cuda.synchronize()
        if r >= 3:
            times.append(s.elapsed_time(e) * 1e-3)
    del buf
    torch.cuda.empty_cache()
    med = reduce_max(statistics.median(times), world, dev)
    return {"gbs": PROBE_BYTES / med / 1e9, "best_gbs": PROBE_BYTES / min(times) / 1e9,
            "bytes": PROBE_BYTES, "reads": len(times),
            "how": "fastocr_read_probe: one read of every 16-byte word, ld.global.nc, "
                   "L2 flushed before each read, CUDA events, median"}


class Bench:
    """One workload on one GPU: case, decoder, graphs and their timings."""

    def __init__(self, args, name, rank, world, dev, flush, tau=None, overrides=()):
        import torch

        import synth
        self.torch = torch
        self.args, self.rank, self.world, self.dev, self.flush = args, rank, world, dev, flush
        wl = synth.workload(name)
        if tau is not None:
            wl = wl.with_(tau=tau)
        for item in overrides:
            key, val = item.split("=", 1)
            wl = wl.with_(**{key: type(getattr(wl, key))(val)})
        self.wl = wl = wl.with_(seed=wl.seed + 1000 * rank)
        K, W = args.steps, args.warmup
        if wl.mode == "fastocr":
            # queries of every decode step: the warm-up reads [0, warmup), the
            # timed steps sample the whole steady decode (lists grow with t)
            self.t0_steady, step0 = wl.warmup, 0
            self.n_gen = wl.steps
        else:   # R-SWA: the last steps before T = wl.steps generated tokens (window full)
            self.t0_steady = step0 = max(0, wl.steps - (W + K))
            self.n_gen = wl.steps - step0
        self.span = wl.steps - self.t0_steady        # steady steps available in the workload
        case = synth.make_case(wl, device=dev, step0=step0, n_steps=self.n_gen)
        self.storage = "full"
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
            self.storage = "ring"
        self.case = case
        self.kind = "rswa" if wl.mode == "rswa" else "fastocr"

    def t_of(self, i):
        """Decode step of the i-th bench step: every K consecutive bench steps
        sample the steady decode at a stride of span/K steps (each group of K
        shifted by one), so every timed pass sees the same mix of cache lengths."""
        K = self.args.steps
        j, p = i % K, i // K
        return self.t0_steady + (j * self.span // K + p) % self.span

    def build(self, tau, kind):
        from dynamic_sparse_kv_gb300 import CapturedStep, DecodeAttention
        wl, case = self.wl, self.case
        dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                              img_range=case.img_range, max_img=wl.n_img, tau=tau, mode=wl.mode,
                              rswa_prefix=wl.rswa_prefix, rswa_window=wl.rswa_window)
        focal = None
        if kind == "fastocr":
            if wl.focal_layers is not None:
                dec.set_focal_layers(wl.focal_layers)
                focal = tuple(wl.focal_layers)
            else:
                qw = self.torch.empty_like(case.q_at(0))
                dec.begin_warmup()
                q_t = None
                for t in range(wl.warmup):   # the method's profiling warm-up (untimed)
                    dec.set_seq_len(wl.seq_len_at(t))
                    q_t = case.q_at(t).contiguous()
                    dec.warmup_step(q_t, qw, select=False)
                focal, _ = dec.finish_warmup(wl.n_focal, q=q_t)
        dec.set_seq_len(self.wl.seq_len_at(self.t_of(0)))
        return dec, focal, CapturedStep(dec, kind)

    def stage(self, dec, cap, i):
        t = self.t_of(i)
        dec.set_seq_len(self.wl.seq_len_at(t))
        cap.q.copy_(self.case.q_at(t))

    def time_graph(self, dec, cap, soak_s, sampler_gpu=None, min_passes=3, max_passes=2000):
        """Warm-up W steps, then repeat the K-step timed pass (L2 flushed before
        every step, untimed) for about soak_s seconds. Returns (median pass ms
        summed over its K steps, all pass totals, wall seconds, clocks)."""
        torch = self.torch
        K, W = self.args.steps, self.args.warmup
        for i in range(W):
            self.stage(dec, cap, i)
            self.flush.zero_()
            cap.replay()
        torch.cuda.synchronize()
        barrier(self.world)

        def one_pass(i0):
            starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
            ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
            for j in range(K):
                self.stage(dec, cap, i0 + j)
                self.flush.zero_()
                starts[j].record()
                cap.replay()
                ends[j].record()
            torch.cuda.synchronize()
            return sum(s.elapsed_time(e) for s, e in zip(starts, ends))

        sampler = ClockSampler(sampler_gpu) if sampler_gpu else None
        wall0 = time.perf_counter()
        passes = [one_pass(W)]
        first = time.perf_counter() - wall0
        n = int(min(max_passes, max(min_passes, math.ceil(soak_s / max(first, 1e-6)))))
        n = int(reduce_max(float(n), self.world, self.dev))   # same pass count on every rank
        for p in range(1, n):
            passes.append(one_pass(W + p * K))
        wall = time.perf_counter() - wall0
        clocks = sampler.stop() if sampler else None
        barrier(self.world)
        med = statistics.median(passes)
        return reduce_max(med, self.world, self.dev), passes, wall, clocks

    def time_replays(self, dec, cap, reps=2):
        """µs of one replay of cap averaged over the decode steps of the timed
        pass (the same K steps, staged the same way, L2 flushed before each):
        each step's time is the median of `reps` replays, and the result is
        their mean, so it is comparable with the step time. Also returns the
        staged decode steps."""
        torch = self.torch
        K, W = self.args.steps, self.args.warmup
        for i in range(W):
            self.stage(dec, cap, i)
            self.flush.zero_()
            cap.replay()
        per_step = [[] for _ in range(K)]
        for _ in range(reps):
            for j in range(K):
                self.stage(dec, cap, W + j)
                self.flush.zero_()
                s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                s.record()
                cap.replay()
                e.record()
                torch.cuda.synchronize()
                per_step[j].append(s.elapsed_time(e) * 1e3)
        us = statistics.fmean(statistics.median(x) for x in per_step)
        return reduce_max(us, self.world, self.dev), [self.t_of(W + j) for j in range(K)]

    # ---- per-kind graphs: the step's layers of one kind, in step order
    def kind_fns(self, dec):
        wl = self.wl
        if self.kind == "rswa":
            def rswa(q, out, stream=None):
                dec.rswa_step(q, out, stream)
            return {"rswa": (rswa, dec.layers, dec.layers)}
        focal = set(dec.sel)

        def only(kind):   # the step's own schedule, issuing just this kind's calls
            def fn(q, out, stream=None):
                dec.step(q, out, stream, only=kind)
            return fn
        n_f = len(focal)
        return {"focal": (only("focal"), n_f, 2 * n_f),
                "sparse": (only("sparse"), wl.layers - n_f, wl.layers - n_f)}

    def single_fn(self, dec, kind):
        """One launch of `kind` (its first layer in the step)."""
        import dynamic_sparse_kv_gb300._native as N
        if kind == "rswa":
            def fn(q, out, stream=None):
                N.fastocr_rswa_attend(dec.handle, q[0], dec.kv[0], self.wl.rswa_prefix,
                                      self.wl.rswa_window, out[0], stream)
            return fn
        first_focal = min(dec.sel)
        first_sparse = next(l for l in range(dec.layers) if l not in dec.sel)

        def fn(q, out, stream=None):
            src = dec.sel[max(dec.focal)]
            if kind == "focal":
                idx, k = dec.sel[first_focal]
                N.fastocr_focal_attend(dec.handle, q[first_focal], dec.kv[first_focal],
                                       dec.img_range, dec.tau, out[first_focal], idx, dec.stride,
                                       k, -1, stream)
            else:
                N.fastocr_sparse_attend(dec.handle, q[first_sparse], dec.kv[first_sparse],
                                        dec.img_range, src[0], dec.stride, src[1],
                                        out[first_sparse], stream)
        return fn

    def kernel_breakdown(self, dec, us_per_step):
        from dynamic_sparse_kv_gb300 import CapturedStep
        wl = self.wl
        kernels, alone = {}, {}
        for kind, (fn, layers, launches) in self.kind_fns(dec).items():
            cap = CapturedStep(dec, kind, fn=fn, launches=launches)
            us, steps = self.time_replays(dec, cap)
            del cap
            k_seq = dec.sel[max(dec.focal)][1].tolist() if self.kind == "fastocr" else None
            bpl = statistics.fmean(kv_bytes(wl, kind, wl.seq_len_at(t), k_seq) for t in steps)
            kernels[kind] = {"layers_per_step": layers, "launches_per_step": launches,
                             "us_in_step": us, "us_per_layer": us / layers,
                             "kv_bytes_per_layer": bpl, "gbs": bpl * layers / (us * 1e-6) / 1e9,
                             "share": us / us_per_step}
            cap1 = CapturedStep(dec, kind + "_alone", fn=self.single_fn(dec, kind),
                                launches=launches // layers)
            us1, steps1 = self.time_replays(dec, cap1)
            del cap1
            b1 = statistics.fmean(kv_bytes(wl, kind, wl.seq_len_at(t), k_seq) for t in steps1)
            alone[kind] = {"us": us1, "kv_bytes": b1, "gbs": b1 / (us1 * 1e-6) / 1e9}
        return kernels, alone

    def e2e(self, dec, cap):
        """Same step through the public API with host buffers: the step's
        queries copied from pinned host memory and its outputs read back
        every step, inside the timing. The headline figure replays a
        CapturedStep(host_io=True), whose graph copies the queries in ahead
        of the first layer and the outputs out while later layers run;
        `serial` is the same step with one copy in, the device-buffer graph,
        and one copy out, back to back."""
        from dynamic_sparse_kv_gb300 import CapturedStep
        torch = self.torch
        K, W = self.args.steps, self.args.warmup
        case, wl = self.case, self.wl
        q_steps = torch.empty((self.n_gen,) + tuple(cap.q.shape), dtype=cap.q.dtype,
                              pin_memory=True)
        q_steps.copy_(case.q)
        n_e = max(K, 50)

        def run(prepare, replay_step):
            s_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_e)]
            e_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_e)]
            for j in range(W + n_e):
                t = self.t_of(j)
                # host side, before the step's timing starts: wait for the
                # previous step, then stage this step's inputs (the L2 flush
                # that follows gives the host time to queue the step)
                torch.cuda.current_stream().synchronize()
                prepare(t - case.step0)
                self.flush.zero_()
                if j >= W:
                    s_ev[j - W].record()
                dec.set_seq_len(wl.seq_len_at(t))
                replay_step(t - case.step0)
                if j >= W:
                    e_ev[j - W].record()
            torch.cuda.synchronize()
            ms = sum(s.elapsed_time(e) for s, e in zip(s_ev, e_ev))
            return reduce_max(ms, self.world, self.dev)

        out_host = torch.empty(tuple(cap.out.shape), dtype=cap.out.dtype, pin_memory=True)

        def serial(i):
            cap.q.copy_(q_steps[i], non_blocking=True)
            cap.replay()
            out_host.copy_(cap.out, non_blocking=True)

        ms_serial = run(lambda i: None, serial)
        io = CapturedStep(dec, cap.kind, host_io=True)

        def stage(i):   # the graph copies from q_host
            io.q_host.copy_(q_steps[i])

        e_ms = run(stage, lambda i: io.replay())
        del io
        qb = cap.q.numel() * cap.q.element_size() + 4 * wl.batch
        return {"value": self.world * n_e / (e_ms * 1e-3), "unit": "steps/s",
                "h2d_bytes_per_step": qb,
                "d2h_bytes_per_step": cap.out.numel() * cap.out.element_size(),
                "us_per_step": e_ms * 1e3 / n_e, "steps": n_e,
                "how": "CapturedStep(host_io=True): queries in by fastocr_copy ahead of "
                       "layer 0, outputs out in chunks overlapped with the later layers, "
                       "all inside the graph; CUDA events around each step",
                "serial": {"value": self.world * n_e / (ms_serial * 1e-3),
                           "us_per_step": ms_serial * 1e3 / n_e,
                           "how": "copy in, device-buffer graph, copy out, back to back"}}

    def launch_chain_floor(self):
        """A CUDA graph of as many dependent one-element kernels as the step
        has layers: the latency floor of a dependent launch chain."""
        torch = self.torch
        tiny = torch.zeros(1, device=self.dev)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            tiny.add_(1.0)
        torch.cuda.current_stream().wait_stream(side)
        chain = torch.cuda.CUDAGraph()
        with torch.cuda.graph(chain):
            for _ in range(self.wl.layers):
                tiny.add_(1.0)
        ts = []
        for _ in range(self.args.warmup + 50):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            chain.replay()
            s1.record()
            torch.cuda.synchronize()
            ts.append(s0.elapsed_time(s1) * 1e3)
        return statistics.median(ts[self.args.warmup:])

    def compare_arms(self, dec):
        """Dense (every layer full) and the tau = 1 FastOCR pipeline, timed like
        the step; a profiling step and the re-capture cost of adaptive layer
        selection."""
        from dynamic_sparse_kv_gb300 import CapturedStep
        torch = self.torch
        compare = {}
        dcap = CapturedStep(dec, "dense")
        ms, _, _, _ = self.time_graph(dec, dcap, 1.0)
        compare["dense_us_per_step"] = ms * 1e3 / self.args.steps
        del dcap
        dec1, _, cap1 = self.build(1.0, "fastocr")
        ms, _, _, _ = self.time_graph(dec1, cap1, 1.0)
        compare["tau1_us_per_step"] = ms * 1e3 / self.args.steps
        del cap1
        dec1.close()
        # a profiling window's step (full attention, mass in the epilogue); the
        # window's end adds one focal layer (config.alone.focal)
        pcap = CapturedStep(dec, "profile_mass")
        ms, _, _, _ = self.time_graph(dec, pcap, 0.5)
        compare["profile_us_per_step"] = ms * 1e3 / self.args.steps
        torch.cuda.synchronize()
        c0 = time.perf_counter()
        del pcap
        pcap = CapturedStep(dec, "fastocr")
        torch.cuda.synchronize()
        compare["recapture_ms"] = (time.perf_counter() - c0) * 1e3
        del pcap
        return compare


def run_workload(args, name, rank, world, dev, flush, *, headline, sampler_gpu=None):
    """Measure one workload; returns (result dict, Bench, peak info)."""
    torch = __import__("torch")
    K = args.steps
    bn = Bench(args, name, rank, world, dev, flush, tau=args.tau if headline else None,
               overrides=args.set if headline else ())
    wl = bn.wl
    dec, focal, cap = bn.build(wl.tau, bn.kind)
    ms_pass, passes, wall, clocks = bn.time_graph(dec, cap, args.soak if headline else 1.0,
                                                  sampler_gpu=sampler_gpu)
    status = dec.device_status()
    assert status == 0, f"device status {status}"
    us_per_step = ms_pass * 1e3 / K
    kernels, alone = bn.kernel_breakdown(dec, us_per_step)
    check = kinds_check(kernels, us_per_step)
    e2e = None if args.no_e2e else bn.e2e(dec, cap)
    compare = {}
    if not args.no_compare and bn.kind == "fastocr":
        compare = bn.compare_arms(dec)
    compare["launch_chain_floor_us_per_step"] = bn.launch_chain_floor()
    step_bytes = sum(v["kv_bytes_per_layer"] * v["layers_per_step"] for v in kernels.values())
    res = {
        "workload": wl.name, "us_per_step": us_per_step, "steps_per_s": world * 1e6 / us_per_step,
        "tau": wl.tau, "batch_per_gpu": wl.batch, "focal_layers": list(focal) if focal else None,
        "kv_bytes_per_step": step_bytes,
        "achieved_step_gbs": step_bytes / (us_per_step * 1e-6) / 1e9,
        "timed_passes": len(passes), "pass_ms_min_median_max": [min(passes), ms_pass, max(passes)],
        "wall_s_timed_passes": wall, "kernels": kernels, **check, "alone": alone,
        "gpu_launches_per_step": cap.launches, **compare, "e2e": e2e,
    }
    if "dense_us_per_step" in compare:
        res["speedup_vs_dense"] = compare["dense_us_per_step"] / us_per_step
        res["speedup_vs_tau1"] = compare["tau1_us_per_step"] / us_per_step
    if wl.mode == "rswa":
        res.update({
            "rswa_prefix": wl.rswa_prefix, "rswa_window": wl.rswa_window,
            "generated_tokens_timed": [bn.t_of(args.warmup) + 1,
                                       bn.t_of(args.warmup + K - 1) + 1],
            "storage": bn.storage,
            "kv_cache_bytes_per_layer": 2 * bn.case.k_cache[0].numel()
            * bn.case.k_cache.element_size()})
    dec.close()
    del cap, dec
    torch.cuda.synchronize()
    return res, bn, clocks


def run_gpu(args, rank, world, local_rank):
    import torch

    import dynamic_sparse_kv_gb300  # noqa: F401  (loads libfastocr.so or raises)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    assert args.warmup >= 3, "at least 3 warm-up steps"
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    K, W = args.steps, args.warmup

    main, bn, clocks = run_workload(args, args.workload, rank, world, dev, flush, headline=True,
                                    sampler_gpu=gpu_uuid)
    wl = bn.wl
    del bn
    torch.cuda.empty_cache()

    peak, peak_src = measured_peaks()
    probe = None if args.no_probe else read_probe(dev, flush, world)
    kernels = main["kernels"]
    dom = max(kernels, key=lambda k: kernels[k]["us_in_step"])
    kd = kernels[dom]
    kname = KERNEL_NAME[dom]
    roofline = {"bound": "hbm", "kernel": kname, "achieved": kd["gbs"], "peak": peak,
                "unit": "GB/s", "frac": kd["gbs"] / peak,
                "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_src == "measured" else "fallback 6.8 TB/s",
                "traffic": recorded_traffic(kname, wl.name),
                "us_per_launch_in_step": kd["us_per_layer"],
                "launches_times_us_over_step": kd["us_in_step"] / main["us_per_step"],
                "how": "algorithmic K/V bytes of the kind's layers / time of those layers "
                       "replayed alone in step order (CUDA graph, L2 flushed)"}
    if dom == "focal":
        roofline["note"] = "a focal layer is the attend kernel plus the selection kernel"
    if probe:
        roofline["peak_readonly"] = probe["gbs"]
        roofline["frac_readonly"] = kd["gbs"] / probe["gbs"]

    secondary = None
    if args.secondary and args.secondary != "none" and args.secondary != args.workload:
        secondary, bn2, _ = run_workload(args, args.secondary, rank, world, dev, flush,
                                         headline=False)
        del bn2
        torch.cuda.empty_cache()

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

    us_per_step = main["us_per_step"]
    value = world * 1e6 / us_per_step
    config = {"workload": wl.name, "batch_per_gpu": wl.batch, "layers": wl.layers,
              "q_heads": wl.q_heads, "kv_heads": wl.kv_heads, "head_dim": wl.head_dim,
              "prompt": wl.prompt, "n_img": wl.n_img, "tau": wl.tau, "page_size": wl.page_size,
              "parallelism": f"replicas{world}",
              "l2": "flushed before every timed step (512 MB memset, untimed)"}
    config.update({k: v for k, v in main.items() if k not in ("workload", "e2e")})
    res = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": us_per_step * 1e-3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": config, "roofline": roofline, "read_probe": probe, "cpu_baseline": cpu,
        "e2e": main["e2e"], "gpu_launches": main["gpu_launches_per_step"] * K,
        "clocks": clocks, "secondary": secondary,
    }
    return res


def run_reference(args):
    """The reference arm: the fp64 oracle on the host cores, on a bounded
    sample of the same workload, reported with the same steps and config keys."""
    import synth
    wl = synth.workload(args.workload)
    tau = args.tau or wl.tau
    t0 = time.perf_counter()
    legs = [run_oracle_leg(args.workload, args.tau, 3.0) for _ in range(max(1, args.steps // 50))]
    el = time.perf_counter() - t0
    v = statistics.fmean(l["value"] for l in legs)
    done = sum(l["steps"] for l in legs)
    sample = (f"fp64 NumPy oracle, 1 thread, {done} steady decode steps of sequence 0 "
              f"over {len(legs)} runs, scaled to the {wl.batch}-sequence step")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "steps/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / v,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "batch_per_gpu": wl.batch, "tau": tau,
                       "oracle_steps_timed": done, "wall_s": el},
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
