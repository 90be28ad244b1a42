"""Shared pieces of the GPU parity tests: run the CUDA path over a synthetic
workload, hand the same inputs to the oracle, and compare.

Selections: the GPU set must have exactly k ascending, distinct positions, and
may differ from the oracle's set only in tokens whose oracle score is within
1e-5 (relative) of the oracle's k-th score. Such a swap is a valid top-k of
the same scores, so the oracle then continues with the GPU's set (it never
takes a value from the GPU that it has not checked first).
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle.attention as A
import oracle.schedule as S

REL_BOUNDARY = 1e-5
TOL = {"bf16": 2e-2, "f32": 1e-5}


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


class KVCache:
    """Logical fp64 copies of (layer, sequence) caches for the oracle, kept in a
    small LRU (a byte budget) so full-size workloads fit in host memory."""

    def __init__(self, case, budget_bytes=3 << 30):
        self.case = case
        self.n_max = case.wl.max_tokens
        self.budget = budget_bytes
        self._memo = {}

    def __call__(self, layer: int, b: int):
        key = (layer, b)
        if key in self._memo:
            val = self._memo.pop(key)
            self._memo[key] = val
            return val
        K, V = self.case.logical_kv(layer, b, self.n_max)
        val = (np64(K), np64(V))
        self._memo[key] = val
        while len(self._memo) > 1 and sum(k.nbytes + v.nbytes for k, v in self._memo.values()) \
                > self.budget:
            self._memo.pop(next(iter(self._memo)))
        return val


def check_selection(gpu, oracle_sel, sigma, img_start, where=""):
    """Returns the number of boundary swaps; raises on anything else."""
    gpu = np.asarray(gpu, dtype=np.int64)
    oracle_sel = np.asarray(oracle_sel, dtype=np.int64)
    k = oracle_sel.size
    assert gpu.size == k, f"{where}: GPU kept {gpu.size}, oracle {k}"
    if k == 0:
        return 0
    assert np.all(np.diff(gpu) > 0), f"{where}: GPU selection not ascending/distinct"
    g, o = set(gpu.tolist()), set(oracle_sel.tolist())
    if g == o:
        return 0
    kth = np.sort(sigma)[::-1][k - 1]
    diff = sorted(g ^ o)
    for pos in diff:
        i = pos - img_start
        assert 0 <= i < sigma.size, f"{where}: position {pos} outside the image"
        assert abs(sigma[i] - kth) <= REL_BOUNDARY * abs(kth), (
            f"{where}: position {pos} (score {sigma[i]:.9g}) differs from the oracle "
            f"and is not within {REL_BOUNDARY} of the k-th score {kth:.9g}")
    return len(diff) // 2


# Largest errors seen per test: [vs the fp64 oracle, vs the oracle rounded to
# the output dtype]. The second isolates the kernels' arithmetic from the final
# rounding of the output; conftest writes the table out at the end of the
# session when FASTOCR_ERR_LOG names a file.
ERRORS: dict = {}


def _test_name() -> str:
    cur = os.environ.get("PYTEST_CURRENT_TEST", "")
    return cur.split(" ")[0] if cur else "?"


def assert_close(gpu: torch.Tensor, ref: np.ndarray, tol: float, where=""):
    got = np64(gpu)
    err = np.max(np.abs(got - ref)) if ref.size else 0.0
    assert np.isfinite(got).all(), f"{where}: non-finite GPU output"
    assert err <= tol, f"{where}: max abs error {err:.3g} > {tol}"
    rounded = torch.from_numpy(np.ascontiguousarray(ref)).to(gpu.dtype).double().numpy()
    err_r = float(np.max(np.abs(got - rounded))) if ref.size else 0.0
    # error in units of the output format's spacing (bf16: 8 significant bits,
    # fp32: 24) at the largest exact value of the same head's output row, i.e.
    # relative to the scale of that output vector
    bits = 8 if gpu.dtype == torch.bfloat16 else 24
    scale = np.max(np.abs(ref), axis=-1, keepdims=True) if ref.size else ref
    ulp = np.exp2(np.floor(np.log2(np.maximum(scale, 2.0 ** -30))) - (bits - 1))
    n_ulp = float(np.max(np.abs(got - ref) / ulp)) if ref.size else 0.0
    rec = ERRORS.setdefault(_test_name(), [0.0, 0.0, str(gpu.dtype), 0.0])
    rec[0], rec[1], rec[3] = max(rec[0], float(err)), max(rec[1], err_r), max(rec[3], n_ulp)
    return float(err)


class CudaDecodeRun:
    """Run the CUDA path step by step, keeping outputs and selections on the host."""

    def __init__(self, case, tau=None, focal_layers=None, splits=None, period=None):
        from dynamic_sparse_kv_gb300 import DecodeAttention, ProfileSchedule

        wl = case.wl
        self.case, self.wl = case, wl
        self.period = period
        self.schedule = ProfileSchedule(wl.warmup, period)
        self.focal_history = []
        self.tau = wl.tau if tau is None else tau
        self.focal_fixed = focal_layers if focal_layers is not None else wl.focal_layers
        self.dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table,
                                   q_heads=wl.q_heads, img_range=case.img_range,
                                   max_img=wl.n_img, tau=self.tau, mode=wl.mode,
                                   rswa_prefix=wl.rswa_prefix, rswa_window=wl.rswa_window,
                                   splits=splits)
        self.outs, self.sels = {}, {}
        self.focal = None
        self.mass = None

    def _selections(self, idx_of_layer):
        d = {}
        for l, (idx, k) in idx_of_layer.items():
            ki = k.cpu().tolist()
            rows = idx.cpu().numpy()
            d[l] = [rows[b, :ki[b]].astype(np.int64) for b in range(self.wl.batch)]
        return d

    def run(self, t_from: int, t_to: int, kind: str = "fastocr"):
        wl, dec = self.wl, self.dec
        for t in range(t_from, t_to):
            dec.set_seq_len(wl.seq_len_at(t))
            q = self.case.q_at(t).contiguous()
            out = torch.empty_like(q)
            if kind == "dense":
                dec.dense_step(q, out)
            elif kind == "rswa":
                dec.rswa_step(q, out)
            elif self.schedule.position(t) >= 0 and self.focal_fixed is None:
                chosen = dec.scheduled_step(t, q, out, self.schedule, wl.n_focal)
                if chosen is not None:
                    self.focal = tuple(chosen)
                    self.focal_history.append((t, self.focal))
                    # a window's end selects on its last step's queries in the
                    # deepest chosen layer only: that selection is F_last
                    d = max(self.focal)
                    self.sels[t] = self._selections({d: dec.sel[d]})
            else:
                if self.focal is None:
                    self.focal = tuple(self.focal_fixed)
                    dec.set_focal_layers(self.focal)
                dec.step(q, out)
                self.sels[t] = self._selections(dec.sel)
            self.outs[t] = out.cpu()
        torch.cuda.synchronize()
        status = dec.device_status()
        assert status == 0, f"device status {status}"
        return self


def oracle_inputs(case, kv: KVCache, batch_idx=None):
    wl = case.wl
    bsel = list(range(wl.batch)) if batch_idx is None else list(batch_idx)
    img = case.img_range.cpu().numpy()[bsel]

    def q_of(t):
        return np64(case.q_at(t))[:, bsel]

    def kv_of(t):
        return lambda l, b: kv(l, bsel[b])

    def n_t_of(t):
        return np.array([wl.seq_len_at(t)] * len(bsel))

    return bsel, img, q_of, kv_of, n_t_of


def compare_decode(run: CudaDecodeRun, steps: int, batch_idx=None, check_focal=True):
    """Oracle schedule over steps [0, steps) on sequences batch_idx, continuing
    with the GPU's (validated) selections; compare every output. Returns stats."""
    case, wl = run.case, run.wl
    kv = KVCache(case)
    bsel, img, q_of, kv_of, n_t_of = oracle_inputs(case, kv, batch_idx)
    swaps = [0]
    tol = TOL[wl.dtype]

    def accept(t, l, b, s, sigma):
        if t not in run.sels or l not in run.sels[t]:
            return s
        gpu = run.sels[t][l][bsel[b]]
        swaps[0] += check_selection(gpu, s, sigma, int(img[b][0]), f"step {t} layer {l} seq {bsel[b]}")
        return gpu

    common = (q_of, kv_of, n_t_of, img, run.tau, wl.layers, len(bsel), wl.q_heads, steps)
    if run.focal_fixed is not None:
        res = S.run_decode(*common, warmup=0, focal_layers=run.focal_fixed, accept=accept)
    elif run.period is not None:
        # re-profiled every run.period steps: every window's C must agree
        res = S.run_decode(*common, warmup=wl.warmup, n_focal=wl.n_focal, accept=accept,
                           period=run.period)
        assert res["focal_history"] == run.focal_history, (res["focal_history"],
                                                           run.focal_history)
    elif check_focal and len(bsel) == wl.batch:
        res = S.run_decode(*common, warmup=wl.warmup, n_focal=wl.n_focal, accept=accept)
        if tuple(res["focal"]) != tuple(run.focal):
            # C may differ only between layers whose profiled mass ties within rounding
            ratio = res["ratio"]
            last = np.sort(ratio)[::-1][wl.n_focal - 1]
            for l in set(res["focal"]) ^ set(run.focal):
                assert abs(ratio[l] - last) <= 1e-6 * abs(last), (res["focal"], run.focal, ratio)
            res = S.run_decode(*common, warmup=wl.warmup, focal_layers=run.focal, accept=accept)
    else:
        # a subset of the batch cannot re-derive C (a batch-wide mean): take the GPU's
        res = S.run_decode(*common, warmup=wl.warmup, focal_layers=run.focal, accept=accept)
    max_err = 0.0
    for t in range(steps):
        for l in range(wl.layers):
            for bi, b in enumerate(bsel):
                e = assert_close(run.outs[t][l, b], res["outs"][t][l, bi], tol,
                                 f"step {t} layer {l} seq {b}")
                max_err = max(max_err, e)
    return dict(max_err=max_err, swaps=swaps[0], focal=res["focal"])
