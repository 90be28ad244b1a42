"""Decode-step schedule of FastOCR in plain Python: warm-up profiling, focal
layers, Cross-Step Fixation Reuse. TEST INFRASTRUCTURE ONLY (see attention.py).

Sources (FastOCR technical summaries on gist.science, ko and fr, sections
"Focal-Guided Pruning" and "Cross-Step Fixation Reuse"):

* Focal layer selection: during a light warm-up of w decode steps the
  image-attention ratio of every layer is profiled; the few layers with the
  highest image concentration become the fixed focal set C.
* Cross-layer propagation: in every later step only layers in C attend to the
  whole cache and select; the selection is handed to the non-focal layers.
* Cross-Step Fixation Reuse: at the start of a step, non-focal layers that come
  before the first focal layer reuse F_last, the previous step's selection of
  its deepest focal layer; the selection is refined at the first focal layer.

Readings (each pinned by a test):

* warm-up steps are the first w decode steps and run full attention in every
  layer; the ratio of layer l is the image probability mass averaged over
  warm-up steps, sequences and query heads; C is shared by all sequences;
  C = the n_focal largest ratios, ties to the lower layer id;
* F_last after warm-up is the selection that the deepest layer of C makes
  in the last warm-up step;
* a non-focal layer uses the selection of the most recent focal layer of the
  same step (each focal layer replaces it), before the first focal layer F_last;
* a step with no F_last yet (no warm-up and step 0) runs the layers before the
  first focal layer on the full cache;
* selections are per sequence and shared by all heads of all non-focal layers.

Adaptive layer selection (named by both summaries' closing section as a
future direction, with no rule given): the plainest form is taken -- the
warm-up profile is re-run for the same w steps every `period` steps (steps
[m*period, m*period + w)), each window's ratio starts from zero, and at the
window's end C is chosen anew and F_last restarts from the new deepest focal
layer's selection, exactly as after the first warm-up. period None is the
published method (one window).
"""
from __future__ import annotations

import numpy as np

from . import attention as A


def choose_focal_layers(ratio, n_focal: int):
    """The n_focal layers with the largest ratio (ties: lower layer id), ascending."""
    ratio = np.asarray(ratio, dtype=np.float64)
    order = sorted(range(ratio.size), key=lambda l: (-ratio[l], l))
    return tuple(sorted(order[:n_focal]))


def warmup_step(q_step, kv, n_t, img, tau, accept=None):
    """One warm-up step: every layer attends to the whole cache.

    q_step: [L, B, H_q, d]; kv(layer, b) -> (K, V) logical [>= n_t[b], H_kv, d];
    n_t: [B]; img: [B, 2] (start, N_img).
    accept(l, b, selection, sigma) -> selection lets a caller continue with
    another valid selection of the same scores (see steady_step).
    Returns (outs [L, B, H_q, d], image mass per layer [L] summed over sequences
    and heads, selection of every layer [L][B])."""
    q_step = np.asarray(q_step, dtype=np.float64)
    n_layers, batch, n_q, d = q_step.shape
    outs = np.zeros((n_layers, batch, n_q, d))
    mass = np.zeros(n_layers)
    sel = [[None] * batch for _ in range(n_layers)]
    for l in range(n_layers):
        for b in range(batch):
            K, V = kv(l, b)
            start, n_img = int(img[b][0]), int(img[b][1])
            out, s, sigma = A.focal_attend(q_step[l, b], K, V, int(n_t[b]), start, n_img, tau)
            outs[l, b] = out
            mass[l] += sigma.sum()
            sel[l][b] = accept(l, b, s, sigma) if accept else s
    return outs, mass, sel


def steady_step(q_step, kv, n_t, img, tau, focal, f_last, accept=None):
    """One decode step after warm-up.

    focal: the focal layer ids C; f_last: [B] selections of the previous step
    (None entries: no selection yet). accept(l, b, selection, sigma), if
    given, returns the selection the step continues with: a parity test uses
    it to continue with the GPU's selection once it has checked that it is a
    valid top-k of these scores (ties within tolerance), so that one allowed
    swap at the boundary does not change every later comparison.
    Returns (outs [L, B, H_q, d],
    selection used or made by each layer [L][B], new F_last [B])."""
    q_step = np.asarray(q_step, dtype=np.float64)
    n_layers, batch, n_q, d = q_step.shape
    focal = set(int(l) for l in focal)
    outs = np.zeros((n_layers, batch, n_q, d))
    used = [[None] * batch for _ in range(n_layers)]
    current = list(f_last)
    for l in range(n_layers):
        for b in range(batch):
            K, V = kv(l, b)
            start, n_img = int(img[b][0]), int(img[b][1])
            if l in focal:
                out, s, sigma = A.focal_attend(q_step[l, b], K, V, int(n_t[b]), start, n_img, tau)
                current[b] = accept(l, b, s, sigma) if accept else s
            elif current[b] is None:
                out = A.full_attend(q_step[l, b], K, V, int(n_t[b]))
            else:
                out = A.sparse_attend(q_step[l, b], K, V, int(n_t[b]), start, n_img, current[b])
            outs[l, b] = out
            used[l][b] = current[b]
    return outs, used, list(current)


def window_position(t: int, warmup: int, period=None) -> int:
    """Position of decode step t in its profiling window, -1 for a steady step.
    Windows are [0, warmup) (period None) or [m*period, m*period + warmup)."""
    pos = t if period is None else t % period
    return pos if pos < warmup else -1


def accumulate_ratio(ratio, mass, pos: int, warmup: int, batch: int, n_q: int):
    """The window's image-attention ratio after its profiling step at window
    position pos: a window starts from zero; each step adds its image mass
    averaged over the window's steps, the sequences and the query heads."""
    base = ratio if pos > 0 else np.zeros_like(ratio)
    return base + mass / (warmup * batch * n_q)


def run_decode(q_of, kv_of, n_t_of, img, tau, n_layers, batch, n_q, steps, warmup=0,
               n_focal=3, focal_layers=None, accept=None, period=None):
    """Whole schedule over decode steps 0 .. steps-1.

    q_of(t) -> [L, B, H_q, d]; kv_of(t) -> kv(layer, b); n_t_of(t) -> [B];
    accept(t, l, b, selection, sigma) as in steady_step; period: re-profile
    every `period` steps (adaptive layer selection), None: profile once.
    Returns dict(outs=[steps] arrays, used=[steps][L][B], focal=C (the last
    chosen), ratio=[L] (of the last window), f_last, focal_history=[(step at
    which a window ended, C chosen)])."""
    if period is not None and period <= warmup:
        raise ValueError("period must exceed the profiling window")
    ratio = np.zeros(n_layers)
    focal = tuple(focal_layers) if focal_layers is not None else None
    f_last = [None] * batch
    outs, used, history = [], [], []
    for t in range(steps):
        q_step, kv, n_t = q_of(t), kv_of(t), n_t_of(t)
        acc = (lambda l, b, s, sg, t=t: accept(t, l, b, s, sg)) if accept else None
        pos = window_position(t, warmup, period)
        if pos >= 0:
            o, mass, sel = warmup_step(q_step, kv, n_t, img, tau, acc)
            ratio = accumulate_ratio(ratio, mass, pos, warmup, batch, n_q)
            outs.append(o)
            used.append([[None] * batch for _ in range(n_layers)])
            if pos == warmup - 1:
                if focal_layers is None:
                    focal = choose_focal_layers(ratio, n_focal)
                f_last = list(sel[max(focal)])
                history.append((t, focal))
        else:
            o, u, f_last = steady_step(q_step, kv, n_t, img, tau, focal, f_last, acc)
            outs.append(o)
            used.append(u)
    return dict(outs=outs, used=used, focal=focal, ratio=ratio, f_last=f_last,
                focal_history=history)
