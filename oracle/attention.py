"""Per-layer decode attention of FastOCR and of R-SWA, in plain fp64 NumPy.

TEST INFRASTRUCTURE ONLY. This is the slow, obviously correct statement of
what the CUDA path must compute. Only tests, the smoke check and the CPU
baseline leg of the benchmark may import it; the product never does.

Every function works on one sequence and on the *logical* cache (token order),
K and V shaped [N, H_kv, d]; paging is a storage detail of the GPU path.

Sources (FastOCR: Dynamic Visual Fixation via KV Cache Pruning for Efficient
Document Parsing, technical summaries on gist.science (ko, fr), and its
abstract; Unlimited OCR summary on my-wiki-6fu.pages.dev):

* Focal-Guided Pruning, "Cross-Layer Propagation": focal layers attend to the
  whole KV cache and pick the top-attended image tokens at keep ratio tau;
  every non-focal layer attends only to that pruned set.
* Unlimited OCR, R-SWA paragraph: attention is limited to a global prefix
  (visual + prompt tokens) plus a causal sliding window of width n over the
  generated text.

Readings taken where the pages are silent (each is pinned by a test):

* softmax scale 1/sqrt(d); query head h reads KV head h // (H_q / H_kv);
* the image score of token i is its softmax probability in the focal layer's
  full-cache attention (denominator over the whole cache), summed over all
  query heads;
* k = ceil(tau * N_img) computed in IEEE double as ceil(tau*N_img - 1e-9),
  clamped to [1, N_img]; ties in the score go to the lower index; the
  selection is returned as absolute cache positions in ascending order;
* a non-focal layer attends to the text prefix [0, img_start), the selected
  image tokens, and the generated tokens [img_start + N_img, N_t);
* R-SWA attends to [0, L_m) and to the last n tokens of [L_m, N_t), the
  current token included;
* an empty attend set yields a zero output.
"""
from __future__ import annotations

import math

import numpy as np


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def attend(q, K, V, positions):
    """Softmax attention of one decode query over the cache rows `positions`.

    q: [H_q, d]; K, V: [N, H_kv, d]; positions: 1-D ints (the attend set A,
    any order). For query head h with KV head j = h // (H_q/H_kv):
        s_h(a) = q_h . K[a, j] / sqrt(d)
        p_h(a) = exp(s_h(a) - max_A s_h) / sum_A exp(s_h - max_A s_h)
        out_h  = sum_A p_h(a) V[a, j]
    Returns (out [H_q, d], p [H_q, |A|]) with p aligned to `positions`.
    """
    q, K, V = _f64(q), _f64(K), _f64(V)
    positions = np.asarray(positions, dtype=np.int64)
    n_q, d = q.shape
    n_kv = K.shape[1]
    group = n_q // n_kv
    out = np.zeros((n_q, d))
    probs = np.zeros((n_q, positions.size))
    if positions.size == 0:
        return out, probs
    for h in range(n_q):
        j = h // group
        keys = K[positions, j, :]
        s = keys @ q[h] / math.sqrt(d)
        e = np.exp(s - s.max())
        p = e / e.sum()
        out[h] = p @ V[positions, j, :]
        probs[h] = p
    return out, probs


def keep_count(tau: float, n_img: int) -> int:
    """k = ceil(tau * N_img) image tokens kept per focal layer (clamped to [1, N_img])."""
    if n_img <= 0:
        return 0
    k = math.ceil(float(tau) * n_img - 1e-9)
    return min(max(k, 1), n_img)


def image_scores(probs_full, img_start: int, n_img: int):
    """sigma_i = sum over all query heads of p_h(img_start + i), i in [0, N_img).

    probs_full: [H_q, N_t], probabilities of a full-cache attention indexed by
    cache position."""
    probs_full = _f64(probs_full)
    return probs_full[:, img_start:img_start + n_img].sum(axis=0)


def select_top(sigma, k: int):
    """Offsets of the k largest scores, ties to the lower offset, ascending."""
    sigma = _f64(sigma)
    order = sorted(range(sigma.size), key=lambda i: (-sigma[i], i))
    return np.array(sorted(order[:k]), dtype=np.int64)


def full_positions(n_t: int):
    return np.arange(n_t, dtype=np.int64)


def focal_attend(q, K, V, n_t: int, img_start: int, n_img: int, tau: float):
    """Focal layer: full-cache attention, head-summed image scores, top-k.

    Returns (out [H_q, d], selected absolute positions ascending, sigma [N_img])."""
    out, probs = attend(q, K, V, full_positions(n_t))
    sigma = image_scores(probs, img_start, n_img)
    sel = img_start + select_top(sigma, keep_count(tau, n_img))
    return out, sel, sigma


def nonfocal_positions(n_t: int, img_start: int, n_img: int, selected):
    """Attend set of a non-focal layer: text prefix, selected image tokens, generated tokens."""
    selected = np.asarray(selected, dtype=np.int64)
    prefix = np.arange(0, min(img_start, n_t), dtype=np.int64)
    generated = np.arange(img_start + n_img, n_t, dtype=np.int64)
    return np.concatenate([prefix, selected, generated])


def sparse_attend(q, K, V, n_t: int, img_start: int, n_img: int, selected):
    """Non-focal layer: attention over nonfocal_positions(...). Returns out [H_q, d]."""
    return attend(q, K, V, nonfocal_positions(n_t, img_start, n_img, selected))[0]


def rswa_positions(n_t: int, prefix_len: int, window: int):
    """R-SWA attend set: [0, L_m) and the last `window` tokens of [L_m, N_t)."""
    prefix = np.arange(0, min(prefix_len, n_t), dtype=np.int64)
    tail = np.arange(max(prefix_len, n_t - window), n_t, dtype=np.int64)
    return np.concatenate([prefix, tail])


def rswa_attend(q, K, V, n_t: int, prefix_len: int, window: int):
    return attend(q, K, V, rswa_positions(n_t, prefix_len, window))[0]


def full_attend(q, K, V, n_t: int):
    return attend(q, K, V, full_positions(n_t))[0]
