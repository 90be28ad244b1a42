"""Plant plausible mistakes in the CPU oracle and check that a pin catches each.

The pins are only worth something if a dropped term, a wrong sign or index,
or a transposed operand in the oracle makes at least one of them fail.
"""
import math

import numpy as np
import pytest

import oracle.attention as A
import oracle.schedule as S
import oracle_pins as P

_attend = A.attend


def _attend_variant(gqa="div", scale="sqrt", use_v=True):
    def attend(q, K, V, positions):
        q, K, V = (np.asarray(x, dtype=np.float64) for x in (q, K, V))
        positions = np.asarray(positions, dtype=np.int64)
        n_q, d = q.shape
        n_kv = K.shape[1]
        group = n_q // n_kv
        out = np.zeros((n_q, d))
        probs = np.zeros((n_q, positions.size))
        if positions.size == 0:
            return out, probs
        for h in range(n_q):
            j = h // group if gqa == "div" else h % n_kv
            s = K[positions, j, :] @ q[h]
            s = s / (math.sqrt(d) if scale == "sqrt" else d)
            e = np.exp(s - s.max())
            p = e / e.sum()
            out[h] = p @ (V if use_v else K)[positions, j, :]
            probs[h] = p
        return out, probs
    return attend


def _select_ties_high(sigma, k):
    sigma = np.asarray(sigma, dtype=np.float64)
    order = sorted(range(sigma.size), key=lambda i: (-sigma[i], -i))
    return np.array(sorted(order[:k]), dtype=np.int64)


def _keep_floor(tau, n_img):
    return 0 if n_img <= 0 else min(max(int(math.floor(tau * n_img)), 1), n_img)


def _scores_image_normalised(probs_full, img_start, n_img):
    p = np.asarray(probs_full)[:, img_start:img_start + n_img]
    return (p / p.sum(axis=1, keepdims=True)).sum(axis=0)


def _scores_one_group(probs_full, img_start, n_img):
    p = np.asarray(probs_full)
    half = max(1, p.shape[0] // 2)
    return p[:half, img_start:img_start + n_img].sum(axis=0)


def _nonfocal_no_generated(n_t, img_start, n_img, selected):
    return np.concatenate([np.arange(0, min(img_start, n_t)), np.asarray(selected, dtype=np.int64)])


def _nonfocal_no_prefix(n_t, img_start, n_img, selected):
    return np.concatenate([np.asarray(selected, dtype=np.int64),
                           np.arange(img_start + n_img, n_t)])


def _rswa_window_plus_one(n_t, prefix_len, window):
    return np.concatenate([np.arange(0, min(prefix_len, n_t)),
                           np.arange(max(prefix_len, n_t - window - 1), n_t)])


def _rswa_without_current(n_t, prefix_len, window):
    return np.concatenate([np.arange(0, min(prefix_len, n_t)),
                           np.arange(max(prefix_len, n_t - 1 - window), n_t - 1)])


def _choose_lowest(ratio, n_focal):
    ratio = np.asarray(ratio)
    return tuple(sorted(sorted(range(ratio.size), key=lambda l: (ratio[l], l))[:n_focal]))


def _steady_first_focal_only(q_step, kv, n_t, img, tau, focal, f_last, accept=None):
    # mistake: later focal layers do not replace the selection
    q_step = np.asarray(q_step, dtype=np.float64)
    n_layers, batch, n_q, d = q_step.shape
    outs = np.zeros((n_layers, batch, n_q, d))
    used = [[None] * batch for _ in range(n_layers)]
    current = list(f_last)
    seen = [False] * batch
    for l in range(n_layers):
        for b in range(batch):
            K, V = kv(l, b)
            start, n_img = int(img[b][0]), int(img[b][1])
            if l in set(focal):
                out, s, _ = A.focal_attend(q_step[l, b], K, V, int(n_t[b]), start, n_img, tau)
                if not seen[b]:
                    current[b] = s
                    seen[b] = True
            elif current[b] is None:
                out = A.full_attend(q_step[l, b], K, V, int(n_t[b]))
            else:
                out = A.sparse_attend(q_step[l, b], K, V, int(n_t[b]), start, n_img, current[b])
            outs[l, b] = out
            used[l][b] = current[b]
    return outs, used, list(current)


def _accumulate_no_reset(ratio, mass, pos, warmup, batch, n_q):
    # mistake: a new profiling window keeps the previous window's mass
    return ratio + mass / (warmup * batch * n_q)


def _window_never_repeats(t, warmup, period=None):
    # mistake: the period is ignored, so the profile runs only once
    return t if t < warmup else -1


MUTATIONS = {
    "gqa_modulo": (A, "attend", _attend_variant(gqa="mod")),
    "scale_1_over_d": (A, "attend", _attend_variant(scale="d")),
    "keys_as_values": (A, "attend", _attend_variant(use_v=False)),
    "ties_to_higher_index": (A, "select_top", _select_ties_high),
    "keep_count_floor": (A, "keep_count", _keep_floor),
    "scores_normalised_over_image": (A, "image_scores", _scores_image_normalised),
    "scores_one_group_only": (A, "image_scores", _scores_one_group),
    "nonfocal_drops_generated": (A, "nonfocal_positions", _nonfocal_no_generated),
    "nonfocal_drops_prefix": (A, "nonfocal_positions", _nonfocal_no_prefix),
    "rswa_window_plus_one": (A, "rswa_positions", _rswa_window_plus_one),
    "rswa_without_current": (A, "rswa_positions", _rswa_without_current),
    "focal_choice_lowest": (S, "choose_focal_layers", _choose_lowest),
    "first_focal_not_replaced": (S, "steady_step", _steady_first_focal_only),
    "reprofile_keeps_old_mass": (S, "accumulate_ratio", _accumulate_no_reset),
    "reprofile_never_repeats": (S, "window_position", _window_never_repeats),
}


def _run_all_pins():
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin()
        except AssertionError:
            failed.append(pin.__name__)
    return failed


def test_pins_pass_unmutated():
    assert _run_all_pins() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    module, attr, bad = MUTATIONS[name]
    monkeypatch.setattr(module, attr, bad)
    failed = _run_all_pins()
    assert failed, f"planted mistake {name!r} passed every pin"
