"""Pins of the CPU oracle: checks against things other than the oracle itself.

Each pin raises AssertionError on a mismatch. They read the oracle through
its modules (oracle.attention / oracle.schedule) so that the mutation tests
can plant a mistake in the oracle with monkeypatch and watch a pin fail.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle.attention as A
import oracle.schedule as S

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "attend_sets.txt")


def _rng(seed):
    return np.random.default_rng(seed)


def _sdpa(q, K, V, positions):
    """PyTorch fp64 scaled_dot_product_attention over `positions`, GQA by
    repeat_interleave of the KV heads (query head h -> KV head h // group)."""
    n_q = q.shape[0]
    group = n_q // K.shape[1]
    pos = torch.as_tensor(np.asarray(positions, dtype=np.int64))
    k = torch.as_tensor(K, dtype=torch.float64)[pos].permute(1, 0, 2)    # [H_kv, n, d]
    v = torch.as_tensor(V, dtype=torch.float64)[pos].permute(1, 0, 2)
    k = k.repeat_interleave(group, dim=0)[None]
    v = v.repeat_interleave(group, dim=0)[None]
    qq = torch.as_tensor(q, dtype=torch.float64)[None, :, None, :]        # [1, H_q, 1, d]
    return F.scaled_dot_product_attention(qq, k, v)[0, :, 0, :].numpy()


def read_golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            mode, params, expected = [x.strip() for x in line.split("|")]
            kv = {}
            for tok in params.split():
                key, val = tok.split("=")
                kv[key] = val
            cases.append((mode, kv, [int(x) for x in expected.split(",")]))
    return cases


# ---------------------------------------------------------------- attention

def pin_attend_matches_sdpa():
    """attend() == torch SDPA (fp64) for GQA shapes, arbitrary position sets;
    its probabilities == SDPA applied to one-hot values."""
    rng = _rng(11)
    for (n_q, n_kv, d, n) in [(6, 2, 16, 37), (4, 4, 8, 5), (7, 1, 32, 50), (28, 4, 128, 70)]:
        q = rng.standard_normal((n_q, d)) * 2.0
        K = rng.standard_normal((n, n_kv, d))
        V = rng.standard_normal((n, n_kv, d))
        for positions in [np.arange(n), rng.permutation(n)[: max(1, n // 3)], np.array([n - 1])]:
            out, p = A.attend(q, K, V, positions)
            np.testing.assert_allclose(out, _sdpa(q, K, V, positions), rtol=1e-12, atol=1e-12)
            m = len(positions)
            onehot = np.zeros((n, n_kv, m))
            onehot[positions, :, np.arange(m)] = 1.0
            np.testing.assert_allclose(p, _sdpa(q, K, onehot, positions), rtol=1e-12, atol=1e-13)


def pin_attend_closed_forms():
    """Constant keys -> uniform weights (out = mean V over the set);
    one position -> out = that V row; empty set -> zeros."""
    rng = _rng(12)
    n_q, n_kv, d, n = 6, 3, 8, 20
    q = rng.standard_normal((n_q, d))
    K = np.broadcast_to(rng.standard_normal((1, n_kv, d)), (n, n_kv, d)).copy()
    V = rng.standard_normal((n, n_kv, d))
    pos = np.array([0, 3, 4, 9, 19])
    out, p = A.attend(q, K, V, pos)
    for h in range(n_q):
        np.testing.assert_allclose(out[h], V[pos, h // 2].mean(axis=0), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(p, np.full((n_q, pos.size), 1.0 / pos.size), rtol=1e-13)
    Kr = rng.standard_normal((n, n_kv, d))
    out1, p1 = A.attend(q, Kr, V, [7])
    for h in range(n_q):
        np.testing.assert_allclose(out1[h], V[7, h // 2], rtol=0, atol=0)
    np.testing.assert_array_equal(p1, np.ones((n_q, 1)))
    out0, p0 = A.attend(q, Kr, V, np.array([], dtype=np.int64))
    assert out0.shape == (n_q, d) and not out0.any() and p0.shape == (n_q, 0)


def pin_gather_order_invariant():
    """The attend set is a set: permuting its order leaves the output unchanged."""
    rng = _rng(13)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((30, 2, 16))
    V = rng.standard_normal((30, 2, 16))
    pos = rng.permutation(30)[:17]
    a, _ = A.attend(q, K, V, pos)
    b, _ = A.attend(q, K, V, pos[::-1].copy())
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- selection

def pin_select_exhaustive():
    """select_top == the unique k-subset in which every kept token beats every
    dropped one (higher score, or equal score and lower index), found by
    trying all k-subsets."""
    rng = _rng(14)
    for trial in range(60):
        n = int(rng.integers(1, 9))
        sigma = rng.choice([0.0, 0.25, 0.5, 0.75, 1.0], size=n) if trial % 2 else rng.random(n)
        for k in range(0, n + 1):
            found = []
            for sub in itertools.combinations(range(n), k):
                kept = set(sub)
                ok = all((sigma[i] > sigma[j]) or (sigma[i] == sigma[j] and i < j)
                         for i in kept for j in range(n) if j not in kept)
                if ok:
                    found.append(list(sub))
            assert len(found) == 1
            np.testing.assert_array_equal(A.select_top(sigma, k), np.array(found[0]))


def pin_keep_counts():
    for mode, kv, expected in read_golden():
        if mode == "keep":
            assert A.keep_count(float(kv["tau"]), int(kv["n_img"])) == expected[0], (kv, expected)


def pin_image_scores():
    """Scores are probabilities of the full-cache softmax summed over ALL query
    heads: constant keys -> every image token scores H_q / N_t; a head that
    puts (almost) all its mass on one image token adds ~1 to that token only."""
    rng = _rng(15)
    n_q, n_kv, d = 8, 2, 16
    P, n_img, n_t = 5, 12, 23
    K = np.broadcast_to(rng.standard_normal((1, n_kv, d)), (n_t, n_kv, d)).copy()
    V = rng.standard_normal((n_t, n_kv, d))
    q = rng.standard_normal((n_q, d))
    _, sel, sigma = A.focal_attend(q, K, V, n_t, P, n_img, 0.25)
    np.testing.assert_allclose(sigma, np.full(n_img, n_q / n_t), rtol=1e-12)
    np.testing.assert_array_equal(sel, P + np.arange(3))            # all tied -> lowest
    # head h stares at image token t_h (distinct per head, across both groups)
    K = rng.standard_normal((n_t, n_kv, d)) * 0.01
    q = np.zeros((n_q, d))
    targets = [P + 2 * h % n_img for h in range(n_q)]
    for h in range(n_q):
        j = h // (n_q // n_kv)
        u = np.zeros(d)
        u[h] = 1.0
        K[targets[h], j] = u
        q[h] = 60.0 * math.sqrt(d) * u
    _, sel, sigma = A.focal_attend(q, K, V, n_t, P, n_img, 1.0)
    expect = np.zeros(n_img)
    for h in range(n_q):
        expect[targets[h] - P] += 1.0
    np.testing.assert_allclose(sigma, expect, atol=1e-6)


def pin_tau_one_is_full():
    """tau = 1 keeps every image token, and a non-focal layer fed that set is
    exactly full attention."""
    rng = _rng(16)
    n_q, n_kv, d, P, n_img, gen = 4, 2, 16, 6, 20, 5
    n_t = P + n_img + gen
    K = rng.standard_normal((n_t, n_kv, d))
    V = rng.standard_normal((n_t, n_kv, d))
    q = rng.standard_normal((n_q, d))
    out_f, sel, _ = A.focal_attend(q, K, V, n_t, P, n_img, 1.0)
    np.testing.assert_array_equal(sel, np.arange(P, P + n_img))
    np.testing.assert_allclose(A.sparse_attend(q, K, V, n_t, P, n_img, sel), out_f, rtol=1e-12,
                               atol=1e-13)
    np.testing.assert_allclose(out_f, _sdpa(q, K, V, np.arange(n_t)), rtol=1e-12, atol=1e-13)


def _attend_set_via_onehot(fn, n_t, **kw):
    """Run `fn` with constant keys and V[a] = e_a: out = indicator(set)/|set|."""
    n_kv, d = 1, max(n_t, 1)
    K = np.ones((n_t, n_kv, d))
    V = np.zeros((n_t, n_kv, d))
    V[np.arange(n_t), 0, np.arange(n_t)] = 1.0
    q = np.ones((2, d))
    out = fn(q, K, V, n_t, **kw)
    support = np.nonzero(out[0] > 1e-12)[0]
    if support.size:
        np.testing.assert_allclose(out[0, support], 1.0 / support.size, rtol=1e-12)
    return support.tolist()


def pin_attend_sets_golden():
    """Non-focal and R-SWA attend sets == the hand-worked cases."""
    for mode, kv, expected in read_golden():
        n_t = int(kv["n_t"]) if "n_t" in kv else None
        if mode == "nonfocal":
            sel = [int(x) for x in kv["selected"].split(",")]
            got = _attend_set_via_onehot(A.sparse_attend, n_t, img_start=int(kv["img_start"]),
                                         n_img=int(kv["n_img"]), selected=sel)
        elif mode == "rswa":
            got = _attend_set_via_onehot(A.rswa_attend, n_t, prefix_len=int(kv["prefix"]),
                                         window=int(kv["window"]))
        else:
            continue
        assert got == expected, (mode, kv, got, expected)


def pin_rswa_short_is_full():
    """R-SWA equals full attention while the generated text fits in the window."""
    rng = _rng(17)
    n_q, n_kv, d, L_m, n = 6, 6, 16, 40, 8
    K = rng.standard_normal((L_m + n, n_kv, d))
    V = rng.standard_normal((L_m + n, n_kv, d))
    q = rng.standard_normal((n_q, d))
    for T in range(1, n + 1):
        n_t = L_m + T
        np.testing.assert_allclose(A.rswa_attend(q, K, V, n_t, L_m, n),
                                   _sdpa(q, K, V, np.arange(n_t)), rtol=1e-12, atol=1e-13)
    n_t = L_m + n + 3
    K = rng.standard_normal((n_t, n_kv, d))
    V = rng.standard_normal((n_t, n_kv, d))
    assert not np.allclose(A.rswa_attend(q, K, V, n_t, L_m, n), _sdpa(q, K, V, np.arange(n_t)))


# ---------------------------------------------------------------- schedule

def pin_focal_layer_choice():
    assert S.choose_focal_layers([0.1, 0.5, 0.5, 0.2, 0.5], 2) == (1, 2)
    assert S.choose_focal_layers([0.3, 0.1, 0.9, 0.4], 3) == (0, 2, 3)
    assert S.choose_focal_layers([1.0, 1.0, 1.0], 1) == (0,)


def _fixation_model(n_layers, onehot_layers, seed, P=3, rows=4, cols=4, gen_max=6, n_q=2):
    """Tiny decode model: layer l has random keys except that its queries point at a
    moving image cell; layers in `onehot_layers` get one-hot-coded values so their
    output reveals their attend set."""
    rng = _rng(seed)
    n_img = rows * cols
    n_max = P + n_img + gen_max
    d = n_max
    Ks, Vs = [], []
    for l in range(n_layers):
        K = rng.standard_normal((n_max, 1, d)) * 0.1
        if l in onehot_layers:
            K = np.ones((n_max, 1, d))
            V = np.zeros((n_max, 1, d))
            V[np.arange(n_max), 0, np.arange(n_max)] = 1.0
        else:
            V = rng.standard_normal((n_max, 1, d))
        Ks.append(K)
        Vs.append(V)

    def q_of(t):
        q = np.zeros((n_layers, 1, n_q, d))
        for l in range(n_layers):
            if l in onehot_layers:
                q[l, 0] = 1.0
                continue
            cell = (3 * t + l) % n_img
            key = Ks[l][P + cell, 0]
            q[l, 0] = 8.0 * key / np.linalg.norm(key)
        return q

    def kv_of(t):
        return lambda l, b: (Ks[l], Vs[l])

    def n_t_of(t):
        return np.array([P + n_img + t + 1])

    img = np.array([[P, n_img]])
    return q_of, kv_of, n_t_of, img, n_img, P


def _support(out_row):
    s = np.nonzero(out_row > 1e-12)[0]
    return s.tolist()


def pin_cross_step_reuse():
    """Layers before the first focal layer read the previous step's selection of
    the deepest focal layer (F_last); later non-focal layers read the latest
    focal selection of the same step. Checked through one-hot-valued layers
    whose output exposes their attend set."""
    n_layers, focal = 5, (1, 3)
    onehot = {0, 2, 4}
    q_of, kv_of, n_t_of, img, n_img, P = _fixation_model(n_layers, onehot, seed=21)
    res = S.run_decode(q_of, kv_of, n_t_of, img, tau=0.25, n_layers=n_layers, batch=1, n_q=2,
                       steps=4, warmup=0, focal_layers=focal)
    prev_deepest = None
    for t in range(4):
        n_t = int(n_t_of(t)[0])
        out = res["outs"][t]
        gen = list(range(P + n_img, n_t))
        sel1 = res["used"][t][1][0]
        sel3 = res["used"][t][3][0]
        # layer 0: F_last (full cache at step 0, where there is none yet)
        want0 = list(range(n_t)) if prev_deepest is None else \
            list(range(P)) + list(prev_deepest) + gen
        assert _support(out[0, 0, 0]) == want0, (t, 0)
        assert _support(out[2, 0, 0]) == list(range(P)) + list(sel1) + gen, (t, 2)
        assert _support(out[4, 0, 0]) == list(range(P)) + list(sel3) + gen, (t, 4)
        # the focal layers' selections are their own top-k of the full cache
        for l, sel in ((1, sel1), (3, sel3)):
            _, own, _ = A.focal_attend(q_of(t)[l, 0], kv_of(t)(l, 0)[0], kv_of(t)(l, 0)[1],
                                       n_t, P, n_img, 0.25)
            np.testing.assert_array_equal(sel, own)
        prev_deepest = sel3
    np.testing.assert_array_equal(res["f_last"][0], prev_deepest)


def pin_warmup_profile():
    """Warm-up ranks layers by image-attention mass: layers whose queries align
    with the image keys (image logits raised by beta_l) are chosen; F_last after
    warm-up is the deepest chosen layer's last-warm-up selection."""
    rng = _rng(22)
    n_layers, n_q, n_kv, d = 6, 4, 2, 16
    P, n_img, steps, w = 4, 16, 3, 2
    beta = [0.0, 3.0, 0.5, 2.0, 0.1, 2.5]       # image pull of each layer's queries
    n_max = P + n_img + steps
    Ks = [0.1 * rng.standard_normal((n_max, n_kv, d)) for _ in range(n_layers)]
    for K in Ks:
        K[P:P + n_img, :, 0] += 1.0                    # image keys share direction e_0
    Vs = [rng.standard_normal((n_max, n_kv, d)) for _ in range(n_layers)]

    def q_of(t):
        q = 0.05 * rng.standard_normal((n_layers, 1, n_q, d))
        for l in range(n_layers):
            q[l, 0, :, 0] += beta[l] * math.sqrt(d)
        return q

    qs = [q_of(t) for t in range(steps)]
    res = S.run_decode(lambda t: qs[t], lambda t: (lambda l, b: (Ks[l], Vs[l])),
                       lambda t: np.array([P + n_img + t + 1]), np.array([[P, n_img]]), 0.25,
                       n_layers, 1, n_q, steps, warmup=w, n_focal=3)
    assert res["focal"] == (1, 3, 5), res["ratio"]
    assert res["ratio"][1] > res["ratio"][5] > res["ratio"][3] > res["ratio"][2]
    # F_last entering step w is layer 5's selection at step w-1
    _, sel5, _ = A.focal_attend(qs[w - 1][5, 0], Ks[5], Vs[5], P + n_img + w, P, n_img, 0.25)
    n_t = P + n_img + w + 1
    out0 = res["outs"][w][0, 0]
    want = A.sparse_attend(qs[w][0, 0], Ks[0], Vs[0], n_t, P, n_img, sel5)
    np.testing.assert_allclose(out0, want, rtol=1e-12, atol=1e-13)


def pin_reprofile_windows():
    """Adaptive layer selection: a second profiling window re-chooses C from its
    own steps only (the first window's mass is not carried over) and F_last
    restarts from the new deepest focal layer's last-window selection; steady
    steps between the windows keep the first C."""
    rng = _rng(23)
    n_layers, n_q, n_kv, d = 6, 4, 2, 16
    P, n_img, w, period, steps = 4, 16, 2, 5, 9
    # window 1 pulls layers 0, 1, 3 to the image and pushes 2, 4, 5 away;
    # window 2 pulls 2, 4, 5 a little harder than 0, 1, 3 -- so the mass of
    # both windows together would still rank 0, 1, 3 first
    beta_1 = [3.0, 3.0, -3.0, 3.0, -3.0, -3.0]
    beta_2 = [1.0, 1.0, 2.0, 1.0, 2.0, 2.0]
    n_max = P + n_img + steps
    Ks = [0.1 * rng.standard_normal((n_max, n_kv, d)) for _ in range(n_layers)]
    for K in Ks:
        K[P:P + n_img, :, 0] += 1.0                    # image keys share direction e_0
    Vs = [rng.standard_normal((n_max, n_kv, d)) for _ in range(n_layers)]
    qs = []
    for t in range(steps):
        beta = beta_1 if t < period else beta_2
        q = 0.05 * rng.standard_normal((n_layers, 1, n_q, d))
        for l in range(n_layers):
            q[l, 0, :, 0] += beta[l] * math.sqrt(d)
        qs.append(q)
    kv_of = lambda t: (lambda l, b: (Ks[l], Vs[l]))  # noqa: E731
    n_t_of = lambda t: np.array([P + n_img + t + 1])  # noqa: E731
    img = np.array([[P, n_img]])
    res = S.run_decode(lambda t: qs[t], kv_of, n_t_of, img, 0.25, n_layers, 1, n_q, steps,
                       warmup=w, n_focal=3, period=period)
    assert res["focal_history"] == [(w - 1, (0, 1, 3)), (period + w - 1, (2, 4, 5))], \
        res["focal_history"]

    def sel_of(t, l):
        return A.focal_attend(qs[t][l, 0], Ks[l], Vs[l], P + n_img + t + 1, P, n_img, 0.25)[1]

    def sparse(t, l, sel):
        return A.sparse_attend(qs[t][l, 0], Ks[l], Vs[l], P + n_img + t + 1, P, n_img, sel)

    # window 2 runs full attention everywhere
    t2 = period
    for l in range(n_layers):
        np.testing.assert_allclose(res["outs"][t2][l, 0],
                                   A.full_attend(qs[t2][l, 0], Ks[l], Vs[l], P + n_img + t2 + 1),
                                   rtol=1e-12, atol=1e-13)
    # a steady step between the windows runs C = (0, 1, 3): layer 2 reads layer 1's selection
    t1 = period - 1
    np.testing.assert_allclose(res["outs"][t1][2, 0], sparse(t1, 2, sel_of(t1, 1)),
                               rtol=1e-12, atol=1e-13)
    # the first step after window 2 runs C = (2, 4, 5): layers 0 and 1 read F_last,
    # layer 5's selection in the window's last step; layer 3 reads layer 2's
    t3 = period + w
    for l in (0, 1):
        np.testing.assert_allclose(res["outs"][t3][l, 0], sparse(t3, l, sel_of(t3 - 1, 5)),
                                   rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["outs"][t3][3, 0], sparse(t3, 3, sel_of(t3, 2)),
                               rtol=1e-12, atol=1e-13)
    # no period: one window, the first C for good
    once = S.run_decode(lambda t: qs[t], kv_of, n_t_of, img, 0.25, n_layers, 1, n_q, steps,
                        warmup=w, n_focal=3)
    assert once["focal_history"] == [(w - 1, (0, 1, 3))]


ALL_PINS = [
    pin_attend_matches_sdpa, pin_attend_closed_forms, pin_gather_order_invariant,
    pin_select_exhaustive, pin_keep_counts, pin_image_scores, pin_tau_one_is_full,
    pin_attend_sets_golden, pin_rswa_short_is_full, pin_focal_layer_choice,
    pin_cross_step_reuse, pin_warmup_profile, pin_reprofile_windows,
]
