"""Seeded input generator: determinism, paged layout, fixation window (no GPU)."""
import numpy as np
import torch

import oracle.attention as A
import synth


def test_same_seed_same_bytes():
    wl = synth.workload("tiny_f32")
    a, b = synth.make_case(wl), synth.make_case(wl)
    for x, y in [(a.k_cache, b.k_cache), (a.v_cache, b.v_cache), (a.q, b.q),
                 (a.block_table, b.block_table)]:
        assert torch.equal(x, y)
    c = synth.make_case(wl, seed=99)
    assert not torch.equal(a.k_cache, c.k_cache)


def test_paged_layout_roundtrip():
    wl = synth.workload("tiny_f32").with_(batch=3, page_size=4)
    case = synth.make_case(wl)
    ps = wl.page_size
    n = wl.seq_len_at(5)
    bt = case.block_table
    assert sorted(bt.flatten().tolist()) == list(range(bt.numel()))   # a permutation
    for b in range(wl.batch):
        K, V = case.logical_kv(1, b, n)
        for pos in [0, 1, ps - 1, ps, n - 1]:
            page = int(bt[b, pos // ps])
            assert torch.equal(K[pos], case.k_cache[1, page, :, pos % ps, :])
            assert torch.equal(V[pos], case.v_cache[1, page, :, pos % ps, :])


def test_fixation_window_clipped_mean():
    wl = synth.workload("tiny_f32")
    cells = torch.tensor([[0], [17], [255]])
    off, valid = synth._window_offsets(wl, cells)
    assert valid[0, 0].sum() == 4 and valid[1, 0].sum() == 9 and valid[2, 0].sum() == 4
    assert sorted(off[1, 0][valid[1, 0]].tolist()) == [0, 1, 2, 16, 17, 18, 32, 33, 34]
    # q - g is 3 * the window mean: recover it by drawing g again from the same seed
    case = synth.make_case(wl, n_steps=3)
    gen = torch.Generator().manual_seed(wl.seed)
    torch.randperm(case.block_table.numel(), generator=gen)
    torch.randn(case.k_cache.shape, generator=gen)
    torch.randn(case.v_cache.shape, generator=gen)
    g = torch.randn(case.q.shape, generator=gen)
    t, layer, h = 2, 1, 3
    K, _ = case.logical_kv(layer, 0, wl.seq_len_at(t))
    cell = int(case.fixation_cells[t, 0])
    r, c = divmod(cell, 16)
    rows = [wl.prompt + rr * 16 + cc for rr in range(r - 1, r + 2) for cc in range(c - 1, c + 2)
            if 0 <= rr < 16 and 0 <= cc < 16]
    want = g[t, layer, 0, h] + 3.0 * K[rows, h // wl.group].mean(0)
    torch.testing.assert_close(case.q[t, layer, 0, h], want, rtol=1e-5, atol=1e-5)


def test_moving_fixation_is_selected():
    """Realism of the generator (not parity): the focal selection of the oracle
    covers most of the 3x3 fixation window, so a 25% keep set follows the gaze."""
    wl = synth.workload("tiny_f32")
    case = synth.make_case(wl, n_steps=8)
    hits = total = 0
    for t in range(8):
        n_t = wl.seq_len_at(t)
        K, V = case.logical_kv(1, 0, n_t)
        _, sel, _ = A.focal_attend(case.q_at(t)[1, 0].double().numpy(), K.double().numpy(),
                                   V.double().numpy(), n_t, wl.prompt, wl.n_img, wl.tau)
        off, valid = synth._window_offsets(wl, case.fixation_cells[t:t + 1])
        window = set((wl.prompt + off[0, 0][valid[0, 0]]).tolist())
        hits += len(window & set(sel.tolist()))
        total += len(window)
    assert hits / total > 0.8
