"""R-SWA with the window kept in a ring of pages (bounded cache memory).

The Unlimited OCR page's R-SWA attends the global prefix [0, L_m) plus the
last n tokens, so a cache only needs L_m + n tokens of storage. The library
needs no special mode for this: `ring_block_table` maps the logical pages
past the prefix onto a ring of ceil(n / page) physical pages, the caller
writes every new token's K/V through that table, and fastocr_rswa_attend
reads only prefix and window rows.

CPU: for every cache length, every row the R-SWA attend set reads still
holds the token it should (simulated writes in token order), for aligned
and unaligned prefixes and windows. GPU: a decode that wraps the ring
several times matches the oracle on the logical cache; the never-written
slots hold NaN, so a read outside the attend set would show.
"""
import numpy as np
import pytest
import torch

import oracle.attention as A
import synth


@pytest.fixture(scope="module")
def ring_fn():
    from conftest import build_library
    build_library()
    from dynamic_sparse_kv_gb300 import ring_block_table
    return ring_block_table


def _violations(t, prefix, window, page, max_tokens):
    """Rows the R-SWA attend set reads that no longer hold their token, when
    tokens are written in order through table row t."""
    holder, bad = {}, 0
    for n_t in range(1, max_tokens + 1):
        p = n_t - 1                                            # the current token is written
        holder[(t[p // page], p % page)] = p
        for q in A.rswa_positions(n_t, prefix, window):        # every row R-SWA reads
            bad += holder[(t[q // page], q % page)] != q
    return bad


@pytest.mark.parametrize("prefix,window,page", [(32, 16, 16), (100, 40, 16), (7, 5, 4),
                                                 (64, 1, 16), (48, 0, 16), (0, 33, 8)])
def test_ring_table_keeps_every_attended_row(ring_fn, prefix, window, page):
    max_tokens = prefix + 12 * (window + page) + 3
    table, per = ring_fn(2, prefix, window, page, max_tokens, first_page=5)
    assert table.shape == (2, -(-max_tokens // page))
    assert per == -(-prefix // page) + max(1, -(-window // page))
    t = table.numpy().astype(np.int64)
    # each sequence owns exactly `per` physical pages, disjoint from the other's
    assert len(set(t[0].tolist())) == per and set(t[0].tolist()).isdisjoint(set(t[1].tolist()))
    assert t.min() == 5 and t.max() == 5 + 2 * per - 1
    for b in range(2):
        assert _violations(t[b], prefix, window, page, max_tokens) == 0
    # one ring page fewer is too few once the window spans more than a page
    if window > page:
        p0, ring = -(-prefix // page), -(-window // page) - 1
        j = np.arange(t.shape[1])
        short = np.where(j < p0, j, p0 + (j - p0) % ring)
        assert _violations(short, prefix, window, page, max_tokens) > 0


@pytest.mark.gpu
def test_rswa_ring_decode_matches_oracle(ring_fn):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dynamic_sparse_kv_gb300 import _native as N
    wl = synth.workload("rswa_b16", batch=3, layers=1, rswa_prefix=100, prompt=100,
                        rswa_window=40, steps=300)
    case = synth.make_case(wl, device="cuda")
    page = wl.page_size
    table, per = ring_fn(wl.batch, wl.rswa_prefix, wl.rswa_window, page, wl.max_tokens)
    pages = wl.batch * per
    shape = (pages, wl.kv_heads, page, wl.head_dim)
    k_ring = torch.full(shape, float("nan"), dtype=case.k_cache.dtype, device="cuda")
    v_ring = torch.full_like(k_ring, float("nan"))
    bt = table.cuda()
    seq = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    kv = N.make_kv(k_ring, v_ring, bt, seq)
    dims_h = N.fastocr_create(wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim, N.FASTOCR_DTYPE_BF16,
                              page, bt.shape[1], 0, 1)
    logical = [case.logical_kv(0, b, wl.max_tokens) for b in range(wl.batch)]

    def write(b, pos):   # token pos of sequence b into its ring slot
        pg, sl = int(table[b, pos // page]), pos % page
        k_ring[pg, :, sl] = logical[b][0][pos]
        v_ring[pg, :, sl] = logical[b][1][pos]

    for b in range(wl.batch):
        for pos in range(wl.rswa_prefix):
            write(b, pos)
    try:
        for t in range(wl.steps):
            n_t = wl.seq_len_at(t)
            for b in range(wl.batch):
                write(b, n_t - 1)
            seq.fill_(n_t)
            q = case.q_at(t)[0].contiguous()
            out = torch.empty_like(q)
            N.fastocr_rswa_attend(dims_h, q, kv, wl.rswa_prefix, wl.rswa_window, out)
            if t % 23 == 0 or t == wl.steps - 1:
                torch.cuda.synchronize()
                for b in range(wl.batch):
                    K = logical[b][0][:n_t].double().cpu().numpy()
                    V = logical[b][1][:n_t].double().cpu().numpy()
                    ref = A.rswa_attend(q[b].double().cpu().numpy(), K, V, n_t, wl.rswa_prefix,
                                        wl.rswa_window)
                    got = out[b].double().cpu().numpy()
                    assert np.isfinite(got).all(), (t, b)
                    assert np.max(np.abs(got - ref)) <= 2e-2, (t, b)
        assert N.fastocr_device_status(dims_h) == 0
    finally:
        N.fastocr_destroy(dims_h)
    # storage per sequence is bounded by the prefix and the window, not the length
    assert per * page <= wl.rswa_prefix + wl.rswa_window + 2 * page < wl.max_tokens
