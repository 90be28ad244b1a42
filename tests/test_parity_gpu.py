"""CUDA path vs the CPU oracle on the same seeded inputs (GPU required).

Small workloads run the whole schedule (warm-up profiling, focal selection,
Cross-Step Fixation Reuse) and compare every output of every layer and step;
sizes span several 16-token tiles, ragged tails, every GQA group the kernels
support and both dtypes. Tolerances: max abs error 2e-2 for bf16 KV with
fp32 accumulation, 1e-5 for fp32; selections exact except boundary ties
within 1e-5 relative of the k-th score.
"""
import numpy as np
import pytest
import torch

import oracle.attention as A
import synth
from gpu_harness import TOL, CudaDecodeRun, KVCache, assert_close, check_selection, compare_decode, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    import dynamic_sparse_kv_gb300  # noqa: F401


def _case(name, **kw):
    return synth.make_case(synth.workload(name, **kw), device="cuda")


def test_tiny_f32_whole_decode():
    """Tiny fp32 workload, all 32 steps: layer 1 focal, layer 0 reuses F_last."""
    case = _case("tiny_f32")
    run = CudaDecodeRun(case).run(0, case.wl.steps)
    stats = compare_decode(run, case.wl.steps)
    assert stats["swaps"] == 0


@pytest.mark.parametrize("variant", [
    dict(batch=2, layers=5, prompt=40, grid=(1, 16, 24), steps=14, warmup=3, n_focal=2),
    dict(batch=3, layers=4, prompt=7, grid=(1, 9, 13), steps=9, warmup=2, n_focal=2, tau=0.3),
    dict(batch=1, layers=3, prompt=64, grid=(1, 32, 32), steps=10, warmup=2, n_focal=1, tau=1.0),
], ids=["qwen_small", "ragged", "tau1"])
def test_qwen_shaped_decode(variant):
    """GQA group 7, d=128, bf16, warm-up chooses C, then steady steps."""
    case = _case("qwen7b_b1", **variant)
    run = CudaDecodeRun(case).run(0, case.wl.steps)
    compare_decode(run, case.wl.steps)


@pytest.mark.parametrize("shape", [
    dict(q_heads=10, kv_heads=10, head_dim=128),   # MHA
    dict(q_heads=16, kv_heads=2, head_dim=128),    # group 8
    dict(q_heads=8, kv_heads=2, head_dim=64),      # d 64
    dict(q_heads=6, kv_heads=3, head_dim=128, dtype="f32"),
    dict(q_heads=5, kv_heads=1, head_dim=64, dtype="f32"),
], ids=["mha", "g8", "d64", "f32_d128", "f32_g5_d64"])
def test_head_shapes(shape):
    case = _case("qwen7b_b1", batch=2, layers=3, prompt=21, grid=(1, 10, 17), steps=6,
                 warmup=2, n_focal=1, tau=0.1, **shape)
    run = CudaDecodeRun(case).run(0, case.wl.steps)
    compare_decode(run, case.wl.steps)


def test_serving_shaped_random_start():
    case = _case("serving_b32", batch=5, layers=3, prompt=37, grid=(1, 12, 20), steps=6,
                 warmup=2, n_focal=1)
    run = CudaDecodeRun(case).run(0, case.wl.steps)
    compare_decode(run, case.wl.steps)


@pytest.mark.parametrize("tau", [0.02, 0.05, 0.1, 1.0])
def test_multipage_tau_sweep(tau):
    case = _case("multipage_b8", batch=3, layers=3, prompt=20, grid=(4, 8, 8), steps=7,
                 warmup=2, n_focal=2, tau=tau)
    run = CudaDecodeRun(case).run(0, case.wl.steps)
    compare_decode(run, case.wl.steps)


def test_tau_one_equals_dense_on_gpu():
    """Invariant: with tau = 1 every layer's output equals full attention."""
    case = _case("qwen7b_b1", batch=2, layers=4, prompt=33, grid=(1, 8, 24), steps=5,
                 warmup=2, n_focal=2, tau=1.0)
    run = CudaDecodeRun(case).run(0, case.wl.steps)
    dense = CudaDecodeRun(case).run(0, case.wl.steps, kind="dense")
    for t in range(case.wl.steps):
        d = (run.outs[t].float() - dense.outs[t].float()).abs().max().item()
        assert d <= 2e-2, (t, d)
        assert set(run.sels.get(t, {}).keys()) <= set(range(case.wl.layers))


def test_rswa_small():
    """R-SWA attend set; equals full attention while T <= n."""
    wl = synth.workload("rswa_b16", batch=3, layers=2, rswa_prefix=100, prompt=100,
                        rswa_window=16, steps=40)
    case = synth.make_case(wl, device="cuda")
    run = CudaDecodeRun(case).run(0, wl.steps, kind="rswa")
    dense = CudaDecodeRun(case).run(0, wl.steps, kind="dense")
    kv = KVCache(case)
    for t in range(wl.steps):
        n_t = wl.seq_len_at(t)
        for l in range(wl.layers):
            for b in range(wl.batch):
                K, V = kv(l, b)
                ref = A.rswa_attend(np64(case.q_at(t)[l, b]), K, V, n_t, wl.rswa_prefix,
                                    wl.rswa_window)
                assert_close(run.outs[t][l, b], ref, TOL["bf16"], f"rswa t={t} l={l} b={b}")
        if t + 1 <= wl.rswa_window:
            d = (run.outs[t].float() - dense.outs[t].float()).abs().max().item()
            assert d <= 2e-2


def _direct(case, n_t, layer=0):
    from dynamic_sparse_kv_gb300 import DecodeAttention
    wl = case.wl
    dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                          img_range=case.img_range, max_img=max(wl.n_img, 1), tau=wl.tau)
    dec.set_seq_len(n_t)
    return dec


def test_constant_keys_ties_to_lowest():
    """All keys equal -> every image token ties; the lowest k positions are kept."""
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=2, layers=1, prompt=19, grid=(1, 10, 10), steps=3, tau=0.13)
    case.k_cache[:] = case.k_cache[:, :1, :1, :1, :]
    wl = case.wl
    n_t = wl.seq_len_at(2)
    dec = _direct(case, n_t)
    q = case.q_at(2)[0].contiguous()
    out = torch.empty_like(q)
    idx = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
    k = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, wl.tau, out, idx,
                           dec.stride, k)
    torch.cuda.synchronize()
    kk = A.keep_count(wl.tau, wl.n_img)
    assert k.tolist() == [kk] * wl.batch
    for b in range(wl.batch):
        assert idx[b, :kk].tolist() == list(range(wl.prompt, wl.prompt + kk))
        Kl, Vl = KVCache(case)(0, b)
        ref = A.full_attend(np64(q[b]), Kl, Vl, n_t)
        assert_close(out[b], ref, TOL["bf16"])


@pytest.mark.parametrize("pattern", ["peaked", "rising"])
def test_large_and_rising_logits(pattern):
    """Logits far apart (a near one-hot softmax) or rising along the cache (the
    running max moves again and again): full, focal and sparse outputs and the
    focal selection still match the oracle."""
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=2, layers=1, prompt=37, grid=(1, 24, 20), steps=40, tau=0.1)
    wl = case.wl
    n_t = wl.seq_len_at(39)
    q = case.q_at(39)[0].contiguous()
    if pattern == "peaked":
        q.mul_(12.0)
    else:   # scale every cached key by a factor growing with its position
        bt = case.block_table.long()
        pos = torch.arange(bt.shape[1] * wl.page_size, device="cuda", dtype=torch.float32)
        grow = (1.0 + 4.0 * pos / wl.max_tokens).to(case.k_cache.dtype)
        for b in range(wl.batch):
            for blk in range(bt.shape[1]):
                page = int(bt[b, blk])
                g = grow[blk * wl.page_size:(blk + 1) * wl.page_size]
                case.k_cache[0, page] *= g.view(1, -1, 1)
    dec = _direct(case, n_t)
    out_full, out_focal, out_sparse = (torch.empty_like(q) for _ in range(3))
    idx = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
    k = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    N.fastocr_full_attend(dec.handle, q, dec.kv[0], out_full)
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, wl.tau, out_focal, idx,
                           dec.stride, k)
    N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], case.img_range, idx, dec.stride, k,
                            out_sparse)
    torch.cuda.synchronize()
    assert dec.device_status() == 0
    kv = KVCache(case)
    for b in range(wl.batch):
        Kl, Vl = kv(0, b)
        qb = np64(q[b])
        assert_close(out_full[b], A.full_attend(qb, Kl, Vl, n_t), TOL["bf16"], f"full b={b}")
        ref_out, ref_sel, sigma = A.focal_attend(qb, Kl, Vl, n_t, wl.prompt, wl.n_img, wl.tau)
        assert_close(out_focal[b], ref_out, TOL["bf16"], f"focal b={b}")
        kk = int(k[b])
        got = idx[b, :kk].cpu().numpy()
        check_selection(got, ref_sel, sigma, wl.prompt, f"focal b={b}")
        ref_sp = A.sparse_attend(qb, Kl, Vl, n_t, wl.prompt, wl.n_img, got)
        assert_close(out_sparse[b], ref_sp, TOL["bf16"], f"sparse b={b}")


def test_adaptive_reprofiling():
    """Adaptive layer selection: the profile re-runs in 2-step windows every 7
    steps; each window re-chooses C from its own steps and F_last restarts.
    From the second window on, the first window's focal layers get queries
    that seek the text prefix, so C must change. Every output, selection and
    window's C matches the oracle's schedule with the same period."""
    import oracle.schedule as S
    from gpu_harness import oracle_inputs
    case = _case("qwen7b_b1", batch=2, layers=6, prompt=24, grid=(1, 12, 16), steps=16,
                 warmup=2, n_focal=2, tau=0.1)
    wl = case.wl
    period = 7
    _, img, q_of, kv_of, n_t_of = oracle_inputs(case, KVCache(case))
    first = S.run_decode(q_of, kv_of, n_t_of, img, wl.tau, wl.layers, wl.batch, wl.q_heads,
                         wl.warmup, warmup=wl.warmup, n_focal=wl.n_focal)["focal"]
    g = wl.q_heads // wl.kv_heads
    for l in first:
        for b in range(wl.batch):
            K, _ = case.logical_kv(l, b, wl.prompt)           # [prompt, H_kv, d]
            m = K.float().mean(0)
            u = m / m.norm(dim=-1, keepdim=True)
            case.q[period - case.step0:, l, b] = (40.0 * u).repeat_interleave(g, 0).to(case.q.dtype)
    run = CudaDecodeRun(case, period=period).run(0, wl.steps)
    compare_decode(run, wl.steps)
    hist = run.focal_history
    assert [t for t, _ in hist] == [wl.warmup - 1 + m * period for m in range(3)]
    assert hist[0][1] == tuple(first)
    assert not set(hist[1][1]) & set(first)


@pytest.mark.parametrize("focal", [(1, 2, 4), (0, 1, 2, 3)])
def test_fixed_adjacent_focal_layers_and_graph(focal):
    """Focal sets with adjacent layers (a focal layer whose selection no
    gather layer uses before the next focal layer selects again): every output
    and every selection of the whole decode matches the oracle, and a
    CUDA-graph replay of the step gives the eager step's outputs and
    selections bit for bit from the same starting selections."""
    from dynamic_sparse_kv_gb300 import CapturedStep
    case = _case("qwen7b_b1", batch=2, layers=6, prompt=24, grid=(1, 12, 16), steps=10,
                 tau=0.1, warmup=0, focal_layers=focal)
    wl = case.wl
    run = CudaDecodeRun(case).run(0, wl.steps)
    assert run.dec.launches_per_step("fastocr") == wl.layers + len(focal)
    compare_decode(run, wl.steps)
    t = wl.steps - 1
    dec = run.dec
    cap = CapturedStep(dec)
    snap = {l: (i.clone(), k.clone()) for l, (i, k) in dec.sel.items()}   # F_last included
    dec.set_seq_len(wl.seq_len_at(t))
    cap.q.copy_(case.q_at(t))
    cap.replay()
    torch.cuda.synchronize()
    got = cap.out.clone()
    got_sel = {l: (i.clone(), k.clone()) for l, (i, k) in dec.sel.items()}
    for l, (i, k) in dec.sel.items():         # the same starting selections for the eager step
        i.copy_(snap[l][0])
        k.copy_(snap[l][1])
    out2 = torch.empty_like(cap.out)
    dec.step(case.q_at(t).contiguous(), out2)
    torch.cuda.synchronize()
    assert torch.equal(out2, got)
    for l, (i, k) in dec.sel.items():
        assert torch.equal(k, got_sel[l][1]) and torch.equal(i, got_sel[l][0]), l
    assert dec.device_status() == 0


@pytest.mark.parametrize("kind,side", [("fastocr", None), ("fastocr", 0), ("dense", 0)])
def test_host_io_graph(kind, side):
    """A CapturedStep that copies its queries in from pinned host memory and
    its outputs back inside the graph (queries by the SM copy kernel, with or
    without the later layers' share on a side stream; outputs in chunks on
    another stream, overlapped with the layers) gives the device-buffer
    graph's outputs and selections bit for bit from the same starting
    selections, and re-reads its host queries at every replay."""
    from dynamic_sparse_kv_gb300 import CapturedStep
    case = _case("qwen7b_b1", batch=2, layers=6, prompt=24, grid=(1, 12, 16), steps=10,
                 tau=0.1, warmup=0, focal_layers=(1, 2, 4))
    wl = case.wl
    run = CudaDecodeRun(case).run(0, wl.steps)
    dec = run.dec
    cap = CapturedStep(dec, kind)
    io = (CapturedStep(dec, kind, host_io=True) if side is None
          else CapturedStep(dec, kind, host_io=True, side_copy_bytes=side))
    assert io.q_host.is_pinned() and io.out_host.is_pinned()
    ptrs = {l: (i.data_ptr(), k.data_ptr()) for l, (i, k) in dec.sel.items()}
    for t in (wl.steps - 1, wl.steps - 2):
        snap = dec.state_dict()
        dec.set_seq_len(wl.seq_len_at(t))
        cap.q.copy_(case.q_at(t))
        cap.replay()
        torch.cuda.synchronize()
        want = cap.out.cpu()
        want_sel = {l: (i.cpu(), k.cpu()) for l, (i, k) in dec.sel.items()}
        dec.load_state_dict(snap)   # same focal set: the graphs' buffers stay
        assert {l: (i.data_ptr(), k.data_ptr()) for l, (i, k) in dec.sel.items()} == ptrs
        io.out_host.fill_(-1.0)
        io.q_host.copy_(case.q_at(t))
        io.replay()
        torch.cuda.synchronize()
        assert torch.equal(io.out_host, want), t
        for l, (i, k) in dec.sel.items():
            assert torch.equal(k.cpu(), want_sel[l][1]) and torch.equal(i.cpu(), want_sel[l][0]), l
    assert dec.device_status() == 0


def test_host_io_graph_rswa():
    """The host-I/O captured R-SWA step (queries split between the SM copy
    and the side copy engine) gives the device-buffer graph's outputs bit for
    bit, and both match the oracle."""
    from dynamic_sparse_kv_gb300 import CapturedStep
    wl = synth.workload("rswa_b16", batch=3, layers=6, rswa_prefix=100, prompt=100,
                        rswa_window=16, steps=40)
    case = synth.make_case(wl, device="cuda")
    dec = CudaDecodeRun(case).run(0, 2, kind="rswa").dec
    cap = CapturedStep(dec, "rswa")
    io = CapturedStep(dec, "rswa", host_io=True, side_copy_bytes=0)
    kv = KVCache(case)
    for t in (wl.steps - 1, 20):
        dec.set_seq_len(wl.seq_len_at(t))
        cap.q.copy_(case.q_at(t))
        cap.replay()
        io.q_host.copy_(case.q_at(t))
        io.replay()
        torch.cuda.synchronize()
        assert torch.equal(io.out_host, cap.out.cpu()), t
        for l in (0, wl.layers - 1):
            for b in range(wl.batch):
                K, V = kv(l, b)
                ref = A.rswa_attend(np64(case.q_at(t)[l, b]), K, V, wl.seq_len_at(t),
                                    wl.rswa_prefix, wl.rswa_window)
                assert_close(io.out_host[l, b], ref, TOL["bf16"], f"t={t} l={l} b={b}")
    assert dec.device_status() == 0


def test_window_end_selection_equals_selecting_warmup():
    """Ending a profiling window by one focal call on the deepest chosen
    layer (finish_warmup(q=...) after profile-only steps) gives the same C,
    the same image mass and the same F_last, bit for bit, as warm-up steps that
    select in every layer and take F_last from the last of them."""
    from dynamic_sparse_kv_gb300 import DecodeAttention
    case = _case("qwen7b_b1", batch=3, layers=5, prompt=24, grid=(1, 12, 16), steps=12,
                 warmup=4, n_focal=2, tau=0.1)
    wl = case.wl
    res = []
    for select in (True, False):
        dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                              img_range=case.img_range, max_img=wl.n_img, tau=wl.tau)
        dec.begin_warmup()
        for t in range(wl.warmup):
            dec.set_seq_len(wl.seq_len_at(t))
            q = case.q_at(t).contiguous()
            dec.warmup_step(q, torch.empty_like(q), select=select)
        focal, mass = dec.finish_warmup(wl.n_focal, q=None if select else q)
        idx, k = dec.sel[max(focal)]
        res.append((focal, mass, idx.cpu(), k.cpu()))
        assert dec.device_status() == 0
        dec.close()
    (f1, m1, i1, k1), (f2, m2, i2, k2) = res
    assert f1 == f2
    assert np.allclose(m1, m2, rtol=1e-6, atol=0)   # the two paths sum the mass differently
    assert torch.equal(k1, k2)
    for b in range(wl.batch):
        assert torch.equal(i1[b, :int(k1[b])], i2[b, :int(k2[b])]), b


def test_checkpoint_resume():
    """The method's state saved mid-warm-up and again in the steady decode and
    loaded into fresh decoders: the resumed decode gives the same outputs and
    selections as the uninterrupted one, bit for bit, and both match the
    oracle. The profiler's mass, the warm-up selections, C and F_last are what
    carry over."""
    case = _case("qwen7b_b1", batch=2, layers=5, prompt=24, grid=(1, 12, 16), steps=14,
                 warmup=4, n_focal=2, tau=0.1)
    wl = case.wl
    whole = CudaDecodeRun(case).run(0, wl.steps)
    t1, t2 = 2, 9                                  # inside the warm-up; steady decode
    part = CudaDecodeRun(case).run(0, t1)
    st = part.dec.state_dict()
    assert st["warm"] is not None and st["focal"] == ()
    assert len(st["warm"][2]) == wl.layers and all(m > 0 for m in st["warm"][2])
    part.dec.close()
    res = CudaDecodeRun(case)
    res.dec.load_state_dict(st)
    res.run(t1, t2)
    st2 = res.dec.state_dict()
    assert st2["focal"] == whole.focal and st2["has_f_last"]
    res.dec.close()
    res2 = CudaDecodeRun(case)
    res2.dec.load_state_dict(st2)
    res2.focal = tuple(st2["focal"])
    res2.run(t2, wl.steps)
    for t in range(wl.steps):
        got = (part if t < t1 else res if t < t2 else res2)
        assert torch.equal(got.outs[t], whole.outs[t]), f"step {t}"
        assert (t in got.sels) == (t in whole.sels), t   # warm-up: only a window's last step selects
        for l, sel in whole.sels.get(t, {}).items():
            for b in range(wl.batch):
                assert np.array_equal(got.sels[t][l][b], sel[b]), f"step {t} layer {l} seq {b}"
    compare_decode(whole, wl.steps)
    with pytest.raises(ValueError):
        bad = CudaDecodeRun(case, tau=0.2)
        bad.dec.load_state_dict(st2)


VARIANTS = {"auto": None, "general": 1, "deep": 2}


def _variants(name):
    v = VARIANTS[name]
    return None if v is None else {0: v, 1: v, 2: v}


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("splits", [None, {0: 5, 1: 4, 2: 5}], ids=["auto", "forced"])
def test_ragged_batch(splits, variant):
    """One launch over sequences that differ in cache length, image position,
    image count (hence k) and R-SWA window position -- as in a continuously
    batched server: every sequence matches the oracle run on its own. Forced
    split counts also give some CTAs of the short sequences little or nothing
    to stream."""
    from dynamic_sparse_kv_gb300 import DecodeAttention
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=4, layers=1, prompt=40, grid=(1, 16, 20), steps=70, tau=0.07)
    wl = case.wl
    n_max = wl.seq_len_at(69)                       # 430
    n_ts = [n_max, n_max - 17, wl.prompt + wl.n_img + 1, n_max - 35]
    ranges = [(40, 320), (23, 300), (40, 250), (0, 320)]   # (start, N_img), inside [0, N_t)
    prefix, window = 100, 24
    dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                          img_range=case.img_range, max_img=wl.n_img, tau=wl.tau, splits=splits,
                          variants=_variants(variant))
    dec.set_seq_len(n_max)                          # length hint: the longest sequence
    dec.set_seq_len(torch.tensor(n_ts, dtype=torch.int32, device="cuda"))
    img = torch.tensor(ranges, dtype=torch.int32, device="cuda")
    q = case.q_at(69)[0].contiguous()
    out_full, out_focal, out_sparse, out_rswa = (torch.empty_like(q) for _ in range(4))
    idx = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
    k = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    N.fastocr_full_attend(dec.handle, q, dec.kv[0], out_full)
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], img, wl.tau, out_focal, idx, dec.stride, k)
    N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], img, idx, dec.stride, k, out_sparse)
    N.fastocr_rswa_attend(dec.handle, q, dec.kv[0], prefix, window, out_rswa)
    torch.cuda.synchronize()
    assert dec.device_status() == 0
    kv = KVCache(case)
    for b, (n_t, (start, n_img)) in enumerate(zip(n_ts, ranges)):
        Kl, Vl = kv(0, b)
        qb = np64(q[b])
        assert_close(out_full[b], A.full_attend(qb, Kl, Vl, n_t), TOL["bf16"], f"full b={b}")
        ref_out, ref_sel, sigma = A.focal_attend(qb, Kl, Vl, n_t, start, n_img, wl.tau)
        assert_close(out_focal[b], ref_out, TOL["bf16"], f"focal b={b}")
        kk = int(k[b])
        assert kk == A.keep_count(wl.tau, n_img)
        got = idx[b, :kk].cpu().numpy()
        check_selection(got, ref_sel, sigma, start, f"focal b={b}")
        assert_close(out_sparse[b], A.sparse_attend(qb, Kl, Vl, n_t, start, n_img, got),
                     TOL["bf16"], f"sparse b={b}")
        assert_close(out_rswa[b], A.rswa_attend(qb, Kl, Vl, n_t, prefix, window), TOL["bf16"],
                     f"rswa b={b}")
    dec.close()


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("splits", [None, {0: 16, 1: 16, 2: 16}], ids=["auto", "split16"])
def test_degenerate_lengths(splits, variant):
    """Edge cases in one launch: a cache of only the current token, an image
    range that is empty, starts at N_t, or holds the current token (which a
    gather layer then attends only if it was selected), and -- with 16
    splits -- CTAs that have nothing at all to stream."""
    from dynamic_sparse_kv_gb300 import DecodeAttention
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=6, layers=1, prompt=16, grid=(1, 4, 8), steps=8, tau=0.5)
    wl = case.wl
    n_ts = [1, 2, 17, 1, 40, 3]
    ranges = [(0, 0), (0, 2), (16, 0), (1, 0), (5, 30), (0, 3)]
    prefix, window = 100, 24
    dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                          img_range=case.img_range, max_img=wl.n_img, tau=wl.tau, splits=splits,
                          variants=_variants(variant))
    dec.set_seq_len(max(n_ts))
    dec.set_seq_len(torch.tensor(n_ts, dtype=torch.int32, device="cuda"))
    img = torch.tensor(ranges, dtype=torch.int32, device="cuda")
    q = case.q_at(0)[0].contiguous()
    out_full, out_focal, out_sparse, out_rswa = (torch.full_like(q, 7.0) for _ in range(4))
    idx = torch.full((wl.batch, dec.stride), -5, dtype=torch.int32, device="cuda")
    k = torch.full((wl.batch,), -5, dtype=torch.int32, device="cuda")
    N.fastocr_full_attend(dec.handle, q, dec.kv[0], out_full)
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], img, wl.tau, out_focal, idx, dec.stride, k)
    N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], img, idx, dec.stride, k, out_sparse)
    N.fastocr_rswa_attend(dec.handle, q, dec.kv[0], prefix, window, out_rswa)
    torch.cuda.synchronize()
    assert dec.device_status() == 0
    kv = KVCache(case)
    for b, (n_t, (start, n_img)) in enumerate(zip(n_ts, ranges)):
        Kl, Vl = kv(0, b)
        qb = np64(q[b])
        assert_close(out_full[b], A.full_attend(qb, Kl, Vl, n_t), TOL["bf16"], f"full b={b}")
        ref_out, ref_sel, sigma = A.focal_attend(qb, Kl, Vl, n_t, start, n_img, wl.tau)
        assert_close(out_focal[b], ref_out, TOL["bf16"], f"focal b={b}")
        kk = int(k[b])
        assert kk == A.keep_count(wl.tau, n_img) == len(ref_sel)
        got = idx[b, :kk].cpu().numpy()
        check_selection(got, ref_sel, sigma, start, f"focal b={b}")
        assert_close(out_sparse[b], A.sparse_attend(qb, Kl, Vl, n_t, start, n_img, got),
                     TOL["bf16"], f"sparse b={b}")
        assert_close(out_rswa[b], A.rswa_attend(qb, Kl, Vl, n_t, prefix, window), TOL["bf16"],
                     f"rswa b={b}")
    dec.close()


def test_sparse_selection_permutation_and_empty():
    """Gather order does not matter; an empty attend list gives zeros."""
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=2, layers=1, prompt=0, grid=(1, 8, 8), steps=3)
    wl = case.wl
    n_img = wl.n_img
    rng = np.random.default_rng(0)
    sel = np.sort(rng.choice(n_img, 9, replace=False))
    dec = _direct(case, wl.seq_len_at(1))
    q = case.q_at(1)[0].contiguous()
    outs = []
    for order in (sel, sel[::-1].copy()):
        idx = torch.tensor(np.tile(order, (wl.batch, 1)), dtype=torch.int32, device="cuda")
        kk = torch.full((wl.batch,), len(order), dtype=torch.int32, device="cuda")
        out = torch.empty_like(q)
        N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], case.img_range, idx, idx.shape[1], kk,
                                out)
        outs.append(out)
    torch.cuda.synchronize()
    for b in range(wl.batch):
        Kl, Vl = KVCache(case)(0, b)
        ref = A.sparse_attend(np64(q[b]), Kl, Vl, wl.seq_len_at(1), 0, n_img, sel)
        assert_close(outs[0][b], ref, TOL["bf16"])
        assert_close(outs[1][b], ref, TOL["bf16"])
    # empty: no prefix, no selection, no generated tokens (seq_len = image end)
    dec.set_seq_len(n_img)
    idx = torch.zeros(wl.batch, 1, dtype=torch.int32, device="cuda")
    kk = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    out = torch.full_like(q, 7.0)
    N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], case.img_range, idx, 1, kk, out)
    torch.cuda.synchronize()
    assert out.abs().max().item() == 0.0
    assert dec.device_status() == 0


def test_device_status_flags_bad_inputs():
    """Bad page ids, lengths and selections are masked and reported, never fault."""
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=2, layers=1, prompt=16, grid=(1, 8, 8), steps=4)
    wl = case.wl
    dec = _direct(case, wl.seq_len_at(1))
    q = case.q_at(1)[0].contiguous()
    out = torch.empty_like(q)
    bt = dec.block_table
    saved = bt[1, 2].item()
    bt[1, 2] = dec.num_pages + 5
    N.fastocr_full_attend(dec.handle, q, dec.kv[0], out)
    assert dec.device_status() & N.DEV_BAD_PAGE
    bt[1, 2] = saved
    dec.set_seq_len(bt.shape[1] * wl.page_size + 3)
    N.fastocr_full_attend(dec.handle, q, dec.kv[0], out)
    assert dec.device_status() & N.DEV_BAD_SEQLEN
    dec.set_seq_len(wl.seq_len_at(1))
    idx = torch.tensor([[2, 20, 30], [17, 18, 9999]], dtype=torch.int32, device="cuda")
    kk = torch.tensor([3, 3], dtype=torch.int32, device="cuda")
    N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], case.img_range, idx, 3, kk, out)
    assert dec.device_status() & N.DEV_BAD_SELECTION
    kk = torch.tensor([3, 500], dtype=torch.int32, device="cuda")
    N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], case.img_range, idx, 3, kk, out)
    assert dec.device_status() & N.DEV_BAD_SELECTION
    N.fastocr_full_attend(dec.handle, q, dec.kv[0], out)
    assert dec.device_status() == 0


def test_host_argument_errors():
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=1, layers=1, prompt=16, grid=(1, 8, 8), steps=2)
    dec = _direct(case, case.wl.seq_len_at(0))
    q = case.q_at(0)[0].contiguous()
    out = torch.empty_like(q)
    idx = torch.zeros(1, dec.stride, dtype=torch.int32, device="cuda")
    k = torch.zeros(1, dtype=torch.int32, device="cuda")
    for tau in (0.0, -0.1, 1.5, float("nan")):
        with pytest.raises(N.FastOCRError) as e:
            N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, tau, out, idx,
                                   dec.stride, k)
        assert e.value.status == N.FASTOCR_ERR_INVALID
    with pytest.raises(N.FastOCRError) as e:
        N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, 1.0, out, idx, 1, k)
    assert e.value.status == N.FASTOCR_ERR_INVALID
    with pytest.raises(N.FastOCRError) as e:
        N.fastocr_full_attend(dec.handle, q.view(-1)[1:], dec.kv[0], out)
    assert e.value.status == N.FASTOCR_ERR_ALIGN
    with pytest.raises(N.FastOCRError) as e:
        N.fastocr_rswa_attend(dec.handle, q, dec.kv[0], -1, 4, out)
    assert e.value.status == N.FASTOCR_ERR_INVALID
    with pytest.raises(N.FastOCRError) as e:
        N.fastocr_set_length_hint(dec.handle, -5)
    assert e.value.status == N.FASTOCR_ERR_INVALID
    with pytest.raises(N.FastOCRError) as e:
        N.fastocr_set_splits(dec.handle, 3, 2)
    assert e.value.status == N.FASTOCR_ERR_INVALID
    for mode, variant in ((3, 1), (0, 3), (1, -1)):
        with pytest.raises(N.FastOCRError) as e:
            N.fastocr_set_variant(dec.handle, mode, variant)
        assert e.value.status == N.FASTOCR_ERR_INVALID
    sigma = torch.zeros(1, case.wl.n_img, dtype=torch.float32, device="cuda")
    with pytest.raises(N.FastOCRError) as e:   # score rows narrower than the image
        N.fastocr_focal_scores(dec.handle, q, dec.kv[0], case.img_range, out, sigma,
                               case.wl.n_img - 1)
    assert e.value.status == N.FASTOCR_ERR_INVALID
    with pytest.raises(N.FastOCRError) as e:
        N.fastocr_select(dec.handle, dec.kv[0], case.img_range, sigma, case.wl.n_img, 0.0, idx,
                         dec.stride, k)
    assert e.value.status == N.FASTOCR_ERR_INVALID
    for flags in (4, 0x80000000, 3):   # FINAL and PENDING exclude each other; no other bits
        with pytest.raises(N.FastOCRError) as e:
            N.fastocr_sparse_attend_ex(dec.handle, q, dec.kv[0], case.img_range, idx, dec.stride,
                                       k, out, flags)
        assert e.value.status == N.FASTOCR_ERR_INVALID


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_selection_final_flag(variant):
    """A gather call told that its selection is final (FASTOCR_SELECTION_FINAL:
    written before the previous kernel began) or pending (FASTOCR_SELECTION_
    PENDING: laid out only after the wait) gives the same outputs, bit for
    bit, as the call that stages it early and checks it after its wait, and
    reports bad entries the same way."""
    from dynamic_sparse_kv_gb300 import DecodeAttention
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=3, layers=1, prompt=40, grid=(1, 24, 24), steps=20, tau=0.1)
    wl = case.wl
    n_t = wl.seq_len_at(19)
    dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                          img_range=case.img_range, max_img=wl.n_img, tau=wl.tau,
                          variants=_variants(variant))
    dec.set_seq_len(n_t)
    q = case.q_at(19)[0].contiguous()
    idx = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
    k = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    out_f = torch.empty_like(q)
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, wl.tau, out_f, idx,
                           dec.stride, k)
    torch.cuda.synchronize()
    outs = []
    for flags in (0, N.SELECTION_FINAL, N.SELECTION_PENDING):
        o = torch.empty_like(q)
        N.fastocr_sparse_attend_ex(dec.handle, q, dec.kv[0], case.img_range, idx, dec.stride, k,
                                   o, flags)
        torch.cuda.synchronize()
        outs.append(o)
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    assert dec.device_status() == 0
    kv = KVCache(case)
    for b in range(wl.batch):
        Kl, Vl = kv(0, b)
        sel = idx[b, :int(k[b])].cpu().numpy()
        ref = A.sparse_attend(np64(q[b]), Kl, Vl, n_t, wl.prompt, wl.n_img, sel)
        assert_close(outs[1][b], ref, TOL["bf16"], f"final b={b}")
    bad = idx.clone()
    bad[0, 0] = wl.prompt - 1                 # outside the image range
    for flags in (0, N.SELECTION_FINAL, N.SELECTION_PENDING):
        o = torch.empty_like(q)
        N.fastocr_sparse_attend_ex(dec.handle, q, dec.kv[0], case.img_range, bad, dec.stride, k,
                                   o, flags)
        assert dec.device_status() & N.DEV_BAD_SELECTION


def test_read_probe_reads_every_word():
    """The bandwidth probe runs on a large buffer and touches every word: its
    device time scales with the bytes it is given."""
    from dynamic_sparse_kv_gb300 import _native as N
    buf = torch.ones(1 << 30, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    times = {}
    for n in (1 << 28, 1 << 30):
        N.fastocr_read_probe(buf, n, sink)          # warm
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        N.fastocr_read_probe(buf, n, sink)
        e.record()
        torch.cuda.synchronize()
        times[n] = s.elapsed_time(e)
    assert times[1 << 30] > 2.0 * times[1 << 28]   # 4x the bytes takes well over 2x the time
    assert (1 << 30) / (times[1 << 30] * 1e-3) < 20e12   # below any plausible HBM rate


def test_cache_offsets_beyond_4gb():
    """One layer whose K and V caches hold 5 GiB each (327,680 pages of 4 KV
    heads x 16 tokens x 128 dims, bf16): a sequence on the last pages (row
    offsets past 4 GiB) and one whose pages alternate between both ends give
    the oracle's outputs and selection in the full, focal and gather calls."""
    from dynamic_sparse_kv_gb300 import DecodeAttention
    from dynamic_sparse_kv_gb300 import _native as N
    H_q, H_kv, d, ps, num_pages = 28, 4, 128, 16, 327680
    B, P, n_img, tau = 2, 24, 320, 0.1
    n_t = P + n_img + 37
    npg = (n_t + ps - 1) // ps
    bt = torch.zeros(B, npg, dtype=torch.int32)
    bt[0] = torch.arange(num_pages - npg, num_pages, dtype=torch.int32)
    for i in range(npg):
        bt[1, i] = 101 * i if i % 2 == 0 else num_pages - 1 - npg - 211 * i
    assert int(bt.max()) * H_kv * ps * d * 2 >= 4 << 30 and int(bt[1].min()) == 0
    k_cache = torch.empty(1, num_pages, H_kv, ps, d, dtype=torch.bfloat16, device="cuda")
    v_cache = torch.empty_like(k_cache)
    used = torch.unique(bt.flatten()).long().cuda()
    g = torch.Generator(device="cuda").manual_seed(41)
    k_cache[0, used] = torch.randn(used.numel(), H_kv, ps, d, generator=g, device="cuda").bfloat16()
    v_cache[0, used] = torch.randn(used.numel(), H_kv, ps, d, generator=g, device="cuda").bfloat16()
    q = (2.0 * torch.randn(B, H_q, d, generator=g, device="cuda")).bfloat16()
    img = torch.tensor([[P, n_img]] * B, dtype=torch.int32, device="cuda")
    dec = DecodeAttention(k_cache, v_cache, bt.cuda(), q_heads=H_q, img_range=img,
                          max_img=n_img, tau=tau)
    dec.set_seq_len(n_t)
    out_f, out_c, out_s = (torch.empty_like(q) for _ in range(3))
    idx = torch.zeros(B, dec.stride, dtype=torch.int32, device="cuda")
    k = torch.zeros(B, dtype=torch.int32, device="cuda")
    N.fastocr_full_attend(dec.handle, q, dec.kv[0], out_f)
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], img, tau, out_c, idx, dec.stride, k)
    N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], img, idx, dec.stride, k, out_s)
    torch.cuda.synchronize()
    assert dec.device_status() == 0
    for b in range(B):
        pages = k_cache[0, bt[b].long().cuda()]
        K = np64(pages.permute(0, 2, 1, 3).reshape(npg * ps, H_kv, d)[:n_t])
        pages = v_cache[0, bt[b].long().cuda()]
        V = np64(pages.permute(0, 2, 1, 3).reshape(npg * ps, H_kv, d)[:n_t])
        qb = np64(q[b])
        assert_close(out_f[b], A.full_attend(qb, K, V, n_t), TOL["bf16"], f"full b={b}")
        ref, sel, sigma = A.focal_attend(qb, K, V, n_t, P, n_img, tau)
        assert_close(out_c[b], ref, TOL["bf16"], f"focal b={b}")
        got = idx[b, :int(k[b])].cpu().numpy()
        check_selection(got, sel, sigma, P, f"selection b={b}")
        assert_close(out_s[b], A.sparse_attend(qb, K, V, n_t, P, n_img, got), TOL["bf16"],
                     f"gather b={b}")
    dec.close()


def test_sm_copy_exact_and_refuses_pageable_memory():
    """fastocr_copy moves bytes exactly between device memory and page-locked
    host memory in every direction (sizes with a ragged grid-stride tail,
    interior pointers of an allocation), and refuses pageable host memory,
    which the device cannot address, before launching anything."""
    from dynamic_sparse_kv_gb300 import _native as N
    g = torch.Generator().manual_seed(5)
    for n in (16, 4096 + 48, 3 * (1 << 20) + 16 * 777):
        src_h = torch.randint(0, 256, (n + 64,), dtype=torch.uint8, generator=g).pin_memory()
        dst_h = torch.zeros(n + 64, dtype=torch.uint8).pin_memory()
        d1 = torch.zeros(n + 64, dtype=torch.uint8, device="cuda")
        d2 = torch.zeros(n + 64, dtype=torch.uint8, device="cuda")
        N.fastocr_copy(d1[16:], src_h[32:], n)      # host -> device
        N.fastocr_copy(d2[48:], d1[16:], n)         # device -> device
        N.fastocr_copy(dst_h[16:], d2[48:], n)      # device -> host
        torch.cuda.synchronize()
        assert torch.equal(d1[16:16 + n].cpu(), src_h[32:32 + n])
        assert torch.equal(dst_h[16:16 + n], src_h[32:32 + n])
        assert int(dst_h[:16].sum()) == 0 and int(dst_h[16 + n:].sum()) == 0
    pageable = np.zeros(4096, dtype=np.uint8)
    addr = (pageable.ctypes.data + 15) // 16 * 16
    d = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    assert N.lib.fastocr_copy(d.data_ptr(), addr, 1024, None) == N.FASTOCR_ERR_INVALID
    assert N.lib.fastocr_copy(addr, d.data_ptr(), 1024, None) == N.FASTOCR_ERR_INVALID
    torch.cuda.synchronize()


def test_length_hint_changes_speed_not_results():
    """Any length hint (none, exact, far too small, far too large) gives the same
    outputs and selection up to summation order; forced split counts likewise."""
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=3, layers=1, prompt=40, grid=(1, 24, 24), steps=12, tau=0.05)
    wl = case.wl
    n_t = wl.seq_len_at(11)
    q = case.q_at(11)[0].contiguous()
    dec = _direct(case, n_t)
    kv = KVCache(case)
    for hint in (0, n_t, 1, 1 << 20):
        N.fastocr_set_length_hint(dec.handle, hint)
        out_f, out_s = torch.empty_like(q), torch.empty_like(q)
        idx = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
        k = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
        N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, wl.tau, out_f, idx,
                               dec.stride, k)
        N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], case.img_range, idx, dec.stride, k,
                                out_s)
        torch.cuda.synchronize()
        for b in range(wl.batch):
            Kl, Vl = kv(0, b)
            qb = np64(q[b])
            ref_out, ref_sel, sigma = A.focal_attend(qb, Kl, Vl, n_t, wl.prompt, wl.n_img, wl.tau)
            assert_close(out_f[b], ref_out, TOL["bf16"], f"focal hint={hint} b={b}")
            got = idx[b, :int(k[b])].cpu().numpy()
            check_selection(got, ref_sel, sigma, wl.prompt, f"hint={hint} b={b}")
            assert_close(out_s[b], A.sparse_attend(qb, Kl, Vl, n_t, wl.prompt, wl.n_img, got),
                         TOL["bf16"], f"sparse hint={hint} b={b}")
    assert dec.device_status() == 0


def test_head_sharded_focal():
    """Head-sharded focal layer on one GPU: two handles each own half of the KV
    heads (whole GQA groups, as two tensor-parallel GPUs would),
    fastocr_focal_scores gives each shard's output heads and score share, the
    shares are summed (the all-reduce) and fastocr_select picks the top k.
    Each shard's heads match the oracle's; the summed scores match the
    oracle's; the selection matches the oracle's and the unsharded call's up
    to ties within 1e-5 of the k-th score."""
    from dynamic_sparse_kv_gb300 import _native as N
    from dynamic_sparse_kv_gb300.sharded import shard_heads
    case = _case("qwen7b_b1", batch=3, layers=1, prompt=40, grid=(1, 24, 24), steps=12, tau=0.05)
    wl = case.wl
    n_t = wl.seq_len_at(11)
    q = case.q_at(11)[0].contiguous()
    dec = _direct(case, n_t)
    idx_u = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
    k_u = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    out_u = torch.empty_like(q)
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, wl.tau, out_u, idx_u,
                           dec.stride, k_u)
    sigma = torch.zeros(wl.batch, wl.n_img, dtype=torch.float32, device="cuda")
    shards = []
    for r in range(2):
        q0, q1, kv0, kv1 = shard_heads(wl.q_heads, wl.kv_heads, r, 2)
        k_s = case.k_cache[0][:, kv0:kv1].contiguous()
        v_s = case.v_cache[0][:, kv0:kv1].contiguous()
        h = N.fastocr_create(wl.batch, q1 - q0, kv1 - kv0, wl.head_dim, N.FASTOCR_DTYPE_BF16,
                             wl.page_size, dec.block_table.shape[1], wl.n_img, 1)
        kv = N.make_kv(k_s, v_s, dec.block_table, dec.seq_len)
        q_s = q[:, q0:q1].contiguous()
        out_s = torch.empty_like(q_s)
        share = torch.full((wl.batch, wl.n_img + 3), -1.0, dtype=torch.float32, device="cuda")
        N.fastocr_focal_scores(h, q_s, kv, case.img_range, out_s, share, share.shape[1])
        shards.append((h, kv, (k_s, v_s), q0, q1, out_s, share))
    for s in shards:
        sigma += s[6][:, :wl.n_img]                 # the all-reduce of two ranks
    idx = torch.full((wl.batch, dec.stride), -1, dtype=torch.int32, device="cuda")
    k = torch.full((wl.batch,), -1, dtype=torch.int32, device="cuda")
    h0, kv0_ = shards[0][0], shards[0][1]
    N.fastocr_select(h0, kv0_, case.img_range, sigma, wl.n_img, wl.tau, idx, dec.stride, k)
    torch.cuda.synchronize()
    kv = KVCache(case)
    for b in range(wl.batch):
        Kl, Vl = kv(0, b)
        qb = np64(q[b])
        ref_out, ref_sel, ref_sigma = A.focal_attend(qb, Kl, Vl, n_t, wl.prompt, wl.n_img, wl.tau)
        for (_, _, _, q0, q1, out_s, share) in shards:
            assert_close(out_s[b], ref_out[q0:q1], TOL["bf16"], f"shard heads {q0}:{q1} b={b}")
            assert (share[b, wl.n_img:] == -1.0).all()   # nothing written past N_img
        got_sigma = np64(sigma[b])
        assert np.max(np.abs(got_sigma - ref_sigma)) <= 1e-4 * np.max(ref_sigma)
        assert int(k[b]) == A.keep_count(wl.tau, wl.n_img)
        got = idx[b, :int(k[b])].cpu().numpy()
        check_selection(got, ref_sel, ref_sigma, wl.prompt, f"sharded b={b}")
        check_selection(got, idx_u[b, :int(k_u[b])].cpu().numpy(), ref_sigma, wl.prompt,
                        f"sharded vs unsharded b={b}")
    for s in shards:
        assert N.fastocr_device_status(s[0]) == 0
        N.fastocr_destroy(s[0])
    assert dec.device_status() == 0


@pytest.mark.parametrize("max_img", [300, 2048, 2049, 5000, 8192, 16384])
@pytest.mark.parametrize("pattern", ["few_values", "constant", "distinct"])
def test_select_kernel_exact(max_img, pattern):
    """The selection kernel alone (fastocr_select on caller scores) against the
    oracle's top-k, exactly: image ranges of 1 to 16384 tokens, so the
    sequence's keys are spread over 1 to 8 CTAs of a cluster; ragged sizes in
    one launch; scores with many ties (a handful of values, or all equal),
    so the k-th score's tie group crosses CTA boundaries and the lowest
    positions must win."""
    from dynamic_sparse_kv_gb300 import _native as N
    B, page = 3, 16
    sizes = [max_img, max(1, max_img - 37), max(1, max_img // 3)]
    starts = [5, 0, 17]
    n_t = max(s + n for s, n in zip(starts, sizes)) + 9
    pages = -(-n_t // page)
    h = N.fastocr_create(B, 4, 2, 64, N.FASTOCR_DTYPE_BF16, page, pages, max_img, 1)
    kc = torch.zeros(B * pages, 2, page, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    bt = torch.arange(B * pages, dtype=torch.int32, device="cuda").view(B, pages)
    seq_len = torch.full((B,), n_t, dtype=torch.int32, device="cuda")
    kv = N.make_kv(kc, vc, bt, seq_len)
    img = torch.tensor(list(zip(starts, sizes)), dtype=torch.int32, device="cuda")
    g = torch.Generator().manual_seed(max_img * 7 + len(pattern))
    if pattern == "few_values":
        sig = torch.randint(0, 5, (B, max_img), generator=g).float() * 0.25
    elif pattern == "constant":
        sig = torch.full((B, max_img), 0.5)
    else:
        sig = torch.rand(B, max_img, generator=g)
    for tau in (0.05, 0.5):
        stride = A.keep_count(tau, max_img)
        idx = torch.full((B, stride), -1, dtype=torch.int32, device="cuda")
        k = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        N.fastocr_select(h, kv, img, sig.cuda(), max_img, tau, idx, stride, k)
        torch.cuda.synchronize()
        for b in range(B):
            n = sizes[b]
            kk = A.keep_count(tau, n)
            assert int(k[b]) == kk
            want = starts[b] + A.select_top(sig[b, :n].double().numpy(), kk)
            got = idx[b, :kk].cpu().numpy()
            assert np.array_equal(got, want), (max_img, pattern, tau, b)
            assert (idx[b, kk:] == -1).all()
    assert N.fastocr_device_status(h) == 0
    N.fastocr_destroy(h)


def test_score_reduce_path_whole_decode():
    """DecodeAttention with a score_reduce hook (one shard: the hook adds
    nothing) runs its focal layers as scores -> reduce -> select; the whole
    decode (warm-up, C, CSFR) matches the oracle like the one-call path."""
    case = _case("qwen7b_b1", batch=2, layers=5, prompt=40, grid=(1, 16, 24), steps=12,
                 warmup=3, n_focal=2)
    calls = []
    run = CudaDecodeRun(case)
    run.dec.score_reduce = lambda sigma: calls.append(sigma.shape)
    run.dec.sigma = torch.zeros(case.wl.batch, case.wl.n_img, dtype=torch.float32, device="cuda")
    run.run(0, case.wl.steps)
    compare_decode(run, case.wl.steps)
    assert len(calls) == 2 * (case.wl.steps - case.wl.warmup)   # two focal layers a step


@pytest.mark.parametrize("variant", ["auto", "general"])
@pytest.mark.parametrize("splits", [None, 1, 5])
@pytest.mark.parametrize("shape", [dict(), dict(q_heads=6, kv_heads=3, head_dim=128, dtype="f32")],
                         ids=["bf16_g7", "f32_g2"])
def test_profile_attend_mass(shape, splits, variant):
    """The profile-only layer (fastocr_profile_attend, the warm-up steps that
    keep no selection): its output is full attention, and the image mass it
    adds to its profiler slot is the oracle's sum over sequences and query
    heads of the image tokens' probabilities, and the mass the focal call
    adds, to within 1e-5 relative; forced split counts merge the mass over a
    cluster, in the automatic variant (deep for these small grids in bf16)
    and the general one."""
    from dynamic_sparse_kv_gb300 import DecodeAttention
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=3, layers=2, prompt=37, grid=(1, 24, 20), steps=40, tau=0.1,
                 **shape)
    wl = case.wl
    t = 35
    n_t = wl.seq_len_at(t)
    dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                          img_range=case.img_range, max_img=wl.n_img, tau=wl.tau,
                          splits={0: splits} if splits else None,
                          variants={0: N.VARIANT_GENERAL} if variant == "general" else None)
    dec.set_seq_len(n_t)
    dec.begin_warmup()                                # profiler slots zeroed
    q = case.q_at(t)[0].contiguous()
    out_p, out_f = torch.empty_like(q), torch.empty_like(q)
    idx = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
    k = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    N.fastocr_profile_attend(dec.handle, q, dec.kv[0], case.img_range, out_p, 0)
    N.fastocr_profile_attend(dec.handle, q, dec.kv[0], case.img_range, out_p, 0)   # adds again
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, wl.tau, out_f, idx,
                           dec.stride, k, profile_layer=1)
    torch.cuda.synchronize()
    assert dec.device_status() == 0
    mass = N.fastocr_profiler_read(dec.handle, 2)
    kv = KVCache(case)
    want, tol = 0.0, TOL[wl.dtype]
    for b in range(wl.batch):
        Kl, Vl = kv(0, b)
        out, probs = A.attend(np64(q[b]), Kl, Vl, A.full_positions(n_t))
        want += float(A.image_scores(probs, wl.prompt, wl.n_img).sum())
        assert_close(out_p[b], out, tol, f"profile b={b}")
        assert_close(out_f[b], out, tol, f"focal b={b}")
    assert abs(mass[0] / 2 - want) <= 1e-5 * want, (mass, want)
    assert abs(mass[1] - want) <= 1e-5 * want, (mass, want)
    dec.close()


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_variants_long_lists(variant):
    """Every kernel variant on lists longer than its row slice (several rounds
    of staging) and on gather lists whose selection spans several tiles per
    warp: full, focal, sparse and R-SWA outputs and the selection match the
    oracle."""
    from dynamic_sparse_kv_gb300 import DecodeAttention
    from dynamic_sparse_kv_gb300 import _native as N
    case = _case("qwen7b_b1", batch=2, layers=1, prompt=300, grid=(1, 40, 64), steps=900,
                 tau=0.3)
    wl = case.wl
    t = 850
    n_t = wl.seq_len_at(t)                          # 300 + 2560 + 851 tokens
    prefix, window = 1500, 700
    dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                          img_range=case.img_range, max_img=wl.n_img, tau=wl.tau,
                          variants=_variants(variant))
    dec.set_seq_len(n_t)
    q = case.q_at(t)[0].contiguous()
    out_full, out_focal, out_sparse, out_rswa = (torch.empty_like(q) for _ in range(4))
    idx = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
    k = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
    N.fastocr_full_attend(dec.handle, q, dec.kv[0], out_full)
    N.fastocr_focal_attend(dec.handle, q, dec.kv[0], case.img_range, wl.tau, out_focal, idx,
                           dec.stride, k)
    N.fastocr_sparse_attend(dec.handle, q, dec.kv[0], case.img_range, idx, dec.stride, k,
                            out_sparse)
    N.fastocr_rswa_attend(dec.handle, q, dec.kv[0], prefix, window, out_rswa)
    torch.cuda.synchronize()
    assert dec.device_status() == 0
    kv = KVCache(case)
    for b in range(wl.batch):
        Kl, Vl = kv(0, b)
        qb = np64(q[b])
        assert_close(out_full[b], A.full_attend(qb, Kl, Vl, n_t), TOL["bf16"], f"full b={b}")
        ref_out, ref_sel, sigma = A.focal_attend(qb, Kl, Vl, n_t, wl.prompt, wl.n_img, wl.tau)
        assert_close(out_focal[b], ref_out, TOL["bf16"], f"focal b={b}")
        got = idx[b, :int(k[b])].cpu().numpy()
        check_selection(got, ref_sel, sigma, wl.prompt, f"focal b={b}")
        assert_close(out_sparse[b], A.sparse_attend(qb, Kl, Vl, n_t, wl.prompt, wl.n_img, got),
                     TOL["bf16"], f"sparse b={b}")
        assert_close(out_rswa[b], A.rswa_attend(qb, Kl, Vl, n_t, prefix, window), TOL["bf16"],
                     f"rswa b={b}")
    dec.close()


@pytest.mark.parametrize("page", [1, 4, 64, 256])
def test_page_sizes(page):
    """Page sizes across the supported range (a power of two, 1..256 tokens):
    the whole FastOCR schedule and an R-SWA pass match the oracle, so block
    table lookups, slot arithmetic and pages that hold several kinds of tokens
    are right at every size."""
    case = _case("qwen7b_b1", batch=2, layers=3, prompt=21, grid=(1, 10, 17), steps=6,
                 warmup=2, n_focal=1, tau=0.1, page_size=page)
    run = CudaDecodeRun(case).run(0, case.wl.steps)
    compare_decode(run, case.wl.steps)
    wl = synth.workload("rswa_b16", batch=2, layers=1, rswa_prefix=70, prompt=70,
                        rswa_window=9, steps=30, page_size=page)
    rcase = synth.make_case(wl, device="cuda")
    rrun = CudaDecodeRun(rcase).run(0, wl.steps, kind="rswa")
    kv = KVCache(rcase)
    for t in (0, 8, 9, 29):
        n_t = wl.seq_len_at(t)
        for b in range(wl.batch):
            K, V = kv(0, b)
            ref = A.rswa_attend(np64(rcase.q_at(t)[0, b]), K, V, n_t, wl.rswa_prefix,
                                wl.rswa_window)
            assert_close(rrun.outs[t][0, b], ref, TOL["bf16"], f"rswa page={page} t={t} b={b}")
