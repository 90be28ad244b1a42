"""Full-size workloads, in the launch configuration the benchmark uses (same
DecodeAttention, automatic split counts), checked against the oracle on
sampled sequences and steps (GPU required).

* qwen7b_b1: every output of every layer of the first warm-up + 3 steady steps.
* serving_b32: three of the 32 sequences, warm-up shortened to 2 steps.
* multipage_b8: two sequences near the start, and a late step (t = 4095, cache
  of ~20.5k tokens) with a fixed focal set, for tau in {0.02, 0.05, 0.1, 1}.
* rswa_b16: two sequences of every layer at T in {1024, 2048, 4096, 8192}.
"""
import numpy as np
import pytest
import torch

import oracle.attention as A
import synth
from gpu_harness import TOL, CudaDecodeRun, KVCache, assert_close, compare_decode, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()
    import dynamic_sparse_kv_gb300  # noqa: F401


def _free():
    torch.cuda.empty_cache()


def test_qwen7b_b1_full_size():
    wl = synth.workload("qwen7b_b1")
    n = wl.warmup + 3
    case = synth.make_case(wl, device="cuda", n_steps=n)
    run = CudaDecodeRun(case).run(0, n)
    stats = compare_decode(run, n)
    assert len(stats["focal"]) == 3
    del case, run
    _free()


def test_serving_b32_full_size_sampled():
    wl = synth.workload("serving_b32", warmup=2)
    n = wl.warmup + 2
    case = synth.make_case(wl, device="cuda", n_steps=n)
    run = CudaDecodeRun(case).run(0, n)
    compare_decode(run, n, batch_idx=[0, 17, 31])
    del case, run
    _free()


@pytest.mark.parametrize("tau", [0.02, 0.05, 0.1, 1.0])
def test_multipage_b8_full_size_sampled(tau):
    wl = synth.workload("multipage_b8", warmup=2, tau=tau)
    n = wl.warmup + 1
    case = synth.make_case(wl, device="cuda", n_steps=n)
    run = CudaDecodeRun(case).run(0, n)
    compare_decode(run, n, batch_idx=[0, 5])
    del case, run
    _free()


@pytest.mark.parametrize("tau", [0.05, 1.0])
def test_multipage_b8_last_step(tau):
    """The last decode step (generated text ~4k tokens), fixed focal set, no F_last:
    layers before the first focal layer see the full cache."""
    wl = synth.workload("multipage_b8", tau=tau, focal_layers=(9, 18, 27), warmup=0)
    t = wl.steps - 1
    case = synth.make_case(wl, device="cuda", step0=t, n_steps=1)
    run = CudaDecodeRun(case).run(t, t + 1)
    kv = KVCache(case)
    n_t = wl.seq_len_at(t)
    q = np64(case.q_at(t))
    for b in (0, 7):
        cur = None
        for l in range(wl.layers):
            K, V = kv(l, b)
            if l in (9, 18, 27):
                ref, sel, sigma = A.focal_attend(q[l, b], K, V, n_t, wl.prompt, wl.n_img, tau)
                from gpu_harness import check_selection
                check_selection(run.sels[t][l][b], sel, sigma, wl.prompt, f"l={l} b={b}")
                cur = run.sels[t][l][b]
            elif cur is None:
                ref = A.full_attend(q[l, b], K, V, n_t)
            else:
                ref = A.sparse_attend(q[l, b], K, V, n_t, wl.prompt, wl.n_img, cur)
            assert_close(run.outs[t][l, b], ref, TOL["bf16"], f"t={t} l={l} b={b}")
    del case, run
    _free()


@pytest.mark.parametrize("T", [1024, 2048, 4096, 8192])
def test_rswa_b16_full_size_sampled(T):
    wl = synth.workload("rswa_b16", steps=T)
    t = T - 1
    case = synth.make_case(wl, device="cuda", step0=t, n_steps=1)
    run = CudaDecodeRun(case).run(t, t + 1, kind="rswa")
    kv = KVCache(case)
    n_t = wl.seq_len_at(t)
    q = np64(case.q_at(t))
    for b in (3, 12):
        for l in range(wl.layers):
            K, V = kv(l, b)
            ref = A.rswa_attend(q[l, b], K, V, n_t, wl.rswa_prefix, wl.rswa_window)
            assert_close(run.outs[t][l, b], ref, TOL["bf16"], f"T={T} l={l} b={b}")
    del case, run
    _free()
