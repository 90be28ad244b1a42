"""A plain C caller of the library (tests/abi_consumer.c), which sees only
include/fastocr.h and the CUDA runtime: it compiles and links with gcc
against the built libfastocr.so (no GPU needed), and on a GPU the full, focal
and gather outputs and the selection it writes match the fp64 oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle.attention as A

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_root() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    from conftest import build_library
    gcc = shutil.which("gcc")
    cuda = _cuda_root()
    if gcc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA toolkit is not available")
    libdir = os.path.dirname(build_library())
    exe = str(tmp_path_factory.mktemp("abi") / "abi_consumer")
    cmd = [gcc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "abi_consumer.c"), "-o", exe,
           "-L", libdir, "-lfastocr", "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_consumer_builds_against_the_header_alone(consumer):
    assert os.access(consumer, os.X_OK)


def _bf16_file(t: torch.Tensor, path: str) -> None:
    t.contiguous().view(torch.int16).cpu().numpy().tofile(path)


def _bf16_read(path: str, shape) -> torch.Tensor:
    return torch.from_numpy(np.fromfile(path, dtype=np.int16)).view(torch.bfloat16).reshape(shape)


@pytest.mark.gpu
def test_consumer_matches_oracle(consumer, tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import synth
    from gpu_harness import TOL, KVCache, assert_close, check_selection, np64
    wl = synth.workload("qwen7b_b1", batch=2, layers=1, prompt=21, grid=(1, 10, 17), steps=20,
                        tau=0.1)
    case = synth.make_case(wl, device="cuda")
    t = 15
    n_t = wl.seq_len_at(t)
    q = case.q_at(t)[0].contiguous()
    d = str(tmp_path)
    _bf16_file(q, os.path.join(d, "q.bin"))
    _bf16_file(case.k_cache[0], os.path.join(d, "k.bin"))
    _bf16_file(case.v_cache[0], os.path.join(d, "v.bin"))
    case.block_table.to(torch.int32).cpu().numpy().tofile(os.path.join(d, "bt.bin"))
    np.full(wl.batch, n_t, dtype=np.int32).tofile(os.path.join(d, "len.bin"))
    case.img_range.to(torch.int32).cpu().numpy().tofile(os.path.join(d, "img.bin"))
    num_pages, max_pages = case.k_cache.shape[1], case.block_table.shape[1]
    args = [consumer, d, wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim, wl.page_size, max_pages,
            num_pages, wl.n_img, wl.tau]
    r = subprocess.run([str(a) for a in args], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert int(open(os.path.join(d, "status.txt")).read()) == 0
    stride = int(open(os.path.join(d, "stride.txt")).read())
    assert stride == A.keep_count(wl.tau, wl.n_img)
    shape = tuple(q.shape)
    out_full = _bf16_read(os.path.join(d, "out_full.bin"), shape)
    out_focal = _bf16_read(os.path.join(d, "out_focal.bin"), shape)
    out_sparse = _bf16_read(os.path.join(d, "out_sparse.bin"), shape)
    idx = np.fromfile(os.path.join(d, "idx.bin"), dtype=np.int32).reshape(wl.batch, stride)
    kept = np.fromfile(os.path.join(d, "kept.bin"), dtype=np.int32)
    kv = KVCache(case)
    for b in range(wl.batch):
        K, V = kv(0, b)
        qb = np64(q[b])
        assert_close(out_full[b], A.full_attend(qb, K, V, n_t), TOL["bf16"], f"full b={b}")
        ref, sel, sigma = A.focal_attend(qb, K, V, n_t, wl.prompt, wl.n_img, wl.tau)
        assert_close(out_focal[b], ref, TOL["bf16"], f"focal b={b}")
        got = idx[b, :kept[b]].astype(np.int64)
        check_selection(got, sel, sigma, wl.prompt, f"selection b={b}")
        assert_close(out_sparse[b], A.sparse_attend(qb, K, V, n_t, wl.prompt, wl.n_img, got),
                     TOL["bf16"], f"gather b={b}")
