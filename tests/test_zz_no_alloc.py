"""The allocation-free focal entry point against the handle-based one (GPU).

fastocr_focal_attend_noalloc serves callers that may not allocate GPU memory
at the point where they run attention (code inside another framework's
memory pool, plugins that may not call cudaMalloc once started, loops that
must not take the driver's allocation locks). It keeps its scratch in a
fixed array inside the library instead of a handle's workspace. Two calls in
a row (different steps, so the second overwrites the first call's scratch)
must each give the same outputs and selection as fastocr_focal_attend, and
match the fp64 oracle on their own (outputs within the test tolerance,
selections exact up to ties within 1e-5 of the k-th score).

This file is collected last on purpose and also passes on its own.
"""
import pytest
import torch

import oracle.attention as A
import synth
from gpu_harness import KVCache, assert_close, check_selection, np64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from conftest import build_library
    build_library()


@pytest.mark.parametrize("name,overrides", [
    ("qwen7b_b1", dict(batch=2, layers=1, prompt=40, grid=(1, 16, 24), steps=6, tau=0.05)),
    ("tiny_f32", dict(steps=6)),
])
def test_noalloc_matches_handle_path(name, overrides):
    from dynamic_sparse_kv_gb300 import _native as N
    from dynamic_sparse_kv_gb300 import DecodeAttention

    wl = synth.workload(name, **overrides)
    case = synth.make_case(wl, device="cuda")
    dec = DecodeAttention(case.k_cache, case.v_cache, case.block_table, q_heads=wl.q_heads,
                          img_range=case.img_range, max_img=wl.n_img, tau=wl.tau)
    dtype = N.FASTOCR_DTYPE_BF16 if wl.dtype == "bf16" else N.FASTOCR_DTYPE_F32
    dims = N.fastocr_dims(wl.batch, wl.q_heads, wl.kv_heads, wl.head_dim, dtype, wl.page_size,
                          dec.block_table.shape[1], wl.n_img, 1)
    assert wl.batch * wl.kv_heads * wl.n_img <= N.NOALLOC_MAX_UNITS_IMG
    tol = 2e-2 if wl.dtype == "bf16" else 1e-5
    layer = wl.layers - 1
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in (2, 5):                       # two calls in a row
        dec.set_seq_len(wl.seq_len_at(t))
        N.fastocr_set_length_hint(dec.handle, 0)   # same split rule as the no-alloc call
        q = case.q_at(t)[layer].contiguous()
        out_ref, out = torch.empty_like(q), torch.full_like(q, float("nan"))
        idx_ref = torch.zeros(wl.batch, dec.stride, dtype=torch.int32, device="cuda")
        k_ref = torch.zeros(wl.batch, dtype=torch.int32, device="cuda")
        idx = torch.full_like(idx_ref, -1)
        k = torch.full_like(k_ref, -1)
        N.fastocr_focal_attend(dec.handle, q, dec.kv[layer], case.img_range, wl.tau, out_ref,
                               idx_ref, dec.stride, k_ref)
        N.fastocr_focal_attend_noalloc(dims, q, dec.kv[layer], case.img_range, wl.tau, out, idx,
                                       dec.stride, k, status)
        torch.cuda.synchronize()
        assert torch.equal(k, k_ref)
        for b in range(wl.batch):
            assert torch.equal(idx[b, :int(k[b])], idx_ref[b, :int(k_ref[b])])
        err = (out.double() - out_ref.double()).abs().max().item()
        assert err <= tol, (t, err)
        # and each call on its own against the fp64 oracle
        n_t = wl.seq_len_at(t)
        kv = KVCache(case)
        for b in range(wl.batch):
            K, V = kv(layer, b)
            ref_out, ref_sel, sigma = A.focal_attend(np64(q[b]), K, V, n_t, wl.prompt, wl.n_img,
                                                     wl.tau)
            assert_close(out[b], ref_out, tol, f"no-alloc t={t} b={b}")
            check_selection(idx[b, :int(k[b])].cpu().numpy(), ref_sel, sigma, wl.prompt,
                            f"no-alloc t={t} b={b}")
    assert int(status.item()) == 0
    assert dec.device_status() == 0
    dec.close()


def test_noalloc_rejects_oversized_problem():
    from dynamic_sparse_kv_gb300 import _native as N
    wl = synth.workload("qwen7b_b1", batch=1, layers=1, steps=2)
    case = synth.make_case(wl, device="cuda")
    dims = N.fastocr_dims(32, wl.q_heads, wl.kv_heads, wl.head_dim, N.FASTOCR_DTYPE_BF16,
                          wl.page_size, case.block_table.shape[1], wl.n_img, 1)
    assert 32 * wl.kv_heads * wl.n_img > N.NOALLOC_MAX_UNITS_IMG
    seq = torch.full((32,), wl.seq_len_at(0), dtype=torch.int32, device="cuda")
    kv = N.make_kv(case.k_cache[0], case.v_cache[0], case.block_table, seq)
    q = torch.zeros(32, wl.q_heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros(32, 256, dtype=torch.int32, device="cuda")
    k = torch.zeros(32, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    img = case.img_range.repeat(32, 1)
    with pytest.raises(N.FastOCRError) as e:
        N.fastocr_focal_attend_noalloc(dims, q, kv, img, wl.tau, q, idx, 256, k, status)
    assert e.value.status == N.FASTOCR_ERR_UNSUPPORTED
