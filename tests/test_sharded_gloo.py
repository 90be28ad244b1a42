"""Head-sharded focal layers on two gloo ranks (CPU, no GPU): each rank owns
half of a sequence's KV heads (whole GQA groups), forms the image-score share
of its own query heads, the shares are summed with the library's all-reduce
callback (dynamic_sparse_kv_gb300.sharded.score_all_reduce), and each rank
selects from the sum. Checked against the unsharded oracle: every rank's
selection equals the unsharded one exactly, and the ranks' head outputs,
gathered in head order, equal the unsharded outputs of the focal layer and of
the non-focal layer that uses the selection.

The per-rank arithmetic is the oracle's, applied to the rank's heads: what is
tested is the decomposition (head partition, score all-reduce, selection from
the summed scores), the host side of the GPU path, whose kernels the GPU test
test_parity_gpu.py::test_head_sharded_focal covers.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import build_library


def shard_heads(*a):
    build_library()   # the package loads its library on import
    from dynamic_sparse_kv_gb300.sharded import shard_heads as f
    return f(*a)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case():
    import synth
    wl = synth.workload("qwen7b_b1", batch=2, layers=2, prompt=20, grid=(1, 12, 16), steps=6,
                        tau=0.1)
    return wl, synth.make_case(wl, device="cpu")


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import oracle.attention as A
    from dynamic_sparse_kv_gb300.sharded import score_all_reduce
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl, case = _case()
        q0, q1, kv0, kv1 = shard_heads(wl.q_heads, wl.kv_heads, rank, world)
        reduce = score_all_reduce()
        t = 4
        n_t = wl.seq_len_at(t)
        res = []
        for b in range(wl.batch):
            K0, V0 = (x.double().numpy() for x in case.logical_kv(0, b, n_t))
            K1, V1 = (x.double().numpy() for x in case.logical_kv(1, b, n_t))
            qs = case.q_at(t).double().numpy()
            # focal layer 1, this rank's heads: output and score share
            out_f, probs = A.attend(qs[1, b, q0:q1], K1[:, kv0:kv1], V1[:, kv0:kv1],
                                    A.full_positions(n_t))
            share = torch.from_numpy(A.image_scores(probs, wl.img_start, wl.n_img).copy())
            reduce(share)                               # sum over ranks, in place
            sel = wl.img_start + A.select_top(share.numpy(), A.keep_count(wl.tau, wl.n_img))
            # non-focal layer 0 over the selection, this rank's heads
            out_s = A.sparse_attend(qs[0, b, q0:q1], K0[:, kv0:kv1], V0[:, kv0:kv1], n_t,
                                    wl.img_start, wl.n_img, sel)
            res.append((sel, out_f, out_s))
        # gather every rank's head outputs and selections on every rank
        gathered = [None] * world
        dist.all_gather_object(gathered, (rank, q0, q1, res))
        q.put((rank, gathered))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_two_rank_head_sharded_selection_matches_unsharded_oracle():
    import oracle.attention as A
    ctx = mp.get_context("spawn")
    qu = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, qu)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(qu.get(timeout=150) for _ in range(2))
    for p in procs:
        p.join(30)
        assert p.exitcode == 0
    wl, case = _case()
    t = 4
    n_t = wl.seq_len_at(t)
    for rank in (0, 1):
        shards = sorted(got[rank], key=lambda x: x[0])
        assert [(s[1], s[2]) for s in shards] == [(0, 14), (14, 28)]
        for b in range(wl.batch):
            K0, V0 = (x.double().numpy() for x in case.logical_kv(0, b, n_t))
            K1, V1 = (x.double().numpy() for x in case.logical_kv(1, b, n_t))
            qs = case.q_at(t).double().numpy()
            ref_f, ref_sel, _ = A.focal_attend(qs[1, b], K1, V1, n_t, wl.img_start, wl.n_img,
                                               wl.tau)
            ref_s = A.sparse_attend(qs[0, b], K0, V0, n_t, wl.img_start, wl.n_img, ref_sel)
            for s in shards:                        # every rank selected the same tokens
                assert np.array_equal(s[3][b][0], ref_sel)
            out_f = np.concatenate([s[3][b][1] for s in shards])
            out_s = np.concatenate([s[3][b][2] for s in shards])
            assert np.array_equal(out_f, ref_f)     # per-head arithmetic is unchanged
            assert np.array_equal(out_s, ref_s)


@pytest.mark.parametrize("q_heads,kv_heads,world", [(28, 4, 2), (28, 4, 4), (10, 10, 3),
                                                    (16, 2, 2), (12, 3, 2)])
def test_shard_heads_partition(q_heads, kv_heads, world):
    """Ranks own disjoint, contiguous, whole GQA groups that cover every head."""
    g = q_heads // kv_heads
    parts = [shard_heads(q_heads, kv_heads, r, world) for r in range(world)]
    assert parts[0][0] == 0 and parts[-1][1] == q_heads and parts[-1][3] == kv_heads
    for (q0, q1, kv0, kv1), nxt in zip(parts, parts[1:] + [None]):
        assert q0 == kv0 * g and q1 == kv1 * g and kv1 > kv0
        if nxt:
            assert nxt[0] == q1 and nxt[2] == kv1
    sizes = [p[3] - p[2] for p in parts]
    assert max(sizes) - min(sizes) <= 1


def test_shard_heads_rejects_bad_layouts():
    with pytest.raises(ValueError):
        shard_heads(28, 4, 0, 5)        # more ranks than KV heads
    with pytest.raises(ValueError):
        shard_heads(27, 4, 0, 2)        # not a GQA layout
    with pytest.raises(ValueError):
        shard_heads(28, 4, 2, 2)        # rank out of range
