"""bench.py's host arithmetic (no GPU): the algorithmic K/V bytes behind the
roofline's `achieved` equal the oracle's attend sets times the bytes of a
token's K and V rows, and the recorded ncu traffic is used only on the
kernel sources it was taken on."""
import numpy as np
import pytest

import bench
import oracle.attention as A
import synth


def _row_bytes(wl):
    return 2 * wl.kv_heads * wl.head_dim * (2 if wl.dtype == "bf16" else 4)


@pytest.mark.parametrize("name", ["qwen7b_b1", "serving_b32", "multipage_b8", "tiny_f32"])
def test_kv_bytes_equal_oracle_attend_sets(name):
    wl = synth.workload(name)
    rng = np.random.default_rng(3)
    for t in (wl.warmup, wl.warmup + 7, wl.steps - 1):
        n_t = wl.seq_len_at(t)
        k = A.keep_count(wl.tau, wl.n_img)
        ks = [k] * wl.batch
        full = sum(A.full_positions(n_t).size for _ in range(wl.batch)) * _row_bytes(wl)
        assert bench.kv_bytes(wl, "focal", n_t, ks) == full
        assert bench.kv_bytes(wl, "full", n_t, ks) == full
        sel = wl.img_start + np.sort(rng.choice(wl.n_img, k, replace=False))
        sparse = sum(A.nonfocal_positions(n_t, wl.img_start, wl.n_img, sel).size
                     for _ in range(wl.batch)) * _row_bytes(wl)
        assert bench.kv_bytes(wl, "sparse", n_t, ks) == sparse


@pytest.mark.parametrize("steps", [1024, 8192])
def test_kv_bytes_rswa_equal_oracle_attend_sets(steps):
    wl = synth.workload("rswa_b16", steps=steps)
    for t in (0, 5, wl.rswa_window - 2, wl.rswa_window, steps - 1):
        n_t = wl.seq_len_at(t)
        want = wl.batch * A.rswa_positions(n_t, wl.rswa_prefix, wl.rswa_window).size
        assert bench.kv_bytes(wl, "rswa", n_t, None) == want * _row_bytes(wl)


def test_recorded_traffic_needs_matching_digest(tmp_path, monkeypatch):
    f = tmp_path / "traffic.md"
    dig = bench.source_digest()
    f.write_text(f"`traffic attend_sparse qwen7b_b1 12345 {dig}`\n"
                 f"`traffic attend_focal qwen7b_b1 999 0000000000000000`\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("attend_sparse", "qwen7b_b1") == 12345.0
    assert bench.recorded_traffic("attend_focal", "qwen7b_b1") is None      # stale digest
    assert bench.recorded_traffic("attend_rswa", "rswa_b16") is None        # not recorded
