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
    import json
    f = tmp_path / "traffic.json"
    dig = bench.source_digest()
    f.write_text(json.dumps({"entries": [
        {"kernel": "attend_sparse", "workload": "qwen7b_b1", "bytes_per_launch": 12345,
         "digest": dig},
        {"kernel": "attend_focal", "workload": "qwen7b_b1", "bytes_per_launch": 999,
         "digest": "0000000000000000"}]}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("attend_sparse", "qwen7b_b1") == 12345.0
    assert bench.recorded_traffic("attend_focal", "qwen7b_b1") is None      # stale digest
    assert bench.recorded_traffic("attend_rswa", "rswa_b16") is None        # not recorded


def test_committed_traffic_file_parses():
    import json
    with open(bench.TRAFFIC_FILE) as f:
        entries = json.load(f)["entries"]
    for e in entries:
        assert e["kernel"] in bench.KERNEL_NAME.values() and e["bytes_per_launch"] > 0
        assert len(e["digest"]) == 16 and e["source"].startswith("profiles/")


def test_kinds_check_flags_shares_above_the_step():
    ok = bench.kinds_check({"focal": {"us_in_step": 300.0}, "sparse": {"us_in_step": 290.0}}, 600.0)
    assert not ok["kinds_exceed_step"] and abs(ok["kinds_sum_over_step"] - 590 / 600) < 1e-12
    bad = bench.kinds_check({"focal": {"us_in_step": 300.0}, "sparse": {"us_in_step": 400.0}},
                            600.0)
    assert bad["kinds_exceed_step"]


def test_reference_arm_echoes_steps_and_config(monkeypatch):
    legs = iter([{"value": 2.0, "steps": 7}])
    monkeypatch.setattr(bench, "run_oracle_leg", lambda *a, **k: next(legs))
    args = bench.parse_args(["--impl", "reference", "--steps", "20", "--warmup", "5"])
    r = bench.run_reference(args)
    assert r["steps"] == 20 and r["warmup"] == 5 and r["impl"] == "reference"
    assert r["config"]["workload"] == args.workload == "serving_b32"
    assert r["config"]["tau"] == synth.workload("serving_b32").tau
    assert r["config"]["batch_per_gpu"] == 32
