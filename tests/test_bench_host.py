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


def test_per_kind_timings_see_the_timed_pass_steps():
    """The per-kind graphs are replayed on exactly the decode steps of the
    timed pass (each step the same number of times), so their times add up
    to the step time for workloads whose lists grow along the decode."""
    import types

    class Ev:
        def record(self):
            pass

        def elapsed_time(self, other):
            return 1.0

    fake_torch = types.SimpleNamespace(cuda=types.SimpleNamespace(
        Event=lambda enable_timing=True: Ev(), synchronize=lambda *a: None))
    bn = object.__new__(bench.Bench)
    bn.torch = fake_torch
    bn.args = bench.parse_args(["--steps", "12", "--warmup", "3"])
    bn.world, bn.dev = 1, None
    bn.flush = types.SimpleNamespace(zero_=lambda: None)
    bn.wl = synth.workload("multipage_b8")
    bn.t0_steady, bn.span = bn.wl.warmup, bn.wl.steps - bn.wl.warmup
    staged = []
    bn.stage = lambda dec, cap, i: staged.append(bn.t_of(i))
    cap = types.SimpleNamespace(replay=lambda: None)
    K, W = 12, 3
    us, steps = bn.time_replays(None, cap, reps=2)
    timed = [bn.t_of(W + j) for j in range(K)]
    assert steps == timed
    assert sorted(staged[W:]) == sorted(timed * 2)
    assert len(set(timed)) == K and max(timed) - min(timed) > bn.span // 2   # the whole decode
    assert us == 1000.0
