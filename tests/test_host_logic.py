"""Host logic of the library compiled for the CPU (no GPU): the keep count the
kernels use against the oracle's, and the split-K choice's invariants."""
import os
import random
import shutil
import subprocess

import pytest

import oracle.attention as A

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# co-resident clusters of 1..16 CTAs of the general variant on a GB300
# (152 SMs, 2 CTAs per SM), as the occupancy query reports them
ACTIVE = [304, 152, 97, 74, 58, 46, 38, 36, 30, 28, 23, 23, 19, 14, 14, 14]


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("probe") / "host_probe")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                    "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "dynamic_sparse_kv_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "host_probe.cu"), "-o", exe], check=True)

    def run(lines):
        r = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True,
                           text=True, check=True)
        return [int(x) for x in r.stdout.split()]
    return run


def test_keep_count_matches_oracle(probe):
    rng = random.Random(7)
    cases = [(tau, n) for tau in (0.02, 0.05, 0.07, 0.1, 0.13, 0.25, 0.3, 0.5, 0.999, 1.0, 1e-6)
             for n in (0, 1, 2, 3, 7, 16, 30, 100, 256, 320, 4096, 8192, 16384, 16390)]
    cases += [(round(rng.uniform(0.0005, 1.0), rng.choice([2, 3, 4])), rng.randrange(0, 20001))
              for _ in range(3000)]
    got = probe([f"k {tau!r} {n}" for tau, n in cases])
    want = [A.keep_count(tau, n) for tau, n in cases]
    bad = [(c, g, w) for c, g, w in zip(cases, got, want) if g != w]
    assert not bad, bad[:10]


def _splits(probe, rows):
    return probe([f"s {u} {n} {mx} 152 " + " ".join(map(str, act)) for u, n, mx, act in rows])


def test_split_choice_in_range_and_schedulable(probe):
    rows = []
    for act in (ACTIVE, [304, 152, 0, 76, 0, 0, 0, 38] + [0] * 8, [300] + [0] * 15):
        for mx in (1, 4, 16):
            for u in (1, 4, 32, 128, 512):
                for n in (1, 300, 5000):
                    rows.append((u, n, mx, act))
    for (u, n, mx, act), s in zip(rows, _splits(probe, rows)):
        assert 1 <= s <= mx and (s == 1 or act[s - 1] >= 1), (u, n, mx, s)


def test_split_choice_grows_with_length(probe):
    lens = [1, 16, 100, 300, 667, 2000, 4417, 8449, 18497, 40000]
    for u in (1, 4, 16, 32, 128):
        got = _splits(probe, [(u, n, 16, ACTIVE) for n in lens])
        assert got == sorted(got), (u, got)


def test_split_choice_on_the_fitted_shapes(probe):
    # (sequence, KV head) units and attend lengths of layers whose split count
    # was swept on a GB300; each expected value is within 3% of the fastest
    # forced count there
    rows = [((4, 4417), 16),      # batch 1, full / focal layer
            ((4, 525), 12),       # batch 1, gather layer
            ((32, 18496), 7),     # 8 sequences of 16k image tokens, focal layer
            ((32, 2932), 4),      # ... gather layer
            ((128, 8449), 2),     # 32 sequences, focal layer
            ((128, 667), 1),      # 32 sequences, gather layer
            ((320, 666), 1),      # 80 sequences, gather layer: one split, not six
            ((512, 8448), 1),     # 128 sequences, focal layer
            ((512, 666), 1),      # 128 sequences, gather layer
            ((640, 666), 1),      # 160 sequences, gather layer
            ((320, 2752), 3),     # R-SWA, 32 sequences x 10 heads
            ((480, 2752), 1),     # R-SWA, 48 sequences
            ((1, 1), 1)]          # one token: nothing to split
    got = _splits(probe, [(u, n, 16, ACTIVE) for (u, n), _ in rows])
    assert got == [want for _, want in rows]


def test_split_choice_one_split_when_one_split_fills_the_device(probe):
    """Short gather lists over more units than the device holds CTAs: extra
    splits only add waves of fixed CTA cost."""
    rows = [(u, n, 16, ACTIVE) for u in (304, 400, 608, 1024, 4096) for n in (300, 700)]
    assert _splits(probe, rows) == [1] * len(rows)
