"""The product path has no CPU fallback and no route through the oracle: the
package imports nothing from oracle/, and without libfastocr.so importing
it fails instead of degrading."""
import os
import re
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "dynamic_sparse_kv_gb300")


def test_package_never_imports_the_oracle():
    pat = re.compile(r"^\s*(from|import)\s+oracle\b|importlib.*oracle", re.M)
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not pat.search(text), f"{f} reaches into oracle/"


def test_import_fails_without_the_library(tmp_path):
    dst = tmp_path / "dynamic_sparse_kv_gb300"
    shutil.copytree(PKG, dst, ignore=shutil.ignore_patterns("*.so", "_build", "__pycache__",
                                                            "csrc"))
    assert not (dst / "libfastocr.so").exists()
    r = subprocess.run([sys.executable, "-c", "import dynamic_sparse_kv_gb300"], cwd=tmp_path,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "libfastocr.so" in (r.stderr + r.stdout)
