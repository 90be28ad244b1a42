import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def build_library(force=False):
    """Build libfastocr.so (nvcc) if needed; return its path. build.py is loaded
    by path because importing the package loads the library it builds."""
    import importlib.util
    path = os.path.join(ROOT, "dynamic_sparse_kv_gb300", "build.py")
    spec = importlib.util.spec_from_file_location("_fastocr_build", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod.build(force=force)


def pytest_sessionfinish(session, exitstatus):
    """Write the per-test maximum output errors (tests/gpu_harness.py) to the
    JSON file FASTOCR_ERR_LOG names, if it is set and any were recorded."""
    path = os.environ.get("FASTOCR_ERR_LOG")
    mod = sys.modules.get("gpu_harness")
    if not path or mod is None or not mod.ERRORS:
        return
    import json
    with open(path, "w") as f:
        json.dump({k: {"max_abs_err": v[0], "max_abs_err_vs_rounded_oracle": v[1], "dtype": v[2],
                       "max_err_in_output_ulps": v[3]}
                   for k, v in sorted(mod.ERRORS.items())}, f, indent=1)
