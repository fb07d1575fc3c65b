"""The bounds-checked library (compiled with MOE_CHECKED: kernels test every
data-dependent global index -- permutation rows, GEMM output rows -- and report
MOE_ERR_DEVICE_BOUNDS instead of accessing out of range) runs the mid-size
parity tests and the expert-parallel kernels' tests clean: a stand-in for a run under a
memory checker.  The tests run in a child process with MOE_CHECKED=1, which makes
the binding load the checked build; each of them requires a clean device
status word after its forward, so any failed check fails the run."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _checked_env():
    import importlib.util
    spec = importlib.util.spec_from_file_location("_moe_build_checked",
                                                  os.path.join(ROOT, "serving_router_gate_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build(checked=True)
    return dict(os.environ, MOE_CHECKED="1")


def test_checked_build_is_loaded_and_runs_mid_size_parity_clean():
    env = _checked_env()
    r = subprocess.run([sys.executable, "-c", "import serving_router_gate_gb300 as m; print(m.lib_path())"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip().endswith("libmoe_gb300_checked.so"), r.stdout
    sel = ("tiny or mid_layer or partial_n or replica_slots or local_ranges or one_hot or stages or "
           "envelope or small_batch_splits")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "tests/test_gpu_small_batch.py",
                        "tests/test_gpu_nvfp4.py", "-q", "-m", "gpu", "-x", "-p", "no:cacheprovider", "-k",
                        sel + " or small_batches or nvfp4_mid or nvfp4_small"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout


def test_checked_build_runs_the_expert_parallel_kernels_clean():
    # the all-to-all reorder, FC2 through a row map and the peer reduction under the
    # bounds-checked build (ranks held by one process; the IPC test stays out: two
    # processes each building their own library)
    env = _checked_env()
    sel = "regroup or scatter or a2a_layer or peer_reduction_of_local or unwritten"
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_gpu_expert_parallel.py", "-q", "-m", "gpu", "-x",
                        "-p", "no:cacheprovider", "-k", sel],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
