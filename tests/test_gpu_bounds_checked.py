"""The parity tests again, on the bounds-checked library (libsvx_checked.so, -DSVX_BOUNDS_CHECK).

No memory checker may run on these GPUs, so the library has a build in which every kernel checks that
each global range it reads or writes lies in the buffer its launch parameters describe (the parts'
K/V rows, Q, the state workspace, the candidates, O and LSE), skips an access that does not and raises
the device error word.  Every round of the parity tests ends with svx_round_finish(timeout_ms > 0), and
every no-allocation round with svx_static_check, which report a raised word as an error; so these tests
passing on the checked library means no kernel computed an address outside its buffers on any of their
shapes (ragged tails, trees, d = 64 head pairs, more than 2^31 elements, full-size sampled rounds).
tests/test_gpu_bounds_hook.py, run here too, shows that the checks fire and are reported.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "speculative_decoding_verification_chunked_gb300")


def test_parity_suite_on_the_bounds_checked_library():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert os.path.exists(os.path.join(PKG, "libsvx_checked.so")), "libsvx_checked.so is not built"
    env = dict(os.environ, SVX_LIBRARY="checked")
    probe = subprocess.run([sys.executable, "-c", "from speculative_decoding_verification_chunked_gb300 import svx; "
                            "print(svx._LIB_PATH)"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert probe.returncode == 0 and probe.stdout.strip().endswith("libsvx_checked.so"), probe.stdout + probe.stderr
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "tests/test_gpu_parity.py", "tests/test_gpu_causality.py", "tests/test_gpu_bounds_hook.py",
           "tests/test_zz_no_alloc.py"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=2400)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout and " failed" not in r.stdout
