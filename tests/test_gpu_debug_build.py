"""The attention, merge, plan and verify kernels under the index-checking
debug build (sources compiled with -DSPECVERIFY_DEBUG): every shared-memory,
TMEM and global index and every TMA / MMA operand address is checked before
its access, a failed check sets SV_DEV_DEBUG_CHECK in the status word and
prints its line.  This is the stand-in for a memory checker: the GPU parity
tests of the attention (bf16 and fp8 KV, both kernel forms, uniform splits
and the balanced plan, the gates, the literal entry point, the seeded sweep)
and the tests that make bounded waits give up run again in a child process
that loads the debug library, and must pass with no check failing.  The
full-size long-context cases are left out for time."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FILES = ["tests/test_gpu_parity.py", "tests/test_gpu_stacked.py", "tests/test_gpu_kv8.py",
         "tests/test_gpu_f4.py", "tests/test_gpu_abi_entry.py", "tests/test_gpu_sweep.py",
         "tests/test_gpu_abort.py"]


def test_parity_under_the_index_checking_build():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verify_mla_gb300 import build as B
    lib = B.build(debug=True)
    env = dict(os.environ, SPECVERIFY_LIBRARY=lib)
    probe = subprocess.run([sys.executable, "-c", "import speculative_decoding_verify_mla_gb300 as sv; "
                            "print(sv.load_library()._name)"], cwd=ROOT, env=env, capture_output=True,
                           text=True, timeout=300)
    assert probe.returncode == 0, probe.stderr[-2000:]
    assert probe.stdout.strip().splitlines()[-1] == lib  # the child loads the debug build
    res = subprocess.run([sys.executable, "-m", "pytest", "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider",
                          *FILES, "-k", "not c4_full"], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=2400)
    out = res.stdout + res.stderr
    assert res.returncode == 0, out[-4000:]
    assert "specverify debug check failed" not in out, out[-4000:]
