"""The AQ_DEBUG_CHECKS build of the library: the kernels also check internal
invariants -- the value bins of every subspace sum to the same total, below
2^31 plus rounding; a streamed share's fixed-point frame keeps the bins' total
within 2^31 and rescales by factors <= 1; split partials land inside the
workspace -- and report a failed one as AQ_DEV_INVARIANT in the status word.
A subset of the parity tests runs in a child process against that build
(selected by AQPQ_DEBUG_CHECKS=1); each of them requires a zero status.
"""
import os
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_checks_build_passes_parity_subset():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, AQPQ_DEBUG_CHECKS="1")
    subprocess.run([sys.executable, "-c", "from decode_attention_product_gb300 import build; build.build(debug=True)"],
                   cwd=ROOT, env=env, check=True, timeout=900)
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "tests/test_gpu_parity.py", "tests/test_gpu_configs.py", "-m", "gpu", "-x",
         "-q", "-p", "no:cacheprovider", "-k",
         "decode_matches_oracle or decode_step_matches_oracle or peaked or qwen_gqa or long"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
