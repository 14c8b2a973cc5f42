"""GPU checks of the two debugging builds of the library (tests/variant_run.py, run as a child
process so that the package loads the variant instead of libjfa.so):

- trace (JFA_TRACE): every role of the persistent forward and backward kernels records one
  event per step or item, the records are ordered, and the results still match the oracle;
- debug (JFA_DEBUG): every tile load is bounds-checked in the kernels; on valid inputs no check
  fires and the results match the oracle.
"""
import os
import subprocess
import sys

import pytest

from varlen_flashattention_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("variant", ["trace", "debug"])
def test_debugging_build(variant):
    build.build(variant=variant)
    env = dict(os.environ, JFA_LIBRARY_VARIANT=variant)
    r = subprocess.run([sys.executable, "-m", "tests.variant_run", variant], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, f"{variant} build checks failed:\n{r.stdout[-4000:]}\n{r.stderr[-4000:]}"
    assert f"{variant} ok" in r.stdout
