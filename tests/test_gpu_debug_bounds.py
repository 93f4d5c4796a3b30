"""The debug build's bounds checks on shapes that stress the kernels' index arithmetic.

libra_debug.so is libra.so compiled with RA_DEBUG_BOUNDS: the tensor-core and f32
kernels check their TMA row coordinates, tensor-memory lanes and columns, ring-walk
state, partial indices, scalar-block indices and output rows, and a failed check
sets a status bit that ra_sync_status / ra_fwd_static_status return as
RA_ERR_BOUNDS.  The cases (tests/bounds_cases.py) run in a child process on the debug
library -- every status check must pass -- and here on libra.so; the two must agree
bit for bit, so the debug build runs the same arithmetic.
"""

import os
import subprocess
import sys

import numpy as np
import pytest

from tests.conftest import ROOT

torch = pytest.importorskip("torch")
ra = pytest.importorskip("context_ring_attention_gb300")

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ra.load_library()


def test_debug_bounds_build_passes_and_matches_release(tmp_path):
    from context_ring_attention_gb300 import build
    if not os.path.exists(build.LIB_DEBUG):
        build.build(debug=True)
    out = tmp_path / "debug.npz"
    env = dict(os.environ, RA_LIBRARY_VARIANT="debug")
    res = subprocess.run([sys.executable, "-m", "tests.bounds_cases", str(out)], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, f"debug-bounds run failed:\n{res.stdout[-2000:]}\n{res.stderr[-4000:]}"
    from tests.bounds_cases import run_cases
    release = run_cases()
    with np.load(out) as dbg:
        assert sorted(dbg.files) == sorted(release)
        for name, want in release.items():
            got = dbg[name]
            assert got.shape == want.shape, name
            # bit for bit (NaN never occurs here: -inf LSEs compare equal)
            assert np.array_equal(got, want), f"{name}: debug build differs from release"
