"""The bounds-checked build (libbitdelta_bounds.so, -DBD_DEBUG_BOUNDS): every
plain global load and store of every kernel is range-checked against the
extent of its buffer, and a check that fails records the kernel in a device
flag word instead of making the access.  These tests run every entry point
(tests/bounds_run.py) once through the normal library and once through the
bounds-checked one, each in a child process of its own (BD_LIBRARY selects
the library), and require that no check fired and that every output of the
two runs is the same bit for bit -- the checks skip no access that the
normal build makes."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from bit_weight_delta_bd_gb300 import bitdelta as bd

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def libs():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    from bit_weight_delta_bd_gb300 import build

    __graft_entry__.build()
    return build.LIB, build.build(debug_bounds=True)


def _run(lib_path: str, out: str) -> dict:
    env = dict(os.environ, BD_LIBRARY=lib_path)
    p = subprocess.run([sys.executable, os.path.join(HERE, "bounds_run.py"), out], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stdout[-2000:] + p.stderr[-4000:]
    return json.loads(p.stdout.strip().splitlines()[-1])


def test_bounds_checked_build_is_silent_and_bit_identical(libs, tmp_path):
    normal, bounded = libs
    rn = _run(normal, str(tmp_path / "normal.npz"))
    rb = _run(bounded, str(tmp_path / "bounds.npz"))
    assert rn["enabled"] is False and rb["enabled"] is True
    assert rn["status"] == bd.BD_OK and rn["bits"] == 0
    assert rb["status"] == bd.BD_OK, f"bounds check fired in kernels 0x{rb['bits']:x}"
    assert rb["bits"] == 0
    a, b = np.load(tmp_path / "normal.npz"), np.load(tmp_path / "bounds.npz")
    assert sorted(a.files) == sorted(b.files) and len(a.files) == rn["arrays"] > 50
    differ = [k for k in a.files if not np.array_equal(a[k], b[k])]
    assert not differ, f"outputs differ between the builds: {differ}"
