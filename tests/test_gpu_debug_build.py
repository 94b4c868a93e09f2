"""The bounds-checked FA_DEBUG build (libfa_debug.so) on a GPU: on valid
inputs no check fires (fa_last_device_error stays FA_OK) and every kernel
family gives the release build's results bit for bit. The debug library
runs in a child process (one library per process)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_matches_release_bitwise(tmp_path):
    from exact_tiled_attention_24_gb300 import build
    build.build()
    build.build(debug=True)
    import debug_cases
    import exact_tiled_attention_24_gb300 as fa
    assert not fa.debug_checks()
    release = debug_cases.run_cases()
    path = tmp_path / "debug.pt"
    env = dict(os.environ, FA_DEBUG_LIBRARY="1")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_cases.py"), str(path)], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    debug = torch.load(path)
    assert sorted(debug) == sorted(release)
    for name, t in release.items():
        assert torch.equal(t, debug[name]), name
