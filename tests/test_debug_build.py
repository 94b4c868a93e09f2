"""Host-side checks of the bounds-checked FA_DEBUG build: it compiles for
sm_103a, exports every entry point the header declares, says it is the
debug build, and rejects bad arguments exactly as the release library does
(no GPU needed)."""
import ctypes

import pytest

from exact_tiled_attention_24_gb300 import build as fabuild
from test_abi import declared_functions


@pytest.fixture(scope="module")
def libs():
    rel = ctypes.CDLL(fabuild.build())
    dbg = ctypes.CDLL(fabuild.build(debug=True))
    return rel, dbg


def test_debug_library_exports_every_declared_symbol(libs):
    _, dbg = libs
    for name in declared_functions():
        assert hasattr(dbg, name), name


def test_flavour_flag(libs):
    rel, dbg = libs
    assert rel.fa_debug_checks() == 0
    assert dbg.fa_debug_checks() == 1


def test_same_argument_checks(libs):
    vp = ctypes.c_void_p
    fake, nul = vp(0x10000), vp(0)
    for L in libs:
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp] + [ctypes.c_int] * 4 + [ctypes.c_float, ctypes.c_int, vp]
        L.fa_status_string.restype = ctypes.c_char_p
        assert L.fa_fwd(nul, fake, fake, fake, fake, 1, 1, 16, 64, 0.125, 0, nul) == 1
        assert L.fa_fwd(fake, fake, fake, fake, fake, 1, 1, 16, 96, 0.125, 0, nul) == 2
        assert L.fa_fwd(vp(0x10002), fake, fake, fake, fake, 1, 1, 16, 64, 0.125, 0, nul) == 3
        assert L.fa_status_string(8) == b"FA_ERR_BOUNDS"
