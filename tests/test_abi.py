"""Host-side checks of the C-ABI library: it loads, exports every entry point
declared in include/fa.h, and rejects bad arguments before touching a GPU
(no compute call is made here)."""
import ctypes
import os
import re

import pytest

import exact_tiled_attention_24_gb300 as fa
from exact_tiled_attention_24_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def L():
    fabuild.build()
    return fa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_binding_symbols():
    assert declared_functions() == sorted(fa.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_status_strings_and_version(L):
    assert L.fa_status_string(0) == b"FA_OK"
    assert L.fa_status_string(6) == b"FA_ERR_WORKSPACE"
    assert L.fa_status_string(99) == b"FA_ERR_UNKNOWN"
    assert re.match(rb"^\d+\.\d+\.\d+$", L.fa_version())


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: checks fail first
MIS = ctypes.c_void_p(0x10002)
NUL = ctypes.c_void_p(0)


def fwd_call(L, q=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=16, d=64, scale=0.125, causal=0):
    return L.fa_fwd(q, FAKE, FAKE, o, lse, B, H, N, d, scale, causal, NUL)


def test_fwd_argument_errors(L):
    assert fwd_call(L, q=NUL) == 1
    assert fwd_call(L, lse=NUL) == 1
    assert fwd_call(L, N=0) == 1
    assert fwd_call(L, B=-1) == 1
    assert fwd_call(L, scale=0.0) == 1
    assert fwd_call(L, scale=float("nan")) == 1
    assert fwd_call(L, scale=float("inf")) == 1
    assert fwd_call(L, d=96) == 2
    assert fwd_call(L, d=256) == 2
    assert fwd_call(L, B=65536, H=65536, N=2) == 2  # more than 2^31 rows
    assert fwd_call(L, q=MIS) == 3
    assert fwd_call(L, o=MIS) == 3


def test_bwd_workspace_size(L):
    B, H, N, d = 2, 3, 100, 64
    assert L.fa_bwd_workspace_bytes(B, H, N, d) == B * H * N * 4  # the fp32 D vector
    assert L.fa_bwd_workspace_bytes(B, H, 0, d) == 0
    assert L.fa_bwd_workspace_bytes(B, H, N, 80) == 0


def test_bwd_argument_errors(L):
    ws = L.fa_bwd_workspace_bytes(1, 1, 16, 64)

    def call(workspace=FAKE, ws_bytes=ws, dq=FAKE, d=64, scale=0.125):
        return L.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dq, FAKE, FAKE, workspace, ws_bytes,
                        1, 1, 16, d, scale, 1, NUL)

    assert call(dq=NUL) == 1
    assert call(scale=-1.0) == 1
    assert call(d=32) == 2
    assert call(workspace=NUL) == 6
    assert call(ws_bytes=ws - 1) == 6
    assert call(workspace=MIS) == 3
    # a misaligned operand of a later stage is rejected before the first
    # stage is queued (nothing reaches the device: no CUDA call is made)
    for pos in range(9):
        args = [FAKE] * 9
        args[pos] = MIS
        assert L.fa_bwd(*args, FAKE, ws, 1, 1, 16, 64, 0.125, 1, NUL) == 3, pos
    # stage entry points
    assert L.fa_bwd_preprocess(FAKE, FAKE, NUL, 1, 1, 16, 64, NUL) == 1
    assert L.fa_bwd_dkdv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, MIS, 1, 1, 1, 16, 64,
                         0.125, 0, NUL) == 3
    assert L.fa_bwd_dkdv(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 3, 16, 64,
                         0.125, 0, NUL) == 1  # 3 K/V heads cannot serve 4 query heads
    assert L.fa_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 1, 16, 64, 0.0, 1, NUL) == 1
    assert L.fa_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 1, 16, 96, 0.1, 1, NUL) == 2
    assert L.fa_bwd_dq(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 0, 16, 64, 0.1, 1, NUL) == 1
    # the dQ sweep that forms D itself: o is an input, Dvec an output
    def dq_d(o=FAKE, Dvec=FAKE, H=1, Hkv=1, d=64, scale=0.1):
        return L.fa_bwd_dq_d(FAKE, FAKE, FAKE, o, FAKE, FAKE, Dvec, FAKE, 1, H, Hkv, 16, d, scale, 1, NUL)

    assert dq_d(o=NUL) == 1 and dq_d(Dvec=NUL) == 1
    assert dq_d(o=MIS) == 3 and dq_d(Dvec=MIS) == 3
    assert dq_d(d=96) == 2
    assert dq_d(H=4, Hkv=3) == 1 and dq_d(scale=0.0) == 1
    # the order fa_bwd takes: never fused with grouped-query heads or bad sizes
    assert L.fa_bwd_fuses_d(2, 32, 8, 8192, 128) == 0
    assert L.fa_bwd_fuses_d(1, 4, 3, 16, 64) == 0
    assert L.fa_bwd_fuses_d(0, 4, 4, 16, 64) == 0
    assert L.fa_bwd_fuses_d(1, 4, 4, 16, 96) == 0


def test_gqa_argument_errors(L):
    def fwd(H=8, Hkv=2, k=FAKE):
        return L.fa_fwd_gqa(FAKE, k, FAKE, FAKE, FAKE, 1, H, Hkv, 16, 64, 0.125, 1, NUL)

    def bwd(H=8, Hkv=2, dk=FAKE):
        ws = L.fa_bwd_workspace_bytes(1, H, 16, 64)
        return L.fa_bwd_gqa(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dk, FAKE, FAKE, ws,
                            1, H, Hkv, 16, 64, 0.125, 1, NUL)

    for call in (fwd, bwd):
        assert call(Hkv=0) == 1
        assert call(Hkv=3) == 1       # does not divide H
        assert call(Hkv=16) == 1      # more K/V heads than query heads
        assert call(H=8, Hkv=-8) == 1
    assert fwd(k=NUL) == 1 and fwd(k=MIS) == 3
    assert bwd(dk=NUL) == 1


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "exact_tiled_attention_24_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle", text, flags=re.M), f


def test_softmax_argument_errors(L):
    for fn in (L.fa_softmax_safe, L.fa_softmax_online):
        assert fn(NUL, FAKE, 4, 16, NUL) == 1
        assert fn(FAKE, NUL, 4, 16, NUL) == 1
        assert fn(FAKE, FAKE, 0, 16, NUL) == 1
        assert fn(FAKE, FAKE, 4, 0, NUL) == 1
        assert fn(FAKE, FAKE, 2**31, 16, NUL) == 2
        assert fn(ctypes.c_void_p(0x10001), FAKE, 4, 16, NUL) == 3


def test_decode_and_merge_argument_errors(L):
    ws = L.fa_decode_workspace_bytes(2, 8, 128, 4)
    assert ws >= 4 * 2 * 8 * 128 * 4 + 4 * 2 * 8 * 4
    assert L.fa_decode_workspace_bytes(2, 8, 96, 4) == 0

    def dec(q=FAKE, table=FAKE, ws_ptr=FAKE, ws_bytes=ws, B=2, H=8, Hkv=2, d=128, num_blocks=10, bs=16,
            max_blocks=8, scale=0.1, S=4):
        return L.fa_decode_paged(q, FAKE, FAKE, table, FAKE, FAKE, FAKE, ws_ptr, ws_bytes, B, H, Hkv, d,
                                 num_blocks, bs, max_blocks, scale, S, NUL)

    assert dec(q=NUL) == 1
    assert dec(table=NUL) == 1
    assert dec(Hkv=3) == 1
    assert dec(S=0) == 1
    assert dec(bs=0) == 1
    assert dec(scale=-1.0) == 1
    assert dec(d=96) == 2
    assert dec(B=70000) == 2                  # more requests than one grid dimension holds
    assert dec(max_blocks=1 << 27, bs=16) == 2   # a context of 2^31 tokens: past the int range
    assert dec(num_blocks=1 << 28, Hkv=2, bs=8) == 2     # 2^32 token rows in the cache: past 32-bit row indices
    assert dec(num_blocks=(1 << 28) - 1, Hkv=2, bs=8, ws_ptr=NUL) == 6  # just below: checks go on
    assert dec(ws_ptr=NUL) == 6
    assert dec(ws_bytes=ws - 1) == 6
    assert dec(q=MIS) == 3
    assert dec(table=ctypes.c_void_p(0x10002)) == 3

    def merge(o_parts=FAKE, n=3, rows=10, d=64):
        return L.fa_attn_merge(o_parts, FAKE, n, FAKE, FAKE, rows, d, NUL)

    assert merge(o_parts=NUL) == 1
    assert merge(n=0) == 1
    assert merge(rows=0) == 1
    assert merge(d=80) == 2
    assert merge(o_parts=MIS) == 3
    assert L.fa_status_string(7) == b"FA_ERR_BAD_INDEX"


def test_host_pipeline_argument_errors(L):
    def ts(**over):
        t = fa.Tensors(*([0x10000] * 9))
        for k, val in over.items():
            setattr(t, k, val)
        return t

    def fwd_h(host=None, dev=None, B=1, H=4, Hkv=2, N=16, d=64, scale=0.125, chunks=0):
        h = ctypes.byref(host if host is not None else ts())
        dv = ctypes.byref(dev if dev is not None else ts())
        return L.fa_fwd_host(h, dv, B, H, Hkv, N, d, scale, 0, chunks, NUL)

    def fb_h(host=None, dev=None, ws=FAKE, ws_bytes=4 * 4 * 16, B=1, H=4, Hkv=2, N=16, d=64, chunks=0):
        h = ctypes.byref(host if host is not None else ts())
        dv = ctypes.byref(dev if dev is not None else ts())
        return L.fa_fwd_bwd_host(h, dv, ws, ws_bytes, B, H, Hkv, N, d, 0.125, 1, chunks, NUL)

    tp = ctypes.POINTER(fa.Tensors)
    assert L.fa_fwd_host(tp(), ctypes.byref(ts()), 1, 4, 2, 16, 64, 0.125, 0, 0, NUL) == 1
    assert fwd_h(host=ts(q=None)) == 1
    assert fwd_h(dev=ts(lse=None)) == 1
    assert fwd_h(Hkv=3) == 1
    assert fwd_h(N=0) == 1
    assert fwd_h(scale=float("inf")) == 1
    assert fwd_h(chunks=-1) == 1
    assert fwd_h(d=96) == 2
    assert fwd_h(dev=ts(o=0x10004)) == 3
    # forward-only calls ignore the gradient slots
    assert fwd_h(host=ts(dO=None, dq=None, dk=None, dv=None), d=96) == 2
    assert fb_h(host=ts(dO=None)) == 1
    assert fb_h(dev=ts(dk=None)) == 1
    assert fb_h(dev=ts(dv=0x10008)) == 3
    assert fb_h(ws=NUL) == 6
    assert fb_h(ws_bytes=4 * 4 * 16 - 1) == 6
    assert fb_h(ws=MIS) == 3
    assert fb_h(d=80) == 2


def test_plain_c_program_compiles_links_and_runs(L, tmp_path):
    """The header is C99 and libfa.so links into a plain C program; the entry
    points that need no GPU (version, status names, argument checks) run."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_fa.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "fa.h"
int main(void) {
  fa_tensors host, dev;
  memset(&host, 0, sizeof host);
  memset(&dev, 0, sizeof dev);
  if (fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 1, 16, 64, 0.125f, 0, NULL) != FA_ERR_INVALID_ARG) return 1;
  if (fa_fwd_host(&host, &dev, 1, 1, 1, 16, 64, 0.125f, 0, 0, NULL) != FA_ERR_INVALID_ARG) return 2;
  if (fa_bwd_workspace_bytes(2, 3, 5, 64) != 2 * 3 * 5 * sizeof(float)) return 3;
  if (strcmp(fa_status_string(FA_ERR_WORKSPACE), "FA_ERR_WORKSPACE") != 0) return 4;
  printf("%s\n", fa_version());
  return 0;
}
''')
    lib_dir = os.path.dirname(fa.lib_path())
    exe = tmp_path / "use_fa"
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", lib_dir, "-lfa", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    assert re.match(r"^\d+\.\d+\.\d+$", r.stdout.strip())


def test_softmax_host_argument_errors(L):
    def call(xh=FAKE, yh=FAKE, xd=FAKE, yd=FAKE, rows=4, n=16, chunks=0):
        return L.fa_softmax_host(xh, yh, xd, yd, rows, n, 1, chunks, NUL)

    assert call(xh=NUL) == 1
    assert call(yd=NUL) == 1
    assert call(rows=0) == 1
    assert call(n=0) == 1
    assert call(chunks=-1) == 1
    assert call(rows=2**31) == 2
    assert call(xd=ctypes.c_void_p(0x10002)) == 3
