"""Exact tiled attention (FlashAttention-style) for GB300 / sm_103a.

Thin ctypes binding over ``libfa.so`` (C ABI in ``include/fa.h``): it only
checks tensors, allocates outputs with torch on the current device, and
passes raw pointers plus the current CUDA stream. Every step of the forward
and backward runs in the library's CUDA kernels; there is no fallback path —
if the library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "FAError",
    "lib",
    "lib_path",
    "fwd",
    "bwd",
    "bwd_preprocess",
    "bwd_dkdv",
    "bwd_dq",
    "bwd_dq_d",
    "bwd_fuses_d",
    "bwd_workspace_bytes",
    "last_device_error",
    "debug_checks",
    "softmax_safe",
    "softmax_online",
    "attn_merge",
    "decode_paged",
    "decode_workspace_bytes",
    "fwd_host",
    "fwd_bwd_host",
    "softmax_host",
    "EXPORTED_SYMBOLS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
# FA_DEBUG_LIBRARY=1 selects the bounds-checked build (libfa_debug.so, made
# by build.build(debug=True)); it computes the same results.
_LIB_PATH = os.path.join(_HERE, "_lib",
                         "libfa_debug.so" if os.environ.get("FA_DEBUG_LIBRARY") == "1" else "libfa.so")
_lib = None

FA_STATUS = {
    0: "FA_OK",
    1: "FA_ERR_INVALID_ARG",
    2: "FA_ERR_UNSUPPORTED",
    3: "FA_ERR_MISALIGNED",
    4: "FA_ERR_CUDA",
    5: "FA_ERR_TIMEOUT",
    6: "FA_ERR_WORKSPACE",
    7: "FA_ERR_BAD_INDEX",
    8: "FA_ERR_BOUNDS",
}

EXPORTED_SYMBOLS = (
    "fa_fwd",
    "fa_fwd_gqa",
    "fa_bwd_workspace_bytes",
    "fa_bwd",
    "fa_bwd_gqa",
    "fa_bwd_preprocess",
    "fa_bwd_dkdv",
    "fa_bwd_dq",
    "fa_bwd_dq_d",
    "fa_bwd_fuses_d",
    "fa_last_device_error",
    "fa_selftest_wait_limit",
    "fa_status_string",
    "fa_version",
    "fa_bwd_noalloc",
    "fa_softmax_safe",
    "fa_softmax_online",
    "fa_attn_merge",
    "fa_decode_workspace_bytes",
    "fa_decode_paged",
    "fa_fwd_host",
    "fa_fwd_bwd_host",
    "fa_softmax_host",
    "fa_debug_checks",
)


class Tensors(ctypes.Structure):
    """fa_tensors: addresses of one problem's q, k, v, dO, o, lse, dq, dk, dv."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "dO", "o", "lse", "dq", "dk", "dv")]


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {FA_STATUS.get(status, status)}")


def lib_path() -> str:
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    """Load libfa.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise FAError(-1, f"libfa.so not built at {_LIB_PATH}; run exact_tiled_attention_24_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_fwd.restype = i
        L.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_fwd_gqa.restype = i
        L.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
        L.fa_bwd_workspace_bytes.restype = sz
        L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, f, i, vp]
        L.fa_bwd.restype = i
        L.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
        L.fa_bwd_gqa.restype = i
        L.fa_bwd_preprocess.argtypes = [vp, vp, vp, i, i, i, i, vp]
        L.fa_bwd_preprocess.restype = i
        L.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_bwd_dkdv.restype = i
        L.fa_bwd_dq.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_bwd_dq_d.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        L.fa_bwd_dq_d.restype = i
        L.fa_bwd_fuses_d.argtypes = [i, i, i, i, i]
        L.fa_bwd_fuses_d.restype = i
        L.fa_bwd_dq.restype = i
        L.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
        L.fa_bwd_noalloc.restype = i
        L.fa_softmax_safe.argtypes = [vp, vp, ctypes.c_longlong, i, vp]
        L.fa_softmax_safe.restype = i
        L.fa_softmax_online.argtypes = [vp, vp, ctypes.c_longlong, i, vp]
        L.fa_softmax_online.restype = i
        L.fa_attn_merge.argtypes = [vp, vp, i, vp, vp, ctypes.c_longlong, i, vp]
        L.fa_attn_merge.restype = i
        L.fa_decode_workspace_bytes.argtypes = [i, i, i, i]
        L.fa_decode_workspace_bytes.restype = sz
        L.fa_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, i, f, i, vp]
        L.fa_decode_paged.restype = i
        tp = ctypes.POINTER(Tensors)
        L.fa_fwd_host.argtypes = [tp, tp, i, i, i, i, i, f, i, i, vp]
        L.fa_fwd_host.restype = i
        L.fa_fwd_bwd_host.argtypes = [tp, tp, vp, sz, i, i, i, i, i, f, i, i, vp]
        L.fa_fwd_bwd_host.restype = i
        L.fa_softmax_host.argtypes = [vp, vp, vp, vp, ctypes.c_longlong, i, i, i, vp]
        L.fa_softmax_host.restype = i
        L.fa_last_device_error.argtypes = [vp]
        L.fa_last_device_error.restype = i
        L.fa_selftest_wait_limit.argtypes = [vp]
        L.fa_selftest_wait_limit.restype = i
        L.fa_status_string.argtypes = [i]
        L.fa_status_string.restype = ctypes.c_char_p
        L.fa_version.argtypes = []
        L.fa_version.restype = ctypes.c_char_p
        L.fa_debug_checks.argtypes = []
        L.fa_debug_checks.restype = i
        _lib = L
    return _lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


# Device type of every tensor the kernels touch. The library launches on the
# current CUDA device, so the tensors must live there as well.
_DEVICE_TYPE = "cuda"


def _on_device(t, name):
    """Raise unless t is a tensor on a device the library can launch on."""
    if not isinstance(t, torch.Tensor) or t.device.type != _DEVICE_TYPE:
        raise ValueError(f"{name} must be a {_DEVICE_TYPE.upper()} tensor")
    if _DEVICE_TYPE == "cuda" and t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device} but the current device is cuda:"
                         f"{torch.cuda.current_device()}: call under torch.cuda.device({t.device})")


def _expect(t, name, shape, dtype, device):
    """Raise unless t is a contiguous `dtype` tensor of exactly `shape` on
    `device`: a buffer the kernels read or write in full, so a smaller one
    would be overrun."""
    if (not isinstance(t, torch.Tensor) or tuple(t.shape) != tuple(shape) or t.dtype != dtype
            or not t.is_contiguous() or t.device != device):
        raise ValueError(f"{name}: expected a contiguous {dtype} tensor of shape {tuple(shape)} on {device}")


def _expect_workspace(ws, device):
    """The workspace's size is checked by the library; here its place."""
    if not isinstance(ws, torch.Tensor) or ws.device != device or not ws.is_contiguous():
        raise ValueError(f"workspace must be a contiguous tensor on {device}")


def _check(status, where):
    if status != 0:
        raise FAError(status, where)


def _check_inputs(q, k, v, *rest):
    """q (and o, dO in rest): [B, H, N, d]; k, v: [B, Hkv, N, d] with Hkv dividing H.
    Returns Hkv."""
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    _on_device(q, "q")
    for t in (q, k, v) + rest:
        if t.device.type != _DEVICE_TYPE:
            raise ValueError("tensors must be on a CUDA device")
        if t.dtype != torch.bfloat16:
            raise ValueError("tensors must be bfloat16")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if t.device != q.device:
            raise ValueError("tensors must be on one device")
    for t in rest:
        if t.shape != q.shape:
            raise ValueError("o and dO must have q's shape")
    if k.shape != (B, Hkv, N, d) or v.shape != k.shape or Hkv < 1 or H % Hkv:
        raise ValueError("k and v must be [B, Hkv, N, d] with Hkv dividing q's head count")
    return Hkv


def _scale(d, scale):
    return (1.0 / d ** 0.5) if scale is None else float(scale)


def fwd(q, k, v, causal=False, scale=None, out=None, lse=None):
    """o, lse = softmax(scale·q kᵀ [causal]) v and its per-row log-sum-exp.

    k and v may hold fewer heads than q (grouped-query attention): query head
    h then uses K/V head h // (H // Hkv)."""
    Hkv = _check_inputs(q, k, v)
    B, H, N, d = q.shape
    if out is not None:
        _expect(out, "out", q.shape, torch.bfloat16, q.device)
    if lse is not None:
        _expect(lse, "lse", (B, H, N), torch.float32, q.device)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse_t), B, H, Hkv, N, d,
                            _scale(d, scale), int(bool(causal)), _stream(q.device)), "fa_fwd_gqa")
    return o, lse_t


def bwd_workspace_bytes(B, H, N, d) -> int:
    return int(lib().fa_bwd_workspace_bytes(B, H, N, d))


def bwd(q, k, v, o, lse, do, causal=False, scale=None, workspace=None):
    """dq, dk, dv of o = softmax(scale·q kᵀ [causal]) v for the output gradient do
    (dk, dv shaped like k, v; with grouped-query heads they sum over the group)."""
    Hkv = _check_inputs(q, k, v, o, do)
    B, H, N, d = q.shape
    _expect(lse, "lse", (B, H, N), torch.float32, q.device)
    ws_bytes = bwd_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    _expect_workspace(workspace, q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    _check(lib().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                            _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                            B, H, Hkv, N, d, _scale(d, scale), int(bool(causal)), _stream(q.device)),
           "fa_bwd_gqa")
    return dq, dk, dv


def bwd_preprocess(o, do, Dvec):
    """Dvec = rowsum(do * o) (fp32 [B, H, N])."""
    _check_inputs(o, o, o, do)
    B, H, N, d = o.shape
    _expect(Dvec, "Dvec", (B, H, N), torch.float32, o.device)
    _check(lib().fa_bwd_preprocess(_ptr(o), _ptr(do), _ptr(Dvec), B, H, N, d, _stream(o.device)),
           "fa_bwd_preprocess")


def bwd_dkdv(q, k, v, do, lse, Dvec, dk, dv, causal=False, scale=None):
    """dk, dv (bf16, written in place) from the recomputed P and dS."""
    Hkv = _check_inputs(q, k, v, do)
    B, H, N, d = q.shape
    _expect(lse, "lse", (B, H, N), torch.float32, q.device)
    _expect(Dvec, "Dvec", (B, H, N), torch.float32, q.device)
    _expect(dk, "dk", k.shape, torch.bfloat16, q.device)
    _expect(dv, "dv", k.shape, torch.bfloat16, q.device)
    _check(lib().fa_bwd_dkdv(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(Dvec), _ptr(dk),
                             _ptr(dv), B, H, Hkv, N, d, _scale(d, scale), int(bool(causal)),
                             _stream(q.device)), "fa_bwd_dkdv")


def bwd_dq_d(q, k, v, o, do, lse, Dvec, dq, causal=False, scale=None):
    """dq (bf16) and Dvec = rowsum(do * o) (fp32), both written in place, by
    the dQ sweep alone (no preprocess); bwd_dkdv can then read Dvec."""
    Hkv = _check_inputs(q, k, v, o, do)
    B, H, N, d = q.shape
    _expect(lse, "lse", (B, H, N), torch.float32, q.device)
    _expect(Dvec, "Dvec", (B, H, N), torch.float32, q.device)
    _expect(dq, "dq", q.shape, torch.bfloat16, q.device)
    _check(lib().fa_bwd_dq_d(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(Dvec), _ptr(dq),
                             B, H, Hkv, N, d, _scale(d, scale), int(bool(causal)), _stream(q.device)),
           "fa_bwd_dq_d")


def bwd_fuses_d(B, H, Hkv, N, d):
    """True when bwd() runs the dQ sweep with D first and the dK/dV sweep
    after it for these sizes on the current device (see fa_bwd_fuses_d)."""
    return bool(lib().fa_bwd_fuses_d(int(B), int(H), int(Hkv), int(N), int(d)))


def bwd_dq(q, k, v, do, lse, Dvec, dq, causal=False, scale=None):
    """dq (bf16, written in place) from the recomputed dS."""
    Hkv = _check_inputs(q, k, v, do)
    B, H, N, d = q.shape
    _expect(lse, "lse", (B, H, N), torch.float32, q.device)
    _expect(Dvec, "Dvec", (B, H, N), torch.float32, q.device)
    _expect(dq, "dq", q.shape, torch.bfloat16, q.device)
    _check(lib().fa_bwd_dq(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(Dvec), _ptr(dq),
                           B, H, Hkv, N, d, _scale(d, scale), int(bool(causal)), _stream(q.device)),
           "fa_bwd_dq")


def selftest_wait_limit(device=None) -> None:
    """Enqueue the error-path self-test on the current stream: a wait that
    nothing satisfies gives up after its limit, so the next
    last_device_error() returns 5 (FA_ERR_TIMEOUT)."""
    dev = torch.device("cuda") if device is None else device
    _check(lib().fa_selftest_wait_limit(_stream(dev)), "fa_selftest_wait_limit")


def debug_checks() -> bool:
    """True when the loaded library is the bounds-checked FA_DEBUG build."""
    return bool(lib().fa_debug_checks())


def last_device_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error status."""
    dev = torch.device("cuda") if device is None else device
    return int(lib().fa_last_device_error(_stream(dev)))


def _softmax(name, x, out):
    if x.device.type != _DEVICE_TYPE or x.dtype != torch.float32 or not x.is_contiguous() or x.dim() < 1:
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    _on_device(x, "x")
    n = x.shape[-1]
    rows = x.numel() // n if n else 0
    if out is not None:
        _expect(out, "out", x.shape, torch.float32, x.device)
    y = torch.empty_like(x) if out is None else out
    _check(getattr(lib(), name)(_ptr(x), _ptr(y), rows, n, _stream(x.device)), name)
    return y


def softmax_safe(x, out=None):
    """Softmax over the last dimension of fp32 x, three passes per row."""
    return _softmax("fa_softmax_safe", x, out)


def softmax_online(x, out=None):
    """Softmax over the last dimension of fp32 x, two passes per row (online)."""
    return _softmax("fa_softmax_online", x, out)


def attn_merge(o_parts, lse_parts, out=None, lse=None):
    """Combine partial attention results: o_parts [S, rows, d] fp32, lse_parts
    [S, rows] fp32 -> (o [rows, d] bf16, lse [rows] fp32)."""
    _on_device(o_parts, "o_parts")
    S, rows, d = o_parts.shape
    if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
        raise ValueError("o_parts and lse_parts must be float32")
    if lse_parts.shape != (S, rows) or not (o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("lse_parts must be a contiguous [S, rows] tensor beside contiguous o_parts")
    if lse_parts.device != o_parts.device:
        raise ValueError("o_parts and lse_parts must be on one device")
    if out is not None:
        _expect(out, "out", (rows, d), torch.bfloat16, o_parts.device)
    if lse is not None:
        _expect(lse, "lse", (rows,), torch.float32, o_parts.device)
    o = torch.empty((rows, d), dtype=torch.bfloat16, device=o_parts.device) if out is None else out
    lse_t = torch.empty((rows,), dtype=torch.float32, device=o_parts.device) if lse is None else lse
    _check(lib().fa_attn_merge(_ptr(o_parts), _ptr(lse_parts), S, _ptr(o), _ptr(lse_t), rows, d,
                               _stream(o_parts.device)), "fa_attn_merge")
    return o, lse_t


def decode_workspace_bytes(B, H, d, n_splits) -> int:
    return int(lib().fa_decode_workspace_bytes(B, H, d, n_splits))


def decode_paged(q, k_cache, v_cache, block_table, seq_lens, n_splits=1, scale=None, workspace=None,
                 out=None, lse=None):
    """One decode step: q [B, H, d] bf16 against the paged cache k_cache,
    v_cache [num_blocks, Hkv, block_size, d] bf16, with block_table
    [B, max_blocks] int32 and seq_lens [B] int32. Returns (o [B, H, d] bf16,
    lse [B, H] fp32)."""
    B, H, d = q.shape
    num_blocks, Hkv, bs, dk = k_cache.shape
    _on_device(q, "q")
    for t in (q, k_cache, v_cache):
        if t.device != q.device or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k_cache, v_cache must be contiguous bfloat16 CUDA tensors on one device")
    if v_cache.shape != k_cache.shape or dk != d:
        raise ValueError("k_cache and v_cache must be [num_blocks, Hkv, block_size, d]")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32 or block_table.dim() != 2 \
            or block_table.shape[0] != B or seq_lens.shape != (B,) or not block_table.is_contiguous():
        raise ValueError("block_table [B, max_blocks] and seq_lens [B] must be int32")
    _expect(block_table, "block_table", block_table.shape, torch.int32, q.device)
    _expect(seq_lens, "seq_lens", (B,), torch.int32, q.device)
    ws_bytes = decode_workspace_bytes(B, H, d, n_splits)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=q.device)
    _expect_workspace(workspace, q.device)
    if out is not None:
        _expect(out, "out", q.shape, torch.bfloat16, q.device)
    if lse is not None:
        _expect(lse, "lse", (B, H), torch.float32, q.device)
    o = torch.empty_like(q) if out is None else out
    lse_t = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _check(lib().fa_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seq_lens),
                                 _ptr(o), _ptr(lse_t), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), B, H, Hkv, d, num_blocks, bs,
                                 block_table.shape[1], _scale(d, scale), n_splits, _stream(q.device)),
           "fa_decode_paged")
    return o, lse_t


_HOST_NAMES = ("q", "k", "v", "dO", "o", "lse", "dq", "dk", "dv")


def _tensors(ts: dict, on_cuda: bool, shapes: dict, names):
    """Check one side's tensors (shape, dtype, contiguity, device kind) and
    pack their addresses into a Tensors struct."""
    st = Tensors()
    for n in names:
        t = ts.get(n)
        if t is None:
            raise ValueError(f"missing tensor {n!r}")
        want_dtype = torch.float32 if n == "lse" else torch.bfloat16
        if tuple(t.shape) != shapes[n] or t.dtype != want_dtype or not t.is_contiguous():
            raise ValueError(f"{n}: expected a contiguous {want_dtype} tensor of shape {shapes[n]}")
        if (t.device.type == _DEVICE_TYPE) != on_cuda or (not on_cuda and t.device.type != "cpu"):
            raise ValueError(f"{n}: expected a {'CUDA' if on_cuda else 'host'} tensor")
        if on_cuda and t.device != ts[names[0]].device:
            raise ValueError(f"{n}: the device tensors must be on one device")
        setattr(st, n, t.data_ptr())
    return st


def _host_shapes(q, k):
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    qs, kvs = (B, H, N, d), (B, Hkv, N, d)
    return {"q": qs, "k": kvs, "v": kvs, "dO": qs, "o": qs, "lse": (B, H, N), "dq": qs, "dk": kvs,
            "dv": kvs}


def fwd_host(host: dict, dev: dict, causal=False, scale=None, n_chunks=0):
    """Forward from host memory: host["q"], ["k"], ["v"] (CPU, ideally
    pinned) are copied into dev["q"], ["k"], ["v"] (CUDA), the forward runs
    there, and dev["o"], ["lse"] are copied back into host["o"], ["lse"], in
    n_chunks pipelined slices (0: the library's default). Asynchronous on the
    current stream: synchronise it before reading host["o"]."""
    names = ("q", "k", "v", "o", "lse")
    q, k = host["q"], host["k"]
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    shapes = _host_shapes(q, k)
    h = _tensors(host, False, shapes, names)
    dv = _tensors(dev, True, shapes, names)
    _on_device(dev["q"], 'dev["q"]')
    _check(lib().fa_fwd_host(ctypes.byref(h), ctypes.byref(dv), B, H, Hkv, N, d, _scale(d, scale),
                             int(bool(causal)), int(n_chunks), _stream(dev["q"].device)), "fa_fwd_host")


def fwd_bwd_host(host: dict, dev: dict, workspace, causal=False, scale=None, n_chunks=0):
    """Forward and backward from host memory: as fwd_host, plus host["dO"]
    in and host["dq"], ["dk"], ["dv"] out; workspace is a CUDA buffer of
    bwd_workspace_bytes(B, H, N, d) bytes."""
    q, k = host["q"], host["k"]
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    shapes = _host_shapes(q, k)
    h = _tensors(host, False, shapes, _HOST_NAMES)
    dv = _tensors(dev, True, shapes, _HOST_NAMES)
    _on_device(dev["q"], 'dev["q"]')
    _expect_workspace(workspace, dev["q"].device)
    _check(lib().fa_fwd_bwd_host(ctypes.byref(h), ctypes.byref(dv), _ptr(workspace),
                                 workspace.numel() * workspace.element_size(), B, H, Hkv, N, d,
                                 _scale(d, scale), int(bool(causal)), int(n_chunks),
                                 _stream(dev["q"].device)), "fa_fwd_bwd_host")


def softmax_host(x_host, y_host, x_dev, y_dev, online=True, n_chunks=0):
    """Row softmax from host memory: x_host (CPU fp32, ideally pinned) is
    copied into x_dev, normalised into y_dev and copied back into y_host, in
    n_chunks pipelined slices of rows (0: the library's default).
    Asynchronous on the current stream: synchronise it before reading y_host."""
    for t, dev_side in ((x_host, False), (y_host, False), (x_dev, True), (y_dev, True)):
        place_ok = t.device == x_dev.device if dev_side else t.device.type == "cpu"
        if not place_ok or t.dtype != torch.float32 or not t.is_contiguous() or t.shape != x_host.shape:
            raise ValueError("x_host, y_host (CPU) and x_dev, y_dev (CUDA) must be contiguous float32 "
                             "tensors of one shape")
    _on_device(x_dev, "x_dev")
    n = x_host.shape[-1]
    rows = x_host.numel() // n if n else 0
    _check(lib().fa_softmax_host(_ptr(x_host), _ptr(y_host), _ptr(x_dev), _ptr(y_dev), rows, n,
                                 int(bool(online)), int(n_chunks), _stream(x_dev.device)), "fa_softmax_host")
