"""float64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library itself never does, and the
oracle shares no code with the CUDA path: the arithmetic lives in
``attn_ref.c`` (plain C, float64, OpenMP over independent rows), compiled
with the host compiler by :func:`build`.

Every entry point takes arrays of any float dtype (numpy arrays or CPU torch
tensors), widens them exactly to float64 and returns float64 numpy arrays.
bf16 and fp32 values widen to float64 without rounding, so the oracle sees
the very bit patterns handed to the GPU.

Parity status: the forward definition is pinned by brute force, by a library
special case (PyTorch's float64 math SDPA) and by closed-form invariants; the
paged decode gather is pinned by an independent scatter and by the worked
layout numbers of the PagedAttention page.  See ``tests/test_oracle_pins.py``.
The FP8 quantization and the FP8 forward's reference live in ``fp8.py``, pinned
by ``tests/test_oracle_fp8.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)
_ip = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile ``attn_ref.c`` into ``_build/liboracle.so`` (gcc, -fopenmp)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    # -ffp-contract=off keeps every multiply and add a separately rounded
    # float64 operation, exactly as written.
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    lib.oracle_forward.argtypes = [_dp, _dp, _dp, _dp, _dp] + [ctypes.c_long] * 4 + [
        ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_forward_rows.argtypes = [_dp, _dp, _dp, _lp, ctypes.c_long, _dp, _dp] + [
        ctypes.c_long] * 4 + [ctypes.c_double, ctypes.c_int, ctypes.c_int]
    lib.oracle_probs_row.argtypes = [_dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_long,
                                     ctypes.c_double, ctypes.c_int, _dp]
    lib.oracle_paged_decode.argtypes = [_dp, _dp, _dp, _ip, _ip, _dp, _dp] + [
        ctypes.c_long] * 7 + [ctypes.c_double, ctypes.c_int]
    lib.oracle_paged_decode_gqa.argtypes = [_dp, _dp, _dp, _ip, _ip, _dp, _dp] + [
        ctypes.c_long] * 8 + [ctypes.c_double, ctypes.c_int]
    lib.oracle_backward.argtypes = [_dp] * 7 + [ctypes.c_long] * 4 + [ctypes.c_double, ctypes.c_int,
                                                                     ctypes.c_int]
    lib.oracle_forward_masked_rows.argtypes = [_dp, _dp, _dp, ctypes.c_void_p, ctypes.c_long, _lp,
                                               ctypes.c_long, _dp, _dp] + [ctypes.c_long] * 4 + [
        ctypes.c_double, ctypes.c_int]
    lib.oracle_max_threads.argtypes = []
    for f in (lib.oracle_forward, lib.oracle_forward_rows, lib.oracle_probs_row,
              lib.oracle_paged_decode, lib.oracle_paged_decode_gqa, lib.oracle_backward,
              lib.oracle_forward_masked_rows,
              lib.oracle_max_threads):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


class use_library:
    """Context manager that routes every entry point through another build of
    ``attn_ref.c`` (a shared object at ``path``).  The pin tests use it to
    show that a deliberately broken copy of the oracle fails them."""

    def __init__(self, path: str):
        self._new = _bind(ctypes.CDLL(path))
        self._old = None

    def __enter__(self):
        global _lib
        _load()
        with _lock:
            self._old, _lib = _lib, self._new
        return self

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._old
        return False


def compile_variant(source_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source into ``out_path``."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(source_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", "-o", out_path, src, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor: widen on the host, exactly
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray, kind=_dp):
    return a.ctypes.data_as(kind)


def max_threads() -> int:
    """Threads the oracle's OpenMP runtime will use by default."""
    return int(_load().oracle_max_threads())


def attention_forward(q, k, v, scale: float, causal: bool, nthreads: int = 0):
    """Exact attention over [B,H,N,d] inputs.  Returns (O [B,H,N,d], LSE [B,H,N])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B,H,N,d] shape")
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d))
    lse = np.zeros((B, H, N))
    rc = _load().oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                B, H, N, d, float(scale), int(bool(causal)), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_forward rejected its arguments")
    return o, lse


def attention_forward_rows(q, k, v, rows, scale: float, causal: bool, nthreads: int = 0):
    """Exact attention for the listed query rows of every (b,h).

    Returns (O [B,H,len(rows),d], LSE [B,H,len(rows)])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64)).astype(np.int_)
    o = np.zeros((B, H, len(r), d))
    lse = np.zeros((B, H, len(r)))
    rc = _load().oracle_forward_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(r, _lp), len(r),
                                     _ptr(o), _ptr(lse), B, H, N, d, float(scale),
                                     int(bool(causal)), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_forward_rows rejected its arguments")
    return o, lse


def probs_row(q, k, i: int, scale: float, causal: bool):
    """Row i of the softmax matrix P for one head (q, k are [N,d])."""
    q, k = _f64(q), _f64(k)
    N, d = q.shape
    p = np.zeros(N)
    rc = _load().oracle_probs_row(_ptr(q), _ptr(k), N, d, int(i), float(scale),
                                  int(bool(causal)), _ptr(p))
    if rc != 0:
        raise ValueError("oracle_probs_row rejected its arguments")
    return p


def attention_backward(q, k, v, dout, scale: float, causal: bool, nthreads: int = 0):
    """Gradients (dQ, dK, dV), each [B,H,N,d], of the loss whose gradient with
    respect to the attention output is ``dout``."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    if q.ndim != 4 or not (k.shape == v.shape == dout.shape == q.shape):
        raise ValueError("q, k, v, dout must share one [B,H,N,d] shape")
    B, H, N, d = q.shape
    dq, dk, dv = np.zeros(q.shape), np.zeros(q.shape), np.zeros(q.shape)
    rc = _load().oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk),
                                 _ptr(dv), B, H, N, d, float(scale), int(bool(causal)),
                                 int(nthreads))
    if rc != 0:
        raise ValueError("oracle_backward rejected its arguments")
    return dq, dk, dv


def attention_forward_masked(q, k, v, mask, scale: float, rows=None, nthreads: int = 0):
    """Forward with a boolean mask (nonzero = the key is visible).  q, k, v are
    [B,H,N,d]; mask is [N,N] (shared by every head) or [B,H,N,N] / [B*H,N,N].
    Returns (O [B,H,R,d], LSE [B,H,R]) for the query rows `rows` (default all);
    a row with no visible key gives O = 0, LSE = -inf."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or not (k.shape == v.shape == q.shape):
        raise ValueError("q, k, v must share one [B,H,N,d] shape")
    B, H, N, d = q.shape
    if hasattr(mask, "detach"):
        mask = mask.detach().cpu().numpy()
    m = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
    if m.shape == (N, N):
        stride = 0
    elif m.size == B * H * N * N and m.shape[-2:] == (N, N):
        stride = N * N
    else:
        raise ValueError("mask must be [N,N] or one [N,N] per head")
    if rows is None:
        rows = np.arange(N)
    rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    R = rr.shape[0]
    o = np.zeros((B, H, R, d))
    lse = np.zeros((B, H, R))
    rc = _load().oracle_forward_masked_rows(_ptr(q), _ptr(k), _ptr(v),
                                            m.ctypes.data_as(ctypes.c_void_p), stride,
                                            _ptr(rr, _lp), R, _ptr(o), _ptr(lse), B, H, N, d,
                                            float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_forward_masked_rows rejected its arguments")
    return o, lse


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                 nthreads: int = 0):
    """Single-query paged decode.  Returns (out [S,H,D], LSE [S,H]).

    q [S,H,D]; k_cache [nb,Hk,D/x,bs,x]; v_cache [nb,Hk,D,bs] with Hk dividing
    H (Hk = H: one key/value head per query head; else query head h reads
    key/value head h // (H // Hk)); block_tables int [S,max_blocks];
    context_lens int [S]."""
    q, kc, vc = _f64(q), _f64(k_cache), _f64(v_cache)
    bt, cl = _i32(block_tables), _i32(context_lens)
    S, H, D = q.shape
    nb, Hk, Dx, bs, x = kc.shape
    if (Hk <= 0 or H % Hk != 0 or Dx * x != D or vc.shape != (nb, Hk, D, bs) or bt.ndim != 2
            or bt.shape[0] != S):
        raise ValueError("inconsistent paged-cache shapes")
    out = np.zeros((S, H, D))
    lse = np.zeros((S, H))
    if Hk == H:
        rc = _load().oracle_paged_decode(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt, _ip),
                                         _ptr(cl, _ip), _ptr(out), _ptr(lse), S, H, D, bs, x,
                                         bt.shape[1], nb, float(scale), int(nthreads))
    else:
        rc = _load().oracle_paged_decode_gqa(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt, _ip),
                                             _ptr(cl, _ip), _ptr(out), _ptr(lse), S, H, Hk, D,
                                             bs, x, bt.shape[1], nb, float(scale), int(nthreads))
    if rc != 0:
        raise ValueError("oracle paged decode rejected its arguments")
    return out, lse
