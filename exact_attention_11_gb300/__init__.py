"""Python binding of libfattn: exact attention forward, backward and paged decode on GB300.

The C ABI (``include/fattn.h``) is reached through ctypes.  The functions
``fa_forward``, ``fa_forward_fp32``, ``fa_backward`` and ``fa_paged_decode`` take the same
arguments as their C counterparts (device pointers as ints, sizes, a stream
handle) and only marshal them; every step of the computation runs in the CUDA
kernels of ``libfattn.so``.  ``forward``, ``backward`` and ``paged_decode`` are torch
conveniences that allocate the outputs and pass the tensors' device pointers.

There is no fallback: if ``libfattn.so`` is missing, cannot be loaded, or the
device is not an sm_103 GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["fa_forward", "fa_forward_f16", "fa_forward_masked", "forward_masked", "fa_forward_fp32", "fa_paged_decode", "fa_paged_decode_noalloc",
           "fa_backward", "fa_backward_workspace_bytes", "backward", "fa_paged_decode_gqa",
           "fa_decode_gqa_select",
           "fa_status_string", "fa_quantize_fp8", "fa_quantize_fp8_workspace_bytes",
           "fa_fp8_vt_stride", "fa_forward_fp8", "quantize_fp8", "forward_fp8", "Fp8Inputs",
           "fa_device_status", "fa_release", "forward", "paged_decode", "FattnError",
           "library_path", "load"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libfattn.so")
_lock = threading.Lock()
_lib = None

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", -1: "FA_ERR_INVALID_ARG", -2: "FA_ERR_UNSUPPORTED",
                -3: "FA_ERR_ALIGNMENT", -4: "FA_ERR_CUDA", -5: "FA_ERR_TIMEOUT",
                -6: "FA_ERR_NO_MEMORY", -7: "FA_ERR_NO_DEVICE"}


class FattnError(RuntimeError):
    def __init__(self, func: str, status: int):
        self.status = status
        super().__init__(f"{func} failed: {STATUS_NAMES.get(status, status)} "
                         f"({fa_status_string(status)})")


def library_path() -> str:
    return _LIB_PATH


_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
EXPORTS = {
    "fa_forward": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_forward_fp32": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_forward_f16": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_forward_masked": ([_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_longlong, _i, _i, _i, _i, _f,
                           _vp], _i),
    "fa_paged_decode": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_paged_decode_noalloc": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_paged_decode_gqa": ([_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp], _i),
    "fa_backward_workspace_bytes": ([_i, _i, _i, _i], ctypes.c_ulonglong),
    "fa_backward": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp,
                     ctypes.c_ulonglong, _vp], _i),
    "fa_quantize_fp8_workspace_bytes": ([_i, _i, _i, _i], ctypes.c_ulonglong),
    "fa_fp8_vt_stride": ([_i], ctypes.c_longlong),
    "fa_quantize_fp8": ([_vp] * 10 + [_i, _i, _i, _i, _vp, ctypes.c_ulonglong, _vp], _i),
    "fa_forward_fp8": ([_vp] * 8 + [_i, _i, _i, _i, _f, _i, _vp], _i),
    "fa_status_string": ([_i], ctypes.c_char_p),
    "fa_device_status": ([], _i),
    "fa_release": ([], None),
    "fa_debug_inject_fault": ([_i], _i),
    "fa_decode_gqa_select": ([_i], _i),
    "fa_version": ([], _i),
}


def load():
    """Loads libfattn.so (raising if it is absent) and declares its exports."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libfattn.so not found at {_LIB_PATH}; build it with "
                "`python -m exact_attention_11_gb300._build` (needs nvcc)")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (args, res) in EXPORTS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(name: str, rc: int) -> int:
    if rc != FA_OK:
        raise FattnError(name, rc)
    return rc


# ---------------------------------------------------------------- raw C ABI
def fa_forward(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    return _check("fa_forward", load().fa_forward(q, k, v, o, lse, B, H, N, d, scale,
                                                  int(causal), stream))


def fa_forward_f16(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    return _check("fa_forward_f16", load().fa_forward_f16(q, k, v, o, lse, B, H, N, d, scale,
                                                          int(causal), stream))


def fa_forward_masked(q, k, v, o, lse, mask, mask_bh_stride, B, H, N, d, scale, stream) -> int:
    return _check("fa_forward_masked", load().fa_forward_masked(
        q, k, v, o, lse, mask, mask_bh_stride, B, H, N, d, scale, stream))


def fa_forward_fp32(q, k, v, o, lse, B, H, N, d, scale, causal, stream) -> int:
    return _check("fa_forward_fp32", load().fa_forward_fp32(q, k, v, o, lse, B, H, N, d, scale,
                                                            int(causal), stream))


def fa_paged_decode(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, num_heads,
                    head_size, block_size, max_num_blocks_per_seq, scale, stream) -> int:
    return _check("fa_paged_decode", load().fa_paged_decode(
        q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, num_heads, head_size,
        block_size, max_num_blocks_per_seq, scale, stream))


def fa_paged_decode_gqa(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs,
                        num_heads, num_kv_heads, head_size, block_size, max_num_blocks_per_seq,
                        scale, stream) -> int:
    return _check("fa_paged_decode_gqa", load().fa_paged_decode_gqa(
        q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, num_heads, num_kv_heads,
        head_size, block_size, max_num_blocks_per_seq, scale, stream))


def fa_paged_decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, out, num_seqs,
                            num_heads, head_size, block_size, max_num_blocks_per_seq, scale,
                            stream) -> int:
    """fa_paged_decode for callers that cannot allocate device memory during
    the call (a process whose memory pool owns all of HBM, a loop that cannot
    afford cudaMalloc's synchronisation).  The split-K scratch is a fixed
    12 MiB device array inside the library; larger problems raise
    FattnError(FA_ERR_UNSUPPORTED).  All calls on a device share that array,
    so calls that overlap on the GPU must not be issued; the first call on a
    device should come before any stream capture."""
    return _check("fa_paged_decode_noalloc", load().fa_paged_decode_noalloc(
        q, k_cache, v_cache, block_tables, context_lens, out, num_seqs, num_heads, head_size,
        block_size, max_num_blocks_per_seq, scale, stream))


def fa_backward_workspace_bytes(B, H, N, d) -> int:
    return int(load().fa_backward_workspace_bytes(B, H, N, d))


def fa_backward(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                workspace_bytes, stream) -> int:
    return _check("fa_backward", load().fa_backward(
        q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, int(causal), workspace,
        workspace_bytes, stream))


def fa_quantize_fp8_workspace_bytes(B, H, N, d) -> int:
    return int(load().fa_quantize_fp8_workspace_bytes(B, H, N, d))


def fa_fp8_vt_stride(N) -> int:
    return int(load().fa_fp8_vt_stride(N))


def fa_quantize_fp8(q, k, v, signs, q8, k8, vt8, q_scale, k_scale, v_scale, B, H, N, d,
                    workspace, workspace_bytes, stream) -> int:
    return _check("fa_quantize_fp8", load().fa_quantize_fp8(
        q, k, v, signs, q8, k8, vt8, q_scale, k_scale, v_scale, B, H, N, d, workspace,
        workspace_bytes, stream))


def fa_forward_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, B, H, N, d, scale, causal,
                   stream) -> int:
    return _check("fa_forward_fp8", load().fa_forward_fp8(
        q8, k8, vt8, q_scale, k_scale, v_scale, o, lse, B, H, N, d, scale, int(causal), stream))


def fa_status_string(status: int) -> str:
    try:
        return load().fa_status_string(status).decode()
    except Exception:  # library missing: still give a name
        return STATUS_NAMES.get(status, "unknown")


def fa_device_status() -> int:
    return load().fa_device_status()


def fa_release() -> None:
    load().fa_release()


def fa_debug_inject_fault(mode: int) -> int:
    """Test hook: arm a lost-copy fault in the next forward (1) or backward
    (2) launch on the current device, or disarm (0) (see fattn.h)."""
    return _check("fa_debug_inject_fault", load().fa_debug_inject_fault(mode))


def fa_decode_gqa_select(impl: int) -> int:
    """Kernel for fa_paged_decode_gqa: 0 = automatic (default), 1 = the
    CUDA-core kernel only, 2 = the tensor-core kernel only (see fattn.h)."""
    return _check("fa_decode_gqa_select", load().fa_decode_gqa_select(impl))


# ---------------------------------------------------------------- torch helpers
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(t):
    import torch
    return torch.cuda.current_stream(t.device).cuda_stream


def forward(q, k, v, scale=None, causal=False, out=None, lse=None, want_lse=True):
    """Exact attention on [B,H,N,d] CUDA tensors (bf16, fp16 or fp32, contiguous).

    Returns (O, LSE) with O in the input dtype and LSE fp32 [B,H,N] (None when
    ``want_lse`` is False).  Runs on the current torch stream."""
    import torch
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B,H,N,d] shape")
    if not (q.is_cuda and q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous CUDA tensors")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in (torch.bfloat16, torch.float16,
                                                                torch.float32):
        raise ValueError("q, k, v must all be bf16, all fp16 or all fp32")
    B, H, N, d = q.shape
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fn = {torch.bfloat16: fa_forward, torch.float16: fa_forward_f16,
          torch.float32: fa_forward_fp32}[q.dtype]
    fn(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, float(scale), bool(causal),
       _stream(q))
    return out, lse


def forward_masked(q, k, v, mask, scale=None, out=None, lse=None):
    """Exact attention with a boolean mask on bf16 [B,H,N,d] CUDA tensors.
    mask: bool or uint8 CUDA tensor, [N,N] (shared) or [B,H,N,N] (nonzero =
    visible).  Returns (O, LSE); rows with no visible key give O = 0,
    LSE = -inf."""
    import torch
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B,H,N,d] shape")
    for t in (q, k, v):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    B, H, N, d = q.shape
    m = mask.to(torch.uint8) if mask.dtype == torch.bool else mask
    if not (m.is_cuda and m.is_contiguous() and m.dtype == torch.uint8):
        raise ValueError("mask must be a contiguous bool or uint8 CUDA tensor")
    if tuple(m.shape) == (N, N):
        stride = 0
    elif tuple(m.shape) == (B, H, N, N):
        stride = N * N
    else:
        raise ValueError("mask must be [N,N] or [B,H,N,N]")
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_forward_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(m), stride, B, H, N,
                      d, float(scale), _stream(q))
    return out, lse


def backward(q, k, v, o, lse, dout, scale=None, causal=False, workspace=None):
    """Gradients (dQ, dK, dV) of the bf16 forward on [B,H,N,d] CUDA tensors.

    ``o`` and ``lse`` are what ``forward`` returned for the same q, k, v,
    scale and causal.  ``workspace`` (optional) is a CUDA tensor of at least
    ``fa_backward_workspace_bytes`` bytes; one is allocated when it is None.
    Runs on the current torch stream."""
    import torch
    for t in (q, k, v, o, dout):
        if t.dim() != 4 or t.shape != q.shape:
            raise ValueError("q, k, v, o, dout must share one [B,H,N,d] shape")
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("q, k, v, o, dout must be contiguous bf16 CUDA tensors")
    B, H, N, d = q.shape
    if lse is None or tuple(lse.shape) != (B, H, N) or lse.dtype != torch.float32 \
            or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B,H,N] tensor")
    if scale is None:
        scale = d ** -0.5
    nbytes = fa_backward_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk),
                _ptr(dv), B, H, N, d, float(scale), bool(causal), _ptr(workspace), ws_bytes,
                _stream(q))
    return dq, dk, dv


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale=None, out=None):
    """Single-query paged decode on CUDA tensors in the layouts of fattn.h.
    The caches' second axis is the key/value head count Hk; Hk < H selects
    the grouped-head decode (fa_paged_decode_gqa)."""
    import torch
    S, H, D = q.shape
    nb, Hk, Dx, bs, x = k_cache.shape
    if Hk <= 0 or H % Hk != 0 or Dx * x != D or tuple(v_cache.shape) != (nb, Hk, D, bs):
        raise ValueError("inconsistent cache shapes")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    for t in (q, k_cache, v_cache, block_tables, context_lens):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError("all decode inputs must be contiguous CUDA tensors")
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if Hk == H:
        fa_paged_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                        _ptr(context_lens), _ptr(out), S, H, D, bs, block_tables.shape[1],
                        float(scale), _stream(q))
    else:
        fa_paged_decode_gqa(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            _ptr(context_lens), _ptr(out), S, H, Hk, D, bs,
                            block_tables.shape[1], float(scale), _stream(q))
    return out


class Fp8Inputs:
    """E4M3 codes and dequantization scales of one attention problem, in the
    layouts of fa_quantize_fp8: q8, k8 uint8 [B,H,N,d]; vt8 uint8 [B,H,d,Npad]
    (V transposed); q_scale, k_scale fp32 [B,H,ceil(N/128)]; v_scale fp32
    [B,H]."""

    def __init__(self, q8, k8, vt8, q_scale, k_scale, v_scale, shape):
        self.q8, self.k8, self.vt8 = q8, k8, vt8
        self.q_scale, self.k_scale, self.v_scale = q_scale, k_scale, v_scale
        self.shape = tuple(shape)


def quantize_fp8(q, k, v, signs=None, workspace=None, out=None):
    """Block-quantizes bf16 [B,H,N,128] CUDA tensors to E4M3 (fa_quantize_fp8).
    ``signs``: optional fp32 CUDA tensor of 128 values +-1 for the random
    orthogonal transform of q and k.  ``out``: an Fp8Inputs of the same shape
    to write into.  Returns an Fp8Inputs.  Runs on the current torch stream."""
    import torch
    for t in (q, k, v):
        if t.dim() != 4 or t.shape != q.shape:
            raise ValueError("q, k, v must share one [B,H,N,d] shape")
        if not (t.is_cuda and t.is_contiguous() and t.dtype == torch.bfloat16):
            raise ValueError("q, k, v must be contiguous bf16 CUDA tensors")
    B, H, N, d = q.shape
    if signs is not None and not (signs.is_cuda and signs.is_contiguous()
                                  and signs.dtype == torch.float32 and signs.numel() == d):
        raise ValueError("signs must be a contiguous fp32 CUDA tensor of d values")
    if out is None:
        dev = q.device
        nblk = (N + 127) // 128
        npad = fa_fp8_vt_stride(N)
        out = Fp8Inputs(torch.empty((B, H, N, d), dtype=torch.uint8, device=dev),
                        torch.empty((B, H, N, d), dtype=torch.uint8, device=dev),
                        torch.empty((B, H, d, npad), dtype=torch.uint8, device=dev),
                        torch.empty((B, H, nblk), dtype=torch.float32, device=dev),
                        torch.empty((B, H, nblk), dtype=torch.float32, device=dev),
                        torch.empty((B, H), dtype=torch.float32, device=dev), q.shape)
    elif out.shape != tuple(q.shape):
        raise ValueError("out was made for another shape")
    nbytes = fa_quantize_fp8_workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=q.device)
    fa_quantize_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(signs), _ptr(out.q8), _ptr(out.k8),
                    _ptr(out.vt8), _ptr(out.q_scale), _ptr(out.k_scale), _ptr(out.v_scale),
                    B, H, N, d, _ptr(workspace), workspace.numel() * workspace.element_size(),
                    _stream(q))
    return out


def forward_fp8(x, scale=None, causal=False, out=None, lse=None, want_lse=True):
    """The FP8 forward (fa_forward_fp8) on an Fp8Inputs.  Returns (O bf16
    [B,H,N,d], LSE fp32 [B,H,N] or None).  Runs on the current torch stream."""
    import torch
    B, H, N, d = x.shape
    if scale is None:
        scale = d ** -0.5
    dev = x.q8.device
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa_forward_fp8(_ptr(x.q8), _ptr(x.k8), _ptr(x.vt8), _ptr(x.q_scale), _ptr(x.k_scale),
                   _ptr(x.v_scale), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                   bool(causal), _stream(x.q8))
    return out, lse
