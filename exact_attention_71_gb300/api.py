"""ctypes binding of libattn_sm103.so (argument marshalling only).

Every step of the attention path runs in the library's CUDA kernels; torch
is used here for device memory, streams and the tensor objects that carry
the pointers.  There is no fallback: if the library is missing or cannot be
loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libattn_sm103.so")

MODE_BLOCK, MODE_BLOCK_HADAMARD, MODE_PER_TENSOR = 0, 1, 2
BLOCK_ROWS = 128

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A call into the attention library returned an error status."""

    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed ({code}): {msg}")
        self.code = code


def library() -> ctypes.CDLL:
    """Load the shared library (built by ``exact_attention_71_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m exact_attention_71_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        P, i, f, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_ulonglong
        L.attn_fwd.argtypes = [P, P, P, P, P, i, i, i, i, i, f, i, P]
        L.attn_fwd.restype = i
        L.attn_fwd_fp8.argtypes = [P, P, P, P, P, i, i, i, i, i, f, i, P, P, P, P]
        L.attn_fwd_fp8.restype = i
        L.attn_fwd_gqa.argtypes = [P, P, P, P, P, i, i, i, i, i, i, f, i, P]
        L.attn_fwd_gqa.restype = i
        L.attn_fwd_fp8_gqa.argtypes = [P, P, P, P, P, i, i, i, i, i, i, f, i, P, P, P, P]
        L.attn_fwd_fp8_gqa.restype = i
        L.attn_fp8_prep.argtypes = [P, P, P, i, i, i, i, i, i, u64, i, P]
        L.attn_fp8_prep_qkv.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, u64, P]
        L.attn_fp8_prep_qkv.restype = i
        L.attn_fp8_prep_rope.argtypes = [P, P, P, P, P, i, i, i, i, i, i, u64, i, P]
        L.attn_fp8_prep_rope.restype = i
        L.attn_fp8_prep.restype = i
        L.attn_fwd_sparse.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, f, i, P]
        L.attn_fwd_sparse.restype = i
        sz = ctypes.c_size_t
        L.attn_bwd_workspace_size.argtypes = [i, i, i, i]
        L.attn_bwd_workspace_size.restype = sz
        L.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, sz, i, i, i, i, i, i, f, i, P]
        L.attn_bwd.restype = i
        L.attn_bwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, f, i, P]
        L.attn_bwd_noalloc.restype = i
        L.attn_bwd_noalloc_max_scratch.argtypes = []
        L.attn_bwd_noalloc_max_scratch.restype = sz
        L.attn_fwd_host_workspace_size.argtypes = [i, i, i, i, i]
        L.attn_fwd_host_workspace_size.restype = sz
        L.attn_fwd_host.argtypes = [P, P, P, P, P, i, i, i, i, i, i, f, i, P, sz, P]
        L.attn_fwd_host.restype = i
        L.attn_fwd_fp8_host_workspace_size.argtypes = [i, i, i, i, i]
        L.attn_fwd_fp8_host_workspace_size.restype = sz
        L.attn_fwd_fp8_host.argtypes = [P, P, P, P, P, i, i, i, i, i, i, f, i, i, u64, P, sz, P]
        L.attn_fwd_fp8_host.restype = i
        L.attn_bwd_host_workspace_size.argtypes = [i, i, i, i, i]
        L.attn_bwd_host_workspace_size.restype = sz
        L.attn_bwd_host.argtypes = [P, P, P, P, P, P, P, P, P, i, i, i, i, i, i, f, i, P, sz, P]
        L.attn_bwd_host.restype = i
        L.attn_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
        L.attn_device_status.restype = i
        L.attn_set_wait_limit.argtypes = [u64]
        L.attn_set_wait_limit.restype = i
        L.attn_last_error_string.argtypes = []
        L.attn_last_error_string.restype = ctypes.c_char_p
        L.attn_fwd_work_order.argtypes = [i, i, i, P, i]
        L.attn_fwd_work_order.restype = i
        _lib = L
        return _lib


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        msg = library().attn_last_error_string().decode(errors="replace")
        raise AttnError(fn, rc, msg)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _torch_stream(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


def _hold_until_done(t, stream):
    """A workspace allocated here is still in use after this function
    returns, by work on `stream` or (host-buffer entries) on the library's
    own streams, which `stream` waits for; recording the tensor on `stream`
    keeps torch's caching allocator from handing the memory out again before
    that work is done."""
    t.record_stream(_torch_stream(stream, t.device))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _check_qkv(q, k, v, dtype):
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q must be (B, N, H, d) and k, v one (B, N, H_kv, d) shape")
    B, N, H, d = q.shape
    if k.shape[0] != B or k.shape[1] != N or k.shape[3] != d or H % k.shape[2] != 0:
        raise ValueError("k, v must be (B, N, H_kv, d) with H_kv dividing the query heads")
    for t in (q, k, v):
        if t.dtype != dtype:
            raise ValueError(f"expected dtype {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")


def _outputs(q, out, lse):
    B, N, H, d = q.shape
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if out.shape != (B, N, H, d) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 (B, N, H, d) tensor")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, N) tensor")
    return out, lse


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, window: int = 0,
             out=None, lse=None, stream=None):
    """bf16 fused attention forward.  q: (B, N, H, d); k, v: (B, N, H_kv, d)
    bf16 CUDA tensors, H_kv dividing H (H_kv < H: grouped-query attention).

    Returns (O (B, N, H, d) bf16, LSE (B, H, N) float32, natural log).
    """
    _check_qkv(q, k, v, torch.bfloat16)
    out, lse = _outputs(q, out, lse)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if Hkv == H:
        rc = library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, int(bool(causal)),
                                float(scale or 0.0), int(window), ctypes.c_void_p(_stream(stream)))
        _check("attn_fwd", rc)
    else:
        rc = library().attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                                    int(bool(causal)), float(scale or 0.0), int(window),
                                    ctypes.c_void_p(_stream(stream)))
        _check("attn_fwd_gqa", rc)
    return out, lse


def fwd_host_workspace_bytes(B: int, H: int, H_kv: int, N: int, d: int) -> int:
    return int(library().attn_fwd_host_workspace_size(B, H, H_kv, N, d))


def attn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, window: int = 0,
                  out=None, lse=None, workspace=None, device=None, stream=None):
    """attn_fwd on HOST tensors: q (B, N, H, d), k, v (B, N, H_kv, d) bf16 CPU
    tensors (page-locked, e.g. ``.pin_memory()``, for overlapped copies).
    The library stages chunks of sequences through ``workspace`` (a uint8
    CUDA tensor of at least fwd_host_workspace_bytes(...) bytes, allocated
    here when omitted) on ``device``.  Returns host (O, LSE); the call is
    asynchronous on ``stream``: synchronize it before reading them.
    """
    B, N, H, Hkv, d, out, lse = _host_args(q, k, v, out, lse)
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    need = fwd_host_workspace_bytes(B, H, Hkv, N, d)
    own = workspace is None
    if own:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    with torch.cuda.device(workspace.device):
        rc = library().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                                     int(bool(causal)), float(scale or 0.0), int(window), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     ctypes.c_void_p(_stream(stream)))
    _check("attn_fwd_host", rc)
    if own:
        _hold_until_done(workspace, stream)
    return out, lse


def fwd_fp8_host_workspace_bytes(B: int, H: int, H_kv: int, N: int, d: int) -> int:
    return int(library().attn_fwd_fp8_host_workspace_size(B, H, H_kv, N, d))


def _host_args(q, k, v, out, lse):
    for t in (q, k, v):
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v must be contiguous 4-d bf16 CPU tensors")
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[1] != N or k.shape[3] != d or H % Hkv != 0:
        raise ValueError("k, v must be (B, N, H_kv, d) with H_kv dividing the query heads")
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.bfloat16, pin_memory=pin)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=pin)
    if out.is_cuda or out.shape != (B, N, H, d) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 (B, N, H, d) CPU tensor")
    if lse.is_cuda or lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, N) CPU tensor")
    return B, N, H, Hkv, d, out, lse


def attn_fwd_fp8_host(q, k, v, mode: int = MODE_BLOCK_HADAMARD, sign_seed: int = 0, causal: bool = False,
                      scale: float | None = None, window: int = 0, out=None, lse=None, workspace=None, device=None,
                      stream=None):
    """The FP8 path on HOST bf16 tensors (prep + e4m3 forward per chunk of
    sequences, staged and overlapped like attn_fwd_host).  mode: MODE_BLOCK or
    MODE_BLOCK_HADAMARD.  Returns host (O, LSE); asynchronous on ``stream``."""
    B, N, H, Hkv, d, out, lse = _host_args(q, k, v, out, lse)
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    own = workspace is None
    if own:
        need = fwd_fp8_host_workspace_bytes(B, H, Hkv, N, d)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    with torch.cuda.device(workspace.device):
        rc = library().attn_fwd_fp8_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                                         int(bool(causal)), float(scale or 0.0), int(window), int(mode),
                                         int(sign_seed) & 0xFFFFFFFFFFFFFFFF, _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         ctypes.c_void_p(_stream(stream)))
    _check("attn_fwd_fp8_host", rc)
    if own:
        _hold_until_done(workspace, stream)
    return out, lse


def attn_fwd_sparse(q, k, v, block_mask, causal: bool = False, scale: float | None = None, window: int = 0,
                    out=None, lse=None, stream=None):
    """bf16 forward with a block-sparse key mask: block_mask is a uint8 (or
    bool) CUDA tensor (B, H, T, T), T = ceil(N / 128); query block i of
    (b, h) sees key block j iff block_mask[b, h, i, j] != 0 (ANDed with the
    causal / window masks).  Rows that see no key get O = 0, LSE = -inf."""
    _check_qkv(q, k, v, torch.bfloat16)
    out, lse = _outputs(q, out, lse)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    T = (N + 127) // 128
    if block_mask.dtype == torch.bool:
        block_mask = block_mask.to(torch.uint8)
    if (block_mask.dtype != torch.uint8 or not block_mask.is_cuda or not block_mask.is_contiguous()
            or tuple(block_mask.shape) != (B, H, T, T)):
        raise ValueError(f"block_mask must be a contiguous uint8 CUDA tensor of shape ({B}, {H}, {T}, {T})")
    rc = library().attn_fwd_sparse(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(block_mask), B, H, Hkv, N,
                                   d, int(bool(causal)), float(scale or 0.0), int(window),
                                   ctypes.c_void_p(_stream(stream)))
    _check("attn_fwd_sparse", rc)
    return out, lse


def bwd_host_workspace_bytes(B: int, H: int, H_kv: int, N: int, d: int) -> int:
    return int(library().attn_bwd_host_workspace_size(B, H, H_kv, N, d))


def attn_bwd_host(dout, q, k, v, out, lse, causal: bool = False, scale: float | None = None, window: int = 0,
                  dq=None, dk=None, dv=None, workspace=None, device=None, stream=None):
    """attn_bwd on HOST tensors (bf16 CPU q, dout, out (B, N, H, d); k, v
    (B, N, H_kv, d); float32 lse (B, H, N)), staged through ``workspace`` (at
    least bwd_host_workspace_bytes(...) bytes on ``device``) like
    attn_fwd_host.  Returns host (dq, dk, dv); asynchronous on ``stream``."""
    B, N, H, Hkv, d, _, _ = _host_args(q, k, v, out, lse)
    if dout.is_cuda or dout.shape != q.shape or dout.dtype != torch.bfloat16 or not dout.is_contiguous():
        raise ValueError("dout must be a contiguous bf16 CPU tensor shaped like q")
    pin = q.is_pinned()
    dq = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pin) if dq is None else dq
    dk = torch.empty(k.shape, dtype=torch.bfloat16, pin_memory=pin) if dk is None else dk
    dv = torch.empty(v.shape, dtype=torch.bfloat16, pin_memory=pin) if dv is None else dv
    for t, ref in ((dq, q), (dk, k), (dv, v)):
        if t.is_cuda or t.shape != ref.shape or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("dq, dk, dv must be contiguous bf16 CPU tensors shaped like q, k, v")
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    own = workspace is None
    if own:
        workspace = torch.empty(max(bwd_host_workspace_bytes(B, H, Hkv, N, d), 256), dtype=torch.uint8,
                                device=device)
    with torch.cuda.device(workspace.device):
        rc = library().attn_bwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                     _ptr(dk), _ptr(dv), B, H, Hkv, N, d, int(bool(causal)), float(scale or 0.0),
                                     int(window), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     ctypes.c_void_p(_stream(stream)))
    _check("attn_bwd_host", rc)
    if own:
        _hold_until_done(workspace, stream)
    return dq, dk, dv


def bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(library().attn_bwd_workspace_size(B, H, N, d))


def attn_bwd(dout, q, k, v, out, lse, causal: bool = False, scale: float | None = None, window: int = 0,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of attn_fwd: (dq, dk, dv) for the upstream gradient dout.

    q, dout, out: bf16 (B, N, H, d); k, v: bf16 (B, N, H_kv, d); lse: the
    forward's float32 (B, H, N).  workspace: optional uint8 CUDA tensor of at
    least bwd_workspace_bytes(B, H, N, d) bytes (allocated per call when
    omitted).
    """
    _check_qkv(q, k, v, torch.bfloat16)
    for t, name in ((dout, "dout"), (out, "out")):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != q.device:
            raise ValueError(f"{name} must be a contiguous bf16 tensor shaped like q")
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if lse.shape != (B, H, N) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 (B, H, N) tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = bwd_workspace_bytes(B, H, N, d)
    own = workspace is None
    if own:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = library().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                            _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(), B, H, Hkv, N, d,
                            int(bool(causal)), float(scale or 0.0), int(window), ctypes.c_void_p(_stream(stream)))
    _check("attn_bwd", rc)
    if own and stream is not None:
        _hold_until_done(workspace, stream)   # the launches run on `stream`, not torch's current one
    return dq, dk, dv


def attn_bwd_noalloc(dout, q, k, v, out, lse, causal: bool = False, scale: float | None = None, window: int = 0,
                     dq=None, dk=None, dv=None, stream=None):
    """attn_bwd without a workspace: the library's built-in device scratch
    buffer is used instead (for callers that may not allocate; calls on one
    device must not overlap on the GPU).  dq, dk, dv are allocated here only
    when not given."""
    _check_qkv(q, k, v, torch.bfloat16)
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    rc = library().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq),
                                    _ptr(dk), _ptr(dv), B, H, Hkv, N, d, int(bool(causal)), float(scale or 0.0),
                                    int(window), ctypes.c_void_p(_stream(stream)))
    _check("attn_bwd_noalloc", rc)
    return dq, dk, dv


def attn_fp8_prep(x, mode: int = MODE_BLOCK_HADAMARD, sign_seed: int = 0, is_v: bool = False,
                  out=None, scales=None, stream=None):
    """Rotation (mode 1, not V) + block quantisation of one bf16 (B,N,H,d) tensor.

    Returns (codes as a torch.uint8 (B,N,H,d) tensor, scales float32 (B,H,ceil(N/128))).
    """
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 4 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 (B, N, H, d) CUDA tensor")
    B, N, H, d = x.shape
    nblk = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    rc = library().attn_fp8_prep(_ptr(x), _ptr(out), _ptr(scales), B, H, N, d, BLOCK_ROWS, int(mode),
                                 int(sign_seed) & 0xFFFFFFFFFFFFFFFF, int(bool(is_v)),
                                 ctypes.c_void_p(_stream(stream)))
    _check("attn_fp8_prep", rc)
    return out, scales


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool = False, scale: float | None = None,
                 window: int = 0, out=None, lse=None, stream=None):
    """FP8 e4m3 fused attention forward on codes from attn_fp8_prep.

    q8, k8, v8: uint8 (or float8_e4m3fn) (B, N, H, d) CUDA tensors; *_scale:
    float32 (B, H, ceil(N/128)).  Returns (O bf16 (B,N,H,d), LSE (B,H,N)).
    """
    for t in (q8, k8, v8):
        if t.dtype not in (torch.uint8, torch.float8_e4m3fn) or not t.is_cuda or not t.is_contiguous():
            raise ValueError("q8, k8, v8 must be contiguous e4m3 codes on the GPU")
    if q8.dim() != 4 or k8.dim() != 4 or k8.shape != v8.shape:
        raise ValueError("q8 must be (B, N, H, d) and k8, v8 one (B, N, H_kv, d) shape")
    B, N, H, d = q8.shape
    Hkv = k8.shape[2]
    if k8.shape[0] != B or k8.shape[1] != N or k8.shape[3] != d or H % Hkv != 0:
        raise ValueError("k8, v8 must be (B, N, H_kv, d) with H_kv dividing the query heads")
    nblk = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    for s, heads in ((q_scale, H), (k_scale, Hkv), (v_scale, Hkv)):
        if s.shape != (B, heads, nblk) or s.dtype != torch.float32 or not s.is_contiguous():
            raise ValueError("scales must be contiguous float32 (B, heads, ceil(N/128)) tensors")
    out, lse = _outputs(q8, out, lse)
    rc = library().attn_fwd_fp8_gqa(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                                    int(bool(causal)), float(scale or 0.0), int(window), _ptr(q_scale),
                                    _ptr(k_scale), _ptr(v_scale), ctypes.c_void_p(_stream(stream)))
    _check("attn_fwd_fp8_gqa", rc)
    return out, lse


def attn_fp8_prep_rope(x, rope_cos, rope_sin, mode: int = MODE_BLOCK_HADAMARD, sign_seed: int = 0,
                       interleaved: bool = False, out=None, scales=None, stream=None):
    """RoPE fused with the FP8 prep of Q or K: each row of token n is turned
    by the (N, d/2) float32 cos / sin tables (pairs (i, i + d/2), or (2i, 2i+1)
    when interleaved), then rotated (mode 1) and block-quantised.

    Returns (codes uint8 (B,N,H,d), scales float32 (B,H,ceil(N/128))).
    """
    if not x.is_cuda or x.dtype != torch.bfloat16 or x.dim() != 4 or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 (B, N, H, d) CUDA tensor")
    B, N, H, d = x.shape
    for t in (rope_cos, rope_sin):
        if (not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or t.shape != (N, d // 2)
                or t.device != x.device):
            raise ValueError("rope_cos / rope_sin must be contiguous float32 (N, d/2) tensors on x's device")
    nblk = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((B, H, nblk), dtype=torch.float32, device=x.device)
    rc = library().attn_fp8_prep_rope(_ptr(x), _ptr(out), _ptr(scales), _ptr(rope_cos), _ptr(rope_sin),
                                      B, H, N, d, BLOCK_ROWS, int(mode), int(sign_seed) & 0xFFFFFFFFFFFFFFFF,
                                      int(bool(interleaved)), ctypes.c_void_p(_stream(stream)))
    _check("attn_fp8_prep_rope", rc)
    return out, scales


def attn_fp8_prep_qkv(q, k, v, mode: int = MODE_BLOCK_HADAMARD, sign_seed: int = 0, stream=None):
    """The prep of Q, K (rotated in mode 1) and V (never rotated) in one call
    (one launch for modes 0 and 1 at head dims 64 and 128).

    Returns (q8, k8, v8, q_scale, k_scale, v_scale)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous bf16 (B, N, H, d) CUDA tensor")
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, N, Hkv, d) or v.shape != k.shape:
        raise ValueError("k and v must be (B, N, H_kv, d) with q's B, N and d")
    nblk = (N + BLOCK_ROWS - 1) // BLOCK_ROWS
    q8 = torch.empty((B, N, H, d), dtype=torch.uint8, device=q.device)
    k8 = torch.empty((B, N, Hkv, d), dtype=torch.uint8, device=q.device)
    v8 = torch.empty((B, N, Hkv, d), dtype=torch.uint8, device=q.device)
    qs = torch.empty((B, H, nblk), dtype=torch.float32, device=q.device)
    ks = torch.empty((B, Hkv, nblk), dtype=torch.float32, device=q.device)
    vs = torch.empty((B, Hkv, nblk), dtype=torch.float32, device=q.device)
    rc = library().attn_fp8_prep_qkv(_ptr(q), _ptr(k), _ptr(v), _ptr(q8), _ptr(k8), _ptr(v8), _ptr(qs), _ptr(ks),
                                     _ptr(vs), B, H, Hkv, N, d, int(mode), int(sign_seed) & 0xFFFFFFFFFFFFFFFF,
                                     ctypes.c_void_p(_stream(stream)))
    _check("attn_fp8_prep_qkv", rc)
    return q8, k8, v8, qs, ks, vs


def fp8_prepare_qkv(q, k, v, mode: int = MODE_BLOCK_HADAMARD, sign_seed: int = 0, stream=None, rope=None):
    """Runs the prep on Q, K (rotated in mode 1) and V (never rotated), one
    launch where the library has it (attn_fp8_prep_qkv).
    rope: optional (cos, sin, interleaved); RoPE is then fused into the prep
    of Q and K."""
    if rope is None:
        return attn_fp8_prep_qkv(q, k, v, mode, sign_seed, stream=stream)
    else:
        c, s_, il = rope
        q8, qs = attn_fp8_prep_rope(q, c, s_, mode, sign_seed, il, stream=stream)
        k8, ks = attn_fp8_prep_rope(k, c, s_, mode, sign_seed, il, stream=stream)
    v8, vs = attn_fp8_prep(v, mode, sign_seed, True, stream=stream)
    return q8, k8, v8, qs, ks, vs


def device_status(stream=None):
    """(status, site): waits for the stream and reads/clears the status word."""
    site = ctypes.c_int(0)
    rc = library().attn_device_status(ctypes.c_void_p(_stream(stream)), ctypes.byref(site))
    return rc, site.value


def fwd_work_order(n_mblocks: int, bh: int, grid: int):
    """The causal d=128 forward's work order (host only): a list of
    (query block, batch*head) per item, or None where the launch uses the
    closed-form order."""
    n = n_mblocks * bh
    buf = (ctypes.c_uint * max(n, 1))()
    got = library().attn_fwd_work_order(n_mblocks, bh, grid, ctypes.cast(buf, ctypes.c_void_p), n)
    if got == 0:
        return None
    return [(buf[k] & 0xFFFF, buf[k] >> 16) for k in range(got)]


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
