"""ctypes front end of the fp64 CPU oracle (``attn_ref.cpp``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use this package; the CUDA path never imports it and it
never imports the CUDA path.  See ``attn_ref.cpp`` for what each function
computes and which passage of the FlashAttention-3 pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with the host C++ compiler (portable C++17)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
               "-ffp-contract=off", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i, d, u64, lng = ctypes.c_int, ctypes.c_double, ctypes.c_ulonglong, ctypes.c_long
            L.oracle_attn_fwd_bf16.argtypes = [P, P, P, P, P, i, i, i, i, i, i, d, i, P, i, i]
            L.oracle_attn_fwd_bf16.restype = i
            L.oracle_attn_fwd_f64.argtypes = [P, P, P, P, P, i, i, i, i, i, i, d, i, P, i, i]
            L.oracle_attn_fwd_f64.restype = i
            L.oracle_attn_fwd_bf16_masked.argtypes = [P, P, P, P, P, i, i, i, i, i, i, d, i, P, P, i, i]
            L.oracle_attn_fwd_bf16_masked.restype = i
            L.oracle_attn_fwd_f64_masked.argtypes = [P, P, P, P, P, i, i, i, i, i, i, d, i, P, P, i, i]
            L.oracle_attn_fwd_f64_masked.restype = i
            L.oracle_attn_bwd_bf16.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, i, d, i, i]
            L.oracle_attn_bwd_bf16.restype = i
            L.oracle_attn_bwd_f64.argtypes = [P, P, P, P, P, P, P, i, i, i, i, i, i, d, i, i]
            L.oracle_attn_bwd_f64.restype = i
            L.oracle_attn_row_probs_f64.argtypes = [P, P, P, i, i, i, i, i, d, i, i, i, i, P]
            L.oracle_attn_row_probs_f64.restype = i
            L.oracle_e4m3_encode_f64.argtypes = [P, P, lng]
            L.oracle_e4m3_encode_f64.restype = None
            L.oracle_e4m3_decode.argtypes = [P, P, lng]
            L.oracle_e4m3_decode.restype = None
            L.oracle_rotation_matrix.argtypes = [i, u64, P]
            L.oracle_rotation_matrix.restype = i
            L.oracle_signs.argtypes = [i, u64, P]
            L.oracle_signs.restype = None
            L.oracle_fp8_quantize.argtypes = [P, P, P, P, i, i, i, i, i, i, u64, i, i]
            L.oracle_fp8_quantize.restype = i
            L.oracle_fp8_quantize_rope.argtypes = [P, P, P, P, P, P, i, i, i, i, i, i, i, u64, i, i]
            L.oracle_fp8_quantize_rope.restype = i
            L.oracle_rope_bf16.argtypes = [P, P, P, P, i, i, i, i, i, i]
            L.oracle_rope_bf16.restype = i
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows_arg(rows, N):
    if rows is None:
        return None, N, None
    r = np.ascontiguousarray(rows, dtype=np.int32)
    return r, len(r), _ptr(r)


def attention(q, k, v, causal=False, scale=None, window=0, rows=None, nthreads=0, block_mask=None):
    """Attention forward in fp64.

    block_mask: optional uint8 (B, H, T, T), T = ceil(N / 128): query block i
    sees key block j of (b, h) iff block_mask[b, h, i, j] != 0 (ANDed with the
    causal and window masks).

    q: (B, N, H, d); k, v: (B, N, Hkv, d) with Hkv dividing H (grouped-query
    attention: query head h reads key/value head h // (H // Hkv)).  Arrays are
    either uint16 bf16 bit patterns or float64.  Returns (o, lse) with o of
    shape (B, H, R, d) and lse (B, H, R), where R indexes ``rows`` (all N rows
    when None).
    """
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rr, R, rp = _rows_arg(rows, N)
    o = np.empty((B, H, R, d), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    bf16 = q.dtype == np.uint16
    if bf16:
        q, k, v = (np.ascontiguousarray(t, dtype=np.uint16) for t in (q, k, v))
    else:
        q, k, v = (np.ascontiguousarray(t, dtype=np.float64) for t in (q, k, v))
    if block_mask is None:
        fn = lib().oracle_attn_fwd_bf16 if bf16 else lib().oracle_attn_fwd_f64
        rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d, int(bool(causal)),
                float(scale), int(window), rp, R, int(nthreads))
    else:
        T = (N + 127) // 128
        m = np.ascontiguousarray(block_mask, dtype=np.uint8)
        if m.shape != (B, H, T, T):
            raise ValueError(f"block_mask must be (B, H, {T}, {T})")
        fn = lib().oracle_attn_fwd_bf16_masked if bf16 else lib().oracle_attn_fwd_f64_masked
        rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d, int(bool(causal)),
                float(scale), int(window), _ptr(m), rp, R, int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_fwd: bad arguments")
    return o, lse


def attention_bwd(q, k, v, dout, causal=False, scale=None, window=0, nthreads=0):
    """Gradients of the attention forward in fp64 for the upstream gradient
    dout = dL/dO.

    q, dout: (B, N, H, d); k, v: (B, N, Hkv, d) (Hkv divides H), either all
    uint16 bf16 bit patterns or all float64.  Returns (dq, dk, dv) in the
    shapes of q, k, v (float64).
    """
    B, N, H, d = q.shape
    Hkv = k.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    if q.dtype == np.uint16:
        fn = lib().oracle_attn_bwd_bf16
        q, k, v, dout = (np.ascontiguousarray(t, dtype=np.uint16) for t in (q, k, v, dout))
    else:
        fn = lib().oracle_attn_bwd_f64
        q, k, v, dout = (np.ascontiguousarray(t, dtype=np.float64) for t in (q, k, v, dout))
    dq = np.empty(q.shape, dtype=np.float64)
    dk = np.empty(k.shape, dtype=np.float64)
    dv = np.empty(v.shape, dtype=np.float64)
    rc = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), B, H, Hkv, N, d,
            int(bool(causal)), float(scale), int(window), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_attn_bwd: bad arguments")
    return dq, dk, dv


def row_probs(q, k, v, b, h, i, causal=False, scale=None, window=0):
    """Softmax weights (length N) of query row i of (b, h); float64 inputs."""
    B, N, H, d = q.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    q, k, v = (np.ascontiguousarray(t, dtype=np.float64) for t in (q, k, v))
    p = np.empty(N, dtype=np.float64)
    rc = lib().oracle_attn_row_probs_f64(_ptr(q), _ptr(k), _ptr(v), B, H, N, d, int(bool(causal)),
                                         float(scale), int(window), b, h, i, _ptr(p))
    if rc != 0:
        raise ValueError("oracle_attn_row_probs: bad arguments")
    return p


def e4m3_encode(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64).ravel()
    out = np.empty(x.size, dtype=np.uint8)
    lib().oracle_e4m3_encode_f64(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8).ravel()
    out = np.empty(c.size, dtype=np.float64)
    lib().oracle_e4m3_decode(_ptr(c), _ptr(out), c.size)
    return out


def rotation_matrix(d: int, seed: int) -> np.ndarray:
    M = np.empty((d, d), dtype=np.float64)
    if lib().oracle_rotation_matrix(d, seed, _ptr(M)) != 0:
        raise ValueError("head_dim must be a power of two")
    return M


def signs(d: int, seed: int) -> np.ndarray:
    s = np.empty(d, dtype=np.float64)
    lib().oracle_signs(d, seed, _ptr(s))
    return s


MODE_BLOCK, MODE_BLOCK_HADAMARD, MODE_PER_TENSOR = 0, 1, 2


def _rope_tables(rope, N, d):
    cos_t, sin_t, interleaved = rope
    cos_t = np.ascontiguousarray(cos_t, dtype=np.float32)
    sin_t = np.ascontiguousarray(sin_t, dtype=np.float32)
    if cos_t.shape != (N, d // 2) or sin_t.shape != (N, d // 2):
        raise ValueError("RoPE tables must be (N, d/2)")
    return cos_t, sin_t, int(bool(interleaved))


def rope(x, cos_t, sin_t, interleaved=False, nthreads=0):
    """RoPE of a (B, N, H, d) bf16 tensor (uint16 bits) with binary32 tables
    (N, d/2); returns float32 (B, N, H, d)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    B, N, H, d = x.shape
    c, s, il = _rope_tables((cos_t, sin_t, interleaved), N, d)
    out = np.empty(x.shape, dtype=np.float32)
    if lib().oracle_rope_bf16(_ptr(x), _ptr(out), _ptr(c), _ptr(s), B, N, H, d, il, int(nthreads)) != 0:
        raise ValueError("oracle_rope: bad arguments")
    return out


def fp8_quantize(x, mode, seed=0, is_v=False, block_rows=128, return_rotated=False, nthreads=0, rope=None):
    """FP8 prep of one (B, N, H, d) bf16 tensor (uint16 bits).

    rope: optional (cos, sin, interleaved) with binary32 tables (N, d/2);
    RoPE is then applied before the rotation and the quantiser (Q, K only).
    Returns (codes uint8 (B,N,H,d), scales float32 (B,H,nblk)[, rotated f32]).
    """
    x = np.ascontiguousarray(x, dtype=np.uint16)
    B, N, H, d = x.shape
    rc_, rs_, ril = (None, None, 0)
    if rope is not None:
        rc_, rs_, ril = _rope_tables(rope, N, d)
    nblk = (N + block_rows - 1) // block_rows
    codes = np.empty(x.shape, dtype=np.uint8)
    scales = np.empty((B, H, nblk), dtype=np.float32)
    rot = np.empty(x.shape, dtype=np.float32) if return_rotated else None
    rc = lib().oracle_fp8_quantize_rope(_ptr(x), _ptr(codes), _ptr(scales),
                                        _ptr(rot) if rot is not None else None,
                                        _ptr(rc_) if rc_ is not None else None,
                                        _ptr(rs_) if rs_ is not None else None, ril,
                                        B, H, N, d, block_rows, mode, seed, int(bool(is_v)), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_fp8_quantize: bad arguments")
    if return_rotated:
        return codes, scales, rot
    return codes, scales
