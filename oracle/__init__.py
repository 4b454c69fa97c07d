"""Float64 CPU oracle for deterministic paged-KV attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
path (``deterministic_paged_kv_gb300``) never imports, loads or calls it, and
this package imports nothing from the product path.

The arithmetic lives in ``rk_oracle.c`` (plain C, float64, OpenMP over
queries).  This module compiles it with gcc on first use and marshals numpy
arrays through ctypes.

Sources followed (page title, section):
  * "WS2 PR7 Fused Attention Backend Alignment", "Current Implementation":
    materialise logical paged K/V before arithmetic; out [B, Hq, Sq, D],
    LSE [B, Hq, Sq].
  * same page, "FlashInfer RoPE Fusion": pre-RoPE Q/K, rotate-half RoPE,
    theta 1e6, scale 1.0, rotary_dim = head_dim.
  * "Add FlashInfer RoPE-fused paged attention scaffold", boundary table:
    GQA packing fixed from head layout, FP32 attention-domain LSE.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
closed forms, invariants, a complex-number statement of the rotation and
dense brute force on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rk_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F64 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile rk_oracle.c into liboracle.so (gcc, OpenMP).  Returns the path."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + ".tmp%d" % os.getpid()
            cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                   "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.rk_oracle_attention.restype = ctypes.c_int
        lib.rk_oracle_attention.argtypes = (
            [ctypes.c_int] * 8
            + [ctypes.c_void_p] * 3
            + [ctypes.c_int, i32p, i32p, i32p,
               ctypes.c_double, ctypes.c_double, ctypes.c_double,
               ctypes.c_void_p, f64p, f64p, ctypes.c_int])
        lib.rk_oracle_rope.restype = None
        lib.rk_oracle_rope.argtypes = [f64p, ctypes.c_int, ctypes.c_double,
                                       ctypes.c_double, ctypes.c_double, f64p]
        lib.rk_oracle_materialize_row.restype = ctypes.c_int
        lib.rk_oracle_materialize_row.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, i32p,
            ctypes.c_int, f64p]
        lib.rk_oracle_attention_backward.restype = ctypes.c_int
        lib.rk_oracle_attention_backward.argtypes = (
            [ctypes.c_int] * 8
            + [ctypes.c_void_p] * 3
            + [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, i32p, i32p, i32p,
               ctypes.c_double, ctypes.c_double, ctypes.c_double]
            + [ctypes.c_void_p] * 8 + [ctypes.c_int])
        lib.rk_oracle_max_threads.restype = ctypes.c_int
        lib.rk_oracle_max_threads.argtypes = []
        _lib = lib
    return _lib


def _as_np(x):
    """numpy view of a numpy array or a CPU torch tensor (bf16 -> raw bits)."""
    if isinstance(x, np.ndarray):
        return x
    try:  # torch tensor
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16)
            return x.numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x)


def _qkv(x):
    """Return (contiguous array, dtype code) for q / k_cache / v_cache."""
    a = _as_np(x)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), BF16
    return np.ascontiguousarray(a, dtype=np.float64), F64


def _i32(x):
    return np.ascontiguousarray(_as_np(x), dtype=np.int32)


def _ptr_i32(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))


def _ptr_f64(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def max_threads() -> int:
    return int(_load().rk_oracle_max_threads())


def rope(x, pos: float, theta: float = 1e6, rope_scale: float = 1.0) -> np.ndarray:
    """Rotate-half RoPE of one float64 vector at position ``pos``."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    assert x.ndim == 1 and x.shape[0] % 2 == 0
    y = np.empty_like(x)
    lib.rk_oracle_rope(_ptr_f64(x), x.shape[0], float(pos), float(theta),
                       float(rope_scale), _ptr_f64(y))
    return y


def materialize_row(cache, block_table, kv_lens, b: int) -> np.ndarray:
    """Logical cache of row ``b`` as float64 [Hkv, kv_len, D]."""
    lib = _load()
    c, code = _qkv(cache)
    NP, P, Hkv, D = c.shape
    bt = _i32(block_table)
    kl = _i32(kv_lens)
    n = int(kl[b])
    dst = np.zeros((Hkv, max(n, 0), D), dtype=np.float64)
    rc = lib.rk_oracle_materialize_row(c.ctypes.data, code, NP, P, Hkv, D,
                                       _ptr_i32(bt), bt.shape[1], _ptr_i32(kl),
                                       int(b), _ptr_f64(dst))
    if rc != 0:
        raise ValueError("oracle materialize_row failed with code %d" % rc)
    return dst


def attention(q, k_cache, v_cache, block_table, kv_lens, position_ids,
              rope_theta: float = 1e6, rope_scale: float = 1.0,
              sm_scale: float | None = None, row_mask=None,
              threads: int | None = None):
    """Float64 paged attention.  Returns ``(out [B,Hq,Sq,D], lse [B,Hq,Sq])``.

    ``q`` is [B, Hq, Sq, D]; caches are [num_pages, page_size, Hkv, D]; inputs
    may be float arrays (used as float64) or bfloat16 bit patterns (uint16 /
    torch.bfloat16).  ``row_mask`` ([B, Sq], optional) limits the work to the
    marked queries; unmarked entries of the result are NaN.
    """
    lib = _load()
    qa, qcode = _qkv(q)
    ka, kcode = _qkv(k_cache)
    va, vcode = _qkv(v_cache)
    if not (qcode == kcode == vcode):
        raise TypeError("q, k_cache and v_cache must share one element type")
    B, Hq, Sq, D = qa.shape
    NP, P, Hkv, D2 = ka.shape
    if D2 != D or va.shape != ka.shape:
        raise ValueError("shape mismatch")
    bt = _i32(block_table)
    kl = _i32(kv_lens)
    pos = _i32(position_ids)
    if bt.shape[0] != B or kl.shape != (B,) or pos.shape != (B, Sq):
        raise ValueError("metadata shape mismatch")
    W = bt.shape[1]
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    out = np.full((B, Hq, Sq, D), np.nan, dtype=np.float64)
    lse = np.full((B, Hq, Sq), np.nan, dtype=np.float64)
    mask_ptr = None
    if row_mask is not None:
        rm = np.ascontiguousarray(_as_np(row_mask), dtype=np.uint8)
        if rm.shape != (B, Sq):
            raise ValueError("row_mask must be [B, Sq]")
        mask_ptr = rm.ctypes.data
    rc = lib.rk_oracle_attention(B, Sq, Hq, Hkv, D, P, NP, W,
                                 qa.ctypes.data, ka.ctypes.data, va.ctypes.data,
                                 qcode, _ptr_i32(bt), _ptr_i32(kl), _ptr_i32(pos),
                                 float(rope_theta), float(rope_scale), float(sm_scale),
                                 mask_ptr, _ptr_f64(out), _ptr_f64(lse),
                                 int(threads or 0))
    if rc != 0:
        raise ValueError("oracle attention failed with code %d" % rc)
    return out, lse


def attention_backward(q, k_cache, v_cache, block_table, kv_lens, position_ids, dout,
                       rope_theta: float = 1e6, rope_scale: float = 1.0,
                       sm_scale: float | None = None, magnitudes: bool = False,
                       threads: int | None = None):
    """Float64 gradient of ``attention`` for L = sum(dout * out).

    Returns ``(dq [B,Hq,Sq,D], dk, dv)`` with dk / dv in the cache layout
    [num_pages, page_size, Hkv, D]: the pages a row references are written in
    full (0 at slots past kv_len), every other entry is NaN.  With
    ``magnitudes`` also returns ``(mag_dq, mag_dk, mag_dv, sens_dq, sens_dk)``:
    per element the sum of the absolute values of its terms, and of its terms'
    dependence on Dq = dout . out scaled by sum_d |dout_d out_d| (how far a
    relative change of out moves it).  ``dout`` is [B, Hq, Sq, D], float or
    bfloat16 bits; q / caches as in ``attention``.
    """
    lib = _load()
    qa, qcode = _qkv(q)
    ka, kcode = _qkv(k_cache)
    va, vcode = _qkv(v_cache)
    ga, gcode = _qkv(dout)
    if not (qcode == kcode == vcode):
        raise TypeError("q, k_cache and v_cache must share one element type")
    B, Hq, Sq, D = qa.shape
    NP, P, Hkv, D2 = ka.shape
    if D2 != D or va.shape != ka.shape or ga.shape != qa.shape:
        raise ValueError("shape mismatch")
    bt = _i32(block_table)
    kl = _i32(kv_lens)
    pos = _i32(position_ids)
    if bt.shape[0] != B or kl.shape != (B,) or pos.shape != (B, Sq):
        raise ValueError("metadata shape mismatch")
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(D)
    dq = np.full((B, Hq, Sq, D), np.nan, dtype=np.float64)
    dk = np.full((NP, P, Hkv, D), np.nan, dtype=np.float64)
    dv = np.full((NP, P, Hkv, D), np.nan, dtype=np.float64)
    mags = ([np.full_like(dq, np.nan), np.full_like(dk, np.nan), np.full_like(dv, np.nan),
             np.full_like(dq, np.nan), np.full_like(dk, np.nan)] if magnitudes else None)
    mp = [m.ctypes.data for m in mags] if mags else [None] * 5
    rc = lib.rk_oracle_attention_backward(B, Sq, Hq, Hkv, D, P, NP, bt.shape[1],
                                          qa.ctypes.data, ka.ctypes.data, va.ctypes.data, qcode,
                                          ga.ctypes.data, gcode, _ptr_i32(bt), _ptr_i32(kl), _ptr_i32(pos),
                                          float(rope_theta), float(rope_scale), float(sm_scale),
                                          dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
                                          mp[0], mp[1], mp[2], mp[3], mp[4], int(threads or 0))
    if rc != 0:
        raise ValueError("oracle attention_backward failed with code %d" % rc)
    if magnitudes:
        return dq, dk, dv, tuple(mags)
    return dq, dk, dv
