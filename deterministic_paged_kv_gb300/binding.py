"""ctypes binding of librk_paged.so (argument marshalling only).

Every step of the attention runs in the library's CUDA kernels; this module
only turns torch tensors into device pointers and the current CUDA stream
into a ``cudaStream_t``, and raises ``RkError`` on a non-zero status.  It
never computes a result itself and has no fallback: if the library is
missing, every call raises.

Names mirror the C ABI in ``include/rk_paged.h``:
``plan`` (rk_paged_plan), ``attn_decode`` (rk_paged_attn_decode),
``attn_prefill`` (rk_paged_attn_prefill), ``decode_split_scratch_bytes``
(rk_paged_decode_split_scratch_bytes), ``attn_decode_split``
(rk_paged_attn_decode_split), ``attn_decode_split_static``
(rk_paged_attn_decode_split_static), ``decode_balanced_scratch_bytes``
(rk_paged_decode_balanced_scratch_bytes), ``attn_decode_balanced``
(rk_paged_attn_decode_balanced), ``kv_append`` (rk_paged_kv_append),
``plan_ragged`` (rk_paged_plan_ragged), ``attn_ragged`` (rk_paged_attn_ragged),
``last_error``, ``policy``, ``abi_version``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "librk_paged.so")

RK_OK = 0
ERRORS = {
    1: "RK_E_ARG", 2: "RK_E_UNSUPPORTED", 3: "RK_E_PAGE_OOB", 4: "RK_E_DUP_PAGE",
    5: "RK_E_PAD", 6: "RK_E_KVLEN", 7: "RK_E_POSITION", 8: "RK_E_CUDA", 9: "RK_E_DEVICE",
}
CODES = {v: k for k, v in ERRORS.items()}
STATUS_PAGE_OOB, STATUS_KVLEN, STATUS_POSITION, STATUS_TIMEOUT, STATUS_RANGE = 1, 2, 4, 8, 16
ABI_VERSION = 3
SPLIT_STATIC_SCRATCH_BYTES = 16 << 20  # RK_PAGED_SPLIT_STATIC_SCRATCH_BYTES
BALANCED_SCRATCH_BYTES = 4096 + 512 * 3088 * 4  # RK_PAGED_BALANCED_SCRATCH_BYTES


class RkError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("%s (%d): %s" % (ERRORS.get(code, "?"), code, msg))
        self.code = code
        self.name = ERRORS.get(code, "?")
        self.msg = msg


class Plan(ctypes.Structure):
    """Mirror of rk_paged_plan_t."""
    _fields_ = [
        ("abi", ctypes.c_uint32),
        ("B", ctypes.c_int32), ("Sq", ctypes.c_int32), ("Hq", ctypes.c_int32),
        ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("W", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("causal", ctypes.c_int32), ("max_kv_len", ctypes.c_int32),
        ("sm_scale", ctypes.c_float), ("validated", ctypes.c_int32), ("pf_units", ctypes.c_int32),
        ("rope_theta", ctypes.c_double), ("rope_scale", ctypes.c_double),
        ("rope_turns", ctypes.c_uint64 * 64),
        ("wait_limit_ns", ctypes.c_uint32), ("timeout_drill", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load the library (once).  Raises if it is missing: there is no fallback."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("librk_paged.so not found at %s; build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % p)
        lib = ctypes.CDLL(p)
        vp, i32p = ctypes.c_void_p, ctypes.c_void_p
        lib.rk_paged_plan.restype = ctypes.c_int
        lib.rk_paged_plan.argtypes = [ctypes.POINTER(Plan)] + [ctypes.c_int32] * 8 + \
            [i32p, i32p, i32p, ctypes.c_double, ctypes.c_double]
        for name in ("rk_paged_attn_decode", "rk_paged_attn_prefill"):
            f = getattr(lib, name)
            f.restype = ctypes.c_int
            f.argtypes = [ctypes.POINTER(Plan)] + [vp] * 10
        lib.rk_paged_decode_split_scratch_bytes.restype = ctypes.c_int
        lib.rk_paged_decode_split_scratch_bytes.argtypes = [ctypes.POINTER(Plan), ctypes.c_int32,
                                                            ctypes.POINTER(ctypes.c_uint64)]
        lib.rk_paged_attn_decode_split.restype = ctypes.c_int
        lib.rk_paged_attn_decode_split.argtypes = [ctypes.POINTER(Plan), ctypes.c_int32] + [vp] * 9 + \
            [ctypes.c_uint64, vp, vp]
        lib.rk_paged_decode_balanced_scratch_bytes.restype = ctypes.c_int
        lib.rk_paged_decode_balanced_scratch_bytes.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(ctypes.c_uint64)]
        lib.rk_paged_attn_decode_balanced.restype = ctypes.c_int
        lib.rk_paged_attn_decode_balanced.argtypes = [ctypes.POINTER(Plan)] + [vp] * 9 + [ctypes.c_uint64, vp, vp]
        lib.rk_paged_attn_decode_split_static.restype = ctypes.c_int
        lib.rk_paged_attn_decode_split_static.argtypes = [ctypes.POINTER(Plan), ctypes.c_int32] + [vp] * 10
        lib.rk_paged_kv_append.restype = ctypes.c_int
        lib.rk_paged_kv_append.argtypes = [ctypes.POINTER(Plan), ctypes.c_int32] + [vp] * 8
        lib.rk_paged_plan_ragged.restype = ctypes.c_int
        lib.rk_paged_plan_ragged.argtypes = [ctypes.POINTER(Plan)] + [ctypes.c_int32] * 8 + \
            [i32p, i32p, i32p, i32p, ctypes.c_double, ctypes.c_double, ctypes.POINTER(ctypes.c_int32)]
        lib.rk_paged_attn_ragged.restype = ctypes.c_int
        lib.rk_paged_attn_ragged.argtypes = [ctypes.POINTER(Plan), ctypes.c_int32] + [vp] * 11
        lib.rk_paged_attn_prefill_backward.restype = ctypes.c_int
        lib.rk_paged_attn_prefill_backward.argtypes = [ctypes.POINTER(Plan)] + [vp] * 13 + \
            [ctypes.c_uint64, vp, vp]
        lib.rk_paged_prefill_backward_workspace_bytes.restype = ctypes.c_int
        lib.rk_paged_prefill_backward_workspace_bytes.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(ctypes.c_uint64)]
        lib.rk_last_error.restype = ctypes.c_char_p
        lib.rk_last_error.argtypes = []
        lib.rk_paged_policy.restype = ctypes.c_char_p
        lib.rk_paged_policy.argtypes = []
        lib.rk_paged_abi_version.restype = ctypes.c_uint32
        lib.rk_paged_abi_version.argtypes = []
        if lib.rk_paged_abi_version() != ABI_VERSION:
            raise RuntimeError("librk_paged.so ABI %d != binding ABI %d"
                               % (lib.rk_paged_abi_version(), ABI_VERSION))
        _lib = lib
        return lib


def last_error() -> str:
    return load().rk_last_error().decode()


def policy() -> str:
    return load().rk_paged_policy().decode()


def abi_version() -> int:
    return int(load().rk_paged_abi_version())


def _check(rc: int):
    if rc != RK_OK:
        raise RkError(rc, last_error())


def _host_i32(t):
    """(keep-alive object, pointer) of a host int32 array (torch or numpy)."""
    if t is None:
        return None, None
    import numpy as np
    try:
        import torch
        if isinstance(t, torch.Tensor):
            t = t.detach().to("cpu", torch.int32).contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(t, dtype=np.int32)
    return a, a.ctypes.data


def plan(B, Sq, Hq, Hkv, D, page_size, num_pages, W, block_table=None, kv_lens=None,
         position_ids=None, rope_theta=1e6, rope_scale=1.0) -> Plan:
    """rk_paged_plan on HOST metadata (or none, for a shape-only plan)."""
    lib = load()
    p = Plan()
    keep = [_host_i32(x) for x in (block_table, kv_lens, position_ids)]
    rc = lib.rk_paged_plan(ctypes.byref(p), int(B), int(Sq), int(Hq), int(Hkv), int(D),
                           int(page_size), int(num_pages), int(W),
                           keep[0][1], keep[1][1], keep[2][1], float(rope_theta), float(rope_scale))
    _check(rc)
    return p


def _dptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _expect(t, shape, name):
    """Raise ValueError unless tensor ``t`` has exactly ``shape``.  The C ABI
    receives bare pointers and cannot see sizes, so a tensor smaller than the
    plan says must be refused here, before anything is launched."""
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError("%s has shape %s, the plan needs %s" % (name, tuple(t.shape), tuple(shape)))


def _check_common(p: Plan, k_cache, v_cache, block_table, kv_lens, status):
    cache = (p.num_pages, p.page_size, p.Hkv, p.D)
    _expect(k_cache, cache, "k_cache")
    _expect(v_cache, cache, "v_cache")
    _expect(block_table, (p.B, p.W), "block_table")
    _expect(kv_lens, (p.B,), "kv_lens")
    if status is not None and status.numel() < 1:
        raise ValueError("status must hold at least one int32")


def _check_shapes(p: Plan, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, status,
                  ragged=False):
    """Every tensor of a decode / prefill / ragged call against the plan's sizes
    (ragged: q / out [total_q, Hq, D], lse [total_q, Hq], position_ids [total_q],
    with total_q = plan.Sq)."""
    _check_common(p, k_cache, v_cache, block_table, kv_lens, status)
    if ragged:
        qs, ls, ps = (p.Sq, p.Hq, p.D), (p.Sq, p.Hq), (p.Sq,)
    else:
        qs, ls, ps = (p.B, p.Hq, p.Sq, p.D), (p.B, p.Hq, p.Sq), (p.B, p.Sq)
    _expect(q, qs, "q")
    _expect(out, qs, "out")
    _expect(lse, ls, "lse")
    _expect(position_ids, ps, "position_ids")


def _launch(fn, p, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, status,
            stream, ragged=False):
    import torch
    for t, dt, name in ((q, torch.bfloat16, "q"), (k_cache, torch.bfloat16, "k_cache"),
                        (v_cache, torch.bfloat16, "v_cache"), (out, torch.bfloat16, "out"),
                        (lse, torch.float32, "lse"), (block_table, torch.int32, "block_table"),
                        (kv_lens, torch.int32, "kv_lens"), (position_ids, torch.int32, "position_ids")):
        if t.dtype != dt:
            raise TypeError("%s must be %s (got %s)" % (name, dt, t.dtype))
    if status is not None and status.dtype != torch.int32:
        raise TypeError("status must be int32")
    _check_shapes(p, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, status, ragged)
    rc = fn(ctypes.byref(p), _dptr(q), _dptr(k_cache), _dptr(v_cache), _dptr(block_table),
            _dptr(kv_lens), _dptr(position_ids), _dptr(out), _dptr(lse), _dptr(status),
            _stream(stream))
    _check(rc)


def attn_decode(p: Plan, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse,
                status=None, stream=None):
    """rk_paged_attn_decode on device tensors; asynchronous on ``stream``."""
    _launch(load().rk_paged_attn_decode, p, q, k_cache, v_cache, block_table, kv_lens,
            position_ids, out, lse, status, stream)


def attn_prefill(p: Plan, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse,
                 status=None, stream=None):
    """rk_paged_attn_prefill on device tensors; asynchronous on ``stream``."""
    _launch(load().rk_paged_attn_prefill, p, q, k_cache, v_cache, block_table, kv_lens,
            position_ids, out, lse, status, stream)


def prefill_backward_workspace_bytes(p: Plan) -> int:
    """rk_paged_prefill_backward_workspace_bytes: device workspace bytes of the backward."""
    n = ctypes.c_uint64(0)
    _check(load().rk_paged_prefill_backward_workspace_bytes(ctypes.byref(p), ctypes.byref(n)))
    return int(n.value)


def attn_prefill_backward(p: Plan, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, dout,
                          dq, dk_cache, dv_cache, workspace, status=None, stream=None):
    """rk_paged_attn_prefill_backward on device tensors: dq [B, Hq, Sq, D] and
    dk_cache / dv_cache [num_pages, 16, Hkv, D] float32; ``workspace`` a CUDA
    tensor of at least ``prefill_backward_workspace_bytes`` bytes (any dtype,
    256-byte aligned); asynchronous on ``stream``."""
    import torch
    for t, dt, name in ((q, torch.bfloat16, "q"), (k_cache, torch.bfloat16, "k_cache"),
                        (v_cache, torch.bfloat16, "v_cache"), (out, torch.bfloat16, "out"),
                        (lse, torch.float32, "lse"), (dout, torch.bfloat16, "dout"),
                        (dq, torch.float32, "dq"), (dk_cache, torch.float32, "dk_cache"),
                        (dv_cache, torch.float32, "dv_cache"),
                        (block_table, torch.int32, "block_table"), (kv_lens, torch.int32, "kv_lens"),
                        (position_ids, torch.int32, "position_ids")):
        if t.dtype != dt:
            raise TypeError("%s must be %s (got %s)" % (name, dt, t.dtype))
    if status is not None and status.dtype != torch.int32:
        raise TypeError("status must be int32")
    _check_shapes(p, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, status)
    _expect(dout, q.shape, "dout")
    _expect(dq, q.shape, "dq")
    _expect(dk_cache, k_cache.shape, "dk_cache")
    _expect(dv_cache, v_cache.shape, "dv_cache")
    nbytes = workspace.numel() * workspace.element_size()
    rc = load().rk_paged_attn_prefill_backward(
        ctypes.byref(p), _dptr(q), _dptr(k_cache), _dptr(v_cache), _dptr(block_table), _dptr(kv_lens),
        _dptr(position_ids), _dptr(out), _dptr(lse), _dptr(dout), _dptr(dq), _dptr(dk_cache), _dptr(dv_cache),
        _dptr(workspace), nbytes, _dptr(status), _stream(stream))
    _check(rc)


def decode_split_scratch_bytes(p: Plan, split_tokens: int) -> int:
    """rk_paged_decode_split_scratch_bytes: device scratch bytes of the split decode."""
    n = ctypes.c_uint64(0)
    _check(load().rk_paged_decode_split_scratch_bytes(ctypes.byref(p), int(split_tokens), ctypes.byref(n)))
    return int(n.value)


def attn_decode_split(p: Plan, split_tokens, q, k_cache, v_cache, block_table, kv_lens, position_ids,
                      out, lse, scratch, status=None, stream=None):
    """rk_paged_attn_decode_split on device tensors; ``scratch`` is a CUDA tensor
    of at least ``decode_split_scratch_bytes`` bytes (any dtype)."""
    import torch
    for t, dt, name in ((q, torch.bfloat16, "q"), (k_cache, torch.bfloat16, "k_cache"),
                        (v_cache, torch.bfloat16, "v_cache"), (out, torch.bfloat16, "out"),
                        (lse, torch.float32, "lse"), (block_table, torch.int32, "block_table"),
                        (kv_lens, torch.int32, "kv_lens"), (position_ids, torch.int32, "position_ids")):
        if t.dtype != dt:
            raise TypeError("%s must be %s (got %s)" % (name, dt, t.dtype))
    if status is not None and status.dtype != torch.int32:
        raise TypeError("status must be int32")
    _check_shapes(p, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, status)
    nbytes = scratch.numel() * scratch.element_size()
    rc = load().rk_paged_attn_decode_split(
        ctypes.byref(p), int(split_tokens), _dptr(q), _dptr(k_cache), _dptr(v_cache), _dptr(block_table),
        _dptr(kv_lens), _dptr(position_ids), _dptr(out), _dptr(lse), _dptr(scratch), nbytes, _dptr(status),
        _stream(stream))
    _check(rc)


def decode_balanced_scratch_bytes(p: Plan) -> int:
    """rk_paged_decode_balanced_scratch_bytes: device scratch bytes of the balanced decode."""
    n = ctypes.c_uint64(0)
    _check(load().rk_paged_decode_balanced_scratch_bytes(ctypes.byref(p), ctypes.byref(n)))
    return int(n.value)


def attn_decode_balanced(p: Plan, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, scratch,
                         status=None, stream=None):
    """rk_paged_attn_decode_balanced on device tensors: the split-free decode on a
    balanced schedule (results bitwise equal to ``attn_decode``).  ``scratch`` is
    a CUDA tensor of at least ``decode_balanced_scratch_bytes`` bytes (any dtype,
    256-byte aligned), zeroed once before its first use and then reused by one
    call at a time."""
    import torch
    for t, dt, name in ((q, torch.bfloat16, "q"), (k_cache, torch.bfloat16, "k_cache"),
                        (v_cache, torch.bfloat16, "v_cache"), (out, torch.bfloat16, "out"),
                        (lse, torch.float32, "lse"), (block_table, torch.int32, "block_table"),
                        (kv_lens, torch.int32, "kv_lens"), (position_ids, torch.int32, "position_ids")):
        if t.dtype != dt:
            raise TypeError("%s must be %s (got %s)" % (name, dt, t.dtype))
    if status is not None and status.dtype != torch.int32:
        raise TypeError("status must be int32")
    _check_shapes(p, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, status)
    nbytes = scratch.numel() * scratch.element_size()
    rc = load().rk_paged_attn_decode_balanced(
        ctypes.byref(p), _dptr(q), _dptr(k_cache), _dptr(v_cache), _dptr(block_table), _dptr(kv_lens),
        _dptr(position_ids), _dptr(out), _dptr(lse), _dptr(scratch), nbytes, _dptr(status), _stream(stream))
    _check(rc)


def attn_decode_split_static(p: Plan, split_tokens, q, k_cache, v_cache, block_table, kv_lens,
                             position_ids, out, lse, status=None, stream=None):
    """rk_paged_attn_decode_split_static: the split decode with the library's own
    static device scratch (no allocation; calls overlapping in time race)."""
    _launch(lambda pp, *r: load().rk_paged_attn_decode_split_static(pp, int(split_tokens), *r), p, q,
            k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, status, stream)


def kv_append(p: Plan, n_new, k_new, v_new, block_table, kv_lens, k_cache, v_cache, status=None,
              stream=None):
    """rk_paged_kv_append: write k_new / v_new (bf16 [B, n_new, Hkv, D]) into the
    pages of positions kv_len - n_new .. kv_len - 1 (kv_lens after the append)."""
    import torch
    for t, dt, name in ((k_new, torch.bfloat16, "k_new"), (v_new, torch.bfloat16, "v_new"),
                        (k_cache, torch.bfloat16, "k_cache"), (v_cache, torch.bfloat16, "v_cache"),
                        (block_table, torch.int32, "block_table"), (kv_lens, torch.int32, "kv_lens")):
        if t.dtype != dt:
            raise TypeError("%s must be %s (got %s)" % (name, dt, t.dtype))
    if status is not None and status.dtype != torch.int32:
        raise TypeError("status must be int32")
    _check_common(p, k_cache, v_cache, block_table, kv_lens, status)
    if int(n_new) > 0:  # n_new <= 0 is judged by the library (0: nothing to do, < 0: RK_E_ARG)
        _expect(k_new, (p.B, int(n_new), p.Hkv, p.D), "k_new")
        _expect(v_new, (p.B, int(n_new), p.Hkv, p.D), "v_new")
    rc = load().rk_paged_kv_append(ctypes.byref(p), int(n_new), _dptr(k_new), _dptr(v_new), _dptr(block_table),
                                   _dptr(kv_lens), _dptr(k_cache), _dptr(v_cache), _dptr(status),
                                   _stream(stream))
    _check(rc)


def plan_ragged(B, total_q, Hq, Hkv, D, page_size, num_pages, W, qo_indptr, block_table=None, kv_lens=None,
                position_ids=None, rope_theta=1e6, rope_scale=1.0):
    """rk_paged_plan_ragged on HOST metadata; returns (plan, max_q_len)."""
    lib = load()
    p = Plan()
    mq = ctypes.c_int32(0)
    keep = [_host_i32(x) for x in (qo_indptr, block_table, kv_lens, position_ids)]
    rc = lib.rk_paged_plan_ragged(ctypes.byref(p), int(B), int(total_q), int(Hq), int(Hkv), int(D),
                                  int(page_size), int(num_pages), int(W), keep[0][1], keep[1][1], keep[2][1],
                                  keep[3][1], float(rope_theta), float(rope_scale), ctypes.byref(mq))
    _check(rc)
    return p, int(mq.value)


def attn_ragged(p: Plan, max_q_len, qo_indptr, q, k_cache, v_cache, block_table, kv_lens, position_ids, out,
                lse, status=None, stream=None):
    """rk_paged_attn_ragged on device tensors: q / out [total_q, Hq, D],
    lse [total_q, Hq], position_ids [total_q], qo_indptr [B + 1]."""
    import torch
    if qo_indptr.dtype != torch.int32:
        raise TypeError("qo_indptr must be int32")
    _expect(qo_indptr, (p.B + 1,), "qo_indptr")
    _launch(lambda pp, *r: load().rk_paged_attn_ragged(pp, int(max_q_len), _dptr(qo_indptr), *r), p, q,
            k_cache, v_cache, block_table, kv_lens, position_ids, out, lse, status, stream, ragged=True)


def run(mode: str, q, k_cache, v_cache, block_table, kv_lens, position_ids, plan_obj=None,
        rope_theta=1e6, rope_scale=1.0, status=None, stream=None, split_tokens=0):
    """Allocate out / lse (and the split scratch) with torch and launch decode,
    split decode (``mode="decode"`` with ``split_tokens`` > 0) or prefill.

    ``plan_obj`` defaults to a shape-only plan; pass one built from host
    metadata to have the contents validated first.
    """
    import torch
    B, Hq, Sq, D = q.shape
    NP, P, Hkv, _ = k_cache.shape
    if plan_obj is None:
        plan_obj = plan(B, Sq, Hq, Hkv, D, P, NP, block_table.shape[1],
                        rope_theta=rope_theta, rope_scale=rope_scale)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if mode == "decode" and split_tokens:
        scratch = torch.empty(decode_split_scratch_bytes(plan_obj, split_tokens), dtype=torch.uint8,
                              device=q.device)
        attn_decode_split(plan_obj, split_tokens, q, k_cache, v_cache, block_table, kv_lens, position_ids,
                          out, lse, scratch, status=status, stream=stream)
        return out, lse
    fn = attn_decode if mode == "decode" else attn_prefill
    fn(plan_obj, q, k_cache, v_cache, block_table, kv_lens, position_ids, out, lse,
       status=status, stream=stream)
    return out, lse
