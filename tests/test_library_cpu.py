"""Host-side tests of the C ABI (no GPU needed): the library loads, exports
every declared symbol, validates metadata with the documented error codes,
reports the pages' fixed policy and derives its RoPE constants correctly."""
import json
import math
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rk_paged.h")


@pytest.fixture(scope="module")
def rk():
    from deterministic_paged_kv_gb300 import build, binding
    build.build()
    binding.load()
    return binding


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rk_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["rk_paged_plan", "rk_paged_attn_decode", "rk_paged_attn_prefill",
              "rk_last_error", "rk_paged_policy", "rk_paged_abi_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(rk):
    out = subprocess.run(["nm", "-D", "--defined-only", rk.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (rk_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    lib = rk.load()
    for n in declared_functions():
        assert hasattr(lib, n)


def test_abi_and_policy_match_the_pages(rk):
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_contract.json")))
    assert rk.abi_version() == rk.ABI_VERSION
    pol = dict(kv.split("=", 1) for kv in rk.policy().split(";"))
    assert pol["split_kv"] == g["split_kv"]["value"]["policy"]
    assert pol["acc"] == g["arithmetic"]["value"]["accumulation"]
    assert pol["lse"].startswith(g["arithmetic"]["value"]["lse"])
    assert pol["downcast"].startswith("final_write")
    assert pol["order"] != g["unsupported_requests"]["value"]["reduction_order"]
    assert int(pol["page_size"]) == g["cache"]["value"]["page_size"]
    assert int(pol["head_dim"]) == g["cache"]["value"]["head_dim"]
    assert "rotate_half" in pol["rope"]


def _ok_case(B=2, Sq=1, W=4, NP=10):
    bt = np.full((B, W), -1, np.int32)
    bt[0, :2] = [3, 7]
    bt[1, :3] = [0, 1, 9]
    kv = np.array([20, 40], np.int32)
    pos = np.array([[20], [40]], np.int32) if Sq == 1 else None
    return bt, kv, pos


def _plan(rk, B, Sq, Hq, Hkv, D, P, NP, W, bt, kv, pos, theta=1e6, scale=1.0):
    return rk.plan(B, Sq, Hq, Hkv, D, P, NP, W, bt, kv, pos, theta, scale)


def test_plan_accepts_valid_decode_and_fills_fields(rk):
    bt, kv, pos = _ok_case()
    p = _plan(rk, 2, 1, 32, 8, 128, 16, 10, 4, bt, kv, pos)
    assert p.abi == rk.ABI_VERSION and p.B == 2 and p.Sq == 1 and p.W == 4 and p.num_pages == 10
    assert p.causal == 1 and p.max_kv_len == 40 and p.validated == 1
    assert p.sm_scale == pytest.approx(1 / math.sqrt(128))
    # also the kv_len-1 convention and a shape-only plan
    _plan(rk, 2, 1, 32, 8, 128, 16, 10, 4, bt, kv, pos - 1)
    q = rk.plan(2, 1, 32, 8, 128, 16, 10, 4)
    assert q.validated == 0


def test_plan_rope_turns_match_oracle_frequencies(rk):
    """The plan's fixed-point rates are the oracle's angular speeds / 2 pi."""
    import oracle
    p = rk.plan(1, 1, 32, 8, 128, 16, 1, 1, rope_theta=1e6, rope_scale=1.0)
    for i in [0, 1, 7, 31, 63]:
        e = np.zeros(128)
        e[i] = 1.0
        y = oracle.rope(e, 1.0)
        speed = math.atan2(y[i + 64], y[i])
        assert p.rope_turns[i] / 2.0 ** 64 * 2 * math.pi == pytest.approx(speed, rel=1e-12)
    p2 = rk.plan(1, 1, 32, 8, 128, 16, 1, 1, rope_theta=1e6, rope_scale=4.0)
    assert p2.rope_turns[5] == pytest.approx(p.rope_turns[5] / 4, rel=1e-12)


@pytest.mark.parametrize("case,code", [
    ("D", "RK_E_UNSUPPORTED"), ("page", "RK_E_UNSUPPORTED"), ("gqa3", "RK_E_UNSUPPORTED"),
    ("gqa16", "RK_E_UNSUPPORTED"), ("kvneg", "RK_E_KVLEN"), ("kvbig", "RK_E_KVLEN"),
    ("oob", "RK_E_PAGE_OOB"), ("neg_page", "RK_E_PAGE_OOB"), ("pad", "RK_E_PAD"),
    ("dup", "RK_E_DUP_PAGE"), ("dup_cross_row", "RK_E_DUP_PAGE"), ("pos_neg", "RK_E_POSITION"),
    ("pos_gap", "RK_E_POSITION"), ("pos_not_trailing", "RK_E_POSITION"),
    ("empty_prefill", "RK_E_POSITION"), ("theta", "RK_E_ARG"), ("scale", "RK_E_ARG"),
    ("Sq0", "RK_E_ARG"), ("partial_meta", "RK_E_ARG"),
])
def test_plan_rejections(rk, case, code):
    B, Sq, Hq, Hkv, D, P, NP, W = 2, 1, 32, 8, 128, 16, 10, 4
    bt, kv, pos = _ok_case()
    theta, scale = 1e6, 1.0
    if case == "D":
        D = 64
    elif case == "page":
        P = 32
    elif case == "gqa3":
        Hq, Hkv = 24, 8
    elif case == "gqa16":
        Hq, Hkv = 32, 2
    elif case == "kvneg":
        kv[0] = -1
    elif case == "kvbig":
        kv[1] = W * 16 + 1
    elif case == "oob":
        bt[1, 2] = NP
    elif case == "neg_page":
        bt[0, 1] = -1
    elif case == "pad":
        bt[0, 3] = 5
    elif case == "dup":
        bt[1, 1] = 0
    elif case == "dup_cross_row":
        bt[1, 0] = 7
    elif case == "pos_neg":
        pos = np.array([[-1], [40]], np.int32)
    elif case == "pos_gap":
        Sq = 3
        pos = np.array([[18, 19, 21], [38, 39, 40]], np.int32)
    elif case == "pos_not_trailing":
        pos = np.array([[18], [40]], np.int32)
    elif case == "empty_prefill":
        Sq = 2
        kv[0] = 0
        bt[0, :] = -1
        pos = np.array([[0, 1], [39, 40]], np.int32)
    elif case == "theta":
        theta = 1.0
    elif case == "scale":
        scale = 0.0
    elif case == "Sq0":
        Sq = 0
        pos = np.zeros((2, 1), np.int32)
    elif case == "partial_meta":
        pos = None
    with pytest.raises(rk.RkError) as ei:
        _plan(rk, B, Sq, Hq, Hkv, D, P, NP, W, bt, kv, pos, theta, scale)
    assert ei.value.name == code, ei.value
    assert rk.last_error()  # a message is set


def test_plan_allows_empty_decode_rows(rk):
    bt = np.full((2, 4), -1, np.int32)
    bt[1, :1] = [2]
    kv = np.array([0, 5], np.int32)
    pos = np.array([[0], [5]], np.int32)
    p = _plan(rk, 2, 1, 32, 8, 128, 16, 4, 4, bt, kv, pos)
    assert p.max_kv_len == 5


def test_launch_without_gpu_fails_closed(rk):
    """With no device, a launch returns an error instead of computing anything."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    p = rk.plan(1, 1, 32, 8, 128, 16, 1, 1)
    lib = rk.load()
    buf = (ctypes_buf := np.zeros(1 << 16, np.uint8)).ctypes.data  # noqa: F841
    al = (buf + 255) & ~255
    import ctypes
    rc = lib.rk_paged_attn_decode(ctypes.byref(p), al, al, al, al, al, al, al, al, None, None)
    assert rc in (rk.CODES["RK_E_CUDA"], rk.CODES["RK_E_DEVICE"])


def test_split_decode_scratch_bytes_host_only(rk):
    """rk_paged_decode_split_scratch_bytes: B * Hq * ceil(W * 16 / split) *
    (D + 1) * 4 bytes; split lengths that are not positive multiples of the
    page size (16) are rejected.  Host only."""
    p = rk.plan(3, 1, 32, 8, 128, 16, 600, 200)
    for split in (16, 528, 1024, 2048, 3072):
        n_splits = -(-200 * 16 // split)
        assert rk.decode_split_scratch_bytes(p, split) == 3 * 32 * n_splits * 129 * 4
    p0 = rk.plan(2, 1, 32, 8, 128, 16, 0, 0)
    assert rk.decode_split_scratch_bytes(p0, 1024) == 2 * 32 * 1 * 129 * 4
    for bad in (0, -1024, 8, 1500, 1001):
        with pytest.raises(rk.RkError) as e:
            rk.decode_split_scratch_bytes(p, bad)
        assert e.value.name == "RK_E_ARG"


def test_ragged_plan_validation_host_only(rk):
    """rk_paged_plan_ragged: qo_indptr must start at 0, not decrease and end at
    total_q; per-row positions follow the padded rules; max_q_len returned."""
    from deterministic_paged_kv_gb300 import workloads
    w = workloads.ragged_case([1, 0, 5, 3], [40, 10, 60, 20], seed=3)
    q, ind, pos = workloads.pack_ragged(w)
    T = q.shape[0]
    p, mq = rk.plan_ragged(w.B, T, 32, 8, 128, 16, w.num_pages, w.W, ind, w.block_table, w.kv_lens, pos)
    assert mq == 5 and p.Sq == T and p.validated == 1
    assert p.pf_units == 2  # rows of 5 and 3 queries: one pair of 32-query q-tiles each
    assert rk.plan(2, 1, 32, 8, 128, 16, 10, 4).pf_units == -1  # padded plan: no count
    for bad_ind in ([1, 1, 1, 6, 9], [0, 1, 0, 6, 9], [0, 1, 1, 6, 8]):
        with pytest.raises(rk.RkError) as e:
            rk.plan_ragged(w.B, T, 32, 8, 128, 16, w.num_pages, w.W, bad_ind, w.block_table, w.kv_lens, pos)
        assert e.value.name == "RK_E_ARG"
    bad_pos = pos.clone()
    bad_pos[1 + 2] += 1  # row 2 no longer contiguous
    with pytest.raises(rk.RkError) as e:
        rk.plan_ragged(w.B, T, 32, 8, 128, 16, w.num_pages, w.W, ind, w.block_table, w.kv_lens, bad_pos)
    assert e.value.name == "RK_E_POSITION"


@pytest.mark.parametrize("Hq,Hkv,expect", [(32, 8, 7), (32, 32, 4), (32, 4, 11)])
def test_ragged_plan_counts_prefill_work_units(rk, Hq, Hkv, expect):
    """pf_units = sum over rows of two or more queries of ceil(q / (2 x 128 / G)):
    q-tiles hold 128 / G query positions and a work unit is a pair of them."""
    from deterministic_paged_kv_gb300 import workloads
    q_lens = [1, 130, 64, 65, 2, 0]
    w = workloads.ragged_case(q_lens, [40, 200, 64, 100, 2, 7], seed=4, Hq=Hq, Hkv=Hkv)
    q, ind, pos = workloads.pack_ragged(w)
    p, mq = rk.plan_ragged(w.B, q.shape[0], Hq, Hkv, 128, 16, w.num_pages, w.W, ind, w.block_table,
                           w.kv_lens, pos)
    span = 2 * 128 // (Hq // Hkv)
    assert mq == 130 and p.pf_units == expect == sum(-(-n // span) for n in q_lens if n >= 2)
    # the count depends on qo_indptr alone: a shape-only ragged plan agrees
    p2, _ = rk.plan_ragged(w.B, q.shape[0], Hq, Hkv, 128, 16, w.num_pages, w.W, ind)
    assert p2.pf_units == expect and p2.validated == 0


def test_backward_workspace_size_host_only(rk):
    """rotated q (FP16) + rotated K and V in token order (2 x 2 B Hkv W 16 D) + delta (FP32),
    each part rounded up to 256 bytes."""
    p = rk.plan(2, 40, 32, 8, 128, 16, 10, 4)
    r = lambda x: (x + 255) // 256 * 256
    want = r(2 * 32 * 40 * 128 * 2) + 2 * r(2 * 8 * 4 * 16 * 128 * 2) + r(2 * 32 * 40 * 4)
    assert rk.prefill_backward_workspace_bytes(p) == want


def _tensors(B=2, Sq=3, Hq=32, Hkv=8, NP=6, W=3, ragged=False):
    import torch
    bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
    if ragged:
        q = torch.zeros((Sq, Hq, 128), dtype=bf)
        lse = torch.zeros((Sq, Hq), dtype=f32)
        pos = torch.zeros((Sq,), dtype=i32)
    else:
        q = torch.zeros((B, Hq, Sq, 128), dtype=bf)
        lse = torch.zeros((B, Hq, Sq), dtype=f32)
        pos = torch.zeros((B, Sq), dtype=i32)
    cache = torch.zeros((NP, 16, Hkv, 128), dtype=bf)
    return dict(q=q, k_cache=cache, v_cache=cache.clone(), block_table=torch.zeros((B, W), dtype=i32),
                kv_lens=torch.zeros((B,), dtype=i32), position_ids=pos, out=q.clone(), lse=lse)


_ORDER = ("q", "k_cache", "v_cache", "block_table", "kv_lens", "position_ids", "out", "lse")


@pytest.mark.parametrize("name,bad_prefill,bad_decode", [
    ("q", (2, 32, 2, 128), (2, 32, 1, 64)), ("out", (2, 32, 3, 64), (1, 32, 1, 128)),
    ("lse", (2, 32, 2), (2, 16, 1)), ("k_cache", (5, 16, 8, 128), (6, 16, 8, 64)),
    ("v_cache", (6, 16, 4, 128), (6, 8, 8, 128)), ("block_table", (2, 2), (2, 4)),
    ("kv_lens", (1,), (3,)), ("position_ids", (2, 2), (2, 2))])
def test_binding_refuses_tensors_smaller_than_the_plan(rk, name, bad_prefill, bad_decode):
    """The C ABI sees only pointers: the binding compares every tensor with the
    plan and raises before any call into the library (here on CPU tensors, so
    a call that got through would fail on the CUDA check instead)."""
    import torch
    p = rk.plan(2, 3, 32, 8, 128, 16, 6, 3)
    t = _tensors()
    with pytest.raises(ValueError, match="expected a CUDA tensor"):  # shapes right: stops at the device check
        rk.attn_prefill(p, *[t[k] for k in _ORDER])
    t[name] = torch.zeros(bad_prefill, dtype=t[name].dtype)
    with pytest.raises(ValueError, match="the plan needs"):
        rk.attn_prefill(p, *[t[k] for k in _ORDER])
    pd = rk.plan(2, 1, 32, 8, 128, 16, 6, 3)
    td = _tensors(Sq=1)
    td[name] = torch.zeros(bad_decode, dtype=td[name].dtype)
    args = [td[k] for k in _ORDER]
    with pytest.raises(ValueError, match="the plan needs"):
        rk.attn_decode(pd, *args)
    with pytest.raises(ValueError, match="the plan needs"):
        rk.attn_decode_split(pd, 1024, *args, torch.zeros(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError, match="the plan needs"):
        rk.attn_decode_split_static(pd, 1024, *args)


def test_binding_refuses_wrong_ragged_append_and_backward_shapes(rk):
    import torch
    p, mq = rk.plan_ragged(2, 5, 32, 8, 128, 16, 6, 3, [0, 2, 5])
    t = _tensors(Sq=5, ragged=True)
    ind = torch.tensor([0, 2, 5], dtype=torch.int32)
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        rk.attn_ragged(p, mq, ind, *[t[k] for k in _ORDER])
    with pytest.raises(ValueError, match="the plan needs"):
        rk.attn_ragged(p, mq, ind[:2], *[t[k] for k in _ORDER])
    t["position_ids"] = torch.zeros((4,), dtype=torch.int32)
    with pytest.raises(ValueError, match="the plan needs"):
        rk.attn_ragged(p, mq, ind, *[t[k] for k in _ORDER])
    # kv_append: new tokens [B, n_new, Hkv, D]
    pa = rk.plan(2, 1, 32, 8, 128, 16, 6, 3)
    ta = _tensors(Sq=1)
    kn = torch.zeros((2, 4, 8, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        rk.kv_append(pa, 4, kn, kn, ta["block_table"], ta["kv_lens"], ta["k_cache"], ta["v_cache"])
    with pytest.raises(ValueError, match="the plan needs"):
        rk.kv_append(pa, 5, kn, kn, ta["block_table"], ta["kv_lens"], ta["k_cache"], ta["v_cache"])
    with pytest.raises(ValueError, match="the plan needs"):
        rk.kv_append(pa, 4, kn, kn, ta["block_table"], ta["kv_lens"], ta["k_cache"][:5], ta["v_cache"])
    # backward: dout / dq like q, dk / dv like the caches
    pb = rk.plan(2, 3, 32, 8, 128, 16, 6, 3)
    tb = _tensors()
    f32 = torch.float32
    good = dict(dout=tb["q"].clone(), dq=torch.zeros(tb["q"].shape, dtype=f32),
                dk=torch.zeros(tb["k_cache"].shape, dtype=f32), dv=torch.zeros(tb["k_cache"].shape, dtype=f32))
    ws = torch.zeros(1 << 20, dtype=torch.uint8)

    def call(g):
        rk.attn_prefill_backward(pb, tb["q"], tb["k_cache"], tb["v_cache"], tb["block_table"], tb["kv_lens"],
                                 tb["position_ids"], tb["out"], tb["lse"], g["dout"], g["dq"], g["dk"], g["dv"], ws)

    with pytest.raises(ValueError, match="expected a CUDA tensor"):
        call(good)
    for k, shape in (("dout", (2, 32, 2, 128)), ("dq", (2, 32, 3, 127)), ("dk", (6, 16, 8, 64)),
                     ("dv", (5, 16, 8, 128))):
        g = dict(good)
        g[k] = torch.zeros(shape, dtype=good[k].dtype)
        with pytest.raises(ValueError, match="the plan needs"):
            call(g)


def test_plan_wait_limit_defaults(rk):
    """Plans start with the 2 s wait limit and no timeout drill."""
    p = rk.plan(2, 1, 32, 8, 128, 16, 6, 3)
    assert p.wait_limit_ns == 2_000_000_000 and p.timeout_drill == 0
    pr, _ = rk.plan_ragged(2, 5, 32, 8, 128, 16, 6, 3, [0, 2, 5])
    assert pr.wait_limit_ns == 2_000_000_000 and pr.timeout_drill == 0
