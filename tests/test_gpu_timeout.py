"""The fail-closed timeout exit of the tensor-core kernels, run for real.

Every pipeline wait inside a kernel gives up after the plan's wait limit; the
CTA then waits out its copies in flight, frees its tensor memory, writes its
rows as failed (out = 0, lse = NaN; NaN gradients) and sets
RK_STATUS_TIMEOUT, so that a lost pipeline participant can neither hang the
GPU nor leave a plausible but wrong result ("Add FlashInfer RoPE-fused paged
attention scaffold": fail closed, no silent fallback).  The plan's
timeout_drill flag makes each CTA's MMA issuer first wait on a barrier that
nothing completes (a bounded wait on a flag nothing sets), with the limit at
its 1 us floor, so the exit runs in every CTA.  Each case then checks that a
normal call on the same stream afterwards is bitwise equal to the same call
made before the drill: the context, the tensor memory and the kernels' state
are intact.
"""
import numpy as np
import pytest
import torch

from deterministic_paged_kv_gb300 import binding, workloads
from helpers import assert_parity, bitwise_equal, oracle_ref, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from deterministic_paged_kv_gb300 import build
    build.build()
    binding.load()


def _plan(w, Sq=None):
    return binding.plan(w.B, Sq or w.Sq, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                        w.position_ids, w.rope_theta, w.rope_scale)


def _drill(p):
    p.wait_limit_ns = 1  # clamped to the 1 us floor by the launch calls
    p.timeout_drill = 1
    return p


def _call(fn, p, d, out_shape, lse_shape, status=None, **kw):
    out = torch.full(out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(lse_shape, 7.0, dtype=torch.float32, device="cuda")
    fn(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"], d["position_ids"], out, lse,
       status=status, **kw)
    return out, lse


def _check_failed(out, lse, st):
    torch.cuda.synchronize()
    assert int(st.item()) & binding.STATUS_TIMEOUT
    assert bool((out.float() == 0).all()), "failed rows must be written as zeros"
    assert bool(torch.isnan(lse).all()), "failed rows must carry a NaN LSE"


@pytest.mark.parametrize("split", [0, 1024])
def test_decode_timeout_exit(split):
    w = workloads.random_case(3, 1, 32, 8, 128, [300, 77, 2500], seed=211, mode="decode")
    d = to_dev(w)
    shp, lshp = (w.B, w.Hq, 1, w.D), (w.B, w.Hq, 1)
    if split:
        p0 = _plan(w)
        scratch = torch.empty(binding.decode_split_scratch_bytes(p0, split), dtype=torch.uint8, device="cuda")
        fn = lambda p, *a, **k: binding.attn_decode_split(p, split, *a[:8], scratch, **k)  # noqa: E731
    else:
        fn = binding.attn_decode
    ref_out, ref_lse = _call(fn, _plan(w), d, shp, lshp)
    torch.cuda.synchronize()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _call(fn, _drill(_plan(w)), d, shp, lshp, status=st)
    _check_failed(out, lse, st)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    out2, lse2 = _call(fn, _plan(w), d, shp, lshp, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert bitwise_equal(out2, ref_out) and bitwise_equal(lse2, ref_lse)
    ro, rl = oracle_ref(w)
    assert_parity(out2, lse2, ro, rl)


def test_prefill_timeout_exit():
    w = workloads.random_case(2, 70, 32, 8, 128, [600, 1333], seed=223, mode="prefill")
    d = to_dev(w)
    shp, lshp = tuple(w.q.shape), (w.B, w.Hq, w.Sq)
    ref_out, ref_lse = _call(binding.attn_prefill, _plan(w), d, shp, lshp)
    torch.cuda.synchronize()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _call(binding.attn_prefill, _drill(_plan(w)), d, shp, lshp, status=st)
    _check_failed(out, lse, st)
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    out2, lse2 = _call(binding.attn_prefill, _plan(w), d, shp, lshp, status=st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert bitwise_equal(out2, ref_out) and bitwise_equal(lse2, ref_lse)
    ro, rl = oracle_ref(w)
    assert_parity(out2, lse2, ro, rl)


def test_ragged_timeout_exit():
    w = workloads.ragged_case([1, 40, 1, 300], [200, 500, 64, 900], seed=227)
    q, ind, pos = workloads.pack_ragged(w)
    p, mq = binding.plan_ragged(w.B, q.shape[0], w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, ind, w.block_table,
                                w.kv_lens, pos, w.rope_theta, w.rope_scale)
    d = to_dev(w)
    dq, dind, dpos = q.cuda(), ind.cuda(), pos.cuda()

    def call(plan, status=None):
        out = torch.full((q.shape[0], w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((q.shape[0], w.Hq), 7.0, dtype=torch.float32, device="cuda")
        binding.attn_ragged(plan, mq, dind, dq, d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"], dpos,
                            out, lse, status=status)
        return out, lse

    ref_out, ref_lse = call(p)
    torch.cuda.synchronize()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pd = binding.Plan.from_buffer_copy(p)
    out, lse = call(_drill(pd), st)
    _check_failed(out, lse, st)  # decode rows and prefill rows alike
    out2, lse2 = call(p)
    torch.cuda.synchronize()
    assert bitwise_equal(out2, ref_out) and bitwise_equal(lse2, ref_lse)


def test_backward_timeout_exit():
    w = workloads.random_case(2, 40, 32, 8, 128, [300, 77], seed=229, mode="prefill")
    d = to_dev(w)
    p = _plan(w)
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device="cuda")
    binding.attn_prefill(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                         d["position_ids"], out, lse)
    dout = torch.randn(w.q.shape, generator=torch.Generator().manual_seed(5)).to(torch.bfloat16).cuda()
    ws = torch.empty(binding.prefill_backward_workspace_bytes(p), dtype=torch.uint8, device="cuda")

    def call(plan, status=None):
        g = [torch.full(w.q.shape, 3.0, dtype=torch.float32, device="cuda"),
             torch.full(w.k_cache.shape, 3.0, dtype=torch.float32, device="cuda"),
             torch.full(w.v_cache.shape, 3.0, dtype=torch.float32, device="cuda")]
        binding.attn_prefill_backward(plan, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                                      d["position_ids"], out, lse, dout, *g, ws, status=status)
        return g

    ref = call(p)
    torch.cuda.synchronize()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = call(_drill(_plan(w)), st)
    torch.cuda.synchronize()
    assert int(st.item()) & binding.STATUS_TIMEOUT
    assert bool(torch.isnan(got[0]).all())
    used = np.zeros(w.num_pages, bool)  # pages the rows reference: written, as NaN
    for b in range(w.B):
        for j in range((int(w.kv_lens[b]) + 15) // 16):
            used[int(w.block_table[b, j])] = True
    for g in got[1:]:
        gc = g.cpu()
        assert bool(torch.isnan(gc[torch.from_numpy(used)]).all())
        assert bool((gc[torch.from_numpy(~used)] == 3.0).all())
    again = call(p)
    torch.cuda.synchronize()
    for a, r in zip(again, ref):
        assert torch.equal(a.view(torch.int32), r.view(torch.int32))
