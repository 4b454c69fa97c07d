"""GPU tests of rk_paged_attn_ragged: a mixed batch of decode rows (one query)
and prefill chunks of any length against the oracle; every row bitwise equal to
the padded entry point that serves its kind and to itself run alone; CUDA graph
replay with new metadata; unsafe qo_indptr."""
import numpy as np
import pytest
import torch

from deterministic_paged_kv_gb300 import binding, workloads
from helpers import assert_parity, bitwise_equal, oracle_ref, run_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from deterministic_paged_kv_gb300 import build
    build.build()
    binding.load()


MIXED_Q = [1, 0, 37, 130, 1, 2, 256, 1]
MIXED_KV = [200, 50, 300, 500, 1, 2, 2048, 4095]


def run_ragged(w, status=None, max_q_len=None):
    q, ind, pos = workloads.pack_ragged(w)
    p, mq = binding.plan_ragged(w.B, q.shape[0], w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, ind, w.block_table,
                                w.kv_lens, pos, w.rope_theta, w.rope_scale)
    d = to_dev(w)
    out = torch.full((q.shape[0], w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((q.shape[0], w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    binding.attn_ragged(p, max_q_len or mq, ind.cuda(), q.cuda(), d["k_cache"], d["v_cache"], d["block_table"],
                        d["kv_lens"], pos.cuda(), out, lse, status=status)
    torch.cuda.synchronize()
    return out, lse, ind


def padded_view(w, out, lse, ind):
    """Packed results laid out as the padded [B, Hq, max_q, D] / [B, Hq, max_q]."""
    B, Hq, mq, D = w.q.shape
    po = torch.zeros((B, Hq, mq, D), dtype=out.dtype)
    pl = torch.full((B, Hq, mq), float("nan"), dtype=torch.float32)
    for b in range(B):
        s, e = int(ind[b]), int(ind[b + 1])
        po[b, :, :e - s] = out[s:e].transpose(0, 1).cpu()
        pl[b, :, :e - s] = lse[s:e].transpose(0, 1).cpu()
    return po, pl


def row_mask(w):
    ql = w.meta["q_lens"]
    m = np.zeros((w.B, w.Sq), np.uint8)
    for b, n in enumerate(ql):
        m[b, :n] = 1
    return m


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (64, 8)])
def test_ragged_mixed_batch_parity(Hq, Hkv):
    w = workloads.ragged_case(MIXED_Q, MIXED_KV, seed=111, Hq=Hq, Hkv=Hkv)
    out, lse, ind = run_ragged(w)
    po, pl = padded_view(w, out, lse, ind)
    m = row_mask(w)
    ro, rl = oracle_ref(w, row_mask=m)
    assert_parity(po, pl, ro, rl, mask=m)


def test_ragged_rows_match_padded_entry_points_and_themselves_alone():
    """Each row: bitwise equal to the padded decode (one query) or padded
    prefill (several) run on that row alone, and to the row as a ragged batch
    of one -- the kernel and the arithmetic depend only on the row."""
    w = workloads.ragged_case(MIXED_Q, MIXED_KV, seed=113)
    out, lse, ind = run_ragged(w)
    for b, n in enumerate(w.meta["q_lens"]):
        if n == 0:
            continue
        s, e = int(ind[b]), int(ind[b + 1])
        one = workloads.select_rows(w, [b])
        pw = workloads.build("row", 1, n, w.Hq, w.Hkv, w.D, [int(w.kv_lens[b])], one.num_pages, one.W, 0, "decode")
        pw.q = one.q[:, :, :n].contiguous()
        pw.k_cache, pw.v_cache, pw.block_table = one.k_cache, one.v_cache, one.block_table
        pw.position_ids = one.position_ids[:, :n].contiguous()
        po, pl = run_gpu(pw, mode="decode" if n == 1 else "prefill")
        assert bitwise_equal(out[s:e], po[0].transpose(0, 1).contiguous()), b
        assert bitwise_equal(lse[s:e], pl[0].transpose(0, 1).contiguous()), b
        solo = workloads.ragged_case([n], [int(w.kv_lens[b])], seed=0)
        solo.q = one.q[:, :, :max(n, 1)].contiguous()
        solo.k_cache, solo.v_cache, solo.block_table = one.k_cache, one.v_cache, one.block_table
        solo.position_ids = one.position_ids[:, :max(n, 1)].contiguous()
        so, sl, _ = run_ragged(solo)
        assert bitwise_equal(out[s:e], so) and bitwise_equal(lse[s:e], sl), b


def test_ragged_graph_replay_with_new_metadata():
    w = workloads.ragged_case(MIXED_Q, MIXED_KV, seed=117)
    ref_out, ref_lse, _ = run_ragged(w)
    q, ind, pos = workloads.pack_ragged(w)
    p, mq = binding.plan_ragged(w.B, q.shape[0], w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, ind)
    d = to_dev(w)
    dq, dind, dpos = q.cuda(), ind.cuda(), pos.cuda()
    out = torch.empty((q.shape[0], w.Hq, w.D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((q.shape[0], w.Hq), dtype=torch.float32, device="cuda")
    args = lambda: (p, mq, dind, dq, d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"], dpos, out, lse)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.attn_ragged(*args(), stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.attn_ragged(*args())
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert bitwise_equal(out, ref_out) and bitwise_equal(lse, ref_lse)
    # new contents: the rows in reverse order (same total_q and max_q_len)
    order = list(range(w.B - 1, -1, -1))
    rw = workloads.select_rows(w, order)
    rw.meta["q_lens"] = [w.meta["q_lens"][b] for b in order]
    rq, rind, rpos = workloads.pack_ragged(rw)
    r_out, r_lse, _ = run_ragged(rw)
    dq.copy_(rq.cuda())
    dind.copy_(rind.cuda())
    dpos.copy_(rpos.cuda())
    d["block_table"].copy_(rw.block_table.cuda())
    d["kv_lens"].copy_(rw.kv_lens.cuda())
    g.replay()
    torch.cuda.synchronize()
    assert bitwise_equal(out, r_out) and bitwise_equal(lse, r_lse)


def test_ragged_status_on_unsafe_indptr_and_oversize_rows():
    w = workloads.ragged_case([2, 40, 1, 3], [100, 200, 300, 400], seed=119)
    good_out, good_lse, ind = run_ragged(w)
    q, ind, pos = workloads.pack_ragged(w)
    p, mq = binding.plan_ragged(w.B, q.shape[0], w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, ind)
    d = to_dev(w)
    bad = ind.clone()
    bad[2] = q.shape[0] + 9            # rows 1 and 2 now out of range
    out = torch.full((q.shape[0], w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((q.shape[0], w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.attn_ragged(p, mq, bad.cuda(), q.cuda(), d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                        pos.cuda(), out, lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & binding.STATUS_POSITION
    s0, e0 = int(ind[0]), int(ind[1])
    assert bitwise_equal(out[s0:e0], good_out[s0:e0]) and bitwise_equal(lse[s0:e0], good_lse[s0:e0])
    # a row longer than max_q_len is not computed and is flagged
    st.zero_()
    out.fill_(float("nan"))
    binding.attn_ragged(p, 3, ind.cuda(), q.cuda(), d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                        pos.cuda(), out, lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & binding.STATUS_POSITION
    s3, e3 = int(ind[3]), int(ind[4])
    assert bitwise_equal(out[s3:e3], good_out[s3:e3])
    # max_q_len 1: only the decode launch runs; it flags the longer rows
    st.zero_()
    out.fill_(float("nan"))
    binding.attn_ragged(p, 1, ind.cuda(), q.cuda(), d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                        pos.cuda(), out, lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & binding.STATUS_POSITION
    s2, e2 = int(ind[2]), int(ind[3])
    assert bitwise_equal(out[s2:e2], good_out[s2:e2]) and bool(torch.isnan(out[s0:e0].float()).all())


def _launch(w, p, max_q_len, ind=None, status=None):
    q, ind0, pos = workloads.pack_ragged(w)
    ind = ind0 if ind is None else ind
    d = to_dev(w)
    out = torch.full((q.shape[0], w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((q.shape[0], w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    binding.attn_ragged(p, max_q_len, ind.cuda(), q.cuda(), d["k_cache"], d["v_cache"], d["block_table"],
                        d["kv_lens"], pos.cuda(), out, lse, status=status)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("case", ["600_rows", "35_levels"])
def test_ragged_many_rows_and_levels_match_oracle_and_the_bounded_grid(case):
    """600 rows (more than the 512 threads that rank rows in one pass), or one
    row of 35 pairs of q-tiles (more than the 32 levels one warp scans at a
    time), G = 8 (32-query pairs): parity with the oracle, and the grid bounded
    over every batch of this shape (pf_units = -1) gives the same bits as the
    exact count."""
    rng = np.random.default_rng(123)
    if case == "600_rows":
        q_lens = [int(x) for x in rng.choice([1, 1, 1, 2, 3, 17, 33, 64, 65], size=600)]
    else:
        q_lens = [1, 1100, 40, 2, 0, 1]
    kv_lens = [int(n + rng.integers(0, 40)) for n in q_lens]
    w = workloads.ragged_case(q_lens, kv_lens, seed=131, Hq=8, Hkv=1)
    q, ind, pos = workloads.pack_ragged(w)
    p, mq = binding.plan_ragged(w.B, q.shape[0], w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, ind, w.block_table,
                                w.kv_lens, pos, w.rope_theta, w.rope_scale)
    assert p.pf_units == sum(-(-n // 32) for n in q_lens if n >= 2)
    out, lse = _launch(w, p, mq)
    po, pl = padded_view(w, out, lse, ind)
    m = row_mask(w)
    ro, rl = oracle_ref(w, row_mask=m)
    assert_parity(po, pl, ro, rl, mask=m)
    p.pf_units = -1
    out2, lse2 = _launch(w, p, mq)
    assert bitwise_equal(out, out2) and bitwise_equal(lse, lse2)


def test_ragged_grid_smaller_than_the_device_batch_is_flagged():
    """A plan counted from another qo_indptr of the same total_q: the units
    that fit are computed (bitwise as usual), the rest flag RK_STATUS_POSITION."""
    w = workloads.ragged_case([2, 2, 1, 1], [100, 300, 50, 60], seed=137)
    good_out, good_lse, ind = run_ragged(w)
    T = int(ind[-1])
    p_small, _ = binding.plan_ragged(w.B, T, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, [0, 3, 4, 5, 6])
    assert p_small.pf_units == 1
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = _launch(w, p_small, 2, status=st)
    assert int(st.item()) & binding.STATUS_POSITION
    # unit 0 (level 0, first row) ran; decode rows ran in their own launch
    assert bitwise_equal(out[0:2], good_out[0:2]) and bitwise_equal(lse[0:2], good_lse[0:2])
    assert bitwise_equal(out[4:6], good_out[4:6]) and bitwise_equal(lse[4:6], good_lse[4:6])
