"""GPU tests of the balanced split-free decode (rk_paged_attn_decode_balanced).

The balanced schedule deals blocks of 1-8 tiles of every (row, KV head) to one
CTA per SM and hands a row's running state from CTA to CTA where it crosses a
boundary (a segment that starts between RoPE anchor tiles replays the angle
steps since the last anchor), so each row is still reduced tile after tile in ascending order by
the operations of the one-CTA-per-(row, KV head) launch.  Every test here
compares the two launches bitwise (the split-free decode's own parity with the
oracle is tested elsewhere, and again here on ragged rows).  The launch epoch
in the first scratch word advances once per balanced launch, which tells the
tests the balanced schedule really ran (it is used only when the batch has at
least as many rows as a KV head's chain has CTAs).
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


@pytest.fixture(scope="module")
def scratch():
    return torch.zeros(binding.BALANCED_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")


def _epoch(scratch):
    torch.cuda.synchronize()
    return int(scratch[:8].view(torch.int32)[0].item()), int(scratch[:8].view(torch.int32)[1].item())


def _plan(w):
    return binding.plan(w.B, 1, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                        w.position_ids, w.rope_theta, w.rope_scale)


def _args(d):
    return (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"], d["position_ids"])


def _outs(w):
    out = torch.full((w.B, w.Hq, 1, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((w.B, w.Hq, 1), 7.0, dtype=torch.float32, device="cuda")
    return out, lse


def _both(w, scratch, p=None, d=None):
    """(per-(row, KV head) out, lse, status), (balanced out, lse, status)."""
    d = d or to_dev(w)
    p = p or _plan(w)
    res = []
    for bal in (False, True):
        out, lse = _outs(w)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        if bal:
            binding.attn_decode_balanced(p, *_args(d), out, lse, scratch, status=st)
        else:
            binding.attn_decode(p, *_args(d), out, lse, status=st)
        torch.cuda.synchronize()
        res.append((out, lse, int(st.item())))
    return res


def _ragged_kv(B, seed, hi=6000):
    rng = np.random.default_rng(seed)
    kv = [int(x) for x in rng.integers(1, hi, size=B)]
    kv[0], kv[1], kv[2], kv[3] = 0, 1024, 2048, 127  # empty, block-aligned and sub-tile rows
    return kv


def test_balanced_ragged_rows_bitwise_and_parity(scratch):
    """40 rows (320 (row, KV head) pairs) of 0..6000 keys: rows cut at every kind
    of block boundary; bitwise equal to the one-CTA launch and within the
    oracle tolerance."""
    kv = _ragged_kv(40, 5)
    w = workloads.random_case(len(kv), 1, 32, 8, 128, kv, seed=301, mode="decode")
    e0, _ = _epoch(scratch)
    (o1, l1, s1), (o2, l2, s2) = _both(w, scratch)
    e1, done = _epoch(scratch)
    assert e1 == e0 + 1 and done == 0, "the balanced schedule did not run"
    assert s1 == 0 and s2 == 0
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)
    ro, rl = oracle_ref(w)
    assert_parity(o2, l2, ro, rl)
    assert bool(torch.isneginf(l2[0]).all()) and bool((o2[0].float() == 0).all())  # the empty row


def test_balanced_decode_throughput_shape_bitwise(scratch):
    """B=64 x kv 4096: 64 rows of 4 blocks over each KV head's chain."""
    w = workloads.decode_throughput()
    e0, _ = _epoch(scratch)
    (o1, l1, s1), (o2, l2, s2) = _both(w, scratch)
    assert _epoch(scratch)[0] == e0 + 1
    assert s1 == s2 == 0
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)


@pytest.mark.parametrize("Hq,Hkv,B", [(64, 8, 20), (8, 8, 20), (16, 4, 40), (4, 1, 160)])
def test_balanced_gqa_groups(scratch, Hq, Hkv, B):
    kv = _ragged_kv(B, 7 + Hq, hi=4000)
    w = workloads.random_case(B, 1, Hq, Hkv, 128, kv, seed=303 + Hq, mode="decode")
    e0, _ = _epoch(scratch)
    (o1, l1, s1), (o2, l2, s2) = _both(w, scratch)
    assert _epoch(scratch)[0] == e0 + 1
    assert s1 == s2 == 0
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)
    ro, rl = oracle_ref(w)
    assert_parity(o2, l2, ro, rl)


def test_balanced_long_row_crosses_many_ctas(scratch):
    """One row of 20000 keys among 18 short ones: its 20 blocks span several
    CTAs of each KV head's chain, so middle segments both take the row over and
    hand it on (a chain of hand-offs, each waiting for the one before); bitwise
    equal to the one-CTA launch and within the oracle tolerance."""
    kv = [20000] + [100 + 37 * i for i in range(18)]
    w = workloads.random_case(len(kv), 1, 32, 8, 128, kv, seed=331, mode="decode")
    e0, _ = _epoch(scratch)
    (o1, l1, s1), (o2, l2, s2) = _both(w, scratch)
    assert _epoch(scratch)[0] == e0 + 1
    assert s1 == s2 == 0
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)
    ro, rl = oracle_ref(w)
    assert_parity(o2, l2, ro, rl)


def test_balanced_fine_blocks_segments_between_anchors(scratch):
    """B=20 x kv 4096: blocks of 8 tiles would leave 3 of each chain's 19 CTAs
    without work, so the kernel cuts the rows in 2-tile blocks and most
    segments start between RoPE anchor tiles (their first angles come from the
    anchor before them and the replayed steps); bitwise equal to the one-CTA
    launch and within the oracle tolerance."""
    w = workloads.random_case(20, 1, 32, 8, 128, [4096] * 20, seed=337, mode="decode")
    e0, _ = _epoch(scratch)
    (o1, l1, s1), (o2, l2, s2) = _both(w, scratch)
    assert _epoch(scratch)[0] == e0 + 1
    assert s1 == s2 == 0
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)
    ro, rl = oracle_ref(w)
    assert_parity(o2, l2, ro, rl)


def test_balanced_single_tile_blocks_odd_segment_starts(scratch):
    """B=20 rows of 1000-1024 keys in a 64-page table: the host allows blocks of
    one tile and no coarser block gives every chain member work, so segments
    start on any tile, 1 to 7 tiles past a RoPE anchor (the replay of up to 7
    tiles of angle steps); bitwise equal to the one-CTA launch and within the
    oracle tolerance."""
    kv = [1024 - 3 * i for i in range(20)]
    w = workloads.random_case(len(kv), 1, 32, 8, 128, kv, seed=341, mode="decode", W=64)
    e0, _ = _epoch(scratch)
    (o1, l1, s1), (o2, l2, s2) = _both(w, scratch)
    assert _epoch(scratch)[0] == e0 + 1
    assert s1 == s2 == 0
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)
    ro, rl = oracle_ref(w)
    assert_parity(o2, l2, ro, rl)


def test_balanced_unsafe_rows_fail_like_the_one_cta_launch(scratch):
    """An out-of-range page id deep inside a long row (a segment other than the
    row's last one meets it) and a kv_len past the table: the same failed rows
    (out = 0, lse = NaN) and status bits as the one-CTA launch; the other rows
    bitwise equal."""
    kv = [3000] * 24
    w = workloads.random_case(len(kv), 1, 32, 8, 128, kv, seed=307, mode="decode")
    w.block_table[5, 10] = w.num_pages + 3  # tokens 160..175 of row 5
    w.kv_lens[9] = w.W * 16 + 1
    (o1, l1, s1), (o2, l2, s2) = _both(w, scratch, p=binding.plan(w.B, 1, 32, 8, 128, 16, w.num_pages, w.W))
    assert s1 == s2 and s2 & binding.STATUS_PAGE_OOB and s2 & binding.STATUS_KVLEN
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)
    for r in (5, 9):
        assert bool(torch.isnan(l2[r]).all()) and bool((o2[r].float() == 0).all())


def test_balanced_repeated_calls_and_graph_replay(scratch):
    """The scratch is reused: three calls in a row, then one captured call
    replayed three times, all bitwise equal to the first."""
    kv = _ragged_kv(32, 11, hi=5000)
    w = workloads.random_case(len(kv), 1, 32, 8, 128, kv, seed=311, mode="decode")
    d = to_dev(w)
    p = _plan(w)
    (o1, l1, _), (ref_o, ref_l, _) = _both(w, scratch, p=p, d=d)
    assert bitwise_equal(o1, ref_o) and bitwise_equal(l1, ref_l)
    e0, _ = _epoch(scratch)
    for _ in range(3):
        out, lse = _outs(w)
        binding.attn_decode_balanced(p, *_args(d), out, lse, scratch)
        torch.cuda.synchronize()
        assert bitwise_equal(out, ref_o) and bitwise_equal(lse, ref_l)
    assert _epoch(scratch)[0] == e0 + 3
    out, lse = _outs(w)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        binding.attn_decode_balanced(p, *_args(d), out, lse, scratch)
    torch.cuda.synchronize()
    e1, _ = _epoch(scratch)
    for _ in range(3):
        out.fill_(float("nan"))
        lse.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert bitwise_equal(out, ref_o) and bitwise_equal(lse, ref_l)
    assert _epoch(scratch) == (e1 + 3, 0)


def test_balanced_timeout_exit_then_recovers(scratch):
    """The timeout drill on the balanced schedule: every row with keys written
    as failed (the empty row has nothing to wait for and stays empty),
    RK_STATUS_TIMEOUT set, the epoch still advanced; the next call is bitwise
    equal to the one-CTA launch."""
    kv = _ragged_kv(24, 13, hi=5000)
    w = workloads.random_case(len(kv), 1, 32, 8, 128, kv, seed=313, mode="decode")
    d = to_dev(w)
    p = _plan(w)
    pdrill = binding.Plan.from_buffer_copy(p)
    pdrill.wait_limit_ns = 1
    pdrill.timeout_drill = 1
    e0, _ = _epoch(scratch)
    out, lse = _outs(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.attn_decode_balanced(pdrill, *_args(d), out, lse, scratch, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & binding.STATUS_TIMEOUT
    assert bool((out.float() == 0).all())
    assert kv[0] == 0 and bool(torch.isneginf(lse[0]).all()) and bool(torch.isnan(lse[1:]).all())
    assert _epoch(scratch) == (e0 + 1, 0)
    (o1, l1, s1), (o2, l2, s2) = _both(w, scratch, p=p, d=d)
    assert s1 == s2 == 0
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)


def test_balanced_small_batch_runs_the_one_cta_launch(scratch):
    """Fewer rows than a KV head's chain has CTAs: the call runs the
    one-CTA-per-pair launch (same results) and leaves the scratch alone."""
    w = workloads.random_case(3, 1, 32, 8, 128, [300, 77, 5000], seed=317, mode="decode")
    before = _epoch(scratch)
    (o1, l1, _), (o2, l2, _) = _both(w, scratch)
    assert _epoch(scratch) == before
    assert bitwise_equal(o1, o2) and bitwise_equal(l1, l2)


def test_balanced_scratch_is_checked(scratch):
    w = workloads.random_case(20, 1, 32, 8, 128, [100] * 20, seed=319, mode="decode")
    d = to_dev(w)
    p = _plan(w)
    out, lse = _outs(w)
    assert binding.decode_balanced_scratch_bytes(p) == binding.BALANCED_SCRATCH_BYTES
    for bad in (scratch[:1024], scratch[1:]):
        with pytest.raises(binding.RkError) as e:
            binding.attn_decode_balanced(p, *_args(d), out, lse, bad)
        assert e.value.name == "RK_E_ARG"
