"""GPU tests of the fixed-split decode (rk_paged_attn_decode_split): parity with
the oracle across several splits, bitwise batch / width / graph invariance for a
given split length, the ordered merge's empty and unsafe cases, and argument
checks."""
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


@pytest.mark.parametrize("split", [16, 528, 1024, 2048, 3072])
def test_split_decode_ragged_parity(split):
    """Rows shorter than, equal to and several times the split length, with a
    ragged last page; every row against the oracle.  Split lengths are any
    multiple of the page size: 16 (one page per split), 528 (splits that start
    and end inside 128-token tiles), multiples of 1024."""
    kv = [1, 1000, 1024, 2048, 3000, 5003]
    w = workloads.random_case(len(kv), 1, 32, 8, 128, kv, seed=41, mode="decode", extra_pages=16)
    out, lse = run_gpu(w, split_tokens=split)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4), (64, 8)])
def test_split_decode_gqa_groups(Hq, Hkv):
    w = workloads.random_case(2, 1, Hq, Hkv, 128, [2500, 4100], seed=43, mode="decode")
    out, lse = run_gpu(w, split_tokens=1024)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_split_decode_long_context_parity():
    """B=1, kv_len 32768: 16 splits of 2048 tokens give the row 128 CTAs."""
    w = workloads.decode_long()
    out, lse = run_gpu(w, split_tokens=2048)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_split_decode_close_to_split_free():
    """A separate arithmetic policy: not bitwise equal to the split-free path,
    but both within the oracle tolerance of each other."""
    w = workloads.decode_invariance(128)
    a_out, a_lse = run_gpu(w)
    b_out, b_lse = run_gpu(w, split_tokens=1024)
    assert float((a_out.float() - b_out.float()).abs().max()) <= 2e-2
    assert float((a_lse - b_lse).abs().max()) <= 1e-3


@pytest.mark.parametrize("split", [16, 528, 1024])
def test_split_decode_batch_width_graph_invariance_bitwise(split):
    """For a fixed split length: the same row alone, reversed in the batch, at
    table widths 128 / 256 (more, empty splits), and under CUDA graph replay
    with new metadata contents -- bitwise equal."""
    w128 = workloads.decode_invariance(128)
    out, lse = run_gpu(w128, split_tokens=split)
    ro, rl = oracle_ref(w128)
    assert_parity(out, lse, ro, rl)
    w256 = workloads.decode_invariance(256)
    w256.block_table = workloads.repad(w128.block_table, 256)
    o2, l2 = run_gpu(w256, split_tokens=split)
    assert bitwise_equal(out, o2) and bitwise_equal(lse, l2)
    rev = workloads.select_rows(w128, list(range(7, -1, -1)))
    o3, l3 = run_gpu(rev, split_tokens=split)
    assert bitwise_equal(out.flip(0), o3) and bitwise_equal(lse.flip(0), l3)
    for b in range(8):
        one = workloads.select_rows(w128, [b], W=256 if b % 2 else 128)
        o4, l4 = run_gpu(one, split_tokens=split)
        assert bitwise_equal(out[b:b + 1], o4) and bitwise_equal(lse[b:b + 1], l4), b
    d = to_dev(w128)
    p = binding.plan(8, 1, 32, 8, 128, 16, w128.num_pages, 128)
    scratch = torch.empty(binding.decode_split_scratch_bytes(p, split), dtype=torch.uint8, device="cuda")
    go = torch.empty_like(d["q"])
    gl = torch.empty((8, 32, 1), dtype=torch.float32, device="cuda")
    args = lambda: (p, split, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                    d["position_ids"], go, gl, scratch)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.attn_decode_split(*args(), stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.attn_decode_split(*args())
    go.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert bitwise_equal(out, go) and bitwise_equal(lse, gl)
    d["q"].copy_(rev.q.cuda())
    d["block_table"].copy_(rev.block_table.cuda())
    d["kv_lens"].copy_(rev.kv_lens.cuda())
    d["position_ids"].copy_(rev.position_ids.cuda())
    g.replay()
    torch.cuda.synchronize()
    assert bitwise_equal(o3, go) and bitwise_equal(l3, gl)


def test_split_decode_empty_rows_and_repeat():
    w = workloads.random_case(3, 1, 32, 8, 128, [0, 2100, 5], seed=47, mode="decode")
    w.position_ids[0, 0] = 0
    out, lse = run_gpu(w, split_tokens=1024)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)
    o2, l2 = run_gpu(w, split_tokens=1024)
    assert bitwise_equal(out, o2) and bitwise_equal(lse, l2)


def test_split_decode_status_on_corrupt_metadata():
    """A page id out of range in one split of a row: that row zeroed with NaN
    LSE and the status bit set; the other rows untouched."""
    w = workloads.random_case(3, 1, 32, 8, 128, [3000, 2500, 1500], seed=53, mode="decode")
    good_out, good_lse = run_gpu(w, split_tokens=1024)
    d = to_dev(w)
    d["block_table"][1, 100] = w.num_pages + 7  # in the row's second split
    p = binding.plan(3, 1, 32, 8, 128, 16, w.num_pages, w.W)
    scratch = torch.empty(binding.decode_split_scratch_bytes(p, 1024), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(d["q"])
    lse = torch.empty((3, 32, 1), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.attn_decode_split(p, 1024, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                              d["position_ids"], out, lse, scratch, status=st)
    torch.cuda.synchronize()
    s = int(st.item())
    assert s & binding.STATUS_PAGE_OOB and not (s & binding.STATUS_TIMEOUT)
    assert torch.all(out[1] == 0) and torch.all(torch.isnan(lse[1]))
    for b in (0, 2):
        assert bitwise_equal(out[b], good_out[b]) and bitwise_equal(lse[b], good_lse[b])


def test_split_decode_argument_checks():
    w = workloads.random_case(1, 1, 32, 8, 128, [100], seed=59, mode="decode")
    d = to_dev(w)
    p = binding.plan(1, 1, 32, 8, 128, 16, w.num_pages, w.W)
    need = binding.decode_split_scratch_bytes(p, 1024)
    n_splits = -(-w.W * 16 // 1024)
    assert need == 1 * 32 * n_splits * (128 + 1) * 4
    out = torch.empty_like(d["q"])
    lse = torch.empty((1, 32, 1), dtype=torch.float32, device="cuda")
    small = torch.empty(need - 4, dtype=torch.uint8, device="cuda")
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"], d["position_ids"], out, lse)
    with pytest.raises(binding.RkError) as e:
        binding.attn_decode_split(p, 1024, *args, small)
    assert e.value.name == "RK_E_ARG"
    ok = torch.empty(need, dtype=torch.uint8, device="cuda")
    for bad in (0, 8, 1000, -1024, 24 + 1):
        with pytest.raises(binding.RkError) as e:
            binding.attn_decode_split(p, bad, *args, ok)
        assert e.value.name == "RK_E_ARG"
