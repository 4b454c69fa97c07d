"""GPU parity and invariance tests of rk_paged_attn_decode (through the C ABI)."""
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


def test_decode_small_parity():
    """B=2, kv_len 128, query at 128 (the pages' strict decode check shape)."""
    w = workloads.decode_small()
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 8), (64, 8), (16, 4), (4, 1)])
def test_decode_ragged_parity(Hq, Hkv):
    kv = [1, 2, 15, 16, 17, 100, 255, 256, 257, 300, 1000]
    w = workloads.random_case(len(kv), 1, Hq, Hkv, 128, kv, seed=7 + Hq + Hkv, mode="decode")
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_decode_query_at_last_key():
    """Trailing convention: query position kv_len-1 (its own key in the cache)."""
    kv = [1, 16, 33, 700]
    w = workloads.random_case(4, 1, 32, 8, 128, kv, seed=99, mode="decode", q_pos_offset=0)
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_decode_empty_rows():
    kv = [0, 37, 0]
    w = workloads.random_case(3, 1, 32, 8, 128, kv, seed=5, mode="decode")
    w.position_ids[0, 0] = 0
    w.position_ids[2, 0] = 0
    out, lse = run_gpu(w)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.all(torch.isneginf(lse[0])) and torch.all(torch.isneginf(lse[2]))
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def _invariance_outputs(W):
    w = workloads.decode_invariance(W)
    return w, run_gpu(w)


def test_decode_batch_width_graph_invariance_bitwise():
    """Same row alone, at two batch positions, at table widths 128/256, and
    under CUDA graph replay: bitwise equal (and matching the oracle)."""
    w128 = workloads.decode_invariance(128)
    out, lse = run_gpu(w128)
    ro, rl = oracle_ref(w128)
    assert_parity(out, lse, ro, rl)
    w256 = workloads.decode_invariance(256)
    w256.block_table = workloads.repad(w128.block_table, 256)
    o2, l2 = run_gpu(w256)
    assert bitwise_equal(out, o2) and bitwise_equal(lse, l2)
    rev = workloads.select_rows(w128, list(range(7, -1, -1)))
    o3, l3 = run_gpu(rev)
    assert bitwise_equal(out.flip(0), o3) and bitwise_equal(lse.flip(0), l3)
    for b in range(8):
        one = workloads.select_rows(w128, [b], W=256 if b % 2 else 128)
        o4, l4 = run_gpu(one)
        assert bitwise_equal(out[b:b + 1], o4) and bitwise_equal(lse[b:b + 1], l4), b
    # CUDA graph: capture once, replay with new metadata contents
    d = to_dev(w128)
    p = binding.plan(8, 1, 32, 8, 128, 16, w128.num_pages, 128)
    go = torch.empty_like(d["q"])
    gl = torch.empty((8, 32, 1), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.attn_decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                            d["position_ids"], go, gl, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.attn_decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                            d["position_ids"], go, gl)
    go.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert bitwise_equal(out, go) and bitwise_equal(lse, gl)
    # replay after swapping the metadata contents (rows reversed)
    d["q"].copy_(rev.q.cuda())
    d["block_table"].copy_(rev.block_table.cuda())
    d["kv_lens"].copy_(rev.kv_lens.cuda())
    d["position_ids"].copy_(rev.position_ids.cuda())
    g.replay()
    torch.cuda.synchronize()
    assert bitwise_equal(o3, go) and bitwise_equal(l3, gl)


def test_decode_rows_in_a_multi_wave_batch_bitwise():
    """The eight ragged invariance rows (partial last pages included) give the
    same bits alone and repeated in a batch whose grid (8 CTAs a row) exceeds
    the SM count, so that rows run in later waves next to other rows.
    Repeated rows share pages, so the host plan (which rejects shared pages)
    is skipped."""
    w = workloads.decode_invariance(128)
    out, lse = run_gpu(w)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    reps = (n_sm // (8 * 8)) + 2
    big = workloads.select_rows(w, list(range(8)) * reps)
    assert big.B * 8 > n_sm
    o2, l2 = run_gpu(big, validate=False)
    for r in range(reps):
        assert bitwise_equal(out, o2[8 * r:8 * r + 8]) and bitwise_equal(lse, l2[8 * r:8 * r + 8]), r


def test_decode_page_permutation_bitwise():
    w = workloads.decode_invariance(128)
    out, lse = run_gpu(w)
    o2, l2 = run_gpu(workloads.permute_pages(w, seed=3))
    assert bitwise_equal(out, o2) and bitwise_equal(lse, l2)


def test_decode_deterministic_repeat():
    w = workloads.decode_invariance(128)
    a = run_gpu(w)
    b = run_gpu(w)
    assert bitwise_equal(a[0], b[0]) and bitwise_equal(a[1], b[1])


def test_decode_throughput_config_sampled_parity():
    """B=64, kv 4096, as timed by the benchmark: 8 sampled rows vs the oracle."""
    w = workloads.decode_throughput()
    out, lse = run_gpu(w, validate=False)
    mask = np.zeros((64, 1), np.uint8)
    mask[[0, 9, 21, 32, 40, 51, 62, 63]] = 1
    ro, rl = oracle_ref(w, row_mask=mask)
    assert_parity(out, lse, ro, rl, mask=mask)


def test_decode_long_context_parity():
    w = workloads.decode_long()
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_decode_row_wider_than_the_page_id_copy():
    """A row of 40000 tokens (2500 pages): the kernel keeps the first 2048 page
    ids of a CTA's range in shared memory and reads the rest from the table;
    both halves of the row against the oracle, and in a batch with a short row."""
    w = workloads.random_case(2, 1, 32, 8, 128, [40000, 333], seed=61, mode="decode")
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_decode_device_status_on_corrupt_metadata():
    """Unsafe device metadata: flagged in status, that row zeroed with NaN LSE,
    other rows untouched; no trap."""
    w = workloads.random_case(3, 1, 32, 8, 128, [40, 50, 60], seed=11, mode="decode")
    good_out, good_lse = run_gpu(w)
    d = to_dev(w)
    d["block_table"][1, 1] = w.num_pages + 5            # out of range page
    d["kv_lens"][2] = w.W * 16 + 1                      # longer than the table
    p = binding.plan(3, 1, 32, 8, 128, 16, w.num_pages, w.W)
    out = torch.empty_like(d["q"])
    lse = torch.empty((3, 32, 1), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.attn_decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                        d["position_ids"], out, lse, status=st)
    torch.cuda.synchronize()
    s = int(st.item())
    assert s & binding.STATUS_PAGE_OOB and s & binding.STATUS_KVLEN
    assert not (s & binding.STATUS_TIMEOUT)
    assert torch.all(out[1:] == 0) and torch.all(torch.isnan(lse[1:]))
    assert bitwise_equal(out[0], good_out[0]) and bitwise_equal(lse[0], good_lse[0])


def test_decode_launch_does_not_synchronize():
    w = workloads.decode_small()
    d = to_dev(w)
    p = binding.plan(2, 1, 32, 8, 128, 16, w.num_pages, w.W)
    out = torch.empty_like(d["q"])
    lse = torch.empty((2, 32, 1), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.set_sync_debug_mode("error")
    try:
        binding.attn_decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                            d["position_ids"], out, lse)
    finally:
        torch.cuda.set_sync_debug_mode("default")
    torch.cuda.synchronize()


def test_decode_range_guard_flags_instead_of_overflowing():
    """A pre-RoPE key element of 40000 (beyond the FP16 score-operand range once
    rotated): that (row, KV head)'s heads get zeros and NaN LSE and the status
    bit is set; all other outputs still match the oracle."""
    w = workloads.random_case(2, 1, 32, 8, 128, [60, 90], seed=43, mode="decode")
    page = int(w.block_table[1, 2])
    w.k_cache[page, 5, 3, 7] = -40000.0
    d = to_dev(w)
    p = binding.plan(2, 1, 32, 8, 128, 16, w.num_pages, w.W)
    out = torch.empty_like(d["q"])
    lse = torch.empty((2, 32, 1), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.attn_decode(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                        d["position_ids"], out, lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == binding.STATUS_RANGE
    assert torch.all(out[1, 12:16] == 0) and torch.all(torch.isnan(lse[1, 12:16]))
    ro, rl = oracle_ref(w)
    keep = np.ones((2, 32), bool)
    keep[1, 12:16] = False
    o = out.float().cpu().numpy()[keep]
    l_ = lse.cpu().numpy()[keep]
    assert np.max(np.abs(o - ro[keep])) <= 2e-2 and np.max(np.abs(l_ - rl[keep])) <= 1e-3
