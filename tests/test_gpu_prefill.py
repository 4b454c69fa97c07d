"""GPU parity and invariance tests of rk_paged_attn_prefill (through the C ABI)."""
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


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 8), (64, 8), (4, 1)])
def test_prefill_small_ragged_parity(Hq, Hkv):
    """Two q-tiles (one partial), ragged prefixes, early positions (few keys per
    query, where the FP16 score operands matter most for the LSE bound)."""
    kv = [300, 77, 41]
    w = workloads.random_case(3, 40, Hq, Hkv, 128, kv, seed=13 + Hq, mode="prefill")
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_prefill_late_positions():
    """Positions past 1024: several KV tiles per q-tile, RoPE anchors and angle
    steps across tiles, a ragged last page."""
    kv = [1100, 1333]
    w = workloads.random_case(2, 70, 32, 8, 128, kv, seed=17, mode="prefill")
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_prefill_query_at_kv_len_convention():
    """Last query position = kv_len (its own key not yet in the cache)."""
    w = workloads.random_case(2, 16, 32, 8, 128, [200, 1500], seed=23, mode="prefill", q_pos_offset=1)
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_prefill_single_query_and_empty_row():
    w = workloads.random_case(3, 1, 32, 8, 128, [0, 1, 513], seed=29, mode="prefill")
    w.position_ids[0, 0] = 0
    out, lse = run_gpu(w)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_prefill_back_to_back_tail_units():
    """Many short rows: every unit is a single KV tile whose last page is partly
    filled, and each CTA of the persistent grid runs several of them in a row,
    so the zeroing of one unit's V tail overlaps the next unit's copies."""
    rng = np.random.default_rng(31)
    kv = [int(x) for x in rng.integers(40, 128, size=48)]
    kv = [x + 1 if x % 16 == 0 else x for x in kv]
    w = workloads.random_case(len(kv), 40, 32, 8, 128, kv, seed=37, mode="prefill")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_gpu(w, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_prefill_chunk_config_parity():
    """B=4, 1536-token prefix + 512-token chunk: every output vs the oracle."""
    w = workloads.prefill_chunk()
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)


def test_prefill_long_sampled_parity():
    """B=1, S=8192 full causal: first 256, last 256 and every 31st position."""
    w = workloads.prefill_long()
    out, lse = run_gpu(w, validate=False)
    mask = np.zeros((1, 8192), np.uint8)
    mask[0, :256] = 1
    mask[0, -256:] = 1
    mask[0, ::31] = 1
    ro, rl = oracle_ref(w, row_mask=mask)
    assert_parity(out, lse, ro, rl, mask=mask)


def test_prefill_batch_width_graph_invariance_bitwise():
    kv = [700, 1200, 1111, 190]
    w = workloads.random_case(4, 96, 32, 8, 128, kv, seed=31, mode="prefill", extra_pages=10)
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)
    wide = workloads.select_rows(w, range(4), W=w.W + 37)
    o2, l2 = run_gpu(wide)
    assert bitwise_equal(out, o2) and bitwise_equal(lse, l2)
    for b in range(4):
        one = workloads.select_rows(w, [b])
        o3, l3 = run_gpu(one)
        assert bitwise_equal(out[b:b + 1], o3) and bitwise_equal(lse[b:b + 1], l3), b
    rev = workloads.select_rows(w, [3, 2, 1, 0])
    o4, l4 = run_gpu(rev)
    assert bitwise_equal(out.flip(0), o4) and bitwise_equal(lse.flip(0), l4)
    perm = workloads.permute_pages(w, seed=8)
    o5, l5 = run_gpu(perm)
    assert bitwise_equal(out, o5) and bitwise_equal(lse, l5)
    d = to_dev(w)
    p = binding.plan(4, 96, 32, 8, 128, 16, w.num_pages, w.W)
    go = torch.empty_like(d["q"])
    gl = torch.empty((4, 32, 96), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        binding.attn_prefill(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                             d["position_ids"], go, gl, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.attn_prefill(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                             d["position_ids"], go, gl)
    go.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert bitwise_equal(out, go) and bitwise_equal(lse, gl)


def test_prefill_device_status_on_corrupt_metadata():
    w = workloads.random_case(2, 8, 32, 8, 128, [60, 90], seed=37, mode="prefill")
    good_out, good_lse = run_gpu(w)
    d = to_dev(w)
    d["block_table"][1, 2] = -7
    p = binding.plan(2, 8, 32, 8, 128, 16, w.num_pages, w.W)
    out = torch.empty_like(d["q"])
    lse = torch.empty((2, 32, 8), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.attn_prefill(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                         d["position_ids"], out, lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == binding.STATUS_PAGE_OOB
    assert torch.all(out[1] == 0) and torch.all(torch.isnan(lse[1]))
    assert bitwise_equal(out[0], good_out[0]) and bitwise_equal(lse[0], good_lse[0])


def test_prefill_deterministic_repeat():
    w = workloads.prefill_chunk()
    a = run_gpu(w, validate=False)
    b = run_gpu(w, validate=False)
    assert bitwise_equal(a[0], b[0]) and bitwise_equal(a[1], b[1])


def test_prefill_range_guard_flags_instead_of_overflowing():
    """A pre-RoPE key element of 40000 (beyond the FP16 score-operand range once
    rotated): that (row, KV head)'s rows are zeroed with NaN LSE and the status
    bit is set; every other output still matches the oracle."""
    w = workloads.random_case(2, 8, 32, 8, 128, [60, 90], seed=41, mode="prefill")
    page = int(w.block_table[1, 0])
    w.k_cache[page, 3, 0, 5] = 40000.0
    d = to_dev(w)
    p = binding.plan(2, 8, 32, 8, 128, 16, w.num_pages, w.W)
    out = torch.empty_like(d["q"])
    lse = torch.empty((2, 32, 8), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.attn_prefill(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                         d["position_ids"], out, lse, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == binding.STATUS_RANGE
    assert torch.all(out[1, 0:4] == 0) and torch.all(torch.isnan(lse[1, 0:4]))
    ro, rl = oracle_ref(w)
    keep = np.ones((2, 32), bool)
    keep[1, 0:4] = False
    o = out.float().cpu().numpy()[keep]
    l_ = lse.cpu().numpy()[keep]
    assert np.max(np.abs(o - ro[keep])) <= 2e-2 and np.max(np.abs(l_ - rl[keep])) <= 1e-3
