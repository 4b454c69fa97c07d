"""rk_paged_attn_decode_split_static (split decode with the library's static
device scratch, no allocation) against rk_paged_attn_decode_split with a
caller buffer, over two calls in a row; oversize inputs are rejected.  Named to
run last, and independent of any earlier test's state."""
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


def _run_both(w, split, d, p, scratch):
    args = (d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"], d["position_ids"])
    o_ref = torch.empty_like(d["q"])
    l_ref = torch.empty((w.B, w.Hq, 1), dtype=torch.float32, device="cuda")
    binding.attn_decode_split(p, split, *args, o_ref, l_ref, scratch)
    o_st = torch.full_like(d["q"], float("nan"))
    l_st = torch.full((w.B, w.Hq, 1), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.attn_decode_split_static(p, split, *args, o_st, l_st, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o_ref, l_ref, o_st, l_st


def test_static_scratch_matches_caller_scratch_two_calls_in_a_row():
    for call, (kv, split, seed) in enumerate((([3000, 1100, 5003, 700], 1024, 61),
                                             ([2048, 9000, 1], 2048, 67),
                                             ([300, 77, 1000], 528, 71),
                                             ([300, 41], 16, 73))):
        w = workloads.random_case(len(kv), 1, 32, 8, 128, kv, seed=seed, mode="decode")
        d = to_dev(w)
        p = binding.plan(w.B, 1, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                         w.position_ids, w.rope_theta, w.rope_scale)
        need = binding.decode_split_scratch_bytes(p, split)
        assert need <= binding.SPLIT_STATIC_SCRATCH_BYTES
        scratch = torch.empty(need, dtype=torch.uint8, device="cuda")
        o_ref, l_ref, o_st, l_st = _run_both(w, split, d, p, scratch)
        assert bitwise_equal(o_ref, o_st) and bitwise_equal(l_ref, l_st), call
        ro, rl = oracle_ref(w)
        assert_parity(o_st, l_st, ro, rl)


def test_static_scratch_rejects_oversize_inputs():
    """A plan whose partials exceed the static array is refused before launch."""
    B, W = 64, 4096  # 64 * 32 * 64 splits of 1024 tokens * 129 * 4 bytes > 16 MiB
    p = binding.plan(B, 1, 32, 8, 128, 16, 8, W)
    assert binding.decode_split_scratch_bytes(p, 1024) > binding.SPLIT_STATIC_SCRATCH_BYTES
    q = torch.zeros((B, 32, 1, 128), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((8, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.full((B, W), -1, dtype=torch.int32, device="cuda")
    kv = torch.zeros(B, dtype=torch.int32, device="cuda")
    pos = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((B, 32, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.RkError) as e:
        binding.attn_decode_split_static(p, 1024, q, cache, cache, bt, kv, pos, out, lse)
    assert e.value.name == "RK_E_ARG"
