"""GPU tests of rk_paged_kv_append: bit-exact against a plain indexing
reference of the page walk, the decode-step and prefill-chunk shapes, an
append followed by attention against the oracle, and the status word."""
import pytest
import torch

from deterministic_paged_kv_gb300 import binding, workloads
from helpers import assert_parity, bitwise_equal, oracle_ref, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from deterministic_paged_kv_gb300 import build
    build.build()
    binding.load()


def reference_append(k_cache, v_cache, block_table, kv_lens, k_new, v_new):
    """Plain loop over rows and tokens: position kv_len - n + j of row b goes
    to slot t % 16 of page block_table[b, t // 16]."""
    k, v = k_cache.clone(), v_cache.clone()
    n = k_new.shape[1]
    for b in range(k_new.shape[0]):
        for j in range(n):
            t = int(kv_lens[b]) - n + j
            pg = int(block_table[b, t // 16])
            k[pg, t % 16] = k_new[b, j]
            v[pg, t % 16] = v_new[b, j]
    return k, v


def _case(B, n_new, kv_after, seed, Hkv=8):
    w = workloads.random_case(B, 1, 4 * Hkv, Hkv, 128, kv_after, seed=seed, mode="decode", extra_pages=4)
    g = torch.Generator().manual_seed(seed + 1)
    k_new = torch.randn((B, n_new, Hkv, 128), generator=g).to(torch.bfloat16)
    v_new = torch.randn((B, n_new, Hkv, 128), generator=g).to(torch.bfloat16)
    return w, k_new, v_new


def _append(w, n_new, k_new, v_new, status=None):
    # the append plan is decode-shaped (Sq = 1, query position kv_len); it
    # validates the table against the lengths after the append
    p = binding.plan(w.B, 1, w.Hq, w.Hkv, 128, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                     w.kv_lens[:, None].clone(), w.rope_theta, w.rope_scale)
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    binding.kv_append(p, n_new, k_new.cuda(), v_new.cuda(), w.block_table.cuda(), w.kv_lens.cuda(), kc, vc,
                      status=status)
    torch.cuda.synchronize()
    return kc.cpu(), vc.cpu()


@pytest.mark.parametrize("B,n_new,kv_after", [
    (4, 1, [1, 17, 32, 4096]),          # decode step: one token, at page starts / inside / at ends
    (3, 37, [37, 100, 160]),            # crosses page boundaries, first page partly filled
    (4, 512, [2048, 2048, 2048, 2048]), # the prefill-chunk shape
])
def test_append_bit_exact(B, n_new, kv_after):
    w, k_new, v_new = _case(B, n_new, kv_after, seed=71 + n_new)
    kc, vc = _append(w, n_new, k_new, v_new)
    rk, rv = reference_append(w.k_cache, w.v_cache, w.block_table, w.kv_lens, k_new, v_new)
    assert bitwise_equal(kc, rk) and bitwise_equal(vc, rv)


def test_append_then_attention_matches_oracle():
    """Decode step of a serving loop: append the new token's K/V, then decode
    over the grown cache; and a prefill chunk appended before its attention."""
    w, k_new, v_new = _case(3, 1, [129, 1000, 2048], seed=83)
    kc, vc = _append(w, 1, k_new, v_new)
    w.k_cache, w.v_cache = kc, vc
    out, lse = run_gpu(w)
    ro, rl = oracle_ref(w)
    assert_parity(out, lse, ro, rl)
    wp = workloads.random_case(2, 64, 32, 8, 128, [300, 700], seed=89, mode="prefill")
    g = torch.Generator().manual_seed(90)
    k_new = torch.randn((2, 64, 8, 128), generator=g).to(torch.bfloat16)
    v_new = torch.randn((2, 64, 8, 128), generator=g).to(torch.bfloat16)
    kc, vc = _append(wp, 64, k_new, v_new)
    wp.k_cache, wp.v_cache = kc, vc
    out, lse = run_gpu(wp)
    ro, rl = oracle_ref(wp)
    assert_parity(out, lse, ro, rl)


def test_append_status_on_unsafe_metadata():
    """kv_len shorter than the append, or a target page out of range: that
    row's tokens are not written, the status word says why, other rows land."""
    w, k_new, v_new = _case(3, 20, [40, 60, 80], seed=97)
    p = binding.plan(3, 1, w.Hq, w.Hkv, 128, 16, w.num_pages, w.W)
    bt = w.block_table.clone()
    kl = w.kv_lens.clone()
    kl[0] = 10                      # shorter than n_new
    bt[1, 3] = w.num_pages + 2      # page of positions 48..63 of row 1 (40..59 appended)
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.kv_append(p, 20, k_new.cuda(), v_new.cuda(), bt.cuda(), kl.cuda(), kc, vc, status=st)
    torch.cuda.synchronize()
    s = int(st.item())
    assert s & binding.STATUS_KVLEN and s & binding.STATUS_PAGE_OOB
    kc, vc = kc.cpu(), vc.cpu()
    # row 2 fully written; row 1 written except positions 48..59; row 0 untouched
    ref_k = w.k_cache.clone()
    for j in range(20):
        t = 80 - 20 + j
        ref_k[int(bt[2, t // 16]), t % 16] = k_new[2, j]
        t = 60 - 20 + j
        if t < 48:
            ref_k[int(bt[1, t // 16]), t % 16] = k_new[1, j]
    assert bitwise_equal(kc, ref_k)


def test_append_argument_checks():
    w, k_new, v_new = _case(2, 4, [10, 20], seed=101)
    p = binding.plan(2, 1, w.Hq, w.Hkv, 128, 16, w.num_pages, w.W)
    kc, vc = w.k_cache.cuda(), w.v_cache.cuda()
    with pytest.raises(binding.RkError) as e:
        binding.kv_append(p, -1, k_new.cuda(), v_new.cuda(), w.block_table.cuda(), w.kv_lens.cuda(), kc, vc)
    assert e.value.name == "RK_E_ARG"
    binding.kv_append(p, 0, k_new.cuda(), v_new.cuda(), w.block_table.cuda(), w.kv_lens.cuda(), kc, vc)
    torch.cuda.synchronize()
    assert bitwise_equal(kc.cpu(), w.k_cache)
