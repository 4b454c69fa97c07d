"""GPU tests of rk_paged_attn_prefill_backward: gradients against the float64
oracle's, bitwise determinism and batch invariance, untouched pages, status.

Tolerance (per element, from the arithmetic of the kernels).  The oracle
returns for every gradient element the sum of the absolute values of its
terms (``mag``) and of their dependence on delta = dout . out scaled by
sum |dout * out| (``sens``).  The kernels round P to BF16 for dV (unit
roundoff 2^-8 of ``mag``), take delta from the BF16 forward output (each out
element within 2^-8, so delta within 2^-8 sum |dout * out|: 2^-8 of ``sens``),
round rotated q / k and dS to FP16 (3 x 2^-11 of ``mag``), and recompute
scores from FP16 operands (a relative P error below 2^-9 for these inputs).
The sum stays under 2^-7 (mag + sens); a floor of 2^-16 of the largest
magnitude covers FP32 accumulation on elements whose terms cancel.
"""
import numpy as np
import pytest
import torch

from deterministic_paged_kv_gb300 import binding, workloads
from helpers import bitwise_equal, run_gpu, to_dev

pytestmark = pytest.mark.gpu

REL = 2.0 ** -7
FLOOR = 2.0 ** -16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from deterministic_paged_kv_gb300 import build
    build.build()
    binding.load()


def _dout(w, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(w.q.shape, generator=g).to(torch.bfloat16)


def run_backward(w, dout, status=None, fill=float("nan")):
    """Forward then backward through the C ABI; returns CPU (dq, dk, dv)."""
    d = to_dev(w)
    out, lse = run_gpu(w, mode="prefill")
    p = binding.plan(w.B, w.Sq, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table, w.kv_lens,
                     w.position_ids, w.rope_theta, w.rope_scale)
    dq = torch.full(w.q.shape, fill, dtype=torch.float32, device="cuda")
    dk = torch.full(w.k_cache.shape, fill, dtype=torch.float32, device="cuda")
    dv = torch.full(w.v_cache.shape, fill, dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.prefill_backward_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    binding.attn_prefill_backward(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                                  d["position_ids"], out, lse, dout.cuda(), dq, dk, dv, ws, status=status)
    torch.cuda.synchronize()
    return dq.cpu(), dk.cpu(), dv.cpu()


def oracle_grads(w, dout):
    import oracle
    return oracle.attention_backward(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids,
                                     dout, w.rope_theta, w.rope_scale, magnitudes=True)


def check(name, got, ref, mag, sens=None, sel=None):
    g = got.double().numpy()
    if sens is None:
        sens = np.zeros_like(mag)
    if sel is not None:
        g, ref, mag, sens = g[sel], ref[sel], mag[sel], sens[sel]
    assert np.isfinite(g).all(), name
    err = np.abs(g - ref)
    bound = REL * (mag + sens) + FLOOR * mag.max()
    ratio = float(np.max(err / np.maximum(mag + sens, 1e-30)))
    print("%s: max err %.3e, max err/(mag+sens) %.3e, max |ref| %.3e" % (name, err.max(), ratio, np.abs(ref).max()))
    assert (err <= bound).all(), (name, float(err.max()), float((err - bound).max()))


def referenced_pages(w):
    m = np.zeros(w.num_pages, bool)
    for b in range(w.B):
        for j in range((int(w.kv_lens[b]) + 15) // 16):
            m[int(w.block_table[b, j])] = True
    return m


CASES = {
    "full_prefill_200": dict(B=1, Sq=200, kv=[200], Hq=32, Hkv=8),
    "full_prefill_1000": dict(B=1, Sq=1000, kv=[1000], Hq=32, Hkv=8),
    "full_prefill_2048": dict(B=1, Sq=2048, kv=[2048], Hq=32, Hkv=8),
    "chunks_300_170": dict(B=2, Sq=70, kv=[300, 170], Hq=32, Hkv=8),
    "mha_G1": dict(B=2, Sq=40, kv=[150, 77], Hq=8, Hkv=8),
    "gqa_G8": dict(B=2, Sq=40, kv=[150, 77], Hq=64, Hkv=8),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_parity_with_oracle(case):
    c = CASES[case]
    npg = sum((n + 15) // 16 for n in c["kv"]) + 3
    W = max((n + 15) // 16 for n in c["kv"]) + 2
    w = workloads.build(case, c["B"], c["Sq"], c["Hq"], c["Hkv"], 128, c["kv"], npg, W, 211, "prefill")
    dout = _dout(w, 212)
    dq, dk, dv = run_backward(w, dout)
    rq, rk, rv, (mq, mk, mv, sq, sk) = oracle_grads(w, dout)
    ref = referenced_pages(w)
    check("dq", dq, rq, mq, sq)
    check("dk", dk, rk, mk, sk, ref)
    check("dv", dv, rv, mv, None, ref)
    assert torch.isnan(dk[torch.from_numpy(~ref)]).all() and torch.isnan(dv[torch.from_numpy(~ref)]).all()


def test_backward_bitwise_deterministic_and_batch_invariant():
    kv = [260, 97, 180]
    w = workloads.build("inv", 3, 64, 32, 8, 128, kv, 40, 20, 223, "prefill")
    dout = _dout(w, 224)
    g1 = run_backward(w, dout)
    g2 = run_backward(w, dout, fill=0.0)
    ref = torch.from_numpy(referenced_pages(w))
    assert bitwise_equal(g1[0], g2[0])
    assert bitwise_equal(g1[1][ref], g2[1][ref]) and bitwise_equal(g1[2][ref], g2[2][ref])
    # row 1 alone (same pages, a batch of one) gives the same bits for its gradients
    one = workloads.select_rows(w, [1])
    d1 = dout[1:2].contiguous()
    s = run_backward(one, d1)
    assert bitwise_equal(s[0][0], g1[0][1])
    pages = [int(one.block_table[0, j]) for j in range((kv[1] + 15) // 16)]
    assert bitwise_equal(s[1][pages], g1[1][pages]) and bitwise_equal(s[2][pages], g1[2][pages])


def test_backward_flags_unsafe_page_and_writes_nothing_there():
    w = workloads.build("bad", 2, 16, 32, 8, 128, [64, 40], 12, 6, 227, "prefill")
    dout = _dout(w, 228)
    good = run_backward(w, dout)
    # corrupt row 1's table after the forward: the backward reads a page id out of range
    d = to_dev(w)
    out, lse = run_gpu(w, mode="prefill")
    p = binding.plan(w.B, w.Sq, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W)
    bt = d["block_table"].clone()
    bt[1, 1] = w.num_pages + 5
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq = torch.full(w.q.shape, float("nan"), dtype=torch.float32, device="cuda")
    dk = torch.full(w.k_cache.shape, float("nan"), dtype=torch.float32, device="cuda")
    dv = torch.full(w.v_cache.shape, float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.prefill_backward_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    binding.attn_prefill_backward(p, d["q"], d["k_cache"], d["v_cache"], bt, d["kv_lens"], d["position_ids"],
                                  out, lse, dout.cuda(), dq, dk, dv, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & binding.STATUS_PAGE_OOB
    # row 0 is untouched by the bad entry: its gradients are the usual bits
    assert bitwise_equal(dq[0].cpu(), good[0][0])
    p0 = [int(w.block_table[0, j]) for j in range(4)]
    assert bitwise_equal(dk.cpu()[p0], good[1][p0]) and bitwise_equal(dv.cpu()[p0], good[2][p0])


def test_backward_range_flag_gives_nan():
    w = workloads.build("rng", 1, 32, 32, 8, 128, [80], 8, 6, 229, "prefill")
    w.q[0, 3, 5, 7] = 40000.0  # pre-RoPE q element beyond 2^15: not representable once rotated in FP16
    dout = _dout(w, 230)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq, dk, dv = run_backward(w, dout, status=st)
    assert int(st.item()) & binding.STATUS_RANGE
    assert torch.isnan(dq[0, 3, 5]).all()


def test_backward_graph_replay_with_new_contents():
    """Captured once, replayed with new q / dout / cache contents of the same
    shape: the same bits as an eager call on those contents."""
    w = workloads.build("graph", 2, 48, 32, 8, 128, [200, 120], 24, 16, 241, "prefill")
    p = binding.plan(w.B, w.Sq, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W)
    d = to_dev(w)
    out, lse = run_gpu(w, mode="prefill")
    dout = _dout(w, 242).cuda()
    dq = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    dk = torch.zeros(w.k_cache.shape, dtype=torch.float32, device="cuda")
    dv = torch.zeros(w.v_cache.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(binding.prefill_backward_workspace_bytes(p), dtype=torch.uint8, device="cuda")
    call = lambda: binding.attn_prefill_backward(p, d["q"], d["k_cache"], d["v_cache"], d["block_table"],
                                                 d["kv_lens"], d["position_ids"], out, lse, dout, dq, dk, dv, ws)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    # new contents: another seed's q / caches / dout and their forward
    w2 = workloads.build("graph2", 2, 48, 32, 8, 128, [200, 120], 24, 16, 243, "prefill")
    w2.block_table, w2.position_ids, w2.kv_lens = w.block_table, w.position_ids, w.kv_lens
    ref = run_backward(w2, _dout(w2, 244), fill=0.0)
    o2, l2 = run_gpu(w2, mode="prefill")
    d["q"].copy_(w2.q.cuda())
    d["k_cache"].copy_(w2.k_cache.cuda())
    d["v_cache"].copy_(w2.v_cache.cuda())
    out.copy_(o2)
    lse.copy_(l2)
    dout.copy_(_dout(w2, 244).cuda())
    g.replay()
    torch.cuda.synchronize()
    pages = torch.from_numpy(referenced_pages(w))
    assert bitwise_equal(dq.cpu(), ref[0])
    assert bitwise_equal(dk.cpu()[pages], ref[1][pages]) and bitwise_equal(dv.cpu()[pages], ref[2][pages])
