"""Pins for the float64 oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or mathematics fix:
closed forms, special cases, invariants, a complex-number statement of the
rotation, and dense brute force on tiny inputs.  A plausible slip anywhere in
the oracle (a wrong pairing or sign in rotate-half, a dropped factor in the
frequencies, an off-by-one in the causal mask, a wrong GQA head mapping, a
transposed cache index, a wrong bf16 decode, a wrong log base) fails at least
one of them.
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
from deterministic_paged_kv_gb300 import workloads

D = 128
THETA = 1e6


def unit(i, d=D):
    e = np.zeros(d)
    e[i] = 1.0
    return e


# ---------------------------------------------------------------- rotation --

def test_rope_unit_vector_closed_form():
    """Rotate-half convention: e_0 at position 1 -> cos(1) e_0 + sin(1) e_64,
    e_64 -> -sin(1) e_0 + cos(1) e_64 (pair 0 has frequency 1)."""
    y = oracle.rope(unit(0), 1.0, THETA)
    want = math.cos(1.0) * unit(0) + math.sin(1.0) * unit(64)
    np.testing.assert_allclose(y, want, atol=1e-15)
    y = oracle.rope(unit(64), 1.0, THETA)
    want = -math.sin(1.0) * unit(0) + math.cos(1.0) * unit(64)
    np.testing.assert_allclose(y, want, atol=1e-15)


def _angular_speeds(theta=THETA, d=D):
    """Angle per position of each pair, measured by rotating unit vectors."""
    w = []
    for i in range(d // 2):
        y = oracle.rope(unit(i, d), 1.0, theta)
        w.append(math.atan2(y[i + d // 2], y[i]))
    return np.array(w)


def test_rope_frequencies_geometric():
    """Frequencies start at 1 and fall by theta^(2/D) per pair (Llama RoPE)."""
    w = _angular_speeds()
    assert w[0] == pytest.approx(1.0, abs=1e-15)
    ratio = w[:-1] / w[1:]
    np.testing.assert_allclose(ratio, THETA ** (2.0 / D), rtol=1e-12)
    # the slowest pair turns by theta^(-(D-2)/D) per position
    assert w[-1] == pytest.approx(THETA ** (-(D - 2) / D), rel=1e-12)


def test_rope_equals_complex_multiplication():
    """Pair i as the complex number x_i + i x_{i+64}, turned by p * w_i."""
    rng = np.random.default_rng(0)
    w = _angular_speeds()
    for p in [0.0, 1.0, 7.0, 1536.0, 32768.0]:
        x = rng.standard_normal(D)
        z = (x[:64] + 1j * x[64:]) * np.exp(1j * p * w)
        want = np.concatenate([z.real, z.imag])
        np.testing.assert_allclose(oracle.rope(x, p, THETA), want, atol=1e-9)


def test_rope_norm_identity_and_composition():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(D)
    np.testing.assert_array_equal(oracle.rope(x, 0.0, THETA), x)
    for p in [1.0, 123.0, 8191.0, 32768.0]:
        assert np.linalg.norm(oracle.rope(x, p, THETA)) == pytest.approx(
            np.linalg.norm(x), rel=1e-13)
    a, b = 37.0, 1500.0
    np.testing.assert_allclose(oracle.rope(oracle.rope(x, a, THETA), b, THETA),
                               oracle.rope(x, a + b, THETA), atol=1e-10)


def test_rope_scale_divides_position():
    rng = np.random.default_rng(2)
    x = rng.standard_normal(D)
    np.testing.assert_allclose(oracle.rope(x, 200.0, THETA, rope_scale=4.0),
                               oracle.rope(x, 50.0, THETA), atol=1e-12)


def test_rope_relative_dot_product():
    """(R(p) q).(R(t) k) depends only on t - p."""
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    base = oracle.rope(q, 10.0).dot(oracle.rope(k, 3.0))
    for c in [1.0, 100.0, 4000.0]:
        assert oracle.rope(q, 10.0 + c).dot(oracle.rope(k, 3.0 + c)) == pytest.approx(
            base, abs=1e-9)


# ------------------------------------------------------------- page walk --

def test_materialize_reads_page_slot_head():
    """An encoded cache: value = page*1000 + slot*10 + head (+ d/1000)."""
    NP, P, Hkv, d = 7, 16, 3, 4
    cache = np.zeros((NP, P, Hkv, d))
    for p in range(NP):
        for s in range(P):
            for h in range(Hkv):
                cache[p, s, h] = p * 1000 + s * 10 + h + np.arange(d) / 1000.0
    bt = np.array([[5, 2, 6, -1], [0, 3, -1, -1]], dtype=np.int32)
    kv = np.array([40, 17], dtype=np.int32)
    for b in range(2):
        m = oracle.materialize_row(cache, bt, kv, b)
        assert m.shape == (Hkv, kv[b], d)
        for t in range(kv[b]):
            page, slot = bt[b, t // 16], t % 16
            for h in range(Hkv):
                assert m[h, t, 0] == page * 1000 + slot * 10 + h
                assert m[h, t, 3] == pytest.approx(page * 1000 + slot * 10 + h + 0.003)


# ------------------------------------------------------- brute force -----

def _brute(q, kc, vc, bt, kv, pos, theta=THETA, scale=1.0, sm=None):
    """Dense attention written independently: contiguous K/V by concatenating
    whole pages, rotation by complex multiplication with speeds measured from
    the oracle's rotation of unit vectors, scipy softmax / logsumexp."""
    B, Hq, Sq, d = q.shape
    Hkv = kc.shape[2]
    G = Hq // Hkv
    sm = 1.0 / math.sqrt(d) if sm is None else sm
    w = _angular_speeds(theta, d) / scale
    half = d // 2

    def rot(x, p):
        z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * np.multiply.outer(p, w))
        return np.concatenate([z.real, z.imag], axis=-1)

    out = np.zeros((B, Hq, Sq, d))
    lse = np.zeros((B, Hq, Sq))
    for b in range(B):
        n = int(kv[b])
        npg = (n + 15) // 16
        K = np.concatenate([kc[bt[b, j]] for j in range(npg)], axis=0)[:n] if n else np.zeros((0, Hkv, d))
        V = np.concatenate([vc[bt[b, j]] for j in range(npg)], axis=0)[:n] if n else np.zeros((0, Hkv, d))
        Kr = rot(np.transpose(K, (1, 0, 2)), np.arange(n, dtype=np.float64)[None, :])
        for h in range(Hq):
            kh = h // G
            for s in range(Sq):
                p = int(pos[b, s])
                nv = max(0, min(n, p + 1))
                if nv == 0:
                    out[b, h, s] = 0.0
                    lse[b, h, s] = -np.inf
                    continue
                qr = rot(q[b, h, s], np.float64(p))
                sc = Kr[kh, :nv] @ qr * sm
                lse[b, h, s] = scipy.special.logsumexp(sc)
                out[b, h, s] = scipy.special.softmax(sc) @ V[:nv, kh]
    return out, lse


@pytest.mark.parametrize("d,Hq,Hkv", [(8, 4, 2), (128, 4, 2), (128, 4, 4), (16, 8, 1)])
def test_oracle_vs_dense_brute_force(d, Hq, Hkv):
    rng = np.random.default_rng(d + Hq + Hkv)
    B, Sq = 2, 3
    kv = np.array([40, 23], dtype=np.int32)
    NP = 6
    kc = rng.standard_normal((NP, 16, Hkv, d))
    vc = rng.standard_normal((NP, 16, Hkv, d))
    bt = np.array([[4, 0, 2], [5, 1, -1]], dtype=np.int32)
    q = rng.standard_normal((B, Hq, Sq, d))
    pos = np.array([[37, 38, 39], [20, 21, 22]], dtype=np.int32)
    o1, l1 = oracle.attention(q, kc, vc, bt, kv, pos)
    o2, l2 = _brute(q, kc, vc, bt, kv, pos)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_oracle_vs_relative_rotation():
    """Rotate only K, by (t - p): q.(R(t-p) k) equals (R(p) q).(R(t) k)."""
    rng = np.random.default_rng(11)
    Hq = Hkv = 1
    kc = rng.standard_normal((3, 16, Hkv, D))
    vc = rng.standard_normal((3, 16, Hkv, D))
    bt = np.array([[2, 0, 1]], dtype=np.int32)
    kv = np.array([45], dtype=np.int32)
    q = rng.standard_normal((1, Hq, 1, D))
    pos = np.array([[45]], dtype=np.int32)
    o1, l1 = oracle.attention(q, kc, vc, bt, kv, pos)
    K = np.concatenate([kc[2], kc[0], kc[1]])[:45, 0]
    V = np.concatenate([vc[2], vc[0], vc[1]])[:45, 0]
    sc = np.array([q[0, 0, 0].dot(oracle.rope(K[t], float(t - 45))) for t in range(45)])
    sc /= math.sqrt(D)
    assert l1[0, 0, 0] == pytest.approx(scipy.special.logsumexp(sc), abs=1e-11)
    np.testing.assert_allclose(o1[0, 0, 0], scipy.special.softmax(sc) @ V, atol=1e-12)


# ----------------------------------------------------- special cases -----

def _one_row(n, q=None, seed=5, Hq=2, Hkv=1, p=None):
    rng = np.random.default_rng(seed)
    npg = (n + 15) // 16
    kc = rng.standard_normal((npg + 1, 16, Hkv, D))
    vc = rng.standard_normal((npg + 1, 16, Hkv, D))
    bt = np.array([list(range(1, npg + 1))], dtype=np.int32)
    kv = np.array([n], dtype=np.int32)
    if q is None:
        q = rng.standard_normal((1, Hq, 1, D))
    pos = np.array([[n if p is None else p]], dtype=np.int32)
    return q, kc, vc, bt, kv, pos


def test_zero_query_gives_mean_and_log_n():
    n = 37
    q, kc, vc, bt, kv, pos = _one_row(n, q=np.zeros((1, 2, 1, D)))
    out, lse = oracle.attention(q, kc, vc, bt, kv, pos)
    V = np.concatenate([vc[j] for j in range(1, 4)])[:n, 0]
    np.testing.assert_allclose(lse[0, :, 0], math.log(n), atol=1e-14)
    np.testing.assert_allclose(out[0, 0, 0], V.mean(axis=0), atol=1e-14)


def test_single_key_closed_form():
    """kv_len 1, q = a e_0 at position p, k = b e_0 at position 0:
    score = a b cos(p) / sqrt(D); out = V[0]."""
    a, b, p = 3.0, -2.5, 5
    q = np.zeros((1, 1, 1, D))
    q[0, 0, 0, 0] = a
    kc = np.zeros((2, 16, 1, D))
    kc[1, 0, 0, 0] = b
    vc = np.random.default_rng(9).standard_normal((2, 16, 1, D))
    bt = np.array([[1]], dtype=np.int32)
    out, lse = oracle.attention(q, kc, vc, bt, np.array([1], np.int32),
                                np.array([[p]], np.int32))
    assert lse[0, 0, 0] == pytest.approx(a * b * math.cos(p) / math.sqrt(D), abs=1e-14)
    np.testing.assert_array_equal(out[0, 0, 0], vc[1, 0, 0])


def test_identical_keys_uniform_softmax():
    n = 50
    rng = np.random.default_rng(13)
    k0 = rng.standard_normal(D)
    kc = np.zeros((5, 16, 1, D))
    # the same key *after* rotation: store R(-t) k0 at token t
    bt = np.array([[3, 1, 4, 0]], dtype=np.int32)
    for t in range(n):
        kc[bt[0, t // 16], t % 16, 0] = oracle.rope(k0, -float(t))
    vc = rng.standard_normal((5, 16, 1, D))
    q = rng.standard_normal((1, 1, 1, D))
    p = n
    out, lse = oracle.attention(q, kc, vc, bt, np.array([n], np.int32),
                                np.array([[p]], np.int32))
    s = oracle.rope(q[0, 0, 0], float(p)).dot(k0) / math.sqrt(D)
    assert lse[0, 0, 0] == pytest.approx(s + math.log(n), abs=1e-10)
    V = np.concatenate([vc[j] for j in bt[0]])[:n, 0]
    np.testing.assert_allclose(out[0, 0, 0], V.mean(axis=0), atol=1e-12)


def test_empty_row():
    q, kc, vc, bt, kv, pos = _one_row(16)
    kv = np.array([0], dtype=np.int32)
    pos = np.array([[0]], dtype=np.int32)
    out, lse = oracle.attention(q, kc, vc, bt, kv, pos)
    assert np.all(out == 0.0)
    assert np.all(np.isneginf(lse))


def test_gqa_head_mapping_matches_repeated_mha():
    """Query head h reads KV head h // G: equal to MHA on repeated KV heads."""
    rng = np.random.default_rng(17)
    Hq, Hkv = 8, 2
    G = Hq // Hkv
    kc = rng.standard_normal((4, 16, Hkv, D))
    vc = rng.standard_normal((4, 16, Hkv, D))
    bt = np.array([[2, 0, 3]], dtype=np.int32)
    kv = np.array([41], dtype=np.int32)
    q = rng.standard_normal((1, Hq, 2, D))
    pos = np.array([[39, 40]], dtype=np.int32)
    o1, l1 = oracle.attention(q, kc, vc, bt, kv, pos)
    kr = np.repeat(kc, G, axis=2)
    vr = np.repeat(vc, G, axis=2)
    o2, l2 = oracle.attention(q, kr, vr, bt, kv, pos)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # and not h % Hkv: heads 1 and 4 must differ in general
    assert not np.allclose(l1[0, 1], l1[0, 4])


def test_causal_prefill_query_equals_decode_at_same_position():
    """A chunk query at position p sees exactly keys 0..p."""
    w = workloads.random_case(1, 5, 4, 2, D, [53], seed=21, mode="prefill")
    o, l = oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids)
    for s in range(5):
        p = int(w.position_ids[0, s])
        od, ld = oracle.attention(w.q[:, :, s:s + 1], w.k_cache, w.v_cache, w.block_table,
                                  np.array([p + 1], np.int32), np.array([[p]], np.int32))
        np.testing.assert_array_equal(o[0, :, s], od[0, :, 0])
        np.testing.assert_array_equal(l[0, :, s], ld[0, :, 0])
    # the last visible key matters: dropping it changes the result
    p = int(w.position_ids[0, 2])
    od, ld = oracle.attention(w.q[:, :, 2:3], w.k_cache, w.v_cache, w.block_table,
                              np.array([p], np.int32), np.array([[p]], np.int32))
    assert not np.allclose(ld[0, :, 0], l[0, :, 2])


def test_page_permutation_bitwise():
    w = workloads.random_case(3, 2, 4, 2, D, [70, 33, 16], seed=31, mode="prefill", extra_pages=6)
    w2 = workloads.permute_pages(w, seed=5)
    o1, l1 = oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids)
    o2, l2 = oracle.attention(w2.q, w2.k_cache, w2.v_cache, w2.block_table, w2.kv_lens,
                              w2.position_ids)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_bf16_bits_decode_exactly():
    """bf16 inputs (raw bits) give the same result as their float64 values."""
    import torch
    w = workloads.random_case(2, 1, 4, 2, D, [19, 40], seed=41, mode="decode")
    o1, l1 = oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids)
    f = lambda t: t.to(torch.float64).numpy()
    o2, l2 = oracle.attention(f(w.q), f(w.k_cache), f(w.v_cache), w.block_table, w.kv_lens,
                              w.position_ids)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    # and the bf16 decode of a known pattern: 0x3F80 is 1.0, 0xC040 is -3.0
    bits = np.zeros((1, 16, 1, D), dtype=np.uint16)
    bits[0, 0, 0, 0] = 0x3F80
    vb = np.zeros((1, 16, 1, D), dtype=np.uint16)
    vb[0, 0, 0, 5] = 0xC040
    qb = np.zeros((1, 1, 1, D), dtype=np.uint16)
    out, lse = oracle.attention(qb, bits, vb, np.array([[0]], np.int32), np.array([1], np.int32),
                                np.array([[0]], np.int32))
    assert out[0, 0, 0, 5] == -3.0
    assert lse[0, 0, 0] == 0.0


def test_row_mask_computes_only_marked_queries():
    w = workloads.random_case(1, 6, 4, 2, D, [60], seed=51, mode="prefill")
    o, l = oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids)
    mask = np.array([[1, 0, 0, 1, 0, 1]], dtype=np.uint8)
    om, lm = oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens,
                              w.position_ids, row_mask=mask)
    for s in range(6):
        if mask[0, s]:
            np.testing.assert_array_equal(om[0, :, s], o[0, :, s])
        else:
            assert np.all(np.isnan(lm[0, :, s]))
