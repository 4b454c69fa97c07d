"""Pins for the oracle's attention gradient (``oracle.attention_backward``),
independent of its code.

The gradient of L = sum(dout * out) is checked against central finite
differences of the (separately pinned) float64 forward, against reverse-mode
autodiff of a dense attention written here in torch, and against closed forms
that hold for the exact gradient: the keys' dv sum to the queries' dout, the
rotated-domain dk sums to zero, a single visible key passes dout straight to
dv and nothing to q or k, and a zero dout gives zero gradients.  A slip in the
softmax derivative (a missing Dq = dout . out term, a wrong sign), in the
scale, in the inverse rotation, in the GQA accumulation or in the page
scatter fails at least one of them.

The tolerance inputs the GPU tests take from the oracle are pinned too: the
term magnitudes must equal |value| on inputs where every term of an element
has one sign, and the delta sensitivities must equal the autograd derivatives
of a torch statement of the gradient (itself pinned to dense autodiff) and
bound the change that a relative 2^-8 perturbation of out makes.  A doubled,
dropped or mis-weighted term in any magnitude or sensitivity fails one of
them.
"""
import math

import numpy as np
import pytest
import torch

import oracle

THETA = 1e6


def _case(seed, D=16, Hq=4, Hkv=2, kv=(37, 20), Sq=3, NP=6, conv=(0, 1)):
    """Two rows on shuffled pages; row b's queries at the trailing positions
    (conv 0: last position kv_len - 1, conv 1: kv_len)."""
    rng = np.random.default_rng(seed)
    B = len(kv)
    kc = rng.standard_normal((NP, 16, Hkv, D))
    vc = rng.standard_normal((NP, 16, Hkv, D))
    perm = rng.permutation(NP)
    W = max((n + 15) // 16 for n in kv)
    bt = np.full((B, W), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(kv):
        for j in range((n + 15) // 16):
            bt[b, j] = perm[k]
            k += 1
    q = rng.standard_normal((B, Hq, Sq, D))
    pos = np.array([[n - Sq + s + conv[b] for s in range(Sq)] for b, n in enumerate(kv)], dtype=np.int32)
    dout = rng.standard_normal((B, Hq, Sq, D))
    return q, kc, vc, bt, np.array(kv, dtype=np.int32), pos, dout


def _loss(q, kc, vc, bt, kv, pos, dout):
    out, _ = oracle.attention(q, kc, vc, bt, kv, pos)
    return float(np.sum(out * dout))


def _referenced(bt, kv, NP):
    """Mask [NP] of pages some row references."""
    m = np.zeros(NP, bool)
    for b, n in enumerate(kv):
        for j in range((int(n) + 15) // 16):
            m[bt[b, j]] = True
    return m


def test_backward_matches_central_differences():
    q, kc, vc, bt, kv, pos, dout = _case(1)
    dq, dk, dv = oracle.attention_backward(q, kc, vc, bt, kv, pos, dout)
    h = 1e-5
    rng = np.random.default_rng(2)
    ref = _referenced(bt, kv, kc.shape[0])
    # every element of dq; a random sample of the referenced cache entries
    for idx in np.ndindex(q.shape):
        e = np.zeros_like(q)
        e[idx] = h
        fd = (_loss(q + e, kc, vc, bt, kv, pos, dout) - _loss(q - e, kc, vc, bt, kv, pos, dout)) / (2 * h)
        assert abs(fd - dq[idx]) <= 1e-6 * (1 + abs(fd)), idx
    pages = np.nonzero(ref)[0]
    for _ in range(120):
        pg = int(rng.choice(pages))
        idx = (pg, int(rng.integers(16)), int(rng.integers(kc.shape[2])), int(rng.integers(kc.shape[3])))
        for cache, grad, name in ((kc, dk, "k"), (vc, dv, "v")):
            e = np.zeros_like(cache)
            e[idx] = h
            args_p = (q, cache + e, vc, bt, kv, pos, dout) if name == "k" else (q, kc, cache + e, bt, kv, pos, dout)
            args_m = (q, cache - e, vc, bt, kv, pos, dout) if name == "k" else (q, kc, cache - e, bt, kv, pos, dout)
            fd = (_loss(*args_p) - _loss(*args_m)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * (1 + abs(fd)), (name, idx)
    # pages no row references are left untouched (NaN)
    assert np.isnan(dk[~ref]).all() and np.isnan(dv[~ref]).all()
    assert np.isfinite(dk[ref]).all() and np.isfinite(dv[ref]).all()


def _torch_dense(q, K, V, kv, pos, Hkv, theta=THETA):
    """Dense causal attention with rotate-half RoPE written with torch ops
    (cos / sin tables, contiguous K/V [B, Hkv, T, D]); autodiff target."""
    B, Hq, Sq, D = q.shape
    G = Hq // Hkv
    half = D // 2
    inv = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / D)

    def rot(x, p):  # x [..., D], p broadcastable positions
        a = p[..., None] * inv
        c, s = torch.cos(a), torch.sin(a)
        lo, hi = x[..., :half], x[..., half:]
        return torch.cat([lo * c - hi * s, hi * c + lo * s], dim=-1)

    outs = []
    for b in range(B):
        n = int(kv[b])
        t = torch.arange(n, dtype=torch.float64)
        Kr = rot(K[b, :, :n], t)  # [Hkv, n, D]
        qp = torch.as_tensor(pos[b], dtype=torch.float64)
        Qr = rot(q[b], qp[None, :])  # [Hq, Sq, D]
        sc = torch.einsum("hsd,htd->hst", Qr, Kr.repeat_interleave(G, dim=0)) / math.sqrt(D)
        vis = torch.arange(n)[None, :] <= torch.as_tensor(pos[b])[:, None]
        sc = sc.masked_fill(~vis[None], float("-inf"))
        outs.append(torch.softmax(sc, dim=-1) @ V[b, :, :n].repeat_interleave(G, dim=0))
    return torch.stack(outs)


def test_backward_matches_dense_autodiff_with_gqa():
    q, kc, vc, bt, kv, pos, dout = _case(3, D=16, Hq=8, Hkv=2, kv=(50, 33), Sq=5, NP=8)
    dq, dk, dv = oracle.attention_backward(q, kc, vc, bt, kv, pos, dout)
    B, Hq, Sq, D = q.shape
    Hkv, T = kc.shape[2], max(kv)
    # contiguous K / V gathered through the table, with their page slots
    K = np.zeros((B, Hkv, T, D))
    V = np.zeros((B, Hkv, T, D))
    for b in range(B):
        for t in range(kv[b]):
            K[b, :, t] = kc[bt[b, t // 16], t % 16]
            V[b, :, t] = vc[bt[b, t // 16], t % 16]
    qt = torch.tensor(q, requires_grad=True)
    Kt = torch.tensor(K, requires_grad=True)
    Vt = torch.tensor(V, requires_grad=True)
    out = _torch_dense(qt, Kt, Vt, kv, pos, Hkv)
    (out * torch.tensor(dout)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-11)
    for b in range(B):
        for t in range(kv[b]):
            np.testing.assert_allclose(dk[bt[b, t // 16], t % 16], Kt.grad[b, :, t].numpy(), atol=1e-11)
            np.testing.assert_allclose(dv[bt[b, t // 16], t % 16], Vt.grad[b, :, t].numpy(), atol=1e-11)
        last = bt[b, (kv[b] - 1) // 16]
        assert (dk[last, (kv[b] - 1) % 16 + 1:] == 0).all()  # slots past kv_len


def test_dv_sums_to_dout_and_rotated_dk_sums_to_zero():
    """sum_t P_t = 1 gives sum over keys of dv = sum over the group's queries
    of dout; sum_t dS_t = 0 gives sum over keys of R(t) dk_t = 0."""
    q, kc, vc, bt, kv, pos, dout = _case(5, D=128, Hq=4, Hkv=2, kv=(45, 30), Sq=4, NP=6)
    dq, dk, dv = oracle.attention_backward(q, kc, vc, bt, kv, pos, dout)
    Hkv, G = kc.shape[2], q.shape[1] // kc.shape[2]
    for b, n in enumerate(kv):
        for kh in range(Hkv):
            sv = sum(dv[bt[b, t // 16], t % 16, kh] for t in range(n))
            sd = dout[b, kh * G:(kh + 1) * G].sum(axis=(0, 1))
            np.testing.assert_allclose(sv, sd, atol=1e-11)
            sk = sum(oracle.rope(dk[bt[b, t // 16], t % 16, kh], float(t)) for t in range(n))
            np.testing.assert_allclose(sk, 0.0, atol=1e-10)


def test_single_key_and_zero_dout():
    rng = np.random.default_rng(7)
    D, Hq, Hkv = 128, 2, 1
    kc = rng.standard_normal((2, 16, Hkv, D))
    vc = rng.standard_normal((2, 16, Hkv, D))
    bt = np.array([[1]], dtype=np.int32)
    kv = np.array([1], dtype=np.int32)
    q = rng.standard_normal((1, Hq, 1, D))
    pos = np.array([[0]], dtype=np.int32)
    dout = rng.standard_normal((1, Hq, 1, D))
    dq, dk, dv = oracle.attention_backward(q, kc, vc, bt, kv, pos, dout)
    # out = v_0 whatever q and k are: dv_0 = sum of the heads' dout, no q / k gradient
    np.testing.assert_allclose(dv[1, 0, 0], dout[0, :, 0].sum(axis=0), atol=1e-14)
    assert np.abs(dq).max() == 0.0 and np.abs(dk[1]).max() == 0.0
    assert (dv[1, 1:] == 0).all()
    z = oracle.attention_backward(q, kc, vc, bt, kv, pos, np.zeros_like(dout))
    assert all(np.nan_to_num(g).max() == 0.0 and np.nan_to_num(g).min() == 0.0 for g in z)


def test_magnitudes_bound_the_values():
    q, kc, vc, bt, kv, pos, dout = _case(9, D=128)
    dq, dk, dv, (mq, mk, mv, sq, sk) = oracle.attention_backward(q, kc, vc, bt, kv, pos, dout, magnitudes=True)
    ref = _referenced(bt, kv, kc.shape[0])
    assert (np.abs(dq) <= mq + 1e-12).all()
    assert (np.abs(dk[ref]) <= mk[ref] + 1e-12).all() and (np.abs(dv[ref]) <= mv[ref] + 1e-12).all()
    assert mq.max() > 0 and mk[ref].max() > 0 and mv[ref].max() > 0
    # Dq sensitivity of dq, restated for one query from its definition with numpy:
    # sum over visible keys of sm_scale * P_t * |k'_t| * sum_d |dout_d out_d|, rotation-combined
    b, h, s_ = 1, 3, 2
    G = q.shape[1] // kc.shape[2]
    p = int(pos[b, s_])
    n = min(p + 1, int(kv[b]))
    kr = np.array([oracle.rope(kc[bt[b, t // 16], t % 16, h // G], float(t)) for t in range(n)])
    qr = oracle.rope(q[b, h, s_], float(p))
    sc = kr @ qr / math.sqrt(q.shape[3])
    P = np.exp(sc - sc.max())
    P /= P.sum()
    out = P @ np.array([vc[bt[b, t // 16], t % 16, h // G] for t in range(n)])
    A = np.sum(np.abs(dout[b, h, s_] * out))
    raw = (P[:, None] * np.abs(kr)).sum(axis=0) * A / math.sqrt(q.shape[3])
    half = q.shape[3] // 2
    want = np.concatenate([raw[:half] + raw[half:], raw[:half] + raw[half:]])
    np.testing.assert_allclose(sq[b, h, s_], want, rtol=1e-12)
    assert (sq >= 0).all() and (sk[ref] >= 0).all() and sq.max() > 0


def test_backward_page_permutation_moves_gradients_with_pages():
    q, kc, vc, bt, kv, pos, dout = _case(11, D=32)
    dq, dk, dv = oracle.attention_backward(q, kc, vc, bt, kv, pos, dout)
    NP = kc.shape[0]
    perm = np.random.default_rng(12).permutation(NP)  # new page id of old page i
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    dq2, dk2, dv2 = oracle.attention_backward(q, kc2, vc2, bt2, kv, pos, dout)
    assert np.array_equal(dq, dq2)
    assert np.array_equal(dk2[perm], dk, equal_nan=True) and np.array_equal(dv2[perm], dv, equal_nan=True)


# ---------------------------------------------------------------------------
# The tolerance inputs: term magnitudes (mag_*) and delta sensitivities (sens_*).
#
# The GPU backward is judged per element against 2^-7 (mag + sens), so these
# numbers need pins of their own.  mag is the sum of |terms| of an element;
# when every term of an element has one sign it must equal |value| exactly
# (a doubled or a dropped term fails).  sens is the sum over the element's
# terms of |d term / d Dq| * sum_d |dout_d out_d|, Dq = dout . out of the
# term's query; it is checked against autograd derivatives of a float64 torch
# statement of the gradient in which every (query, key) term takes Dq from its
# own entry of an explicit ``delta`` tensor.  That statement is itself pinned
# to autodiff of the dense forward.
# ---------------------------------------------------------------------------


def _rot_t(x, p, theta=THETA, scale=1.0):
    """Rotate-half RoPE of x [..., D] at positions p (broadcast), float64 torch."""
    D = x.shape[-1]
    half = D // 2
    inv = theta ** (-2.0 * torch.arange(half, dtype=torch.float64) / D)
    a = torch.as_tensor(p, dtype=torch.float64)[..., None] * inv / scale
    c, s = torch.cos(a), torch.sin(a)
    lo, hi = x[..., :half], x[..., half:]
    return torch.cat([lo * c - hi * s, hi * c + lo * s], dim=-1)


def _logical(cache, bt, kv):
    """Logical [B, Hkv, T, D] float64 copy of a paged cache (plain gather)."""
    B, T = len(kv), int(max(kv))
    out = np.zeros((B, cache.shape[2], T, cache.shape[3]))
    for b in range(B):
        for t in range(int(kv[b])):
            out[b, :, t] = cache[bt[b, t // 16], t % 16]
    return out


def _restated_grads(q, K, V, kv, pos, dout, delta, theta=THETA, scale=1.0):
    """Gradient of L = sum(dout * out) with the softmax correction taken from
    ``delta`` [B, Hq, Sq, T] (one entry per query-key term):
    dS = P (dout . v - delta), dq' = s dS K', dk' = s dS^T Q', dv = P^T dout,
    then dq = R(p)^T dq', dk = R(t)^T dk'.  Returns dq, dk, dv [B, Hkv, T, D]
    and the rotated-domain dq', dk'."""
    B, Hq, Sq, D = q.shape
    Hkv, T = K.shape[1], K.shape[2]
    G = Hq // Hkv
    sm = 1.0 / math.sqrt(D)
    dq, dqr, dk, dkr, dv = [], [], [], [], []
    for b in range(B):
        n = int(kv[b])
        t = torch.arange(T, dtype=torch.float64)
        Kr = _rot_t(K[b], t, theta, scale).repeat_interleave(G, dim=0)  # [Hq, T, D]
        Vg = V[b].repeat_interleave(G, dim=0)
        Qr = _rot_t(q[b], torch.as_tensor(pos[b], dtype=torch.float64)[None, :], theta, scale)
        vis = (torch.arange(T)[None, :] <= torch.as_tensor(pos[b])[:, None]) & (torch.arange(T)[None, :] < n)
        sc = torch.einsum("hsd,htd->hst", Qr, Kr) * sm
        P = torch.softmax(sc.masked_fill(~vis[None], float("-inf")), dim=-1)
        dp = torch.einsum("hsd,htd->hst", dout[b], Vg)
        dS = torch.where(vis[None], P * (dp - delta[b]), torch.zeros_like(P))
        gq = sm * torch.einsum("hst,htd->hsd", dS, Kr)
        gk = (sm * torch.einsum("hst,hsd->htd", dS, Qr)).view(Hkv, G, T, D).sum(1)
        gv = torch.einsum("hst,hsd->htd", P, dout[b]).view(Hkv, G, T, D).sum(1)
        dqr.append(gq)
        dkr.append(gk)
        dq.append(_rot_t(gq, -torch.as_tensor(pos[b], dtype=torch.float64)[None, :], theta, scale))
        dk.append(_rot_t(gk, -t, theta, scale))
        dv.append(gv)
    return (torch.stack(dq), torch.stack(dk), torch.stack(dv), torch.stack(dqr), torch.stack(dkr))


def _pair_bound(x):
    """Rotation-pair combination the oracle uses: x[i] + x[i + D/2] in both slots."""
    half = x.shape[-1] // 2
    c = x[..., :half] + x[..., half:]
    return np.concatenate([c, c], axis=-1)


def test_restated_gradient_with_explicit_delta_is_the_gradient():
    q, kc, vc, bt, kv, pos, dout = _case(21, D=16, Hq=4, Hkv=2, kv=(37, 20), Sq=3, NP=6)
    K, V = _logical(kc, bt, kv), _logical(vc, bt, kv)
    out, _ = oracle.attention(q, kc, vc, bt, kv, pos)
    Dq = np.sum(dout * out, axis=-1)
    T = K.shape[2]
    delta = torch.tensor(np.repeat(Dq[..., None], T, axis=-1))
    dq, dk, dv, _, _ = _restated_grads(torch.tensor(q), torch.tensor(K), torch.tensor(V), kv, pos,
                                       torch.tensor(dout), delta)
    # against reverse-mode autodiff of the dense forward
    qt = torch.tensor(q, requires_grad=True)
    Kt = torch.tensor(K, requires_grad=True)
    Vt = torch.tensor(V, requires_grad=True)
    (_torch_dense(qt, Kt, Vt, kv, pos, kc.shape[2]) * torch.tensor(dout)).sum().backward()
    np.testing.assert_allclose(dq.numpy(), qt.grad.numpy(), atol=1e-11)
    for b, n in enumerate(kv):
        np.testing.assert_allclose(dk[b, :, :n].numpy(), Kt.grad[b, :, :n].numpy(), atol=1e-11)
        np.testing.assert_allclose(dv[b, :, :n].numpy(), Vt.grad[b, :, :n].numpy(), atol=1e-11)


def test_delta_sensitivities_are_the_autograd_derivatives():
    q, kc, vc, bt, kv, pos, dout = _case(23, D=16, Hq=4, Hkv=2, kv=(37, 20), Sq=3, NP=6)
    B, Hq, Sq, D = q.shape
    Hkv, G = kc.shape[2], Hq // kc.shape[2]
    K, V = _logical(kc, bt, kv), _logical(vc, bt, kv)
    out, _ = oracle.attention(q, kc, vc, bt, kv, pos)
    Dq = np.sum(dout * out, axis=-1)
    A = np.sum(np.abs(dout * out), axis=-1)  # [B, Hq, Sq]
    T = K.shape[2]
    qt, Kt, Vt, gt = (torch.tensor(x) for x in (q, K, V, dout))
    delta0 = torch.tensor(np.repeat(Dq[..., None], T, axis=-1))

    def f(delta):
        _, _, _, gq, gk = _restated_grads(qt, Kt, Vt, kv, pos, gt, delta)
        return torch.cat([gq.reshape(-1), gk.reshape(-1)])

    J = torch.autograd.functional.jacobian(f, delta0, vectorize=True).numpy()  # [outputs, B*Hq*Sq*T]
    J = J.reshape(J.shape[0], -1)
    w = np.repeat(A[..., None], T, axis=-1).reshape(-1)  # A of each term's query
    sens_rot = np.abs(J) @ w
    nq = B * Hq * Sq * D
    sq_rot = sens_rot[:nq].reshape(B, Hq, Sq, D)
    sk_rot = sens_rot[nq:].reshape(B, Hkv, T, D)

    _, _, _, (_, _, _, sq, sk) = oracle.attention_backward(q, kc, vc, bt, kv, pos, dout, magnitudes=True)
    np.testing.assert_allclose(sq, _pair_bound(sq_rot), rtol=1e-10, atol=1e-14)
    skc = _pair_bound(sk_rot)
    for b, n in enumerate(kv):
        for t in range(n):
            np.testing.assert_allclose(sk[bt[b, t // 16], t % 16], skc[b, :, t], rtol=1e-10, atol=1e-14)
    # the pair combination bounds the sensitivity after the inverse rotation
    def fpre(delta):
        gq, gk, _, _, _ = _restated_grads(qt, Kt, Vt, kv, pos, gt, delta)
        return torch.cat([gq.reshape(-1), gk.reshape(-1)])

    Jp = torch.autograd.functional.jacobian(fpre, delta0, vectorize=True).numpy().reshape(len(sens_rot), -1)
    pre = np.abs(Jp) @ w
    assert (pre[:nq] <= _pair_bound(sq_rot).reshape(-1) * (1 + 1e-12) + 1e-15).all()
    # a relative change of 2^-8 in every element of out (signs taken so that each
    # query's Dq moves by the full 2^-8 A) moves the gradients by at most 2^-8 sens
    eps = 2.0 ** -8 * np.sign(dout * out)
    Dq2 = np.sum(dout * out * (1 + eps), axis=-1)
    delta2 = torch.tensor(np.repeat(Dq2[..., None], T, axis=-1))
    g0 = _restated_grads(qt, Kt, Vt, kv, pos, gt, delta0)
    g1 = _restated_grads(qt, Kt, Vt, kv, pos, gt, delta2)
    dqd = np.abs((g1[0] - g0[0]).numpy())
    assert (dqd <= 2.0 ** -8 * sq * (1 + 1e-9) + 1e-15).all()
    assert dqd.max() > 0.25 * (2.0 ** -8 * sq).max()  # the bound is reached, not vacuous
    dkd = np.abs((g1[1] - g0[1]).numpy())
    for b, n in enumerate(kv):
        for t in range(n):
            assert (dkd[b, :, t] <= 2.0 ** -8 * sk[bt[b, t // 16], t % 16] * (1 + 1e-9) + 1e-15).all()


def test_magnitudes_equal_the_values_when_every_term_has_one_sign():
    """Keys +-u and values +-w with the same signs a_t, queries positive multiples
    of one vector z, dout > 0, and RoPE made the identity (rope_scale 1e14):
    every dq' term has the sign of u, every dk'_t term the sign of a_t z and every
    dv term is positive, so each magnitude equals |value|.  With u and z zero in
    the upper half of the dims, the rotation-pair combination adds nothing for
    the lower half."""
    rng = np.random.default_rng(31)
    D, Hq, Hkv, Sq, NP = 32, 4, 2, 3, 6
    half = D // 2
    kvl = (40, 23)
    B = len(kvl)
    scale = 1e14
    u = np.concatenate([rng.standard_normal(half), np.zeros(half)])
    z = np.concatenate([rng.standard_normal(half), np.zeros(half)])
    wv = np.abs(rng.standard_normal(D)) + 0.1
    perm = rng.permutation(NP)
    W = max((n + 15) // 16 for n in kvl)
    bt = np.full((B, W), -1, dtype=np.int32)
    kc = rng.standard_normal((NP, 16, Hkv, D))  # slots past kv_len stay random
    vc = rng.standard_normal((NP, 16, Hkv, D))
    k = 0
    for b, n in enumerate(kvl):
        for j in range((n + 15) // 16):
            bt[b, j] = perm[k]
            k += 1
        for t in range(n):
            for kh in range(Hkv):
                a = rng.choice([-1.0, 1.0])
                kc[bt[b, t // 16], t % 16, kh] = a * u
                vc[bt[b, t // 16], t % 16, kh] = a * wv
    q = (np.abs(rng.standard_normal((B, Hq, Sq, 1))) + 0.2) * 3.0 * z
    dout = np.abs(rng.standard_normal((B, Hq, Sq, D))) + 0.05
    kv = np.array(kvl, dtype=np.int32)
    pos = np.array([[n - Sq + s for s in range(Sq)] for n in kvl], dtype=np.int32)
    dq, dk, dv, (mq, mk, mv, _, _) = oracle.attention_backward(q, kc, vc, bt, kv, pos, dout,
                                                               rope_scale=scale, magnitudes=True)
    ref = _referenced(bt, kv, NP)
    np.testing.assert_allclose(mv[ref], np.abs(dv[ref]), rtol=1e-12)
    np.testing.assert_allclose(mq[..., :half], np.abs(dq[..., :half]), rtol=1e-9)
    np.testing.assert_allclose(mk[ref][..., :half], np.abs(dk[ref][..., :half]), rtol=1e-9)
    # the case is not degenerate: many-term elements with sizeable values
    assert np.abs(dq[..., :half]).min() > 1e-6 and np.abs(dk[ref][..., :half]).max() > 1e-3
