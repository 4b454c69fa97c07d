"""Shared helpers for the GPU parity tests (inputs from workloads, reference
from the oracle, kernels through the C ABI binding)."""
import numpy as np
import torch

OUT_TOL = 2e-2   # max abs error, BF16 out vs float64 oracle
LSE_TOL = 1e-3   # max abs error, FP32 LSE vs float64 oracle


def to_dev(w, device="cuda"):
    return {k: getattr(w, k).to(device) for k in
            ("q", "k_cache", "v_cache", "block_table", "kv_lens", "position_ids")}


def run_gpu(w, mode=None, validate=True, status=None, stream=None, split_tokens=0):
    """Launch through the C ABI; returns device (out, lse).  split_tokens > 0
    selects the fixed-split decode entry point."""
    from deterministic_paged_kv_gb300 import binding
    mode = mode or w.mode
    d = to_dev(w)
    p = None
    if validate:
        p = binding.plan(w.B, w.Sq, w.Hq, w.Hkv, w.D, 16, w.num_pages, w.W, w.block_table,
                         w.kv_lens, w.position_ids, w.rope_theta, w.rope_scale)
    return binding.run(mode, d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["kv_lens"],
                       d["position_ids"], plan_obj=p, rope_theta=w.rope_theta,
                       rope_scale=w.rope_scale, status=status, stream=stream, split_tokens=split_tokens)


def oracle_ref(w, row_mask=None):
    import oracle
    return oracle.attention(w.q, w.k_cache, w.v_cache, w.block_table, w.kv_lens, w.position_ids,
                            w.rope_theta, w.rope_scale, row_mask=row_mask)


def compare(out, lse, ref_out, ref_lse, mask=None):
    """Max abs errors over the compared entries (mask [B, Sq] of queries)."""
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.float().cpu().numpy().astype(np.float64)
    if mask is not None:
        sel = np.asarray(mask, bool)
        o = o.transpose(0, 2, 1, 3)[sel]
        l = l.transpose(0, 2, 1)[sel]
        ref_out = ref_out.transpose(0, 2, 1, 3)[sel]
        ref_lse = ref_lse.transpose(0, 2, 1)[sel]
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(l), fin), "LSE finiteness differs"
    assert np.array_equal(np.isneginf(l), np.isneginf(ref_lse))
    eo = float(np.max(np.abs(o - ref_out))) if o.size else 0.0
    el = float(np.max(np.abs(l[fin] - ref_lse[fin]))) if fin.any() else 0.0
    return eo, el


def assert_parity(out, lse, ref_out, ref_lse, mask=None, out_tol=OUT_TOL, lse_tol=LSE_TOL):
    eo, el = compare(out, lse, ref_out, ref_lse, mask)
    assert eo <= out_tol and el <= lse_tol, "out err %.3g (tol %.3g), lse err %.3g (tol %.3g)" % (
        eo, out_tol, el, lse_tol)
    return eo, el


def bitwise_equal(a, b):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
