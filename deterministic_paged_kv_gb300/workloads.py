"""Seeded synthetic inputs for paged-KV attention.

This module only draws random inputs and lays out page tables; it holds none
of the attention arithmetic.  Both the CUDA path's tests/benchmark and the
oracle's tests take their inputs from here, so both sides see identical bytes.

Recipe (all on the CPU, ``torch.Generator`` seeded per workload; draw order
Q, K cache, V cache, then the page permutation; ragged lengths come from a
second generator seeded from the workload seed):
  * Q, K cache, V cache ~ N(0, 1) drawn in float32, rounded to bfloat16;
  * the K cache is stored pre-RoPE, NHD: [num_pages, page_size, Hkv, D];
  * each row's pages come from a random permutation of the page pool, unused
    block-table entries are -1;
  * decode rows put the query at position kv_len (keys 0..kv_len-1), chunked
    prefill rows put the chunk's queries at the trailing positions
    kv_len-Sq .. kv_len-1 (the chunk's own K/V already in the cache).

The named workloads mirror the shapes of the pages' decode/prefill runs
(page 16, head_dim 128, NHD, theta 1e6, GQA 32/8).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

PAGE = 16


@dataclass
class Workload:
    name: str
    q: torch.Tensor            # bf16 [B, Hq, Sq, D]
    k_cache: torch.Tensor      # bf16 [NP, PAGE, Hkv, D]
    v_cache: torch.Tensor      # bf16 [NP, PAGE, Hkv, D]
    block_table: torch.Tensor  # int32 [B, W]
    kv_lens: torch.Tensor      # int32 [B]
    position_ids: torch.Tensor  # int32 [B, Sq]
    mode: str                  # "decode" or "prefill"
    rope_theta: float = 1e6
    rope_scale: float = 1.0
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return self.q.shape[0]

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def Sq(self):
        return self.q.shape[2]

    @property
    def D(self):
        return self.q.shape[3]

    @property
    def Hkv(self):
        return self.k_cache.shape[2]

    @property
    def num_pages(self):
        return self.k_cache.shape[0]

    @property
    def W(self):
        return self.block_table.shape[1]


def _randn_bf16(gen, shape):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def build(name, B, Sq, Hq, Hkv, D, kv_lens, num_pages, W, seed, mode,
          q_pos_offset=None, rope_theta=1e6, rope_scale=1.0, page_perm=True):
    """Generic builder.

    ``kv_lens``: list of ints (one per row).  Row b gets ceil(kv_len/PAGE)
    pages, taken in order from a seeded permutation of the pool.
    ``q_pos_offset``: position of query s is ``kv_len - Sq + s + q_pos_offset``
    (decode default: offset 1, i.e. the query sits at kv_len; prefill default:
    offset 0, trailing positions ending at kv_len-1).
    """
    gen = torch.Generator().manual_seed(int(seed))
    q = _randn_bf16(gen, (B, Hq, Sq, D))
    k_cache = _randn_bf16(gen, (num_pages, PAGE, Hkv, D))
    v_cache = _randn_bf16(gen, (num_pages, PAGE, Hkv, D))
    perm = (torch.randperm(num_pages, generator=gen) if page_perm
            else torch.arange(num_pages)).to(torch.int32)
    kv = [int(x) for x in kv_lens]
    need = [(n + PAGE - 1) // PAGE for n in kv]
    if sum(need) > num_pages:
        raise ValueError("page pool too small")
    if max(need + [0]) > W:
        raise ValueError("table width too small")
    bt = torch.full((B, W), -1, dtype=torch.int32)
    cur = 0
    for b in range(B):
        bt[b, :need[b]] = perm[cur:cur + need[b]]
        cur += need[b]
    if q_pos_offset is None:
        q_pos_offset = 1 if mode == "decode" else 0
    pos = torch.empty((B, Sq), dtype=torch.int32)
    for b in range(B):
        start = max(kv[b] - Sq + q_pos_offset, 0)
        pos[b] = torch.arange(start, start + Sq, dtype=torch.int32)
    return Workload(name, q, k_cache, v_cache, bt, torch.tensor(kv, dtype=torch.int32),
                    pos, mode, rope_theta, rope_scale)


def ragged_case(q_lens, kv_lens, seed, Hq=32, Hkv=8, D=128, extra_pages=3):
    """A ragged batch, kept padded to max(q_lens) queries per row (the pack
    step below gives the packed layout).  Row b has q_lens[b] queries: one
    query sits at position kv_len (a decode row), longer rows take the
    trailing positions kv_len - q_len .. kv_len - 1 (a prefill chunk); padding
    entries repeat the row's last position and are never read."""
    B = len(q_lens)
    mq = max(list(q_lens) + [1])
    need = sum((int(n) + PAGE - 1) // PAGE for n in kv_lens)
    W = max([(int(n) + PAGE - 1) // PAGE for n in kv_lens] + [1])
    w = build("ragged", B, mq, Hq, Hkv, D, kv_lens, need + extra_pages, W, seed, "prefill")
    pos = torch.zeros((B, mq), dtype=torch.int32)
    for b, n in enumerate(q_lens):
        n = int(n)
        if n == 0:
            continue
        start = max(int(kv_lens[b]) - n + (1 if n == 1 else 0), 0)
        pos[b, :n] = torch.arange(start, start + n, dtype=torch.int32)
        pos[b, n:] = start + n - 1
    w.position_ids = pos
    w.meta["q_lens"] = [int(n) for n in q_lens]
    return w


def pack_ragged(w):
    """(q [total_q, Hq, D], qo_indptr [B + 1], position_ids [total_q]) of a
    ragged_case workload: row b's first q_lens[b] queries, rows in order."""
    ql = w.meta["q_lens"]
    indptr = [0]
    for n in ql:
        indptr.append(indptr[-1] + n)
    q = torch.cat([w.q[b, :, :n].transpose(0, 1) for b, n in enumerate(ql)], 0).contiguous()
    pos = torch.cat([w.position_ids[b, :n] for b, n in enumerate(ql)]).contiguous()
    return q, torch.tensor(indptr, dtype=torch.int32), pos


def decode_small():
    """B=2, q_len 1, kv_len 128, query at 128; 16 pages shuffled."""
    return build("decode_small: B=2 kv=128 Hq=32 Hkv=8 d=128", 2, 1, 32, 8, 128,
                 [128, 128], 16, 8, 1001, "decode")


def decode_invariance(W=128):
    """B=8 ragged kv_len ~ U[1, 2048]; 1024 pages shuffled; width W."""
    gen = torch.Generator().manual_seed(1002 + 7919)
    kv = torch.randint(1, 2049, (8,), generator=gen).tolist()
    return build("decode_invariance: B=8 kv~U[1,2048] Hq=32 Hkv=8 d=128", 8, 1, 32, 8, 128,
                 kv, 1024, W, 1002, "decode")


def decode_throughput():
    """B=64, kv_len 4096 each (256 pages/row), 16384 pages shuffled."""
    return build("decode_throughput: B=64 kv=4096 Hq=32 Hkv=8 d=128", 64, 1, 32, 8, 128,
                 [4096] * 64, 16384, 256, 1003, "decode")


def prefill_chunk():
    """B=4, 1536-token paged prefix + 512-token causal chunk (pos 1536..2047)."""
    return build("prefill_chunk: B=4 prefix=1536 chunk=512 Hq=32 Hkv=8 d=128", 4, 512, 32, 8,
                 128, [2048] * 4, 512, 128, 1004, "prefill")


def decode_long():
    """B=1, kv_len 32768 (2048 pages), query at 32768, no split-KV."""
    return build("decode_long: B=1 kv=32768 Hq=32 Hkv=8 d=128", 1, 1, 32, 8, 128,
                 [32768], 2048, 2048, 1005, "decode")


def prefill_long():
    """B=1 full causal prefill, S=8192 (512 pages), positions 0..8191."""
    return build("prefill_long: B=1 S=8192 Hq=32 Hkv=8 d=128", 1, 8192, 32, 8, 128,
                 [8192], 512, 512, 1006, "prefill")


NAMED = {
    "decode_small": decode_small,
    "decode_invariance": decode_invariance,
    "decode_throughput": decode_throughput,
    "prefill_chunk": prefill_chunk,
    "decode_long": decode_long,
    "prefill_long": prefill_long,
}


def repad(block_table: torch.Tensor, W: int) -> torch.Tensor:
    """Same page lists in a wider (or narrower) table, padded with -1."""
    B, W0 = block_table.shape
    out = torch.full((B, W), -1, dtype=torch.int32)
    n = min(W, W0)
    out[:, :n] = block_table[:, :n]
    if W < W0 and bool((block_table[:, W:] >= 0).any()):
        raise ValueError("narrower table would drop pages")
    return out


def select_rows(w: Workload, rows, W=None) -> Workload:
    """A sub-batch of ``w`` with the given rows (same pool, same pages)."""
    idx = torch.tensor(list(rows), dtype=torch.long)
    bt = w.block_table[idx]
    if W is not None:
        bt = repad(bt, W)
    return Workload(w.name + " rows=%s" % list(rows), w.q[idx].contiguous(), w.k_cache,
                    w.v_cache, bt.contiguous(), w.kv_lens[idx].contiguous(),
                    w.position_ids[idx].contiguous(), w.mode, w.rope_theta, w.rope_scale)


def permute_pages(w: Workload, seed: int) -> Workload:
    """Move every page to a new physical slot and rewrite the table to match."""
    gen = torch.Generator().manual_seed(int(seed))
    NP = w.num_pages
    perm = torch.randperm(NP, generator=gen)          # new slot of old page p
    k = torch.empty_like(w.k_cache)
    v = torch.empty_like(w.v_cache)
    k[perm] = w.k_cache
    v[perm] = w.v_cache
    bt = w.block_table.clone()
    live = bt >= 0
    bt[live] = perm[bt[live].long()].to(torch.int32)
    return Workload(w.name + " permuted", w.q, k, v, bt, w.kv_lens, w.position_ids,
                    w.mode, w.rope_theta, w.rope_scale)


def random_case(B, Sq, Hq, Hkv, D, kv_lens, seed, mode, W=None, extra_pages=3,
                q_pos_offset=None):
    """Small ragged case for parity tests: pool just large enough plus spare pages."""
    need = sum((int(n) + PAGE - 1) // PAGE for n in kv_lens)
    maxp = max([(int(n) + PAGE - 1) // PAGE for n in kv_lens] + [1])
    return build("random", B, Sq, Hq, Hkv, D, kv_lens, need + extra_pages,
                 W or maxp, seed, mode, q_pos_offset=q_pos_offset)
