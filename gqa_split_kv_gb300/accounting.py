"""Algorithmic byte counts of one decode-attention call (for GB/s and rooflines).

The bytes a call must move at minimum, by tensor:
  kv        = 2 * D * 2 B * Hkv * sum_b L_b        (every cached K and V row once)
  q         = B * Hq * D * 2 B
  out       = B * Hq * D * 2 B
  partials  = per (b, h) with n >= 2 pieces: n * (D + 2) * 4 B, written once by the
              split kernel and read once by the combine
  page_table= 4 B * sum_b ceil(L_b / page_size)    (paged caches)
  seq_lens  = 4 B * B

"algorithmic" = kv + q + partials read + page_table + seq_lens (what the combine
and split kernels must read); "strict" = kv + q + out.  Which segments are cut
into pieces, and into how many, is asked of the library's own planner
(decode_plan_pieces, host only).
"""
from __future__ import annotations

from typing import Optional

import numpy as np


def split_part_rows(seq_lens, Hq: int, Hkv: int, D: int, S: int, q_len: int = 1) -> int:
    """Rows x pieces of the partials one call writes: the sum, over the pieces of
    segments cut into two or more, of the piece's query rows."""
    from . import binding
    lens = np.asarray(seq_lens, dtype=np.int32)
    if S < 2 or lens.size == 0 or int(lens.max()) == 0:
        return 0
    rec = binding.plan_pieces(lens, Hq, Hkv, D, int(lens.max()), S, q_len=q_len)
    return int(rec[rec[:, 4] >= 2, 2].sum())


def traffic_bytes(B: int, Hq: int, Hkv: int, D: int, seq_lens, S: int, page_size: Optional[int] = None,
                  q_len: int = 1, kv_dtype: str = "bf16") -> dict:
    """Bytes of one call; with q_len > 1 (multi-query decode) the rows of a KV head
    are its G query heads x q_len query tokens, and K/V are still read once.  An
    int8 cache moves D bytes plus a 4-byte scale per (token, KV head) and tensor."""
    lens = np.asarray(seq_lens, dtype=np.int64)
    kv = 2 * (D + 4 if kv_dtype == "int8" else 2 * D) * Hkv * int(lens.sum())
    q = B * Hq * q_len * D * 2
    out = B * Hq * q_len * D * 2
    partials = split_part_rows(lens, Hq, Hkv, D, S, q_len) * (D + 2) * 4
    pt = 0 if page_size is None else 4 * int(((lens + page_size - 1) // page_size).sum())
    sl = 4 * B
    return {"kv": kv, "q": q, "out": out, "partials_read": partials, "partials_written": partials,
            "page_table": pt, "seq_lens": sl,
            "algorithmic": kv + q + partials + pt + sl, "strict": kv + q + out}


def prefill_visible(seq_lens, q_len: int) -> int:
    """Keys seen by all query tokens of a causal chunk, summed over sequences (per
    query head): query i of a sequence of L tokens sees max(0, min(L, L - q_len + 1 + i))."""
    total = 0
    for L in np.asarray(seq_lens, dtype=np.int64):
        L = int(L)
        lo = L - q_len + 1  # keys of query 0
        # sum over i of clamp(lo + i, 0, L)
        for_i = np.clip(lo + np.arange(q_len, dtype=np.int64), 0, L)
        total += int(for_i.sum())
    return total


def prefill_work(B: int, Hq: int, Hkv: int, D: int, seq_lens, q_len: int) -> dict:
    """Algorithmic flops and bytes of one causal prefill call: 2 D flops for each
    (query, key) score and 2 D for its share of P V, per query head; bytes of q,
    out and of K/V read once."""
    vis = prefill_visible(seq_lens, q_len)
    flops = 4 * D * Hq * vis
    kv = 2 * 2 * D * Hkv * int(np.clip(np.asarray(seq_lens, dtype=np.int64), 0, None).sum())
    qo = 2 * 2 * B * q_len * Hq * D
    return {"flops": flops, "visible_pairs_per_head": vis, "kv_bytes": kv, "q_out_bytes": qo}
