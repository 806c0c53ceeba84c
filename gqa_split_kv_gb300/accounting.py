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
and split kernels must read); "strict" = kv + q + out.  The piece count per
segment restates the library's split rule (see include/decode_attn.h) for
counting only.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

BLOCK = 16


def _groups(G: int):
    ng = -(-G // 8)
    gr = -(-G // ng)
    return ng, gr


def _passes(G: int, D: int):
    """(sub-groups per pass, passes per KV head, rows per sub-group): a pass runs the
    largest power of two of sub-groups that divides their number, at most 2 at
    D = 128, else 4."""
    ng, gr = _groups(G)
    per, cap = 1, (2 if D == 128 else 4)
    while per * 2 <= cap and ng % (per * 2) == 0:
        per *= 2
    return per, -(-ng // per), gr


def piece_counts(seq_lens, Hkv: int, G: int, S: int, D: int) -> np.ndarray:
    """Pieces of every segment, shape [B, Hkv * passes].

    The library's split plan: segments lie end to end on one line in (u, b)
    order (slot-major), each taking
    gap + 4 ceil(n_b / 4) positions (gap = 4 ceil((2816 / D) / 4) positions
    without blocks, then its blocks, then padding); the line is cut into ranges
    of q positions."""
    lens = np.asarray(seq_lens, dtype=np.int64)
    _, npass, _ = _passes(G, D)
    U = Hkv * npass
    nblk = (lens + BLOCK - 1) // BLOCK
    B = len(lens)
    if S == 1:
        return np.where(nblk[:, None] > 0, 1, 0) * np.ones((B, U), dtype=np.int64)
    gap = (2816 // D + 3) // 4 * 4
    w = np.where(nblk > 0, (nblk + 3) // 4 * 4 + gap, 0)
    P = np.concatenate([[0], np.cumsum(w)])
    NB = U * int(P[-1])
    R = (S - 1) * U
    q = max(4, -(-max(1, -(-NB // R)) // 4) * 4)
    s0 = np.arange(U)[None, :] * int(P[-1]) + P[:-1, None] + gap
    s1 = s0 + nblk[:, None]
    n = (s1 - 1) // q - s0 // q + 1
    return np.where(nblk[:, None] > 0, n, 0)


def traffic_bytes(B: int, Hq: int, Hkv: int, D: int, seq_lens, S: int, page_size: Optional[int] = None,
                  q_len: int = 1, kv_dtype: str = "bf16") -> dict:
    """Bytes of one call; with q_len > 1 (multi-query decode) the rows of a KV head
    are its G query heads x q_len query tokens, and K/V are still read once.  An
    int8 cache moves D bytes plus a 4-byte scale per (token, KV head) and tensor."""
    lens = np.asarray(seq_lens, dtype=np.int64)
    G = Hq // Hkv * q_len
    per, npass, gr = _passes(G, D)
    kv = 2 * (D + 4 if kv_dtype == "int8" else 2 * D) * Hkv * int(lens.sum())
    q = B * Hq * q_len * D * 2
    out = B * Hq * q_len * D * 2
    n = piece_counts(lens, Hkv, G, S, D)                      # [B, U]
    # rows of segment slot u = h * npass + pass
    heads = np.array([min(per * gr, G - (u % npass) * per * gr) for u in range(Hkv * npass)])
    part_rows = int(((n >= 2) * n * heads[None, :]).sum())
    partials = part_rows * (D + 2) * 4
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
