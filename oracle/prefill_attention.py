"""CPU oracle for causal GQA prefill / chunked-prefill attention (test
infrastructure only; the CUDA library never calls it and shares no code with it).

"gqa_prefill_attn" appears on the AstrAI commit page ("csrc", commit 988e013) as a
tiled shared-memory K/V kernel with mask support, and the page on the double-buffered
cp.async rewrite compares its prefill against torch SDPA.  The pages fix neither the
mask nor the layouts, so this module takes the plain causal reading, the same one as
multi-query decode:

- sequence b holds L_b cached tokens, of which the last q_len are the chunk being
  prefilled (full prefill: L_b == q_len);
- query token i (0-based) sits at position L_b - q_len + i and attends to positions
  0 .. L_b - q_len + i (itself included); a query that sees no token (L_b < q_len - i)
  gives zeros;
- query head h reads KV head h // G;
- q and the output are token-major [B, q_len, Hq, D] (the layout a QKV projection
  writes); the cache is the decode cache, contiguous [B, max_ctx, Hkv, D] or paged.

Every value is computed in float64 from the bf16 inputs (exact widening), with the
attention definition softmax(q K^T * scale) V per query row.
"""
from __future__ import annotations

from typing import Iterable, Optional, Tuple

import numpy as np

from .decode_attention import _kv_rows, visible_tokens, widen_bf16

__all__ = ["prefill", "prefill_row_count"]


def _causal_attend(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, L: int, q_len: int) -> np.ndarray:
    """Q [q_len, D], K/V [L, D] float64 -> [q_len, D]: row i sees K[:visible_tokens(L, q_len, i)]."""
    out = np.zeros((q_len, Q.shape[1]))
    if L == 0:
        return out
    s = (Q @ K.T) * float(scale)  # [q_len, L]
    vis = np.array([visible_tokens(L, q_len, i) for i in range(q_len)])
    seen = np.arange(L)[None, :] < vis[:, None]
    s = np.where(seen, s, -np.inf)
    has = vis > 0
    M = np.where(has, s.max(axis=1), 0.0)[:, None]
    w = np.where(seen, np.exp(s - M), 0.0)
    den = w.sum(axis=1, keepdims=True)
    out[has] = (w @ V)[has] / den[has]
    return out


def prefill(inp: dict, rows: Optional[Iterable[Tuple[int, int, int]]] = None) -> np.ndarray:
    """fp64 causal prefill.  inp["q"] is [B, q_len, Hq, D] bf16 bits; the cache is
    contiguous ("k", "v") or paged ("k_pool", "v_pool", "page_table", "page_size");
    inp["seq_lens"] [B], inp["scale"].  Returns [B, q_len, Hq, D], or [n, D] for the
    selected (b, i, h) rows."""
    q = inp["q"]
    B, q_len, Hq, D = q.shape
    Hkv = (inp["k"] if "k" in inp else inp["k_pool"]).shape[2]
    G = Hq // Hkv
    full = rows is None
    want = None if full else list(rows)
    out = np.zeros((B, q_len, Hq, D))
    for b in range(B):
        if not full and not any(w[0] == b for w in want):
            continue
        L = int(inp["seq_lens"][b])
        Kb, Vb = _kv_rows(inp, b, L)
        heads = range(Hq) if full else sorted({w[2] for w in want if w[0] == b})
        for h in heads:
            g = h // G
            out[b, :, h] = _causal_attend(widen_bf16(q[b, :, h]), widen_bf16(Kb[:, g]), widen_bf16(Vb[:, g]),
                                          inp["scale"], L, q_len)
    if full:
        return out
    return np.stack([out[b, i, h] for b, i, h in want]) if want else np.zeros((0, D))


def prefill_row_count(seq_lens, q_len: int) -> int:
    """Sum over sequences and query tokens of the keys each query sees (per head)."""
    return int(sum(visible_tokens(int(L), q_len, i) for L in seq_lens for i in range(q_len)))
