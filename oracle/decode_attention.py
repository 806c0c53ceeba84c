"""Plain fp64 CPU oracle for single-token GQA decode attention.

TEST INFRASTRUCTURE.  This module is the reference that the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import it.  It shares no code with the CUDA
path (no kernels, headers, helpers, tables or pre/post-processing); both are
fed the same seeded inputs by a separate generator module.

What is computed (the decode-attention definition that the source pages build
their kernels around; none of the pages writes it as an equation):
for sequence b, query head h and its KV head g = h // G (G = Hq / Hkv, the G
query heads of one KV head are consecutive), over the L_b cached tokens t,

    s_t   = scale * sum_d q[b,h,d] * k[b,t,g,d]
    out   = sum_t exp(s_t - M) v[b,t,g,:] / sum_t exp(s_t - M),   M = max_t s_t

in float64 from the exactly widened bf16 inputs, then rounded once to bf16
(round to nearest, ties to even).

Split-KV (AstrAI commit 988e013 "csrc", split-KV items; "perf(qwen3.8):
split the flash-decode KV range across warp-groups", section "Mechanism"):
a piece of the token range yields unnormalised partials (acc, m, l) with
m = max over the piece, acc = sum exp(s - m) v, l = sum exp(s - m); pieces
are merged by the log-sum-exp rescale in ascending piece order.  Which
partition of the token range a GPU call uses is not the oracle's business
(the pages fix only caps on the split count, and any partition merges to the
same result): ``range_partials`` computes the partials of whatever token
ranges it is given.

Paged caches (AstrAI commit 69fecaf "csrc/tests", paged decode items): token
t of sequence b is row t % page_size of physical page page_table[b, t // page_size].

Every function here is pinned by tests/test_oracle.py against closed forms,
invariants, a high-precision brute force and torch's scaled_dot_product_attention.
"""
from __future__ import annotations

import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "widen_bf16",
    "round_to_bf16",
    "attend",
    "attend_partial",
    "merge_partials",
    "gather_paged",
    "decode_contig",
    "decode_paged",
    "decode_rows",
    "range_partials",
    "combine_partials",
    "visible_tokens",
    "decode_multi",
    "dequant_rows",
    "decode_int8",
]


# ---------------------------------------------------------------- bf16 bits

def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64, exactly (a bf16 is the top half of a float32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, one rounding: nearest, ties to even.

    bf16 has an 8-bit significand (7 stored bits) and float32's exponent range.
    Normal numbers are rounded to 8 significant bits; below 2**-126 the grid is
    the subnormal spacing 2**-133; results of magnitude >= 2**128 after rounding
    overflow to infinity.  NaN maps to the canonical quiet NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    flat = x.reshape(-1)
    res = out.reshape(-1)
    nan = np.isnan(flat)
    sign = np.signbit(flat)
    a = np.abs(np.where(nan, 0.0, flat))
    mant, expo = np.frexp(a)                       # a = mant * 2**expo, mant in [0.5, 1)
    normal = expo - 1 >= -126
    # significand as an integer in [128, 256]: a = n * 2**(expo - 8)
    n_norm = np.rint(np.ldexp(mant, 8))
    v_norm = np.ldexp(n_norm, expo - 8)
    v_sub = np.ldexp(np.rint(np.ldexp(a, 133)), -133)
    v = np.where(normal, v_norm, v_sub)
    v = np.where(v >= 2.0 ** 128, np.inf, v)
    v32 = np.where(sign, -v, v).astype(np.float32)  # exact: v is on the bf16 grid
    bits = (v32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits[nan] = 0x7FC0
    res[:] = bits
    return out


# ------------------------------------------------------------ the definition

def attend(q_rows: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(q K^T * scale) V for each query row, in float64.

    q_rows [n, D], K [L, D], V [L, D] (float64).  Returns [n, D] float64.
    L == 0 gives zeros (an empty context has nothing to attend to).
    """
    n, D = q_rows.shape
    if K.shape[0] == 0:
        return np.zeros((n, D), dtype=np.float64)
    s = (q_rows @ K.T) * float(scale)              # [n, L]
    M = s.max(axis=1, keepdims=True)
    w = np.exp(s - M)
    return (w @ V) / w.sum(axis=1, keepdims=True)


def attend_partial(q_rows: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float):
    """Unnormalised partials over one piece of the context.

    Returns (acc [n, D], m [n], l [n]) with m = max_t s_t,
    acc = sum_t exp(s_t - m) V_t, l = sum_t exp(s_t - m).
    An empty piece gives (0, -inf, 0).
    """
    n, D = q_rows.shape
    if K.shape[0] == 0:
        return np.zeros((n, D)), np.full(n, -np.inf), np.zeros(n)
    s = (q_rows @ K.T) * float(scale)
    m = s.max(axis=1)
    w = np.exp(s - m[:, None])
    return w @ V, m, w.sum(axis=1)


def merge_partials(parts: Sequence[Tuple[np.ndarray, np.ndarray, np.ndarray]]) -> np.ndarray:
    """Log-sum-exp merge of partials, in the order given.

    M = max_j m_j over pieces with l_j > 0; w_j = exp(m_j - M);
    out = sum_j w_j acc_j / sum_j w_j l_j.  Pieces with l_j == 0 are skipped;
    if every piece is empty the result is zero.
    """
    acc0 = parts[0][0]
    n, D = acc0.shape
    out = np.zeros((n, D))
    for r in range(n):
        live = [(a[r], m[r], l[r]) for (a, m, l) in parts if l[r] > 0]
        if not live:
            continue
        M = max(m for (_, m, _) in live)
        num = np.zeros(D)
        den = 0.0
        for a, m, l in live:
            w = math.exp(m - M)
            num += w * a
            den += w * l
        out[r] = num / den
    return out


# --------------------------------------------------------------- KV access

def gather_paged(pool: np.ndarray, page_table: np.ndarray, b: int, L: int, page_size: int) -> np.ndarray:
    """Logical token rows [L, Hkv, D] of sequence b from a paged pool, one token at a time."""
    rows = [pool[page_table[b, t // page_size], t % page_size] for t in range(L)]
    if not rows:
        return pool[:0, 0]
    return np.stack(rows)


def _kv_rows(inp: dict, b: int, L: int):
    """(K, V) for sequence b as bf16 bits [L, Hkv, D]."""
    if "k" in inp:
        return inp["k"][b, :L], inp["v"][b, :L]
    ps = int(inp["page_size"])
    return (gather_paged(inp["k_pool"], inp["page_table"], b, L, ps),
            gather_paged(inp["v_pool"], inp["page_table"], b, L, ps))


def decode_rows(inp: dict, pairs: Iterable[Tuple[int, int]], scale: Optional[float] = None) -> np.ndarray:
    """fp64 outputs for selected (b, query head) pairs only.  Returns [n, D]."""
    q = inp["q"]
    Hq = q.shape[1]
    Hkv = (inp["k"] if "k" in inp else inp["k_pool"]).shape[2]
    G = Hq // Hkv
    scale = inp["scale"] if scale is None else scale
    res = []
    cache = {}
    for b, h in pairs:
        L = int(inp["seq_lens"][b])
        if b not in cache:
            cache = {b: _kv_rows(inp, b, L)}
        Kb, Vb = cache[b]
        g = h // G
        res.append(attend(widen_bf16(q[b, h])[None], widen_bf16(Kb[:, g]), widen_bf16(Vb[:, g]), scale)[0])
    return np.stack(res) if res else np.zeros((0, q.shape[2]))


def decode_contig(q, k, v, seq_lens, scale) -> np.ndarray:
    """Contiguous cache k, v [B, max_ctx, Hkv, D] (bf16 bits).  Returns fp64 [B, Hq, D]."""
    inp = {"q": q, "k": k, "v": v, "seq_lens": seq_lens, "scale": scale}
    return _decode_all(inp)


def decode_paged(q, k_pool, v_pool, page_table, seq_lens, page_size, scale) -> np.ndarray:
    """Paged cache pools [num_pages, page_size, Hkv, D] + page_table [B, max_pages].  fp64 [B, Hq, D]."""
    inp = {"q": q, "k_pool": k_pool, "v_pool": v_pool, "page_table": page_table,
           "seq_lens": seq_lens, "page_size": page_size, "scale": scale}
    return _decode_all(inp)


def _decode_all(inp: dict) -> np.ndarray:
    q = inp["q"]
    B, Hq, D = q.shape
    Hkv = (inp["k"] if "k" in inp else inp["k_pool"]).shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(inp["seq_lens"][b])
        Kb, Vb = _kv_rows(inp, b, L)
        for g in range(Hkv):
            Kg, Vg = widen_bf16(Kb[:, g]), widen_bf16(Vb[:, g])
            out[b, g * G:(g + 1) * G] = attend(widen_bf16(q[b, g * G:(g + 1) * G]), Kg, Vg, inp["scale"])
    return out


# ------------------------------------------------------------ partials of given ranges

def range_partials(inp: dict, ranges: Iterable[Tuple[int, int, int, int, int, int]], num_splits: int):
    """fp64 unnormalised partials of given query rows over given token ranges,
    laid out as a GPU call's partial buffers.

    inp is a decode input (q [B, Hq, D]), a multi-query input (q [B, Hq, q_len, D])
    or an int8-cache input, with a contiguous or paged cache.  The rows of a
    sequence are its Hq * q_len (query head h, query token i) pairs, head-major
    (row r = h * q_len + i; q_len = 1 for single-token decode); query token i sees
    visible_tokens(L_b, q_len, i) tokens.  Each range (b, row0, nrows, slot, t0, t1)
    asks for the partials of rows row0 .. row0 + nrows - 1 of sequence b over
    tokens [t0, t1), cut at what each row sees, stored in partial slot `slot`:
    attend_partial of that row and token range (an empty range gives (0, -inf, 0)).

    Returns (acc [B, R, S, D], ml [B, R, S, 2]) with R = Hq * q_len; slots that no
    range fills are NaN.
    """
    q = inp["q"]
    B, Hq = q.shape[:2]
    D = q.shape[-1]
    qlen = q.shape[2] if q.ndim == 4 else 1
    qrows = q.reshape(B, Hq * qlen, D)
    kname = next(n for n in ("k", "k_pool", "k_i8", "k_pool_i8") if n in inp)
    Hkv = inp[kname].shape[2]
    G = Hq // Hkv
    acc = np.full((B, Hq * qlen, num_splits, D), np.nan)
    ml = np.full((B, Hq * qlen, num_splits, 2), np.nan)
    cache = {}
    for b, row0, nrows, slot, t0, t1 in ranges:
        L = int(inp["seq_lens"][b])
        if b not in cache:
            if kname in ("k_i8", "k_pool_i8"):
                cache = {b: dequant_rows(inp, b, L)}
            else:
                Kb, Vb = _kv_rows(inp, b, L)
                cache = {b: (widen_bf16(Kb), widen_bf16(Vb))}
        K, V = cache[b]
        for r in range(row0, row0 + nrows):
            h, i = r // qlen, r % qlen
            hi = min(t1, visible_tokens(L, qlen, i))
            lo = min(t0, hi)
            a, m, l = attend_partial(widen_bf16(qrows[b, r])[None], K[lo:hi, h // G], V[lo:hi, h // G], inp["scale"])
            acc[b, r, slot] = a[0]
            ml[b, r, slot] = (m[0], l[0])
    return acc, ml


def combine_partials(part_acc: np.ndarray, part_ml: np.ndarray) -> np.ndarray:
    """The stand-alone merge: all S slots of each (b, h), skipping slots with l == 0.

    part_acc [B, Hq, S, D], part_ml [B, Hq, S, 2] = (m, l).  Returns fp64 [B, Hq, D].
    """
    B, Hq, S, D = part_acc.shape
    out = np.zeros((B, Hq, D))
    for b in range(B):
        for h in range(Hq):
            parts = [(part_acc[b, h, j][None].astype(np.float64),
                      np.array([float(part_ml[b, h, j, 0])]),
                      np.array([float(part_ml[b, h, j, 1])])) for j in range(S)]
            out[b, h] = merge_partials(parts)[0]
    return out


# ------------------------------------------------------------ multi-query decode
#
# Speculative verification ("perf(dspark): overlap KV staging with compute via
# cp.async", section "sparkinfer DSpark auto-eval — eval-dspark:XL", which scores a
# draft block of 7): a sequence of L cached tokens whose last q_len tokens are the
# new block scores q_len queries at once.  Query token i (0-based) sits at position
# L - q_len + i and sees every token up to and including itself.  q and the output
# are [B, Hq, q_len, D]; the pages do not fix the layout (head-major is this
# library's choice).

def visible_tokens(L: int, q_len: int, i: int) -> int:
    """Tokens that query token i of the block sees: positions 0 .. L - q_len + i."""
    return max(0, min(L, L - q_len + 1 + i))


def decode_multi(inp: dict, rows: Optional[Iterable[Tuple[int, int, int]]] = None) -> np.ndarray:
    """fp64 multi-query outputs.  inp["q"] is [B, Hq, q_len, D] bf16 bits; the cache
    is contiguous ("k", "v") or paged ("k_pool", "v_pool", "page_table", "page_size").
    Returns [B, Hq, q_len, D], or [n, D] for the selected (b, h, i) rows.  A query
    that sees no token gives zeros."""
    q = inp["q"]
    B, Hq, qlen, D = q.shape
    Hkv = (inp["k"] if "k" in inp else inp["k_pool"]).shape[2]
    G = Hq // Hkv
    want = [(b, h, i) for b in range(B) for h in range(Hq) for i in range(qlen)] if rows is None else list(rows)
    res = np.zeros((len(want), D))
    cache = {}
    for n, (b, h, i) in enumerate(want):
        L = int(inp["seq_lens"][b])
        if b not in cache:
            cache = {b: _kv_rows(inp, b, L)}
        Kb, Vb = cache[b]
        t = visible_tokens(L, qlen, i)
        if t == 0:
            continue
        g = h // G
        res[n] = attend(widen_bf16(q[b, h, i])[None], widen_bf16(Kb[:t, g]), widen_bf16(Vb[:t, g]), inp["scale"])[0]
    return res.reshape(B, Hq, qlen, D) if rows is None else res


# ------------------------------------------------------------ int8 KV cache
#
# "perf(dspark): overlap KV staging with compute via cp.async", section "Cost and
# fallbacks", names an int8 KV pool read through a dequant-into-shared-memory path
# but fixes no format.  Reading used here: symmetric int8 per (token, KV head),
# K[t, g, :] = k_i8[t, g, :] * k_scale[g, t] (V likewise), with fp32 scales stored
# head-major ([B, Hkv, max_ctx] contiguous, [num_pages, Hkv, page_size] paged).

def dequant_rows(inp: dict, b: int, L: int):
    """fp64 (K, V) rows [L, Hkv, D] of sequence b of an int8 cache, dequantized."""
    if "k_i8" in inp:
        k = inp["k_i8"][b, :L].astype(np.float64) * inp["k_scale"][b, :, :L].T.astype(np.float64)[:, :, None]
        v = inp["v_i8"][b, :L].astype(np.float64) * inp["v_scale"][b, :, :L].T.astype(np.float64)[:, :, None]
        return k, v
    ps = int(inp["page_size"])
    table = inp["page_table"]
    ks, vs = [], []
    for t in range(L):
        page, row = table[b, t // ps], t % ps
        ks.append(inp["k_pool_i8"][page, row].astype(np.float64) * inp["k_scale_pool"][page, :, row][:, None])
        vs.append(inp["v_pool_i8"][page, row].astype(np.float64) * inp["v_scale_pool"][page, :, row][:, None])
    if not ks:
        Hkv, D = inp["k_pool_i8"].shape[2:]
        return np.zeros((0, Hkv, D)), np.zeros((0, Hkv, D))
    return np.stack(ks), np.stack(vs)


def decode_int8(inp: dict, rows: Optional[Iterable[Tuple[int, int]]] = None) -> np.ndarray:
    """fp64 decode over an int8 KV cache (single query token per sequence): the
    attention definition with K, V the dequantized values.  Returns [B, Hq, D], or
    [n, D] for the selected (b, h) rows."""
    q = inp["q"]
    B, Hq, D = q.shape
    Hkv = (inp["k_i8"] if "k_i8" in inp else inp["k_pool_i8"]).shape[2]
    G = Hq // Hkv
    want = [(b, h) for b in range(B) for h in range(Hq)] if rows is None else list(rows)
    res = np.zeros((len(want), D))
    cache = {}
    for n, (b, h) in enumerate(want):
        L = int(inp["seq_lens"][b])
        if L == 0:
            continue
        if b not in cache:
            cache = {b: dequant_rows(inp, b, L)}
        K, V = cache[b]
        res[n] = attend(widen_bf16(q[b, h])[None], K[:, h // G], V[:, h // G], inp["scale"])[0]
    return res.reshape(B, Hq, D) if rows is None else res
