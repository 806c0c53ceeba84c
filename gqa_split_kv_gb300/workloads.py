"""Seeded synthetic inputs for split-KV GQA decode attention.

This module only draws and lays out numbers.  It holds none of the attention
arithmetic, so both the CPU oracle and the CUDA library can be fed from it
without sharing any of the method's code.

Every tensor is drawn as float32 from a seeded ``numpy.random.Generator``
(PCG64) and rounded once to bfloat16 (round to nearest, ties to even) with
integer bit operations, so the oracle and the GPU see identical bits.

Workload shapes follow the decode shapes the source pages discuss: GQA-6 with
head_dim 256 at ctx 4096 ("perf(dspark): overlap KV staging with compute via
cp.async", section "Why there was still headroom"), paged caches resolved
through a page table (AstrAI commit 69fecaf, paged decode items), G=8 query
rows per KV head (AstrAI commit 988e013, scalar decode items) and head_dim
32/64/128/256 (same commit, dispatch items).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "draw_seq_lens",
    "make_inputs",
    "contig_to_paged",
    "quantize_int8_rows",
    "make_int8_cache",
    "int8_to_paged",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 bit patterns (ties to even).

    Input generation only: the inputs are defined as these bf16 values.
    Inputs are finite, so NaN handling is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic decode-attention problem.

    layout:      "contig" -> K/V are [B, max_ctx, Hkv, D];
                 "paged"  -> K/V pools are [num_pages, page_size, Hkv, D] with a
                 page table [B, max_pages_per_seq].
    lens:        "full" (every sequence has max_ctx tokens), "uniform" (integers in
                 [lens_lo, lens_hi]) or "loguniform" (floor(exp(U(0, ln lens_hi))),
                 clamped to [1, lens_hi]).
    outlier_frac: fraction of key rows (token positions, shared by all KV heads)
                 multiplied by ``outlier_mult`` before the bf16 rounding.
    """

    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    max_ctx: int
    layout: str = "contig"
    page_size: int = 0
    lens: str = "full"
    lens_lo: int = 0
    lens_hi: int = 0
    outlier_frac: float = 0.0
    outlier_mult: float = 20.0
    seed: int = 1234
    q_len: int = 1  # query tokens per sequence (> 1: multi-query decode, q is [B, Hq, q_len, D])
    kv_dtype: str = "bf16"  # "int8": symmetric int8 K/V with fp32 scales per (token, KV head)
    kind: str = "decode"    # "prefill": causal attention of the last q_len tokens, q is [B, q_len, Hq, D]

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return float(np.float32(1.0 / math.sqrt(self.D)))

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workload families of the decode configurations, plus two multi-query
# (verification) workloads; each name states its shape.
WORKLOADS = {
    "tiny_contig_b1_hq8_hkv2_d64_ctx512": Workload(
        "tiny_contig_b1_hq8_hkv2_d64_ctx512", B=1, Hq=8, Hkv=2, D=64, max_ctx=512, seed=1235),
    "gqa6_contig_b1_hq24_hkv4_d256_ctx4096": Workload(
        "gqa6_contig_b1_hq24_hkv4_d256_ctx4096", B=1, Hq=24, Hkv=4, D=256, max_ctx=4096, seed=1236),
    "gqa6_contig_b1_hq24_hkv4_d256_ctx16384": Workload(
        "gqa6_contig_b1_hq24_hkv4_d256_ctx16384", B=1, Hq=24, Hkv=4, D=256, max_ctx=16384, seed=1236),
    "paged_b16_hq32_hkv8_d128_u256_8192_ps32": Workload(
        "paged_b16_hq32_hkv8_d128_u256_8192_ps32", B=16, Hq=32, Hkv=8, D=128, max_ctx=8192,
        layout="paged", page_size=32, lens="uniform", lens_lo=256, lens_hi=8192, seed=1237),
    "long_contig_b1_hq32_hkv8_d128_ctx65536_outliers": Workload(
        "long_contig_b1_hq32_hkv8_d128_ctx65536_outliers", B=1, Hq=32, Hkv=8, D=128,
        max_ctx=65536, outlier_frac=0.001, seed=1238),
    "mixed_paged_b64_hq64_hkv8_d128_log1_32768_ps16": Workload(
        "mixed_paged_b64_hq64_hkv8_d128_log1_32768_ps16", B=64, Hq=64, Hkv=8, D=128,
        max_ctx=32768, layout="paged", page_size=16, lens="loguniform", lens_hi=32768, seed=1239),
    "sweep_contig_b64_hq64_hkv8_d32_ctx2048": Workload(
        "sweep_contig_b64_hq64_hkv8_d32_ctx2048", B=64, Hq=64, Hkv=8, D=32, max_ctx=2048, seed=1240),
    "sweep_contig_b64_hq64_hkv8_d64_ctx2048": Workload(
        "sweep_contig_b64_hq64_hkv8_d64_ctx2048", B=64, Hq=64, Hkv=8, D=64, max_ctx=2048, seed=1241),
    "sweep_paged_b64_hq64_hkv8_d64_ctx2048_ps16": Workload(
        "sweep_paged_b64_hq64_hkv8_d64_ctx2048_ps16", B=64, Hq=64, Hkv=8, D=64, max_ctx=2048,
        layout="paged", page_size=16, seed=1242),
    "sweep_paged_b64_hq64_hkv8_d32_ctx2048_ps16": Workload(
        "sweep_paged_b64_hq64_hkv8_d32_ctx2048_ps16", B=64, Hq=64, Hkv=8, D=32, max_ctx=2048,
        layout="paged", page_size=16, seed=1250),
    # multi-query decode (speculative verification of a draft block)
    "verify_contig_b1_hq24_hkv4_d256_ctx4096_q7": Workload(
        "verify_contig_b1_hq24_hkv4_d256_ctx4096_q7", B=1, Hq=24, Hkv=4, D=256, max_ctx=4096, q_len=7,
        seed=1243),
    "verify_paged_b16_hq32_hkv8_d128_u256_8192_ps32_q4": Workload(
        "verify_paged_b16_hq32_hkv8_d128_u256_8192_ps32_q4", B=16, Hq=32, Hkv=8, D=128, max_ctx=8192,
        layout="paged", page_size=32, lens="uniform", lens_lo=256, lens_hi=8192, q_len=4, seed=1244),
    # int8 KV cache (per (token, KV head) fp32 scales)
    "int8_long_contig_b1_hq32_hkv8_d128_ctx65536": Workload(
        "int8_long_contig_b1_hq32_hkv8_d128_ctx65536", B=1, Hq=32, Hkv=8, D=128, max_ctx=65536, kv_dtype="int8",
        seed=1245),
    "int8_paged_b16_hq32_hkv8_d128_u256_8192_ps32": Workload(
        "int8_paged_b16_hq32_hkv8_d128_u256_8192_ps32", B=16, Hq=32, Hkv=8, D=128, max_ctx=8192,
        layout="paged", page_size=32, lens="uniform", lens_lo=256, lens_hi=8192, kv_dtype="int8", seed=1246),
    # causal prefill: a full 4096-token prompt, a 1024-token chunk after 7168 cached
    # tokens (paged), and the GQA-6 head_dim 256 shape of the decode configurations
    "prefill_contig_b1_hq32_hkv8_d128_L4096": Workload(
        "prefill_contig_b1_hq32_hkv8_d128_L4096", B=1, Hq=32, Hkv=8, D=128, max_ctx=4096, q_len=4096,
        kind="prefill", seed=1247),
    "prefill_chunk_paged_b4_hq32_hkv8_d128_ctx8192_q1024_ps32": Workload(
        "prefill_chunk_paged_b4_hq32_hkv8_d128_ctx8192_q1024_ps32", B=4, Hq=32, Hkv=8, D=128, max_ctx=8192,
        layout="paged", page_size=32, q_len=1024, kind="prefill", seed=1248),
    "prefill_gqa6_contig_b1_hq24_hkv4_d256_L4096": Workload(
        "prefill_gqa6_contig_b1_hq24_hkv4_d256_L4096", B=1, Hq=24, Hkv=4, D=256, max_ctx=4096, q_len=4096,
        kind="prefill", seed=1249),
}


def draw_seq_lens(wl: Workload, rng: np.random.Generator) -> np.ndarray:
    if wl.lens == "full":
        return np.full(wl.B, wl.max_ctx, dtype=np.int32)
    if wl.lens == "uniform":
        return rng.integers(wl.lens_lo, wl.lens_hi + 1, size=wl.B).astype(np.int32)
    if wl.lens == "loguniform":
        u = rng.uniform(0.0, math.log(wl.lens_hi), size=wl.B)
        return np.clip(np.floor(np.exp(u)), 1, wl.lens_hi).astype(np.int32)
    raise ValueError(f"unknown length distribution {wl.lens!r}")


def workload_lens(wl: Workload) -> np.ndarray:
    """The sequence lengths make_inputs(wl) draws (its first draw from the seed)."""
    return draw_seq_lens(wl, np.random.default_rng(wl.seed))


def _normal_bf16(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    """N(0,1) float32 draws rounded to bf16 bits, generated in chunks to bound host memory."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(rng.standard_normal(e - s, dtype=np.float32))
    return out.reshape(shape)


def _outlier_keys(rng: np.random.Generator, shape, frac: float, mult: float, token_axis: int,
                  ntok: int) -> np.ndarray:
    """Key cache with round(frac * ntok) token rows (all KV heads) scaled by ``mult`` in fp32."""
    k32 = rng.standard_normal(int(np.prod(shape)), dtype=np.float32).reshape(shape)
    n_out = int(round(frac * ntok))
    pos = np.sort(rng.choice(ntok, size=n_out, replace=False))
    idx = [slice(None)] * len(shape)
    idx[token_axis] = pos
    k32[tuple(idx)] *= np.float32(mult)
    return f32_to_bf16_bits(k32), pos


def make_inputs(wl: Workload, seed: Optional[int] = None) -> dict:
    """Draw one problem.  Returns a dict of numpy arrays (bf16 as uint16 bits).

    Keys: q [B,Hq,D] ([B,Hq,q_len,D] when q_len > 1); seq_lens int32[B]; for "contig": k, v [B,max_ctx,Hkv,D];
    for "paged": k_pool, v_pool [num_pages,page_size,Hkv,D] and page_table
    int32[B,max_pages_per_seq] (unused entries are -1, never read); plus
    "scale" (float32 value 1/sqrt(D)) and "outlier_pos" when present.
    The pool holds exactly sum(ceil(L_b/page_size)) pages and the logical
    pages of all sequences are scattered over it by a random permutation.
    """
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    seq_lens = draw_seq_lens(wl, rng)
    if wl.kind == "prefill":  # token-major chunk queries
        q = _normal_bf16(rng, (wl.B, wl.q_len, wl.Hq, wl.D))
    else:
        q = _normal_bf16(rng, (wl.B, wl.Hq, wl.D) if wl.q_len == 1 else (wl.B, wl.Hq, wl.q_len, wl.D))
    out = {"q": q, "seq_lens": seq_lens, "scale": wl.scale}
    if wl.kv_dtype == "int8":  # keys k_i8, v_i8, k_scale, v_scale (or their page pools)
        cache = make_int8_cache(rng, wl.B, wl.max_ctx, wl.Hkv, wl.D)
        if wl.layout == "contig":
            out.update(cache)
        else:
            out.update(int8_to_paged(cache, seq_lens, wl.page_size, rng), page_size=wl.page_size)
        return out
    if wl.layout == "contig":
        shape = (wl.B, wl.max_ctx, wl.Hkv, wl.D)
        if wl.outlier_frac > 0:
            k, pos = _outlier_keys(rng, shape, wl.outlier_frac, wl.outlier_mult, 1, wl.max_ctx)
            out["outlier_pos"] = pos
        else:
            k = _normal_bf16(rng, shape)
        out["k"] = k
        out["v"] = _normal_bf16(rng, shape)
        return out
    if wl.layout != "paged":
        raise ValueError(f"unknown layout {wl.layout!r}")
    ps = wl.page_size
    npages_b = (seq_lens.astype(np.int64) + ps - 1) // ps
    num_pages = int(npages_b.sum())
    max_pages = (wl.max_ctx + ps - 1) // ps
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((wl.B, max_pages), -1, dtype=np.int32)
    cur = 0
    for b in range(wl.B):
        n = int(npages_b[b])
        table[b, :n] = perm[cur:cur + n]
        cur += n
    shape = (max(num_pages, 1), ps, wl.Hkv, wl.D)
    if wl.outlier_frac > 0:
        k, pos = _outlier_keys(rng, shape, wl.outlier_frac, wl.outlier_mult, 1, ps)
        out["outlier_pos"] = pos
    else:
        k = _normal_bf16(rng, shape)
    out.update(k_pool=k, v_pool=_normal_bf16(rng, shape), page_table=table, page_size=ps)
    return out


def contig_to_paged(k: np.ndarray, v: np.ndarray, seq_lens: np.ndarray, page_size: int,
                    rng: np.random.Generator, spare_pages: int = 0):
    """Scatter a contiguous cache into a shuffled page pool (same logical data).

    Returns (k_pool, v_pool, page_table).  Pool pages that no sequence uses
    (``spare_pages`` of them) are filled with NaN bit patterns so that a kernel
    reading a page it does not own produces a visible error.
    """
    B, max_ctx, Hkv, D = k.shape
    ps = page_size
    npages_b = (seq_lens.astype(np.int64) + ps - 1) // ps
    used = int(npages_b.sum())
    num_pages = used + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    max_pages = (max_ctx + ps - 1) // ps
    table = np.full((B, max_pages), -1, dtype=np.int32)
    kp = np.full((max(num_pages, 1), ps, Hkv, D), 0x7FC0, dtype=np.uint16)
    vp = np.full((max(num_pages, 1), ps, Hkv, D), 0x7FC0, dtype=np.uint16)
    cur = 0
    for b in range(B):
        L = int(seq_lens[b])
        for p in range(int(npages_b[b])):
            phys = int(perm[cur])
            cur += 1
            table[b, p] = phys
            t0, t1 = p * ps, min(L, (p + 1) * ps)
            kp[phys, : t1 - t0] = k[b, t0:t1]
            vp[phys, : t1 - t0] = v[b, t0:t1]
    return kp, vp, table


def quantize_int8_rows(x: np.ndarray):
    """Symmetric int8 quantization of the last axis: scale = max|x| / 127 per row
    (1 for an all-zero row), values rint(x / scale) clipped to [-127, 127].
    Returns (int8 values, float32 scales with the last axis dropped)."""
    x = x.astype(np.float32)
    amax = np.abs(x).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(127.0), np.float32(1.0)).astype(np.float32)
    q = np.clip(np.rint(x / scale[..., None]), -127, 127).astype(np.int8)
    return q, scale


def make_int8_cache(rng: np.random.Generator, B: int, ctx: int, Hkv: int, D: int):
    """A contiguous int8 KV cache from N(0, 1) values: k_i8, v_i8 [B, ctx, Hkv, D]
    and fp32 scales k_scale, v_scale stored head-major, [B, Hkv, ctx]."""
    out = {}
    for name in ("k", "v"):
        x = rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32)
        q, s = quantize_int8_rows(x)
        out[name + "_i8"] = q
        out[name + "_scale"] = np.ascontiguousarray(s.transpose(0, 2, 1))
    return out


def int8_to_paged(cache: dict, seq_lens: np.ndarray, page_size: int, rng: np.random.Generator,
                  spare_pages: int = 0):
    """Scatter a contiguous int8 cache (make_int8_cache) into a shuffled page pool.

    Returns dict(k_pool_i8, v_pool_i8 [num_pages, page_size, Hkv, D] int8,
    k_scale_pool, v_scale_pool [num_pages, Hkv, page_size] fp32, page_table).
    Pages no sequence uses carry NaN scales."""
    B, max_ctx, Hkv, D = cache["k_i8"].shape
    ps = page_size
    npages_b = (seq_lens.astype(np.int64) + ps - 1) // ps
    num_pages = int(npages_b.sum()) + spare_pages
    perm = rng.permutation(num_pages).astype(np.int32)
    table = np.full((B, (max_ctx + ps - 1) // ps), -1, dtype=np.int32)
    out = {n: np.zeros((max(num_pages, 1), ps, Hkv, D), np.int8) for n in ("k_pool_i8", "v_pool_i8")}
    for n in ("k_scale_pool", "v_scale_pool"):
        out[n] = np.full((max(num_pages, 1), Hkv, ps), np.nan, np.float32)
    cur = 0
    for b in range(B):
        L = int(seq_lens[b])
        for p in range(int(npages_b[b])):
            phys = int(perm[cur])
            cur += 1
            table[b, p] = phys
            t0, t1 = p * ps, min(L, (p + 1) * ps)
            out["k_pool_i8"][phys, : t1 - t0] = cache["k_i8"][b, t0:t1]
            out["v_pool_i8"][phys, : t1 - t0] = cache["v_i8"][b, t0:t1]
            out["k_scale_pool"][phys, :, : t1 - t0] = cache["k_scale"][b, :, t0:t1]
            out["v_scale_pool"][phys, :, : t1 - t0] = cache["v_scale"][b, :, t0:t1]
    out["page_table"] = table
    return out
