"""Thin Python binding of libdecode_attn.so (argument marshalling only).

Every step of the attention runs in the library's CUDA kernels; this module
only checks tensor shapes and dtypes, allocates outputs and partial buffers
with PyTorch when the caller does not pass them, and forwards raw device
pointers and the current CUDA stream through the C ABI of
``include/decode_attn.h``.  There is no fallback: if the library is missing
or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from .build import LIB

__all__ = [
    "load",
    "DecodeAttnError",
    "num_splits",
    "num_splits_multi",
    "decode_attn_contig",
    "decode_attn_paged",
    "decode_attn_multi_contig",
    "decode_attn_multi_paged",
    "decode_attn_int8_contig",
    "decode_attn_int8_paged",
    "decode_combine",
    "device_error",
    "selftest_bounded_wait",
    "counters_len",
    "plan_pieces",
    "max_batch",
    "PIECE_FIELDS",
    "STATUS",
]

STATUS = {0: "DA_OK", 1: "DA_ERR_INVALID_ARG", 2: "DA_ERR_UNSUPPORTED", 3: "DA_ERR_WORKSPACE",
          4: "DA_ERR_CUDA", 5: "DA_ERR_TIMEOUT"}

_lib = None


class DecodeAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (built in-tree by gqa_split_kv_gb300.build); raises if it is absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built; run gqa_split_kv_gb300.build.build() (needs nvcc)")
    lib = ctypes.CDLL(p)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.decode_num_splits.argtypes = [i, i, i, i, i]
    lib.decode_num_splits.restype = i
    lib.decode_attn_contig.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, vp, vp]
    lib.decode_attn_contig.restype = i
    lib.decode_attn_paged.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, vp, vp, vp, vp]
    lib.decode_attn_paged.restype = i
    lib.decode_num_splits_multi.argtypes = [i, i, i, i, i, i, i]
    lib.decode_num_splits_multi.restype = i
    lib.decode_attn_multi_contig.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, vp, vp, vp, vp]
    lib.decode_attn_multi_contig.restype = i
    lib.decode_attn_multi_paged.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, i, vp, vp, vp, vp, vp]
    lib.decode_attn_multi_paged.restype = i
    lib.decode_attn_int8_contig.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, vp, vp, vp, vp]
    lib.decode_attn_int8_contig.restype = i
    lib.decode_attn_int8_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp, vp, vp, vp,
                                           vp]
    lib.decode_attn_int8_paged.restype = i
    lib.prefill_attn_contig.argtypes = [vp, vp, vp, vp, i, i, i, i, i, i, f, vp, vp]
    lib.prefill_attn_contig.restype = i
    lib.prefill_attn_paged.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, f, vp, vp]
    lib.prefill_attn_paged.restype = i
    lib.decode_combine.argtypes = [vp, vp, i, i, i, i, vp, vp]
    lib.decode_combine.restype = i
    lib.decode_status_string.argtypes = [i]
    lib.decode_status_string.restype = ctypes.c_char_p
    lib.decode_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.decode_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, vp]
    lib.decode_selftest_bounded_wait.restype = i
    lib.decode_device_error.restype = i
    lib.decode_plan_pieces.argtypes = [vp, i, i, i, i, i, i, i, vp, i, ctypes.POINTER(i)]
    lib.decode_plan_pieces.restype = i
    lib.decode_max_batch.argtypes = [i, i, i, i, i, i]
    lib.decode_max_batch.restype = i
    if path is None:
        _lib = lib
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise DecodeAttnError(fn, status)


def _need(t, name, dtype, ndim):
    import torch
    if t.dtype != dtype or t.dim() != ndim or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA {dtype} tensor with {ndim} dims, "
                         f"got {tuple(t.shape)} {t.dtype} on {t.device}")


def num_splits(batch: int, num_kv_heads: int, max_seq_len: int, head_dim: int, num_sms: int = 0) -> int:
    s = load().decode_num_splits(batch, num_kv_heads, max_seq_len, head_dim, num_sms)
    if s < 0:
        raise DecodeAttnError("decode_num_splits", -s)
    return s


def num_splits_multi(batch: int, q_len: int, num_q_heads: int, num_kv_heads: int, max_seq_len: int,
                     head_dim: int, num_sms: int = 0) -> int:
    """Split count that counts every pass over a KV head (multi-query or G > 8)."""
    s = load().decode_num_splits_multi(batch, q_len, num_q_heads, num_kv_heads, max_seq_len, head_dim, num_sms)
    if s < 0:
        raise DecodeAttnError("decode_num_splits_multi", -s)
    return s


# Fields of one decode_plan_pieces record.
PIECE_FIELDS = ("b", "row0", "nrows", "j", "npieces", "t0", "t1", "held_t0", "held_t1")


def plan_pieces(seq_lens, num_q_heads: int, num_kv_heads: int, head_dim: int, max_len: int, num_splits: int,
                q_len: int = 1):
    """The pieces a decode call computes (host only): an int32 array [n, 9] of
    PIECE_FIELDS records, in the order the library's planner walks them.

    seq_lens: host sequence lengths (a sequence of ints or an int array), or an int
    batch size meaning every sequence has max_len tokens."""
    import numpy as np
    lib = load()
    if isinstance(seq_lens, (int, np.integer)):
        batch, lens_ptr, keep = int(seq_lens), None, None
    else:
        keep = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
        batch, lens_ptr = int(keep.shape[0]), keep.ctypes.data_as(ctypes.c_void_p)
    count = ctypes.c_int(0)
    st = lib.decode_plan_pieces(lens_ptr, batch, q_len, num_q_heads, num_kv_heads, head_dim, max_len, num_splits,
                                None, 0, ctypes.byref(count))
    if st not in (0, 3):
        raise DecodeAttnError("decode_plan_pieces", st)
    rec = np.zeros((count.value, len(PIECE_FIELDS)), dtype=np.int32)
    st = lib.decode_plan_pieces(lens_ptr, batch, q_len, num_q_heads, num_kv_heads, head_dim, max_len, num_splits,
                                rec.ctypes.data_as(ctypes.c_void_p), count.value, ctypes.byref(count))
    _check("decode_plan_pieces", st)
    del keep
    return rec


def max_batch(num_q_heads: int, num_kv_heads: int, head_dim: int, q_len: int = 1, kv_int8: bool = False,
              paged: bool = False) -> int:
    """Largest batch the decode kernels accept for this shape (host only)."""
    m = load().decode_max_batch(q_len, num_q_heads, num_kv_heads, head_dim, int(kv_int8), int(paged))
    if m < 0:
        raise DecodeAttnError("decode_max_batch", -m)
    return m


def counters_len(batch: int, num_q_heads: int, num_kv_heads: int, q_len: int = 1) -> int:
    """Entries of the per-segment counter array: batch * Hkv * ceil(G * q_len / 8)."""
    G = num_q_heads // num_kv_heads * q_len
    return batch * num_kv_heads * ((G + 7) // 8)


def _workspace(B, Hq, Hkv, D, S, part_acc, part_ml, seg_counters, device):
    import torch
    if S >= 2:
        if part_acc is None:
            part_acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device=device)
        if part_ml is None:
            part_ml = torch.empty((B, Hq, S, 2), dtype=torch.float32, device=device)
        if seg_counters is None:
            seg_counters = torch.zeros(counters_len(B, Hq, Hkv), dtype=torch.int64, device=device)
    return part_acc, part_ml, seg_counters


def decode_attn_contig(q, k, v, seq_lens=None, scale: Optional[float] = None, splits: Optional[int] = None,
                       part_acc=None, part_ml=None, seg_counters=None, out=None, stream=None):
    """q [B,Hq,D], k/v [B,max_ctx,Hkv,D] bf16; seq_lens int32 [B] or None.  Returns out [B,Hq,D] bf16."""
    import torch
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    B, Hq, D = q.shape
    _, ctx, Hkv, _ = k.shape
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, 1)
    scale = D ** -0.5 if scale is None else float(scale)
    S = num_splits(B, Hkv, ctx, D) if splits is None else int(splits)
    part_acc, part_ml, seg_counters = _workspace(B, Hq, Hkv, D, S, part_acc, part_ml, seg_counters, q.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    st = load().decode_attn_contig(_ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, Hq, Hkv, D, ctx, scale, S,
                                   _ptr(part_acc), _ptr(part_ml), _ptr(seg_counters), _ptr(out), _stream(stream))
    _check("decode_attn_contig", st)
    return out


def decode_attn_paged(q, k_pool, v_pool, page_table, seq_lens, max_seq_len: int, scale: Optional[float] = None,
                      splits: Optional[int] = None, part_acc=None, part_ml=None, seg_counters=None, out=None,
                      stream=None):
    """q [B,Hq,D]; pools [num_pages,page_size,Hkv,D] bf16; page_table int32 [B,max_pages]; seq_lens int32 [B]."""
    import torch
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, D = q.shape
    num_pages, ps, Hkv, _ = k_pool.shape
    max_pages = page_table.shape[1]
    scale = D ** -0.5 if scale is None else float(scale)
    S = num_splits(B, Hkv, max_seq_len, D) if splits is None else int(splits)
    part_acc, part_ml, seg_counters = _workspace(B, Hq, Hkv, D, S, part_acc, part_ml, seg_counters, q.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    st = load().decode_attn_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), B, Hq, Hkv,
                                  D, ps, max_pages, num_pages, int(max_seq_len), scale, S, _ptr(part_acc),
                                  _ptr(part_ml), _ptr(seg_counters), _ptr(out), _stream(stream))
    _check("decode_attn_paged", st)
    return out


def _multi_workspace(B, Hq, qlen, Hkv, D, S, part_acc, part_ml, seg_counters, device):
    import torch
    if S >= 2:
        if part_acc is None:
            part_acc = torch.empty((B, Hq, qlen, S, D), dtype=torch.float32, device=device)
        if part_ml is None:
            part_ml = torch.empty((B, Hq, qlen, S, 2), dtype=torch.float32, device=device)
        if seg_counters is None:
            seg_counters = torch.zeros(counters_len(B, Hq, Hkv, qlen), dtype=torch.int64, device=device)
    return part_acc, part_ml, seg_counters


def decode_attn_multi_contig(q, k, v, seq_lens=None, scale: Optional[float] = None, splits: Optional[int] = None,
                             part_acc=None, part_ml=None, seg_counters=None, out=None, stream=None):
    """Multi-query decode: q [B,Hq,q_len,D]; k/v [B,max_ctx,Hkv,D] bf16; seq_lens int32 [B] or None.
    Query token i of sequence b sees its first seq_lens[b] - q_len + 1 + i tokens.  Returns out [B,Hq,q_len,D]."""
    import torch
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    B, Hq, qlen, D = q.shape
    _, ctx, Hkv, _ = k.shape
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, 1)
    scale = D ** -0.5 if scale is None else float(scale)
    S = num_splits_multi(B, qlen, Hq, Hkv, ctx, D) if splits is None else int(splits)
    part_acc, part_ml, seg_counters = _multi_workspace(B, Hq, qlen, Hkv, D, S, part_acc, part_ml, seg_counters,
                                                       q.device)
    if out is None:
        out = torch.empty((B, Hq, qlen, D), dtype=torch.bfloat16, device=q.device)
    st = load().decode_attn_multi_contig(_ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, qlen, Hq, Hkv, D, ctx, scale,
                                         S, _ptr(part_acc), _ptr(part_ml), _ptr(seg_counters), _ptr(out),
                                         _stream(stream))
    _check("decode_attn_multi_contig", st)
    return out


def decode_attn_multi_paged(q, k_pool, v_pool, page_table, seq_lens, max_seq_len: int,
                            scale: Optional[float] = None, splits: Optional[int] = None, part_acc=None, part_ml=None,
                            seg_counters=None, out=None, stream=None):
    """Multi-query decode over a paged cache: q [B,Hq,q_len,D]; pools [num_pages,page_size,Hkv,D] bf16."""
    import torch
    _need(q, "q", torch.bfloat16, 4)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, qlen, D = q.shape
    num_pages, ps, Hkv, _ = k_pool.shape
    max_pages = page_table.shape[1]
    scale = D ** -0.5 if scale is None else float(scale)
    S = num_splits_multi(B, qlen, Hq, Hkv, max_seq_len, D) if splits is None else int(splits)
    part_acc, part_ml, seg_counters = _multi_workspace(B, Hq, qlen, Hkv, D, S, part_acc, part_ml, seg_counters,
                                                       q.device)
    if out is None:
        out = torch.empty((B, Hq, qlen, D), dtype=torch.bfloat16, device=q.device)
    st = load().decode_attn_multi_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), B,
                                        qlen, Hq, Hkv, D, ps, max_pages, num_pages, int(max_seq_len), scale, S,
                                        _ptr(part_acc), _ptr(part_ml), _ptr(seg_counters), _ptr(out),
                                        _stream(stream))
    _check("decode_attn_multi_paged", st)
    return out


def decode_attn_int8_contig(q, k_i8, v_i8, k_scale, v_scale, seq_lens=None, scale: Optional[float] = None,
                            splits: Optional[int] = None, part_acc=None, part_ml=None, seg_counters=None, out=None,
                            stream=None):
    """Decode over an int8 cache: q [B,Hq,D] bf16; k_i8/v_i8 int8 [B,max_ctx,Hkv,D]; k_scale/v_scale fp32
    [B,Hkv,max_ctx] (K = k_i8 * k_scale per token and KV head).  Returns out [B,Hq,D] bf16."""
    import torch
    _need(q, "q", torch.bfloat16, 3)
    _need(k_i8, "k_i8", torch.int8, 4)
    _need(v_i8, "v_i8", torch.int8, 4)
    _need(k_scale, "k_scale", torch.float32, 3)
    _need(v_scale, "v_scale", torch.float32, 3)
    B, Hq, D = q.shape
    _, ctx, Hkv, _ = k_i8.shape
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, 1)
    scale = D ** -0.5 if scale is None else float(scale)
    S = num_splits_multi(B, 1, Hq, Hkv, ctx, D) if splits is None else int(splits)
    part_acc, part_ml, seg_counters = _workspace(B, Hq, Hkv, D, S, part_acc, part_ml, seg_counters, q.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    st = load().decode_attn_int8_contig(_ptr(q), _ptr(k_i8), _ptr(v_i8), _ptr(k_scale), _ptr(v_scale),
                                        _ptr(seq_lens), B, Hq, Hkv, D, ctx, scale, S, _ptr(part_acc), _ptr(part_ml),
                                        _ptr(seg_counters), _ptr(out), _stream(stream))
    _check("decode_attn_int8_contig", st)
    return out


def decode_attn_int8_paged(q, k_pool_i8, v_pool_i8, k_scale_pool, v_scale_pool, page_table, seq_lens,
                           max_seq_len: int, scale: Optional[float] = None, splits: Optional[int] = None,
                           part_acc=None, part_ml=None, seg_counters=None, out=None, stream=None):
    """Decode over a paged int8 cache: pools int8 [num_pages,page_size,Hkv,D], scale pools fp32
    [num_pages,Hkv,page_size]; page_table int32 [B,max_pages]; seq_lens int32 [B]."""
    import torch
    _need(q, "q", torch.bfloat16, 3)
    _need(k_pool_i8, "k_pool_i8", torch.int8, 4)
    _need(v_pool_i8, "v_pool_i8", torch.int8, 4)
    _need(k_scale_pool, "k_scale_pool", torch.float32, 3)
    _need(v_scale_pool, "v_scale_pool", torch.float32, 3)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, Hq, D = q.shape
    num_pages, ps, Hkv, _ = k_pool_i8.shape
    max_pages = page_table.shape[1]
    scale = D ** -0.5 if scale is None else float(scale)
    S = num_splits_multi(B, 1, Hq, Hkv, max_seq_len, D) if splits is None else int(splits)
    part_acc, part_ml, seg_counters = _workspace(B, Hq, Hkv, D, S, part_acc, part_ml, seg_counters, q.device)
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    st = load().decode_attn_int8_paged(_ptr(q), _ptr(k_pool_i8), _ptr(v_pool_i8), _ptr(k_scale_pool),
                                       _ptr(v_scale_pool), _ptr(page_table), _ptr(seq_lens), B, Hq, Hkv, D, ps,
                                       max_pages, num_pages, int(max_seq_len), scale, S, _ptr(part_acc),
                                       _ptr(part_ml), _ptr(seg_counters), _ptr(out), _stream(stream))
    _check("decode_attn_int8_paged", st)
    return out


def prefill_attn_contig(q, k, v, seq_lens=None, scale: Optional[float] = None, out=None, stream=None):
    """Causal prefill of the last q_len tokens: q [B, q_len, Hq, D] bf16 (token-major); k/v
    [B, max_ctx, Hkv, D] bf16; seq_lens int32 [B] (None: max_ctx each).  Returns out like q."""
    import torch
    _need(q, "q", torch.bfloat16, 4)
    _need(k, "k", torch.bfloat16, 4)
    _need(v, "v", torch.bfloat16, 4)
    B, q_len, Hq, D = q.shape
    _, ctx, Hkv, _ = k.shape
    if seq_lens is not None:
        _need(seq_lens, "seq_lens", torch.int32, 1)
    scale = D ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    st = load().prefill_attn_contig(_ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, q_len, Hq, Hkv, D, ctx, scale,
                                    _ptr(out), _stream(stream))
    _check("prefill_attn_contig", st)
    return out


def prefill_attn_paged(q, k_pool, v_pool, page_table, seq_lens, max_seq_len: int, scale: Optional[float] = None,
                       out=None, stream=None):
    """Causal prefill over a paged cache: pools [num_pages, page_size, Hkv, D] bf16, page_table
    int32 [B, max_pages], seq_lens int32 [B]; q/out [B, q_len, Hq, D] bf16."""
    import torch
    _need(q, "q", torch.bfloat16, 4)
    _need(k_pool, "k_pool", torch.bfloat16, 4)
    _need(v_pool, "v_pool", torch.bfloat16, 4)
    _need(page_table, "page_table", torch.int32, 2)
    _need(seq_lens, "seq_lens", torch.int32, 1)
    B, q_len, Hq, D = q.shape
    num_pages, ps, Hkv, _ = k_pool.shape
    scale = D ** -0.5 if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    st = load().prefill_attn_paged(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), B, q_len,
                                   Hq, Hkv, D, ps, page_table.shape[1], num_pages, int(max_seq_len), scale, _ptr(out),
                                   _stream(stream))
    _check("prefill_attn_paged", st)
    return out


def decode_combine(part_acc, part_ml, out=None, stream=None):
    """part_acc [B,Hq,S,D], part_ml [B,Hq,S,2] fp32 -> out [B,Hq,D] bf16."""
    import torch
    _need(part_acc, "part_acc", torch.float32, 4)
    _need(part_ml, "part_ml", torch.float32, 4)
    B, Hq, S, D = part_acc.shape
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=part_acc.device)
    st = load().decode_combine(_ptr(part_acc), _ptr(part_ml), B, Hq, D, S, _ptr(out), _stream(stream))
    _check("decode_combine", st)
    return out


def selftest_bounded_wait(timeout_ns: int, stream=None) -> None:
    """Enqueue the diagnostic kernel whose wait can never complete; it gives up
    after timeout_ns and sets bit 0 of the device error word (see device_error)."""
    st = load().decode_selftest_bounded_wait(int(timeout_ns), _stream(stream))
    if st != 0:
        raise DecodeAttnError("decode_selftest_bounded_wait", st)


def device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    flags = ctypes.c_uint(0)
    st = load().decode_device_error(_stream(stream), ctypes.byref(flags))
    if st not in (0, 5):
        raise DecodeAttnError("decode_device_error", st)
    return int(flags.value)
