"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
call the library through its C ABI, and compare with the CPU oracle.

Tolerances (decode-attention output is bf16, partials fp32):
  output:   |gpu - ref| <= 2e-2 + 2e-2 * |ref| elementwise, ref the unrounded fp64 oracle
  partials: m  |dm| <= 1e-4 * max(1, |m|);  l  |dl| <= 1e-4 * l;
            acc  max|d acc| <= 1e-4 * max|acc_ref| over each (b, h, piece) row
"""
import numpy as np
import torch

import oracle
from gqa_split_kv_gb300 import binding
from gqa_split_kv_gb300.workloads import bf16_bits_to_f32

OUT_ATOL = 2e-2
OUT_RTOL = 2e-2
PART_RTOL = 1e-4


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_i32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.int32)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def num_splits_for(inp: dict) -> int:
    q = inp["q"]
    Hkv = (inp["k"] if "k" in inp else inp["k_pool"]).shape[2]
    max_len = inp["k"].shape[1] if "k" in inp else inp["page_table"].shape[1] * inp["page_size"]
    return binding.num_splits(q.shape[0], Hkv, max_len, q.shape[2])


def run(inp: dict, S: int = None, lens_null: bool = False, dev_inputs: dict = None, max_seq_len: int = None,
        counters=None):
    """One library call on inp; returns (out bits, part_acc, part_ml, S) as numpy."""
    if S is None:
        S = num_splits_for(inp)
    d = dev_inputs if dev_inputs is not None else to_device(inp)
    B, Hq, D = inp["q"].shape
    acc = torch.full((B, Hq, max(S, 1), D), float("nan"), dtype=torch.float32, device="cuda")
    ml = torch.full((B, Hq, max(S, 1), 2), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    Hkv = (inp["k"] if "k" in inp else inp["k_pool"]).shape[2]
    ctr = counters if counters is not None else torch.zeros(binding.counters_len(B, Hq, Hkv), dtype=torch.int64,
                                                            device="cuda")
    if "k" in inp:
        binding.decode_attn_contig(d["q"], d["k"], d["v"], None if lens_null else d["seq_lens"], scale=inp["scale"],
                                   splits=S, part_acc=acc, part_ml=ml, seg_counters=ctr, out=out)
    else:
        msl = max_seq_len if max_seq_len is not None else inp["page_table"].shape[1] * inp["page_size"]
        binding.decode_attn_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"], msl,
                                  scale=inp["scale"], splits=S, part_acc=acc, part_ml=ml, seg_counters=ctr, out=out)
    torch.cuda.synchronize()
    assert binding.device_error() == 0, "a kernel gave up on a bounded wait"
    return host_bits(out), acc.cpu().numpy(), ml.cpu().numpy(), S


def to_device(inp: dict) -> dict:
    d = {"q": dev_bf16(inp["q"]), "seq_lens": dev_i32(inp["seq_lens"])}
    if "k" in inp:
        d["k"] = dev_bf16(inp["k"])
        d["v"] = dev_bf16(inp["v"])
    else:
        d["k_pool"] = dev_bf16(inp["k_pool"])
        d["v_pool"] = dev_bf16(inp["v_pool"])
        d["page_table"] = dev_i32(inp["page_table"])
    return d


def check_out(out_bits: np.ndarray, ref: np.ndarray, what: str = ""):
    got = bf16_bits_to_f32(out_bits).astype(np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > OUT_ATOL + OUT_RTOL * np.abs(ref)
    assert not bad.any(), (f"{what}: {bad.sum()} outputs out of tolerance, max abs err {err.max():.3e} "
                           f"at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def plan_max_len(inp: dict, max_seq_len: int = None) -> int:
    """The length cap a call on inp uses: max_ctx, or min(max_pages * page_size, max_seq_len)."""
    for name in ("k", "k_i8"):
        if name in inp:
            return int(inp[name].shape[1])
    cap = int(inp["page_table"].shape[1]) * int(inp["page_size"])
    return cap if max_seq_len is None else min(cap, int(max_seq_len))


def check_plan_partials(acc: np.ndarray, ml: np.ndarray, inp: dict, S: int, max_seq_len: int = None,
                        segments: int = None, rng=None, what: str = ""):
    """Every partial slot a call leaves filled, against the oracle's partials of the
    token range the slot holds.  The pieces come from the library's planner
    (decode_plan_pieces): any partition is correct, so the oracle is not told which
    one the library uses.  acc/ml are the call's buffers ([B, Hq(, q_len), S, ...]);
    segments: check only this many randomly chosen multi-piece segments."""
    q = inp["q"]
    B, Hq = q.shape[:2]
    qlen = q.shape[2] if q.ndim == 4 else 1
    D = q.shape[-1]
    Hkv = next(inp[n] for n in ("k", "k_pool", "k_i8", "k_pool_i8") if n in inp).shape[2]
    rec = binding.plan_pieces(inp["seq_lens"], Hq, Hkv, D, plan_max_len(inp, max_seq_len), S, q_len=qlen)
    rec = rec[rec[:, 8] > rec[:, 7]]  # slots that hold a partial when the call returns
    if segments is not None and len(rec):
        segs = sorted({(int(r[0]), int(r[1])) for r in rec})
        rng = rng if rng is not None else np.random.default_rng(0)
        keep = {segs[i] for i in rng.choice(len(segs), size=min(segments, len(segs)), replace=False)}
        rec = np.array([r for r in rec if (int(r[0]), int(r[1])) in keep]).reshape(-1, rec.shape[1])
    ranges = [(int(r[0]), int(r[1]), int(r[2]), int(r[3]), int(r[7]), int(r[8])) for r in rec]
    ref_acc, ref_ml = oracle.range_partials(inp, ranges, S)
    acc = acc.reshape(B, Hq * qlen, S, D)
    ml = ml.reshape(B, Hq * qlen, S, 2)
    checked = 0
    for b, row0, nrows, j, t0, t1 in ranges:
        for r in range(row0, row0 + nrows):
            m_ref, l_ref = ref_ml[b, r, j]
            m_got, l_got = ml[b, r, j]
            if l_ref == 0:  # a row that sees no token of this range
                assert m_got == -np.inf and l_got == 0 and np.all(acc[b, r, j] == 0), (what, b, r, j)
                continue
            assert abs(m_got - m_ref) <= PART_RTOL * max(1.0, abs(m_ref)), (what, b, r, j, m_got, m_ref)
            assert abs(l_got - l_ref) <= PART_RTOL * l_ref, (what, b, r, j, l_got, l_ref)
            da = np.abs(acc[b, r, j].astype(np.float64) - ref_acc[b, r, j]).max()
            assert da <= PART_RTOL * np.abs(ref_acc[b, r, j]).max(), (what, b, r, j, da)
            checked += 1
    return checked


def run_multi(inp, S=None, max_seq_len=None, dev_inputs=None):
    """One multi-query call (q [B, Hq, q_len, D]); returns (out bits, part_acc, part_ml, S) as numpy."""
    B, Hq, qlen, D = inp["q"].shape
    d = dev_inputs if dev_inputs is not None else to_device(inp)
    q = d["q"]
    if "k" in inp:
        Hkv, ctx = inp["k"].shape[2], inp["k"].shape[1]
    else:
        Hkv, ctx = inp["k_pool"].shape[2], max_seq_len
    S = binding.num_splits_multi(B, qlen, Hq, Hkv, ctx, D) if S is None else S
    acc = torch.full((B, Hq, qlen, S, D), float("nan"), dtype=torch.float32, device="cuda")
    ml = torch.full((B, Hq, qlen, S, 2), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full((B, Hq, qlen, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ctr = torch.zeros(binding.counters_len(B, Hq, Hkv, qlen), dtype=torch.int64, device="cuda")
    if "k" in inp:
        binding.decode_attn_multi_contig(q, d["k"], d["v"], d["seq_lens"],
                                         scale=inp["scale"], splits=S, part_acc=acc, part_ml=ml, seg_counters=ctr,
                                         out=out)
    else:
        binding.decode_attn_multi_paged(q, d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"], max_seq_len,
                                        scale=inp["scale"], splits=S, part_acc=acc, part_ml=ml, seg_counters=ctr,
                                        out=out)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return host_bits(out), acc.cpu().numpy(), ml.cpu().numpy(), S


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run_int8(inp, S=None, max_seq_len=None):
    """One int8-cache call (contiguous k_i8/v_i8/k_scale/v_scale or paged pools).
    Returns (out bits, part_acc, part_ml, S)."""
    B, Hq, D = inp["q"].shape
    q = dev_bf16(inp["q"])
    paged = "k_pool_i8" in inp
    Hkv = (inp["k_pool_i8"] if paged else inp["k_i8"]).shape[2]
    ctx = max_seq_len if paged else inp["k_i8"].shape[1]
    S = binding.num_splits_multi(B, 1, Hq, Hkv, ctx, D) if S is None else S
    acc = torch.full((B, Hq, S, D), float("nan"), dtype=torch.float32, device="cuda")
    ml = torch.full((B, Hq, S, 2), float("nan"), dtype=torch.float32, device="cuda")
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    ctr = torch.zeros(binding.counters_len(B, Hq, Hkv), dtype=torch.int64, device="cuda")
    if paged:
        binding.decode_attn_int8_paged(q, dev(inp["k_pool_i8"]), dev(inp["v_pool_i8"]), dev(inp["k_scale_pool"]),
                                       dev(inp["v_scale_pool"]), dev_i32(inp["page_table"]),
                                       dev_i32(inp["seq_lens"]), max_seq_len, scale=inp["scale"], splits=S,
                                       part_acc=acc, part_ml=ml, seg_counters=ctr, out=out)
    else:
        binding.decode_attn_int8_contig(q, dev(inp["k_i8"]), dev(inp["v_i8"]), dev(inp["k_scale"]),
                                        dev(inp["v_scale"]), dev_i32(inp["seq_lens"]), scale=inp["scale"], splits=S,
                                        part_acc=acc, part_ml=ml, seg_counters=ctr, out=out)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return host_bits(out), acc.cpu().numpy(), ml.cpu().numpy(), S
