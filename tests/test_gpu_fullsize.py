"""Full-size parity: every benchmark workload at its full size, in the launch
configuration bench.py times (the planner's split count), checked on sampled
outputs the oracle computes one by one (whole KV-head groups), on every output
against a property that holds at any size (a softmax-weighted mean of V rows
lies between their smallest and largest value, per column), on the partials of
sampled multi-piece segments, and for bitwise run-to-run determinism."""
import numpy as np
import pytest

import oracle
from gqa_split_kv_gb300.workloads import WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_helpers import (OUT_ATOL, OUT_RTOL, check_plan_partials, run, run_int8, run_multi,  # noqa: E402
                         to_device)
from gqa_split_kv_gb300.workloads import bf16_bits_to_f32  # noqa: E402

N_ROWS = 24       # sampled (b, query head) outputs per workload (multi-query, int8)
N_GROUPS = 24     # sampled (b, KV head) groups, all G query heads each (decode)
N_SEGMENTS = 3    # sampled multi-piece segments whose partials are checked


def _v_rows(inp, b):
    """V rows [L, Hkv, D] of sequence b as float32."""
    L = int(inp["seq_lens"][b])
    if "v" in inp:
        bits = inp["v"][b, :L]
    else:
        ps = int(inp["page_size"])
        pages = inp["page_table"][b, :(L + ps - 1) // ps]
        bits = inp["v_pool"][pages].reshape(-1, *inp["v_pool"].shape[2:])[:L]
    return bf16_bits_to_f32(bits)


def _check_convex_bounds(inp, out_bits, G, name):
    """Every output row is a convex combination of its V rows: per column it lies
    between their smallest and largest value (an empty sequence gives zeros)."""
    out = bf16_bits_to_f32(out_bits).astype(np.float64)
    B, Hq, D = out.shape
    for b in range(B):
        if int(inp["seq_lens"][b]) == 0:
            assert np.all(out[b] == 0), (name, b)
            continue
        V = _v_rows(inp, b)
        lo = np.repeat(V.min(axis=0), G, axis=0).astype(np.float64)  # [Hq, D]
        hi = np.repeat(V.max(axis=0), G, axis=0).astype(np.float64)
        tol = OUT_ATOL + OUT_RTOL * np.maximum(np.abs(lo), np.abs(hi))
        assert np.all(out[b] >= lo - tol) and np.all(out[b] <= hi + tol), (name, b)


def _sample_rows(inp, rng):
    B, Hq, _ = inp["q"].shape
    lens = inp["seq_lens"]
    # always include the longest sequence and an empty or shortest one
    picks = {(int(np.argmax(lens)), 0), (int(np.argmin(lens)), Hq - 1)}
    want = min(N_ROWS, B * Hq)
    while len(picks) < want:
        picks.add((int(rng.integers(B)), int(rng.integers(Hq))))
    return sorted(picks)


def _full_size_multi(wl, inp, d):
    """Multi-query workloads: sampled (b, h, i) outputs against the oracle, and bitwise
    run-to-run determinism (partials are checked at parity sizes)."""
    max_len = wl.max_ctx if "k_pool" in inp else None
    out, acc, ml, S = run_multi(inp, None, max_seq_len=max_len, dev_inputs=d)
    assert np.all(np.isfinite(bf16_bits_to_f32(out)))
    rng = np.random.default_rng(4343)
    lens = inp["seq_lens"]
    picks = {(int(np.argmax(lens)), 0, wl.q_len - 1), (int(np.argmin(lens)), wl.Hq - 1, 0)}
    while len(picks) < min(N_ROWS, wl.B * wl.Hq * wl.q_len):
        picks.add((int(rng.integers(wl.B)), int(rng.integers(wl.Hq)), int(rng.integers(wl.q_len))))
    rows = sorted(picks)
    ref = oracle.decode_multi(inp, rows)
    got = np.stack([bf16_bits_to_f32(out[b, h, i]).astype(np.float64) for b, h, i in rows])
    err = np.abs(got - ref)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref)), f"{wl.name}: max abs err {err.max():.3e}"
    if S >= 2:
        check_plan_partials(acc, ml, inp, S, max_seq_len=max_len, segments=2, rng=rng, what=wl.name)
    out2, *_ = run_multi(inp, S, max_seq_len=max_len, dev_inputs=d)
    assert np.array_equal(out, out2)


def _full_size_int8(wl, inp):
    """int8-cache workloads: sampled outputs against the oracle, and bitwise run-to-run
    determinism (partials are checked at parity sizes)."""
    max_len = wl.max_ctx if wl.layout == "paged" else None
    out, acc, ml, S = run_int8(inp, None, max_seq_len=max_len)
    assert np.all(np.isfinite(bf16_bits_to_f32(out)))
    pairs = _sample_rows(inp, np.random.default_rng(4444))
    ref = oracle.decode_int8(inp, pairs)
    got = np.stack([bf16_bits_to_f32(out[b, h]).astype(np.float64) for b, h in pairs])
    err = np.abs(got - ref)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref)), f"{wl.name}: max abs err {err.max():.3e}"
    if S >= 2:
        check_plan_partials(acc, ml, inp, S, max_seq_len=max_len, segments=2, rng=np.random.default_rng(4445),
                            what=wl.name)
    out2, *_ = run_int8(inp, S, max_seq_len=max_len)
    assert np.array_equal(out, out2)


def _full_size_prefill(wl, inp):
    """Causal prefill workloads: sampled (b, i, h) outputs against the oracle (a few
    query heads, each over the whole chunk) and bitwise run-to-run determinism."""
    from gqa_split_kv_gb300 import binding
    d = to_device(inp)
    out = torch.empty_like(d["q"])

    def call():
        if wl.layout == "paged":
            binding.prefill_attn_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"], wl.max_ctx,
                                       scale=inp["scale"], out=out)
        else:
            binding.prefill_attn_contig(d["q"], d["k"], d["v"], d["seq_lens"], scale=inp["scale"], out=out)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        return out.view(torch.int16).cpu().numpy().view(np.uint16).copy()

    got_bits = call()
    assert np.all(np.isfinite(bf16_bits_to_f32(got_bits)))
    rng = np.random.default_rng(4545)
    heads = [0, wl.Hq - 1, int(rng.integers(wl.Hq))]
    rows = sorted({(int(rng.integers(wl.B)), i, h) for h in heads
                   for i in [0, wl.q_len - 1] + [int(x) for x in rng.integers(wl.q_len, size=6)]})
    ref = oracle.prefill(inp, rows)
    got = np.stack([bf16_bits_to_f32(got_bits[b, i, h]).astype(np.float64) for b, i, h in rows])
    err = np.abs(got - ref)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref)), f"{wl.name}: max abs err {err.max():.3e}"
    assert np.array_equal(call(), got_bits)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_workload(name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl)
    if wl.kind == "prefill":
        return _full_size_prefill(wl, inp)
    if wl.kv_dtype == "int8":
        return _full_size_int8(wl, inp)
    d = to_device(inp)
    if wl.q_len > 1:
        return _full_size_multi(wl, inp, d)
    max_len = wl.max_ctx
    out, acc, ml, S = run(inp, None, dev_inputs=d, max_seq_len=max_len if "k_pool" in inp else None)
    assert np.all(np.isfinite(bf16_bits_to_f32(out)))
    # sampled whole KV-head groups, row by row against the oracle
    rng = np.random.default_rng(4242)
    G = wl.Hq // wl.Hkv
    lens = inp["seq_lens"]
    groups = {(int(np.argmax(lens)), 0), (int(np.argmin(lens)), wl.Hkv - 1)}
    while len(groups) < min(N_GROUPS, wl.B * wl.Hkv):
        groups.add((int(rng.integers(wl.B)), int(rng.integers(wl.Hkv))))
    pairs = [(b, g * G + i) for b, g in sorted(groups) for i in range(G)]
    ref = oracle.decode_rows(inp, pairs)
    got = np.stack([bf16_bits_to_f32(out[b, h]).astype(np.float64) for b, h in pairs])
    err = np.abs(got - ref)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref)), f"{name}: max abs err {err.max():.3e}"
    # every output row, against the convex-combination bounds
    _check_convex_bounds(inp, out, G, name)
    # partials of sampled segments cut into several pieces, at the same plan
    if S >= 2:
        check_plan_partials(acc, ml, inp, S, max_seq_len=max_len if "k_pool" in inp else None,
                            segments=N_SEGMENTS, rng=rng, what=name)
    # the same launch again: identical bits
    out2, *_ = run(inp, S, dev_inputs=d, max_seq_len=max_len if "k_pool" in inp else None)
    assert np.array_equal(out, out2)
