"""Full-size parity: every benchmark workload at its full size, in the launch
configuration bench.py times (the planner's split count), checked on sampled
outputs the oracle computes one by one, on the partials of sampled
multi-piece segments, and for bitwise run-to-run determinism."""
import numpy as np
import pytest

import oracle
from gqa_split_kv_gb300.workloads import WORKLOADS, make_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_helpers import OUT_ATOL, OUT_RTOL, PART_RTOL, run, run_int8, run_multi, to_device  # noqa: E402
from gqa_split_kv_gb300.workloads import bf16_bits_to_f32  # noqa: E402

N_ROWS = 24       # sampled (b, query head) outputs per workload
N_SEGMENTS = 3    # sampled multi-piece segments whose partials are checked


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
    # sampled outputs, one by one against the oracle
    rng = np.random.default_rng(4242)
    pairs = _sample_rows(inp, rng)
    ref = oracle.decode_rows(inp, pairs)
    got = np.stack([bf16_bits_to_f32(out[b, h]).astype(np.float64) for b, h in pairs])
    err = np.abs(got - ref)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref)), f"{name}: max abs err {err.max():.3e}"
    # partials of sampled segments cut into several pieces, at the same plan
    if S >= 2:
        G = wl.Hq // wl.Hkv
        pieces = [pc for pc in oracle.split_pieces(inp["seq_lens"], wl.Hkv, G, S, oracle.piece_gap_blocks(wl.D),
                                                    oracle.groups_per_pass(G, wl.D)) if pc["npieces"] >= 2]
        if pieces:
            segs = sorted({(pc["b"], pc["u"]) for pc in pieces})
            chosen = [segs[i] for i in rng.choice(len(segs), size=min(N_SEGMENTS, len(segs)), replace=False)]
            for pc in pieces:
                if (pc["b"], pc["u"]) not in chosen:
                    continue
                b, h = pc["b"], pc["h"]
                first, count = pc["group"]
                heads = list(range(h * G + first, h * G + first + count))
                L = int(inp["seq_lens"][b])
                if "k" in inp:
                    K, V = inp["k"][b, pc["t0"]:pc["t1"], h], inp["v"][b, pc["t0"]:pc["t1"], h]
                else:
                    K = oracle.gather_paged(inp["k_pool"], inp["page_table"], b, L, inp["page_size"])[pc["t0"]:pc["t1"], h]
                    V = oracle.gather_paged(inp["v_pool"], inp["page_table"], b, L, inp["page_size"])[pc["t0"]:pc["t1"], h]
                a, m, l = oracle.attend_partial(oracle.widen_bf16(inp["q"][b, heads]), oracle.widen_bf16(K),
                                                oracle.widen_bf16(V), inp["scale"])
                for r, hq in enumerate(heads):
                    j = pc["piece"]
                    assert abs(ml[b, hq, j, 0] - m[r]) <= PART_RTOL * max(1.0, abs(m[r]))
                    assert abs(ml[b, hq, j, 1] - l[r]) <= PART_RTOL * l[r]
                    assert np.abs(acc[b, hq, j].astype(np.float64) - a[r]).max() <= PART_RTOL * np.abs(a[r]).max()
    # the same launch again: identical bits
    out2, *_ = run(inp, S, dev_inputs=d, max_seq_len=max_len if "k_pool" in inp else None)
    assert np.array_equal(out, out2)
