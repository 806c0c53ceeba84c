"""Pins of the causal prefill oracle against facts that do not come from the oracle
itself: torch's float64 SDPA with its causal mask, a long-double brute force with
no max subtraction, slices of a full prefill, multi-query decode (pinned on its
own), paged == contiguous, and planted off-by-one limits."""
import math

import numpy as np
import pytest

from oracle import decode_attention as od
from oracle import prefill_attention as op
from gqa_split_kv_gb300.workloads import contig_to_paged, f32_to_bf16_bits


def _case(seed, B, q_len, Hq, Hkv, D, ctx, lens):
    rng = np.random.default_rng(seed)
    return {
        "q": f32_to_bf16_bits(rng.standard_normal((B, q_len, Hq, D), dtype=np.float32)),
        "k": f32_to_bf16_bits(rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32)),
        "v": f32_to_bf16_bits(rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32)),
        "seq_lens": np.asarray(lens, np.int32),
        "scale": float(np.float32(1 / math.sqrt(D))),
    }


@pytest.mark.parametrize("G,Hkv,D", [(1, 2, 16), (4, 2, 32), (6, 1, 64)])
def test_full_prefill_matches_torch_sdpa_causal_float64(G, Hkv, D):
    torch = pytest.importorskip("torch")
    L = 37
    inp = _case(G * 10 + D, 1, L, G * Hkv, Hkv, D, L, [L])
    got = op.prefill(inp)
    q = torch.from_numpy(od.widen_bf16(inp["q"][0]).transpose(1, 0, 2))              # [Hq, L, D]
    k = torch.from_numpy(od.widen_bf16(inp["k"][0]).transpose(1, 0, 2)).repeat_interleave(G, 0)
    v = torch.from_numpy(od.widen_bf16(inp["v"][0]).transpose(1, 0, 2)).repeat_interleave(G, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=inp["scale"]).numpy()
    assert np.abs(got[0] - ref.transpose(1, 0, 2)).max() <= 1e-12


def _brute(inp):
    """Long-double softmax with explicit masks and no max subtraction (tiny values only)."""
    B, q_len, Hq, D = inp["q"].shape
    Hkv = inp["k"].shape[2]
    G = Hq // Hkv
    out = np.zeros((B, q_len, Hq, D))
    for b in range(B):
        L = int(inp["seq_lens"][b])
        for i in range(q_len):
            pos = L - q_len + i
            for h in range(Hq):
                num = np.zeros(D, dtype=np.longdouble)
                den = np.longdouble(0)
                for t in range(L):
                    if t > pos:
                        continue
                    s = np.longdouble(0)
                    for d in range(D):
                        s += np.longdouble(od.widen_bf16(inp["q"][b, i, h, d])) * \
                            np.longdouble(od.widen_bf16(inp["k"][b, t, h // G, d]))
                    w = np.exp(s * np.longdouble(inp["scale"]))
                    den += w
                    num += w * od.widen_bf16(inp["v"][b, t, h // G]).astype(np.longdouble)
                if den > 0:
                    out[b, i, h] = (num / den).astype(np.float64)
    return out


def test_matches_long_double_brute_force_with_ragged_chunks():
    # chunk of 5 over lengths 9 (chunk at 4..8), 5 (full prefill), 3 (two queries see nothing)
    inp = _case(7, 3, 5, 4, 2, 4, 9, [9, 5, 3])
    got = op.prefill(inp)
    assert np.abs(got - _brute(inp)).max() <= 1e-12
    assert np.all(got[2, :2] == 0.0)  # positions -2 and -1: no visible token


def test_chunks_are_rows_of_the_full_prefill():
    L, Hq, Hkv, D = 40, 6, 3, 16
    full = _case(11, 1, L, Hq, Hkv, D, L, [L])
    ref = op.prefill(full)
    for q0, q_len in [(0, 8), (13, 9), (31, 9), (39, 1)]:
        # the cache holds q0 + q_len tokens; the chunk is tokens q0 .. q0 + q_len - 1
        chunk = dict(full, q=full["q"][:, q0:q0 + q_len], seq_lens=np.array([q0 + q_len], np.int32))
        assert np.abs(op.prefill(chunk)[0] - ref[0, q0:q0 + q_len]).max() <= 1e-12


def test_small_chunks_equal_multi_query_decode():
    inp = _case(13, 3, 7, 8, 2, 32, 50, [50, 7, 20])
    multi = dict(inp, q=np.ascontiguousarray(inp["q"].transpose(0, 2, 1, 3)))  # [B, Hq, q_len, D]
    want = od.decode_multi(multi).transpose(0, 2, 1, 3)
    assert np.abs(op.prefill(inp) - want).max() <= 1e-12


def test_paged_equals_contiguous():
    inp = _case(17, 2, 6, 4, 2, 32, 64, [64, 23])
    rng = np.random.default_rng(3)
    k_pool, v_pool, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], 16, rng, spare_pages=2)
    paged = dict(k_pool=k_pool, v_pool=v_pool, page_table=table, q=inp["q"], seq_lens=inp["seq_lens"],
                 scale=inp["scale"], page_size=16)
    assert np.array_equal(op.prefill(paged), op.prefill(inp))


def test_selected_rows_equal_full_output():
    inp = _case(19, 2, 5, 6, 3, 16, 30, [30, 12])
    full = op.prefill(inp)
    rows = [(0, 4, 5), (1, 0, 0), (1, 3, 2)]
    assert np.array_equal(op.prefill(inp, rows), np.stack([full[b, i, h] for b, i, h in rows]))


def test_row_count():
    assert op.prefill_row_count([5], 5) == 15            # 1 + 2 + ... + 5
    assert op.prefill_row_count([9, 3], 5) == (5 + 6 + 7 + 8 + 9) + (0 + 0 + 1 + 2 + 3)


def test_planted_off_by_one_limits_are_caught(monkeypatch):
    inp = _case(23, 1, 6, 2, 1, 8, 10, [10])
    ref = _brute(inp)
    assert np.abs(op.prefill(inp) - ref).max() <= 1e-12
    good = op.visible_tokens
    for bad in (lambda L, n, i: good(L, n, i) + 1 if good(L, n, i) < L else good(L, n, i),
                lambda L, n, i: max(0, good(L, n, i) - 1)):
        with monkeypatch.context() as m:
            m.setattr(op, "visible_tokens", bad)
            assert np.abs(op.prefill(inp) - ref).max() > 1e-6


def test_bench_flop_count_matches_the_oracle_row_count():
    from gqa_split_kv_gb300.accounting import prefill_visible, prefill_work
    for lens, q_len in [([5], 5), ([9, 3], 5), ([205, 75, 40, 0], 75), ([4096], 4096), ([8192] * 4, 1024)]:
        assert prefill_visible(lens, q_len) == op.prefill_row_count(lens, q_len)
    w = prefill_work(1, 32, 8, 128, [4096], 4096)
    assert w["flops"] == 4 * 128 * 32 * (4096 * 4097 // 2)
