"""GPU parity of multi-query decode (speculative verification: q_len new tokens per
sequence, causal within the block) through the C ABI, against the CPU oracle."""
import math

import numpy as np
import pytest

import oracle
from gqa_split_kv_gb300.workloads import contig_to_paged, f32_to_bf16_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_helpers import check_out, check_plan_partials, run_multi  # noqa: E402

RAGGED = [1, 7, 15, 16, 17, 100, 300, 777]


def multi_case(seed, B, Hq, Hkv, D, qlen, ctx, lens):
    rng = np.random.default_rng(seed)
    return dict(q=f32_to_bf16_bits(rng.standard_normal((B, Hq, qlen, D), dtype=np.float32)),
                k=f32_to_bf16_bits(rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32)),
                v=f32_to_bf16_bits(rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32)),
                seq_lens=np.asarray(lens, np.int32), scale=float(np.float32(1 / math.sqrt(D))))


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv,qlen", [(8, 2, 2), (24, 4, 7), (16, 2, 4), (16, 2, 8), (4, 4, 8), (24, 4, 1)])
def test_multi_contig_matches_oracle(D, Hq, Hkv, qlen):
    inp = multi_case(D + 10 * qlen + Hq, len(RAGGED), Hq, Hkv, D, qlen, ctx=max(RAGGED), lens=RAGGED)
    ref = oracle.decode_multi(inp)
    checked = 0
    for S in (None, 1, 5, 40):
        out, acc, ml, S_used = run_multi(inp, S)
        check_out(out, ref, f"D={D} G={Hq // Hkv} q_len={qlen} S={S_used}")
        # queries that see no token (sequence shorter than the block) are zero
        for b, L in enumerate(RAGGED):
            for i in range(qlen):
                if oracle.visible_tokens(L, qlen, i) == 0:
                    assert np.all(out[b, :, i] == 0)
        if S_used >= 2:
            checked += check_plan_partials(acc, ml, inp, S_used, what=f"multi D={D} q_len={qlen}")
    assert checked > 0


def test_multi_with_one_query_token_is_plain_decode_bitwise():
    inp = multi_case(5, 4, 16, 4, 128, 1, ctx=900, lens=[900, 33, 1, 500])
    single = dict(inp, q=np.ascontiguousarray(inp["q"][:, :, 0]))
    from gpu_helpers import run
    for S in (1, 6, 20):
        m_out = run_multi(inp, S)[0][:, :, 0]
        s_out = run(single, S)[0]
        assert np.array_equal(m_out, s_out)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("ps", [16, 32, 64])
def test_multi_paged_matches_contiguous_bitwise(D, ps):
    inp = multi_case(ps + D, len(RAGGED), 32, 8, D, 4, ctx=max(RAGGED), lens=RAGGED)
    rng = np.random.default_rng(ps + 1)
    kp, vp, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], ps, rng, spare_pages=2)
    pin = dict(q=inp["q"], k_pool=kp, v_pool=vp, page_table=table, seq_lens=inp["seq_lens"], page_size=ps,
               scale=inp["scale"])
    ref = oracle.decode_multi(pin)
    for S in (None, 1, 7):
        out_c, acc_c, ml_c, S_used = run_multi(inp, S)
        out_p, acc_p, ml_p, _ = run_multi(pin, S_used, max_seq_len=max(RAGGED))
        check_out(out_p, ref, f"paged D={D} ps={ps} S={S_used}")
        assert np.array_equal(out_p, out_c)
        if S_used >= 2:
            check_plan_partials(acc_p, ml_p, pin, S_used, max_seq_len=max(RAGGED), what=f"multi paged D={D}")
        used = ~np.isnan(ml_c[..., 1])
        assert np.array_equal(acc_p[used], acc_c[used]) and np.array_equal(ml_p[used], ml_c[used])


def test_multi_deterministic():
    inp = multi_case(9, 3, 24, 4, 256, 7, ctx=2000, lens=[2000, 1500, 5])
    first = run_multi(inp)
    for _ in range(2):
        again = run_multi(inp)
        assert np.array_equal(first[0], again[0])
        assert np.array_equal(first[1], again[1], equal_nan=True)
