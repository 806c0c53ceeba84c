"""GPU parity of decode over an int8 KV cache (per (token, KV head) fp32 scales)
through the C ABI, against the CPU oracle."""
import math

import numpy as np
import pytest

import oracle
from gqa_split_kv_gb300.workloads import f32_to_bf16_bits, int8_to_paged, make_int8_cache

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_helpers import check_out, check_plan_partials, run_int8  # noqa: E402

RAGGED = [1, 15, 16, 17, 100, 300, 777]


def int8_case(seed, B, Hq, Hkv, D, ctx, lens):
    rng = np.random.default_rng(seed)
    inp = make_int8_cache(rng, B, ctx, Hkv, D)
    inp.update(q=f32_to_bf16_bits(rng.standard_normal((B, Hq, D), dtype=np.float32)),
               seq_lens=np.asarray(lens, np.int32), scale=float(np.float32(1 / math.sqrt(D))))
    return inp


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (24, 4), (16, 2), (4, 4), (24, 2)])
def test_int8_contig_matches_oracle(D, Hq, Hkv):
    inp = int8_case(D * 7 + Hq, len(RAGGED), Hq, Hkv, D, ctx=780, lens=RAGGED)
    ref = oracle.decode_int8(inp)
    checked = 0
    for S in (None, 1, 5, 40):
        out, acc, ml, S_used = run_int8(inp, S)
        check_out(out, ref, f"int8 D={D} G={Hq // Hkv} S={S_used}")
        if S_used >= 2:
            checked += check_plan_partials(acc, ml, inp, S_used, what=f"int8 D={D} S={S_used}")
    assert checked > 0


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("ps", [16, 32, 48, 64, 96])  # 48, 96: no shift, boxes of 16 / 32 rows
def test_int8_paged_matches_oracle_and_contiguous_bitwise(D, ps):
    inp = int8_case(3 * D + ps, len(RAGGED), 32, 8, D, ctx=780, lens=RAGGED)
    pin = dict(int8_to_paged(inp, inp["seq_lens"], ps, np.random.default_rng(ps), spare_pages=3),
               q=inp["q"], seq_lens=inp["seq_lens"], page_size=ps, scale=inp["scale"])
    ref = oracle.decode_int8(pin)
    for S in (None, 1, 4):
        out_c, acc_c, ml_c, S_used = run_int8(inp, S)
        out_p, acc_p, ml_p, _ = run_int8(pin, S_used, max_seq_len=780)
        check_out(out_p, ref, f"int8 paged D={D} ps={ps} S={S_used}")
        assert np.array_equal(out_p, out_c)
        used = ~np.isnan(ml_c[..., 1])
        assert np.array_equal(acc_p[used], acc_c[used]) and np.array_equal(ml_p[used], ml_c[used])


def test_int8_deterministic_and_edge_lengths():
    inp = int8_case(11, 4, 16, 2, 128, ctx=1200, lens=[1200, 0, 1, 640])
    ref = oracle.decode_int8(inp)
    first = run_int8(inp)
    check_out(first[0], ref, "int8 edges")
    assert np.all(first[0][1] == 0)
    for _ in range(2):
        assert np.array_equal(run_int8(inp)[0], first[0])


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("lens", [[512], [500, 512], [0, 9]])
def test_int8_small_batches_whose_lengths_differ_from_the_cache(D, lens):
    """The guessed first tiles of small contiguous batches (kept or drained) with an int8 cache."""
    inp = int8_case(41 + D + sum(lens), len(lens), 16, 4, D, ctx=512, lens=lens)
    ref = oracle.decode_int8(inp)
    for S in (None, 1, 5):
        out, acc, ml, S_used = run_int8(inp, S)
        check_out(out, ref, f"int8 D={D} lens={lens} S={S_used}")
        if S_used >= 2:
            check_plan_partials(acc, ml, inp, S_used, what=f"int8 D={D} lens={lens}")
