"""GPU parity of causal prefill / chunked prefill through the C ABI against the
CPU oracle: element by element over several query blocks and key tiles with
ragged tails, full prefill, chunks longer than the cache, every head size and
several group sizes; paged == contiguous bitwise; run-to-run determinism; a bad
page-table entry flagged."""
import math

import numpy as np
import pytest

import oracle
from gqa_split_kv_gb300.workloads import bf16_bits_to_f32, contig_to_paged, f32_to_bf16_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_helpers import OUT_ATOL, OUT_RTOL, dev_bf16, dev_i32, host_bits  # noqa: E402
from gqa_split_kv_gb300 import binding  # noqa: E402


def prefill_case(seed, B, q_len, Hq, Hkv, D, ctx, lens):
    rng = np.random.default_rng(seed)
    return {
        "q": f32_to_bf16_bits(rng.standard_normal((B, q_len, Hq, D), dtype=np.float32)),
        "k": f32_to_bf16_bits(rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32)),
        "v": f32_to_bf16_bits(rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32)),
        "seq_lens": np.asarray(lens, np.int32),
        "scale": float(np.float32(1 / math.sqrt(D))),
    }


def run_prefill(inp, max_seq_len=None):
    q = dev_bf16(inp["q"])
    out = torch.full(q.shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    if "k_pool" in inp:
        binding.prefill_attn_paged(q, dev_bf16(inp["k_pool"]), dev_bf16(inp["v_pool"]), dev_i32(inp["page_table"]),
                                   dev_i32(inp["seq_lens"]), max_seq_len, scale=inp["scale"], out=out)
    else:
        binding.prefill_attn_contig(q, dev_bf16(inp["k"]), dev_bf16(inp["v"]), dev_i32(inp["seq_lens"]),
                                    scale=inp["scale"], out=out)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return host_bits(out)


def check(out_bits, ref, what):
    got = bf16_bits_to_f32(out_bits).astype(np.float64)
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - ref)
    bad = err > OUT_ATOL + OUT_RTOL * np.abs(ref)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, max abs err {err.max():.3e}"


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (24, 4), (16, 2)])
def test_prefill_matches_oracle(D, Hq, Hkv):
    # q_len 75 spans several query blocks (64 / G tokens each) with a ragged last one;
    # lengths: chunk after a prefix crossing key tiles, full prefill, chunk longer than
    # the cache (the first queries see nothing), and an empty sequence
    lens = [75 + 130, 75, 40, 0]
    inp = prefill_case(D + Hq, len(lens), 75, Hq, Hkv, D, 256, lens)
    check(run_prefill(inp), oracle.prefill(inp), f"D={D} G={Hq // Hkv}")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("scale", [-0.125, 0.0, 0.5])
def test_prefill_any_scale(D, scale):
    # the kernels take a positive scale into the exponent and the row maximum;
    # a negative or zero one is applied to the scores first: every sign is exact
    # to the oracle (zero: uniform weights over the visible keys)
    lens = [75 + 130, 75, 40]
    inp = prefill_case(7 * D + 3, len(lens), 75, 16, 4, D, 256, lens)
    inp["scale"] = scale
    check(run_prefill(inp), oracle.prefill(inp), f"D={D} scale={scale}")


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 2, 64), (64, 1, 32), (64, 1, 128)])
def test_prefill_large_groups(Hq, Hkv, D):
    # G = 16 (4 query tokens per block) and G = 64 (one token per block, all 64 rows)
    lens = [90, 33]
    inp = prefill_case(Hq + D, len(lens), 33, Hq, Hkv, D, 96, lens)
    check(run_prefill(inp), oracle.prefill(inp), f"G={Hq // Hkv} D={D}")


@pytest.mark.parametrize("D,ps", [(64, 16), (128, 32), (256, 64), (32, 48),
                                  # many page boxes per key tile, split over the two
                                  # producer warps; pages that are not powers of two
                                  (128, 16), (128, 48), (256, 16), (256, 96), (64, 96)])
def test_prefill_paged_equals_contiguous_bitwise(D, ps):
    lens = [300, 64, 17]
    inp = prefill_case(3 * D + ps, len(lens), 64, 16, 4, D, 320, lens)
    k_pool, v_pool, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], ps, np.random.default_rng(ps),
                                            spare_pages=3)
    paged = dict(inp, k_pool=k_pool, v_pool=v_pool, page_table=table, page_size=ps)
    del paged["k"], paged["v"]
    out_c = run_prefill(inp)
    out_p = run_prefill(paged, max_seq_len=320)
    check(out_p, oracle.prefill(paged), f"paged D={D} ps={ps}")
    assert np.array_equal(out_c, out_p)


def test_prefill_deterministic_and_long_chunk():
    # 1000-token chunk after a 1500-token prefix: 63 query blocks, up to 40 key tiles
    inp = prefill_case(99, 1, 1000, 32, 8, 128, 2500, [2500])
    a = run_prefill(inp)
    b = run_prefill(inp)
    assert np.array_equal(a, b)
    rows = [(0, i, h) for i in (0, 1, 63, 500, 998, 999) for h in (0, 5, 31)]
    ref = oracle.prefill(inp, rows)
    got = np.stack([bf16_bits_to_f32(a[0, i, h]).astype(np.float64) for _, i, h in rows])
    err = np.abs(got - ref)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref)), err.max()


def test_prefill_null_lengths_mean_full_cache():
    inp = prefill_case(5, 2, 40, 8, 2, 64, 100, [100, 100])
    q = dev_bf16(inp["q"])
    out = binding.prefill_attn_contig(q, dev_bf16(inp["k"]), dev_bf16(inp["v"]), None, scale=inp["scale"])
    torch.cuda.synchronize()
    check(host_bits(out), oracle.prefill(inp), "null seq_lens")


def test_prefill_bad_page_entry_is_flagged():
    lens = [200, 90]
    inp = prefill_case(7, 2, 32, 8, 2, 64, 256, lens)
    k_pool, v_pool, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], 16, np.random.default_rng(1))
    table = table.copy()
    table[0, 3] = 1 << 30  # sequence 0 reads a page outside the pool
    paged = dict(inp, k_pool=k_pool, v_pool=v_pool, page_table=table, page_size=16)
    q = dev_bf16(inp["q"])
    out = binding.prefill_attn_paged(q, dev_bf16(k_pool), dev_bf16(v_pool), dev_i32(table), dev_i32(inp["seq_lens"]),
                                     256, scale=inp["scale"])
    torch.cuda.synchronize()
    assert binding.device_error() == 4  # bit 2: an entry outside the pool (read and cleared)
    assert binding.device_error() == 0
    # the other sequence is unaffected
    ref = oracle.prefill(dict(paged, page_table=table), [(1, i, h) for i in range(32) for h in range(8)])
    got = bf16_bits_to_f32(host_bits(out)[1]).astype(np.float64).reshape(-1, 64)
    err = np.abs(got - ref)
    assert np.all(err <= OUT_ATOL + OUT_RTOL * np.abs(ref))


@pytest.mark.parametrize("D", [64, 128, 256])
def test_prefill_ignores_cache_rows_past_the_sequence(D):
    """Cache rows at or past a sequence's length may hold anything, NaN included:
    they are masked out of the scores and their V rows never reach the output."""
    lens = [300, 129, 64]
    inp = prefill_case(8 + D, 3, 64, 16, 4, D, 384, lens)
    ref = oracle.prefill(inp)
    for b, L in enumerate(lens):
        inp["k"][b, L:] = 0x7FC0  # bf16 quiet NaN
        inp["v"][b, L:] = 0x7FC0
    check(run_prefill(inp), ref, f"NaN past the sequence, D={D}")
    kp, vp, table = contig_to_paged(inp["k"], inp["v"], np.full(3, 384, np.int32), 32, np.random.default_rng(D))
    paged = dict(inp, k_pool=kp, v_pool=vp, page_table=table, page_size=32)
    check(run_prefill(paged, max_seq_len=384), ref, f"paged, NaN past the sequence, D={D}")
