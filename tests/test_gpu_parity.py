"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by
element, on seeded inputs spanning several tiles, ragged tails and every
supported head_dim / group size, plus the bitwise determinism and
paged-vs-contiguous identities the split plan guarantees."""
import math

import numpy as np
import pytest

import oracle
from gqa_split_kv_gb300.workloads import Workload, contig_to_paged, f32_to_bf16_bits, make_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_helpers import check_out, check_plan_partials, run, to_device  # noqa: E402

RAGGED = [1, 15, 16, 17, 100, 300, 777]


def contig_case(seed, B, Hq, Hkv, D, ctx, lens=None, kstd=1.0):
    rng = np.random.default_rng(seed)
    q = f32_to_bf16_bits(rng.standard_normal((B, Hq, D), dtype=np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32) * np.float32(kstd))
    v = f32_to_bf16_bits(rng.standard_normal((B, ctx, Hkv, D), dtype=np.float32))
    seq = np.full(B, ctx, np.int32) if lens is None else np.asarray(lens, np.int32)
    return dict(q=q, k=k, v=v, seq_lens=seq, scale=float(np.float32(1 / math.sqrt(D))))


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (24, 4), (16, 2), (4, 4), (24, 2)])
def test_contig_matches_oracle(D, Hq, Hkv):
    inp = contig_case(D * 1000 + Hq, len(RAGGED), Hq, Hkv, D, ctx=max(RAGGED), lens=RAGGED)
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    checked = 0
    for S in (None, 1, 5, 40):
        out, acc, ml, S_used = run(inp, S)
        check_out(out, ref, f"D={D} G={Hq // Hkv} S={S_used}")
        if S_used >= 2:
            checked += check_plan_partials(acc, ml, inp, S_used, what=f"D={D} S={S_used}")
    assert checked > 0  # some segment was cut into several pieces


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("ps", [16, 32, 48, 64, 96])  # 48, 96: no shift, boxes of 16 / 32 rows
def test_paged_matches_oracle_and_contiguous_bitwise(D, ps):
    inp = contig_case(7 * D + ps, len(RAGGED), 32, 8, D, ctx=max(RAGGED), lens=RAGGED)
    rng = np.random.default_rng(ps)
    kp, vp, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], ps, rng, spare_pages=3)
    pin = dict(q=inp["q"], k_pool=kp, v_pool=vp, page_table=table, seq_lens=inp["seq_lens"], page_size=ps,
               scale=inp["scale"])
    ref = oracle.decode_paged(inp["q"], kp, vp, table, inp["seq_lens"], ps, inp["scale"])
    for S in (None, 1, 4):
        out_c, acc_c, ml_c, S_used = run(inp, S)
        out_p, acc_p, ml_p, _ = run(pin, S_used, max_seq_len=max(RAGGED))
        check_out(out_p, ref, f"paged D={D} ps={ps} S={S_used}")
        # same tokens, same plan, same order: identical bits
        assert np.array_equal(out_p, out_c)
        if S_used >= 2:
            check_plan_partials(acc_p, ml_p, pin, S_used, max_seq_len=max(RAGGED), what="paged")
            used = ~np.isnan(ml_c[..., 1])
            assert np.array_equal(acc_p[used], acc_c[used]) and np.array_equal(ml_p[used], ml_c[used])


@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("ps", [16, 64])
def test_paged_long_pieces_cycle_every_producer_warp(D, ps):
    # paged caches have two producer warps (four at D = 32) that issue the tiles of
    # a piece in turn; a 3001-token sequence in one piece (S = 1) gives each of them
    # many tiles and many passes over the stage ring, and the planner's split gives
    # pieces whose tile counts are not multiples of the producer count
    lens = [3001, 1, 2048, 700]
    inp = contig_case(11 * D + ps, len(lens), 16, 4, D, ctx=max(lens), lens=lens)
    rng = np.random.default_rng(D + ps)
    kp, vp, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], ps, rng, spare_pages=2)
    pin = dict(q=inp["q"], k_pool=kp, v_pool=vp, page_table=table, seq_lens=inp["seq_lens"], page_size=ps,
               scale=inp["scale"])
    ref = oracle.decode_paged(inp["q"], kp, vp, table, inp["seq_lens"], ps, inp["scale"])
    for S in (1, None):
        out_c, _, _, S_used = run(inp, S)
        out_p, _, _, _ = run(pin, S_used, max_seq_len=max(lens))
        check_out(out_p, ref, f"paged D={D} ps={ps} S={S_used}")
        assert np.array_equal(out_p, out_c)


def test_page_table_permutation_gives_identical_bits():
    inp = contig_case(5, 5, 16, 2, 128, ctx=700, lens=[700, 333, 64, 1, 519])
    rng = np.random.default_rng(1)
    outs = []
    for trial in range(3):
        kp, vp, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], 16, rng, spare_pages=trial * 5)
        pin = dict(q=inp["q"], k_pool=kp, v_pool=vp, page_table=table, seq_lens=inp["seq_lens"], page_size=16,
                   scale=inp["scale"])
        outs.append(run(pin, 6, max_seq_len=700)[0])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


@pytest.mark.parametrize("G", [9, 12, 16, 64])
def test_large_groups(G):
    inp = contig_case(G, 2, 2 * G, 2, 64, ctx=300, lens=[300, 77])
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    for S in (None, 1, 3):
        out, acc, ml, S_used = run(inp, S)
        check_out(out, ref, f"G={G}")
        if S_used >= 2:
            check_plan_partials(acc, ml, inp, S_used, what=f"G={G}")


def test_deterministic_across_runs():
    inp = contig_case(9, 3, 32, 8, 128, ctx=2000, lens=[2000, 1500, 37])
    d = to_device(inp)
    first = run(inp, None, dev_inputs=d)
    for _ in range(2):
        again = run(inp, None, dev_inputs=d)
        assert np.array_equal(first[0], again[0])
        assert np.array_equal(first[1], again[1], equal_nan=True)
        assert np.array_equal(first[2], again[2], equal_nan=True)


def test_null_seq_lens_means_full_context():
    inp = contig_case(10, 2, 8, 2, 64, ctx=200)
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    out, *_ = run(inp, None, lens_null=True)
    check_out(out, ref, "null seq_lens")


def test_empty_and_single_token_sequences():
    inp = contig_case(11, 4, 8, 2, 128, ctx=100, lens=[0, 1, 0, 100])
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    for S in (1, 2, 7):
        out, *_ = run(inp, S)
        check_out(out, ref, f"empty S={S}")
        assert np.all(out[0] == 0) and np.all(out[2] == 0)
        assert np.array_equal(out[1], inp["v"][1, 0][np.arange(8) // 4])  # one key: its V row


def test_lengths_beyond_the_cache_are_clamped():
    inp = contig_case(12, 2, 8, 2, 64, ctx=64, lens=[64, 64])
    inp_big = dict(inp, seq_lens=np.array([1000, -5], np.int32))
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], np.array([64, 0], np.int32), inp["scale"])
    out, *_ = run(inp_big, 3)
    check_out(out, ref, "clamped")


def test_outlier_keys_small():
    wl = Workload("o", B=1, Hq=32, Hkv=8, D=128, max_ctx=4096, outlier_frac=0.001, seed=77)
    inp = make_inputs(wl)
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    out, acc, ml, S = run(inp, None)
    check_out(out, ref, "outliers")
    assert check_plan_partials(acc, ml, inp, S, what="outliers") > 0


def test_combine_alone_matches_oracle_merge():
    rng = np.random.default_rng(13)
    inp = contig_case(13, 3, 8, 2, 64, ctx=900, lens=[900, 40, 0])
    S = 6
    # partials of arbitrary pieces (any partition merges to the same output)
    ranges = []
    for b, L in enumerate([900, 40, 0]):
        cuts = [0, *sorted(rng.integers(0, L + 1, size=S - 1).tolist()), L]
        ranges += [(b, 0, 8, j, cuts[j], cuts[j + 1]) for j in range(S)]
    ra, rm = oracle.range_partials(inp, ranges, S)
    acc = np.nan_to_num(ra, nan=0.0).astype(np.float32)
    ml = rm.copy()
    ml[..., 0] = np.where(np.isnan(ml[..., 0]), -np.inf, ml[..., 0])
    ml[..., 1] = np.nan_to_num(ml[..., 1], nan=0.0)
    ml = ml.astype(np.float32)
    want = oracle.combine_partials(acc.astype(np.float64), ml.astype(np.float64))
    from gqa_split_kv_gb300 import binding
    out = binding.decode_combine(torch.from_numpy(acc).cuda(), torch.from_numpy(ml).cuda())
    torch.cuda.synchronize()
    from gpu_helpers import host_bits
    check_out(host_bits(out), want, "combine")
    assert np.all(host_bits(out)[2] == 0)


def test_counters_are_reused_without_reset():
    """Segment counters are zeroed once; later calls (any shape) reuse them as they are."""
    from gqa_split_kv_gb300 import binding
    inp = contig_case(14, 3, 16, 4, 128, ctx=1500, lens=[1500, 900, 20])
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    ctr = torch.zeros(binding.counters_len(3, 16, 4), dtype=torch.int64, device="cuda")
    first = run(inp, 9, counters=ctr)[0]
    check_out(first, ref, "first")
    other = contig_case(15, 2, 16, 4, 128, ctx=700, lens=[700, 300])  # another shape on the same counters
    run(other, 5, counters=ctr)
    for _ in range(2):
        assert np.array_equal(run(inp, 9, counters=ctr)[0], first)
    # counters left with arbitrary values by someone else
    ctr.copy_(torch.randint(0, 2 ** 31, ctr.shape, device="cuda"))
    assert np.array_equal(run(inp, 9, counters=ctr)[0], first)


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """A wait that nothing completes (the diagnostic kernel's mbarrier) ends after its
    limit with the timeout bit set in the device error word; later calls still work."""
    import time

    from gqa_split_kv_gb300 import binding
    assert binding.device_error() == 0
    t0 = time.perf_counter()
    binding.selftest_bounded_wait(2_000_000)  # 2 ms
    assert binding.device_error() == 1        # bit 0: a bounded wait ran out (read and cleared)
    assert time.perf_counter() - t0 < 5.0
    assert binding.device_error() == 0
    inp = contig_case(16, 2, 8, 2, 64, ctx=300, lens=[300, 45])
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    check_out(run(inp, 3)[0], ref, "after the self-test")


def test_out_of_range_page_entry_is_flagged_not_followed():
    """A page-table entry outside the pool sets bit 2 of the device error word; the
    box is read from page 0 instead, so nothing outside the pool is read and the
    sequences whose entries are valid are still exact."""
    from gqa_split_kv_gb300 import binding
    inp = contig_case(17, 3, 16, 4, 128, ctx=300, lens=[300, 90, 200])
    rng = np.random.default_rng(17)
    kp, vp, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], 32, rng)
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    for bad in (-7, kp.shape[0], 1 << 30):
        t = table.copy()
        t[1, 1] = bad  # sequence 1, tokens 32..63
        pin = dict(q=inp["q"], k_pool=kp, v_pool=vp, page_table=t, seq_lens=inp["seq_lens"], page_size=32,
                   scale=inp["scale"])
        B, Hq, D = inp["q"].shape
        d = to_device(pin)
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
        binding.decode_attn_paged(d["q"], d["k_pool"], d["v_pool"], d["page_table"], d["seq_lens"], 300,
                                  scale=inp["scale"], splits=1, out=out)
        assert binding.device_error() == 4
        from gpu_helpers import host_bits
        got = host_bits(out)
        check_out(got[[0, 2]], ref[[0, 2]], "valid sequences beside a bad entry")
    assert binding.device_error() == 0


def test_kernels_write_nothing_outside_their_buffers():
    """Guard bands (canaries) around the output and partial buffers stay untouched."""
    from gqa_split_kv_gb300 import binding
    inp = contig_case(18, 4, 24, 4, 256, ctx=700, lens=[700, 1, 333, 0])
    B, Hq, D = inp["q"].shape
    d = to_device(inp)
    GUARD = 4096
    for S in (1, 6, 40):
        out_raw = torch.full((2 * GUARD + B * Hq * D,), -3.0, dtype=torch.bfloat16, device="cuda")
        acc_raw = torch.full((2 * GUARD + B * Hq * S * D,), 7.0, dtype=torch.float32, device="cuda")
        ml_raw = torch.full((2 * GUARD + B * Hq * S * 2,), 9.0, dtype=torch.float32, device="cuda")
        out = out_raw[GUARD:GUARD + B * Hq * D].view(B, Hq, D)
        acc = acc_raw[GUARD:GUARD + B * Hq * S * D].view(B, Hq, S, D)
        ml = ml_raw[GUARD:GUARD + B * Hq * S * 2].view(B, Hq, S, 2)
        binding.decode_attn_contig(d["q"], d["k"], d["v"], d["seq_lens"], scale=inp["scale"], splits=S,
                                   part_acc=acc, part_ml=ml, out=out)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        for raw, val in ((out_raw, -3.0), (acc_raw, 7.0), (ml_raw, 9.0)):
            assert torch.all(raw[:GUARD] == val) and torch.all(raw[-GUARD:] == val), S
        ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
        from gpu_helpers import host_bits
        check_out(host_bits(out), ref, f"canaries S={S}")


@pytest.mark.parametrize("S", [5, 40])
def test_cuda_graph_replays_are_exact(S):
    """A call captured in a CUDA graph carries one epoch for every replay; the
    segment counters still restart at zero each replay (the completing piece resets
    them), so in-kernel merges (S=5) and the combine path (S=40) stay exact."""
    from gqa_split_kv_gb300 import binding
    from gpu_helpers import host_bits
    inp = contig_case(19, 3, 16, 4, 128, ctx=1500, lens=[1500, 900, 40])
    B, Hq, D = inp["q"].shape
    d = to_device(inp)
    acc = torch.empty((B, Hq, S, D), dtype=torch.float32, device="cuda")
    ml = torch.empty((B, Hq, S, 2), dtype=torch.float32, device="cuda")
    ctr = torch.zeros(binding.counters_len(B, Hq, 4), dtype=torch.int64, device="cuda")
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device="cuda")
    q = d["q"].clone()

    def call():
        binding.decode_attn_contig(q, d["k"], d["v"], d["seq_lens"], scale=inp["scale"], splits=S, part_acc=acc,
                                   part_ml=ml, seg_counters=ctr, out=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()  # first call outside capture: device attributes and kernel attributes are set here
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    rng = np.random.default_rng(19)
    for rep in range(4):
        qbits = f32_to_bf16_bits(rng.standard_normal((B, Hq, D), dtype=np.float32))
        q.copy_(torch.from_numpy(qbits.view(np.int16)).cuda().view(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        ref = oracle.decode_contig(qbits, inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
        check_out(host_bits(out), ref, f"graph replay {rep} S={S}")


@pytest.mark.parametrize("D,paged", [(128, False), (64, True)])
def test_batch_at_the_limit_and_past_it(D, paged):
    """The plan keeps 8 bytes per sequence in shared memory: decode_max_batch
    sequences run and match the oracle; one more returns DA_ERR_UNSUPPORTED and
    launches nothing (the output stays untouched)."""
    from gqa_split_kv_gb300 import binding
    Bmax = binding.max_batch(8, 2, D, paged=paged)
    rng = np.random.default_rng(D + paged)
    lens = rng.integers(0, 33, size=Bmax + 1).astype(np.int32)
    inp = contig_case(21 + D, Bmax + 1, 8, 2, D, ctx=32, lens=lens)
    if paged:
        kp, vp, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], 16, rng, spare_pages=1)
        inp = dict(q=inp["q"], k_pool=kp, v_pool=vp, page_table=table, seq_lens=inp["seq_lens"], page_size=16,
                   scale=inp["scale"])
    cut = {k: (v[:Bmax] if k in ("q", "k", "v", "seq_lens", "page_table") else v) for k, v in inp.items()}
    ref = oracle.decode_paged(cut["q"], kp, vp, cut["page_table"], cut["seq_lens"], 16, inp["scale"]) if paged \
        else oracle.decode_contig(cut["q"], cut["k"], cut["v"], cut["seq_lens"], cut["scale"])
    out, *_ = run(cut, None, max_seq_len=32 if paged else None)
    check_out(out, ref, f"B={Bmax}")
    with pytest.raises(binding.DecodeAttnError) as e:
        run(inp, None, max_seq_len=32 if paged else None)
    assert e.value.status == 2


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("lens", [[700], [699, 700], [640, 1], [0, 700, 33, 700], [5]])
def test_small_batches_whose_lengths_differ_from_the_cache(D, lens):
    """Small contiguous batches start their first tiles from a guess (every sequence
    max_ctx tokens) before seq_lens is read; the plan then keeps or drains them.
    Lengths that match the guess, and lengths that do not, against the oracle."""
    inp = contig_case(31 + D + sum(lens), len(lens), 24, 4, D, ctx=700, lens=lens)
    ref = oracle.decode_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["scale"])
    d = to_device(inp)
    for S in (None, 1, 3, 9):
        out, acc, ml, S_used = run(inp, S, dev_inputs=d)
        check_out(out, ref, f"D={D} lens={lens} S={S_used}")
        if S_used >= 2:
            check_plan_partials(acc, ml, inp, S_used, what=f"D={D} lens={lens}")
        assert np.array_equal(run(inp, S_used, dev_inputs=d)[0], out)
