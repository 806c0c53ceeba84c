"""Pins for the CPU oracle: closed forms, invariants, brute force and a library routine.

Each check is chosen so that a plausible mistake in the oracle (a dropped
normalisation, a wrong sign in the exponent, the wrong query-head -> KV-head
map, K and V swapped, a wrong page index, a wrong piece boundary, double
rounding to bf16) fails at least one of them; ``test_planted_mistakes_are_caught``
plants such mistakes in the oracle and checks that.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import decode_attention as od
from gqa_split_kv_gb300.workloads import Workload, contig_to_paged, f32_to_bf16_bits, make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand_bits(rng, shape, std=1.0):
    return f32_to_bf16_bits((rng.standard_normal(shape) * std).astype(np.float32))


def _contig_case(rng, B, Hq, Hkv, D, ctx, lens=None, kstd=1.0):
    q = _rand_bits(rng, (B, Hq, D))
    k = _rand_bits(rng, (B, ctx, Hkv, D), kstd)
    v = _rand_bits(rng, (B, ctx, Hkv, D))
    seq = np.full(B, ctx, np.int32) if lens is None else np.asarray(lens, np.int32)
    return dict(q=q, k=k, v=v, seq_lens=seq, scale=float(np.float32(1 / math.sqrt(D))))


# ------------------------------------------------------------ bf16 rounding

def _pos_finite_bf16():
    bits = np.arange(0x0000, 0x7F80, dtype=np.uint16)  # +0 .. largest finite
    return bits, od.widen_bf16(bits)


def test_round_to_bf16_fixes_every_grid_point():
    bits, vals = _pos_finite_bf16()
    assert np.array_equal(od.round_to_bf16(vals), bits)
    assert np.array_equal(od.round_to_bf16(-vals), bits | np.uint16(0x8000))


def test_round_to_bf16_midpoints_ties_to_even_and_nearest():
    bits, vals = _pos_finite_bf16()
    lo, hi = vals[:-1], vals[1:]
    mid = (lo + hi) / 2  # exact in fp64
    even = np.where(bits[:-1] % 2 == 0, bits[:-1], bits[1:])
    assert np.array_equal(od.round_to_bf16(mid), even)
    above = np.nextafter(mid, np.inf)
    below = np.nextafter(mid, -np.inf)
    assert np.array_equal(od.round_to_bf16(above), bits[1:])
    assert np.array_equal(od.round_to_bf16(below), bits[:-1])
    # past the largest finite value: the midpoint to 2**128 rounds to infinity
    top = float(vals[-1])
    assert od.round_to_bf16(np.array([top + 2.0 ** 119]))[0] == 0x7F80
    assert od.round_to_bf16(np.array([np.nextafter(top + 2.0 ** 119, 0)]))[0] == 0x7F7F


def test_round_to_bf16_matches_torch_on_float32_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(200000) * 10.0 ** rng.integers(-30, 30, 200000),
                        (od.widen_bf16(np.arange(1, 0x7F7F, 97, dtype=np.uint16)) * (1 + 2.0 ** -8))])
    x32 = x.astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(od.round_to_bf16(x32.astype(np.float64)), want)


# ---------------------------------------------------------- closed forms

@pytest.mark.parametrize("D,Hq,Hkv", [(32, 4, 1), (64, 8, 2), (128, 32, 8), (256, 24, 4)])
def test_single_key_returns_its_value_row(D, Hq, Hkv):
    rng = np.random.default_rng(D)
    inp = _contig_case(rng, 2, Hq, Hkv, D, ctx=5, lens=[1, 1])
    out = od.round_to_bf16(od.decode_contig(**inp))
    G = Hq // Hkv
    for b in range(2):
        for h in range(Hq):
            assert np.array_equal(out[b, h], inp["v"][b, 0, h // G])


def test_identical_keys_give_mean_of_values():
    rng = np.random.default_rng(3)
    inp = _contig_case(rng, 1, 6, 1, 64, ctx=37)
    inp["k"][:] = inp["k"][:, :1]
    out = od.decode_contig(**inp)
    mean = od.widen_bf16(inp["v"][0, :, 0]).mean(axis=0)
    assert np.allclose(out[0], mean[None], rtol=0, atol=1e-12)


def test_zero_scale_gives_mean_of_values():
    rng = np.random.default_rng(4)
    inp = _contig_case(rng, 2, 8, 2, 32, ctx=19, lens=[19, 7])
    inp["scale"] = 0.0
    out = od.decode_contig(**inp)
    for b, L in enumerate([19, 7]):
        for h in range(8):
            mean = od.widen_bf16(inp["v"][b, :L, h // 4]).mean(axis=0)
            assert np.allclose(out[b, h], mean, rtol=0, atol=1e-12)


def test_empty_sequence_gives_zeros():
    rng = np.random.default_rng(5)
    inp = _contig_case(rng, 2, 4, 2, 32, ctx=8, lens=[0, 8])
    out = od.decode_contig(**inp)
    assert np.all(out[0] == 0)
    assert np.any(out[1] != 0)


def test_hand_worked_example():
    """Two keys, scores (1, 0) for head 0 and (0, 0) for head 1 -> weights e/(e+1), 1/(e+1) and 1/2, 1/2."""
    one, zero = 0x3F80, 0x0000
    q = np.array([[[one, zero], [zero, zero]]], np.uint16)          # heads 0 and 1, D=2
    k = np.array([[[[one, zero]], [[zero, one]]]], np.uint16)        # tokens 0 and 1, one KV head
    v = f32_to_bf16_bits(np.array([[[[2.0, -1.0]], [[4.0, 3.0]]]], np.float32))
    out = od.decode_contig(q, k, v, np.array([2], np.int32), 1.0)
    e = math.e
    assert np.allclose(out[0, 0], [(2 * e + 4) / (e + 1), (-e + 3) / (e + 1)], atol=1e-15)
    assert np.allclose(out[0, 1], [3.0, 1.0], atol=1e-15)


# --------------------------------------------------------- brute force

def test_matches_high_precision_brute_force():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 40
    rng = np.random.default_rng(11)
    for trial in range(6):
        B, Hkv, G, D = 2, 2, 1 + trial % 3, 2 + trial % 3
        lens = [1 + (trial * 3) % 8, 8]
        inp = _contig_case(rng, B, G * Hkv, Hkv, D, ctx=8, lens=lens, kstd=3.0)
        inp["scale"] = 0.37
        out = od.decode_contig(**inp)
        qf = od.widen_bf16(inp["q"])
        kf = od.widen_bf16(inp["k"])
        vf = od.widen_bf16(inp["v"])
        for b in range(B):
            for h in range(G * Hkv):
                g = h // G
                w = [mpmath.exp(mpmath.mpf(0.37) * mpmath.fsum(mpmath.mpf(qf[b, h, d]) * mpmath.mpf(kf[b, t, g, d])
                                                            for d in range(D))) for t in range(lens[b])]
                den = mpmath.fsum(w)
                for d in range(D):
                    ref = mpmath.fsum(w[t] * mpmath.mpf(vf[b, t, g, d]) for t in range(lens[b])) / den
                    assert abs(float(ref) - out[b, h, d]) <= 1e-12 * max(1.0, abs(float(ref)))


def test_outlier_scores_stay_finite_and_exact():
    """Scores of magnitude ~100 (keys x20): the max subtraction keeps exp finite."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    rng = np.random.default_rng(12)
    inp = _contig_case(rng, 1, 2, 1, 16, ctx=12, kstd=20.0)
    inp["scale"] = 1.0
    out = od.decode_contig(**inp)
    assert np.all(np.isfinite(out))
    qf, kf, vf = (od.widen_bf16(inp[n]) for n in ("q", "k", "v"))
    for h in range(2):
        s = [mpmath.fsum(mpmath.mpf(qf[0, h, d]) * mpmath.mpf(kf[0, t, 0, d]) for d in range(16)) for t in range(12)]
        w = [mpmath.exp(x) for x in s]
        for d in range(16):
            ref = mpmath.fsum(w[t] * mpmath.mpf(vf[0, t, 0, d]) for t in range(12)) / mpmath.fsum(w)
            assert abs(float(ref) - out[0, h, d]) <= 1e-12 * max(1.0, abs(float(ref)))


# ------------------------------------------------------- library routine

@pytest.mark.parametrize("G,Hkv,D", [(1, 4, 64), (4, 2, 64), (6, 4, 256), (8, 8, 128), (12, 2, 32)])
def test_matches_torch_sdpa_float64(G, Hkv, D):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(G * 100 + D)
    lens = [33, 70, 1]
    inp = _contig_case(rng, 3, G * Hkv, Hkv, D, ctx=70, lens=lens)
    out = od.decode_contig(**inp)
    for b, L in enumerate(lens):
        q = torch.from_numpy(od.widen_bf16(inp["q"][b]))[None, :, None, :]                 # [1,Hq,1,D]
        k = torch.from_numpy(od.widen_bf16(inp["k"][b, :L])).permute(1, 0, 2)[None]        # [1,Hkv,L,D]
        v = torch.from_numpy(od.widen_bf16(inp["v"][b, :L])).permute(1, 0, 2)[None]
        k = k.repeat_interleave(G, dim=1)
        v = v.repeat_interleave(G, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=inp["scale"])[0, :, 0].numpy()
        assert np.allclose(out[b], ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------ invariants

def test_paged_matches_contiguous_and_ignores_page_order():
    rng = np.random.default_rng(21)
    lens = [1, 16, 17, 100, 63]
    inp = _contig_case(rng, 5, 8, 2, 64, ctx=100, lens=lens)
    ref = od.decode_contig(**inp)
    for ps, spare in [(16, 0), (32, 3), (1, 2), (64, 1)]:
        kp, vp, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], ps, rng, spare)
        got = od.decode_paged(inp["q"], kp, vp, table, inp["seq_lens"], ps, inp["scale"])
        assert np.array_equal(got, ref)
        # shuffle the physical pages again: same logical data, same bits out
        perm = rng.permutation(kp.shape[0])
        inv = np.argsort(perm)
        table2 = np.where(table >= 0, inv[np.maximum(table, 0)], -1).astype(np.int32)
        got2 = od.decode_paged(inp["q"], kp[perm], vp[perm], table2, inp["seq_lens"], ps, inp["scale"])
        assert np.array_equal(od.round_to_bf16(got2), od.round_to_bf16(ref))


def test_joint_token_permutation_invariance():
    rng = np.random.default_rng(22)
    inp = _contig_case(rng, 1, 8, 2, 128, ctx=90)
    ref = od.decode_contig(**inp)
    perm = rng.permutation(90)
    inp2 = dict(inp, k=inp["k"][:, perm], v=inp["v"][:, perm])
    assert np.allclose(od.decode_contig(**inp2), ref, rtol=0, atol=1e-12)


def test_linear_in_values():
    rng = np.random.default_rng(23)
    inp = _contig_case(rng, 2, 4, 1, 32, ctx=40, lens=[40, 9])
    v2 = _rand_bits(rng, inp["v"].shape)
    a = od.decode_contig(**inp)
    b = od.decode_contig(**dict(inp, v=v2))
    # v + v2 is not on the bf16 grid; the definition is linear in the widened values
    qf = inp["q"]
    both = np.zeros_like(a)
    for bb, L in enumerate([40, 9]):
        for h in range(4):
            K = od.widen_bf16(inp["k"][bb, :L, 0])
            V = od.widen_bf16(inp["v"][bb, :L, 0]) + od.widen_bf16(v2[bb, :L, 0])
            both[bb, h] = od.attend(od.widen_bf16(qf[bb, h])[None], K, V, inp["scale"])[0]
    assert np.allclose(both, a + b, rtol=0, atol=1e-12)


def test_single_group_is_per_head_attention():
    """G=1: every query head reads its own KV head (multi-head attention)."""
    rng = np.random.default_rng(24)
    inp = _contig_case(rng, 1, 4, 4, 64, ctx=30)
    out = od.decode_contig(**inp)
    for h in range(4):
        ref = od.attend(od.widen_bf16(inp["q"][0, h])[None], od.widen_bf16(inp["k"][0, :, h]),
                        od.widen_bf16(inp["v"][0, :, h]), inp["scale"])[0]
        assert np.array_equal(out[0, h], ref)


# ------------------------------------------- partials of arbitrary ranges
#
# The pages fix only caps on the split count; any partition of a row's tokens
# into pieces must merge back to the unsplit result.  These pins cut the token
# ranges at random places (pieces of any length, empty ones included), so they
# do not depend on the partition the library happens to use.

def _random_ranges(rng, lens, rows, S, group=1):
    """Random partitions of every (sequence, row group) token range into at most S
    pieces: [(b, row0, nrows, slot, t0, t1)], slots 0.. in token order."""
    out = []
    for b, L in enumerate(lens):
        for row0 in range(0, rows, group):
            n = int(rng.integers(1, S + 1))
            cuts = np.sort(rng.integers(0, L + 1, size=n - 1)) if L > 0 else np.zeros(n - 1, np.int64)
            edges = [0, *cuts.tolist(), L]
            for j in range(n):
                out.append((b, row0, min(group, rows - row0), j, edges[j], edges[j + 1]))
    return out


def _merge_rows(acc, ml, n_of):
    """Merge slots 0 .. n - 1 of every (b, r) with merge_partials."""
    B, R, S, D = acc.shape
    out = np.zeros((B, R, D))
    for b in range(B):
        for r in range(R):
            n = n_of[b, r]
            parts = [(acc[b, r, j][None], ml[b, r, j, :1], ml[b, r, j, 1:]) for j in range(n)]
            out[b, r] = od.merge_partials(parts)[0]
    return out


def _slot_counts(ranges, B, R):
    n = np.zeros((B, R), np.int64)
    for b, row0, nrows, j, t0, t1 in ranges:
        n[b, row0:row0 + nrows] = np.maximum(n[b, row0:row0 + nrows], j + 1)
    return n


def test_merge_of_partials_over_any_partition_equals_unsplit():
    rng = np.random.default_rng(33)
    lens = [5, 130, 64, 1000, 0]
    inp = _contig_case(rng, 5, 12, 2, 64, ctx=1000, lens=lens)
    ref = od.decode_contig(**inp)
    kp, vp, table = contig_to_paged(inp["k"], inp["v"], inp["seq_lens"], 32, rng, 2)
    pin = dict(q=inp["q"], k_pool=kp, v_pool=vp, page_table=table, seq_lens=inp["seq_lens"], scale=inp["scale"],
               page_size=32)
    for trial, S in enumerate((1, 2, 3, 5, 17, 39)):
        ranges = _random_ranges(rng, lens, 12, S, group=int(rng.choice([1, 3, 6])))
        for case in (inp, pin):
            acc, ml = od.range_partials(case, ranges, S)
            got = _merge_rows(acc, ml, _slot_counts(ranges, 5, 12))
            assert np.allclose(got, ref, rtol=0, atol=1e-12), (S, trial)


def test_range_partials_follow_their_definition():
    """acc / l of a range is attention over that range alone; m is its largest
    score; an empty range gives (0, -inf, 0)."""
    rng = np.random.default_rng(34)
    inp = _contig_case(rng, 1, 4, 1, 32, ctx=200)
    ranges = [(0, 0, 4, 0, 0, 64), (0, 1, 2, 1, 64, 77), (0, 3, 1, 2, 77, 200), (0, 0, 1, 3, 50, 50)]
    acc, ml = od.range_partials(inp, ranges, 4)
    qf, kf, vf = (od.widen_bf16(inp[n]) for n in ("q", "k", "v"))
    for b, row0, nrows, j, t0, t1 in ranges:
        for h in range(row0, row0 + nrows):
            if t1 == t0:
                assert ml[0, h, j, 0] == -np.inf and ml[0, h, j, 1] == 0 and np.all(acc[0, h, j] == 0)
                continue
            K, V = kf[0, t0:t1, 0], vf[0, t0:t1, 0]
            sc = K @ qf[0, h] * inp["scale"]
            assert ml[0, h, j, 0] == sc.max()
            assert np.allclose(ml[0, h, j, 1], np.exp(sc - sc.max()).sum(), rtol=1e-14)
            assert np.allclose(acc[0, h, j] / ml[0, h, j, 1], od.attend(qf[0, h][None], K, V, inp["scale"])[0],
                               atol=1e-13)
    assert np.isnan(acc[0, 2, 2]).all()  # slot 2 of row 2 was not asked for


def test_combine_skips_empty_slots():
    rng = np.random.default_rng(35)
    inp = _contig_case(rng, 2, 4, 1, 32, ctx=300, lens=[300, 40])
    ranges = _random_ranges(rng, [300, 40], 4, 6)
    acc, ml = od.range_partials(inp, ranges, 6)
    acc = np.nan_to_num(acc, nan=0.0)
    ml[..., 0] = np.where(np.isnan(ml[..., 0]), -np.inf, ml[..., 0])
    ml[..., 1] = np.nan_to_num(ml[..., 1], nan=0.0)
    out = od.combine_partials(acc, ml)
    assert np.allclose(out, od.decode_contig(**inp), rtol=0, atol=1e-12)


# --------------------------------------------------- planted mistakes

def _pins(monkey_od):
    """A small battery of the checks above, run against a (possibly mutated) oracle."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(99)
    inp = _contig_case(rng, 2, 6, 2, 16, ctx=200, lens=[200, 11], kstd=2.0)
    out = monkey_od.decode_contig(**inp)
    for b, L in enumerate([200, 11]):
        q = torch.from_numpy(od.widen_bf16(inp["q"][b]))[None, :, None, :]
        k = torch.from_numpy(od.widen_bf16(inp["k"][b, :L])).permute(1, 0, 2)[None].repeat_interleave(3, 1)
        v = torch.from_numpy(od.widen_bf16(inp["v"][b, :L])).permute(1, 0, 2)[None].repeat_interleave(3, 1)
        ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=inp["scale"])[0, :, 0].numpy()
        if not np.allclose(out[b], ref, rtol=0, atol=1e-12):
            return False
    ranges = _random_ranges(np.random.default_rng(98), [200, 11], 6, 40, group=3)
    acc, ml = monkey_od.range_partials(inp, ranges, 40)
    npc = _slot_counts(ranges, 2, 6)
    assert npc.max() >= 2  # the merge must be exercised
    for b in range(2):
        for h in range(6):
            parts = [(acc[b, h, j][None], ml[b, h, j, :1], ml[b, h, j, 1:]) for j in range(npc[b, h])]
            if not np.allclose(monkey_od.merge_partials(parts)[0], out[b, h], atol=1e-12):
                return False
    return True


def test_planted_mistakes_are_caught(monkeypatch):
    assert _pins(od)
    good_attend, good_partial, good_merge = od.attend, od.attend_partial, od.merge_partials

    def no_norm(q, K, V, scale):
        s = (q @ K.T) * scale
        return np.exp(s - s.max(1, keepdims=True)) @ V

    def wrong_sign(q, K, V, scale):
        s = -(q @ K.T) * scale
        w = np.exp(s - s.max(1, keepdims=True))
        return (w @ V) / w.sum(1, keepdims=True)

    def swapped_kv(q, K, V, scale):
        return good_attend(q, V, K, scale)

    def scale_twice(q, K, V, scale):
        return good_attend(q, K, V, scale * scale)

    def merge_without_rescale(parts):
        out = np.zeros_like(parts[0][0])
        num = sum(a for a, m, l in parts)
        den = sum(l for a, m, l in parts)
        return num / den[:, None]

    def partial_off_by_one(q, K, V, scale):
        return good_partial(q, K[:-1] if len(K) > 1 else K, V[:-1] if len(V) > 1 else V, scale)

    for name, fn in [("attend", no_norm), ("attend", wrong_sign), ("attend", swapped_kv),
                     ("attend", scale_twice), ("merge_partials", merge_without_rescale),
                     ("attend_partial", partial_off_by_one)]:
        with monkeypatch.context() as m:
            m.setattr(od, name, fn)
            assert not _pins(od), f"planted mistake in {name} ({fn.__name__}) went unnoticed"

    # wrong query-head -> KV-head map (h % Hkv instead of h // G)
    def decode_all_modmap(inp):
        q = inp["q"]
        B, Hq, D = q.shape
        Hkv = inp["k"].shape[2]
        out = np.zeros((B, Hq, D))
        for b in range(B):
            L = int(inp["seq_lens"][b])
            for h in range(Hq):
                out[b, h] = od.attend(od.widen_bf16(q[b, h])[None], od.widen_bf16(inp["k"][b, :L, h % Hkv]),
                                      od.widen_bf16(inp["v"][b, :L, h % Hkv]), inp["scale"])[0]
        return out

    with monkeypatch.context() as m:
        m.setattr(od, "_decode_all", decode_all_modmap)
        assert not _pins(od)


# ------------------------------------------------------ generator sanity

def test_generator_workloads_have_the_stated_structure():
    wl = Workload("t", B=8, Hq=16, Hkv=4, D=32, max_ctx=256, layout="paged", page_size=16,
                  lens="uniform", lens_lo=10, lens_hi=256, seed=5)
    inp = make_inputs(wl)
    lens = inp["seq_lens"]
    assert lens.min() >= 10 and lens.max() <= 256
    used = inp["page_table"][inp["page_table"] >= 0]
    assert sorted(used.tolist()) == list(range(inp["k_pool"].shape[0]))
    wl2 = Workload("o", B=1, Hq=8, Hkv=2, D=64, max_ctx=5000, outlier_frac=0.001, seed=6)
    inp2 = make_inputs(wl2)
    assert len(inp2["outlier_pos"]) == 5
    big = np.abs(od.widen_bf16(inp2["k"][0])).max(axis=(1, 2))
    assert np.all(big[inp2["outlier_pos"]] > 8.0)


# ------------------------------------------------------------ multi-query decode

def _multi_case(rng, B, Hq, Hkv, D, qlen, ctx, lens, kstd=1.0):
    inp = _contig_case(rng, B, Hq, Hkv, D, ctx, lens, kstd)
    inp["q"] = _rand_bits(rng, (B, Hq, qlen, D))
    return inp


def _masked_softmax_reference(inp):
    """Independent formulation: all L scores per query row, a causal mask matrix
    mask[i, t] = (t <= L - q_len + i), softmax over the unmasked entries."""
    q = inp["q"]
    B, Hq, qlen, D = q.shape
    Hkv = inp["k"].shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, qlen, D))
    for b in range(B):
        L = int(inp["seq_lens"][b])
        t = np.arange(L)
        mask = t[None, :] <= (L - qlen + np.arange(qlen))[:, None]
        for h in range(Hq):
            K = od.widen_bf16(inp["k"][b, :L, h // G])
            V = od.widen_bf16(inp["v"][b, :L, h // G])
            s = od.widen_bf16(q[b, h]) @ K.T * inp["scale"]
            for i in range(qlen):
                if not mask[i].any():
                    continue
                m = s[i][mask[i]].max()
                w = np.where(mask[i], np.exp(np.where(mask[i], s[i], m) - m), 0.0)
                out[b, h, i] = w @ V / w.sum()
    return out


def test_multi_query_matches_a_masked_softmax():
    rng = np.random.default_rng(60)
    for qlen, lens in [(1, [9, 40]), (3, [3, 40]), (7, [7, 100]), (4, [2, 33]), (8, [1, 17])]:
        inp = _multi_case(rng, 2, 6, 2, 16, qlen, ctx=max(lens), lens=lens)
        got = od.decode_multi(inp)
        assert np.allclose(got, _masked_softmax_reference(inp), rtol=0, atol=1e-12), qlen


def test_multi_query_row_is_decode_over_its_visible_prefix():
    rng = np.random.default_rng(61)
    inp = _multi_case(rng, 2, 8, 2, 32, 5, ctx=60, lens=[60, 23])
    out = od.decode_multi(inp)
    for b in range(2):
        for i in range(5):
            n = od.visible_tokens(int(inp["seq_lens"][b]), 5, i)
            one = dict(inp, q=inp["q"][:, :, i], seq_lens=np.array([n if bb == b else 1 for bb in range(2)], np.int32))
            for h in range(8):
                assert np.array_equal(out[b, h, i], od.decode_rows(one, [(b, h)])[0])
    # the last query token sees the whole sequence; one token equals plain decode
    single = dict(inp, q=inp["q"][:, :, 4])
    assert np.allclose(out[:, :, 4], od.decode_contig(**single), rtol=0, atol=1e-12)
    one = dict(inp, q=inp["q"][:, :, :1])
    assert np.allclose(od.decode_multi(one)[:, :, 0], od.decode_contig(**dict(inp, q=inp["q"][:, :, 0])),
                       rtol=0, atol=1e-12)


def test_multi_query_edge_lengths():
    assert [od.visible_tokens(10, 4, i) for i in range(4)] == [7, 8, 9, 10]
    assert [od.visible_tokens(2, 4, i) for i in range(4)] == [0, 0, 1, 2]
    assert od.visible_tokens(0, 1, 0) == 0
    rng = np.random.default_rng(62)
    inp = _multi_case(rng, 1, 2, 1, 16, 4, ctx=2, lens=[2])
    out = od.decode_multi(inp)
    assert np.all(out[0, :, :2] == 0)  # queries that see no token
    assert np.array_equal(od.round_to_bf16(out[0, :, 2]),
                          inp["v"][0, 0, 0][None].repeat(2, 0))  # one visible key: its V row


def test_multi_query_merge_of_partials_equals_unsplit():
    """Rows are (head, query token) pairs, head-major; a row's range is cut at what
    its query token sees, so pieces past it are empty and merge to nothing."""
    rng = np.random.default_rng(63)
    inp = _multi_case(rng, 3, 4, 1, 32, 6, ctx=400, lens=[400, 5, 130])
    ref = od.decode_multi(inp).reshape(3, 24, 32)
    for S in (1, 3, 9, 40):
        ranges = _random_ranges(rng, [400, 5, 130], 24, S, group=int(rng.choice([1, 6, 8])))
        acc, ml = od.range_partials(inp, ranges, S)
        got = _merge_rows(acc, ml, _slot_counts(ranges, 3, 24))
        assert np.allclose(got, ref, rtol=0, atol=1e-12), S


def test_multi_query_planted_off_by_one_is_caught(monkeypatch):
    rng = np.random.default_rng(64)
    inp = _multi_case(rng, 2, 4, 2, 16, 4, ctx=30, lens=[30, 6])
    ref = _masked_softmax_reference(inp)
    assert np.allclose(od.decode_multi(inp), ref, rtol=0, atol=1e-12)
    for wrong in (lambda L, q, i: max(0, min(L, L - q + i)), lambda L, q, i: max(0, min(L, L - q + 2 + i)),
                  lambda L, q, i: max(0, min(L, L - i))):
        with monkeypatch.context() as m:
            m.setattr(od, "visible_tokens", wrong)
            assert not np.allclose(od.decode_multi(inp), ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------ int8 KV cache

def _int8_case(seed, B, Hq, Hkv, D, ctx, lens):
    from gqa_split_kv_gb300.workloads import make_int8_cache
    rng = np.random.default_rng(seed)
    inp = make_int8_cache(rng, B, ctx, Hkv, D)
    inp.update(q=_rand_bits(rng, (B, Hq, D)), seq_lens=np.asarray(lens, np.int32),
               scale=float(np.float32(1 / math.sqrt(D))))
    return inp


def test_int8_with_unit_scales_is_decode_of_the_integers():
    inp = _int8_case(70, 2, 8, 2, 32, 50, [50, 9])
    inp["k_scale"][:] = 1.0
    inp["v_scale"][:] = 1.0
    from gqa_split_kv_gb300.workloads import f32_to_bf16_bits
    k = f32_to_bf16_bits(inp["k_i8"].astype(np.float32))  # integers |x| <= 127 are exact in bf16
    v = f32_to_bf16_bits(inp["v_i8"].astype(np.float32))
    ref = od.decode_contig(inp["q"], k, v, inp["seq_lens"], inp["scale"])
    assert np.allclose(od.decode_int8(inp), ref, rtol=0, atol=1e-12)


def test_int8_scales_act_as_documented():
    inp = _int8_case(71, 2, 6, 2, 16, 40, [40, 13])
    base = od.decode_int8(inp)
    # V scales multiply the output; K scales multiply the softmax scale
    twice_v = dict(inp, v_scale=inp["v_scale"] * 2)
    assert np.allclose(od.decode_int8(twice_v), 2 * base, rtol=1e-13, atol=0)
    twice_k = dict(inp, k_scale=inp["k_scale"] * 2)
    assert np.allclose(od.decode_int8(twice_k), od.decode_int8(dict(inp, scale=inp["scale"] * 2)), rtol=0,
                       atol=1e-12)


def test_int8_brute_force_and_paged():
    from gqa_split_kv_gb300.workloads import int8_to_paged
    inp = _int8_case(72, 2, 4, 2, 8, 12, [12, 5])
    got = od.decode_int8(inp)
    for b, L in enumerate([12, 5]):
        for h in range(4):
            g = h // 2
            q = od.widen_bf16(inp["q"][b, h])
            num, den = np.zeros(8), 0.0
            s = [inp["scale"] * sum(q[d] * float(inp["k_i8"][b, t, g, d]) * float(inp["k_scale"][b, g, t])
                                    for d in range(8)) for t in range(L)]
            m = max(s)
            for t in range(L):
                w = math.exp(s[t] - m)
                den += w
                num += w * inp["v_i8"][b, t, g].astype(np.float64) * float(inp["v_scale"][b, g, t])
            assert np.allclose(got[b, h], num / den, rtol=0, atol=1e-12)
    pin = dict(int8_to_paged(inp, inp["seq_lens"], 4, np.random.default_rng(1), spare_pages=2),
               q=inp["q"], seq_lens=inp["seq_lens"], page_size=4, scale=inp["scale"])
    assert np.array_equal(od.decode_int8(pin), got)


def test_int8_merge_of_partials_equals_unsplit():
    inp = _int8_case(73, 3, 8, 2, 64, 600, [600, 70, 0])
    ref = od.decode_int8(inp)
    rng = np.random.default_rng(75)
    for S in (1, 4, 40):
        ranges = _random_ranges(rng, [600, 70, 0], 8, S, group=4)
        acc, ml = od.range_partials(inp, ranges, S)
        got = _merge_rows(acc, ml, _slot_counts(ranges, 3, 8))
        assert np.allclose(got, ref, rtol=0, atol=1e-12), S


def test_int8_planted_mistakes_are_caught(monkeypatch):
    inp = _int8_case(74, 2, 4, 2, 16, 30, [30, 7])
    ref = _int8_reference_by_hand(inp)
    assert np.allclose(od.decode_int8(inp), ref, rtol=0, atol=1e-12)
    good = od.dequant_rows

    def k_scale_for_v(inp_, b, L):
        k, v = good(inp_, b, L)
        return k, v / inp_["v_scale"][b, :, :L].T[:, :, None] * inp_["k_scale"][b, :, :L].T[:, :, None]

    def scales_transposed(inp_, b, L):
        k, v = good(inp_, b, L)
        ks = inp_["k_scale"][b, :, :L].T[:, :, None]
        return k / ks * ks[::-1], v

    for bad in (k_scale_for_v, scales_transposed):
        with monkeypatch.context() as m:
            m.setattr(od, "dequant_rows", bad)
            assert not np.allclose(od.decode_int8(inp), ref, rtol=0, atol=1e-12), bad.__name__


def _int8_reference_by_hand(inp):
    """Dequantize with explicit loops (independent of dequant_rows), then attend."""
    B, Hq, D = inp["q"].shape
    Hkv = inp["k_i8"].shape[2]
    out = np.zeros((B, Hq, D))
    for b in range(B):
        L = int(inp["seq_lens"][b])
        K = np.zeros((L, Hkv, D))
        V = np.zeros((L, Hkv, D))
        for t in range(L):
            for g in range(Hkv):
                K[t, g] = inp["k_i8"][b, t, g].astype(np.float64) * float(inp["k_scale"][b, g, t])
                V[t, g] = inp["v_i8"][b, t, g].astype(np.float64) * float(inp["v_scale"][b, g, t])
        for h in range(Hq):
            g = h // (Hq // Hkv)
            out[b, h] = od.attend(od.widen_bf16(inp["q"][b, h])[None], K[:, g], V[:, g], inp["scale"])[0]
    return out


def test_int8_traffic_counts_values_and_scales():
    """The bench's int8 byte count: D int8 bytes plus one fp32 scale per (token, KV
    head) for each of K and V, against the bf16 count of 2 D bytes per tensor."""
    from gqa_split_kv_gb300.accounting import traffic_bytes
    lens = [100, 7, 0, 300]
    for D in (32, 64, 128, 256):
        t8 = traffic_bytes(4, 16, 4, D, lens, 1, kv_dtype="int8")
        t16 = traffic_bytes(4, 16, 4, D, lens, 1)
        assert t8["kv"] == 2 * 4 * sum(lens) * (D + 4)
        assert t16["kv"] == 2 * 4 * sum(lens) * 2 * D
        assert t8["q"] == t16["q"] and t8["partials_read"] == t16["partials_read"]
