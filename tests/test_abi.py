"""C ABI checks that need no GPU: the library loads, exports every declared
symbol, the host planner's values, and argument validation (every rejected
call returns its status before touching CUDA)."""
import ctypes
import os
import re

import pytest

from gqa_split_kv_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def clib():
    build_mod.build()
    from gqa_split_kv_gb300 import binding
    return binding.load()


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return names


def test_every_declared_symbol_is_exported(clib):
    names = declared_functions()
    assert {"decode_num_splits", "decode_attn_contig", "decode_attn_paged", "decode_combine",
            "decode_num_splits_multi", "decode_attn_multi_contig", "decode_attn_multi_paged"} <= set(names)
    for n in names:
        assert hasattr(clib, n), n


def test_status_strings(clib):
    assert clib.decode_status_string(0) == b"DA_OK"
    assert clib.decode_status_string(3) == b"DA_ERR_WORKSPACE"
    assert clib.decode_status_string(99) == b"unknown status"


@pytest.mark.parametrize("args,want", [
    ((1, 4, 4096, 256, 152), 39),     # GQA-6 ctx 4096: 38 ranges per KV head fill 152 SMs
    ((1, 8, 65536, 128, 152), 20),
    ((16, 8, 8192, 128, 152), 20),
    ((64, 8, 32768, 128, 152), 20),
    ((1, 2, 512, 64, 152), 32),       # capped by the 32 blocks of 16 tokens
    ((1, 2, 16, 64, 152), 1),         # one block: nothing to split
    ((1, 2, 17, 64, 152), 2),
    ((4, 1, 10 ** 6, 128, 2000), 1024),
])
def test_num_splits_values(clib, args, want):
    assert clib.decode_num_splits(*args) == want


def test_num_splits_multi(clib):
    # 42 rows (GQA-6 x 7 tokens) = 6 sub-groups of 7; 2 per pass at D=256 -> 3 passes x 4 KV heads = 12 segments
    assert clib.decode_num_splits_multi(1, 7, 24, 4, 4096, 256, 152) == clib.decode_num_splits(1, 12, 4096, 256, 152)
    assert clib.decode_num_splits_multi(1, 7, 24, 4, 4096, 256, 152) == 14
    # 16 rows at D=128: 2 sub-groups in one pass -> as many segments as KV heads
    assert clib.decode_num_splits_multi(16, 4, 32, 8, 8192, 128, 152) == clib.decode_num_splits(16, 8, 8192, 128, 152)
    for args in [(1, 4, 4096, 256, 152), (16, 8, 8192, 128, 152), (64, 8, 32768, 128, 152)]:
        B, Hkv, L, D, sms = args
        assert clib.decode_num_splits_multi(B, 1, 6 * Hkv, Hkv, L, D, sms) == clib.decode_num_splits(*args)
    assert clib.decode_num_splits_multi(1, 0, 8, 2, 64, 64, 152) == -1
    assert clib.decode_num_splits_multi(1, 9, 16, 2, 64, 64, 152) == -1   # 72 rows per KV head
    assert clib.decode_num_splits_multi(1, 2, 8, 2, 64, 48, 152) == -2


def test_num_splits_rejects_bad_shapes(clib):
    assert clib.decode_num_splits(1, 0, 100, 64, 152) == -1
    assert clib.decode_num_splits(-1, 2, 100, 64, 152) == -1
    assert clib.decode_num_splits(1, 2, -5, 64, 152) == -1


A = 0x10000  # a fake 16-byte-aligned address: never dereferenced by rejected calls


def contig(clib, q=A, k=A, v=A, lens=None, B=1, Hq=8, Hkv=2, D=64, ctx=64, scale=0.125, S=2, pa=A, pm=A, ctr=A,
           out=A):
    return clib.decode_attn_contig(q, k, v, lens, B, Hq, Hkv, D, ctx, scale, S, pa, pm, ctr, out, None)


def paged(clib, ps=16, lens=A, table=A, D=64, S=2, maxp=4, npages=4, maxlen=64, pa=A, pm=A, ctr=A):
    return clib.decode_attn_paged(A, A, A, table, lens, 1, 8, 2, D, ps, maxp, npages, maxlen, 0.125, S, pa, pm, ctr,
                                  A, None)


def test_contig_argument_errors(clib):
    assert contig(clib, Hq=6, Hkv=4) == 1                 # Hq % Hkv
    assert contig(clib, D=48) == 2                        # head_dim not built
    assert contig(clib, D=512) == 2
    assert contig(clib, Hq=130, Hkv=2) == 2               # G > 64
    assert contig(clib, S=0) == 1
    assert contig(clib, S=1025) == 1
    assert contig(clib, pa=None) == 3                     # partial slots missing
    assert contig(clib, pm=None) == 3
    assert contig(clib, ctr=None) == 3
    assert contig(clib, ctr=A + 4) == 1
    assert contig(clib, q=A + 2) == 1                     # misaligned
    assert contig(clib, out=A + 8) == 1
    assert contig(clib, k=A + 4) == 1
    assert contig(clib, pa=A + 4) == 1
    assert contig(clib, pm=A + 4) == 1
    assert contig(clib, q=None) == 1
    assert contig(clib, k=None) == 1
    assert contig(clib, scale=float("inf")) == 1
    assert contig(clib, scale=float("nan")) == 1
    assert contig(clib, ctx=-1) == 1
    assert contig(clib, B=-1) == 1
    assert contig(clib, Hkv=0) == 1
    assert contig(clib, B=0) == 0                         # empty batch: nothing to do


def test_paged_argument_errors(clib):
    assert paged(clib, ps=24) == 2                        # page size not a multiple of 16
    assert paged(clib, ps=8) == 2
    assert paged(clib, ps=0) == 1
    assert paged(clib, lens=None) == 1                    # seq_lens required
    assert paged(clib, table=None) == 1
    assert paged(clib, table=A + 2) == 1
    assert paged(clib, D=100) == 2
    assert paged(clib, pa=None) == 3
    assert paged(clib, ctr=None) == 3
    assert paged(clib, maxp=-1) == 1
    assert paged(clib, maxlen=-3) == 1


def test_multi_argument_errors(clib):
    def multi(qlen=4, Hq=8, Hkv=2, D=64):
        return clib.decode_attn_multi_contig(A, A, A, None, 1, qlen, Hq, Hkv, D, 64, ctypes.c_float(0.125), 2, A, A,
                                             A, A, None)
    assert multi(qlen=0) == 1
    assert multi(qlen=17) == 1
    assert multi(Hq=6, Hkv=4) == 1          # Hq % Hkv
    assert multi(Hq=32, Hkv=2, qlen=5) == 2  # G * q_len = 80 > 64
    assert multi(D=48) == 2
    assert clib.decode_attn_multi_paged(A, A, A, A, A, 1, 2, 8, 2, 64, 24, 4, 4, 64, ctypes.c_float(0.125), 2, A, A,
                                        A, A, None) == 2  # page size not a multiple of 16


def test_combine_argument_errors(clib):
    assert clib.decode_combine(A, A, 1, 8, 48, 4, A, None) == 2
    assert clib.decode_combine(A, A, 1, 8, 64, 0, A, None) == 1
    assert clib.decode_combine(None, A, 1, 8, 64, 4, A, None) == 1
    assert clib.decode_combine(A, A, 1, 8, 64, 4, None, None) == 1
    assert clib.decode_combine(A + 4, A, 1, 8, 64, 4, A, None) == 1
    assert clib.decode_combine(A, A, 0, 8, 64, 4, A, None) == 0


def test_device_error_rejects_null(clib):
    assert clib.decode_device_error(None, None) == 1


def test_selftest_rejects_bad_timeouts(clib):
    clib.decode_selftest_bounded_wait.argtypes = [ctypes.c_ulonglong, ctypes.c_void_p]
    assert clib.decode_selftest_bounded_wait(0, None) == 1
    assert clib.decode_selftest_bounded_wait(10 ** 9 + 1, None) == 1


def test_int8_argument_errors(clib):
    def i8(ks=A, vs=A, ctx=64, D=64):
        return clib.decode_attn_int8_contig(A, A, A, ks, vs, None, 1, 8, 2, D, ctx, ctypes.c_float(0.125), 2, A, A,
                                            A, A, None)
    assert i8(ks=None) == 1
    assert i8(vs=A + 4) == 1
    assert i8(ctx=66) == 2   # scale rows need 16-byte strides: max_ctx a multiple of 4
    assert i8(D=48) == 2
    assert clib.decode_attn_int8_paged(A, A, A, None, A, A, A, 1, 8, 2, 64, 16, 4, 4, 64, ctypes.c_float(0.125), 2,
                                       A, A, A, A, None) == 1


def test_prefill_argument_checks_return_before_cuda(clib):
    V = ctypes.c_void_p
    q = V(1 << 20)  # never dereferenced: every call below is rejected or has nothing to do
    nan = float("nan")
    # (batch, q_len, Hq, Hkv, D, max_ctx, scale) -> status
    cases = [((1, 4, 6, 4, 128, 64, 0.1), 1),      # Hq not a multiple of Hkv
             ((1, 4, 8, 2, 48, 64, 0.1), 2),       # head_dim
             ((1, 4, 130, 2, 64, 64, 0.1), 2),     # G = 65 rows per token
             ((1, 4, 8, 2, 64, 64, nan), 1),       # scale
             ((-1, 4, 8, 2, 64, 64, 0.1), 1),
             ((1, -4, 8, 2, 64, 64, 0.1), 1),
             ((1, 4, 8, 2, 64, -1, 0.1), 1),
             ((0, 4, 8, 2, 64, 64, 0.1), 0),       # nothing to do
             ((3, 0, 8, 2, 64, 64, 0.1), 0)]
    for (B, n, Hq, Hkv, D, ctx, sc), want in cases:
        got = clib.prefill_attn_contig(q, q, q, None, B, n, Hq, Hkv, D, ctx, sc, q, None)
        assert got == want, (B, n, Hq, Hkv, D, ctx, sc, got)
    # misaligned q / out
    assert clib.prefill_attn_contig(V((1 << 20) + 2), q, q, None, 1, 4, 8, 2, 64, 64, 0.1, q, None) == 1
    assert clib.prefill_attn_contig(q, q, q, None, 1, 4, 8, 2, 64, 64, 0.1, V((1 << 20) + 8), None) == 1
    # paged: page size, missing table / lengths, negative sizes
    assert clib.prefill_attn_paged(q, q, q, q, q, 1, 4, 8, 2, 64, 8, 4, 16, 64, 0.1, q, None) == 2
    assert clib.prefill_attn_paged(q, q, q, None, q, 1, 4, 8, 2, 64, 16, 4, 16, 64, 0.1, q, None) == 1
    assert clib.prefill_attn_paged(q, q, q, q, None, 1, 4, 8, 2, 64, 16, 4, 16, 64, 0.1, q, None) == 1
    assert clib.prefill_attn_paged(q, q, q, q, q, 1, 4, 8, 2, 64, 16, -1, 16, 64, 0.1, q, None) == 1
    assert clib.prefill_attn_paged(q, q, q, q, q, 1, 4, 8, 3, 64, 16, 4, 16, 64, 0.1, q, None) == 1


def test_binding_rejects_host_and_mistyped_tensors(clib):
    """The Python binding only marshals arguments: host tensors, wrong dtypes and
    wrong ranks raise before the library is called."""
    torch = pytest.importorskip("torch")
    from gqa_split_kv_gb300 import binding
    q = torch.zeros((1, 8, 64), dtype=torch.bfloat16)
    k = torch.zeros((1, 32, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="q"):
        binding.decode_attn_contig(q, k, k)                      # host tensors
    with pytest.raises(ValueError, match="q"):
        binding.prefill_attn_contig(q, k, k)                     # q must be [B, q_len, Hq, D]
    with pytest.raises(ValueError, match="q"):
        binding.decode_attn_int8_contig(q, k, k, q, q)
    with pytest.raises(ValueError, match="q"):
        binding.prefill_attn_paged(q.float().unsqueeze(0), k, k, None, None, 32)


# ---------------------------------------------------- the library's split plan
#
# The pages fix only caps on the split count (AstrAI commit 988e013 "csrc",
# split-KV items: at most the tile count and 32 splits), and any partition of a
# row's tokens gives the same output.  So the partition the library uses is not
# restated anywhere; decode_plan_pieces reports it from the planner code the
# kernels run, and these checks hold it to the properties every valid partition
# must have.

def check_library_plan(lens, Hq, Hkv, D, S, q_len=1):
    from gqa_split_kv_gb300 import binding
    max_len = max(lens) if len(lens) else 0
    rec = binding.plan_pieces(list(lens), Hq, Hkv, D, max_len, S, q_len=q_len)
    R, G = Hq * q_len, Hq // Hkv * q_len
    segs = {}
    for r in rec:
        segs.setdefault((int(r[0]), int(r[1])), []).append([int(x) for x in r])
    for b, L in enumerate(lens):
        mine = sorted(k for k in segs if k[0] == b)
        if L == 0:
            assert not mine, (b, "an empty sequence has no pieces")
            continue
        rows = sorted(r for (bb, row0) in mine for r in range(row0, row0 + segs[(bb, row0)][0][2]))
        assert rows == list(range(R)), (b, "every row in exactly one pass")
    for (b, row0), ps in segs.items():
        ps.sort(key=lambda p: p[3])
        n, L = len(ps), int(lens[b])
        nrows = ps[0][2]
        assert 1 <= nrows <= 32 and row0 // G == (row0 + nrows - 1) // G, "a pass stays within one KV head"
        assert [p[3] for p in ps] == list(range(n)) and all(p[4] == n for p in ps)
        assert 1 <= n <= S
        assert all(p[2] == nrows for p in ps)
        assert ps[0][5] == 0 and ps[-1][6] == L, "the pieces cover [0, L)"
        for a, c in zip(ps, ps[1:]):
            assert a[6] == c[5], "in order, no gap, no overlap"
        assert all(p[5] < p[6] for p in ps), "no empty piece"
        assert all(p[5] % 64 == 0 for p in ps), "pieces start on 64-token boundaries"
        for p in ps:  # what slot j holds when the call returns
            t0, t1, h0, h1 = p[5], p[6], p[7], p[8]
            assert (h0, h1) == ((0, 0) if n == 1 else (t0, t1))
    return rec


def test_library_plan_is_a_valid_partition_random_shapes():
    import numpy as np
    rng = np.random.default_rng(41)
    for trial in range(300):
        B = int(rng.integers(1, 7))
        lens = rng.integers(0, 3000, size=B)
        lens[rng.random(B) < 0.2] = 0
        Hkv = int(rng.integers(1, 9))
        G = int(rng.choice([1, 2, 4, 6, 8, 9, 12, 16, 24, 32, 64]))
        D = int(rng.choice([32, 64, 128, 256]))
        S = int(rng.integers(1, 80))
        check_library_plan(lens.tolist(), G * Hkv, Hkv, D, S)


def test_library_plan_is_a_valid_partition_multi_query():
    import numpy as np
    rng = np.random.default_rng(42)
    for trial in range(100):
        B = int(rng.integers(1, 5))
        lens = rng.integers(0, 2000, size=B).tolist()
        Hkv, G, q_len = int(rng.integers(1, 5)), int(rng.choice([1, 4, 6, 8])), int(rng.integers(1, 9))
        if G * q_len > 64:
            continue
        D = int(rng.choice([64, 128, 256]))
        check_library_plan(lens, G * Hkv, Hkv, D, int(rng.integers(2, 40)), q_len=q_len)


@pytest.mark.parametrize("name", ["gqa6_contig_b1_hq24_hkv4_d256_ctx4096", "gqa6_contig_b1_hq24_hkv4_d256_ctx16384",
                                  "paged_b16_hq32_hkv8_d128_u256_8192_ps32",
                                  "long_contig_b1_hq32_hkv8_d128_ctx65536_outliers",
                                  "mixed_paged_b64_hq64_hkv8_d128_log1_32768_ps16"])
def test_library_plan_on_the_workloads(name):
    from gqa_split_kv_gb300 import binding
    from gqa_split_kv_gb300.workloads import WORKLOADS, workload_lens
    wl = WORKLOADS[name]
    lens = workload_lens(wl)
    S = binding.num_splits(wl.B, wl.Hkv, wl.max_ctx, wl.D, 152)
    rec = check_library_plan(lens.tolist(), wl.Hq, wl.Hkv, wl.D, S)
    assert rec[:, 4].max() <= S


def test_gqa6_pieces():
    """GQA-6 at ctx 4096 with the planner's 39 slots: 32 or 33 pieces per KV head, every
    slot holding its own piece's partial."""
    rec = check_library_plan([4096], 24, 4, 256, 39)
    for h in range(4):
        seg = rec[rec[:, 1] == 6 * h]
        assert 32 <= len(seg) <= 39 and set(seg[:, 2].tolist()) == {6}


def test_max_batch_values(clib):
    from gqa_split_kv_gb300 import binding
    assert binding.max_batch(32, 8, 128) == 1159
    for D in (32, 64, 128, 256):
        for paged in (False, True):
            for kv8 in (False, True):
                m = binding.max_batch(8 * 4, 8, D, kv_int8=kv8, paged=paged)
                assert 500 <= m <= 20000, (D, paged, kv8, m)
    assert clib.decode_max_batch(1, 8, 2, 48, 0, 0) == -2
    assert clib.decode_max_batch(0, 8, 2, 64, 0, 0) == -1
    assert clib.decode_max_batch(2, 8, 2, 64, 1, 0) == -2  # int8 caches take one query token
