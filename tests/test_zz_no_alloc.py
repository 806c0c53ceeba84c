"""The allocation-free entry point, decode_attn_contig_noalloc.

It serves callers that cannot allocate device memory or hold a workspace (a
runtime that hands its plugins only input and output buffers, a serving loop
that must not call cudaMalloc between steps): the segment counters and split
partials live in a fixed array inside the library.  Its outputs are checked
against the allocating entry point and against the CPU oracle.  This file is
collected last, so a run that stops at the first failure has already run every
other test.  It needs no state from other tests and passes alone in a fresh
process.
"""
import ctypes
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from gqa_split_kv_gb300 import binding  # noqa: E402
from gqa_split_kv_gb300.workloads import bf16_bits_to_f32, f32_to_bf16_bits  # noqa: E402

ATOL = RTOL = 2e-2


def _noalloc_fn():
    fn = binding.load().decode_attn_contig_noalloc
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, vp]
    fn.restype = i
    return fn


def _case(seed, B, Hq, Hkv, D, ctx, lens):
    rng = np.random.default_rng(seed)
    host = {}

    def dev(name, shape):
        bits = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        host[name] = bits
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)

    scale = float(np.float32(1.0 / math.sqrt(D)))
    c = dict(q=dev("q", (B, Hq, D)), k=dev("k", (B, ctx, Hkv, D)), v=dev("v", (B, ctx, Hkv, D)),
             lens=torch.tensor(lens, dtype=torch.int32, device="cuda"), B=B, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx,
             scale=scale)
    c["ref"] = oracle.decode_contig(host["q"], host["k"], host["v"], np.asarray(lens, np.int32), scale)
    return c


def _call(fn, c):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.full((c["B"], c["Hq"], c["D"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    st = fn(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["lens"].data_ptr(), c["B"], c["Hq"],
            c["Hkv"], c["D"], c["ctx"], c["scale"], out.data_ptr(), stream)
    assert st == 0, binding.STATUS.get(st, st)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return _as_f64(out)


def _close(got, ref):
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    assert np.all(err <= ATOL + RTOL * np.abs(ref)), f"max abs err {err.max():.3e}"


def _as_f64(t):
    return bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def test_noalloc_matches_the_allocating_entry_point_on_two_calls_in_a_row():
    fn = _noalloc_fn()
    # two calls in a row, different inputs, sharing the library's array; the first
    # cuts its long sequence into more than 8 pieces (merged by the combine kernel)
    cases = [_case(101, 3, 24, 4, 128, 1500, [1500, 700, 33]), _case(202, 2, 32, 8, 64, 3000, [3000, 1])]
    for c in cases:
        want = binding.decode_attn_contig(c["q"], c["k"], c["v"], c["lens"], scale=c["scale"])
        got = _call(fn, c)
        _close(got, _as_f64(want))
        _close(got, c["ref"])


def test_noalloc_shapes_in_turn_match_the_oracle():
    """One shape, another, then the first again: counters and partials left in the
    array by a call of another shape must not disturb the next."""
    fn = _noalloc_fn()
    a = _case(303, 1, 24, 4, 256, 4096, [4096])            # GQA-6: 32-33 pieces per KV head
    b = _case(404, 5, 16, 2, 64, 900, [900, 17, 0, 450, 64])
    for c in (a, b, a, b, a):
        _close(_call(fn, c), c["ref"])


def test_noalloc_rejects_partials_beyond_its_array():
    fn = _noalloc_fn()
    A = 0x10000  # never dereferenced: every call below returns before any launch
    # 64 x 64 heads x 20 slots x 256 columns of fp32 partials is far beyond 8 MiB
    assert fn(A, A, A, None, 64, 64, 8, 256, 4096, 0.0625, A, None) == 3
    assert fn(A, A, A, None, 1, 6, 4, 64, 64, 0.125, A, None) == 1  # Hq % Hkv
    # the statuses of decode_attn_contig for the same bad arguments, whatever the size
    alloc = binding.load().decode_attn_contig
    for args in [(64, 65 * 8, 8, 256, 4096, 0.0625),      # G = 65 > 64
                 (1, 65, 1, 64, 64, 0.125),
                 (64, 64, 8, 256, 4096, float("inf")),    # non-finite scale
                 (1, 8, 2, 48, 64, 0.125)]:               # head_dim 48
        B, Hq, Hkv, D, ctx, scale = args
        want = alloc(A, A, A, None, B, Hq, Hkv, D, ctx, scale, 1, None, None, None, A, None)
        assert want in (1, 2)
        assert fn(A, A, A, None, B, Hq, Hkv, D, ctx, scale, A, None) == want, args
