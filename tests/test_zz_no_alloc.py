"""The allocation-free entry point, decode_attn_contig_noalloc.

It serves callers that cannot allocate device memory or hold a workspace (a
runtime that hands its plugins only input and output buffers, a serving loop
that must not call cudaMalloc between steps): the split partials live in a
fixed array inside the library.  This file is collected last, so a run that
stops at the first failure has already run every other test.  It needs no
state from other tests and passes alone in a fresh process.
"""
import ctypes
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

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

    def dev(shape):
        bits = f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)

    return dict(q=dev((B, Hq, D)), k=dev((B, ctx, Hkv, D)), v=dev((B, ctx, Hkv, D)),
                lens=torch.tensor(lens, dtype=torch.int32, device="cuda"), B=B, Hq=Hq, Hkv=Hkv, D=D, ctx=ctx,
                scale=1.0 / math.sqrt(D))


def _as_f64(t):
    return bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)


def test_noalloc_matches_the_allocating_entry_point_on_two_calls_in_a_row():
    fn = _noalloc_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [_case(101, 3, 24, 4, 128, 1500, [1500, 700, 33]), _case(202, 2, 32, 8, 64, 3000, [3000, 1])]
    for c in cases:  # two calls in a row, different inputs, sharing the library's array
        want = binding.decode_attn_contig(c["q"], c["k"], c["v"], c["lens"], scale=c["scale"])
        out = torch.full((c["B"], c["Hq"], c["D"]), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = fn(c["q"].data_ptr(), c["k"].data_ptr(), c["v"].data_ptr(), c["lens"].data_ptr(), c["B"], c["Hq"],
                c["Hkv"], c["D"], c["ctx"], c["scale"], out.data_ptr(), stream)
        assert st == 0, binding.STATUS.get(st, st)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        got, ref = _as_f64(out), _as_f64(want)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))


def test_noalloc_rejects_partials_beyond_its_array():
    fn = _noalloc_fn()
    A = 0x10000  # never dereferenced: the call returns before any launch
    # 64 x 64 heads x 20 slots x 256 columns of fp32 partials is far beyond 8 MiB
    assert fn(A, A, A, None, 64, 64, 8, 256, 4096, 0.0625, A, None) == 3
    assert fn(A, A, A, None, 1, 6, 4, 64, 64, 0.125, A, None) == 1  # Hq % Hkv
