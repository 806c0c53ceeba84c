"""CPU oracle for split-KV GQA decode attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.
"""
from .decode_attention import *  # noqa: F401,F403
from .prefill_attention import *  # noqa: F401,F403
