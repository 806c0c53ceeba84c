"""Split-KV GQA decode attention for GB300 (sm_103a).

The compute path is libdecode_attn.so (CUDA, C ABI in include/decode_attn.h);
``binding`` forwards PyTorch tensors to it, ``workloads`` draws seeded inputs.
"""
from .binding import (DecodeAttnError, decode_attn_contig, decode_attn_paged, decode_combine,  # noqa: F401
                      device_error, load, num_splits)
