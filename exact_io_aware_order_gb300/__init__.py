"""GB300 (sm_103a) exact attention forward: causal prefill, split-KV decode
and the LSE combine, behind a C ABI (``include/attn.h``, ``libattn.so``).

The functions here only marshal torch tensors into the C calls; every step of
the computation runs in the library's CUDA kernels.
"""

from .api import (  # noqa: F401
    prefill,
    prefill_varlen,
    decode_splitkv,
    combine,
    decode,
    decode_num_splits,
    check_device_status,
    set_wait_timeout_ns,
    selftest_bounded_wait,
    decode_noalloc,
    decode_append_splitkv,
    decode_append,
    quantize_fp8,
    quantize_fp8_qkv,
    quantize_fp8_varlen,
    prefill_fp8,
    prefill_fp8_varlen,
)
from ._lib import AttnError, lib  # noqa: F401
