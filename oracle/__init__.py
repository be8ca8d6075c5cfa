"""Test infrastructure: a float64 CPU oracle for exact attention forward.

Only the test-suite, the package's ``smoke()`` check and the benchmark's CPU
baseline leg may import this package.  The library's own compute path never
imports, calls or links anything in here, and nothing in here imports the
library.
"""

from .attention_ref import (  # noqa: F401
    masked_attention,
    prefill,
    prefill_rows,
    gather_sequence,
    decode,
    decode_partials,
    combine,
    append_token,
    decode_append,
    prefill_varlen,
    prefill_varlen_rows,
)
from . import fp8_ref  # noqa: F401  (FP8 block quantisation and its attention)
