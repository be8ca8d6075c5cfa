"""ctypes view of ``libattn.so``: symbol table, argument types, status codes.

The library must have been built (``exact_io_aware_order_gb300.build.build()``
or ``__graft_entry__.build()``); loading a missing library raises instead of
falling back to anything else.
"""

from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "attn.h")

c_int, c_float, c_void_p, c_uint64, c_char_p = (ctypes.c_int, ctypes.c_float, ctypes.c_void_p,
                                                 ctypes.c_uint64, ctypes.c_char_p)
c_uint = ctypes.c_uint

# name -> (restype, argtypes); pointers are passed as c_void_p (raw addresses).
SIGNATURES = {
    "attn_status_string": (c_char_p, [c_int]),
    "attn_version": (c_char_p, []),
    "attn_prefill": (c_int, [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int, c_void_p]),
    "attn_prefill_ex": (c_int, [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int, c_int, c_float,
                                                                c_void_p, c_void_p]),
    "attn_decode_splitkv_ex": (c_int, [c_void_p] * 5 + [c_int] + [c_void_p] * 2 + [c_int] * 8
                               + [c_float, c_int, c_float, c_void_p, c_void_p]),
    "attn_decode_splitkv_ex2": (c_int, [c_void_p] * 5 + [c_int] + [c_void_p] * 2 + [c_int] * 8
                                + [c_float, c_int, c_float, c_void_p, c_uint, c_void_p]),
    "attn_prefill_varlen": (c_int, [c_void_p] * 6 + [c_int] * 5 + [c_float, c_int, c_void_p]),
    "attn_prefill_varlen_ex": (c_int, [c_void_p] * 6 + [c_int] * 5
                               + [c_float, c_int, c_int, c_float, c_void_p, c_void_p]),
    "attn_prefill_ex2": (c_int, [c_void_p] * 5 + [c_int] * 5 + [c_float, c_int, c_int, c_float,
                                                                 c_void_p, c_uint, c_void_p]),
    "attn_prefill_varlen_ex2": (c_int, [c_void_p] * 6 + [c_int] * 5
                                + [c_float, c_int, c_int, c_float, c_void_p, c_uint, c_void_p]),
    "attn_decode_num_splits": (c_int, [c_int] * 4),
    "attn_decode_splitkv": (c_int, [c_void_p] * 5 + [c_int] + [c_void_p] * 2 + [c_int] * 8
                            + [c_float, c_void_p]),
    "attn_decode_append_splitkv": (c_int, [c_void_p] * 7 + [c_int] + [c_void_p] * 2
                                   + [c_int] * 8 + [c_float, c_void_p]),
    "attn_decode_append_splitkv_ex": (c_int, [c_void_p] * 7 + [c_int] + [c_void_p] * 2
                                      + [c_int] * 8 + [c_float, c_int, c_float, c_void_p,
                                                       c_void_p]),
    "attn_prefill_fp8": (c_int, [c_void_p] * 8 + [c_int] * 5 + [c_float, c_int, c_void_p]),
    "attn_prefill_fp8_varlen": (c_int, [c_void_p] * 9 + [c_int] * 5
                                + [c_float, c_int, c_void_p]),
    "attn_quantize_fp8_varlen": (c_int, [c_void_p] * 5 + [c_int] * 4 + [c_void_p]),
    "attn_quantize_fp8": (c_int, [c_void_p] * 4 + [c_int] * 5 + [c_void_p]),
    "attn_quantize_fp8_qkv": (c_int, [c_void_p] * 10 + [c_int] * 4 + [c_void_p]),
    "attn_combine": (c_int, [c_void_p, c_void_p] + [c_int] * 4 + [c_void_p, c_void_p, c_void_p]),
    "attn_check_device_status": (c_int, [c_void_p]),
    "attn_set_wait_timeout_ns": (c_uint64, [c_uint64]),
    "attn_selftest_bounded_wait": (c_int, [c_void_p]),
    "attn_decode_noalloc": (c_int, [c_void_p] * 5 + [c_int] + [c_void_p] * 2 + [c_int] * 8
                            + [c_float, c_void_p]),
}

ATTN_MAX_SPLITS = 1024
ATTN_NOALLOC_SCRATCH_BYTES = 8 << 20


class AttnError(RuntimeError):
    """A nonzero attn_status returned by the library."""

    def __init__(self, fn: str, status: int, message: str):
        super().__init__(f"{fn} failed with status {status}: {message}")
        self.status = status


_LIB = None


def status_codes() -> dict[str, int]:
    """The attn_status enum, parsed from the public header."""
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(ATTN_\w+)\s*=\s*(\d+)", text)}


def header_functions() -> list[str]:
    """Every function the public header declares."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(attn_\w+)\s*\(", text, re.M)))


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run exact_io_aware_order_gb300.build.build() first")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def check(fn: str, status: int) -> None:
    if status != 0:
        msg = lib().attn_status_string(status).decode()
        raise AttnError(fn, status, msg)
