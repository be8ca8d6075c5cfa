"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

* libattn.so builds, loads and exports every function include/attn.h declares;
* every status code has a name;
* argument validation rejects bad calls with the documented status before
  touching the device (fake, never-dereferenced addresses are used);
* the split-count policy and the split rule behave as documented.
"""

import ctypes
import os

import pytest

from exact_io_aware_order_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return _lib.lib()


def test_exports_every_header_function(L):
    names = _lib.header_functions()
    assert {"attn_prefill", "attn_decode_splitkv", "attn_combine", "attn_decode_num_splits",
            "attn_status_string", "attn_check_device_status"} <= set(names)
    raw = ctypes.CDLL(_lib.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), f"{n} is declared in include/attn.h but not exported"
    assert set(names) == set(_lib.SIGNATURES), "binding signatures out of sync with the header"


def test_status_strings(L):
    codes = _lib.status_codes()
    assert codes["ATTN_OK"] == 0 and len(set(codes.values())) == len(codes)
    for name, val in codes.items():
        s = L.attn_status_string(val).decode()
        assert s.startswith(name), (name, s)
    assert L.attn_status_string(999).decode() == "ATTN_ERR_UNKNOWN"
    assert L.attn_version().decode().endswith("sm_103a")


# Fake 16-byte-aligned addresses; validation fails before any is used.
P = 0x10000


def _prefill(L, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, batch=1, hq=4, hkv=2, n=128, d=128, scale=0.1, causal=1)
    a.update(kw)
    return L.attn_prefill(a["q"], a["k"], a["v"], a["o"], a["lse"], a["batch"], a["hq"], a["hkv"],
                          a["n"], a["d"], a["scale"], a["causal"], None)


def test_prefill_ex2_flags(L):
    """attn_prefill_ex2 / attn_prefill_varlen_ex2: unknown flag bits are
    refused before any launch; the rest of the validation is the _ex calls'."""
    c = _lib.status_codes()
    f = L.attn_prefill_ex2
    base = (P, P, P, P, P, 1, 4, 2, 128, 128, 0.1, 1, -1, 0.0, None)
    assert f(*base, 2, None) == c["ATTN_ERR_SHAPE"]
    assert f(*base, 1 << 31, None) == c["ATTN_ERR_SHAPE"]
    assert f(P, P, P, None, P, 1, 4, 2, 128, 128, 0.1, 1, -1, 0.0, None, 1, None) == c["ATTN_ERR_NULL"]
    assert f(P, P, P, P + 8, P, 1, 4, 2, 128, 128, 0.1, 1, -1, 0.0, None, 1, None) == c["ATTN_ERR_ALIGN"]
    g = L.attn_prefill_varlen_ex2
    vbase = (P, P, P, P, P, P, 3, 512, 8, 2, 128, 0.1, 1, -1, 0.0, None)
    assert g(*vbase, 4, None) == c["ATTN_ERR_SHAPE"]
    assert g(P, P, P, P, P, P, 3, 512, 8, 2, 96, 0.1, 1, -1, 0.0, None, 1, None) == c["ATTN_ERR_HEADDIM"]


def test_prefill_validation(L):
    c = _lib.status_codes()
    assert _prefill(L, q=None) == c["ATTN_ERR_NULL"]
    assert _prefill(L, lse=None) == c["ATTN_ERR_NULL"]
    assert _prefill(L, n=0) == c["ATTN_ERR_SHAPE"]
    assert _prefill(L, batch=0) == c["ATTN_ERR_SHAPE"]
    assert _prefill(L, n=(1 << 24) + 1) == c["ATTN_ERR_SHAPE"]
    assert _prefill(L, batch=1, hq=1 << 20, hkv=1, n=1 << 24) == c["ATTN_ERR_SHAPE"]  # items > 2^31
    assert _prefill(L, scale=0.0) == c["ATTN_ERR_SHAPE"]
    assert _prefill(L, scale=float("nan")) == c["ATTN_ERR_SHAPE"]
    assert _prefill(L, d=96) == c["ATTN_ERR_HEADDIM"]
    assert _prefill(L, d=192) == c["ATTN_ERR_HEADDIM"]
    assert _prefill(L, d=512) == c["ATTN_ERR_HEADDIM"]
    assert _prefill(L, hq=6, hkv=4) == c["ATTN_ERR_GQA"]
    assert _prefill(L, q=P + 8) == c["ATTN_ERR_ALIGN"]
    assert _prefill(L, o=P + 4) == c["ATTN_ERR_ALIGN"]
    assert _prefill(L, lse=P + 2) == c["ATTN_ERR_ALIGN"]


def test_variant_validation(L):
    c = _lib.status_codes()
    ex = lambda w, cap, al=None: L.attn_prefill_ex(P, P, P, P, P, 1, 4, 2, 128, 128, 0.1, 1, w, cap,
                                                   al, None)
    assert ex(-2, 0.0) == c["ATTN_ERR_SHAPE"]
    assert ex(0, -1.0) == c["ATTN_ERR_SHAPE"]
    assert ex(0, float("nan")) == c["ATTN_ERR_SHAPE"]
    assert ex(0, float("inf")) == c["ATTN_ERR_SHAPE"]
    assert L.attn_prefill_ex(None, P, P, P, P, 1, 4, 2, 128, 128, 0.1, 1, 5, 1.0, None, None) == \
        c["ATTN_ERR_NULL"]
    assert ex(-1, 2.0, P) == c["ATTN_ERR_SHAPE"]            # ALiBi with soft-capping
    assert L.attn_prefill_ex(P, P, P, P, P, 1, 4, 2, 128, 512, 0.1, 1, 16, 0.0, None, None) == \
        c["ATTN_ERR_HEADDIM"]
    assert ex(-1, 0.0, P + 2) == c["ATTN_ERR_ALIGN"]        # misaligned slopes
    dx = lambda w, cap, al=None: L.attn_decode_splitkv_ex(P, P, P, P, P, 4, P, P, 2, 8, 2, 128, 16,
                                                          8, 16, 128, 0.1, w, cap, al, None)
    assert dx(-3, 0.0) == c["ATTN_ERR_SHAPE"] and dx(4, -0.5) == c["ATTN_ERR_SHAPE"]
    assert dx(-1, 1.0, P) == c["ATTN_ERR_SHAPE"] and dx(-1, 0.0, P + 1) == c["ATTN_ERR_ALIGN"]


@pytest.mark.parametrize("kv_len,S,W", [(100, 3, 10), (1000, 7, 0), (33, 2, 16), (5000, 9, 4095),
                                        (17, 4, 100), (0, 3, 5), (64, 1, 15)])
def test_split_rule_with_window(kv_len, S, W):
    from gpu_util import split_ranges

    r = split_ranges(kv_len, S, W)
    lo = max(0, kv_len - 1 - W)
    covered = [t for a, b in r for t in range(a, b)]
    assert covered == list(range(lo, kv_len))          # exactly the window, in order
    assert all(a % 16 == 0 or a == lo for a, b in r if a < b)


def _varlen(L, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, cu=P, S=3, T=500, hq=4, hkv=2, d=128, scale=0.1, causal=1)
    a.update(kw)
    return L.attn_prefill_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu"], a["S"], a["T"],
                                 a["hq"], a["hkv"], a["d"], a["scale"], a["causal"], None)


def test_prefill_varlen_validation(L):
    c = _lib.status_codes()
    assert _varlen(L, cu=None) == c["ATTN_ERR_NULL"]
    assert _varlen(L, S=0) == c["ATTN_ERR_SHAPE"]
    assert _varlen(L, S=(1 << 20) + 1) == c["ATTN_ERR_SHAPE"]   # 513 .. 2^20 run in slices
    assert _varlen(L, hq=1 << 20, hkv=1, T=1 << 24) == c["ATTN_ERR_SHAPE"]   # item count > 2^31
    assert _varlen(L, T=0) == c["ATTN_ERR_SHAPE"]
    assert _varlen(L, T=(1 << 24) + 1) == c["ATTN_ERR_SHAPE"]
    assert _varlen(L, d=96) == c["ATTN_ERR_HEADDIM"]
    assert _varlen(L, d=512) == c["ATTN_ERR_HEADDIM"]
    assert _varlen(L, hq=6, hkv=4) == c["ATTN_ERR_GQA"]
    assert _varlen(L, cu=P + 2) == c["ATTN_ERR_ALIGN"]
    assert _varlen(L, q=P + 8) == c["ATTN_ERR_ALIGN"]


def _varlen_ex(L, w=-1, cap=0.0, al=None, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, cu=P, S=3, T=1000, hq=8, hkv=2, d=128, scale=0.1, causal=1)
    a.update(kw)
    return L.attn_prefill_varlen_ex(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cu"], a["S"],
                                    a["T"], a["hq"], a["hkv"], a["d"], a["scale"], a["causal"],
                                    w, cap, al, None)


def test_prefill_varlen_ex_validation(L):
    """The packed prefill's variant arguments are checked as attn_prefill_ex's."""
    c = _lib.status_codes()
    assert _varlen_ex(L, w=-2) == c["ATTN_ERR_SHAPE"]
    assert _varlen_ex(L, cap=-1.0) == c["ATTN_ERR_SHAPE"]
    assert _varlen_ex(L, cap=float("nan")) == c["ATTN_ERR_SHAPE"]
    assert _varlen_ex(L, cap=2.0, al=P) == c["ATTN_ERR_SHAPE"]      # ALiBi with soft-capping
    assert _varlen_ex(L, al=P + 2) == c["ATTN_ERR_ALIGN"]
    assert _varlen_ex(L, w=5, cu=None) == c["ATTN_ERR_NULL"]
    assert _varlen_ex(L, w=5, S=(1 << 20) + 1) == c["ATTN_ERR_SHAPE"]


def _decode(L, **kw):
    a = dict(q=P, k=P, v=P, bt=P, lens=P, S=4, op=P, lp=P, B=2, hq=8, hkv=2, d=128, bs=16,
             mb=8, nb=16, maxlen=128, scale=0.1)
    a.update(kw)
    return L.attn_decode_splitkv(a["q"], a["k"], a["v"], a["bt"], a["lens"], a["S"], a["op"],
                                 a["lp"], a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["mb"],
                                 a["nb"], a["maxlen"], a["scale"], None)


def test_decode_validation(L):
    c = _lib.status_codes()
    assert _decode(L, q=None) == c["ATTN_ERR_NULL"]
    assert _decode(L, lens=None) == c["ATTN_ERR_NULL"]
    assert _decode(L, B=0) == c["ATTN_ERR_SHAPE"]
    assert _decode(L, bs=0) == c["ATTN_ERR_SHAPE"]
    assert _decode(L, nb=0) == c["ATTN_ERR_SHAPE"]
    assert _decode(L, bt=None, maxlen=0) == c["ATTN_ERR_SHAPE"]
    assert _decode(L, scale=-1.0) == c["ATTN_ERR_SHAPE"]
    assert _decode(L, d=80) == c["ATTN_ERR_HEADDIM"]
    assert _decode(L, d=512) == c["ATTN_ERR_HEADDIM"]
    assert _decode(L, hq=6, hkv=4) == c["ATTN_ERR_GQA"]
    assert _decode(L, hq=130, hkv=2) == c["ATTN_ERR_GQA"]      # g = 65 > 64
    assert _decode(L, S=-1) == c["ATTN_ERR_SPLITS"]
    assert _decode(L, S=_lib.ATTN_MAX_SPLITS + 1) == c["ATTN_ERR_SPLITS"]
    assert _decode(L, k=P + 8) == c["ATTN_ERR_ALIGN"]
    assert _decode(L, op=P + 4) == c["ATTN_ERR_ALIGN"]
    assert _decode(L, bt=P + 2) == c["ATTN_ERR_ALIGN"]


def _decode_ex2(L, flags, **kw):
    a = dict(q=P, k=P, v=P, bt=P, lens=P, S=4, op=P, lp=P, B=2, hq=8, hkv=2, d=128, bs=16, mb=8,
             nb=16, maxlen=128, scale=0.1)
    a.update(kw)
    return L.attn_decode_splitkv_ex2(a["q"], a["k"], a["v"], a["bt"], a["lens"], a["S"], a["op"],
                                     a["lp"], a["B"], a["hq"], a["hkv"], a["d"], a["bs"], a["mb"],
                                     a["nb"], a["maxlen"], a["scale"], -1, 0.0, None, flags, None)


def test_decode_flags_validation(L):
    """Unknown flag bits are refused before anything is launched; the
    argument checks of attn_decode_splitkv_ex apply with the early flag too."""
    c = _lib.status_codes()
    assert _decode_ex2(L, 2) == c["ATTN_ERR_SHAPE"]
    assert _decode_ex2(L, 0x80000000) == c["ATTN_ERR_SHAPE"]
    assert _decode_ex2(L, 1, q=None) == c["ATTN_ERR_NULL"]
    assert _decode_ex2(L, 1, hq=130, hkv=2) == c["ATTN_ERR_GQA"]
    assert _decode_ex2(L, 1, d=80) == c["ATTN_ERR_HEADDIM"]


def _append(L, **kw):
    a = dict(q=P, kn=P, vn=P, k=P, v=P, bt=P, lens=P, S=4, op=P, lp=P, B=2, hq=8, hkv=2, d=128,
             bs=16, mb=8, nb=16, maxlen=128, scale=0.1)
    a.update(kw)
    return L.attn_decode_append_splitkv(a["q"], a["kn"], a["vn"], a["k"], a["v"], a["bt"],
                                        a["lens"], a["S"], a["op"], a["lp"], a["B"], a["hq"],
                                        a["hkv"], a["d"], a["bs"], a["mb"], a["nb"], a["maxlen"],
                                        a["scale"], None)


def _append_ex(L, w=-1, cap=0.0, al=None, **kw):
    a = dict(q=P, kn=P, vn=P, k=P, v=P, bt=P, lens=P, S=4, op=P, lp=P, B=2, hq=8, hkv=2, d=128,
             bs=16, mb=8, nb=16, maxlen=128, scale=0.1)
    a.update(kw)
    return L.attn_decode_append_splitkv_ex(a["q"], a["kn"], a["vn"], a["k"], a["v"], a["bt"],
                                           a["lens"], a["S"], a["op"], a["lp"], a["B"], a["hq"],
                                           a["hkv"], a["d"], a["bs"], a["mb"], a["nb"],
                                           a["maxlen"], a["scale"], w, cap, al, None)


def test_decode_append_ex_validation(L):
    c = _lib.status_codes()
    assert _append_ex(L, kn=None) == c["ATTN_ERR_NULL"]
    assert _append_ex(L, w=-3) == c["ATTN_ERR_SHAPE"]                # window below -1
    assert _append_ex(L, cap=-1.0) == c["ATTN_ERR_SHAPE"]
    assert _append_ex(L, cap=float("nan")) == c["ATTN_ERR_SHAPE"]
    assert _append_ex(L, cap=2.0, al=P) == c["ATTN_ERR_SHAPE"]       # ALiBi with soft-capping
    assert _append_ex(L, w=10, al=P + 2) == c["ATTN_ERR_ALIGN"]      # misaligned slopes
    assert _append_ex(L, w=10, vn=P + 2) == c["ATTN_ERR_ALIGN"]
    assert _append_ex(L, w=10, d=96) == c["ATTN_ERR_HEADDIM"]


def test_decode_append_validation(L):
    c = _lib.status_codes()
    assert _append(L, kn=None) == c["ATTN_ERR_NULL"]
    assert _append(L, vn=None) == c["ATTN_ERR_NULL"]
    assert _append(L, kn=P + 8) == c["ATTN_ERR_ALIGN"]
    assert _append(L, vn=P + 2) == c["ATTN_ERR_ALIGN"]
    # the rest is the plain decode's validation
    assert _append(L, k=None) == c["ATTN_ERR_NULL"]
    assert _append(L, d=80) == c["ATTN_ERR_HEADDIM"]
    assert _append(L, hq=6, hkv=4) == c["ATTN_ERR_GQA"]
    assert _append(L, S=-1) == c["ATTN_ERR_SPLITS"]
    assert _append(L, bs=0) == c["ATTN_ERR_SHAPE"]


def test_combine_validation(L):
    c = _lib.status_codes()
    f = L.attn_combine
    assert f(None, P, 4, 1, 8, 128, P, P, None) == c["ATTN_ERR_NULL"]
    assert f(P, P, 4, 0, 8, 128, P, P, None) == c["ATTN_ERR_SHAPE"]
    assert f(P, P, 4, 1, 8, 32, P, P, None) == c["ATTN_ERR_HEADDIM"]
    assert f(P, P, 4, 1, 8, 512, P, P, None) == c["ATTN_ERR_HEADDIM"]
    assert f(P, P, 0, 1, 8, 128, P, P, None) == c["ATTN_ERR_SPLITS"]
    assert f(P, P, 1025, 1, 8, 128, P, P, None) == c["ATTN_ERR_SPLITS"]
    assert f(P + 8, P, 4, 1, 8, 128, P, P, None) == c["ATTN_ERR_ALIGN"]


def test_split_policy(L):
    f = L.attn_decode_num_splits
    assert f(0, 4, 1000, 152) == 1 and f(1, 4, 0, 152) == 1
    for B, H, Lk, sms in [(1, 4, 30720, 152), (1, 8, 32768, 152), (16, 8, 32768, 152),
                          (3, 1, 77, 152), (1, 1, 1000, 152), (256, 8, 30000, 152),
                          (1, 4, 30720, 148)]:
        s = f(B, H, Lk, sms)
        assert 1 <= s <= _lib.ATTN_MAX_SPLITS
        # splits never cut a sequence into chunks much shorter than 256 tokens
        assert s == 1 or -(-Lk // s) >= 256 - 16
        # small batch: enough (sequence, kv head, split) blocks to cover every SM
        if B * H < sms and Lk >= 256 * sms:
            assert B * H * s >= sms
    # large batch: already enough (sequence, head) pairs -> one split
    assert f(256, 8, 30000, 152) == 1


def _rule(kv_len, S):
    """The split rule as the header states it, restated independently."""
    if kv_len == 0:
        return [(0, 0)] * S
    c = ((kv_len + S - 1) // S + 15) // 16 * 16
    out = []
    for s in range(S):
        lo = min(s * c, kv_len)
        out.append((lo, min(lo + c, kv_len)))
    return out


@pytest.mark.parametrize("kv_len,S", [(30720, 1), (30720, 16), (30720, 148), (1, 4), (17, 2),
                                      (1000, 7), (0, 3), (15, 16)])
def test_split_rule(kv_len, S):
    from gpu_util import split_ranges

    r = split_ranges(kv_len, S)
    assert r == _rule(kv_len, S)
    covered = [t for a, b in r for t in range(a, b)]
    assert covered == list(range(kv_len))            # a partition, in order


def test_header_documents_each_entry_point():
    text = open(os.path.join(ROOT, "include", "attn.h")).read()
    for name in ["attn_prefill", "attn_decode_splitkv", "attn_combine", "attn_decode_num_splits",
                 "attn_decode_append_splitkv", "attn_prefill_varlen"]:
        block = text[:text.index(name + "(")]
        doc = block[block.rindex("/*"):]
        assert "Page:" in doc or "section" in doc, f"{name} lacks its citation"


def _fp8_varlen(L, **kw):
    a = dict(q=P, k=P, v=P, qs=P, ks=P, vs=P, o=P, lse=P, cu=P, S=3, T=512, hq=8, hkv=2, d=128,
             scale=0.1, causal=1)
    a.update(kw)
    return L.attn_prefill_fp8_varlen(a["q"], a["k"], a["v"], a["qs"], a["ks"], a["vs"], a["o"],
                                     a["lse"], a["cu"], a["S"], a["T"], a["hq"], a["hkv"], a["d"],
                                     a["scale"], a["causal"], None)


def test_prefill_fp8_varlen_validation(L):
    c = _lib.status_codes()
    assert _fp8_varlen(L, cu=None) == c["ATTN_ERR_NULL"]
    assert _fp8_varlen(L, vs=None) == c["ATTN_ERR_NULL"]
    assert _fp8_varlen(L, T=500) == c["ATTN_ERR_SHAPE"]      # V^T rows must be 16-byte multiples
    assert _fp8_varlen(L, T=0) == c["ATTN_ERR_SHAPE"]
    assert _fp8_varlen(L, S=513) == c["ATTN_ERR_SHAPE"]
    assert _fp8_varlen(L, d=96) == c["ATTN_ERR_HEADDIM"]
    assert _fp8_varlen(L, d=256) == c["ATTN_ERR_HEADDIM"]
    assert _fp8_varlen(L, hq=6, hkv=4) == c["ATTN_ERR_GQA"]
    assert _fp8_varlen(L, cu=P + 2) == c["ATTN_ERR_ALIGN"]
    assert _fp8_varlen(L, v=P + 8) == c["ATTN_ERR_ALIGN"]


def _quant_varlen(L, **kw):
    a = dict(x=P, codes=P, scales=P, signs=None, cu=P, S=3, T=500, planes=4, d=128)
    a.update(kw)
    return L.attn_quantize_fp8_varlen(a["x"], a["codes"], a["scales"], a["signs"], a["cu"], a["S"],
                                      a["T"], a["planes"], a["d"], None)


def test_quantize_fp8_varlen_validation(L):
    c = _lib.status_codes()
    assert _quant_varlen(L, cu=None) == c["ATTN_ERR_NULL"]
    assert _quant_varlen(L, S=0) == c["ATTN_ERR_SHAPE"]
    assert _quant_varlen(L, planes=0) == c["ATTN_ERR_SHAPE"]
    assert _quant_varlen(L, T=(1 << 24) + 1) == c["ATTN_ERR_SHAPE"]
    assert _quant_varlen(L, d=256) == c["ATTN_ERR_HEADDIM"]
    assert _quant_varlen(L, codes=P + 8) == c["ATTN_ERR_ALIGN"]
    assert _quant_varlen(L, signs=P + 2) == c["ATTN_ERR_ALIGN"]
