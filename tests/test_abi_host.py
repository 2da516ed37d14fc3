"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports every declared entry point; helper values; argument validation rejects
bad calls before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest

from quantized_kv_cache_store_gb300 import _build, tqkv

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "tqkv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tqkv.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"tq_store", "tq_verify_stage1", "tq_verify_stage2", "tq_page_bytes",
            "tq_partials_bytes", "tq_codebook", "tq_status_string", "tq_device_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_page_and_partials_bytes(lib):
    assert tqkv.tq_page_bytes(0) == 3136 and tqkv.tq_page_bytes(1) == 1920 and tqkv.tq_page_bytes(2) == 1920
    assert tqkv.tq_page_bytes(3) == 1920
    assert tqkv.tq_page_bytes(4) == 2176 and tqkv.tq_page_bytes(5) == 1664
    assert tqkv.tq_page_bytes(7) == 0
    assert tqkv.tq_partials_bytes(8, 4, 32, 8) == 8 * 4 * 32 * 8 * 129 * 4
    assert tqkv.tq_partials_bytes(0, 4, 32, 8) == 0


def test_status_strings(lib):
    for s in range(6):
        assert tqkv.tq_status_string(s) and tqkv.tq_status_string(s) != "unknown status"
    assert tqkv.tq_status_string(99) == "unknown status"


def test_codebook_matches_oracle(lib, oracle_lib):
    ours = tqkv.tq_codebook(1)
    ref = oracle_lib.codebook16().view(np.float16).astype(np.float32)
    assert np.array_equal(ours, ref)
    for preset, n in ((2, 8), (3, 8), (4, 16), (5, 4)):
        assert tqkv.tq_key_levels(preset) == n == oracle_lib.key_levels(preset)
        ref = oracle_lib.codebook_n(n).view(np.float16).astype(np.float32)
        assert np.array_equal(tqkv.tq_codebook(preset), ref)
    assert tqkv.tq_key_levels(0) == 0 and tqkv.tq_key_levels(9) == 0
    out = np.zeros(8, np.float32)
    assert lib.tq_codebook(0, ctypes.c_void_p(out.ctypes.data)) == tqkv.TQ_ERR_UNSUPPORTED
    assert lib.tq_codebook(1, None) == tqkv.TQ_ERR_INVALID_ARG


def _desc(preset=0, hk=4, nb=8, ptr=0x10000, head_dim=128, block=16, reserved=0):
    return tqkv.tq_cache_desc(preset, head_dim, block, hk, nb, reserved, ptr)


FAKE = 0x7f0000000000  # 16-byte aligned fake device address; never dereferenced on these paths


def _s1(lib, d, q=FAKE, bt=FAKE, mb=4, sl=FAKE, n=8, B=1, Hq=32, S=2, causal=1, po=FAKE, pl=FAKE):
    return lib.tq_verify_stage1(ctypes.byref(d) if d is not None else None, q, bt, mb, sl, n, B, Hq, S,
                                causal, po, pl, None)


def test_store_validation(lib):
    P = ctypes.c_void_p
    st = lambda d, k=FAKE, v=FAKE, s=FAKE, T=4: lib.tq_store(ctypes.byref(d) if d else None, P(k), P(v),
                                                             P(s), T, None)
    assert st(None) == tqkv.TQ_ERR_INVALID_ARG
    assert st(_desc(ptr=0)) == tqkv.TQ_ERR_INVALID_ARG
    assert st(_desc(preset=6, ptr=FAKE)) == tqkv.TQ_ERR_UNSUPPORTED
    assert st(_desc(head_dim=64, ptr=FAKE)) == tqkv.TQ_ERR_UNSUPPORTED
    assert st(_desc(block=32, ptr=FAKE)) == tqkv.TQ_ERR_UNSUPPORTED
    assert st(_desc(hk=0, ptr=FAKE)) == tqkv.TQ_ERR_INVALID_ARG
    assert st(_desc(reserved=1, ptr=FAKE)) == tqkv.TQ_ERR_INVALID_ARG
    assert st(_desc(ptr=FAKE + 8)) == tqkv.TQ_ERR_MISALIGNED
    assert st(_desc(ptr=FAKE), k=0) == tqkv.TQ_ERR_INVALID_ARG
    assert st(_desc(ptr=FAKE), k=FAKE + 2) == tqkv.TQ_ERR_MISALIGNED
    assert st(_desc(ptr=FAKE), s=FAKE + 2) == tqkv.TQ_ERR_MISALIGNED
    assert st(_desc(ptr=FAKE), T=-1) == tqkv.TQ_ERR_INVALID_ARG
    assert st(_desc(ptr=FAKE), T=0) == tqkv.TQ_OK  # nothing to enqueue


def test_stage1_validation(lib):
    d = _desc(ptr=FAKE)
    assert _s1(lib, None) == tqkv.TQ_ERR_INVALID_ARG
    assert _s1(lib, d, q=0) == tqkv.TQ_ERR_INVALID_ARG
    assert _s1(lib, d, n=0) == tqkv.TQ_ERR_INVALID_ARG
    assert _s1(lib, d, n=129) == tqkv.TQ_ERR_UNSUPPORTED     # more than 128 query tokens per sequence
    assert _s1(lib, d, Hq=30) == tqkv.TQ_ERR_INVALID_ARG       # Hq % Hk != 0
    assert _s1(lib, d, n=64, Hq=128) == tqkv.TQ_ERR_UNSUPPORTED  # 64 x 32 rows per kv-head > 1024
    assert _s1(lib, d, S=0) == tqkv.TQ_ERR_INVALID_ARG
    assert _s1(lib, d, S=70000) == tqkv.TQ_ERR_UNSUPPORTED
    assert _s1(lib, d, causal=2) == tqkv.TQ_ERR_INVALID_ARG
    assert _s1(lib, d, mb=0) == tqkv.TQ_ERR_INVALID_ARG
    assert _s1(lib, d, q=FAKE + 4) == tqkv.TQ_ERR_MISALIGNED
    assert _s1(lib, d, po=FAKE + 4) == tqkv.TQ_ERR_MISALIGNED
    assert _s1(lib, d, sl=FAKE + 1) == tqkv.TQ_ERR_MISALIGNED
    assert _s1(lib, d, B=-1) == tqkv.TQ_ERR_INVALID_ARG
    assert _s1(lib, d, B=0) == tqkv.TQ_OK  # nothing to enqueue


def test_stage2_validation(lib):
    s2 = lambda po=FAKE, pl=FAKE, n=8, B=1, Hq=8, D=128, S=2, out=FAKE: lib.tq_verify_stage2(
        po, pl, n, B, Hq, D, S, out, None)
    assert s2(po=0) == tqkv.TQ_ERR_INVALID_ARG
    assert s2(out=0) == tqkv.TQ_ERR_INVALID_ARG
    assert s2(S=0) == tqkv.TQ_ERR_INVALID_ARG
    assert s2(D=64) == tqkv.TQ_ERR_UNSUPPORTED
    assert s2(out=FAKE + 4) == tqkv.TQ_ERR_MISALIGNED
    assert s2(pl=FAKE + 2) == tqkv.TQ_ERR_MISALIGNED


def test_single_call_validation(lib):
    d = _desc(ptr=FAKE)
    v = lambda q=FAKE, t=FAKE, out=FAKE, S=2, B=1: lib.tq_verify(ctypes.byref(d), q, FAKE, 4, FAKE, 8, B, 32, S, 1,
                                                               FAKE, FAKE, t, out, None)
    assert v(out=0) == tqkv.TQ_ERR_INVALID_ARG
    assert v(t=0) == tqkv.TQ_ERR_INVALID_ARG
    assert v(t=FAKE + 2) == tqkv.TQ_ERR_MISALIGNED
    assert v(out=FAKE + 4) == tqkv.TQ_ERR_MISALIGNED
    assert v(q=0) == tqkv.TQ_ERR_INVALID_ARG
    assert v(S=0) == tqkv.TQ_ERR_INVALID_ARG
    assert v(B=0) == tqkv.TQ_OK  # nothing to enqueue


def test_store_verify_validation(lib):
    d = _desc(ptr=FAKE)
    v = lambda k=FAKE, vv=FAKE, q=FAKE, t=FAKE, out=FAKE, B=1: lib.tq_store_verify(
        ctypes.byref(d), k, vv, q, FAKE, 4, FAKE, 8, B, 32, 2, 1, FAKE, FAKE, t, out, None)
    assert v(k=0) == tqkv.TQ_ERR_INVALID_ARG
    assert v(vv=0) == tqkv.TQ_ERR_INVALID_ARG
    assert v(out=0) == tqkv.TQ_ERR_INVALID_ARG
    assert v(k=FAKE + 8) == tqkv.TQ_ERR_MISALIGNED
    assert v(vv=FAKE + 2) == tqkv.TQ_ERR_MISALIGNED
    assert v(t=FAKE + 2) == tqkv.TQ_ERR_MISALIGNED
    assert v(q=0) == tqkv.TQ_ERR_INVALID_ARG
    assert v(B=0) == tqkv.TQ_OK  # nothing to enqueue


def test_header_enums_match_the_binding():
    """The preset and status values the header declares are the binding's and
    the input recipe's."""
    from quantized_kv_cache_store_gb300 import inputs

    text = open(HEADER).read()
    decl = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(TQ_[A-Z0-9_]+)\s*=\s*(\d+)", text)}
    for name in ("TQ_OK", "TQ_ERR_INVALID_ARG", "TQ_ERR_UNSUPPORTED", "TQ_ERR_MISALIGNED", "TQ_ERR_CUDA",
                 "TQ_ERR_TIMEOUT", "TQ_PRESET_K8V4", "TQ_PRESET_K3V4_NC", "TQ_PRESET_K3V4", "TQ_PRESET_K3V4_NC_RS",
                 "TQ_PRESET_K4V4_NC", "TQ_PRESET_K2V4_NC"):
        assert decl[name] == getattr(tqkv, name), name
    assert tqkv.PRESETS == inputs.PRESETS
    for preset in tqkv.PRESETS.values():
        assert tqkv.tq_page_bytes(preset) > 0
