"""CPU oracle for TurboQuant speculative-verify attention (test infrastructure).

TEST INFRASTRUCTURE ONLY: the product path (the CUDA library and its Python
binding) never imports this package.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg call it.  It shares no code with the CUDA library.

The arithmetic lives in ``tq_oracle.c`` (plain C, fp32 encoder in a fixed
operation order, fp64 attention); this module compiles it with gcc and wraps it
with ctypes and numpy.  Every function cites the page section it follows in the
C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libtqoracle.so")
_lock = threading.Lock()
_lib = None

PRESET_K8V4 = 0
PRESET_K3V4_NC = 1
PRESET_K3V4 = 2  # k3v4_nc's coding with the plain norm as key factor
PRESET_K3V4_NC_RS = 3  # k3v4_nc with a randomised-sign Hadamard rotation
HEAD_DIM = 128
BLOCK = 16


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off, OpenMP on)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_page_bytes.restype = ctypes.c_long
            lib.oracle_page_bytes.argtypes = [I]
            lib.oracle_h2f.restype = ctypes.c_float
            lib.oracle_h2f.argtypes = [ctypes.c_uint16]
            lib.oracle_d2h_rn.restype = ctypes.c_uint16
            lib.oracle_d2h_rn.argtypes = [ctypes.c_double]
            lib.oracle_f2h_rn.restype = ctypes.c_uint16
            lib.oracle_f2h_rn.argtypes = [ctypes.c_float]
            lib.oracle_e4m3_to_double.restype = ctypes.c_double
            lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_from_half.restype = ctypes.c_uint8
            lib.oracle_e4m3_from_half.argtypes = [ctypes.c_uint16]
            lib.oracle_lloyd_max8.restype = I
            lib.oracle_lloyd_max8.argtypes = [P]
            lib.oracle_codebook16.restype = I
            lib.oracle_codebook16.argtypes = [P]
            lib.oracle_lloyd_max.restype = I
            lib.oracle_lloyd_max.argtypes = [I, P]
            lib.oracle_codebook_n.restype = I
            lib.oracle_codebook_n.argtypes = [I, P]
            lib.oracle_key_bits.restype = I
            lib.oracle_key_bits.argtypes = [I]
            lib.oracle_key_levels.restype = I
            lib.oracle_key_levels.argtypes = [I]
            lib.oracle_quant_index_n.restype = I
            lib.oracle_quant_index_n.argtypes = [ctypes.c_float, P, I]
            lib.oracle_pack_bits.argtypes = [P, I, P]
            lib.oracle_unpack_bits.argtypes = [P, I, P]
            lib.oracle_encode_keyq.argtypes = [P, P, I, P, P, I, I]
            lib.oracle_wht_f32.argtypes = [P]
            lib.oracle_wht_f64.argtypes = [P]
            lib.oracle_tree_sum.restype = ctypes.c_float
            lib.oracle_tree_sum.argtypes = [P]
            lib.oracle_quant_index.restype = I
            lib.oracle_quant_index.argtypes = [ctypes.c_float, P]
            lib.oracle_pack3.argtypes = [P, P]
            lib.oracle_unpack3.argtypes = [P, P]
            lib.oracle_encode_key3.argtypes = [P, P, P, P]
            lib.oracle_splitmix64.restype = ctypes.c_uint64
            lib.oracle_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
            lib.oracle_rs_sign.restype = I
            lib.oracle_rs_sign.argtypes = [I]
            lib.oracle_encode_key8.argtypes = [P, P]
            lib.oracle_encode_value4.argtypes = [P, P, P, P]
            lib.oracle_store.restype = I
            lib.oracle_store.argtypes = [I, P, I, I, P, P, P, I]
            lib.oracle_decode_key.argtypes = [I, P, I, P, P]
            lib.oracle_decode_value.argtypes = [I, P, I, P]
            lib.oracle_visible.restype = I
            lib.oracle_visible.argtypes = [I, I, I, I]
            lib.oracle_verify_rows.restype = I
            lib.oracle_verify_rows.argtypes = [I, P, I, I, P, P, I, P, I, I, I, I, I, P, P]
            lib.oracle_verify.restype = I
            lib.oracle_verify.argtypes = [I, P, I, I, P, P, I, P, I, I, I, I, P]
            lib.oracle_partials.restype = I
            lib.oracle_partials.argtypes = [I, P, I, I, P, P, I, P, I, I, I, I, I, P, P]
            lib.oracle_merge.argtypes = [P, P, ctypes.c_long, I, P]
            lib.oracle_attend_raw.argtypes = [P, I, P, P, P, P, P, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "arrays passed to the oracle must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _u16(a) -> np.ndarray:
    """fp16 data as a contiguous uint16 bit-pattern array."""
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=np.uint16)


# ----------------------------------------------------------------- scalars

def page_bytes(preset: int) -> int:
    return int(_load().oracle_page_bytes(preset))


def h2f(h: int) -> float:
    return float(_load().oracle_h2f(h))


def d2h(x: float) -> int:
    return int(_load().oracle_d2h_rn(x))


def f2h(x: float) -> int:
    return int(_load().oracle_f2h_rn(x))


def e4m3_to_double(b: int) -> float:
    return float(_load().oracle_e4m3_to_double(b))


def e4m3_from_half(h: int) -> int:
    return int(_load().oracle_e4m3_from_half(h))


def lloyd_max8() -> tuple[np.ndarray, int]:
    c = np.zeros(8, np.float64)
    it = _load().oracle_lloyd_max8(_ptr(c))
    return c, int(it)


def codebook16() -> np.ndarray:
    """The k3v4_nc key codebook, fp16 bit patterns, ascending."""
    cb = np.zeros(8, np.uint16)
    _load().oracle_codebook16(_ptr(cb))
    return cb


def lloyd_max(n: int) -> tuple[np.ndarray, int]:
    """n-level Lloyd-Max levels of the standard normal (fp64) and the iteration count."""
    c = np.zeros(n, np.float64)
    it = _load().oracle_lloyd_max(n, _ptr(c))
    return c, int(it)


def codebook_n(n: int) -> np.ndarray:
    """n-level key codebook for N(0, 1/128), fp16 bit patterns, ascending."""
    cb = np.zeros(n, np.uint16)
    _load().oracle_codebook_n(n, _ptr(cb))
    return cb


def key_bits(preset: int) -> int:
    return int(_load().oracle_key_bits(preset))


def key_levels(preset: int) -> int:
    return int(_load().oracle_key_levels(preset))


def codebook(preset: int) -> np.ndarray:
    """The key codebook of a coded-key preset (fp16 bit patterns)."""
    return codebook_n(key_levels(preset))


def wht_f32(x) -> np.ndarray:
    t = np.ascontiguousarray(x, dtype=np.float32).copy()
    _load().oracle_wht_f32(_ptr(t))
    return t


def wht_f64(x) -> np.ndarray:
    t = np.ascontiguousarray(x, dtype=np.float64).copy()
    _load().oracle_wht_f64(_ptr(t))
    return t


def tree_sum(a) -> float:
    a = np.ascontiguousarray(a, dtype=np.float32)
    return float(_load().oracle_tree_sum(_ptr(a)))


def quant_index(y: float, cb: np.ndarray | None = None) -> int:
    cb = codebook16() if cb is None else _u16(cb)
    return int(_load().oracle_quant_index(ctypes.c_float(y), _ptr(cb)))


def quant_index_n(y: float, cb) -> int:
    cb = _u16(cb)
    return int(_load().oracle_quant_index_n(ctypes.c_float(y), _ptr(cb), len(cb)))


def pack_bits(idx, bits: int) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    out = np.zeros(HEAD_DIM * bits // 8, np.uint8)
    _load().oracle_pack_bits(_ptr(idx), bits, _ptr(out))
    return out


def unpack_bits(b, bits: int) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.zeros(HEAD_DIM, np.uint8)
    _load().oracle_unpack_bits(_ptr(b), bits, _ptr(out))
    return out


def encode_keyq(k, bits: int, corrected: bool = True) -> tuple[np.ndarray, int]:
    """Coded key with a 2^bits-level codebook: (code bytes, fp16 key factor bits)."""
    k = _u16(k)
    cb = codebook_n(1 << bits)
    codes = np.zeros(HEAD_DIM * bits // 8, np.uint8)
    nc = np.zeros(1, np.uint16)
    _load().oracle_encode_keyq(_ptr(k), _ptr(cb), bits, _ptr(codes), _ptr(nc), int(corrected), 0)
    return codes, int(nc[0])


def pack3(idx) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.uint8)
    out = np.zeros(48, np.uint8)
    _load().oracle_pack3(_ptr(idx), _ptr(out))
    return out


def unpack3(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint8)
    out = np.zeros(HEAD_DIM, np.uint8)
    _load().oracle_unpack3(_ptr(b), _ptr(out))
    return out


def splitmix64(seed: int, j: int) -> int:
    """Output j (0-based) of SplitMix64 seeded with seed."""
    return int(_load().oracle_splitmix64(seed, j))


def rs_signs() -> np.ndarray:
    """The sign vector s of preset k3v4_nc_rs (keys rotated by H diag(s))."""
    return np.array([_load().oracle_rs_sign(j) for j in range(128)], np.int32)


def encode_key3(k) -> tuple[np.ndarray, int]:
    k = _u16(k)
    cb = codebook16()
    codes = np.zeros(48, np.uint8)
    nc = np.zeros(1, np.uint16)
    _load().oracle_encode_key3(_ptr(k), _ptr(cb), _ptr(codes), _ptr(nc))
    return codes, int(nc[0])


def encode_key8(k) -> np.ndarray:
    k = _u16(k)
    out = np.zeros(HEAD_DIM, np.uint8)
    _load().oracle_encode_key8(_ptr(k), _ptr(out))
    return out


def encode_value4(v) -> tuple[np.ndarray, int, int]:
    """Returns (codes uint8[128] in 0..15, scale fp16 bits, zero fp16 bits)."""
    v = _u16(v)
    out = np.zeros(HEAD_DIM, np.uint8)
    s = np.zeros(1, np.uint16)
    z = np.zeros(1, np.uint16)
    _load().oracle_encode_value4(_ptr(v), _ptr(out), _ptr(s), _ptr(z))
    return out, int(s[0]), int(z[0])


def decode_key(preset: int, page: np.ndarray, off: int) -> np.ndarray:
    page = np.ascontiguousarray(page, dtype=np.uint8)
    cb = codebook(preset) if key_bits(preset) else codebook16()
    out = np.zeros(HEAD_DIM, np.float64)
    _load().oracle_decode_key(preset, _ptr(page), off, _ptr(cb), _ptr(out))
    return out


def decode_value(preset: int, page: np.ndarray, off: int) -> np.ndarray:
    page = np.ascontiguousarray(page, dtype=np.uint8)
    out = np.zeros(HEAD_DIM, np.float64)
    _load().oracle_decode_value(preset, _ptr(page), off, _ptr(out))
    return out


def visible(L: int, n_spec: int, n: int, causal: bool) -> int:
    return int(_load().oracle_visible(L, n_spec, n, int(causal)))


# ----------------------------------------------------------------- arrays

def store(preset: int, cache: np.ndarray, k, v, slot_mapping) -> np.ndarray:
    """Encode T tokens into ``cache`` (uint8 [num_blocks][Hk][page]) in place.
    k, v: fp16 [T][Hk][D]; slot_mapping int32 [T]."""
    assert cache.dtype == np.uint8 and cache.ndim == 3 and cache.flags["C_CONTIGUOUS"]
    nb, hk, pb = cache.shape
    assert pb == page_bytes(preset)
    k = _u16(k)
    v = _u16(v)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    T = sm.shape[0]
    assert k.shape == (T, hk, HEAD_DIM) and v.shape == (T, hk, HEAD_DIM)
    rc = _load().oracle_store(preset, _ptr(cache), nb, hk, _ptr(k), _ptr(v), _ptr(sm), T)
    assert rc == 0
    return cache


def verify(preset: int, cache: np.ndarray, q, block_table, seq_lens, causal: bool = True,
           rows=None) -> np.ndarray:
    """fp64 spec-verify attention.  q fp16 [n_spec][B][Hq][D].  Returns
    [n_spec][B][Hq][D], or [len(rows)][D] when ``rows`` lists (n, b, h)."""
    nb, hk, _ = cache.shape
    q = _u16(q)
    n_spec, B, Hq, _ = q.shape
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    assert bt.shape[0] == B and sl.shape == (B,)
    lib = _load()
    if rows is None:
        out = np.zeros((n_spec, B, Hq, HEAD_DIM), np.float64)
        rc = lib.oracle_verify(preset, _ptr(cache), nb, hk, _ptr(q), _ptr(bt), bt.shape[1], _ptr(sl),
                               n_spec, B, Hq, int(causal), _ptr(out))
    else:
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        out = np.zeros((r.shape[0], HEAD_DIM), np.float64)
        rc = lib.oracle_verify_rows(preset, _ptr(cache), nb, hk, _ptr(q), _ptr(bt), bt.shape[1],
                                    _ptr(sl), n_spec, B, Hq, int(causal), r.shape[0], _ptr(r),
                                    _ptr(out))
    assert rc == 0
    return out


def partials(preset: int, cache: np.ndarray, q, block_table, seq_lens, num_kv_splits: int,
             causal: bool = True) -> tuple[np.ndarray, np.ndarray]:
    """Split-KV partials: o [n_spec][B][Hq][S][D], lse [n_spec][B][Hq][S] (natural log)."""
    nb, hk, _ = cache.shape
    q = _u16(q)
    n_spec, B, Hq, _ = q.shape
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    S = int(num_kv_splits)
    po = np.zeros((n_spec, B, Hq, S, HEAD_DIM), np.float64)
    pl = np.zeros((n_spec, B, Hq, S), np.float64)
    rc = _load().oracle_partials(preset, _ptr(cache), nb, hk, _ptr(q), _ptr(bt), bt.shape[1],
                                 _ptr(sl), n_spec, B, Hq, S, int(causal), _ptr(po), _ptr(pl))
    assert rc == 0
    return po, pl


def merge(part_o, part_lse) -> np.ndarray:
    """Stage-2 log-sum-exp merge.  part_o [..., S, D], part_lse [..., S]."""
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    S = pl.shape[-1]
    lead = pl.shape[:-1]
    nrows = int(np.prod(lead)) if lead else 1
    out = np.zeros(lead + (HEAD_DIM,), np.float64)
    _load().oracle_merge(_ptr(po), _ptr(pl), nrows, S, _ptr(out))
    return out


def attend_raw(q, k, v, lo, hi) -> tuple[np.ndarray, np.ndarray]:
    """Quantisation-bypass attention: q fp16 [nr][D], k/v fp16 [L][D], rows see
    positions [lo_r, hi_r).  Returns (out fp64 [nr][D], lse [nr])."""
    q = _u16(q)
    k = _u16(k)
    v = _u16(v)
    lo = np.ascontiguousarray(lo, dtype=np.int32)
    hi = np.ascontiguousarray(hi, dtype=np.int32)
    nr = q.shape[0]
    out = np.zeros((nr, HEAD_DIM), np.float64)
    lse = np.zeros(nr, np.float64)
    _load().oracle_attend_raw(_ptr(q), nr, _ptr(k), _ptr(v), _ptr(lo), _ptr(hi), _ptr(out), _ptr(lse))
    return out, lse
