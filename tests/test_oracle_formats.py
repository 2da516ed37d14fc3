"""Pins for the oracle's number formats: fp16 and e4m3 conversions.

Each conversion is checked against an independent library routine (numpy's
float16, torch's float8_e4m3fn) and, for e4m3, against exhaustive brute force
(nearest representable value, ties to the even code)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_h2f_exhaustive(oracle_lib):
    O = oracle_lib
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([O.h2f(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f2h_matches_numpy(oracle_lib):
    O = oracle_lib
    rng = np.random.default_rng(7)
    xs = [rng.standard_normal(3000).astype(np.float32) * s for s in (1e-8, 1e-6, 1e-4, 1.0, 1e3, 6e4)]
    edges = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e9, np.inf, -np.inf,
                      2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -25 * 1.0000001, 2.0 ** -14,
                      2.0 ** -14 - 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
                      2049.0, 2051.0, 4097.0], np.float32)
    xs = np.concatenate(xs + [edges])
    ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([O.f2h(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


def test_d2h_matches_numpy(oracle_lib):
    O = oracle_lib
    rng = np.random.default_rng(8)
    xs = np.concatenate([rng.standard_normal(2000) * s for s in (1e-6, 0.1, 1.0, 100.0)])
    ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([O.d2h(float(x)) for x in xs], np.uint16)
    assert np.array_equal(got, ref)


def _e4m3_table():
    """Decoded value of every e4m3 code, written from the format definition
    (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, subnormals at
    exponent 0, S.1111.111 = NaN, no infinities)."""
    vals = np.zeros(256)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            vals[c] = np.nan
            continue
        v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        vals[c] = -v if s else v
    return vals


def test_e4m3_decode_all_codes(oracle_lib):
    O = oracle_lib
    ours = np.array([O.e4m3_to_double(c) for c in range(256)])
    table = _e4m3_table()
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for ref in (table, lib):
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(ours), nan)
        assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_encode_exhaustive_bruteforce(oracle_lib):
    """All 65,536 fp16 inputs: nearest e4m3 value, ties to the even code,
    |x| >= 448 saturates to +-448, NaN -> 0x7F, sign kept (also for zero)."""
    O = oracle_lib
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16).astype(np.float64)
    got = np.array([O.e4m3_from_half(int(b)) for b in bits], np.uint8)
    table = _e4m3_table()
    pos = table[:127]  # codes 0x00..0x7E, non-negative finite, ascending
    assert np.all(np.diff(pos) > 0)
    a = np.abs(x)
    sign = np.signbit(x).astype(np.uint8) << 7
    exp = np.zeros(65536, np.uint8)
    fin = np.isfinite(a) & (a < 448.0)
    d = np.abs(a[fin, None] - pos[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    codes = np.arange(127)
    # among the nearest codes, the even one wins a tie
    pick = np.where(cand & (codes[None, :] % 2 == 0), codes[None, :], 1000).min(axis=1)
    single = cand.sum(axis=1) == 1
    pick[single] = np.argmax(cand[single], axis=1)
    exp[fin] = pick.astype(np.uint8)
    exp[np.isfinite(a) & (a >= 448.0)] = 0x7E
    exp[np.isinf(a)] = 0x7E
    exp = exp | sign
    exp[np.isnan(x)] = 0x7F
    assert np.array_equal(got, exp)


def test_e4m3_encode_matches_torch_in_range(oracle_lib):
    O = oracle_lib
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = bits.view(np.float16)
    ok = np.isfinite(x) & (np.abs(x.astype(np.float32)) < 448.0)
    ref = torch.from_numpy(x[ok].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([O.e4m3_from_half(int(b)) for b in bits[ok]], np.uint8)
    assert np.array_equal(got, ref)
