"""Pins for the other key widths: the 16-level (k4v4_nc) and 4-level
(k2v4_nc) Lloyd-Max codebooks, b-bit packing and the coded-key encoder.

The levels are compared with Max's published table and re-checked against
Lloyd's conditions by quadrature (scipy), an independent route from the
oracle's closed-form cell means; packing is compared with a big-integer bit
stream; cell indices with a brute-force nearest-centroid search."""
import os

import numpy as np
import pytest
from scipy import integrate, stats

D = 128
GOLD = os.path.join(os.path.dirname(__file__), "golden")
WIDTHS = {4: ("lloyd_max_gaussian_16level.txt", 16), 2: ("lloyd_max_gaussian_4level.txt", 4)}
PRESET_OF_BITS = {4: 4, 2: 5, 3: 1}


def _golden(name):
    out = {}
    for line in open(os.path.join(GOLD, name)):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = line.split("=", 1)
            out[k.strip()] = [float(t) for t in v.split()]
    return out


def _cells(c):
    return np.concatenate([[-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]])


@pytest.mark.parametrize("bits", [4, 2])
def test_matches_max_table(oracle_lib, bits):
    name, n = WIDTHS[bits]
    g = _golden(name)
    c, it = oracle_lib.lloyd_max(n)
    assert it > 0 and np.all(np.diff(c) > 0)
    h = n // 2
    assert np.allclose(c[h:], g["levels"], atol=6e-4)
    assert np.allclose(-c[:h][::-1], g["levels"], atol=6e-4)
    assert np.allclose(_cells(c)[1:-1][h - 1:], g["boundaries"], atol=6e-4)
    bb = _cells(c)
    mse = sum(integrate.quad(lambda x: (x - c[m]) ** 2 * stats.norm.pdf(x), bb[m], bb[m + 1], epsabs=1e-14)[0]
              for m in range(n))
    assert abs(mse / g["mse"][0] - 1) < 2e-3


@pytest.mark.parametrize("n", [4, 16])
def test_lloyd_conditions_by_quadrature(oracle_lib, n):
    c, _ = oracle_lib.lloyd_max(n)
    b = _cells(c)
    for m in range(n):
        num = integrate.quad(lambda x: x * stats.norm.pdf(x), b[m], b[m + 1], epsabs=1e-14, epsrel=1e-13)[0]
        den = integrate.quad(stats.norm.pdf, b[m], b[m + 1], epsabs=1e-14, epsrel=1e-13)[0]
        assert abs(num / den - c[m]) < 1e-9


def test_eight_levels_unchanged(oracle_lib):
    c8, _ = oracle_lib.lloyd_max8()
    c, _ = oracle_lib.lloyd_max(8)
    assert np.array_equal(c, c8)
    assert np.array_equal(oracle_lib.codebook_n(8), oracle_lib.codebook16())


@pytest.mark.parametrize("n", [4, 16])
def test_codebook_is_scaled_levels(oracle_lib, n):
    c, _ = oracle_lib.lloyd_max(n)
    cb = oracle_lib.codebook_n(n)
    assert np.array_equal(cb, (c / np.sqrt(128.0)).astype(np.float16).view(np.uint16))
    f = cb.view(np.float16).astype(np.float64)
    assert np.array_equal(f, -f[::-1]) and np.all(np.diff(f) > 0)


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_bits_definition(oracle_lib, bits):
    rng = np.random.default_rng(40 + bits)
    n = 1 << bits
    pats = [np.zeros(D, np.uint8), np.full(D, n - 1, np.uint8), (np.arange(D) % n).astype(np.uint8)]
    pats += [rng.integers(0, n, D).astype(np.uint8) for _ in range(20)]
    for idx in pats:
        packed = oracle_lib.pack_bits(idx, bits)
        stream = 0
        for j, c in enumerate(idx):
            stream |= int(c) << (bits * j)
        assert bytes(packed) == stream.to_bytes(D * bits // 8, "little")
        assert np.array_equal(oracle_lib.unpack_bits(packed, bits), idx)
    if bits == 3:
        idx = rng.integers(0, 8, D).astype(np.uint8)
        assert np.array_equal(oracle_lib.pack_bits(idx, 3), oracle_lib.pack3(idx))


@pytest.mark.parametrize("n", [4, 16])
def test_quant_index_is_nearest_centroid(oracle_lib, n):
    """The cell index equals a brute-force nearest-centroid search (ties,
    which sit exactly on an fp32 midpoint, go to the lower level)."""
    cb16 = oracle_lib.codebook_n(n)
    cb = cb16.view(np.float16).astype(np.float64)
    rng = np.random.default_rng(n)
    ys = np.concatenate([rng.standard_normal(3000) / np.sqrt(D), cb, 0.5 * (cb[:-1] + cb[1:]), [0.0, -1.0, 1.0]])
    for y in ys.astype(np.float32):
        d = np.abs(float(y) - cb)
        best = int(np.flatnonzero(d == d.min())[0])
        assert oracle_lib.quant_index_n(float(y), cb16) == best


def _H():
    h = np.array([[1.0]])
    while h.shape[0] < D:
        h = np.block([[h, h], [h, -h]])
    return h


@pytest.mark.parametrize("bits", [2, 4])
def test_centroid_vectors_round_trip(oracle_lib, bits):
    """A key built as a multiple of H c (c a vector of centroids) is coded back to c,
    and the stored page decodes to the key up to the fp16 factor."""
    O = oracle_lib
    n = 1 << bits
    cb = O.codebook_n(n).view(np.float16).astype(np.float64)
    bnd = 0.5 * (cb[:-1] + cb[1:])
    rng = np.random.default_rng(60 + bits)
    done = 0
    while done < 20:
        # the encoder codes y = c / |c| for k = 2 H c: take idx at a fixed point
        # of idx -> cell(c[idx] / |c[idx]|), away from every boundary
        idx = np.searchsorted(bnd, rng.standard_normal(D) / np.sqrt(D), side="left")
        for _ in range(10):
            y = cb[idx] / np.linalg.norm(cb[idx])
            nxt = np.searchsorted(bnd, y, side="left")
            if np.array_equal(nxt, idx):
                break
            idx = nxt
        if not np.array_equal(nxt, idx) or np.min(np.abs(y[:, None] - bnd[None, :])) < 1e-4:
            continue
        done += 1
        idx = idx.astype(np.uint8)
        k = (2.0 * (_H() @ cb[idx])).astype(np.float16)
        codes, nc = O.encode_keyq(k, bits)
        assert np.array_equal(O.unpack_bits(codes, bits), idx)
        preset = PRESET_OF_BITS[bits]
        cache = np.zeros((1, 1, O.page_bytes(preset)), np.uint8)
        O.store(preset, cache, k.reshape(1, 1, D), np.zeros((1, 1, D), np.float16), np.array([0], np.int32))
        assert np.array_equal(cache[0, 0, :D * bits // 8], codes)
        kh = O.decode_key(preset, cache[0, 0], 0)
        kk = k.astype(np.float64)
        assert np.max(np.abs(kh - kk)) <= 2.0 ** -9 * np.max(np.abs(kk))


@pytest.mark.parametrize("bits,d", [(4, 0.009497), (2, 0.1175), (3, 0.03454)])
def test_distortion_matches_lloyd_max(oracle_lib, bits, d):
    """Mean relative squared error of norm-corrected keys: the rescaled
    reconstruction has cos = sqrt(1 - d), so the relative error is
    2 - 2 sqrt(1 - d) (high-dimension limit), d from Max's table."""
    O = oracle_lib
    preset = PRESET_OF_BITS[bits]
    rng = np.random.default_rng(70 + bits)
    errs = []
    for _ in range(600):
        k = rng.standard_normal(D).astype(np.float16)
        cache = np.zeros((1, 1, O.page_bytes(preset)), np.uint8)
        O.store(preset, cache, k.reshape(1, 1, D), np.zeros((1, 1, D), np.float16), np.array([0], np.int32))
        kh = O.decode_key(preset, cache[0, 0], 0)
        kk = k.astype(np.float64)
        errs.append(np.sum((kk - kh) ** 2) / np.sum(kk ** 2))
    expect = 2 - 2 * np.sqrt(1 - d)
    assert abs(np.mean(errs) / expect - 1) < 0.06


def test_page_sizes_and_layout(oracle_lib):
    """Slots 134 B (k4v4_nc) and 102 B (k2v4_nc), rounded up to 4 bytes like
    k3v4_nc's 118 -> 120; the value fields follow the key factor."""
    O = oracle_lib
    assert O.page_bytes(4) == 16 * 136 and O.page_bytes(5) == 16 * 104
    rng = np.random.default_rng(9)
    for preset, bits in ((4, 4), (5, 2)):
        k = rng.standard_normal((3, 1, D)).astype(np.float16)
        v = rng.standard_normal((3, 1, D)).astype(np.float16)
        cache = np.zeros((1, 1, O.page_bytes(preset)), np.uint8)
        O.store(preset, cache, k, v, np.array([0, 5, 15], np.int32))
        page = cache[0, 0]
        cbytes = D * bits // 8
        vo = 16 * cbytes + 32
        for t, off in enumerate((0, 5, 15)):
            codes, nc = O.encode_keyq(k[t, 0], bits)
            assert np.array_equal(page[off * cbytes:(off + 1) * cbytes], codes)
            assert int(page[16 * cbytes + 2 * off]) | (int(page[16 * cbytes + 2 * off + 1]) << 8) == nc
            code, s, z = O.encode_value4(v[t, 0])
            got = [(page[vo + 8 * d + off // 2] >> (4 * (off % 2))) & 15 for d in range(D)]
            assert np.array_equal(np.array(got, np.uint8), code)
            so, zo = vo + 1024, vo + 1024 + 32
            assert int(page[so + 2 * off]) | (int(page[so + 2 * off + 1]) << 8) == s
            assert int(page[zo + 2 * off]) | (int(page[zo + 2 * off + 1]) << 8) == z
        assert not page[zo + 32:].any()  # padding
