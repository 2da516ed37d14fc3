"""Pins for the oracle's encoder: rotation, centroid coding, bit packing, norm
correction, value quantisation and the page layout."""
import numpy as np
import pytest

D = 128


def _H():
    i = np.arange(D)
    pc = np.vectorize(lambda x: bin(x).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1.0, -1.0)


# ----------------------------------------------------------------- rotation

def test_wht_is_sylvester_hadamard(oracle_lib):
    O = oracle_lib
    H = _H()
    M32 = np.stack([O.wht_f32(np.eye(D)[j]) for j in range(D)], axis=1)
    M64 = np.stack([O.wht_f64(np.eye(D)[j]) for j in range(D)], axis=1)
    assert np.array_equal(M32, H)
    assert np.array_equal(M64, H)
    assert np.array_equal(H @ H.T, D * np.eye(D))


def test_wht_twice_scales_by_D(oracle_lib):
    rng = np.random.default_rng(1)
    x = rng.integers(-50, 50, D).astype(np.float64)
    assert np.array_equal(oracle_lib.wht_f64(oracle_lib.wht_f64(x)), D * x)
    assert np.array_equal(oracle_lib.wht_f32(oracle_lib.wht_f32(x)), (D * x).astype(np.float32))


def test_wht_matches_matrix_product(oracle_lib):
    rng = np.random.default_rng(2)
    H = _H()
    for _ in range(5):
        x = rng.standard_normal(D)
        assert np.allclose(oracle_lib.wht_f64(x), H @ x, atol=1e-12, rtol=0)
        x16 = x.astype(np.float16).astype(np.float64)
        y = oracle_lib.wht_f32(x16)
        assert np.allclose(y, H @ x16, atol=1e-5, rtol=0)


def test_tree_sum_close_to_exact(oracle_lib):
    rng = np.random.default_rng(3)
    for _ in range(20):
        a = (rng.standard_normal(D) ** 2).astype(np.float32)
        exact = float(np.sum(a.astype(np.float64)))
        assert abs(oracle_lib.tree_sum(a) - exact) <= 8 * np.spacing(np.float32(exact))
    ints = rng.integers(0, 1000, D).astype(np.float32)
    assert oracle_lib.tree_sum(ints) == float(ints.sum())


def test_tree_sum_association_order(oracle_lib):
    """The documented order, fixed by hand on inputs where fp32 rounding
    (spacing 2 at 2^24, ties to even) tells the orders apart:
    lane partials p_l = (a[4l] + a[4l+1]) + (a[4l+2] + a[4l+3]), then
    p_l <- p_l + p_(l xor off) for off = 16, 8, 4, 2, 1."""
    big = np.float32(2.0 ** 24)
    # within a lane: (2^24 + 1) + (1 + 1) = 2^24 + 2 (the first sum ties to
    # 2^24); left to right gives 2^24, right to left 2^24 + 4
    a = np.zeros(D, np.float32)
    a[0], a[1], a[2], a[3] = big, 1, 1, 1
    assert oracle_lib.tree_sum(a) == 2.0 ** 24 + 2
    # across lanes: lanes 1 and 17 meet first (offset 16) and give 2, added to
    # lane 0's 2^24 last (offset 1): 2^24 + 2; with offset 1 first, each 1
    # meets 2^24 alone and ties away: 2^24
    a = np.zeros(D, np.float32)
    a[0], a[4], a[68] = big, 1, 1
    assert oracle_lib.tree_sum(a) == 2.0 ** 24 + 2
    # offset 8 before offset 2: lanes 2 and 10 (1 each) meet at offset 8,
    # then join lane 0 at offset 2
    a = np.zeros(D, np.float32)
    a[0], a[8], a[40] = big, 1, 1
    assert oracle_lib.tree_sum(a) == 2.0 ** 24 + 2


# ---------------------------------------------------------- centroid coding

def test_quant_index_cells(oracle_lib):
    O = oracle_lib
    cb16 = O.codebook16()
    cb = cb16.view(np.float16).astype(np.float32)
    for m in range(8):
        assert O.quant_index(float(cb[m]), cb16) == m
    for m in range(7):
        bm = np.float32((np.float64(cb[m]) + np.float64(cb[m + 1])) / 2)
        assert O.quant_index(float(bm), cb16) == m            # a tie goes low
        up = np.nextafter(bm, np.float32(np.inf))
        assert O.quant_index(float(up), cb16) == m + 1
    assert O.quant_index(0.0, cb16) == 3
    assert O.quant_index(-1.0, cb16) == 0 and O.quant_index(1.0, cb16) == 7


def test_pack3_bit_definition(oracle_lib):
    rng = np.random.default_rng(4)
    pats = [np.zeros(D, np.uint8), np.full(D, 7, np.uint8), np.arange(D, dtype=np.uint8) % 8,
            (7 - np.arange(D) % 8).astype(np.uint8)] + [rng.integers(0, 8, D).astype(np.uint8)
                                                         for _ in range(20)]
    for idx in pats:
        packed = oracle_lib.pack3(idx)
        stream = 0
        for j, c in enumerate(idx):
            stream |= int(c) << (3 * j)
        assert bytes(packed) == stream.to_bytes(48, "little")
        assert np.array_equal(oracle_lib.unpack3(packed), idx)


def _one_token_page(O, preset, k, v):
    cache = np.zeros((1, 1, O.page_bytes(preset)), np.uint8)
    O.store(preset, cache, k.reshape(1, 1, D), v.reshape(1, 1, D), np.array([0], np.int32))
    return cache[0, 0]


def test_centroid_vectors_round_trip(oracle_lib):
    """A key built as H c (c a vector of centroids) is coded back to c."""
    O = oracle_lib
    rng = np.random.default_rng(5)
    cb16 = O.codebook16()
    cb = cb16.view(np.float16).astype(np.float64)
    bnd = 0.5 * (cb[:-1] + cb[1:])
    for _ in range(30):
        y = rng.standard_normal(D) / np.sqrt(D)
        idx = np.searchsorted(bnd, y, side="left").astype(np.uint8)
        c = cb[idx]
        k = (2.0 * (_H() @ c)).astype(np.float16)
        codes, nc = O.encode_key3(k)
        assert np.array_equal(O.unpack3(codes), idx)


def test_norm_correction_preserves_norm(oracle_lib):
    O = oracle_lib
    rng = np.random.default_rng(6)
    for scale in (0.01, 1.0, 30.0):
        for _ in range(20):
            k = (rng.standard_normal(D) * scale).astype(np.float16)
            page = _one_token_page(O, 1, k, np.zeros(D, np.float16))
            kh = O.decode_key(1, page, 0)
            nk = np.linalg.norm(k.astype(np.float64))
            assert abs(np.linalg.norm(kh) / nk - 1.0) <= 2.0 ** -10


def test_plain_norm_preset_differs_only_in_the_factor(oracle_lib):
    """Preset k3v4 codes keys exactly like k3v4_nc and stores fp16(|k|) as the
    key factor: its pages equal k3v4_nc's except in the factor field, the
    factor is |k| to fp16 rounding, and the decoded key keeps the centroid
    vector's own norm, |k_hat| = factor * |c_hat| (H / sqrt(D) is orthonormal)."""
    O = oracle_lib
    rng = np.random.default_rng(14)
    cb = O.codebook16().view(np.float16).astype(np.float64)
    for scale in (0.01, 1.0, 30.0):
        for _ in range(10):
            k = (rng.standard_normal(D) * scale).astype(np.float16)
            v = rng.standard_normal(D).astype(np.float16)
            pnc = _one_token_page(O, 1, k, v)
            ppl = _one_token_page(O, 2, k, v)
            diff = np.nonzero(pnc != ppl)[0]
            assert set(diff) <= {768, 769}  # the fp16 factor of token 0
            fac = float(ppl[768:770].view(np.float16)[0])
            nk = np.linalg.norm(k.astype(np.float64))
            assert abs(fac / nk - 1.0) <= 2.0 ** -11
            chat = np.linalg.norm(cb[O.unpack3(ppl[0:48])])
            assert abs(np.linalg.norm(O.decode_key(2, ppl, 0)) - fac * chat) <= 1e-12 * fac * chat


def test_splitmix64_published_outputs(oracle_lib):
    """The sign generator is SplitMix64: its first outputs for seed 0 are the
    generator's published reference values."""
    O = oracle_lib
    assert O.splitmix64(0, 0) == 0xE220A8397B1DCDAF
    assert O.splitmix64(0, 1) == 0x6E789E6AA1B965F4
    s = O.rs_signs()
    assert set(np.unique(s)) == {-1, 1} and 40 < (s < 0).sum() < 88  # a Rademacher-like vector
    seed = 0x54515F5349474E53
    assert all((s[j] < 0) == bool(O.splitmix64(seed, j) >> 63) for j in range(128))


def test_signed_rotation_round_trips_centroid_vectors(oracle_lib):
    """Preset k3v4_nc_rs rotates by H diag(s): a key built as s * (H c) from a
    centroid vector c codes back to c exactly, decodes to the key itself, and
    the unsigned preset does not recover c from it."""
    O = oracle_lib
    rng = np.random.default_rng(15)
    cb = O.codebook16().view(np.float16).astype(np.float64)
    bnd = (cb[:-1] + cb[1:]) / 2
    s = O.rs_signs().astype(np.float64)
    for _ in range(10):
        y = rng.standard_normal(D) / np.sqrt(D)
        idx = np.searchsorted(bnd, y, side="left").astype(np.uint8)
        c = cb[idx]
        kk = 2.0 * s * (_H() @ c)
        k = kk.astype(np.float16)
        page = _one_token_page(O, 3, k, np.zeros(D, np.float16))
        assert np.array_equal(O.unpack3(page[0:48]), idx)
        kh = O.decode_key(3, page, 0)  # = nc s (H c) / sqrt(D): the key up to fp16 rounding
        assert np.max(np.abs(kh - kk)) <= 2.0 ** -9 * np.max(np.abs(kk))
        plain = _one_token_page(O, 1, k, np.zeros(D, np.float16))
        assert not np.array_equal(O.unpack3(plain[0:48]), idx)


def test_key3_distortion_matches_lloyd_max(oracle_lib):
    """Mean relative squared error of norm-corrected 3-bit keys: with
    distortion d = 0.03454 of the unit-Gaussian Lloyd-Max quantiser, the
    rescaled reconstruction has cos = sqrt(1 - d), so the relative error is
    2 - 2 sqrt(1 - d) = 0.0348 (high-dimension limit)."""
    O = oracle_lib
    rng = np.random.default_rng(7)
    errs = []
    for _ in range(1500):
        k = rng.standard_normal(D).astype(np.float16)
        page = _one_token_page(O, 1, k, np.zeros(D, np.float16))
        kh = O.decode_key(1, page, 0)
        kk = k.astype(np.float64)
        errs.append(np.sum((kk - kh) ** 2) / np.sum(kk ** 2))
    expect = 2 - 2 * np.sqrt(1 - 0.03454)
    assert abs(np.mean(errs) / expect - 1) < 0.04


def test_zero_key(oracle_lib):
    codes, nc = oracle_lib.encode_key3(np.zeros(D, np.float16))
    assert nc == 0
    assert np.array_equal(oracle_lib.unpack3(codes), np.full(D, 3, np.uint8))


def test_key8_is_per_coordinate_e4m3(oracle_lib):
    O = oracle_lib
    rng = np.random.default_rng(8)
    k = (rng.standard_normal(D) * 20).astype(np.float16)
    out = O.encode_key8(k)
    ref = np.array([O.e4m3_from_half(int(b)) for b in k.view(np.uint16)], np.uint8)
    assert np.array_equal(out, ref)


# ------------------------------------------------------------------ values

def _decode_v(codes, s, z):
    sf = np.float64(np.array([s], np.uint16).view(np.float16)[0])
    zf = np.float64(np.array([z], np.uint16).view(np.float16)[0])
    codes = codes.astype(np.int64)
    return codes, codes * sf + zf, sf, zf


def test_value_error_bound(oracle_lib):
    rng = np.random.default_rng(9)
    for scale in (1e-3, 1.0, 100.0):
        for _ in range(50):
            v = (rng.standard_normal(D) * scale).astype(np.float16)
            packed, s, z = oracle_lib.encode_value4(v)
            codes, vh, sf, zf = _decode_v(packed, s, z)
            vv = v.astype(np.float64)
            assert codes.min() >= 0 and codes.max() <= 15
            assert sf * 15 >= (vv.max() - vv.min()) * (1 - 1e-7)
            assert np.all(np.abs(vv - vh) <= sf / 2 * (1 + 1e-6) + 1e-12)
            assert zf == vv.min()


def test_value_constant_and_signed_zero(oracle_lib):
    for c in (0.0, -0.0, 1.5, -3.25):
        v = np.full(D, c, np.float16)
        packed, s, z = oracle_lib.encode_value4(v)
        codes, vh, sf, zf = _decode_v(packed, s, z)
        assert s == 0 and np.all(codes == 0)
        assert np.array_equal(vh, v.astype(np.float64))
        if c == 0.0:
            assert z == 0  # -0 is stored as +0


def test_value_grid_is_lossless(oracle_lib):
    rng = np.random.default_rng(10)
    for s, z in ((0.125, -1.0), (0.0625, 0.5), (0.25, -2.0)):
        codes = rng.integers(0, 16, D)
        codes[:2] = (0, 15)
        v = (z + codes * s).astype(np.float16)
        packed, sh, zh = oracle_lib.encode_value4(v)
        got, vh, sf, zf = _decode_v(packed, sh, zh)
        assert np.array_equal(got, codes) and sf == s and zf == z


# -------------------------------------------------------------- page layout

@pytest.mark.parametrize("preset,offs", [(0, dict(k=0, v=2048, s=3072, z=3104, page=3136)),
                                          (1, dict(k=0, nc=768, v=800, s=1824, z=1856, page=1920))])
def test_page_layout_and_skips(oracle_lib, preset, offs):
    O = oracle_lib
    rng = np.random.default_rng(11)
    nb, hk = 3, 2
    assert O.page_bytes(preset) == offs["page"]
    cache = np.zeros((nb, hk, offs["page"]), np.uint8)
    T = 7
    k = rng.standard_normal((T, hk, D)).astype(np.float16)
    v = rng.standard_normal((T, hk, D)).astype(np.float16)
    slots = np.array([17, -1, 3, nb * 16, 40, 16, 2], np.int32)  # 16/17 and 2/3 share value bytes
    O.store(preset, cache, k, v, slots)
    expect = np.zeros_like(cache)
    for t, slot in enumerate(slots):
        if slot < 0 or slot >= nb * 16:
            continue
        blk, off = divmod(int(slot), 16)
        for h in range(hk):
            pg = expect[blk, h]
            vp, s, z = O.encode_value4(v[t, h])
            if preset == 0:
                pg[off * 128:(off + 1) * 128] = O.encode_key8(k[t, h])
            else:
                codes, nc = O.encode_key3(k[t, h])
                pg[off * 48:(off + 1) * 48] = codes
                pg[offs["nc"] + 2 * off: offs["nc"] + 2 * off + 2] = np.array([nc], "<u2").view(np.uint8)
            # value codes coordinate-major: byte 8d + off/2, low nibble = even off
            for d in range(D):
                byte = offs["v"] + 8 * d + off // 2
                sh = 4 * (off % 2)
                pg[byte] = (int(pg[byte]) & (0xFF ^ (0xF << sh))) | (int(vp[d]) << sh)
            pg[offs["s"] + 2 * off: offs["s"] + 2 * off + 2] = np.array([s], "<u2").view(np.uint8)
            pg[offs["z"] + 2 * off: offs["z"] + 2 * off + 2] = np.array([z], "<u2").view(np.uint8)
    assert np.array_equal(cache, expect)
