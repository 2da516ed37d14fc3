"""Pins for the oracle's attention: brute force in the quantisation-bypass
mode, softmax normalisation, causal visibility, split invariance, paging,
fused-equals-looped and lossless-cache cases."""
import numpy as np
import pytest

from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs, scaled
from tests.helpers import oracle_cache

D = 128


def _bruteforce(q, k, v, lo, hi):
    """softmax(q k^T / sqrt(D)) v per row over [lo, hi), numpy fp64."""
    q = q.astype(np.float64)
    k = k.astype(np.float64)
    v = v.astype(np.float64)
    out = np.zeros((q.shape[0], D))
    lse = np.full(q.shape[0], -np.inf)
    for r in range(q.shape[0]):
        if hi[r] <= lo[r]:
            continue
        s = k[lo[r]:hi[r]] @ q[r] / np.sqrt(D)
        m = s.max()
        w = np.exp(s - m)
        out[r] = w @ v[lo[r]:hi[r]] / w.sum()
        lse[r] = m + np.log(w.sum())
    return out, lse


def test_bypass_matches_bruteforce(oracle_lib):
    rng = np.random.default_rng(20)
    L, nr = 300, 12
    q = rng.standard_normal((nr, D)).astype(np.float16)
    k = (rng.standard_normal((L, D)) * 2).astype(np.float16)
    v = rng.standard_normal((L, D)).astype(np.float16)
    lo = rng.integers(0, 50, nr).astype(np.int32)
    hi = (lo + rng.integers(0, 250, nr)).astype(np.int32)
    hi[0] = lo[0]  # one empty row
    o, l = oracle_lib.attend_raw(q, k, v, lo, hi)
    ro, rl = _bruteforce(q, k, v, lo, hi)
    assert np.allclose(o, ro, atol=1e-12, rtol=0)
    assert np.array_equal(np.isinf(l), np.isinf(rl))
    fin = np.isfinite(rl)
    assert np.allclose(l[fin], rl[fin], atol=1e-12, rtol=0)


def _small(preset="k8v4", **kw):
    base = WORKLOADS["tiny_k8v4"] if preset == "k8v4" else scaled(WORKLOADS["tiny_k8v4"], preset="k3v4_nc")
    return scaled(base, **kw)


@pytest.mark.parametrize("preset", ["k8v4", "k3v4_nc"])
def test_weights_sum_to_one(oracle_lib, preset):
    """With every value row constant 1 the output is exactly the sum of the
    softmax weights."""
    O = oracle_lib
    inp = make_inputs(_small(preset, seq_len=100), 1)
    inp.v[:] = 1.0
    cache = oracle_cache(O, inp)
    out = O.verify(inp.wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens)
    assert np.allclose(out, 1.0, atol=1e-12, rtol=0)


@pytest.mark.parametrize("preset", ["k8v4", "k3v4_nc"])
def test_causal_visibility(oracle_lib, preset):
    """Draft n sees exactly L - n_spec + n + 1 positions: changing K/V at any
    later position leaves its row bit-identical and changes the next row."""
    O = oracle_lib
    wl = _small(preset, seq_len=77, B=2, Hq=4, Hk=2)
    inp = make_inputs(wl, 2)
    cache = oracle_cache(O, inp)
    ref = O.verify(wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens)
    for n in range(wl.n_spec - 1):
        vis = O.visible(int(inp.seq_lens[0]), wl.n_spec, n, True)
        assert vis == 77 - wl.n_spec + n + 1
        inp2 = make_inputs(wl, 2)
        row = inp2.tok_off[0] + vis  # first invisible position of draft n, sequence 0
        inp2.k[row:inp2.tok_off[0] + 77] *= -3
        inp2.v[row:inp2.tok_off[0] + 77] += 5
        c2 = oracle_cache(O, inp2)
        out = O.verify(wl.preset_id, c2, inp2.q.numpy(), inp2.block_table, inp2.seq_lens)
        assert np.array_equal(out[: n + 1, 0], ref[: n + 1, 0])
        assert not np.allclose(out[n + 1, 0], ref[n + 1, 0])
        assert np.array_equal(out[:, 1], ref[:, 1])


def test_noncausal_sees_everything(oracle_lib):
    O = oracle_lib
    wl = _small("k8v4", seq_len=50, causal=False)
    inp = make_inputs(wl, 3)
    cache = oracle_cache(O, inp)
    out = O.verify(0, cache, inp.q.numpy(), inp.block_table, inp.seq_lens, causal=False)
    for n in range(wl.n_spec):
        assert O.visible(50, wl.n_spec, n, False) == 50
    # every draft row of the same head equals attention over all 50 positions
    one = O.verify(0, cache, inp.q.numpy()[:1], inp.block_table, inp.seq_lens, causal=False)
    assert np.array_equal(out[0], one[0])


@pytest.mark.parametrize("preset", ["k8v4", "k3v4_nc"])
@pytest.mark.parametrize("S", [1, 2, 3, 8, 32])
def test_split_merge_equals_direct(oracle_lib, preset, S):
    O = oracle_lib
    wl = _small(preset, seq_len=200)
    inp = make_inputs(wl, 4)
    cache = oracle_cache(O, inp)
    direct = O.verify(wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens)
    po, pl = O.partials(wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens, S)
    merged = O.merge(po, pl)
    assert np.allclose(merged, direct, atol=1e-12, rtol=0)
    if S == 32:  # 200 tokens in 13 pages: most of 32 splits are empty
        assert np.isinf(pl).any()
        assert np.all(po[np.isinf(pl)] == 0)


def test_paging_is_transparent(oracle_lib):
    """A shuffled block table over permuted pages gives the same result as a
    contiguous one."""
    O = oracle_lib
    wl = _small("k3v4_nc", seq_len=150, B=3, Hq=4, Hk=2)
    a = make_inputs(wl, 5)
    b = make_inputs(scaled(wl, shuffled_blocks=True), 5)
    assert not np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(a.k.numpy(), b.k.numpy())
    oa = O.verify(1, oracle_cache(O, a), a.q.numpy(), a.block_table, a.seq_lens)
    ob = O.verify(1, oracle_cache(O, b), b.q.numpy(), b.block_table, b.seq_lens)
    assert np.array_equal(oa, ob)


def test_fused_equals_looped(oracle_lib):
    """A causal N_spec=8 verify equals 8 single-query calls on growing prefixes
    (the fused-versus-looped check of the fused kernel's test)."""
    O = oracle_lib
    wl = _small("k8v4", seq_len=120)
    inp = make_inputs(wl, 6)
    cache = oracle_cache(O, inp)
    fused = O.verify(0, cache, inp.q.numpy(), inp.block_table, inp.seq_lens)
    for n in range(8):
        sl = inp.seq_lens - 8 + n + 1
        one = O.verify(0, cache, inp.q.numpy()[n:n + 1], inp.block_table, sl, causal=True)
        assert np.array_equal(one[0], fused[n])


def test_lossless_k8v4_cache_equals_bruteforce(oracle_lib):
    """K on the e4m3 grid and V rows on exact 16-level grids make the k8v4
    cache lossless, so quantised attention equals unquantised brute force."""
    O = oracle_lib
    rng = np.random.default_rng(12)
    wl = _small("k8v4", seq_len=90)
    inp = make_inputs(wl, 7)
    T = inp.k.shape[0]
    e4 = np.array([O.e4m3_to_double(c) for c in range(127)])
    kk = rng.choice(np.concatenate([e4, -e4]), size=(T, 1, D)) / 64
    kk = (kk * 64).astype(np.float16)
    codes = rng.integers(0, 16, (T, 1, D))
    codes[..., 0], codes[..., 1] = 0, 15
    s = rng.choice([0.0625, 0.125, 0.25], size=(T, 1, 1))
    z = rng.choice([-1.0, -0.5, -2.0], size=(T, 1, 1))
    vv = (z + codes * s).astype(np.float16)
    inp.k[:] = __import__("torch").from_numpy(kk)
    inp.v[:] = __import__("torch").from_numpy(vv)
    cache = oracle_cache(O, inp)
    out = O.verify(0, cache, inp.q.numpy(), inp.block_table, inp.seq_lens)
    L = int(inp.seq_lens[0])
    for n in range(8):
        vis = L - 8 + n + 1
        qr = inp.q.numpy()[n, 0]
        ref, _ = _bruteforce(qr, kk[:L, 0], vv[:L, 0], np.zeros(8, int), np.full(8, vis))
        assert np.allclose(out[n, 0], ref, atol=1e-12, rtol=0)


@pytest.mark.parametrize("preset,max_rel", [("k8v4", 0.15), ("k3v4_nc", 0.3)])
def test_quantised_attention_tracks_unquantised(oracle_lib, preset, max_rel):
    """Coarse sanity of the decode: quantised attention stays close to
    unquantised attention (relative error of 4-bit values ~0.1, plus ~0.1 from
    3-bit keys); a broken rotation inverse or code gather decorrelates it."""
    O = oracle_lib
    wl = _small(preset, seq_len=256)
    inp = make_inputs(wl, 8)
    cache = oracle_cache(O, inp)
    out = O.verify(wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens)
    for h in range(wl.Hq):
        ref, _ = _bruteforce(inp.q.numpy()[7, 0, h:h + 1], inp.k.numpy()[:, 0], inp.v.numpy()[:, 0],
                             np.zeros(1, int), np.full(1, 256))
        o, r = out[7, 0, h], ref[0]
        assert np.linalg.norm(o - r) / np.linalg.norm(r) < max_rel
        assert np.corrcoef(o, r)[0, 1] > 0.95
