"""Spec-verify stage 1 + stage 2 on the GPU against the oracle, and the
properties the method fixes (causality, split invariance, paging, fused equals
looped, lossless cache)."""
import dataclasses

import numpy as np
import pytest
import torch

from quantized_kv_cache_store_gb300 import tqkv
from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs, scaled
from tests.helpers import ATOL, RTOL, assert_close, gpu_run, oracle_cache, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _oracle_out(O, inp, causal=None, rows=None):
    causal = inp.wl.causal if causal is None else causal
    cache = oracle_cache(O, inp)
    return O.verify(inp.wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens, causal, rows)


SMALL = [
    # (preset, n_spec, B, Hq, Hk, seq_len / len_range, S, causal)
    ("k8v4", 8, 1, 8, 1, 256, 2, True),     # the tiny workload
    ("k3v4_nc", 8, 1, 8, 1, 256, 2, True),
    ("k8v4", 8, 2, 4, 2, 203, 3, True),     # ragged last page
    ("k3v4_nc", 8, 2, 4, 2, 203, 3, False),
    ("k8v4", 1, 3, 8, 2, (17, 300), 4, True),
    ("k3v4_nc", 1, 5, 32, 8, (1, 90), 2, True),
    ("k8v4", 16, 1, 8, 1, 100, 5, True),    # 128 rows per kv-head
    ("k3v4_nc", 4, 2, 6, 3, 40, 1, True),
    ("k8v4", 3, 2, 2, 2, 3, 4, True),       # cached_len 0, splits mostly empty
    ("k3v4_nc", 8, 1, 32, 4, 555, 7, True),
    ("k8v4", 4, 2, 8, 1, 300, 3, True),     # 32 rows per kv-head
    ("k3v4", 8, 2, 4, 2, 203, 3, True),     # plain-norm preset
    ("k3v4", 1, 3, 8, 2, (17, 300), 4, False),
    ("k3v4_nc_rs", 8, 2, 4, 2, 203, 3, True),  # randomised-sign Hadamard
    ("k3v4_nc_rs", 16, 1, 8, 1, 100, 5, True),  # 128 rows: two row tiles
    ("k3v4_nc", 2, 1, 16, 1, 77, 2, True),
    ("k3v4_nc", 16, 1, 16, 2, 190, 3, True),  # 128 rows per kv-head
    ("k4v4_nc", 8, 1, 8, 1, 256, 2, True),    # the other key widths
    ("k2v4_nc", 8, 1, 8, 1, 256, 2, True),
    ("k4v4_nc", 8, 2, 4, 2, 203, 3, False),
    ("k2v4_nc", 1, 5, 32, 8, (1, 90), 2, True),
    ("k4v4_nc", 1, 3, 8, 2, (17, 300), 4, True),
    ("k2v4_nc", 16, 1, 16, 2, 190, 3, True),
    ("k4v4_nc", 4, 2, 8, 1, 300, 3, True),
]


def _wl(preset, n, B, Hq, Hk, L, S, causal, shuffled=True):
    kw = dict(len_range=L, seq_len=0) if isinstance(L, tuple) else dict(seq_len=L, len_range=())
    return scaled(WORKLOADS["tiny_k8v4"], preset=preset, n_spec=n, B=B, Hq=Hq, Hk=Hk, num_kv_splits=S,
                  causal=causal, shuffled_blocks=shuffled, **kw)


@pytest.mark.parametrize("case", SMALL)
@pytest.mark.parametrize("seed", [42, 101])
def test_small_cases_match_oracle(oracle_lib, case, seed):
    wl = _wl(*case)
    inp = make_inputs(wl, seed)
    cache, po, pl, out = gpu_run(inp)
    assert np.array_equal(cache, oracle_cache(oracle_lib, inp))
    assert_close(out, _oracle_out(oracle_lib, inp))
    # the partials agree too (same split boundaries on both sides)
    rpo, rpl = oracle_lib.partials(wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens,
                                   wl.num_kv_splits, wl.causal)
    assert np.array_equal(np.isinf(pl), np.isinf(rpl))
    fin = np.isfinite(rpl)
    assert_close(pl[fin], rpl[fin], atol=1e-3, rtol=0, what="lse")
    assert_close(po, rpo, what="partial o")


def test_stage2_alone(oracle_lib):
    rng = np.random.default_rng(3)
    n, B, Hq, S = 3, 2, 5, 9
    po = rng.standard_normal((n, B, Hq, S, 128)).astype(np.float32)
    pl = (rng.standard_normal((n, B, Hq, S)) * 5).astype(np.float32)
    pl[0, 0, 0, :4] = -np.inf
    pl[1, 1, 2, :] = -np.inf           # every split empty -> zeros
    po[np.isinf(pl)] = 0
    out = torch.empty((n, B, Hq, 128), dtype=torch.float32, device="cuda")
    tqkv.tq_verify_stage2(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), out)
    ref = oracle_lib.merge(po.astype(np.float64), pl.astype(np.float64))
    got = out.cpu().numpy()
    assert_close(got, ref, atol=1e-5, rtol=1e-5)
    assert np.all(got[1, 1, 2] == 0)


@pytest.mark.parametrize("name", ["tiny_k8v4", "poc_k8v4", "poc_k3v4_nc", "decode_k3v4_nc"])
def test_workload_matches_oracle(oracle_lib, name):
    inp = make_inputs(WORKLOADS[name], 42)
    cache, po, pl, out = gpu_run(inp)
    ref = _oracle_out(oracle_lib, inp)
    err = assert_close(out, ref)
    assert err < ATOL


def test_longctx_sampled_rows(oracle_lib):
    """Full-size long context: sampled rows against the oracle (each row needs
    the whole 262,144-token sequence)."""
    wl = WORKLOADS["longctx_k3v4_nc"]
    inp = make_inputs(wl, 42)
    cache, po, pl, out = gpu_run(inp)
    rows = [(0, 0, 0), (7, 0, 5), (3, 1, 31), (7, 1, 17), (0, 1, 9), (5, 0, 26)]
    ref = oracle_lib.verify(wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens, True, rows)
    got = np.stack([out[n, b, h] for n, b, h in rows])
    assert_close(got, ref)


# Different split counts only change which running maximum each probability is
# rounded to fp16 against (relative rounding <= 2^-11 per weight); a wrong
# split boundary would drop or double tokens and move outputs by ~1e-2.
SPLIT_ATOL = 5e-4


@pytest.mark.parametrize("preset", ["k8v4", "k3v4_nc"])
def test_split_invariance(preset):
    wl = _wl(preset, 8, 2, 16, 2, 1000, 1, True)
    inp = make_inputs(wl, 5)
    outs = [gpu_run(inp, S=S)[3] for S in (1, 2, 8, 32, 80)]
    for o in outs[1:]:
        assert_close(o, outs[0], atol=SPLIT_ATOL, rtol=0, what="split invariance")


@pytest.mark.parametrize("preset", ["k8v4", "k3v4_nc"])
def test_causal_rows_bit_identical(preset):
    """Changing K/V at positions a draft cannot see leaves its output row
    bit-identical."""
    wl = _wl(preset, 8, 1, 8, 1, 180, 3, True, shuffled=False)
    base = make_inputs(wl, 9)
    out0 = gpu_run(base)[3]
    for n in (0, 3, 6):
        inp = make_inputs(wl, 9)
        vis = 180 - 8 + n + 1
        inp.k[vis:180] = -inp.k[vis:180] * 2
        inp.v[vis:180] = inp.v[vis:180] + 3
        out = gpu_run(inp)[3]
        assert np.array_equal(out[: n + 1], out0[: n + 1])
        assert not np.allclose(out[n + 1], out0[n + 1])


@pytest.mark.parametrize("preset", ["k8v4", "k3v4_nc"])
def test_fused_equals_looped(preset):
    """One causal N_spec=8 call equals eight N_spec=1 calls on growing prefixes."""
    wl = _wl(preset, 8, 2, 8, 2, 333, 4, True)
    inp = make_inputs(wl, 10)
    fused = gpu_run(inp)[3]
    from quantized_kv_cache_store_gb300.step import SpecVerify

    sv = SpecVerify(inp)
    sv.prefill()
    sv.store()
    for n in range(8):
        q1 = sv.q[n:n + 1].contiguous()
        sl = (sv.seq_lens - 8 + n + 1).contiguous()
        po = torch.empty((1, wl.B, wl.Hq, 4, 128), dtype=torch.float32, device="cuda")
        pl = torch.empty((1, wl.B, wl.Hq, 4), dtype=torch.float32, device="cuda")
        out = torch.empty((1, wl.B, wl.Hq, 128), dtype=torch.float32, device="cuda")
        tqkv.tq_verify_stage1(sv.caches[0], sv.preset, q1, sv.block_table, sl, 4, True, po, pl)
        tqkv.tq_verify_stage2(po, pl, out)
        assert_close(out.cpu().numpy()[0], fused[n], atol=SPLIT_ATOL, rtol=0, what=f"looped draft {n}")


@pytest.mark.parametrize("preset", ["k8v4", "k3v4_nc"])
def test_paging_bit_identical(preset):
    wl = _wl(preset, 8, 3, 8, 2, 150, 3, True, shuffled=False)
    a = make_inputs(wl, 11)
    b = make_inputs(dataclasses.replace(wl, shuffled_blocks=True), 11)
    assert not np.array_equal(a.block_table, b.block_table)
    assert np.array_equal(gpu_run(a)[3], gpu_run(b)[3])


def test_lossless_k8v4_matches_unquantised_bruteforce(oracle_lib):
    """K on the e4m3 grid and V rows on exact 16-level grids: the k8v4 cache
    is lossless, so the GPU result must match plain softmax(QK^T/sqrt D)V."""
    rng = np.random.default_rng(12)
    wl = _wl("k8v4", 8, 1, 8, 1, 240, 2, True, shuffled=False)
    inp = make_inputs(wl, 13)
    T = inp.k.shape[0]
    e4 = np.array([oracle_lib.e4m3_to_double(c) for c in range(127)])
    e4 = e4[e4 <= 4.0]
    kk = rng.choice(np.concatenate([e4, -e4]), size=(T, 1, 128)).astype(np.float16)
    codes = rng.integers(0, 16, (T, 1, 128))
    codes[..., 0], codes[..., 1] = 0, 15
    s = rng.choice([0.0625, 0.125, 0.25], size=(T, 1, 1))
    z = rng.choice([-1.0, -0.5, -2.0], size=(T, 1, 1))
    vv = (z + codes * s).astype(np.float16)
    inp.k[:] = torch.from_numpy(kk)
    inp.v[:] = torch.from_numpy(vv)
    out = gpu_run(inp)[3]
    q = inp.q.numpy().astype(np.float64)
    for n in range(8):
        vis = 240 - 8 + n + 1
        for h in range(8):
            sc = kk[:vis, 0].astype(np.float64) @ q[n, 0, h] / np.sqrt(128)
            w = np.exp(sc - sc.max())
            ref = w @ vv[:vis, 0].astype(np.float64) / w.sum()
            assert_close(out[n, 0, h], ref)


def test_invalid_block_ids_are_invisible(oracle_lib):
    wl = _wl("k3v4_nc", 8, 2, 8, 2, 200, 3, True)
    inp = make_inputs(wl, 14)
    cache_ref = oracle_cache(oracle_lib, inp)
    bt = inp.block_table.copy()
    bt[0, 3] = -1
    bt[1, 5] = inp.num_blocks + 7
    inp2 = dataclasses.replace(inp, block_table=bt)
    from quantized_kv_cache_store_gb300.step import SpecVerify

    sv = SpecVerify(inp2)
    sv.caches[0].copy_(torch.from_numpy(cache_ref))
    sv.verify()
    torch.cuda.synchronize()
    ref = oracle_lib.verify(1, cache_ref, inp.q.numpy(), bt, inp.seq_lens)
    assert_close(sv.out.cpu().numpy(), ref)


def test_device_status_clean():
    """No bounded device-side wait expired in any of the runs above."""
    torch.cuda.synchronize()
    assert tqkv.tq_device_status() == tqkv.TQ_OK


def test_unused_slots_with_garbage_do_not_leak():
    """Slots past seq_len in the last page hold arbitrary bytes (here 0xFF:
    NaN scales); the output must not change."""
    wl = _wl("k8v4", 8, 1, 8, 1, 200, 2, True, shuffled=False)
    inp = make_inputs(wl, 15)
    from quantized_kv_cache_store_gb300.step import SpecVerify

    sv = SpecVerify(inp)
    sv.prefill()
    sv.store()
    ref = sv.verify().clone()
    last = int(inp.block_table[0, (200 - 1) // 16])
    page = sv.caches[0][last, 0]
    assert 200 % 16 == 8  # tokens 8..15 of the last page are unused
    for off in range(8, 16):
        page[off * 128:(off + 1) * 128] = 0xFF            # NaN e4m3 keys
        page[3072 + 2 * off: 3072 + 2 * off + 2] = 0xFF   # NaN scale
        page[3104 + 2 * off: 3104 + 2 * off + 2] = 0xFF   # NaN zero
    for d in range(128):                                   # value codes of tokens 8..15:
        page[2048 + 8 * d + 4: 2048 + 8 * d + 8] = 0xFF    # bytes 4..7 of each coordinate row
    out = sv.verify()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)


# ---- tq_verify: both stages in one call (one launch whose splits merge through
# per-pair counters when every CTA is resident and S <= 32; else stage 1 + stage 2)

FUSED = [
    # (preset, n_spec, B, Hq, Hk, seq_len / len_range, S, causal)
    ("k8v4", 8, 1, 8, 1, 256, 2, True),
    ("k3v4_nc", 8, 2, 4, 2, 203, 3, False),
    ("k8v4", 1, 3, 8, 2, (17, 300), 4, True),
    ("k3v4_nc", 8, 1, 32, 4, 555, 7, True),
    ("k8v4", 4, 2, 8, 1, 300, 8, True),     # eight splits: one row per split to merge
    ("k3v4_nc", 4, 2, 6, 3, 40, 1, True),
    ("k3v4_nc", 8, 2, 16, 2, 900, 6, True),  # rows not a multiple of the splits
    ("k8v4", 8, 1, 8, 1, 64, 8, True),      # most splits empty
    ("k8v4", 3, 2, 2, 2, 3, 5, True),       # splits mostly empty
    ("k3v4_nc", 2, 1, 16, 1, 77, 16, True),
    ("k3v4", 8, 1, 8, 1, 256, 4, True),
    ("k3v4_nc_rs", 8, 1, 32, 4, 555, 7, True),
    ("k8v4", 1, 2, 8, 1, 2000, 32, True),   # the most splits one launch merges
    ("k8v4", 2, 3, 8, 4, 700, 40, False),   # more splits than one launch merges: two launches
    ("k8v4", 16, 1, 8, 1, 100, 3, True),    # 128 rows: two row tiles in one launch
    ("k4v4_nc", 8, 1, 32, 4, 555, 7, True),
    ("k2v4_nc", 8, 2, 16, 2, 900, 6, True),
    ("k4v4_nc", 16, 1, 16, 2, 190, 3, True),
]


def _fused_run(inp):
    from quantized_kv_cache_store_gb300.step import SpecVerify

    sv = SpecVerify(inp)
    sv.prefill()
    sv.step_fused()
    torch.cuda.synchronize()
    fused = sv.out.cpu().numpy()
    assert not sv.tickets.any()  # left zeroed for the next call
    sv.verify_call()             # and a second call gives the same result
    torch.cuda.synchronize()
    assert np.array_equal(sv.out.cpu().numpy(), fused)
    sv.verify()
    torch.cuda.synchronize()
    return sv.caches[0].cpu().numpy(), fused, sv.out.cpu().numpy()


@pytest.mark.parametrize("case", FUSED)
def test_single_call_verify_matches_oracle(oracle_lib, case):
    inp = make_inputs(_wl(*case), 77)
    cache, fused, staged = _fused_run(inp)
    assert np.array_equal(cache, oracle_cache(oracle_lib, inp))
    assert_close(fused, _oracle_out(oracle_lib, inp))
    # same arithmetic as stage 1 + stage 2 up to the order of the merge sums
    assert_close(fused, staged, atol=1e-5, rtol=1e-5, what="single call vs two calls")


@pytest.mark.parametrize("name", ["poc_k8v4", "poc_k3v4_nc"])
def test_single_call_verify_poc(oracle_lib, name):
    inp = make_inputs(WORKLOADS[name], 1001)
    cache, fused, staged = _fused_run(inp)
    assert_close(fused, _oracle_out(oracle_lib, inp))
    assert_close(fused, staged, atol=1e-5, rtol=1e-5, what="single call vs two calls")
    assert tqkv.tq_device_status() == tqkv.TQ_OK


# ---- continuation chunks ("spec-decode-intel-arc", backend-integration
# section: chunks of up to 128 query tokens take the spec-verify path): up to
# 1024 query rows per kv-head, tiled 64 rows per CTA on the tensor cores.

@pytest.mark.parametrize("preset", ["k8v4", "k3v4_nc", "k4v4_nc", "k2v4_nc"])
@pytest.mark.parametrize("q_len,group,L,S", [(16, 8, 300, 3), (64, 4, 700, 2), (128, 8, 600, 2), (128, 2, 1500, 5)])
def test_continuation_chunks_match_oracle(oracle_lib, preset, q_len, group, L, S):
    from quantized_kv_cache_store_gb300.step import SpecVerify

    wl = _wl(preset, q_len, 2, 2 * group, 2, L, S, True)
    inp = make_inputs(wl, 31)
    ref = _oracle_out(oracle_lib, inp)
    # stage 1 + stage 2
    cache, po, pl, out = gpu_run(inp)
    assert np.array_equal(cache, oracle_cache(oracle_lib, inp))
    assert_close(out, ref)
    # one tq_verify call and one tq_store_verify call
    sv = SpecVerify(inp, n_caches=2)
    sv.prefill()
    sv.store(0)
    fused = sv.verify_call(0).cpu().numpy()
    assert_close(fused, ref)
    sv.step_one(1)
    torch.cuda.synchronize()
    assert torch.equal(sv.caches[1], sv.caches[0])
    assert_close(sv.out.cpu().numpy(), ref)
    assert not sv.tickets.any()
