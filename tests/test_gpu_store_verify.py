"""tq_store_verify (drafts stored inside the verify launch) against tq_store
followed by tq_verify: the same cache bytes and the same outputs, bit for
bit, whether the drafts land in the first chunk of their split, in its last
chunk, across two splits, or the call falls back to two launches."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs, scaled
from tests.helpers import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


CASES = [
    # (workload, overrides)
    ("tiny_k8v4", {}),                                                   # drafts in chunk 0 of split 1
    ("tiny_k8v4", dict(preset="k3v4_nc")),
    ("tiny_k8v4", dict(preset="k3v4", n_spec=8, B=2, Hq=16, Hk=2, seq_len=500, num_kv_splits=3)),
    ("tiny_k8v4", dict(preset="k3v4_nc_rs", n_spec=8, B=2, Hq=16, Hk=2, seq_len=333, num_kv_splits=2)),
    ("tiny_k8v4", dict(n_spec=16, B=1, Hq=4, Hk=1, seq_len=200, num_kv_splits=4)),  # drafts across two splits
    ("tiny_k8v4", dict(preset="k3v4_nc", n_spec=8, B=2, Hq=4, Hk=2, seq_len=203, num_kv_splits=3, causal=False)),
    ("tiny_k8v4", dict(preset="k3v4_nc", n_spec=1, B=5, Hq=32, Hk=8, seq_len=0, len_range=(1, 900),
                       num_kv_splits=2)),                                # ragged, shuffled pages
    ("tiny_k8v4", dict(n_spec=3, B=2, Hq=2, Hk=2, seq_len=3, num_kv_splits=4)),  # no cached prefix
    ("tiny_k8v4", dict(n_spec=2, B=3, Hq=8, Hk=4, seq_len=700, num_kv_splits=40)),  # two launches
    ("tiny_k8v4", dict(preset="k4v4_nc", n_spec=8, B=2, Hq=16, Hk=2, seq_len=500, num_kv_splits=3)),
    ("tiny_k8v4", dict(preset="k2v4_nc", n_spec=16, B=1, Hq=4, Hk=1, seq_len=200, num_kv_splits=4)),
    ("poc_k8v4", {}),
    ("poc_k3v4_nc", {}),
    ("poc_k3v4_nc", dict(preset="k4v4_nc")),
]


@pytest.mark.parametrize("name,kw", CASES)
def test_store_verify_equals_store_then_verify(name, kw):
    from quantized_kv_cache_store_gb300.step import SpecVerify

    wl = scaled(WORKLOADS[name], **kw) if kw else WORKLOADS[name]
    sv = SpecVerify(make_inputs(wl, 9), n_caches=2)
    sv.prefill()
    sv.store(0)
    ref = sv.verify_call(0).clone()
    sv.step_one(1)
    torch.cuda.synchronize()
    assert torch.equal(sv.caches[1], sv.caches[0])
    assert torch.equal(sv.out, ref)
    assert not sv.tickets.any()
    # a second call on the same cache rewrites the same bytes and gives the same result
    sv.step_one(1)
    torch.cuda.synchronize()
    assert torch.equal(sv.caches[1], sv.caches[0])
    assert torch.equal(sv.out, ref)


# ---- tq_store_verify (the bench step) against the oracle itself: the cache
# bytes after the call (prefix stored by tq_store, drafts by the call) and the
# attention outputs, at the full workload sizes.

@pytest.mark.parametrize("name", ["poc_k8v4", "poc_k3v4_nc", "decode_k3v4_nc"])
def test_store_verify_matches_oracle(oracle_lib, name):
    from quantized_kv_cache_store_gb300.step import SpecVerify
    from tests.helpers import ATOL, assert_close, oracle_cache

    inp = make_inputs(WORKLOADS[name], 1001)
    sv = SpecVerify(inp)
    sv.prefill()
    sv.step_one(0)
    torch.cuda.synchronize()
    cache = oracle_cache(oracle_lib, inp)
    assert np.array_equal(sv.caches[0].cpu().numpy(), cache)
    wl = inp.wl
    ref = oracle_lib.verify(wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens, wl.causal)
    assert assert_close(sv.out.cpu().numpy(), ref) < ATOL
    assert not sv.tickets.any()


def test_store_verify_longctx_sampled_rows(oracle_lib):
    """Full-size long context through tq_store_verify: every page the drafts
    touch is bit-exact against the oracle's encoding, and sampled output rows
    match the oracle (each row needs the whole 262,144-token sequence)."""
    from quantized_kv_cache_store_gb300.step import SpecVerify
    from tests.helpers import assert_close

    wl = WORKLOADS["longctx_k3v4_nc"]
    inp = make_inputs(wl, 1001)
    sv = SpecVerify(inp)
    sv.prefill()
    before = sv.caches[0].cpu().numpy()
    sv.step_one(0)
    torch.cuda.synchronize()
    got = sv.caches[0].cpu().numpy()
    # the oracle stores the drafts into the prefix-only cache the GPU started from
    want = before.copy()
    d = inp.draft_rows()
    oracle_lib.store(wl.preset_id, want, inp.k.numpy()[d], inp.v.numpy()[d], inp.slots[d])
    assert np.array_equal(got, want)
    rows = [(0, 0, 0), (7, 0, 5), (3, 1, 31), (7, 1, 17), (1, 1, 8)]
    ref = oracle_lib.verify(wl.preset_id, want, inp.q.numpy(), inp.block_table, inp.seq_lens, True, rows)
    out = sv.out.cpu().numpy()
    assert_close(np.stack([out[n, b, h] for n, b, h in rows]), ref)
