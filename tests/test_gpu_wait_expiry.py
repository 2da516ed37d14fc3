"""Failure detection of the single-launch verify without a GPU fault: a
cross-split wait that runs out.

The splits of each (sequence, kv-head) count themselves in on the arrival
counter in `tickets` and wait, for a bounded time, until it reaches the split
count.  Here the counter of one pair starts at 0xFFFFFFFF, so the S
arrivals leave it at 0 .. S-1 and it never reaches S: every split of that
pair waits out its limit (well under a second of polling), then writes NaN
for the pair's rows and sets the device error word.  The test checks the
status, the NaN rows, that every other row is untouched by the failure, and
that the next calls (with the caller's counters zeroed, and through
tq_verify_noalloc, whose own scratch is set up again after the reported
expiry) give the normal result bit for bit."""
import time

import pytest
import torch

from quantized_kv_cache_store_gb300 import tqkv
from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs, scaled
from tests.helpers import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_expired_merge_wait_reports_timeout_and_recovers():
    from quantized_kv_cache_store_gb300.step import SpecVerify

    wl = scaled(WORKLOADS["tiny_k8v4"], n_spec=8, B=2, Hq=8, Hk=2, seq_len=300, num_kv_splits=3)
    sv = SpecVerify(make_inputs(wl, 21))
    sv.prefill()
    sv.store()
    torch.cuda.synchronize()
    assert tqkv.tq_device_status() == tqkv.TQ_OK
    ref = sv.verify_call().clone()
    torch.cuda.synchronize()
    assert not torch.isnan(ref).any()

    b_bad, kvh_bad, group = 1, 0, wl.Hq // wl.Hk
    sv.tickets[b_bad, kvh_bad, 0] = -1  # 0xFFFFFFFF: the arrivals wrap to 0 .. S-1
    sv.out.zero_()
    t0 = time.time()
    out = sv.verify_call()
    torch.cuda.synchronize()
    waited = time.time() - t0
    assert tqkv.tq_device_status() == tqkv.TQ_ERR_TIMEOUT
    assert tqkv.tq_device_status() == tqkv.TQ_OK  # reading cleared the word
    heads = slice(kvh_bad * group, (kvh_bad + 1) * group)
    assert torch.isnan(out[:, b_bad, heads]).all()
    keep = torch.ones_like(out, dtype=torch.bool)
    keep[:, b_bad, heads] = False
    assert torch.equal(out[keep], ref[keep])
    assert waited < 30.0

    # recovery: the caller zeroes its counters, the next call is the normal one
    sv.tickets.zero_()
    again = sv.verify_call().clone()
    torch.cuda.synchronize()
    assert torch.equal(again, ref)
    assert not sv.tickets.any()
    assert tqkv.tq_device_status() == tqkv.TQ_OK

    # tq_verify_noalloc sets its own scratch up again after the reported expiry
    na = torch.full_like(ref, float("nan"))
    tqkv.tq_verify_noalloc(sv.caches[0], sv.preset, sv.q, sv.block_table, sv.seq_lens, sv.S, wl.causal, na)
    torch.cuda.synchronize()
    assert torch.equal(na, ref)
    assert tqkv.tq_device_status() == tqkv.TQ_OK
