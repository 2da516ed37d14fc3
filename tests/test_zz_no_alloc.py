"""tq_verify_noalloc (the allocation-free entry point) against tq_verify on
the same inputs: two calls in a row each, identical outputs.  Collected last
and independent of earlier tests: the library's scratch is set up by the
first call, whichever test makes it, and left ready for the next."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_store_gb300 import tqkv
from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs, scaled
from tests.helpers import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


CASES = [
    ("tiny_k8v4", {}),
    ("tiny_k8v4", dict(preset="k3v4_nc", n_spec=8, B=2, Hq=4, Hk=2, seq_len=203, num_kv_splits=3)),
    ("tiny_k8v4", dict(n_spec=2, B=3, Hq=8, Hk=4, seq_len=700, num_kv_splits=40, causal=False)),  # two launches
    ("poc_k8v4", {}),
    ("poc_k3v4_nc", {}),
]


@pytest.mark.parametrize("name,kw", CASES)
def test_noalloc_matches_tq_verify(name, kw):
    from quantized_kv_cache_store_gb300.step import SpecVerify

    wl = scaled(WORKLOADS[name], **kw) if kw else WORKLOADS[name]
    sv = SpecVerify(make_inputs(wl, 5))
    sv.prefill()
    ref = sv.verify_call().clone()
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row: the counters are left zero for the next
        out = torch.full_like(ref, float("nan"))
        tqkv.tq_verify_noalloc(sv.caches[0], sv.preset, sv.q, sv.block_table, sv.seq_lens, sv.S,
                               wl.causal, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    assert tqkv.tq_device_status() == tqkv.TQ_OK


def test_noalloc_rejects_oversized():
    from quantized_kv_cache_store_gb300.step import SpecVerify

    wl = WORKLOADS["tiny_k8v4"]
    sv = SpecVerify(make_inputs(wl, 5))
    out = torch.empty((wl.n_spec, wl.B, wl.Hq, 128), dtype=torch.float32, device="cuda")
    # 8 x 1 x 8 x 9000 split rows of 129 floats exceed the 16 MiB scratch
    with pytest.raises(tqkv.TqError) as e:
        tqkv.tq_verify_noalloc(sv.caches[0], sv.preset, sv.q, sv.block_table, sv.seq_lens, 9000, True, out)
    assert e.value.status == tqkv.TQ_ERR_UNSUPPORTED
