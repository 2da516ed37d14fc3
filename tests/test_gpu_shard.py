"""The sequence-sharded verify of quantized_kv_cache_store_gb300.shard on one
GPU: each rank's stage 1 (its page range, local block table and lengths, the
causal rule on the last rank only) run one after another through the C ABI,
the partials concatenated along the split axis as the all-gather would, and
merged by stage 2 -- against the oracle over the whole sequences."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_store_gb300 import shard
from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs, scaled
from tests.helpers import assert_close, oracle_cache, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("preset,world,n,L,S", [("k8v4", 2, 8, 2000, 2), ("k3v4_nc", 3, 8, (40, 900), 3),
                                                ("k3v4_nc", 4, 1, (1, 600), 2), ("k8v4", 2, 64, 1200, 2)])
def test_seq_sharded_matches_oracle(oracle_lib, preset, world, n, L, S):
    from quantized_kv_cache_store_gb300.step import SpecVerify

    kw = dict(len_range=L, seq_len=0) if isinstance(L, tuple) else dict(seq_len=L, len_range=())
    wl = scaled(WORKLOADS["tiny_k8v4"], preset=preset, n_spec=n, B=3, Hq=8, Hk=2, num_kv_splits=S,
                shuffled_blocks=True, **kw)
    inp = make_inputs(wl, 5)
    sv = SpecVerify(inp)
    sv.prefill()
    sv.store()
    backend = shard.GpuBackend(sv.caches[0], sv.preset)
    pos, pls = [], []
    for r in range(world):
        sh = shard.page_ranges(inp.seq_lens, n, world, r)
        po, pl = backend.stage1(sv.q, sh.block_table(inp.block_table), sh.local_lens, S, sh.causal)
        pos.append(po)
        pls.append(pl)
    out = backend.stage2(torch.cat(pos, dim=3), torch.cat(pls, dim=3))
    torch.cuda.synchronize()
    ref = oracle_lib.verify(wl.preset_id, oracle_cache(oracle_lib, inp), inp.q.numpy(), inp.block_table,
                            inp.seq_lens, True)
    assert_close(out.cpu().numpy(), ref)
