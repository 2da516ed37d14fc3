"""One verify call spread over two ranks (gloo, CPU): the host side of
quantized_kv_cache_store_gb300.shard -- which pages and heads each rank owns,
its local block table and lengths, the causal rule only where the drafts
are, the all-gather of the split partials and the log-sum-exp merge -- with
the oracle as each rank's compute.  The merged result must equal the
single-process oracle over the whole sequences."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = {
    # name: (preset, n_spec, B, Hq, Hk, seq_len or (lo, hi), S per rank, shuffled)
    "poc_like": (0, 8, 2, 8, 2, 1000, 2, False),
    "ragged_k3": (1, 8, 3, 8, 2, (20, 700), 3, True),
    "decode": (1, 1, 3, 8, 4, (1, 300), 2, True),
}


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(case):
    from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs, scaled

    preset, n, B, Hq, Hk, L, S, shuffled = CASES[case]
    names = {v: k for k, v in __import__("quantized_kv_cache_store_gb300.inputs", fromlist=["PRESETS"]).PRESETS.items()}
    kw = dict(len_range=L, seq_len=0) if isinstance(L, tuple) else dict(seq_len=L, len_range=())
    wl = scaled(WORKLOADS["tiny_k8v4"], preset=names[preset], n_spec=n, B=B, Hq=Hq, Hk=Hk, num_kv_splits=S,
                shuffled_blocks=shuffled, **kw)
    return wl, make_inputs(wl, 77)


def _rank(rank: int, world: int, port: int, case: str, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from quantized_kv_cache_store_gb300 import shard
    from tests.helpers import oracle_cache

    class OracleBackend(shard.Backend):
        def __init__(self, preset, cache):
            self.preset, self.cache = preset, cache

        def stage1(self, q, block_table, seq_lens, num_kv_splits, causal):
            po, pl = oracle.partials(self.preset, self.cache, q.numpy(), block_table, np.asarray(seq_lens, np.int32),
                                     num_kv_splits, causal)
            return torch.from_numpy(po), torch.from_numpy(pl)

        def stage2(self, partial_o, partial_lse):
            return torch.from_numpy(oracle.merge(partial_o.numpy(), partial_lse.numpy()))

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        oracle.build()
        wl, inp = _inputs(case)
        cache = oracle_cache(oracle, inp)
        # sequence sharding: every rank ends with the full output
        sh = shard.page_ranges(inp.seq_lens, wl.n_spec, world, rank)
        seq_out = shard.verify_seq_sharded(OracleBackend(wl.preset_id, cache), sh, inp.q, inp.block_table,
                                           wl.num_kv_splits).numpy()
        # kv-head sharding: each rank its heads, gathered for the comparison
        lo, hi = shard.head_range(wl.Hk, world, rank)
        g = wl.Hq // wl.Hk
        q_loc = np.ascontiguousarray(inp.q.numpy()[:, :, lo * g:hi * g])
        c_loc = np.ascontiguousarray(cache[:, lo:hi])
        head_loc = oracle.verify(wl.preset_id, c_loc, q_loc, inp.block_table, inp.seq_lens, True) if hi > lo else \
            np.zeros((wl.n_spec, wl.B, 0, 128))
        head_out = shard.gather_heads(torch.from_numpy(head_loc), wl.Hk, g).numpy()
        out.put((rank, seq_out, head_out, sh.page_lo.tolist(), sh.page_hi.tolist(), bool(sh.causal)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", list(CASES))
def test_two_ranks_equal_one_process(oracle_lib, case):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, case, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((out.get(timeout=300) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    wl, inp = _inputs(case)
    from tests.helpers import oracle_cache

    cache = oracle_cache(oracle_lib, inp)
    ref = oracle_lib.verify(wl.preset_id, cache, inp.q.numpy(), inp.block_table, inp.seq_lens, True)
    for rank, seq_out, head_out, lo, hi, causal in res:
        np.testing.assert_allclose(seq_out, ref, rtol=0, atol=1e-10)
        assert np.array_equal(head_out, ref)
        assert causal == (rank == 1)
    # the two ranges tile every sequence and the drafts sit in the last one
    pages = (inp.seq_lens + 15) // 16
    assert res[0][3] == [0] * wl.B and res[0][4] == res[1][3] and res[1][4] == pages.tolist()
    assert all(16 * lo1 <= L - wl.n_spec for lo1, L in zip(res[1][3], inp.seq_lens))


def test_page_ranges_properties():
    from quantized_kv_cache_store_gb300.shard import head_range, page_ranges

    rng = np.random.default_rng(3)
    for _ in range(200):
        world = int(rng.integers(1, 9))
        n = int(rng.integers(1, 20))
        L = rng.integers(n, 5000, size=int(rng.integers(1, 6)))
        shards = [page_ranges(L, n, world, r) for r in range(world)]
        pages = (L + 15) // 16
        assert np.array_equal(shards[0].page_lo, np.zeros_like(L))
        for a, b in zip(shards, shards[1:]):
            assert np.array_equal(a.page_hi, b.page_lo)
        assert np.array_equal(shards[-1].page_hi, pages)
        assert np.all(16 * shards[-1].page_lo <= L - n)
        assert np.array_equal(sum(s.local_lens.astype(np.int64) for s in shards), L)
        Hk = int(rng.integers(1, 17))
        rs = [head_range(Hk, world, r) for r in range(world)]
        assert rs[0][0] == 0 and rs[-1][1] == Hk and all(a[1] == b[0] for a, b in zip(rs, rs[1:]))
