"""The seeded input recipe: deterministic per seed, and the drafts' cache
slots follow the rule tq_store_verify applies (draft n of sequence b at
position min(L_b, 16 max_blocks) - n_spec + n through the block table)."""
import numpy as np
import pytest

from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs, scaled

CASES = {
    "tiny": WORKLOADS["tiny_k8v4"],
    "poc": WORKLOADS["poc_k3v4_nc"],
    # the decode recipe (ragged lengths, shuffled pages) at a smaller size
    "decode_small": scaled(WORKLOADS["decode_k3v4_nc"], B=6, len_range=(1, 700)),
}


@pytest.mark.parametrize("name", list(CASES))
def test_draft_slots_follow_the_block_table(name):
    inp = make_inputs(CASES[name], 7)
    n = inp.wl.n_spec
    bt = inp.block_table
    slots = inp.slots[inp.draft_rows()]
    want = []
    for b, L in enumerate(inp.seq_lens):
        Lc = min(int(L), 16 * bt.shape[1])
        for j in range(n):
            pos = Lc - n + j
            want.append(int(bt[b, pos // 16]) * 16 + pos % 16)
    assert np.array_equal(slots, np.array(want, np.int32))


def test_seeded_inputs_are_deterministic():
    a = make_inputs(WORKLOADS["tiny_k8v4"], 11)
    b = make_inputs(WORKLOADS["tiny_k8v4"], 11)
    c = make_inputs(WORKLOADS["tiny_k8v4"], 12)
    assert np.array_equal(a.q.numpy(), b.q.numpy()) and np.array_equal(a.k.numpy(), b.k.numpy())
    assert np.array_equal(a.block_table, b.block_table) and np.array_equal(a.slots, b.slots)
    assert not np.array_equal(a.q.numpy(), c.q.numpy())
