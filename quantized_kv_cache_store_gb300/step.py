"""Device buffers for one spec-verify workload and the step that runs it.

A step is the whole hot path over one batch: ``tq_store`` of the n_spec draft
tokens of every sequence into the paged cache, then ``tq_verify_stage1`` and
``tq_verify_stage2`` (``step``) or the single ``tq_verify`` call
(``step_fused``).  Everything is allocated once here (PyTorch device
memory); the calls themselves allocate nothing.
"""
from __future__ import annotations

import numpy as np
import torch

from . import tqkv
from .inputs import Inputs


class SpecVerify:
    def __init__(self, inp: Inputs, device="cuda", num_kv_splits: int | None = None,
                 n_caches: int = 1):
        wl = inp.wl
        self.inp = inp
        self.wl = wl
        self.preset = wl.preset_id
        self.S = int(num_kv_splits or wl.num_kv_splits)
        self.device = torch.device(device)
        dev = self.device
        self.caches = [tqkv.alloc_cache(inp.num_blocks, wl.Hk, self.preset, dev) for _ in range(n_caches)]
        self.q = inp.q.to(dev).contiguous()
        self.block_table = torch.from_numpy(inp.block_table).to(dev).contiguous()
        self.seq_lens = torch.from_numpy(inp.seq_lens.astype(np.int32)).to(dev).contiguous()
        drafts = inp.draft_rows()
        self.k_new = inp.k[drafts].to(dev).contiguous()
        self.v_new = inp.v[drafts].to(dev).contiguous()
        self.slots_new = torch.from_numpy(inp.slots[drafts]).to(dev).contiguous()
        n, B, Hq = wl.n_spec, wl.B, wl.Hq
        self.part_o = torch.empty((n, B, Hq, self.S, 128), dtype=torch.float32, device=dev)
        self.part_lse = torch.empty((n, B, Hq, self.S), dtype=torch.float32, device=dev)
        self.out = torch.empty((n, B, Hq, 128), dtype=torch.float32, device=dev)
        self.tickets = torch.zeros((B, wl.Hk, 4), dtype=torch.int32, device=dev)

    def prefill(self, chunk_tokens: int = 1 << 18) -> None:
        """Store the cached prefix of every sequence (untimed set-up)."""
        rows = self.inp.prefix_rows()
        for c in self.caches[:1]:
            for s in range(0, len(rows), chunk_tokens):
                r = rows[s:s + chunk_tokens]
                k = self.inp.k[r].to(self.device)
                v = self.inp.v[r].to(self.device)
                sl = torch.from_numpy(self.inp.slots[r]).to(self.device)
                tqkv.tq_store(c, self.preset, k, v, sl)
        for c in self.caches[1:]:
            c.copy_(self.caches[0])

    def store(self, i: int = 0, stream=None) -> None:
        tqkv.tq_store(self.caches[i], self.preset, self.k_new, self.v_new, self.slots_new, stream)

    def verify(self, i: int = 0, stream=None) -> torch.Tensor:
        tqkv.tq_verify_stage1(self.caches[i], self.preset, self.q, self.block_table, self.seq_lens,
                              self.S, self.wl.causal, self.part_o, self.part_lse, stream)
        tqkv.tq_verify_stage2(self.part_o, self.part_lse, self.out, stream)
        return self.out

    def verify_call(self, i: int = 0, stream=None) -> torch.Tensor:
        """Both stages through tq_verify (one launch when every CTA fits on the device at once)."""
        tqkv.tq_verify(self.caches[i], self.preset, self.q, self.block_table, self.seq_lens, self.S,
                       self.wl.causal, self.part_o, self.part_lse, self.tickets, self.out, stream)
        return self.out

    def step(self, i: int = 0, stream=None) -> torch.Tensor:
        """Store the drafts, then stage 1 and stage 2 as two calls."""
        self.store(i, stream)
        return self.verify(i, stream)

    def step_fused(self, i: int = 0, stream=None) -> torch.Tensor:
        """Store the drafts, then one tq_verify call."""
        self.store(i, stream)
        return self.verify_call(i, stream)

    def step_one(self, i: int = 0, stream=None) -> torch.Tensor:
        """The whole step as one tq_store_verify call (one launch where possible)."""
        tqkv.tq_store_verify(self.caches[i], self.preset, self.k_new, self.v_new, self.q, self.block_table,
                             self.seq_lens, self.S, self.wl.causal, self.part_o, self.part_lse, self.tickets,
                             self.out, stream)
        return self.out
