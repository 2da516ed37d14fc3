"""Seeded synthetic workloads for spec-verify attention.

This module draws random numbers and lays out indices only; it holds none of
the method's arithmetic (no rotation, quantisation or attention).  The tests,
the benchmark and the smoke check all draw their inputs from here, so the CUDA
path and the CPU oracle see the same bytes.

Recipe (one ``torch.Generator('cpu')`` seeded per call, drawn in this order):
  1. ragged sequence lengths (only for workloads with a length range),
  2. Q  ~ N(0, 1) float32 -> fp16, shape [n_spec, B, Hq, D],
  3. K  ~ N(0, 1) float32, shape [tokens, Hk, D],
  4. V  ~ N(0, 1) float32 -> fp16, same shape,
  5. per-kv-head key scale ~ U(k_scale_lo, k_scale_hi) (1.0 when both are 1),
     applied to K before the fp16 cast,
  6. block permutation (only for workloads with shuffled blocks).
Tokens are laid out sequence-major: sequence b owns rows
[tok_off[b], tok_off[b] + L_b) of K and V, position p at row tok_off[b] + p.
The last n_spec positions of each sequence are the draft tokens that a verify
step stores; the earlier ones are the cached prefix.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch

HEAD_DIM = 128
BLOCK = 16
PRESETS = {"k8v4": 0, "k3v4_nc": 1, "k3v4": 2, "k3v4_nc_rs": 3, "k4v4_nc": 4, "k2v4_nc": 5}


@dataclass(frozen=True)
class Workload:
    name: str
    preset: str            # "k8v4" | "k3v4_nc" | "k3v4" | "k3v4_nc_rs" | "k4v4_nc" | "k2v4_nc"
    n_spec: int
    B: int
    Hq: int
    Hk: int
    seq_len: int = 0       # fixed total length per sequence (includes the drafts)
    len_range: tuple = ()  # (lo, hi) inclusive: ragged lengths drawn per sequence
    num_kv_splits: int = 8
    causal: bool = True
    shuffled_blocks: bool = False
    k_scale: tuple = (1.0, 1.0)
    store_in_step: bool = True   # a step stores the drafts, then verifies

    @property
    def preset_id(self) -> int:
        return PRESETS[self.preset]

    @property
    def group(self) -> int:
        return self.Hq // self.Hk


# The five workloads, named by what they are.  The split counts are the
# implementation's choice (results do not depend on them beyond rounding):
# PoC 8 (the pages' value; 128 CTAs of 8 chunks), decode 4 (1024 CTAs: the
# ragged lengths balance over the 152 SMs of a GB300 while each CTA's fixed
# cost stays small), long context 19 (8 (sequence, kv-head) pairs x 19 = 152
# CTAs: one wave, one launch).
WORKLOADS = {
    "tiny_k8v4": Workload("tiny_k8v4", "k8v4", n_spec=8, B=1, Hq=8, Hk=1, seq_len=256,
                          num_kv_splits=2),
    "poc_k8v4": Workload("poc_k8v4", "k8v4", n_spec=8, B=4, Hq=32, Hk=4, seq_len=8192,
                         num_kv_splits=8),
    "poc_k3v4_nc": Workload("poc_k3v4_nc", "k3v4_nc", n_spec=8, B=4, Hq=32, Hk=4, seq_len=8192,
                            num_kv_splits=8),
    "decode_k3v4_nc": Workload("decode_k3v4_nc", "k3v4_nc", n_spec=1, B=32, Hq=32, Hk=8,
                               len_range=(1024, 32768), num_kv_splits=4, shuffled_blocks=True),
    "longctx_k3v4_nc": Workload("longctx_k3v4_nc", "k3v4_nc", n_spec=8, B=2, Hq=32, Hk=4,
                                seq_len=262144, num_kv_splits=19, k_scale=(0.5, 2.0)),
    # the PoC shape with the other key widths (4-bit and 2-bit codes)
    "poc_k4v4_nc": Workload("poc_k4v4_nc", "k4v4_nc", n_spec=8, B=4, Hq=32, Hk=4, seq_len=8192,
                            num_kv_splits=8),
    "poc_k2v4_nc": Workload("poc_k2v4_nc", "k2v4_nc", n_spec=8, B=4, Hq=32, Hk=4, seq_len=8192,
                            num_kv_splits=8),
    # a continuation chunk of 128 query tokens (1024 rows per kv-head: 16 row
    # tiles of 64 over the same pages) on the PoC cache
    "cont_k8v4": Workload("cont_k8v4", "k8v4", n_spec=128, B=1, Hq=32, Hk=4, seq_len=8192,
                          num_kv_splits=8),
}


@dataclass
class Inputs:
    wl: Workload
    seed: int
    seq_lens: np.ndarray        # int32 [B], total length incl. drafts
    q: torch.Tensor             # fp16 [n_spec, B, Hq, D]
    k: torch.Tensor             # fp16 [tokens, Hk, D]
    v: torch.Tensor             # fp16 [tokens, Hk, D]
    tok_off: np.ndarray         # int64 [B]
    block_table: np.ndarray     # int32 [B, max_blocks] (-1 past the end)
    num_blocks: int
    slots: np.ndarray           # int32 [tokens]: cache slot of every token row
    extra: dict = field(default_factory=dict)

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    def prefix_rows(self) -> np.ndarray:
        """Rows of K/V holding the cached prefix (all but the last n_spec per sequence)."""
        n = self.wl.n_spec
        return np.concatenate([np.arange(o, o + L - n) for o, L in zip(self.tok_off, self.seq_lens)])

    def draft_rows(self) -> np.ndarray:
        """Rows of K/V holding the draft tokens, ordered [b][n]."""
        n = self.wl.n_spec
        return np.concatenate([np.arange(o + L - n, o + L) for o, L in zip(self.tok_off, self.seq_lens)])


def make_inputs(wl: Workload, seed: int) -> Inputs:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    B = wl.B
    if wl.len_range:
        lo, hi = wl.len_range
        seq_lens = torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).numpy()
    else:
        seq_lens = np.full(B, wl.seq_len, np.int64)
    seq_lens = seq_lens.astype(np.int32)
    if np.any(seq_lens < wl.n_spec):
        raise ValueError("every sequence must hold at least n_spec tokens")
    tokens = int(seq_lens.sum())
    q = torch.randn((wl.n_spec, B, wl.Hq, HEAD_DIM), generator=g, dtype=torch.float32).half()
    k32 = torch.randn((tokens, wl.Hk, HEAD_DIM), generator=g, dtype=torch.float32)
    v = torch.randn((tokens, wl.Hk, HEAD_DIM), generator=g, dtype=torch.float32).half()
    lo_s, hi_s = wl.k_scale
    if (lo_s, hi_s) != (1.0, 1.0):
        sc = torch.rand((wl.Hk,), generator=g, dtype=torch.float32) * (hi_s - lo_s) + lo_s
        k32 = k32 * sc.view(1, wl.Hk, 1)
    k = k32.half()
    del k32
    nblk = (seq_lens.astype(np.int64) + BLOCK - 1) // BLOCK
    num_blocks = int(nblk.sum())
    if wl.shuffled_blocks:
        perm = torch.randperm(num_blocks, generator=g).numpy().astype(np.int32)
    else:
        perm = np.arange(num_blocks, dtype=np.int32)
    max_blocks = int(nblk.max())
    bt = np.full((B, max_blocks), -1, np.int32)
    start = 0
    for b in range(B):
        bt[b, : nblk[b]] = perm[start : start + nblk[b]]
        start += int(nblk[b])
    tok_off = np.zeros(B, np.int64)
    tok_off[1:] = np.cumsum(seq_lens[:-1].astype(np.int64))
    slots = np.empty(tokens, np.int32)
    for b in range(B):
        p = np.arange(seq_lens[b], dtype=np.int64)
        slots[tok_off[b] : tok_off[b] + seq_lens[b]] = (bt[b, p // BLOCK].astype(np.int64) * BLOCK
                                                          + p % BLOCK).astype(np.int32)
    return Inputs(wl, seed, seq_lens, q, k, v, tok_off, bt, num_blocks, slots)


def scaled(wl: Workload, **kw) -> Workload:
    """A copy of a workload with some fields replaced (smaller parity cases)."""
    return replace(wl, **kw)


def algorithmic_kv_bytes(wl: Workload, seq_lens: np.ndarray, page_bytes: int) -> int:
    """Compressed KV bytes one verify call must read: every page of every
    (sequence, kv-head) once."""
    pages = int(((seq_lens.astype(np.int64) + BLOCK - 1) // BLOCK).sum())
    return pages * wl.Hk * page_bytes
