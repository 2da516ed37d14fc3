"""The page-printed figures pin the cache byte budget and the roofline
arithmetic (tests/golden/page_figures.txt lists each with its citation)."""
import os

import numpy as np

from quantized_kv_cache_store_gb300.inputs import WORKLOADS, algorithmic_kv_bytes, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")


def _figs():
    out = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if "=" in line:
            k, v = line.split("=", 1)
            out[k.strip()] = float(v)
    return out


def test_k8v4_slot_size(oracle_lib):
    f = _figs()
    assert oracle_lib.page_bytes(0) == 16 * f["k8v4_slot_bytes"]


def test_poc_bytes_per_call(oracle_lib):
    f = _figs()
    wl = WORKLOADS["poc_k8v4"]
    assert (wl.n_spec, wl.B, wl.Hq, wl.Hk, wl.seq_len) == (f["poc_n_spec"], f["poc_B"], f["poc_Hq"],
                                                         f["poc_Hk"], f["poc_seqlen"])
    lens = np.full(wl.B, wl.seq_len)
    nbytes = algorithmic_kv_bytes(wl, lens, oracle_lib.page_bytes(0))
    assert nbytes == f["poc_blocks"] * 16 * f["poc_kv_heads"] * f["k8v4_slot_bytes"]
    assert round(nbytes / 1e6, 1) == f["poc_kv_megabytes"]


def test_arithmetic_intensity_pins_slot_sizes(oracle_lib):
    """FLOP per KV byte of the fused kernel: 4 * R * D per token-head with
    R = n_spec * Hq / Hk = 64 rows, over the slot size."""
    f = _figs()
    flop_per_token_head = 4 * 64 * f["poc_D"]
    assert round(flop_per_token_head / (oracle_lib.page_bytes(0) / 16), 1) == f["fused_ai_k8v4"]
    assert round(flop_per_token_head / (oracle_lib.page_bytes(1) / 16), 1) == f["fused_ai_k3v4_nc"]


def test_single_query_flops():
    f = _figs()
    flops = 2 * f["poc_B"] * f["poc_Hq"] * f["poc_seqlen"] * f["poc_D"] * 2
    assert round(flops / 1e9, 2) == f["single_query_gflop"]
