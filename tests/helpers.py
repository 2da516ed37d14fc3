"""Shared test helpers: oracle-side cache building and tolerance checks."""
import numpy as np

from quantized_kv_cache_store_gb300.inputs import Inputs

# Attention-output tolerance: |gpu - oracle| <= ATOL + RTOL * |oracle|, and the
# plain absolute error must stay under ATOL as well for the fp16-operand path.
ATOL = 2e-3
RTOL = 1e-2


def oracle_cache(O, inp: Inputs) -> np.ndarray:
    """Encode every token (cached prefix and drafts) with the oracle."""
    cache = np.zeros((inp.num_blocks, inp.wl.Hk, O.page_bytes(inp.wl.preset_id)), np.uint8)
    O.store(inp.wl.preset_id, cache, inp.k.numpy(), inp.v.numpy(), inp.slots)
    return cache


def assert_close(got, ref, atol=ATOL, rtol=RTOL, what="output"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bad = err > atol + rtol * np.abs(ref)
    assert not np.any(np.isnan(got)), f"{what}: NaN in result"
    assert not bad.any(), (f"{what}: {bad.sum()} elements out of tolerance, max err "
                           f"{err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}")
    return float(err.max())


def require_gpu():
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from quantized_kv_cache_store_gb300 import _build, tqkv

    _build.build()
    tqkv.load()


def gpu_run(inp: Inputs, S=None, causal=None, prefill=True, step=True):
    """Fill a GPU cache with the prefix via tq_store, then run one step (store
    the drafts, stage 1, stage 2).  Returns numpy (cache, part_o, part_lse, out)."""
    import torch

    from quantized_kv_cache_store_gb300.step import SpecVerify

    wl = inp.wl if causal is None else __import__("dataclasses").replace(inp.wl, causal=causal)
    inp = __import__("dataclasses").replace(inp, wl=wl)
    sv = SpecVerify(inp, num_kv_splits=S)
    if prefill:
        sv.prefill()
    if step:
        sv.step()
    torch.cuda.synchronize()
    return (sv.caches[0].cpu().numpy(), sv.part_o.cpu().numpy(), sv.part_lse.cpu().numpy(),
            sv.out.cpu().numpy())
