"""tq_store on the GPU: cache bytes bit-exact against the oracle's encoder."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_store_gb300 import tqkv
from quantized_kv_cache_store_gb300.inputs import WORKLOADS, make_inputs
from tests.helpers import oracle_cache, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _store_both(O, preset, k, v, slots, nb, hk):
    cache = tqkv.alloc_cache(nb, hk, preset)
    tqkv.tq_store(cache, preset, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                  torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    ref = np.zeros((nb, hk, O.page_bytes(preset)), np.uint8)
    O.store(preset, ref, k, v, slots)
    return cache.cpu().numpy(), ref


@pytest.mark.parametrize("preset", [0, 1, 2, 3, 4, 5])
@pytest.mark.parametrize("seed", [42, 101, 202])
def test_store_random_ragged(oracle_lib, preset, seed):
    rng = np.random.default_rng(seed)
    nb, hk, T = 9, 3, 37
    scale = rng.choice([1e-3, 1.0, 50.0], size=(T, hk, 1))
    k = (rng.standard_normal((T, hk, 128)) * scale).astype(np.float16)
    v = (rng.standard_normal((T, hk, 128)) * scale[::-1]).astype(np.float16)
    slots = rng.permutation(nb * 16)[:T].astype(np.int32)
    slots[3] = -1
    slots[7] = nb * 16 + 5  # out of range: skipped
    got, ref = _store_both(oracle_lib, preset, k, v, slots, nb, hk)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("preset", [0, 1, 2, 3, 4, 5])
def test_store_special_values(oracle_lib, preset):
    hk, T = 1, 8
    k = np.zeros((T, hk, 128), np.float16)
    v = np.zeros((T, hk, 128), np.float16)
    k[1] = 448.0
    k[2, 0, ::2] = -0.0
    k[3] = np.float16(6e-8)            # fp16 subnormal keys
    k[4] = np.linspace(-60000, 60000, 128).astype(np.float16)
    k[5, 0, 0] = 1.0                   # one-hot key
    k[6] = np.float16(-2.5)
    k[7, 0, :64] = 1e-4
    v[1] = -0.0                        # constant negative zero
    v[2] = 3.0                         # constant
    v[3] = np.linspace(-1, 1, 128).astype(np.float16)
    v[4] = np.float16(6e-8)
    v[4, 0, 5] = 0
    v[5] = np.linspace(-60000, 60000, 128).astype(np.float16)
    v[6, 0, ::3] = 1e-5
    v[7] = np.arange(128) % 16
    got, ref = _store_both(oracle_lib, preset, k, v, np.arange(T, dtype=np.int32), 1, hk)
    assert np.array_equal(got, ref)


def test_store_e4m3_exhaustive(oracle_lib):
    """Every fp16 bit pattern (NaN and infinities included) as a k8v4 key."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    k = bits.view(np.float16).reshape(512, 1, 128)
    v = np.zeros_like(k)
    got, ref = _store_both(oracle_lib, 0, k, v, np.arange(512, dtype=np.int32), 32, 1)
    assert np.array_equal(got, ref)


def test_store_zero_tokens():
    cache = tqkv.alloc_cache(2, 1, 0)
    e = torch.empty((0, 1, 128), dtype=torch.float16, device="cuda")
    tqkv.tq_store(cache, 0, e, e, torch.empty((0,), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert int(cache.sum()) == 0


@pytest.mark.parametrize("name", ["tiny_k8v4", "poc_k8v4", "poc_k3v4_nc", "decode_k3v4_nc",
                                  "longctx_k3v4_nc"])
def test_store_full_workload_cache(oracle_lib, name):
    """The whole cache of each workload (prefix and drafts) is bit-exact."""
    inp = make_inputs(WORKLOADS[name], 1000)
    from quantized_kv_cache_store_gb300.step import SpecVerify

    sv = SpecVerify(inp)
    sv.prefill()
    sv.store()
    torch.cuda.synchronize()
    got = sv.caches[0].cpu().numpy()
    ref = oracle_cache(oracle_lib, inp)
    assert np.array_equal(got, ref)
