"""ctypes binding of libtqkv (include/tqkv.h), same names as the C ABI.

Argument marshalling only: tensors are checked for device, dtype and
contiguity, and their data pointers plus the current CUDA stream are handed to
the C entry points.  Every step of the path runs in the CUDA kernels; there is
no CPU fallback, and a missing library raises instead of degrading.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import _build

TQ_OK = 0
TQ_ERR_INVALID_ARG = 1
TQ_ERR_UNSUPPORTED = 2
TQ_ERR_MISALIGNED = 3
TQ_ERR_CUDA = 4
TQ_ERR_TIMEOUT = 5
TQ_PRESET_K8V4 = 0
TQ_PRESET_K3V4_NC = 1
TQ_PRESET_K3V4 = 2
TQ_PRESET_K3V4_NC_RS = 3
TQ_PRESET_K4V4_NC = 4
TQ_PRESET_K2V4_NC = 5
PRESETS = {"k8v4": TQ_PRESET_K8V4, "k3v4_nc": TQ_PRESET_K3V4_NC, "k3v4": TQ_PRESET_K3V4,
           "k3v4_nc_rs": TQ_PRESET_K3V4_NC_RS, "k4v4_nc": TQ_PRESET_K4V4_NC, "k2v4_nc": TQ_PRESET_K2V4_NC}

_lock = threading.Lock()
_lib = None


class TqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tq_status_string(status)} (status {status})")


class tq_cache_desc(ctypes.Structure):
    _fields_ = [("preset", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("num_blocks", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cache", ctypes.c_void_p)]


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libtqkv.so.  Raises if it is missing (after an optional build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            if not build_if_missing:
                raise RuntimeError(f"libtqkv.so not found at {_build.LIB}; build it with "
                                   "quantized_kv_cache_store_gb300._build.build()")
            _build.build()
        lib = ctypes.CDLL(_build.LIB)
        P, I, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        lib.tq_page_bytes.restype = S
        lib.tq_page_bytes.argtypes = [I]
        lib.tq_partials_bytes.restype = S
        lib.tq_partials_bytes.argtypes = [I, I, I, I]
        lib.tq_codebook.restype = I
        lib.tq_codebook.argtypes = [I, P]
        lib.tq_key_levels.restype = I
        lib.tq_key_levels.argtypes = [I]
        lib.tq_status_string.restype = ctypes.c_char_p
        lib.tq_status_string.argtypes = [I]
        D = ctypes.POINTER(tq_cache_desc)
        lib.tq_store.restype = I
        lib.tq_store.argtypes = [D, P, P, P, I, P]
        lib.tq_verify_stage1.restype = I
        lib.tq_verify_stage1.argtypes = [D, P, P, I, P, I, I, I, I, I, P, P, P]
        lib.tq_verify_stage2.restype = I
        lib.tq_verify_stage2.argtypes = [P, P, I, I, I, I, I, P, P]
        lib.tq_verify.restype = I
        lib.tq_verify.argtypes = [D, P, P, I, P, I, I, I, I, I, P, P, P, P, P]
        lib.tq_store_verify.restype = I
        lib.tq_store_verify.argtypes = [D, P, P, P, P, I, P, I, I, I, I, I, P, P, P, P, P]
        lib.tq_verify_noalloc.restype = I
        lib.tq_verify_noalloc.argtypes = [D, P, P, I, P, I, I, I, I, I, P, P]
        lib.tq_device_status.restype = I
        lib.tq_device_status.argtypes = []
        _lib = lib
        return lib


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, dtype, name: str) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _check(status: int, where: str):
    if status != TQ_OK:
        raise TqError(status, where)


# ------------------------------------------------------------ host helpers

def tq_page_bytes(preset: int) -> int:
    return int(load().tq_page_bytes(int(preset)))


def tq_partials_bytes(n_spec: int, B: int, Hq: int, num_kv_splits: int) -> int:
    return int(load().tq_partials_bytes(n_spec, B, Hq, num_kv_splits))


def tq_key_levels(preset: int) -> int:
    return int(load().tq_key_levels(int(preset)))


def tq_codebook(preset: int = TQ_PRESET_K3V4_NC) -> np.ndarray:
    out = np.zeros(max(tq_key_levels(preset), 1), np.float32)
    _check(load().tq_codebook(int(preset), ctypes.c_void_p(out.ctypes.data)), "tq_codebook")
    return out


def tq_device_status() -> int:
    """Reads and clears the sticky device-side error word (synchronises)."""
    return int(load().tq_device_status())


def tq_status_string(status: int) -> str:
    return load().tq_status_string(int(status)).decode()


def cache_desc(cache: torch.Tensor, preset: int) -> tq_cache_desc:
    """Descriptor of a uint8 CUDA tensor shaped [num_blocks, Hk, page_bytes]."""
    _dev(cache, torch.uint8, "cache")
    if cache.dim() != 3 or cache.shape[2] != tq_page_bytes(preset):
        raise ValueError("cache must be [num_blocks, num_kv_heads, tq_page_bytes(preset)]")
    return tq_cache_desc(int(preset), 128, 16, int(cache.shape[1]), int(cache.shape[0]), 0,
                         cache.data_ptr())


def alloc_cache(num_blocks: int, num_kv_heads: int, preset: int, device="cuda") -> torch.Tensor:
    """A zeroed cache tensor (allocation is the caller's, done with torch)."""
    return torch.zeros((num_blocks, num_kv_heads, tq_page_bytes(preset)), dtype=torch.uint8, device=device)


# ------------------------------------------------------------- entry points

def tq_store(cache: torch.Tensor, preset: int, k: torch.Tensor, v: torch.Tensor,
             slot_mapping: torch.Tensor, stream=None) -> None:
    d = cache_desc(cache, preset)
    T = int(slot_mapping.shape[0])
    if k.shape != (T, d.num_kv_heads, 128) or v.shape != k.shape:
        raise ValueError("k and v must be [T, num_kv_heads, 128]")
    st = load().tq_store(ctypes.byref(d), _dev(k, torch.float16, "k"), _dev(v, torch.float16, "v"),
                         _dev(slot_mapping, torch.int32, "slot_mapping"), T, _stream(stream))
    _check(st, "tq_store")


def tq_verify_stage1(cache: torch.Tensor, preset: int, q: torch.Tensor, block_table: torch.Tensor,
                     seq_lens: torch.Tensor, num_kv_splits: int, causal: bool,
                     partial_o: torch.Tensor, partial_lse: torch.Tensor, stream=None) -> None:
    d = cache_desc(cache, preset)
    n_spec, B, Hq, D = q.shape
    S = int(num_kv_splits)
    if D != 128 or block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("q [n_spec,B,Hq,128], block_table [B,max_blocks], seq_lens [B]")
    if partial_o.shape != (n_spec, B, Hq, S, 128) or partial_lse.shape != (n_spec, B, Hq, S):
        raise ValueError("partial_o [n_spec,B,Hq,S,128] and partial_lse [n_spec,B,Hq,S]")
    st = load().tq_verify_stage1(ctypes.byref(d), _dev(q, torch.float16, "q"),
                                 _dev(block_table, torch.int32, "block_table"), int(block_table.shape[1]),
                                 _dev(seq_lens, torch.int32, "seq_lens"), n_spec, B, Hq, S, int(bool(causal)),
                                 _dev(partial_o, torch.float32, "partial_o"),
                                 _dev(partial_lse, torch.float32, "partial_lse"), _stream(stream))
    _check(st, "tq_verify_stage1")


def tq_verify_stage2(partial_o: torch.Tensor, partial_lse: torch.Tensor, out: torch.Tensor,
                     stream=None) -> None:
    n_spec, B, Hq, S, D = partial_o.shape
    if partial_lse.shape != (n_spec, B, Hq, S) or out.shape != (n_spec, B, Hq, D):
        raise ValueError("partial_lse [n_spec,B,Hq,S], out [n_spec,B,Hq,128]")
    st = load().tq_verify_stage2(_dev(partial_o, torch.float32, "partial_o"),
                                 _dev(partial_lse, torch.float32, "partial_lse"), n_spec, B, Hq, D, S,
                                 _dev(out, torch.float32, "out"), _stream(stream))
    _check(st, "tq_verify_stage2")


def tq_verify(cache: torch.Tensor, preset: int, q: torch.Tensor, block_table: torch.Tensor,
              seq_lens: torch.Tensor, num_kv_splits: int, causal: bool, partial_o: torch.Tensor,
              partial_lse: torch.Tensor, tickets: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """Both stages in one call (one launch when S <= 32 and every CTA fits on the device at once).
    tickets: int32 [B, Hk, 4], zero before the first call, zero again after each."""
    d = cache_desc(cache, preset)
    n_spec, B, Hq, D = q.shape
    S = int(num_kv_splits)
    if D != 128 or block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("q [n_spec,B,Hq,128], block_table [B,max_blocks], seq_lens [B]")
    if partial_o.shape != (n_spec, B, Hq, S, 128) or partial_lse.shape != (n_spec, B, Hq, S):
        raise ValueError("partial_o [n_spec,B,Hq,S,128] and partial_lse [n_spec,B,Hq,S]")
    if out.shape != (n_spec, B, Hq, 128) or tickets.shape != (B, d.num_kv_heads, 4):
        raise ValueError("out [n_spec,B,Hq,128], tickets [B,Hk,4]")
    st = load().tq_verify(ctypes.byref(d), _dev(q, torch.float16, "q"),
                          _dev(block_table, torch.int32, "block_table"), int(block_table.shape[1]),
                          _dev(seq_lens, torch.int32, "seq_lens"), n_spec, B, Hq, S, int(bool(causal)),
                          _dev(partial_o, torch.float32, "partial_o"), _dev(partial_lse, torch.float32, "partial_lse"),
                          _dev(tickets, torch.int32, "tickets"), _dev(out, torch.float32, "out"), _stream(stream))
    _check(st, "tq_verify")


def tq_store_verify(cache: torch.Tensor, preset: int, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
                    block_table: torch.Tensor, seq_lens: torch.Tensor, num_kv_splits: int, causal: bool,
                    partial_o: torch.Tensor, partial_lse: torch.Tensor, tickets: torch.Tensor, out: torch.Tensor,
                    stream=None) -> None:
    """Store the drafts (k_new, v_new: fp16 [B * n_spec, Hk, 128], sequence-major)
    at the last n_spec positions of each sequence, then verify (one launch
    where tq_verify takes one)."""
    d = cache_desc(cache, preset)
    n_spec, B, Hq, D = q.shape
    if k_new.shape != (B * n_spec, d.num_kv_heads, 128) or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be [B * n_spec, Hk, 128]")
    if D != 128 or block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("q [n_spec,B,Hq,128], block_table [B,max_blocks], seq_lens [B]")
    S = int(num_kv_splits)
    if partial_o.shape != (n_spec, B, Hq, S, 128) or partial_lse.shape != (n_spec, B, Hq, S):
        raise ValueError("partial_o [n_spec,B,Hq,S,128] and partial_lse [n_spec,B,Hq,S]")
    if out.shape != (n_spec, B, Hq, 128) or tickets.shape != (B, d.num_kv_heads, 4):
        raise ValueError("out [n_spec,B,Hq,128], tickets [B,Hk,4]")
    st = load().tq_store_verify(ctypes.byref(d), _dev(k_new, torch.float16, "k_new"),
                                _dev(v_new, torch.float16, "v_new"), _dev(q, torch.float16, "q"),
                                _dev(block_table, torch.int32, "block_table"), int(block_table.shape[1]),
                                _dev(seq_lens, torch.int32, "seq_lens"), n_spec, B, Hq, S, int(bool(causal)),
                                _dev(partial_o, torch.float32, "partial_o"),
                                _dev(partial_lse, torch.float32, "partial_lse"), _dev(tickets, torch.int32, "tickets"),
                                _dev(out, torch.float32, "out"), _stream(stream))
    _check(st, "tq_store_verify")


def tq_verify_noalloc(cache: torch.Tensor, preset: int, q: torch.Tensor, block_table: torch.Tensor,
                      seq_lens: torch.Tensor, num_kv_splits: int, causal: bool, out: torch.Tensor,
                      stream=None) -> None:
    """tq_verify with the library's own scratch: no partial or counter buffers.
    The first call on a device sets the scratch up (synchronising); calls on
    one device must not overlap."""
    d = cache_desc(cache, preset)
    n_spec, B, Hq, D = q.shape
    if D != 128 or block_table.dim() != 2 or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("q [n_spec,B,Hq,128], block_table [B,max_blocks], seq_lens [B]")
    if out.shape != (n_spec, B, Hq, 128):
        raise ValueError("out [n_spec,B,Hq,128]")
    st = load().tq_verify_noalloc(ctypes.byref(d), _dev(q, torch.float16, "q"),
                                  _dev(block_table, torch.int32, "block_table"), int(block_table.shape[1]),
                                  _dev(seq_lens, torch.int32, "seq_lens"), n_spec, B, Hq, int(num_kv_splits),
                                  int(bool(causal)), _dev(out, torch.float32, "out"), _stream(stream))
    _check(st, "tq_verify_noalloc")
