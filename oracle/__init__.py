"""CPU oracle for paged decode attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library (``paged_kv_cache_311_gb300``) never imports it and shares no code
with it.

The arithmetic lives in ``pkv_oracle.c`` (plain C, fp64, built by
``oracle.build``); this module only marshals numpy arrays.  The block
manager used by the pins is ``oracle.block_manager`` (plain Python).

Every function here is pinned by ``tests/test_oracle_pins.py`` against
facts that the pages and the mathematics fix (the worked block-count example,
closed forms, library softmax attention, paging invariants).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import build_oracle, library_path

F32, F16, BF16 = 0, 1, 2
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16}
BAD_BLOCK, BAD_SLOT, BAD_LEN = 1, 2, 8

_lib = None


def lib():
    global _lib
    if _lib is None:
        # PKV_ORACLE_LIB lets the mutation tests load a deliberately broken
        # build of the same source; it is never set outside the test suite.
        path = os.environ.get("PKV_ORACLE_LIB") or library_path()
        if not os.path.exists(path):
            build_oracle()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, u32, f64, sz = (ctypes.c_int, ctypes.c_int64, ctypes.c_uint32,
                                  ctypes.c_double, ctypes.c_size_t)
        L.pkv_oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.pkv_oracle_f16_to_f64.restype = f64
        L.pkv_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.pkv_oracle_bf16_to_f64.restype = f64
        L.pkv_oracle_blocks_for_tokens.argtypes = [i64, i64]
        L.pkv_oracle_blocks_for_tokens.restype = i64
        L.pkv_oracle_paged_attention.argtypes = [P, P, P, P, i32, P, i32, P, i32, i32, i32, i32,
                                                 i32, i64, f64, i32, i32]
        L.pkv_oracle_paged_attention.restype = u32
        L.pkv_oracle_contiguous_attention.argtypes = [P, P, P, P, i32, i32, i32, i32, f64]
        L.pkv_oracle_contiguous_attention.restype = None
        L.pkv_oracle_reshape_and_cache.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i64]
        L.pkv_oracle_reshape_and_cache.restype = u32
        L.pkv_oracle_copy_blocks.argtypes = [P, P, i32, P, i32, sz, i64]
        L.pkv_oracle_copy_blocks.restype = u32
        L.pkv_oracle_swap_blocks.argtypes = [P, P, P, P, i32, P, i32, sz, i64, i64, i32]
        L.pkv_oracle_swap_blocks.restype = u32
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _raw(a: np.ndarray) -> np.ndarray:
    """A C-contiguous view of the array's raw elements (bf16 arrives as uint16)."""
    return np.ascontiguousarray(a)


def f16_to_f64(bits: int) -> float:
    return lib().pkv_oracle_f16_to_f64(int(bits))


def bf16_to_f64(bits: int) -> float:
    return lib().pkv_oracle_bf16_to_f64(int(bits))


def blocks_for_tokens(n_tokens: int, block_size: int) -> int:
    return int(lib().pkv_oracle_blocks_for_tokens(int(n_tokens), int(block_size)))


def paged_attention(q, k_cache, v_cache, dtype: str, block_tables, context_lens,
                    num_kv_heads: int, scale: float, partition_size: int = 0,
                    nthreads: int = 1):
    """fp64 [B, H, D] output of single-query attention over the paged cache.

    q: [B, H, D]; k_cache, v_cache: [NB, Hk, bs, D]; all three as raw element
    arrays of ``dtype`` (float32, float16, or uint16 holding bf16 bits).
    block_tables: int32 [B, MB]; context_lens: int32 [B].  ``scale`` is used
    as given (pass the float32 value the GPU sees).  Returns (out, status)."""
    q = _raw(q); k_cache = _raw(k_cache); v_cache = _raw(v_cache)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H, D = q.shape
    NB, Hk, bs, D2 = k_cache.shape
    assert D2 == D and Hk == num_kv_heads and v_cache.shape == k_cache.shape
    out = np.zeros((B, H, D), dtype=np.float64)
    st = lib().pkv_oracle_paged_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), DTYPE_CODES[dtype], _ptr(bt),
        int(bt.shape[1]), _ptr(cl), B, H, Hk, D, bs, NB, float(scale), int(partition_size),
        int(nthreads))
    return out, int(st)


def contiguous_attention(q, K, V, scale: float):
    """fp64 attention of q [H, D] over contiguous K, V [L, Hk, D] (fp64 inputs)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    H, D = q.shape
    L, Hk, _ = K.shape
    out = np.zeros((H, D), dtype=np.float64)
    lib().pkv_oracle_contiguous_attention(_ptr(out), _ptr(q), _ptr(K), _ptr(V), L, H, Hk, D,
                                          float(scale))
    return out


def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping):
    """In-place scatter of key/value [T, Hk, D] into k_cache/v_cache [NB, Hk, bs, D]."""
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    key = _raw(key); value = _raw(value)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T, Hk, D = key.shape
    NB, Hk2, bs, D2 = k_cache.shape
    assert Hk2 == Hk and D2 == D
    code = {4: F32, 2: F16}[k_cache.dtype.itemsize]   # 2-byte types are copied as bits
    return int(lib().pkv_oracle_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache),
                                                  _ptr(v_cache), code, _ptr(sm), T, Hk, D, bs, NB))


def copy_blocks(k_caches, v_caches, src_dst_pairs):
    """In-place copy-on-write block copies over every layer's caches."""
    nl = len(k_caches)
    for c in list(k_caches) + list(v_caches):
        assert c.flags.c_contiguous
    kp = (ctypes.c_void_p * nl)(*[c.ctypes.data for c in k_caches])
    vp = (ctypes.c_void_p * nl)(*[c.ctypes.data for c in v_caches])
    pairs = np.ascontiguousarray(src_dst_pairs, dtype=np.int64).reshape(-1, 2)
    NB = k_caches[0].shape[0]
    block_bytes = k_caches[0][0].nbytes
    return int(lib().pkv_oracle_copy_blocks(kp, vp, nl, _ptr(pairs), pairs.shape[0],
                                            block_bytes, NB))



def swap_blocks(gpu_k, gpu_v, host_k, host_v, pairs, direction):
    """Block swap between two pools of every layer: pairs of (gpu block,
    host block); direction 0 copies gpu -> host, 1 host -> gpu."""
    nl = len(gpu_k)
    for c in list(gpu_k) + list(gpu_v) + list(host_k) + list(host_v):
        assert c.flags.c_contiguous
    arr = lambda cs: (ctypes.c_void_p * nl)(*[c.ctypes.data for c in cs])
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    return int(lib().pkv_oracle_swap_blocks(arr(gpu_k), arr(gpu_v), arr(host_k), arr(host_v), nl,
                                            _ptr(pr), pr.shape[0], gpu_k[0][0].nbytes,
                                            gpu_k[0].shape[0], host_k[0].shape[0], int(direction)))