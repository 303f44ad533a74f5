"""paged_kv_cache_311_gb300 -- GB300-native paged KV-cache decode attention.

A thin ctypes binding over ``libpkv.so`` (C ABI in ``include/pkv.h``).  Every
step of the path runs in the library's CUDA kernels; this module only turns
torch tensors into pointers, sizes and the current CUDA stream.  torch is
used for device memory and streams, nothing else.  There is no CPU fallback:
calling into the library without a built ``libpkv.so`` raises.

Operations (PagedAttention: Efficient LLM Serving with vLLM, "The
PagedAttention Algorithm" and "Advanced Features"):
  paged_attention_decode  single-query attention over a block-table-mapped cache
  reshape_and_cache       scatter of new tokens' K/V into their slots
  copy_blocks             copy-on-write copy of shared blocks
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

import torch

from .build import library_path

__all__ = [
    "PkvError", "load_library", "paged_attention_decode", "reshape_and_cache", "copy_blocks",
    "paged_attention_workspace_bytes", "status_string", "last_decode_launches",
    "paged_attention_decode_shared", "plan_shared_prefix", "SharedPrefixPlan",
    "set_decode_engine", "last_decode_engine", "kv_cache_usage", "KvCacheUsage", "swap_blocks",
    "SWAP_OUT", "SWAP_IN", "BlockPool",
    "DEV_BAD_BLOCK", "DEV_BAD_SLOT", "DEV_TIMEOUT", "DEV_BAD_CONTEXT_LEN", "DEV_DRAIN_TIMEOUT",
    "HEADER_PATH", "bounded_wait_hook",
]

HEADER_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                           "include", "pkv.h")

PKV_F32, PKV_F16, PKV_BF16 = 0, 1, 2
_DTYPE = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}

DEV_BAD_BLOCK, DEV_BAD_SLOT, DEV_TIMEOUT, DEV_BAD_CONTEXT_LEN, DEV_DRAIN_TIMEOUT = 1, 2, 4, 8, 16

_lib = None


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Loads libpkv.so (built by ``paged_kv_cache_311_gb300.build``)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise ImportError(f"libpkv.so not built at {p}; run python -m paged_kv_cache_311_gb300.build")
    L = ctypes.CDLL(p)
    vp, i32, i64, u64, f32 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                              ctypes.c_float)
    L.pkv_paged_attention_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.pkv_paged_attention_workspace_bytes.restype = u64
    L.pkv_paged_attention_decode.argtypes = [vp, i32, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32,
                                             i32, i32, i64, i32, f32, i32, vp, u64, vp, vp]
    L.pkv_paged_attention_decode.restype = i32
    L.pkv_paged_attention_decode_shared.argtypes = [vp, i32, vp, vp, vp, i32, vp, i32, vp, i32,
                                                    i32, i32, i32, i32, i64, i32, f32, vp, i32,
                                                    i32, i32, vp, u64, vp, vp]
    L.pkv_paged_attention_decode_shared.restype = i32
    L.pkv_plan_shared_prefix.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp, u64,
                                         ctypes.POINTER(ctypes.c_size_t),
                                         ctypes.POINTER(ctypes.c_size_t)]
    L.pkv_plan_shared_prefix.restype = i32
    L.pkv_shared_plan_max_ints.argtypes = [i32, i32, i32, i32, i32]
    L.pkv_shared_plan_max_ints.restype = u64
    L.pkv_kv_cache_usage.argtypes = [vp, vp, i32, i32, i32, i64, ctypes.POINTER(i64),
                                     ctypes.POINTER(i64), ctypes.POINTER(i64)]
    L.pkv_kv_cache_usage.restype = i32
    L.pkv_block_pool_create.argtypes = [i64, i32]
    L.pkv_block_pool_create.restype = vp
    L.pkv_block_pool_destroy.argtypes = [vp]
    L.pkv_block_pool_destroy.restype = None
    L.pkv_block_pool_allocate_prompt.argtypes = [vp, vp, i32, vp, i32, ctypes.POINTER(i32)]
    L.pkv_block_pool_allocate_prompt.restype = i32
    L.pkv_block_pool_commit_prompt.argtypes = [vp, vp, i32, vp]
    L.pkv_block_pool_commit_prompt.restype = i32
    L.pkv_block_pool_allocate.argtypes = [vp, i32, vp]
    L.pkv_block_pool_allocate.restype = i32
    L.pkv_block_pool_fork.argtypes = [vp, vp, i32]
    L.pkv_block_pool_fork.restype = i32
    L.pkv_block_pool_release.argtypes = [vp, vp, i32]
    L.pkv_block_pool_release.restype = i32
    L.pkv_block_pool_prepare_write.argtypes = [vp, vp, i32, vp]
    L.pkv_block_pool_prepare_write.restype = i32
    L.pkv_block_pool_append_slots.argtypes = [vp, vp, i32, vp, i32, vp, vp, ctypes.POINTER(i32),
                                              ctypes.POINTER(i32)]
    L.pkv_block_pool_append_slots.restype = i32
    L.pkv_block_pool_available.argtypes = [vp]
    L.pkv_block_pool_available.restype = i64
    L.pkv_block_pool_refcount.argtypes = [vp, i32]
    L.pkv_block_pool_refcount.restype = i32
    L.pkv_block_pool_is_cached.argtypes = [vp, i32]
    L.pkv_block_pool_is_cached.restype = i32
    L.pkv_block_pool_stats.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                       ctypes.POINTER(i64), ctypes.POINTER(u64), ctypes.POINTER(u64)]
    L.pkv_block_pool_stats.restype = i32
    L.pkv_reshape_and_cache.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64, vp, vp]
    L.pkv_reshape_and_cache.restype = i32
    L.pkv_copy_blocks.argtypes = [vp, vp, i32, vp, i32, u64, i64, vp, vp]
    L.pkv_copy_blocks.restype = i32
    L.pkv_swap_blocks.argtypes = [vp, vp, vp, vp, i32, vp, i32, u64, i64, i64, i32, vp, vp]
    L.pkv_swap_blocks.restype = i32
    L.pkv_status_string.argtypes = [i32]
    L.pkv_status_string.restype = ctypes.c_char_p
    L.pkv_last_decode_launches.argtypes = []
    L.pkv_last_decode_launches.restype = i32
    L.pkv_last_decode_engine.argtypes = []
    L.pkv_last_decode_engine.restype = i32
    L.pkv_decode_set_engine.argtypes = [i32]
    L.pkv_decode_set_engine.restype = i32
    L.pkv_test_bounded_wait.argtypes = [ctypes.c_uint64, ctypes.c_uint64, vp, vp]
    L.pkv_test_bounded_wait.restype = i32
    if path is None:
        _lib = L
    return L


def declared_functions(header: str = HEADER_PATH) -> list:
    """Names of the functions include/pkv.h declares."""
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return load_library().pkv_status_string(int(status)).decode()


def last_decode_launches() -> int:
    return int(load_library().pkv_last_decode_launches())


ENGINES = {"auto": 0, "cuda_core": 1, "tensor_core": 2, "tcgen05": 3}


def set_decode_engine(engine: str) -> None:
    """Process-wide engine of the decode kernels: "auto", "cuda_core", "tensor_core"
    (warp-level MMA) or "tcgen05" (the shared-prefix kernel on tcgen05 MMAs with
    TMEM accumulators; the per-sequence kernel keeps the warp-level MMA)."""
    _check(load_library().pkv_decode_set_engine(ENGINES[engine]), "pkv_decode_set_engine")


def last_decode_engine() -> str:
    code = int(load_library().pkv_last_decode_engine())
    return {1: "cuda_core", 2: "tensor_core", 3: "tcgen05"}.get(code, "none")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise PkvError(rc, what)


def _need_cuda(*ts: torch.Tensor) -> None:
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def paged_attention_workspace_bytes(num_seqs: int, num_heads: int, max_context_len: int,
                                    head_dim: int, partition_size: int = 0) -> int:
    return int(load_library().pkv_paged_attention_workspace_bytes(
        num_seqs, num_heads, max_context_len, head_dim, partition_size))


def paged_attention_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                           v_cache: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, scale: float,
                           block_size: Optional[int] = None, num_kv_heads: Optional[int] = None,
                           *, max_context_len: Optional[int] = None, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None,
                           device_status: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """out[s, h] = attention of q[s, h] over sequence s's paged K/V.

    q, out: [B, H, D]; k_cache, v_cache: [NB, Hk, bs, D]; block_tables int32
    [B, MB]; context_lens int32 [B].  ``max_context_len`` is a host-side bound
    of context_lens (read from the device, with a sync, if omitted).  A
    workspace is allocated here when the split-context path needs one and
    none is given.  device_status: optional uint32/int32 [1] tensor that the
    kernels OR error bits into."""
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, workspace, device_status)
    B, H, D = q.shape
    NB, Hk, bs, D2 = k_cache.shape
    if block_size is not None and block_size != bs:
        raise ValueError("block_size does not match k_cache")
    if num_kv_heads is not None and num_kv_heads != Hk:
        raise ValueError("num_kv_heads does not match k_cache")
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != (B, H, D):
        raise ValueError("shape mismatch")
    if q.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise ValueError("q, k_cache and v_cache must share a dtype")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0
    if workspace is None:
        nbytes = paged_attention_workspace_bytes(B, H, max_context_len, D, partition_size)
        if nbytes:
            workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    L = load_library()
    rc = L.pkv_paged_attention_decode(
        _ptr(out), _DTYPE[out.dtype], _ptr(q), _ptr(k_cache), _ptr(v_cache), _DTYPE[k_cache.dtype],
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), B, H, Hk, D, bs, NB,
        int(max_context_len), float(scale), int(partition_size), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(device_status), _stream(stream))
    _check(rc, "pkv_paged_attention_decode")
    return out


class SharedPrefixPlan:
    """A host-made plan of the shared-prefix decode (see plan_shared_prefix).

    host: the int32 plan; num_lists (CTAs per kv head), num_items, slots,
    workspace_bytes: its sizes.  to(device) gives the device copy the decode
    call takes (read only by the device, so one device copy serves every call
    with the same tables and lengths)."""

    def __init__(self, host, num_lists: int, num_items: int, slots: int, workspace_bytes: int):
        self.host = host
        self.num_lists = int(num_lists)
        self.num_items = int(num_items)
        self.slots = int(slots)
        self.workspace_bytes = int(workspace_bytes)

    def to(self, device) -> torch.Tensor:
        return torch.from_numpy(self.host).to(device)


class BlockPool:
    """Host allocator of one paged cache's blocks with prefix caching (the C
    pkv_block_pool_*).  Tables are numpy int32 arrays of block ids."""

    def __init__(self, num_blocks: int, block_size: int):
        self._L = load_library()
        self._p = self._L.pkv_block_pool_create(int(num_blocks), int(block_size))
        if not self._p:
            raise PkvError(-1, "pkv_block_pool_create")
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)

    def __del__(self):
        p, self._p = getattr(self, "_p", None), None
        if p:
            self._L.pkv_block_pool_destroy(p)

    @staticmethod
    def _i32(a):
        import numpy as np
        return np.ascontiguousarray(np.asarray(a), dtype=np.int32)

    def allocate_prompt(self, tokens):
        """-> (table, cached_tokens) for a new request's prompt tokens."""
        import numpy as np
        t = self._i32(tokens)
        table = np.empty(max(1, -(-t.size // self.block_size)), np.int32)
        cached = ctypes.c_int32(0)
        rc = self._L.pkv_block_pool_allocate_prompt(self._p, t.ctypes.data, t.size,
                                                    table.ctypes.data, table.size,
                                                    ctypes.byref(cached))
        _check(rc, "pkv_block_pool_allocate_prompt")
        return table[: -(-t.size // self.block_size)].copy(), cached.value

    def commit_prompt(self, tokens, table) -> None:
        t, tb = self._i32(tokens), self._i32(table)
        _check(self._L.pkv_block_pool_commit_prompt(self._p, t.ctypes.data, t.size, tb.ctypes.data),
               "pkv_block_pool_commit_prompt")

    def allocate(self, n: int):
        import numpy as np
        out = np.empty(max(n, 1), np.int32)
        _check(self._L.pkv_block_pool_allocate(self._p, int(n), out.ctypes.data),
               "pkv_block_pool_allocate")
        return out[:n].copy()

    def fork(self, table) -> None:
        tb = self._i32(table)
        _check(self._L.pkv_block_pool_fork(self._p, tb.ctypes.data, tb.size), "pkv_block_pool_fork")

    def release(self, table) -> None:
        tb = self._i32(table)
        _check(self._L.pkv_block_pool_release(self._p, tb.ctypes.data, tb.size),
               "pkv_block_pool_release")

    def prepare_write(self, table, logical_block: int):
        """-> (src, dst) copy pair if the block had to be copied first (the
        table, a numpy int32 array, is updated in place), else None."""
        import numpy as np
        assert table.dtype == np.int32 and table.flags.c_contiguous
        pair = np.zeros(2, np.int64)
        rc = self._L.pkv_block_pool_prepare_write(self._p, table.ctypes.data, int(logical_block),
                                                  pair.ctypes.data)
        if rc < 0:
            _check(rc, "pkv_block_pool_prepare_write")
        return (int(pair[0]), int(pair[1])) if rc == 1 else None

    def append_slots(self, tables, lens):
        """Room for one more token in every sequence of a batch, in one call:
        tables (numpy int32 [n, MB], C-contiguous, rewritten in place where a
        block is added or copied) and lens (the tokens each holds before this
        one) -> (slots int64 [n], copy pairs int64 [k, 2]).  If the pool runs
        out, raises PkvError with ``done``, the number of sequences served."""
        import numpy as np
        assert tables.dtype == np.int32 and tables.flags.c_contiguous and tables.ndim == 2
        ln = self._i32(lens)
        n = tables.shape[0]
        assert ln.shape == (n,)
        slots = np.empty(max(n, 1), np.int64)
        pairs = np.empty((max(n, 1), 2), np.int64)
        k, done = ctypes.c_int32(0), ctypes.c_int32(0)
        rc = self._L.pkv_block_pool_append_slots(self._p, tables.ctypes.data, tables.shape[1],
                                                 ln.ctypes.data, n, slots.ctypes.data,
                                                 pairs.ctypes.data, ctypes.byref(k), ctypes.byref(done))
        if rc != 0:
            e = PkvError(rc, "pkv_block_pool_append_slots")
            e.done = done.value
            raise e
        return slots[:n].copy(), pairs[:k.value].copy()

    def available(self) -> int:
        return int(self._L.pkv_block_pool_available(self._p))

    def refcount(self, block: int) -> int:
        return int(self._L.pkv_block_pool_refcount(self._p, int(block)))

    def is_cached(self, block: int) -> bool:
        return bool(self._L.pkv_block_pool_is_cached(self._p, int(block)) == 1)

    def stats(self) -> dict:
        f, c, e = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
        lk, h = ctypes.c_uint64(0), ctypes.c_uint64(0)
        _check(self._L.pkv_block_pool_stats(self._p, ctypes.byref(f), ctypes.byref(c), ctypes.byref(e),
                                            ctypes.byref(lk), ctypes.byref(h)), "pkv_block_pool_stats")
        return {"free": f.value, "cached": c.value, "evictable": e.value, "lookups": lk.value,
                "hits": h.value}


class KvCacheUsage:
    """What kv_cache_usage counted: cached tokens, distinct blocks and the
    token slots of those blocks that hold a token, for one block size."""

    def __init__(self, tokens: int, blocks: int, occupied_slots: int, block_size: int, num_seqs: int):
        self.tokens = tokens
        self.blocks = blocks
        self.occupied_slots = occupied_slots
        self.block_size = block_size
        self.num_seqs = num_seqs

    @property
    def paged_waste(self) -> float:
        """Share of the allocated slots that hold no token."""
        slots = self.blocks * self.block_size
        return 1.0 - self.occupied_slots / slots if slots else 0.0

    def reserved_waste(self, reserve_tokens: int) -> float:
        """Share unused if every sequence reserved reserve_tokens slots."""
        total = self.num_seqs * reserve_tokens
        return 1.0 - self.tokens / total if total else 0.0


def kv_cache_usage(block_tables, context_lens, block_size: int, num_blocks: int) -> KvCacheUsage:
    """Memory accounting of a paged cache from its host block tables and
    lengths (the C function pkv_kv_cache_usage)."""
    import numpy as np
    bt = np.ascontiguousarray(np.asarray(block_tables), dtype=np.int32)
    cl = np.ascontiguousarray(np.asarray(context_lens), dtype=np.int32)
    B, MB = bt.shape
    t, b, o = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    rc = load_library().pkv_kv_cache_usage(bt.ctypes.data, cl.ctypes.data, B, MB, block_size,
                                           int(num_blocks), ctypes.byref(t), ctypes.byref(b),
                                           ctypes.byref(o))
    _check(rc, "pkv_kv_cache_usage")
    return KvCacheUsage(t.value, b.value, o.value, block_size, B)


def plan_shared_prefix(block_tables, context_lens, num_heads: int, num_kv_heads: int,
                       head_dim: int, block_size: int, max_context_len: Optional[int] = None,
                       partition_size: int = 0) -> SharedPrefixPlan:
    """Host planner: orders the sequences by their block tables so that those
    whose tables start with the same block ids become neighbours, groups them
    and cuts the attention into work items.
    block_tables, context_lens: host int32 arrays (numpy or CPU tensors)."""
    import numpy as np
    bt = np.ascontiguousarray(np.asarray(block_tables), dtype=np.int32)
    cl = np.ascontiguousarray(np.asarray(context_lens), dtype=np.int32)
    B, MB = bt.shape
    if max_context_len is None:
        max_context_len = int(cl.max()) if B else 0
    L = load_library()
    cap = int(L.pkv_shared_plan_max_ints(B, num_heads, num_kv_heads, max_context_len,
                                          partition_size))
    plan = np.empty(max(cap, 16), dtype=np.int32)   # the planner writes every int it returns
    n_ints, ws = ctypes.c_size_t(0), ctypes.c_size_t(0)
    rc = L.pkv_plan_shared_prefix(bt.ctypes.data, cl.ctypes.data, B, MB, block_size, num_heads,
                                  num_kv_heads, head_dim, max_context_len, partition_size,
                                  plan.ctypes.data, plan.size, ctypes.byref(n_ints), ctypes.byref(ws))
    _check(rc, "pkv_plan_shared_prefix")
    plan = plan[: n_ints.value].copy()
    return SharedPrefixPlan(plan, plan[0], plan[7], plan[1], ws.value)


def paged_attention_decode_shared(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                  v_cache: torch.Tensor, block_tables: torch.Tensor,
                                  context_lens: torch.Tensor, scale: float, plan: SharedPrefixPlan,
                                  plan_device: torch.Tensor, *,
                                  max_context_len: Optional[int] = None,
                                  workspace: Optional[torch.Tensor] = None,
                                  device_status: Optional[torch.Tensor] = None,
                                  stream=None, **_unused) -> torch.Tensor:
    """As paged_attention_decode, reading the blocks that a plan's groups
    share once for all their members' query heads."""
    _need_cuda(out, q, k_cache, v_cache, block_tables, context_lens, plan_device, workspace,
               device_status)
    B, H, D = q.shape
    NB, Hk, bs, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != (B, H, D):
        raise ValueError("shape mismatch")
    if q.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise ValueError("q, k_cache and v_cache must share a dtype")
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or
            plan_device.dtype != torch.int32):
        raise ValueError("block_tables, context_lens and the plan must be int32")
    if max_context_len is None:
        max_context_len = int(context_lens.max().item()) if B else 0
    if workspace is None:
        workspace = torch.empty(max(plan.workspace_bytes, 16), dtype=torch.uint8, device=q.device)
    rc = load_library().pkv_paged_attention_decode_shared(
        _ptr(out), _DTYPE[out.dtype], _ptr(q), _ptr(k_cache), _ptr(v_cache), _DTYPE[k_cache.dtype],
        _ptr(block_tables), int(block_tables.shape[1]), _ptr(context_lens), B, H, Hk, D, bs, NB,
        int(max_context_len), float(scale), _ptr(plan_device), plan.num_lists, plan.num_items,
        plan.slots,
        _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(device_status),
        _stream(stream))
    _check(rc, "pkv_paged_attention_decode_shared")
    return out


def bounded_wait_hook(device_status: torch.Tensor, limit_ns: int, max_polls: int = 0,
                      stream=None) -> None:
    """Test hook: one CTA whose bounded wait (and the drain after it) must
    give up; device_status then holds DEV_TIMEOUT | DEV_DRAIN_TIMEOUT."""
    _need_cuda(device_status)
    _check(load_library().pkv_test_bounded_wait(int(limit_ns), int(max_polls), _ptr(device_status),
                                                _stream(stream)), "pkv_test_bounded_wait")


def reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, slot_mapping: torch.Tensor, *,
                      device_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """k_cache/v_cache[slot // bs, :, slot % bs, :] = key/value[t] for every slot >= 0."""
    _need_cuda(key, value, k_cache, v_cache, slot_mapping, device_status)
    T, Hk, D = key.shape
    NB, Hk2, bs, D2 = k_cache.shape
    if (Hk2, D2) != (Hk, D) or value.shape != key.shape or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch")
    if key.dtype != k_cache.dtype or value.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise ValueError("dtype mismatch")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    rc = load_library().pkv_reshape_and_cache(
        _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _DTYPE[k_cache.dtype],
        _ptr(slot_mapping), T, Hk, D, bs, NB, _ptr(device_status), _stream(stream))
    _check(rc, "pkv_reshape_and_cache")


def copy_blocks(k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor],
                src_dst_pairs: torch.Tensor, *, device_status: Optional[torch.Tensor] = None,
                stream=None) -> None:
    """Block dst of every layer's K and V cache becomes a copy of block src."""
    if len(k_caches) != len(v_caches) or not k_caches:
        raise ValueError("need one K and one V cache per layer")
    _need_cuda(*k_caches, *v_caches, src_dst_pairs, device_status)
    if src_dst_pairs.dtype != torch.int64:
        raise ValueError("src_dst_pairs must be int64")
    shape = tuple(k_caches[0].shape)
    for c in list(k_caches) + list(v_caches):
        if tuple(c.shape) != shape or c.dtype != k_caches[0].dtype:
            raise ValueError("all caches must share shape and dtype")
    nl = len(k_caches)
    kp = (ctypes.c_void_p * nl)(*[c.data_ptr() for c in k_caches])
    vp = (ctypes.c_void_p * nl)(*[c.data_ptr() for c in v_caches])
    block_bytes = k_caches[0][0].numel() * k_caches[0].element_size()
    rc = load_library().pkv_copy_blocks(kp, vp, nl, _ptr(src_dst_pairs),
                                        int(src_dst_pairs.numel() // 2), block_bytes, shape[0],
                                        _ptr(device_status), _stream(stream))
    _check(rc, "pkv_copy_blocks")


SWAP_OUT, SWAP_IN = 0, 1


def swap_blocks(gpu_k: Sequence[torch.Tensor], gpu_v: Sequence[torch.Tensor],
                host_k: Sequence[torch.Tensor], host_v: Sequence[torch.Tensor],
                pairs: torch.Tensor, direction: int, *,
                device_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Moves whole blocks between every layer's GPU caches and pinned host
    pools: pairs (gpu block, host block), SWAP_OUT copies gpu -> host,
    SWAP_IN host -> gpu."""
    if not (len(gpu_k) == len(gpu_v) == len(host_k) == len(host_v)) or not gpu_k:
        raise ValueError("need one K and one V pool per layer on each side")
    _need_cuda(*gpu_k, *gpu_v, pairs, device_status)
    if pairs.dtype != torch.int64:
        raise ValueError("pairs must be int64")
    gshape, hshape = tuple(gpu_k[0].shape), tuple(host_k[0].shape)
    for c in list(gpu_k) + list(gpu_v):
        if tuple(c.shape) != gshape or c.dtype != gpu_k[0].dtype:
            raise ValueError("all GPU caches must share shape and dtype")
    for c in list(host_k) + list(host_v):
        if tuple(c.shape[1:]) != gshape[1:] or c.shape[0] != hshape[0] or c.dtype != gpu_k[0].dtype:
            raise ValueError("host pools must hold blocks of the GPU caches' shape and dtype")
        if c.is_cuda or not c.is_pinned():
            raise ValueError("host pools must be pinned CPU tensors")
    nl = len(gpu_k)
    arr = lambda cs: (ctypes.c_void_p * nl)(*[c.data_ptr() for c in cs])
    block_bytes = gpu_k[0][0].numel() * gpu_k[0].element_size()
    rc = load_library().pkv_swap_blocks(arr(gpu_k), arr(gpu_v), arr(host_k), arr(host_v), nl,
                                        _ptr(pairs), int(pairs.numel() // 2), block_bytes,
                                        gshape[0], hshape[0], int(direction),
                                        _ptr(device_status), _stream(stream))
    _check(rc, "pkv_swap_blocks")
