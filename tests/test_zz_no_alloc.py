"""pkv_paged_attention_decode_static: decode attention without any allocation.

This entry point exists for callers that cannot allocate device memory --
plugins whose host engine owns all device memory and gives them none, code
under an allocator that is full or must not grow, and latency-critical loops
that must not call cudaMalloc because it may synchronise the device.  When a
context spans several partitions it keeps the split-context partials in a
buffer inside the library instead of a caller workspace.

The test calls it through the C ABI twice in a row (on two different
batches, each at two partition sizes) and compares each result with the
allocating entry point pkv_paged_attention_decode and with the CPU oracle, at
the tolerance the other attention tests use.  It also checks that a large
batch whose contexts fit one partition runs (single pass, no buffer) and that
a split request beyond the buffer is refused.  It runs last so that a
failure here cannot hide other results.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.gpu_support import TOL, max_err, oracle_decode
from tests.util import small_case

pytestmark = pytest.mark.gpu


def _lib():
    import paged_kv_cache_311_gb300 as pkv
    L = pkv.load_library()
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    L.pkv_paged_attention_decode_static.argtypes = [vp, i32, vp, vp, vp, i32, vp, i32, vp, i32, i32,
                                                    i32, i32, i32, i64, i32, ctypes.c_float, i32,
                                                    vp, vp]
    L.pkv_paged_attention_decode_static.restype = i32
    L.pkv_static_workspace_capacity.argtypes = []
    L.pkv_static_workspace_capacity.restype = ctypes.c_size_t
    return L


def _device(case):
    d = {k: case[k].cuda() for k in ("q", "k_cache", "v_cache")}
    d["bt"] = torch.as_tensor(case["block_tables"], dtype=torch.int32).cuda()
    d["cl"] = torch.as_tensor(case["context_lens"], dtype=torch.int32).cuda()
    return d


def _static_call(L, case, d, out, status, P):
    B, H, D = d["q"].shape
    NB, Hk, bs, _ = d["k_cache"].shape
    vp = ctypes.c_void_p
    return L.pkv_paged_attention_decode_static(
        vp(out.data_ptr()), 0, vp(d["q"].data_ptr()), vp(d["k_cache"].data_ptr()),
        vp(d["v_cache"].data_ptr()), {"f32": 0, "f16": 1, "bf16": 2}[case["dtype"]],
        vp(d["bt"].data_ptr()), d["bt"].shape[1], vp(d["cl"].data_ptr()), B, H, Hk, D, bs, NB,
        int(max(case["context_lens"])), ctypes.c_float(case["scale"]), P, vp(status.data_ptr()),
        vp(torch.cuda.current_stream().cuda_stream))


def _allocating(case, d, P):
    import paged_kv_cache_311_gb300 as pkv
    out = torch.empty(d["q"].shape, dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(out, d["q"], d["k_cache"], d["v_cache"], d["bt"], d["cl"],
                               case["scale"], max_context_len=int(max(case["context_lens"])),
                               partition_size=P)
    return out


def test_static_workspace_matches_allocating_decode_and_oracle_twice():
    L = _lib()
    cases = [
        small_case(41, dtype="bf16", B=5, H=16, Hk=2, D=128, bs=16, lens=(1, 700, 513, 2000, 4097)),
        small_case(42, dtype="f16", B=3, H=8, Hk=8, D=64, bs=8, lens=(3000, 17, 1024)),
    ]
    for case in cases:                      # two calls in a row, different batches
        d = _device(case)
        ref, ost = oracle_decode(case)
        assert ost == 0
        for P in (512, 256):
            alloc = _allocating(case, d, P)
            out = torch.full_like(alloc, float("nan"))
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            rc = _static_call(L, case, d, out, st, P)
            assert rc == 0
            torch.cuda.synchronize()
            assert st.item() == 0
            assert torch.isfinite(out).all()
            got = out.double().cpu().numpy()
            assert max_err(got, alloc.double().cpu().numpy()) <= TOL[case["dtype"]]
            assert max_err(got, ref) <= TOL[case["dtype"]]


def test_single_partition_batch_needs_no_buffer():
    """2048 sequences x 64 heads whose contexts fit one partition: the split
    path's partials would take 2048 * 64 * (2 + 128) * 4 bytes (> 32 MiB), but
    the single pass uses none, so the call runs and matches the oracle."""
    L = _lib()
    B = 2048
    lens = tuple(int(x) for x in np.random.default_rng(5).integers(1, 65, B))
    case = small_case(44, dtype="bf16", B=B, H=64, Hk=8, D=128, bs=16, lens=lens)
    assert B * 64 * (2 + 128) * 4 > L.pkv_static_workspace_capacity()
    d = _device(case)
    out = torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _static_call(L, case, d, out, st, 512) == 0
    torch.cuda.synchronize()
    assert st.item() == 0
    ref, ost = oracle_decode(case)
    assert ost == 0 and max_err(out.double().cpu().numpy(), ref) <= TOL["bf16"]


def test_static_workspace_rejects_oversized_requests():
    L = _lib()
    cap = L.pkv_static_workspace_capacity()
    assert cap == 32 << 20
    case = small_case(43, dtype="bf16", B=2, H=8, Hk=1, D=128, bs=16, lens=(5, 9))
    d = _device(case)
    out = torch.empty(d["q"].shape, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B, H, D = d["q"].shape
    NB, Hk, bs, _ = d["k_cache"].shape
    vp = ctypes.c_void_p
    # 2 seqs x 8 heads x ceil(2**20 / 32) partitions x (2 + 128) x 4 bytes > 32 MiB
    rc = L.pkv_paged_attention_decode_static(
        vp(out.data_ptr()), 0, vp(d["q"].data_ptr()), vp(d["k_cache"].data_ptr()),
        vp(d["v_cache"].data_ptr()), 2, vp(d["bt"].data_ptr()), 1 << 16, vp(d["cl"].data_ptr()),
        B, H, Hk, D, bs, NB, 1 << 20, ctypes.c_float(0.1), 32, vp(st.data_ptr()), None)
    assert rc == -4
