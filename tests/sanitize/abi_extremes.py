"""Scalar arguments at and past their limits through the host-side checks of
the GPU entry points.  Meant to run with no CUDA device visible (the caller
sets CUDA_VISIBLE_DEVICES to an empty string): a call that passes its checks
then stops at its first CUDA call with PKV_ECUDA, so the non-null pointers
below, which nothing may read, are never used.  Run by
tests/test_host_sanitizers.py against a build of the library whose host code
has UndefinedBehaviorSanitizer; a report aborts this process."""
import ctypes
import itertools
import sys

import torch

if torch.cuda.is_available():   # never with a device: the pointers below are not real
    sys.exit("a CUDA device is visible; refusing to run")

L = ctypes.CDLL(sys.argv[1])
vp, i32, i64, u64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
L.pkv_paged_attention_workspace_bytes.argtypes = [i32] * 5
L.pkv_paged_attention_workspace_bytes.restype = u64
L.pkv_paged_attention_decode.argtypes = [vp, i32, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32, i32,
                                         i32, i64, i32, f32, i32, vp, u64, vp, vp]
L.pkv_paged_attention_decode_shared.argtypes = [vp, i32, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32,
                                                i32, i32, i64, i32, f32, vp, i32, i32, i32, vp, u64,
                                                vp, vp]
L.pkv_paged_attention_decode_static.argtypes = [vp, i32, vp, vp, vp, i32, vp, i32, vp, i32, i32, i32,
                                                i32, i32, i64, i32, f32, i32, vp, vp]
L.pkv_reshape_and_cache.argtypes = [vp, vp, vp, vp, i32, vp, i32, i32, i32, i32, i64, vp, vp]

INTS = [-2**31, -1, 0, 1, 8, 16, 64, 128, 65535, 65536, 2**31 - 16, 2**31 - 1]
I64S = [-2**63, -1, 0, 1, 1 << 20, 2**31 - 1, 2**31, 2**63 - 1]
P = 16 * 1024   # non-null and 16-byte aligned

n = 0
for a in itertools.product(INTS, repeat=5):
    L.pkv_paged_attention_workspace_bytes(*a)
    n += 1
for mb, B, H, Hk, D, bs, mcl, part in itertools.product(
        [1, 8, 65535, 2**31 - 1], [0, 1, 65535, 65536, 2**31 - 1], [1, 8, 2**31 - 1], [1, 8, 65536],
        [64, 128, 2**31 - 1], [8, 32, 2**31 - 1], [0, 1, 2**31 - 1], [0, 32, 2**31 - 32]):
    for nb in (1, 2**31 - 1):
        L.pkv_paged_attention_decode(P, 0, P, P, P, 2, P, mb, P, B, H, Hk, D, bs, nb, mcl, 1.0, part,
                                     P, 2**62, P, None)
        L.pkv_paged_attention_decode_static(P, 0, P, P, P, 2, P, mb, P, B, H, Hk, D, bs, nb, mcl, 1.0,
                                            part, P, None)
        for slots in (1, 2**31 - 1):
            L.pkv_paged_attention_decode_shared(P, 0, P, P, P, 2, P, mb, P, B, H, Hk, D, bs, nb, mcl,
                                                1.0, P, 1, 1, slots, P, 2**62, P, None)
        n += 4
for T, Hk, D, bs in itertools.product([0, 1, 2**31 - 1], [1, 2**31 - 1], [1, 8, 2**29, 2**31 - 1],
                                      [1, 2**31 - 1]):
    for nb in I64S:
        L.pkv_reshape_and_cache(P, P, P, P, 2, P, T, Hk, D, bs, nb, P, None)
        n += 1
print("calls", n)
