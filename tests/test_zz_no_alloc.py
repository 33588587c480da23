"""vcattn_prep_noalloc, the preprocessing entry point for callers that cannot
allocate device memory at call time (a plugin that only receives its input
and output tensors, or a program that forbids allocation after start-up).
It must produce exactly what vcattn_prep produces with a caller workspace,
call after call, although every call reuses the same library-owned scratch.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from bit_smoothed_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    assert torch.cuda.is_available()
    return vcattn


def _c_entry(vc):
    f = vc.lib().vcattn_prep_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(vc.Shape), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.POINTER(vc.PreppedStruct), ctypes.c_void_p]
    return f


def _same(a, b):
    for key, x in a.items():
        x = x.cpu().numpy()
        y = b[key].cpu().numpy()
        if x.dtype == np.float32:
            x, y = x.view(np.uint32), y.view(np.uint32)
        assert np.array_equal(x, y), key


def test_prep_noalloc_matches_prep_on_consecutive_calls(vc):
    f = _c_entry(vc)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # a large call, a smaller one (stale scratch from the first must not leak
    # in), then the first again
    for H, N, seed in ((4, 3000, 11), (3, 1777, 12), (4, 3000, 11)):
        Q, K, V = W.make_qkv(1, H, N, 8, seed, device="cuda")
        _, perm = vc.group(V, 8, 3)
        ref = vc.prep(Q, K, V, perm)
        out = vc.Prepped(tuple(Q.shape), Q.device)
        st = f(ctypes.byref(out.shape), ctypes.c_void_p(Q.data_ptr()), ctypes.c_void_p(K.data_ptr()),
               ctypes.c_void_p(V.data_ptr()), ctypes.c_void_p(perm.data_ptr()),
               ctypes.byref(out.struct), stream)
        assert st == 0
        torch.cuda.synchronize()
        _same(out.views(), ref.views())
    assert vc.last_device_error() == 0


def test_prep_noalloc_refuses_problems_beyond_its_scratch(vc):
    f = _c_entry(vc)
    big = vc.Shape(1, 64, 1 << 20, 128)      # needs 512 MiB of scratch
    fake = ctypes.c_void_p(1 << 20)          # never dereferenced: refused first
    pp = vc.PreppedStruct(*([1 << 20] * len(vc.PreppedStruct._fields_)))
    assert f(ctypes.byref(big), fake, fake, fake, None, ctypes.byref(pp), None) == 2
