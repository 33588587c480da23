"""The C-ABI library builds, loads and exports every symbol its headers declare;
host-side argument validation works without a GPU (no compute calls)."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    return vcattn.lib()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(vcattn_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert {"vcattn_group", "vcattn_prep", "vcattn_attn", "vcattn_fwd",
            "vcattn_last_device_error"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n


def _shape(B=1, H=2, N=1000, D=128):
    from bit_smoothed_attention_gb300.vcattn import Shape
    return Shape(B, H, N, D)


def test_status_strings(lib):
    for s in range(6):
        assert lib.vcattn_status_string(s)


def test_workspace_queries(lib):
    s = _shape()
    g = lib.vcattn_group_workspace_bytes(ctypes.byref(s), 8)
    p = lib.vcattn_prep_workspace_bytes(ctypes.byref(s))
    pb = lib.vcattn_prepped_bytes(ctypes.byref(s))
    f = lib.vcattn_fwd_workspace_bytes(ctypes.byref(s))
    assert g > 0 and p > 0 and pb > 0 and f >= pb + p
    assert lib.vcattn_group_workspace_bytes(ctypes.byref(s), 0) == 0
    assert lib.vcattn_group_workspace_bytes(ctypes.byref(s), 65) == 0
    bad = _shape(D=64)
    assert lib.vcattn_prepped_bytes(ctypes.byref(bad)) == 0
    big = _shape(N=4096)
    assert lib.vcattn_prepped_bytes(ctypes.byref(big)) > pb
    assert lib.vcattn_npad(1) == 128 and lib.vcattn_npad(128) == 128 and lib.vcattn_npad(129) == 256


def test_prepped_carve_layout(lib):
    from bit_smoothed_attention_gb300.vcattn import PreppedStruct
    s = _shape(N=777)
    nb = lib.vcattn_prepped_bytes(ctypes.byref(s))
    base = 1 << 20   # carving only computes addresses; nothing is touched
    out = PreppedStruct()
    assert lib.vcattn_prepped_carve(ctypes.byref(s), ctypes.c_void_p(base), nb, ctypes.byref(out)) == 0
    addrs = sorted((getattr(out, f), f) for f, _ in PreppedStruct._fields_)
    assert all(a % 256 == 0 for a, _ in addrs)
    assert addrs[0][0] == base and addrs[-1][0] < base + nb
    assert lib.vcattn_prepped_carve(ctypes.byref(s), ctypes.c_void_p(base), nb - 1,
                                    ctypes.byref(out)) == 1
    assert lib.vcattn_prepped_carve(ctypes.byref(s), ctypes.c_void_p(base + 8), nb,
                                    ctypes.byref(out)) == 1


def test_argument_validation_without_gpu(lib):
    """Invalid arguments are rejected before any CUDA call."""
    P = ctypes.c_void_p
    s = _shape()
    fake = P(1 << 20)
    # D != 128
    bad = _shape(D=64)
    assert lib.vcattn_group(ctypes.byref(bad), fake, 8, 5, fake, fake, None, fake, 1 << 30, None) == 2
    # k outside [1, 64]
    assert lib.vcattn_group(ctypes.byref(s), fake, 0, 5, fake, fake, None, fake, 1 << 30, None) == 2
    assert lib.vcattn_group(ctypes.byref(s), fake, 65, 5, fake, fake, None, fake, 1 << 30, None) == 2
    # null pointers, zero iterations, misalignment, short workspace
    assert lib.vcattn_group(ctypes.byref(s), None, 8, 5, fake, fake, None, fake, 1 << 30, None) == 1
    assert lib.vcattn_group(ctypes.byref(s), fake, 8, 0, fake, fake, None, fake, 1 << 30, None) == 1
    assert lib.vcattn_group(ctypes.byref(s), P((1 << 20) + 4), 8, 5, fake, fake, None, fake,
                            1 << 30, None) == 1
    assert lib.vcattn_group(ctypes.byref(s), fake, 8, 5, fake, fake, None, fake, 16, None) == 1
    # shape errors
    for B, H, N in ((0, 1, 10), (1, 0, 10), (1, 1, 0)):
        z = _shape(B, H, N)
        assert lib.vcattn_prepped_bytes(ctypes.byref(z)) == 0
    from bit_smoothed_attention_gb300.vcattn import PreppedStruct
    pp = PreppedStruct()
    assert lib.vcattn_prep(ctypes.byref(s), fake, fake, fake, None, ctypes.byref(pp), fake, 1 << 30,
                           None) == 1
    assert lib.vcattn_attn(ctypes.byref(s), ctypes.byref(pp), ctypes.c_float(0.1), None, fake, None,
                           None) == 1
    assert lib.vcattn_fwd(ctypes.byref(s), fake, fake, fake, None, ctypes.c_float(0.1), None, fake,
                          None, fake, 16, None) == 1


def test_fwd_host_validation_without_gpu(lib):
    """The host-pipeline entry point sizes two chunk slots and rejects bad
    arguments before any CUDA call."""
    P = ctypes.c_void_p
    s = _shape(B=2, H=5, N=1000)
    one = _shape(B=1, H=1, N=1000)
    w8 = lib.vcattn_fwd_host_workspace_bytes(ctypes.byref(s), 8, 0)    # default chunk: all 10 > 8 -> 8
    w2 = lib.vcattn_fwd_host_workspace_bytes(ctypes.byref(s), 8, 2)
    w1 = lib.vcattn_fwd_host_workspace_bytes(ctypes.byref(one), 8, 0)  # chunk clamps to B*H = 1
    assert w8 > w2 > 0 and w1 > 0
    assert lib.vcattn_fwd_host_workspace_bytes(ctypes.byref(s), 8, 20) == \
        lib.vcattn_fwd_host_workspace_bytes(ctypes.byref(s), 8, 10)
    # two slots of a one-head chunk hold at least Q, K, V and O of that head twice
    assert w1 >= 2 * 4 * 1000 * 128 * 2
    assert lib.vcattn_fwd_host_workspace_bytes(ctypes.byref(s), 0, 2) == 0
    assert lib.vcattn_fwd_host_workspace_bytes(ctypes.byref(s), 8, -1) == 0
    assert lib.vcattn_fwd_host_workspace_bytes(ctypes.byref(_shape(D=64)), 8, 2) == 0
    fake, ws = P(1 << 20), P(1 << 24)
    streams = (P * 4)(P(1), P(2), P(3), P(4))
    same = (P * 4)(P(1), P(2), P(3), P(3))
    shared = (P * 4)(P(1), P(2), P(1), P(4))

    def call(hQ=fake, k=8, iters=5, hO=fake, chunk=2, w=ws, nbytes=w2, st=streams, shape=s):
        return lib.vcattn_fwd_host(ctypes.byref(shape), hQ, fake, fake, k, iters, ctypes.c_float(0.1),
                                   None, hO, None, chunk, w, nbytes, st)
    assert call(hQ=None) == 1
    assert call(hO=None) == 1
    assert call(iters=0) == 1
    assert call(chunk=-1) == 1
    assert call(k=65) == 2
    assert call(shape=_shape(D=64)) == 2
    assert call(w=P((1 << 24) + 16)) == 1        # not 256-byte aligned
    assert call(nbytes=w2 - 1) == 1
    assert call(st=same) == 1
    assert call(st=shared) == 1
    assert call(st=None) == 1


def test_group_warm_validation_without_gpu(lib):
    P = ctypes.c_void_p
    s = _shape()
    fake = P(1 << 20)
    # the starting centroids are required and must be 16-byte aligned
    assert lib.vcattn_group_warm(ctypes.byref(s), fake, 8, 1, None, fake, fake, None, fake, 1 << 30,
                                 None) == 1
    assert lib.vcattn_group_warm(ctypes.byref(s), fake, 8, 1, P((1 << 20) + 4), fake, fake, None, fake,
                                 1 << 30, None) == 1
    assert lib.vcattn_group_warm(ctypes.byref(s), fake, 65, 1, fake, fake, fake, None, fake, 1 << 30,
                                 None) == 2


def test_strided_validation_without_gpu(lib):
    """The strided entry points need strides, and each stride must be a
    positive multiple of 8 elements."""
    from bit_smoothed_attention_gb300.vcattn import PreppedStruct, Strides
    P = ctypes.c_void_p
    s = _shape()
    fake = P(1 << 20)
    good = Strides(2 * 1000 * 128, 128, 2 * 128)
    for bad in (Strides(0, 128, 256), Strides(2 * 1000 * 128, 100, 256), Strides(-8, 128, 256)):
        assert lib.vcattn_group_strided(ctypes.byref(s), fake, ctypes.byref(bad), 8, 1, None, fake, fake,
                                        None, fake, 1 << 30, None) == 1
    assert lib.vcattn_group_strided(ctypes.byref(s), fake, None, 8, 1, None, fake, fake, None, fake,
                                    1 << 30, None) == 1
    pp = PreppedStruct()
    assert lib.vcattn_prep_strided(ctypes.byref(s), fake, ctypes.byref(good), fake, None, fake,
                                   ctypes.byref(good), None, ctypes.byref(pp), fake, 1 << 30, None) == 1
    assert lib.vcattn_attn_strided(ctypes.byref(s), ctypes.byref(pp), ctypes.c_float(0.1), 8,
                                   ctypes.c_float(6.0), 0, None, fake, None, None, None) == 1


def test_test_hooks_validation_without_gpu(lib):
    """The test hooks reject bad sizes and pointers before any CUDA call."""
    P = ctypes.c_void_p
    f = lib.vcattn_test_expcast
    f.restype = ctypes.c_int
    f.argtypes = [P, P, P, P, ctypes.c_int64, P]
    fake = P(1 << 20)
    assert f(fake, fake, fake, fake, 6, None) == 1           # not a multiple of 4
    assert f(fake, fake, fake, fake, -4, None) == 1
    assert f(fake, fake, fake, fake, 0, None) == 0           # nothing to do
    assert f(None, fake, fake, fake, 8, None) == 1
    assert f(P((1 << 20) + 4), fake, fake, fake, 8, None) == 1
    g = lib.vcattn_test_attn_stalled_after
    g.restype = ctypes.c_int
    from bit_smoothed_attention_gb300.vcattn import PreppedStruct
    pp = PreppedStruct()
    s = _shape()
    assert g(ctypes.byref(s), ctypes.byref(pp), ctypes.c_float(0.1), None, 0, fake, None, None) == 1
