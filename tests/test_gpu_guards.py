"""Guard bands around every buffer the library writes (a memory checker is
not available here, so out-of-bounds writes are caught this way): each
output and workspace is placed between two 4 KiB bands of a known byte
pattern, the whole path runs through the C ABI (grouping, preprocessing,
attention), and afterwards every band must be intact and the device error
word clear.  Covered: ragged and tiny sequence lengths, one head of the
32,626-token live shape, dense and block-sparse attention, bf16 and f32
output, contiguous and (B, N, H, D)-strided output, and the preprocessing
entry point without a caller workspace."""
import ctypes
import math

import numpy as np
import pytest
import torch

from bit_smoothed_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096
PATTERN = 0xA5
SM = float(np.float32(1 / math.sqrt(128)))


@pytest.fixture(scope="module")
def vc():
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    assert torch.cuda.is_available()
    return vcattn


class Guarded:
    """`nbytes` of device memory between two bands of PATTERN bytes."""

    def __init__(self, nbytes, name):
        self.n = int(nbytes)
        self.name = name
        self.buf = torch.full((GUARD + ((self.n + 255) // 256) * 256 + GUARD,), PATTERN, dtype=torch.uint8,
                              device="cuda")

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr() + GUARD)

    def tensor(self, dtype, shape):
        esz = torch.empty((), dtype=dtype).element_size()
        return self.buf[GUARD:GUARD + self.n].view(dtype).view(*shape)

    def check(self):
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.n:]          # includes the rounding slack
        bad_h = int((head != PATTERN).sum())
        bad_t = int((tail != PATTERN).sum())
        assert bad_h == 0 and bad_t == 0, "%s: %d bytes before and %d after the buffer were written" % (
            self.name, bad_h, bad_t)


def _run_guarded(vc, B, H, N, k, seed, masked, o_layout, out_f32):
    L = vc.lib()
    Q, K, V = W.make_qkv(B, H, N, k, seed, device="cuda")
    shape = vc.Shape(B, H, N, 128)
    s = ctypes.byref(shape)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    guards = []

    def g(nbytes, name):
        x = Guarded(nbytes, name)
        guards.append(x)
        return x

    labels = g(B * H * N * 4, "labels")
    perm = g(B * H * N * 4, "perm")
    cent = g(B * H * k * 128 * 4, "centroids")
    gws_n = L.vcattn_group_workspace_bytes(s, k)
    gws = g(gws_n, "group workspace")
    assert L.vcattn_group(s, P(V), k, 5, labels.ptr, perm.ptr, cent.ptr, gws.ptr, gws_n, stream) == 0

    pb = L.vcattn_prepped_bytes(s)
    prepped = g(pb, "prepped")
    pp = vc.PreppedStruct()
    assert L.vcattn_prepped_carve(s, prepped.ptr, pb, ctypes.byref(pp)) == 0
    pws_n = L.vcattn_prep_workspace_bytes(s)
    pws = g(pws_n, "prep workspace")
    assert L.vcattn_prep(s, P(Q), P(K), P(V), perm.ptr, ctypes.byref(pp), pws.ptr, pws_n, stream) == 0

    mask = W.make_tile_mask(B, H, N, seed + 1, keep_frac=0.3).cuda() if masked else None
    esz = 4 if out_f32 else 2
    O = g(B * H * N * 128 * esz, "O")
    lse = g(B * H * N * 4, "lse2")
    mptr = None if mask is None else P(mask)
    if o_layout == "bnhd":
        st = vc.Strides(N * H * 128, 128, H * 128)
        assert L.vcattn_attn_strided(s, ctypes.byref(pp), ctypes.c_float(SM), 8, ctypes.c_float(6.0),
                                     int(out_f32), mptr, O.ptr, ctypes.byref(st), lse.ptr, stream) == 0
    else:
        assert L.vcattn_attn_ex(s, ctypes.byref(pp), ctypes.c_float(SM), 8, ctypes.c_float(6.0), int(out_f32),
                                mptr, O.ptr, lse.ptr, stream) == 0

    # the preprocessing without a caller workspace, into a second guarded buffer
    prepped2 = g(pb, "prepped (no-alloc entry)")
    pp2 = vc.PreppedStruct()
    assert L.vcattn_prepped_carve(s, prepped2.ptr, pb, ctypes.byref(pp2)) == 0
    f = L.vcattn_prep_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(vc.Shape), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.POINTER(vc.PreppedStruct), ctypes.c_void_p]
    assert f(s, P(Q), P(K), P(V), perm.ptr, ctypes.byref(pp2), stream) == 0

    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    for x in guards:
        x.check()
    # the guarded run computed what the ordinary calls compute
    lab_ref, perm_ref = vc.group(V, k, 5)
    assert torch.equal(perm.tensor(torch.int32, (B, H, N)), perm_ref)
    assert torch.equal(prepped.buf[GUARD:GUARD + pb], prepped2.buf[GUARD:GUARD + pb])
    ppr = vc.prep(Q, K, V, perm_ref)
    Or, Lr = vc.attn(ppr, SM, mask=mask, out_f32=out_f32)
    dt = torch.float32 if out_f32 else torch.bfloat16
    if o_layout == "bnhd":
        Og = O.tensor(dt, (B, N, H, 128)).transpose(1, 2)
    else:
        Og = O.tensor(dt, (B, H, N, 128))
    torch.cuda.synchronize()
    assert torch.equal(Og, Or)
    assert torch.equal(lse.tensor(torch.float32, (B, H, N)), Lr)


@pytest.mark.parametrize("N", [1, 63, 65, 127, 129, 777])
@pytest.mark.parametrize("masked,o_layout,out_f32", [(False, "bhnd", False), (True, "bhnd", True),
                                                     (False, "bnhd", True), (True, "bnhd", False)])
def test_guard_bands_small(vc, N, masked, o_layout, out_f32):
    _run_guarded(vc, 1, 2, N, 8, 1300 + N, masked, o_layout, out_f32)


@pytest.mark.parametrize("masked,o_layout", [(False, "bhnd"), (True, "bnhd")])
def test_guard_bands_live_head(vc, masked, o_layout):
    """One head of the live shape (N = 32626: a partial last block and tile)."""
    _run_guarded(vc, 1, 1, 32626, 64, 1400, masked, o_layout, False)
