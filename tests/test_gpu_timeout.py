"""Failure detection on the GPU without a fault: the attention kernel's
bounded waits.  With the K/V loader switched off (a test hook), no tile ever
arrives; every wait gives up after its 2 s limit, the kernel records a
timeout in the device error word and exits, and the CUDA context stays
usable for the next, normal call."""
import math

import numpy as np
import pytest
import torch

from bit_smoothed_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SM = float(np.float32(1 / math.sqrt(128)))


def test_stalled_loader_reports_timeout_and_context_survives():
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    Q, K, V = W.make_qkv(1, 1, 256, 4, 77, device="cuda")
    _, perm = vcattn.group(V, 4, 5)
    pp = vcattn.prep(Q, K, V, perm)
    torch.cuda.synchronize()
    assert vcattn.last_device_error() == vcattn.OK
    vcattn.test_attn_stalled(pp, SM)
    assert vcattn.last_device_error() == vcattn.ERR_TIMEOUT
    assert vcattn.last_device_error() == vcattn.OK          # read and cleared
    O, L = vcattn.attn(pp, SM)                               # the context still works
    torch.cuda.synchronize()
    assert vcattn.last_device_error() == vcattn.OK
    assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()


@pytest.mark.parametrize("masked", [False, True])
def test_loader_stopping_midway_drains_and_context_survives(masked):
    """The loader stops after two KV tiles, with copies and MMAs of every CTA
    already issued: the consumers give up after their 2 s limit, the kernel
    waits for what it issued before it releases TMEM and exits, records the
    timeout, and the next normal call gives the same output as before.  With
    a tile mask this is the block-sparse kernel, whose two loaders per CTA
    each walk their own slot's tiles through stages of their own."""
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    Q, K, V = W.make_qkv(1, 2, 2000, 4, 78, device="cuda")
    _, perm = vcattn.group(V, 4, 5)
    pp = vcattn.prep(Q, K, V, perm)
    mask = W.make_tile_mask(1, 2, 2000, 79, keep_frac=0.4).cuda() if masked else None
    O_ref, L_ref = vcattn.attn(pp, SM, mask=mask)
    torch.cuda.synchronize()
    assert vcattn.last_device_error() == vcattn.OK
    vcattn.test_attn_stalled_after(pp, SM, 2, mask=mask)
    assert vcattn.last_device_error() == vcattn.ERR_TIMEOUT
    O, L = vcattn.attn(pp, SM, mask=mask)
    torch.cuda.synchronize()
    assert vcattn.last_device_error() == vcattn.OK
    assert torch.equal(O, O_ref) and torch.equal(L, L_ref)
