"""The whole step (grouping, preprocessing, attention) captured into one CUDA
graph and replayed.

Every entry point enqueues only stream work (kernels, memsets, device-to-device
copies) on the caller's stream and never synchronises, so a caller can capture
a step once and replay it: the replay must give the eager results bit for bit,
also after new inputs are copied into the captured input buffers.
"""
import math

import numpy as np
import pytest
import torch

from bit_smoothed_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SM = float(np.float32(1 / math.sqrt(128)))


@pytest.fixture(scope="module")
def vc():
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return vcattn


def _eager(vc, Q, K, V, k, mask):
    labels, perm = vc.group(V, k, 5)
    pp = vc.prep(Q, K, V, perm)
    O, L = vc.attn(pp, SM, mask=mask)
    torch.cuda.synchronize()
    return labels.clone(), perm.clone(), O.clone(), L.clone()


@pytest.mark.parametrize("masked", [False, True])
def test_step_replays_from_a_cuda_graph(vc, masked):
    B, H, N, k = 1, 3, 1500, 8
    Q, K, V = W.make_qkv(B, H, N, k, 71, device="cuda")
    mask = W.make_tile_mask(B, H, N, 72, keep_frac=0.4).cuda() if masked else None
    ref = _eager(vc, Q, K, V, k, mask)

    # warm up on a side stream (first-call set-up happens outside the capture)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _eager(vc, Q, K, V, k, mask)
    torch.cuda.current_stream().wait_stream(side)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        labels, perm = vc.group(V, k, 5)
        pp = vc.prep(Q, K, V, perm)
        O, L = vc.attn(pp, SM, mask=mask)
    g.replay()
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    for got, want in zip((labels, perm, O, L), ref):
        assert torch.equal(got, want)

    # new inputs in the captured buffers: the replay follows them
    Q2, K2, V2 = W.make_qkv(B, H, N, k, 73, device="cuda")
    ref2 = _eager(vc, Q2, K2, V2, k, mask)
    Q.copy_(Q2)
    K.copy_(K2)
    V.copy_(V2)
    g.replay()
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    for got, want in zip((labels, perm, O, L), ref2):
        assert torch.equal(got, want)
