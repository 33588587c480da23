"""The k-means assignment's tensor-core filter, measured on real inputs.

km_assign_tc computes an approximation T_c of every FP32 k-means score on the
tensor core and keeps only the clusters within a bound E of the largest T_c;
exact FP32 chains then decide among those.  The labels are exact provided
|T_c - score_c| <= E / 2 for every token and cluster (the bound proven in
tests/test_km_bound.py for any FP32 accumulation order and rounding).  These
tests read T_c and E out of the kernel (vcattn_test_km_scores) and compare
them with the oracle's FP32 chain scores, so the margin that the hardware
leaves is observed rather than assumed.
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


def _scores(vc, V, k, cent):
    B, H, N, _ = V.shape
    s = vc.Shape(B, H, N, 128)
    L = vc.lib()
    nb = L.vcattn_group_workspace_bytes(ctypes.byref(s), k)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    labels = torch.empty(B, H, N, dtype=torch.int32, device="cuda")
    T = torch.empty(B, H, N, 65, dtype=torch.float32, device="cuda")
    c = torch.from_numpy(np.ascontiguousarray(cent, np.float32)).cuda()
    f = L.vcattn_test_km_scores
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    st = f(ctypes.byref(s), P(V.data_ptr()), k, P(c.data_ptr()), P(labels.data_ptr()), P(T.data_ptr()),
           P(ws.data_ptr()), ctypes.c_size_t(nb), P(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    return labels.cpu().numpy(), T.cpu().numpy()


def _margin(orc, Vb_head, cent_head, T_head, k):
    s = orc.kmeans_scores(Vb_head, cent_head).astype(np.float64)      # FP32 chain scores
    Tc = T_head[:, :k].astype(np.float64)
    E = T_head[:, 64].astype(np.float64)
    assert np.all(E > 0) and np.all(np.isneginf(T_head[:, k:64]))
    return (np.abs(Tc - s) / E[:, None]).max(), s


def test_filter_margin_on_the_live_workload(vc, orc):
    """One head of the 32,626-token workload, centroids after two Lloyd
    iterations: every |T_c - score_c| stays below E / 2, and the step's
    labels are the FP32 argmax (lowest index on ties)."""
    w = W.WORKLOADS["live"]
    Q, K, V = W.make_workload(W.Workload("live_h1", 1, 1, w.N, w.k_lat, w.k, seed=w.seed), device="cuda")
    Vb = W.bf16_bits(V).reshape(1, w.N, 128)
    _, cent = orc.kmeans(Vb, w.k, 2)
    labels, T = _scores(vc, V, w.k, cent)
    ratio, s = _margin(orc, Vb[0], cent[0], T[0, 0], w.k)
    print("live head: max |T - score| / E = %.3e (exactness needs <= 0.5)" % ratio)
    assert ratio <= 0.5
    best = np.argmax(s == s.max(axis=1, keepdims=True), axis=1)
    assert np.array_equal(labels[0, 0], best)


def test_filter_margin_near_ties(vc, orc):
    """Centroid pairs one bf16 ulp apart and tokens copied from them (scores
    equal in all but the last bits): the margin still holds."""
    H, N, k = 1, 2048, 16
    g = torch.Generator(device="cpu").manual_seed(4242)
    V = (torch.randn(1, H, N, 128, generator=g) * 2.0).to(torch.bfloat16)
    bits = V.view(torch.int16)
    for c in range(1, k, 2):
        j0, j1 = (c - 1) * N // k, c * N // k
        bits[:, :, j1] = bits[:, :, j0]
        bits[:, :, j1, c % 128] += 1
        for r in range(1, 9):
            bits[:, :, j1 + r] = bits[:, :, j0 if r % 2 else j1]
    V = V.cuda()
    Vb = W.bf16_bits(V).reshape(1, N, 128)
    cent = np.stack([(Vb[0, (c * N) // k].astype(np.uint32) << 16).view(np.float32) for c in range(k)])[None]
    labels, T = _scores(vc, V, k, cent)
    ratio, s = _margin(orc, Vb[0], cent[0], T[0, 0], k)
    print("near ties: max |T - score| / E = %.3e" % ratio)
    assert ratio <= 0.5
    best = np.argmax(s == s.max(axis=1, keepdims=True), axis=1)
    assert np.array_equal(labels[0, 0], best)
