"""ExpCast-FP8 byte for byte: the attention kernel's own cast (through the
vcattn_test_expcast hook, which runs the kernel's expcast4 and its handling
of excluded keys) against the oracle's definition of the byte
(code = rint(fmaf(x, A, B)), ties to even; codes below 8 flush to 0; -inf
scores give 0).  "VC-Attention: Value Smoothing and Softmax Casting for
Low-bit Attention", Key Contribution 2: one FMA and one integer rounding
write the probability's E4M3 byte.

The kernel's form differs from the definition (a saturated FMA or a compare
for the flush, a magic-number add for the rounding), so every boundary of
the definition is swept: every half-integer t in [7.5, 126.5] and the two
floats on each side, the flush edge at 7.5, the largest t the kernel can
produce (C + tau8 at the library's default off = 8, tau8 = 6), the dropped
blocks (A = B = 0) and the excluded keys (-inf), and ten million random
(x, A, B) in the ranges the attention produces.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vc():
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    assert torch.cuda.is_available()
    return vcattn


def _gpu_codes(vc, x, A, B):
    """x [4m] f32, A and B [m] f32 (one per four scores) -> GPU bytes [4m]."""
    xt, At, Bt = (torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda() for a in (x, A, B))
    codes = vc.test_expcast(xt, At, Bt)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    return codes.cpu().numpy()


def _compare(vc, orc, x, A, B):
    g = _gpu_codes(vc, x, A, B)
    r = orc.expcast_v(x, np.repeat(A, 4), np.repeat(B, 4))
    bad = np.nonzero(g != r)[0]
    assert bad.size == 0, "%d byte mismatches, first at x=%r A=%r B=%r: gpu %d oracle %d" % (
        bad.size, x[bad[0]], A[bad[0] // 4], B[bad[0] // 4], g[bad[0]], r[bad[0]])
    return r


def _pad4(x):
    n = (-x.size) % 4
    return np.concatenate([x, np.zeros(n, np.float32)]) if n else x


def _neighbours(t, k=2):
    """t and the k floats on each side of it (FP32)."""
    t = np.asarray(t, np.float32)
    out = [t]
    up, dn = t.copy(), t.copy()
    for _ in range(k):
        up = np.nextafter(up, np.float32(np.inf))
        dn = np.nextafter(dn, np.float32(-np.inf))
        out += [up, dn]
    return np.concatenate(out).astype(np.float32)


def test_expcast_boundaries_bit_exact(vc, orc):
    """With A = 1 and an integer B the scores are t - B exactly, so t itself
    is swept: half-integers (the rounding ties), integers, the flush edge and
    the largest t the kernel reaches."""
    C = orc.expcast_C(8)
    t_max = np.float32(C + 6.0)                      # C + tau8 < 126.5
    halves = np.arange(7, 127, dtype=np.float32) + np.float32(0.5)
    ints = np.arange(-4, 127, dtype=np.float32)
    ts = np.concatenate([_neighbours(halves), _neighbours(ints), _neighbours([7.5, t_max, 8.0], 8)])
    ts = ts[ts <= np.float32(126.5)]
    for Bi in (0.0, -3.0, 17.0, 100.0):
        x = _pad4((ts - np.float32(Bi)).astype(np.float32))
        m = x.size // 4
        A = np.ones(m, np.float32)
        B = np.full(m, Bi, np.float32)
        assert np.array_equal(np.float32(x + np.float32(Bi)), np.float32(x) + np.float32(Bi))
        r = _compare(vc, orc, x, A, B)
        if Bi == 0.0:
            # the definition's edges, stated directly
            t = x
            assert np.all(r[t < np.float32(7.5)] == 0)
            assert np.all(r[(t >= np.float32(7.5)) & (t <= np.float32(126.5))] >= 8)
            assert r[np.argmax(t == np.float32(7.5))] == 8           # tie 7.5 -> 8 (even)
            assert r[np.argmax(t == np.float32(8.5))] == 8           # tie 8.5 -> 8 (even)
            assert r[np.argmax(t == np.float32(9.5))] == 10          # tie 9.5 -> 10
            assert r[np.argmax(t == np.float32(126.5))] == 126


def test_expcast_dropped_blocks_and_excluded_keys(vc, orc):
    """A dropped block is cast with A = B = 0 (every byte 0 for finite
    scores); a key past the end of the sequence has score -inf (byte 0)."""
    rng = np.random.default_rng(11)
    n = 1 << 20
    x = (rng.standard_normal(n) * 1e4).astype(np.float32)
    m = n // 4
    A = np.zeros(m, np.float32)
    B = np.zeros(m, np.float32)
    g = _compare(vc, orc, x, A, B)
    assert not g.any()
    A = rng.uniform(1e-4, 1e-2, m).astype(np.float32)
    zmax = (x.reshape(m, 4).astype(np.float64) * A[:, None]).max(axis=1)
    B = (np.float32(orc.expcast_C(8)) - (zmax - rng.uniform(0.0, 6.0, m))).astype(np.float32)
    x[rng.random(n) < 0.3] = -np.inf
    g = _compare(vc, orc, x, A, B)
    assert not g[np.isneginf(x)].any()


def test_expcast_random_scores_bit_exact(vc, orc):
    """Ten million scores in the ranges the attention produces: x is an FP32
    sum of E4M3 products (up to 448^2 * 128 in magnitude), A = c0 * q_scale *
    k_scale, and B = C - m with m at least the group's largest code minus
    tau8 (so t <= C + tau8, as in the kernel)."""
    rng = np.random.default_rng(2024)
    C = np.float32(orc.expcast_C(8))
    sm = np.float32(1 / math.sqrt(128))
    c0 = np.float32(8.0 * 1.4426950408889634 * float(sm))
    total = 0
    for chunk in range(5):
        m = 1 << 19                                        # groups of four
        qs = np.exp(rng.uniform(np.log(1e-3), np.log(0.2), m)).astype(np.float32)
        ks = np.exp(rng.uniform(np.log(1e-3), np.log(0.2), m)).astype(np.float32)
        A = ((c0 * qs).astype(np.float32) * ks).astype(np.float32)
        mag = np.exp(rng.uniform(np.log(10.0), np.log(448.0 * 448 * 128), m))
        x = (rng.uniform(-1.0, 1.0, (m, 4)) * mag[:, None]).astype(np.float32)
        # half of the scores on a coarse grid (exact sums of few products)
        grid = rng.random((m, 4)) < 0.5
        x[grid] = np.round(x[grid] * 64) / 64
        z = x.astype(np.float64) * A[:, None].astype(np.float64)
        zmax = z.max(axis=1)
        slack = rng.uniform(0.0, 6.0, m)                  # lazy threshold: m >= max - tau8
        mrun = (zmax - slack + rng.exponential(8.0, m) * (rng.random(m) < 0.5)).astype(np.float32)
        B = (C - mrun).astype(np.float32)
        _compare(vc, orc, x.ravel(), A, B)
        total += x.size
    assert total >= 10_000_000


def test_expcast_hook_rejects_bad_sizes(vc):
    x = torch.zeros(6, dtype=torch.float32, device="cuda")
    A = torch.zeros(1, dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        vc.test_expcast(x, A, A)
