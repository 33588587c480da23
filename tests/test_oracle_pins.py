"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a library
routine (torch float8 conversion, numpy stable argsort, torch SDPA), a closed
form (the ExpCast round trip and Proposition 3.1's bound), an invariant
(centring, joint permutation, rank-one restoration) or brute force on tiny
inputs.  None of these needs a GPU.
"""
import math
import os

import numpy as np
import pytest
import torch

from bit_smoothed_attention_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")
CSTAR = (math.log2(1.5) - 0.5) / 2
# the oracle takes sm_scale as FP32; references use the same rounded value
SM = float(np.float32(1 / math.sqrt(128)))


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLD, name)):
        line = line.split("#")[0].strip()
        if "=" in line:
            k, v = line.split("=")
            vals[k.strip()] = float(v)
        elif line:
            a, b = line.split()
            vals[int(a, 16)] = float(b)
    return vals


# ----------------------------------------------------------------- E4M3 codec
def test_e4m3_decode_matches_torch_all_bytes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_e4m3_format_golden(orc):
    for code, val in _golden("e4m3fn_format.txt").items():
        got = orc.e4m3_decode(np.array([code], np.uint8))[0]
        assert got == val and np.signbit(got) == np.signbit(val)


def _e4m3_probe_values():
    rng = np.random.default_rng(7)
    vals = [rng.uniform(-500, 500, 1_000_000).astype(np.float32),
            (np.sign(rng.standard_normal(1_000_000)) *
             np.exp2(rng.uniform(-12, 9.2, 1_000_000))).astype(np.float32)]
    # every finite E4M3 value, every midpoint (a tie) and its fp32 neighbours
    pos = np.unique(np.abs(torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
                           .float().numpy()))
    pos = pos[np.isfinite(pos)]
    mids = ((pos[1:].astype(np.float64) + pos[:-1]) / 2).astype(np.float32)
    for arr in (pos, mids, np.nextafter(mids, np.float32(np.inf)),
                np.nextafter(mids, np.float32(0))):
        vals += [arr, -arr]
    vals.append(np.array([448.0, 448.5, 463.9, 464.0, 465.0, 1e30, -1e30, 0.0, -0.0,
                          1e-30, -1e-30], np.float32))
    return np.concatenate(vals)


def test_e4m3_encode_matches_torch(orc):
    x = _e4m3_probe_values()
    ours = orc.e4m3_encode(x)
    ref = torch.from_numpy(x).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, (x[bad[:5]], ours[bad[:5]], ref[bad[:5]])


def test_e4m3_tie_detector(orc):
    pos = np.array([1.0, 1.125, 0.015625, 0.001953125, 256, 288], np.float32)
    mids = np.array([1.0625, 0.0009765625, 272.0, 0.0146484375], np.float32)
    assert not orc.e4m3_is_tie(pos).any()
    assert orc.e4m3_is_tie(mids).all()
    assert not orc.e4m3_is_tie(np.nextafter(mids, np.float32(0))).any()


def test_prep_counts_quantiser_ties(orc):
    """The preprocessing's tie count (R15): a Q block whose largest |q| is 448
    quantises with inv = 1, so q = 1.0625 (halfway between the E4M3 values 1
    and 1.125) is a tie and 448, 1.0 and 0 are not; a constant K centres to
    zero and a constant V leaves a zero residual (no quantiser input at all)."""
    N = 64
    q = np.zeros((1, N, 128), np.float32)
    q[0, 0, 0] = 448.0
    q[0, 1:11, 3] = 1.0625
    q[0, 11:20, 5] = 1.0
    k = np.full((1, N, 128), 0.75, np.float32)
    v = np.full((1, N, 128), -2.5, np.float32)
    bits = [W.bf16_bits(torch.from_numpy(t).to(torch.bfloat16)) for t in (q, k, v)]
    out = orc.prep(*bits, count_ties=True)
    assert out["ties"].tolist() == [[10, 0, 0]]
    plain = orc.prep(*bits)
    for key in plain:
        assert np.array_equal(plain[key], out[key]), key


# ------------------------------------------------------------------- ExpCast
@pytest.mark.parametrize("off", [0, 8])
def test_expcast_round_trip_identity(orc, off):
    """For every normal E4M3 value v, ExpCast of its exact log2-domain score
    returns v's own byte (the affine-log construction of the byte)."""
    C = orc.expcast_C(off)
    codes = np.arange(8, 127, dtype=np.uint8)
    v = orc.e4m3_decode(codes)
    y = np.log2(v) - off                      # log2 of the probability
    x = (8.0 * y).astype(np.float32)          # score in code units, m = 0
    out = orc.expcast(x, 1.0, C)
    ok = codes <= 56 + 8 * off                # p <= 1 (the max-subtracted domain)
    assert np.array_equal(out[ok], codes[ok])


@pytest.mark.parametrize("off", [0, 8])
def test_expcast_max_maps_to_power_of_two(orc, off):
    C = orc.expcast_C(off)
    assert orc.expcast(np.zeros(1, np.float32), 1.0, C)[0] == 56 + 8 * off
    v = orc.e4m3_decode(np.array([56 + 8 * off], np.uint8))[0]
    assert v == 2.0 ** off


def test_expcast_log_ratio_bound(orc):
    """|log2(decoded / exact)| <= 1/16 + c*, attained up to the sweep step."""
    off = 8
    C = orc.expcast_C(off)
    y = np.linspace(-13.9, 0.0, 2_000_001)       # log2 p over the normal range
    x = (8.0 * y).astype(np.float32)
    codes = orc.expcast(x, 1.0, C)
    assert (codes >= 8).all()
    dec = orc.e4m3_decode(codes) / 2.0 ** off
    err = np.log2(dec) - x.astype(np.float64) / 8.0
    bound = 1.0 / 16 + CSTAR
    assert np.abs(err).max() <= bound + 1e-6
    assert np.abs(err).max() >= bound - 1e-4


def test_expcast_underflow_and_clip(orc):
    C = orc.expcast_C(8)
    x = np.array([-1e30, -np.inf, -200.0, -113.0, 50.0, 1e30], np.float32)
    out = orc.expcast(x, 1.0, C)
    assert list(out[:3]) == [0, 0, 0]
    assert out[3] == 0                   # t = 6.66 -> k = 7 -> underflow to 0
    assert out[4] == 126 and out[5] == 126


def test_expcast_half_integers_round_to_even(orc):
    """The integer conversion of ExpCast rounds half to even (the default
    rounding of a float-to-integer conversion): every half-integer t in
    [7.5, 126.5] gives numpy's round-half-even of t, then the flush below 8
    and the clip at 126."""
    t = np.arange(7, 127, dtype=np.float32) + np.float32(0.5)   # exact in FP32
    out = orc.expcast(t, 1.0, 0.0)                                # fmaf(t, 1, 0) = t
    k = np.rint(t.astype(np.float64))                             # half to even
    want = np.where(k < 8, 0, np.minimum(k, 126)).astype(np.uint8)
    assert np.array_equal(out, want)


def _row_tv(orc, logits2, off=8):
    """Exact vs ExpCast distributions for one row of log2-domain scores."""
    C = orc.expcast_C(off)
    m = logits2.max()
    x = (8.0 * (logits2 - m)).astype(np.float32)
    codes = orc.expcast(x, 1.0, C)
    p = np.exp2(x.astype(np.float64) / 8.0)
    p /= p.sum()
    ph = orc.e4m3_decode(codes)
    ph /= ph.sum()
    tail = p[codes == 0].sum()
    return 0.5 * np.abs(p - ph).sum(), tail, p, ph


def test_prop31_row_tv_bound(orc):
    """Proposition 3.1 (VC-Attention, Key Contribution 4): row TV <= 3.64%
    plus the underflow tail."""
    g = _golden("prop31_expcast.txt")
    derived = math.tanh(math.log(2) * (1 / 16 + CSTAR) / 2)
    assert round(100 * derived, 2) == g["row_tv_bound_percent"]
    rng = np.random.default_rng(3)
    worst = 0.0
    for r in range(300):
        n = int(rng.integers(2, 4096))
        s = rng.standard_normal(n) * rng.uniform(0.2, 6.0)
        tv, tail, _, _ = _row_tv(orc, s)
        assert tv <= derived + tail + 1e-12
        worst = max(worst, tv - tail)
    assert worst > 0.005
    # An adversarial row reaches the bound: two groups of keys sitting where
    # the encoding error is most positive and most negative, carrying almost
    # all of the mass (the row max itself is encoded exactly).
    C = orc.expcast_C(8)
    y = np.linspace(-6, -1, 400001)
    x = (8.0 * y).astype(np.float32)
    err = np.log2(orc.e4m3_decode(orc.expcast(x, 1.0, C)) / 256.0) - x.astype(np.float64) / 8
    yp, ym = x[np.argmax(err)] / 8.0, x[np.argmin(err)] / 8.0
    best = 0.0
    n1 = 4000
    for n2 in range(int(n1 * 2 ** (yp - ym) * 0.8), int(n1 * 2 ** (yp - ym) * 1.25), 7):
        tv, tail, _, _ = _row_tv(orc, np.array([0.0] + [yp] * n1 + [ym] * n2))
        assert tail == 0
        best = max(best, tv)
    assert best > 0.0363 and best <= derived + 1e-12


def test_prop31_output_bound(orc):
    """||o - o_hat|| <= TV * diam(V) for the ExpCast row (same Proposition)."""
    rng = np.random.default_rng(4)
    for _ in range(50):
        n = int(rng.integers(2, 1000))
        s = rng.standard_normal(n) * 3
        tv, tail, p, ph = _row_tv(orc, s)
        V = rng.standard_normal((n, 16)) * rng.uniform(0.1, 10)
        diam = max(np.linalg.norm(V[i] - V[j]) for i in range(min(n, 60)) for j in range(n)) \
            if n <= 60 else None
        if diam is None:
            # diameter of a random cloud via all pairs on a subset plus extremes
            D2 = ((V[:, None, :] - V[None, :, :]) ** 2).sum(-1)
            diam = math.sqrt(D2.max())
        assert np.linalg.norm(p @ V - ph @ V) <= tv * diam + 1e-12


# ------------------------------------------------------------------ tree sum
def test_tree_sum_adjacent_pairing(orc):
    rng = np.random.default_rng(5)
    for n in (1, 2, 64, 512):
        x = rng.standard_normal(n).astype(np.float32) * 1e3
        s = orc.tree_sum(x)
        exact = math.fsum(x.astype(np.float64))
        assert abs(s - exact) <= (math.log2(n) + 1) * 2 ** -24 * np.abs(x).sum() + 1e-30
    # adjacent pairs that cancel exactly give exactly 0 only under adjacent pairing
    x = np.array([1e8, -1e8, 1.0, -1.0, 3.0, -3.0, 1e-3, -1e-3], np.float32)
    assert orc.tree_sum(x) == 0.0
    y = np.array([1e8, 1.0, -1e8, -1.0], np.float32)    # pairs (1e8+1), (-1e8-1)
    assert orc.tree_sum(y) == 0.0
    z = np.array([1e8, 1.0, 1.0, -1e8], np.float32)    # (1e8+1)=1e8, (1-1e8)=-1e8
    assert orc.tree_sum(z) == 0.0 and math.fsum(z) == 2.0


# -------------------------------------------------------------------- k-means
def _bits(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def test_kmeans_recovers_separated_clusters(orc):
    """Well-separated clusters laid out so that the evenly spaced seeds take
    one point of each: Lloyd's iterations recover the generating partition."""
    rng = np.random.default_rng(11)
    k, N = 6, 240
    cent = rng.standard_normal((k, 128)) * 10
    lab = np.repeat(np.arange(k), N // k)          # seed c falls in cluster c
    V = _bits(cent[lab] + rng.standard_normal((N, 128)) * 0.1)[None]
    labels, C = orc.kmeans(V, k, 4)
    assert np.array_equal(labels[0], lab)
    v = _f(V[0])
    for c in range(k):
        assert np.allclose(C[0, c], v[lab == c].mean(0), rtol=1e-6, atol=1e-6)


def test_kmeans_empty_cluster_keeps_centroid(orc):
    a = np.full((1, 128), -2.0, np.float32)
    b = np.full((1, 128), 3.0, np.float32)
    V = _bits(np.concatenate([a, b, b]))[None]     # seeds a, b, b
    labels, C = orc.kmeans(V, 3, 2)
    assert list(labels[0]) == [0, 1, 1]            # ties go to the lower cluster
    assert np.all(C[0, 2] == 3.0) and np.all(C[0, 1] == 3.0) and np.all(C[0, 0] == -2.0)


def test_kmeans_brute_force_invariants(orc):
    rng = np.random.default_rng(12)
    for trial in range(4):
        N, k = int(rng.integers(20, 256)), int(rng.integers(1, 9))
        V = _bits(rng.standard_normal((N, 128)) * 2 + rng.standard_normal((1, 128)))[None]
        v = _f(V[0])
        prev_obj = np.inf
        prev_labels, prev_C = None, None
        for iters in range(1, 6):
            labels, C = orc.kmeans(V, k, iters)
            labels, C = labels[0], C[0].astype(np.float64)
            if iters == 1:
                init = v[[(c * N) // k for c in range(k)]]
                # assign of iteration 1 is the brute-force argmin distance to init
                d2 = ((v[:, None, :] - init[None]) ** 2).sum(-1)
                best = d2.min(1)
                chosen = d2[np.arange(N), labels]
                assert np.all(chosen <= best + 1e-6 * (1 + best))
            else:
                # labels are the argmin distance to the previous centroids
                d2 = ((v[:, None, :] - prev_C[None]) ** 2).sum(-1)
                best = d2.min(1)
                chosen = d2[np.arange(N), labels]
                assert np.all(chosen <= best + 1e-6 * (1 + best))
            # centroids are the member means (empty clusters keep the old one)
            for c in range(k):
                m = labels == c
                if m.any():
                    assert np.allclose(C[c], v[m].mean(0), rtol=2e-6, atol=2e-6)
                elif prev_C is not None:
                    assert np.array_equal(C[c], prev_C[c])
            obj = ((v - C[labels]) ** 2).sum()
            assert obj <= prev_obj * (1 + 1e-9)
            prev_obj, prev_labels, prev_C = obj, labels, C


def test_kmeans_warm_start_continues_the_iterations(orc):
    """Starting from the centroids after n iterations and running m more is
    the same computation as n + m iterations from the usual seeds (labels
    and centroids bit for bit); a warm start from arbitrary centroids makes
    the first assign the brute-force nearest centroid."""
    rng = np.random.default_rng(14)
    V = _bits(rng.standard_normal((2, 300, 128)) * 2 + rng.standard_normal((2, 1, 128)))
    k = 7
    for n, m in ((1, 1), (2, 3), (4, 1)):
        _, Cn = orc.kmeans(V, k, n)
        lw, Cw = orc.kmeans(V, k, m, init=Cn)
        lc, Cc = orc.kmeans(V, k, n + m)
        assert np.array_equal(lw, lc) and np.array_equal(Cw, Cc)
    init = rng.standard_normal((2, k, 128)).astype(np.float32)
    lab, C = orc.kmeans(V, k, 1, init=init)
    for h in range(2):
        v = _f(V[h])
        d2 = ((v[:, None, :] - init[h][None].astype(np.float64)) ** 2).sum(-1)
        chosen = d2[np.arange(v.shape[0]), lab[h]]
        assert np.all(chosen <= d2.min(1) + 1e-6 * (1 + d2.min(1)))
        for c in range(k):
            mem = lab[h] == c
            if mem.any():
                assert np.allclose(C[h, c], v[mem].mean(0), rtol=2e-6, atol=2e-6)
            else:
                assert np.array_equal(C[h, c], init[h, c])


def test_kmeans_tie_goes_to_lowest_cluster(orc):
    # two identical points as the only data: both seeds equal, every score ties
    v = np.ones((2, 128), np.float32)
    labels, C = orc.kmeans(_bits(v)[None], 2, 1)
    assert list(labels[0]) == [0, 0]


def test_kmeans_scores_match_fp64(orc):
    rng = np.random.default_rng(13)
    V = _bits(rng.standard_normal((50, 128)))
    C = rng.standard_normal((7, 128)).astype(np.float32)
    s = orc.kmeans_scores(V, C).astype(np.float64)
    v = _f(V)
    ref = v @ C.T.astype(np.float64) - 0.5 * (C.astype(np.float64) ** 2).sum(1)
    assert np.allclose(s, ref, rtol=0, atol=1e-4)


# ----------------------------------------------------------------------- sort
def test_stable_sort_matches_numpy(orc):
    rng = np.random.default_rng(14)
    lab = rng.integers(0, 17, (3, 5000)).astype(np.int32)
    perm = orc.stable_sort(lab, 17)
    for h in range(3):
        assert np.array_equal(perm[h], np.argsort(lab[h], kind="stable"))
        assert np.array_equal(np.sort(perm[h]), np.arange(5000))
        assert np.all(np.diff(lab[h][perm[h]]) >= 0)


# ----------------------------------------------------------------------- prep
def _small_inputs(N=777, H=2, k_lat=8, seed=21):
    Q, K, V = W.make_qkv(1, H, N, k_lat, seed)
    return W.bf16_bits(Q)[0], W.bf16_bits(K)[0], W.bf16_bits(V)[0]


def test_prep_means_and_quantisers(orc):
    Q, K, V = _small_inputs()
    BH, N, _ = Q.shape
    labels, _ = orc.kmeans(V, 8, 3)
    perm = orc.stable_sort(labels, 8)
    pp = orc.prep(Q, K, V, perm)
    Np = orc.npad(N)
    nb = (N + 63) // 64
    for h in range(BH):
        q, k, v = _f(Q[h]), _f(K[h]), _f(V[h])
        # K mean: the FP32 tree mean of K
        assert np.allclose(pp["k_mean"][h], k.mean(0), rtol=1e-6, atol=1e-6)
        # Q bytes: within E4M3 rounding of q / scale; the block max maps to 448
        for b in range(nb):
            r0, r1 = 64 * b, min(64 * b + 64, N)
            s = pp["q_scale"][h, b]
            deq = orc.e4m3_decode(pp["q8"][h, r0:r1]) * s
            x = q[r0:r1]
            assert np.all(np.abs(deq - x) <= np.maximum(np.abs(x) * 2 ** -4, s * 2 ** -10) + 1e-12)
            assert np.abs(orc.e4m3_decode(pp["q8"][h, r0:r1])).max() == 448.0
        # centred, permuted K
        kc = k[perm[h]] - pp["k_mean"][h].astype(np.float64)
        for b in range(nb):
            r0, r1 = 64 * b, min(64 * b + 64, N)
            s = pp["k_scale"][h, b]
            deq = orc.e4m3_decode(pp["k8"][h, r0:r1]) * s
            assert np.all(np.abs(deq - kc[r0:r1]) <= np.maximum(np.abs(kc[r0:r1]) * 2 ** -4, s * 2 ** -10) + 1e-5 * s)
        # V: block means of the gathered V; residual within rounding; pad zero
        vg = v[perm[h]]
        for b in range(nb):
            r0, r1 = 64 * b, min(64 * b + 64, N)
            assert np.allclose(pp["v_mean"][h, b], vg[r0:r1].mean(0), rtol=1e-6, atol=1e-6)
        res = vg - pp["v_mean"][h][np.arange(N) // 64].astype(np.float64)
        deq = orc.e4m3_decode(pp["r8t"][h][:, :N]).T * pp["v_scale"][h].astype(np.float64)
        sv = pp["v_scale"][h].astype(np.float64)
        assert np.all(np.abs(deq - res) <= np.maximum(np.abs(res) * 2 ** -4, sv * 2 ** -10) + 1e-5 * sv)
        assert np.all(pp["q8"][h, N:] == 0) and np.all(pp["k8"][h, N:] == 0)
        assert np.all(pp["r8t"][h][:, N:] == 0)
        assert np.all(pp["q_scale"][h, nb:] == 1) and np.all(pp["v_mean"][h, nb:] == 0)
        # qmu = q . mu_K
        assert np.allclose(pp["qmu"][h], q @ pp["k_mean"][h].astype(np.float64), rtol=1e-5, atol=1e-4)


def test_prep_residual_block_means_vanish(orc):
    """After demeaning, each block's FP32 residual averages to ~0 (the
    'dequanted V's mean' effect of the smoothing)."""
    Q, K, V = _small_inputs(N=640)
    pp = orc.prep(Q, K, V, None)
    for h in range(Q.shape[0]):
        v = _f(V[h]).astype(np.float32)
        for b in range(10):
            r = (v[64 * b:64 * b + 64] - pp["v_mean"][h, b]).astype(np.float64)
            assert np.all(np.abs(r.mean(0)) <= 64 * 2 ** -23 * np.abs(v[64 * b:64 * b + 64]).max(0) + 1e-30)


def test_prep_zero_block_rule(orc):
    N = 130
    Q = np.zeros((1, N, 128), np.uint16)
    K = np.zeros((1, N, 128), np.uint16)
    V = _bits(np.full((N, 128), 3.0, np.float32))[None]
    pp = orc.prep(Q, K, V, None)
    assert np.all(pp["q8"] == 0) and np.all(pp["q_scale"] == 1)
    assert np.all(pp["k8"] == 0) and np.all(pp["k_scale"] == 1)
    assert np.all(pp["r8t"] == 0) and np.all(pp["v_scale"] == 1)
    assert np.all(pp["v_mean"][0, :3] == 3.0)


# ------------------------------------------------------------------ attention
def _deq(orc, pp, h, N):
    Np = orc.npad(N)
    q = orc.e4m3_decode(pp["q8"][h, :N]) * np.repeat(pp["q_scale"][h], 64)[:N, None]
    k = orc.e4m3_decode(pp["k8"][h, :N]) * np.repeat(pp["k_scale"][h], 64)[:N, None]
    v = orc.e4m3_decode(pp["r8t"][h][:, :N]).T * pp["v_scale"][h].astype(np.float64) \
        + pp["v_mean"][h][np.arange(N) // 64]
    return q, k, v


def _softmax_attn(q, k, v, sm, allowed=None):
    s = (q @ k.T) * sm
    if allowed is not None:
        s = np.where(allowed, s, -np.inf)
    m = s.max(1, keepdims=True)
    e = np.exp(s - np.where(np.isfinite(m), m, 0))
    l = e.sum(1, keepdims=True)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(l > 0, (e @ v) / l, 0.0)
        lse2 = np.where(l[:, 0] > 0, (m[:, 0] + np.log(l[:, 0])) / math.log(2), -np.inf)
    return o, lse2


@pytest.mark.parametrize("N", [1, 63, 129, 777])
def test_emul_exact_exp_equals_softmax_of_dequantised(orc, N):
    """With ExpCast replaced by the exact exponential, the tiled online
    recurrence (rescaling, partial tiles, rank-one mean restoration) equals
    plain softmax attention on the dequantised tensors."""
    Q, K, V = _small_inputs(N=N, H=1, seed=30 + N)
    labels, _ = orc.kmeans(V, 4, 2)
    perm = orc.stable_sort(labels, 4)
    pp = orc.prep(Q, K, V, perm)
    sm = SM
    O1, L1 = orc.attn_emul(pp, 0, N, sm, flags=1)
    O3, L3 = orc.attn_emul(pp, 0, N, sm, flags=3)
    q, k, v = _deq(orc, pp, 0, N)
    o, lse2 = _softmax_attn(q, k, v, sm)
    assert np.allclose(O1, o, rtol=1e-10, atol=1e-10)
    assert np.allclose(O3, O1, rtol=1e-11, atol=1e-12)
    lq = L1 - pp["qmu"][0].astype(np.float64) * sm / math.log(2)
    assert np.allclose(lq, lse2, rtol=0, atol=1e-9)


def test_single_block_is_global_v_centring(orc):
    """With one 64-token block over the whole sequence the block mean is the
    sequence mean of V, and the restoration reduces to plain V centring: the
    output equals attention on the centred (residual) values plus the mean,
    since every softmax row sums to 1."""
    N = 50
    Q, K, V = _small_inputs(N=N, H=1, seed=55)
    pp = orc.prep(Q, K, V, None)
    mu = pp["v_mean"][0][0].astype(np.float64)
    v64 = torch.from_numpy(V[0].view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.allclose(mu, v64.mean(0), rtol=1e-6, atol=1e-6)
    O1, _ = orc.attn_emul(pp, 0, N, SM, flags=1)
    q, k, _ = _deq(orc, pp, 0, N)
    resid = orc.e4m3_decode(pp["r8t"][0][:, :N]).T * pp["v_scale"][0].astype(np.float64)
    o_res, _ = _softmax_attn(q, k, resid, SM)
    assert np.allclose(O1, o_res + mu[None, :], rtol=1e-10, atol=1e-10)
    # the centred values carry (almost) no mean: what is left is E4M3 rounding
    assert np.abs(resid.mean(0)).max() <= 0.02 * np.abs(v64).max()


def test_emul_mask_and_empty_rows(orc):
    N = 300
    Q, K, V = _small_inputs(N=N, H=1, seed=40)
    pp = orc.prep(Q, K, V, None)
    sm = SM
    nq, nbp = (N + 63) // 64, orc.npad(N) // 64
    rng = np.random.default_rng(41)
    mask = (rng.random((nq, nbp)) < 0.4).astype(np.uint8)
    mask[2, :] = 0                       # an empty selection
    O, L = orc.attn_emul(pp, 0, N, sm, mask=mask, flags=1)
    q, k, v = _deq(orc, pp, 0, N)
    allowed = mask[np.arange(N) // 64][:, np.arange(N) // 64].astype(bool)
    o, lse2 = _softmax_attn(q, k, v, sm, allowed)
    assert np.allclose(O, o, rtol=1e-10, atol=1e-10)
    assert np.all(O[128:192] == 0) and np.all(np.isneginf(L[128:192]))
    lq = L - pp["qmu"][0] * sm / math.log(2)
    fin = np.isfinite(lse2)
    assert np.allclose(lq[fin], lse2[fin], atol=1e-9)


def _cut_down(pp, qt, steps, N):
    """The prepped tensors of one head cut down to query tile qt and the KV
    blocks of `steps`, laid out two per 128-key tile in step order (a step of
    one block takes the first half of the last tile).  Only the last block of
    the sequence may be partial, and only as the last block of the cut."""
    blocks = [b for st in steps for b in st]
    nkeys = [min(64, N - 64 * b) for b in blocks]
    assert all(n == 64 for n in nkeys[:-1])
    Nc = 64 * (len(blocks) - 1) + nkeys[-1]
    Npc = ((Nc + 127) // 128) * 128
    nbc = Npc // 64
    rows = np.arange(64 * qt, min(64 * qt + 64, N))
    cut = {"q8": np.zeros((1, Npc, 128), np.uint8), "k8": np.zeros((1, Npc, 128), np.uint8),
           "r8t": np.zeros((1, 128, Npc), np.uint8), "q_scale": np.ones((1, nbc), np.float32),
           "k_scale": np.ones((1, nbc), np.float32), "v_scale": pp["v_scale"].copy(),
           "k_mean": pp["k_mean"].copy(), "v_mean": np.zeros((1, nbc, 128), np.float32),
           "qmu": np.zeros((1, max(Nc, 64)), np.float32)}
    cut["q8"][0, :rows.size] = pp["q8"][0, rows]
    cut["q_scale"][0, 0] = pp["q_scale"][0, qt]
    cut["qmu"][0, :rows.size] = pp["qmu"][0, rows]
    for c, b in enumerate(blocks):
        n = nkeys[c]
        cut["k8"][0, 64 * c:64 * c + n] = pp["k8"][0, 64 * b:64 * b + n]
        cut["r8t"][0, :, 64 * c:64 * c + n] = pp["r8t"][0, :, 64 * b:64 * b + n]
        cut["k_scale"][0, c] = pp["k_scale"][0, b]
        cut["v_mean"][0, c] = pp["v_mean"][0, b]
    return cut, Nc, rows


@pytest.mark.parametrize("tau8", [0.0, 6.0])
def test_emul_mask_steps_are_the_query_tiles_own_blocks(orc, tau8):
    """With a 64x64 tile mask, a row's KV steps are the blocks its own query
    tile keeps, in ascending order, two per step; only the last step of an
    odd count has one block ("[perf] Add opt-in SM120 sparse attention
    forward kernel for MiniMax-H3", Changes: the kept KV tiles of each query
    tile are visited).  The expected steps of each case are written out
    below, and the masked rows must equal the unmasked emulation of a
    problem cut down to those steps' blocks, two per 128-key step.  A
    different pairing of the same blocks gives different bytes, so the
    comparison decides the steps; the masks of other query tiles do not
    matter; a mask that keeps everything is no mask."""
    N = 1000                                      # 16 blocks, the last has 40 keys
    Q, K, V = _small_inputs(N=N, H=1, seed=60)
    labels, _ = orc.kmeans(V, 4, 2)
    perm = orc.stable_sort(labels, 4)
    pp = orc.prep(Q, K, V, perm)
    nq, nbp = (N + 63) // 64, orc.npad(N) // 64
    rng = np.random.default_rng(61)
    mask = (rng.random((nq, nbp)) < 0.3).astype(np.uint8)
    # query tile: (blocks it keeps, its KV steps written out by hand)
    cases = {
        3: ([1, 3, 4], [(1, 3), (4,)]),
        4: ([0, 1, 2, 3], [(0, 1), (2, 3)]),
        8: ([9], [(9,)]),
        10: ([2, 7, 11, 15], [(2, 7), (11, 15)]),
        11: ([2, 3, 7, 8, 15], [(2, 3), (7, 8), (15,)]),
        15: ([0, 5, 6, 12, 13, 14], [(0, 5), (6, 12), (13, 14)]),
    }
    for qt, (blocks, _) in cases.items():
        mask[qt, :] = 0
        mask[qt, blocks] = 1
    O, L = orc.attn_emul(pp, 0, N, SM, tau8=tau8, mask=mask)
    for qt, (blocks, steps) in cases.items():
        assert [b for st in steps for b in st] == blocks
        cut, Nc, rows = _cut_down(pp, qt, steps, N)
        Oc, Lc = orc.attn_emul(cut, 0, Nc, SM, tau8=tau8, qidx=np.arange(rows.size))
        assert np.array_equal(O[rows], Oc) and np.array_equal(L[rows], Lc), qt
    # another pairing of the same blocks changes the output of tile 10
    cut, Nc, rows = _cut_down(pp, 10, [(2, 11), (7, 15)], N)
    assert not np.array_equal(O[rows], orc.attn_emul(cut, 0, Nc, SM, tau8=tau8, qidx=np.arange(rows.size))[0])
    # what the other query tiles keep does not matter
    m2 = 1 - mask
    for qt, (blocks, _) in cases.items():
        m2[qt] = mask[qt]
    O2, L2 = orc.attn_emul(pp, 0, N, SM, tau8=tau8, mask=m2)
    for qt in cases:
        r = np.arange(64 * qt, min(64 * qt + 64, N))
        assert np.array_equal(O2[r], O[r]) and np.array_equal(L2[r], L[r])
    Of, Lf = orc.attn_emul(pp, 0, N, SM, tau8=tau8, mask=np.ones((nq, nbp), np.uint8))
    Od, Ld = orc.attn_emul(pp, 0, N, SM, tau8=tau8)
    assert np.array_equal(Of, Od) and np.array_equal(Lf, Ld)


def test_emul_expcast_within_prop31(orc):
    """With ExpCast on, every row stays within (3.6368% + tail) * diam(V) of
    the exact-exponential row (Proposition 3.1's output bound)."""
    N = 900
    Q, K, V = _small_inputs(N=N, H=1, seed=50)
    pp = orc.prep(Q, K, V, None)
    sm = SM
    Oe, _ = orc.attn_emul(pp, 0, N, sm, flags=1)
    Oc, _ = orc.attn_emul(pp, 0, N, sm, flags=0)
    q, k, v = _deq(orc, pp, 0, N)
    s = (q @ k.T) * sm
    p = np.exp(s - s.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    tail = np.where(p / p.max(1, keepdims=True) < 2.0 ** -13.5, p, 0).sum(1)
    D2 = ((v[:, None, :] - v[None, :, :]) ** 2).sum(-1)
    diam = math.sqrt(D2.max())
    bound = math.tanh(math.log(2) * (1 / 16 + CSTAR) / 2)
    err = np.linalg.norm(Oc - Oe, axis=1)
    assert np.all(err <= (bound + tail) * diam + 1e-9)
    assert err.max() > 0


def test_emul_lazy_rescale_threshold_is_consistent(orc):
    """A lazy running max (threshold tau) changes only the reference of the
    codes; the normalised output stays within the ExpCast bound."""
    N = 600
    Q, K, V = _small_inputs(N=N, H=1, seed=60)
    pp = orc.prep(Q, K, V, None)
    sm = SM
    O0, L0 = orc.attn_emul(pp, 0, N, sm, tau8=0.0, flags=1)
    O6, L6 = orc.attn_emul(pp, 0, N, sm, tau8=6.0, flags=1)
    assert np.allclose(O0, O6, rtol=1e-10, atol=1e-10)
    assert np.allclose(L0, L6, atol=1e-9)


def test_dense_matches_torch_sdpa(orc):
    N = 333
    Q, K, V = _small_inputs(N=N, H=1, seed=70)
    sm = SM
    O, L = orc.attn_dense(Q[0], K[0], V[0], sm)
    q, k, v = (torch.from_numpy(_f(x[0]))[None, None] for x in (Q, K, V))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=sm)[0, 0].numpy()
    assert np.allclose(O, ref, rtol=1e-12, atol=1e-12)
    s = (q[0, 0] @ k[0, 0].T).numpy() * sm
    assert np.allclose(L, np.logaddexp.reduce(s, axis=1) / math.log(2), atol=1e-10)


def test_dense_centring_and_joint_permutation_invariance(orc):
    """K centring (attention-equivalent) and a joint K/V permutation leave
    exact attention unchanged."""
    rng = np.random.default_rng(80)
    N = 200
    q = rng.integers(-4, 5, (N, 128)).astype(np.float32)
    mu = rng.integers(-8, 9, (1, 128)).astype(np.float32)
    kc = rng.integers(-4, 5, (N, 128)).astype(np.float32)
    v = rng.standard_normal((N, 128)).astype(np.float32)
    Qb, Kc, Kb, Vb = _bits(q), _bits(kc), _bits(kc + mu), _bits(v)
    sm = 0.05
    Oa, _ = orc.attn_dense(Qb, Kb, Vb, sm)
    Ob, _ = orc.attn_dense(Qb, Kc, Vb, sm)
    assert np.allclose(Oa, Ob, rtol=1e-12, atol=1e-12)
    perm = rng.permutation(N)
    Oc, _ = orc.attn_dense(Qb, Kb[perm], Vb[perm], sm)
    assert np.allclose(Oa, Oc, rtol=1e-12, atol=1e-12)


def test_dense_mask_matches_torch(orc):
    N = 256
    Q, K, V = _small_inputs(N=N, H=1, seed=90)
    sm = SM
    rng = np.random.default_rng(91)
    perm = rng.permutation(N).astype(np.int32)
    mask = (rng.random((4, 4)) < 0.5).astype(np.uint8)
    mask[np.arange(4), np.arange(4)] = 1
    O, _ = orc.attn_dense(Q[0], K[0], V[0], sm, mask=mask, perm=perm)
    allowed = np.zeros((N, N), bool)
    for i in range(N):
        for p in range(N):
            allowed[i, perm[p]] = mask[i // 64, p // 64]
    q, k, v = (torch.from_numpy(_f(x[0])) for x in (Q, K, V))
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[None, None], k[None, None], v[None, None], attn_mask=torch.from_numpy(allowed)[None, None],
        scale=sm)[0, 0].numpy()
    assert np.allclose(O, ref, rtol=1e-12, atol=1e-12)


def test_emul_end_to_end_close_to_dense(orc):
    """The whole quantised pipeline against exact attention on the tiny
    workload: rel-L2 <= 0.05 and cosine >= 0.998."""
    w = W.WORKLOADS["tiny"]
    Q, K, V = (W.bf16_bits(t)[0] for t in W.make_workload(w))
    labels, _ = orc.kmeans(V, w.k, w.iters)
    perm = orc.stable_sort(labels, w.k)
    pp = orc.prep(Q, K, V, perm)
    qidx = np.arange(0, w.N, 3)
    for h in range(w.H):
        Oe, Le = orc.attn_emul(pp, h, w.N, w.sm_scale, qidx=qidx)
        Od, Ld = orc.attn_dense(Q[h], K[h], V[h], w.sm_scale, qidx=qidx)
        rel = np.linalg.norm(Oe - Od) / np.linalg.norm(Od)
        cos = (Oe * Od).sum() / (np.linalg.norm(Oe) * np.linalg.norm(Od))
        assert rel <= 0.05 and cos >= 0.998, (rel, cos)
        assert np.abs(Le - Ld).max() < 0.05


# ------------------------------------------------------ QK Hadamard rotation
def test_hadamard_butterfly_is_the_sylvester_matrix(orc):
    """The butterfly maps the unit vectors to the rows of the 128-point
    Sylvester-Hadamard matrix (scipy.linalg.hadamard), so it computes x H
    with H H^T = 128 I."""
    from scipy.linalg import hadamard
    H = hadamard(128).astype(np.float64)
    Y = orc.hadamard128(np.eye(128, dtype=np.float32)).astype(np.float64)
    assert np.array_equal(Y, H)
    assert np.array_equal(Y @ Y.T, 128.0 * np.eye(128))


def test_hadamard_butterfly_fp32_error_bound(orc):
    """Seven stages of FP32 additions: each output is within 7 u sum|x| of
    the exact x H (u = 2^-24), and a row of powers of two with no
    cancellation is exact."""
    from scipy.linalg import hadamard
    H = hadamard(128).astype(np.float64)
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((2000, 128)) * np.exp(rng.uniform(-8, 8, (2000, 1)))).astype(np.float32)
    x[::7, 3] *= 1000.0                        # outlier channels
    y = orc.hadamard128(x).astype(np.float64)
    exact = x.astype(np.float64) @ H
    bound = 7 * 2.0 ** -24 * np.abs(x).astype(np.float64).sum(1, keepdims=True)
    assert np.all(np.abs(y - exact) <= bound + 1e-30)
    assert not np.array_equal(y, exact)       # FP32 rounding does happen
    e = np.zeros((1, 128), np.float32)
    e[0, :] = 2.0 ** -3
    assert np.array_equal(orc.hadamard128(e)[0].astype(np.float64), e[0].astype(np.float64) @ H)


def test_prep_hadamard_rotates_only_q_and_k(orc):
    """With the rotation, the V side, the K mean and qmu are those of the
    plain preprocessing; Q8 and K8 quantise x H / 16 and (k - mu_K) H / 8,
    so the dequantised scores still approximate q . (k - mu_K) (the
    rotation is orthogonal up to the power-of-two scaling), and on inputs
    with outlier channels more closely than without the rotation."""
    Q, K, V = _small_inputs(N=700, H=1, seed=71)
    # a few outlier channels in Q and K (bf16 bit patterns scaled by 2^5)
    Qo, Ko = Q.copy(), K.copy()
    for t in (Qo, Ko):
        t[..., 5] = ((t[..., 5].astype(np.uint32) + (5 << 7)) & 0xFFFF).astype(np.uint16)
    labels, _ = orc.kmeans(V, 8, 2)
    perm = orc.stable_sort(labels, 8)
    for q, k in ((Q, K), (Qo, Ko)):
        p0 = orc.prep(q, k, V, perm)
        p1 = orc.prep(q, k, V, perm, flags=orc.PREP_QK_HADAMARD)
        for key in ("r8t", "v_scale", "v_mean", "k_mean", "qmu"):
            assert np.array_equal(p0[key], p1[key]), key
        assert not np.array_equal(p0["q8"], p1["q8"]) and not np.array_equal(p0["k8"], p1["k8"])
    N = Q.shape[1]

    def scores(pp, q, k):
        qd = orc.e4m3_decode(pp["q8"][0, :N]) * np.repeat(pp["q_scale"][0], 64)[:N, None]
        kd = orc.e4m3_decode(pp["k8"][0, :N]) * np.repeat(pp["k_scale"][0], 64)[:N, None]
        qf = (q[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        kf = (k[0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)[perm[0]]
        kc = kf - pp["k_mean"][0].astype(np.float64)
        exact = qf @ kc.T
        return np.linalg.norm(qd @ kd.T - exact) / np.linalg.norm(exact)

    e_plain = scores(orc.prep(Qo, Ko, V, perm), Qo, Ko)
    e_rot = scores(orc.prep(Qo, Ko, V, perm, flags=orc.PREP_QK_HADAMARD), Qo, Ko)
    assert e_rot < 0.05 and e_plain < 0.2
    assert e_rot < e_plain, (e_rot, e_plain)


def test_emul_with_hadamard_close_to_dense(orc):
    """The whole pipeline with the QK rotation meets the same bar against
    exact attention (rel-L2 <= 0.05, cosine >= 0.998); with the exact
    exponential it is softmax attention of the dequantised rotated tensors."""
    w = W.WORKLOADS["tiny"]
    Q, K, V = (W.bf16_bits(t)[0] for t in W.make_workload(w))
    labels, _ = orc.kmeans(V, w.k, w.iters)
    perm = orc.stable_sort(labels, w.k)
    pp = orc.prep(Q, K, V, perm, flags=orc.PREP_QK_HADAMARD)
    qidx = np.arange(0, w.N, 3)
    for h in range(w.H):
        Oe, Le = orc.attn_emul(pp, h, w.N, SM, qidx=qidx, tau8=6.0)
        Od, Ld = orc.attn_dense(Q[h], K[h], V[h], SM, qidx=qidx)
        rel = np.linalg.norm(Oe - Od) / np.linalg.norm(Od)
        cos = (Oe * Od).sum() / (np.linalg.norm(Oe) * np.linalg.norm(Od))
        assert rel <= 0.05 and cos >= 0.998, (rel, cos)
        assert np.abs(Le - Ld).max() < 0.05
    O1, L1 = orc.attn_emul(pp, 0, w.N, SM, flags=1)
    q, k, v = _deq(orc, pp, 0, w.N)
    o, lse2 = _softmax_attn(q, k, v, SM)
    assert np.allclose(O1, o, rtol=1e-10, atol=1e-10)
