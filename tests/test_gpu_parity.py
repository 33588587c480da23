"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars (the stated tolerances of the method's hot path):
* k-means labels, centroids and the permutation: bit-exact;
* quantised bytes, scales and means: bit-exact (E4M3 rounding ties are
  counted and reported; both sides round half to even so they must agree);
* attention output (FP32 output mode) vs the emulating oracle: rel-L2 <= 2e-3
  and max-abs <= 4e-3; vs exact FP64 attention: rel-L2 <= 0.05 and cosine >=
  0.998; log2-LSE vs the emulating oracle: max-abs <= 1e-3;
* bf16 output: within the FP32 bar plus half a bf16 ulp of the output.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from bit_smoothed_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SM = float(np.float32(1 / math.sqrt(128)))
REL_EMUL, ABS_EMUL = 2e-3, 4e-3
REL_DENSE, COS_DENSE = 0.05, 0.998
LSE_EMUL = 1e-3
TAU8 = 6.0   # the library's default lazy-rescale threshold (code units)


@pytest.fixture(scope="module")
def vc():
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    major, minor = torch.cuda.get_device_capability()
    assert (major, minor) == (10, 3), "the library is built for sm_103a"
    return vcattn


def _inputs(B, H, N, k_lat, seed):
    Q, K, V = W.make_qkv(B, H, N, k_lat, seed, device="cuda")
    return Q, K, V


def _bits(t):
    return W.bf16_bits(t).reshape(-1, t.shape[-2], t.shape[-1])


def _metrics(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(got - ref).max()
    cos = (got * ref).sum() / max(np.linalg.norm(got) * np.linalg.norm(ref), 1e-30)
    return rel, mx, cos


def _oracle_pipeline(orc, Qb, Kb, Vb, k, iters):
    labels, cent = orc.kmeans(Vb, k, iters)
    perm = orc.stable_sort(labels, k)
    pp = orc.prep(Qb, Kb, Vb, perm)
    return labels, cent, perm, pp


# ------------------------------------------------------------------- group
@pytest.mark.parametrize("N,H,k", [(1024, 2, 8), (777, 2, 5), (1, 1, 1), (63, 1, 3), (129, 2, 64),
                                   (3000, 1, 32), (2049, 1, 16)])
def test_group_bit_exact(vc, orc, N, H, k):
    Q, K, V = _inputs(1, H, N, max(k, 1), 100 + N + k)
    labels, perm, cent = vc.group(V, k, 5, centroids=True)
    torch.cuda.synchronize()
    Vb = _bits(V)
    ol, oc = orc.kmeans(Vb, k, 5)
    op = orc.stable_sort(ol, k)
    gl = labels.reshape(H, N).cpu().numpy()
    gp = perm.reshape(H, N).cpu().numpy()
    gc = cent.reshape(H, k, 128).cpu().numpy()
    assert np.array_equal(gl, ol), "labels differ at %d tokens" % (gl != ol).sum()
    assert np.array_equal(gc.view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(gp, op)
    assert vc.last_device_error() == 0


def test_group_degenerate_inputs(vc, orc):
    """All-zero V and constant V: every score ties, everything goes to cluster 0."""
    for fill in (0.0, 1.5):
        V = torch.full((1, 1, 300, 128), fill, dtype=torch.bfloat16, device="cuda")
        labels, perm = vc.group(V, 4, 3)
        assert (labels == 0).all()
        assert torch.equal(perm[0, 0].cpu(), torch.arange(300, dtype=torch.int32))
        ol, _ = orc.kmeans(_bits(V), 4, 3)
        assert np.array_equal(labels.reshape(1, 300).cpu().numpy(), ol)


def test_group_all_clusters_tied(vc, orc):
    """The seeds are 64 sign patterns of one bf16 vector u, so every h_c is
    the same float (the squares come in the same order), and a third of the
    tokens are zero: their 64 scores are one value, every cluster stays a
    candidate through both filters (two rounds of exact chains), and the
    lowest index must win.  Other tokens are small multiples of the seeds
    and random rows.  Bit-exact after one and two iterations."""
    H, N, k = 2, 4096, 64
    g = torch.Generator(device="cpu")
    g.manual_seed(777)
    V = (torch.randn(1, H, N, 128, generator=g) * 0.5).to(torch.bfloat16)
    u = (torch.rand(128, generator=g) + 0.5).to(torch.bfloat16)
    sign = torch.randint(0, 2, (k, 128), generator=g).to(torch.bool)
    seeds = [(c * N) // k for c in range(k)]
    zero = torch.rand(N, generator=g) < 0.33
    for h in range(H):
        V[0, h, zero] = 0.0
        for c, j in enumerate(seeds):
            V[0, h, j] = torch.where(sign[c], -u, u)
        for c, j in enumerate(seeds):       # a few scaled copies next to each seed
            if j + 1 < N and (j + 1) not in seeds:
                V[0, h, j + 1] = (torch.where(sign[c], -u, u).float() * 0.5).to(torch.bfloat16)
    V = V.cuda()
    for iters in (1, 2):
        labels, perm, cent = vc.group(V, k, iters, centroids=True)
        torch.cuda.synchronize()
        ol, oc = orc.kmeans(_bits(V), k, iters)
        op = orc.stable_sort(ol, k)
        assert np.array_equal(labels.reshape(H, N).cpu().numpy(), ol)
        assert np.array_equal(cent.reshape(H, k, 128).cpu().numpy().view(np.uint32), oc.view(np.uint32))
        assert np.array_equal(perm.reshape(H, N).cpu().numpy(), op)
        if iters == 1:   # the zero tokens all went to cluster 0
            z = zero.numpy().copy()
            z[seeds] = False
            z[[j + 1 for j in seeds if j + 1 < N]] = False
            assert z.sum() > 1000 and np.all(ol[:, z] == 0)
    assert vc.last_device_error() == 0


def test_group_near_ties(vc, orc):
    """Pairs of initial centroids one bf16 ulp apart in one channel, and
    tokens repeated from them: most scores of the first iterations differ in
    the last bits only, so the tensor-core bound keeps several candidates and
    the FP32 filter and the exact chains decide.  Still bit-exact."""
    H, N, k = 2, 2048, 16
    g = torch.Generator(device="cpu")
    g.manual_seed(4242)
    V = (torch.randn(1, H, N, 128, generator=g) * 2.0).to(torch.bfloat16)
    bits = V.view(torch.int16)
    for c in range(1, k, 2):
        j0, j1 = (c - 1) * N // k, c * N // k
        bits[:, :, j1] = bits[:, :, j0]
        bits[:, :, j1, c % 128] += 1          # one ulp in one channel
        # copies of the pair, each tied exactly or nearly between the two
        for r in range(1, 9):
            bits[:, :, j1 + r] = bits[:, :, j0 if r % 2 else j1]
    V = V.cuda()
    labels, perm, cent = vc.group(V, k, 5, centroids=True)
    torch.cuda.synchronize()
    ol, oc = orc.kmeans(_bits(V), k, 5)
    op = orc.stable_sort(ol, k)
    assert np.array_equal(labels.reshape(H, N).cpu().numpy(), ol)
    assert np.array_equal(cent.reshape(H, k, 128).cpu().numpy().view(np.uint32), oc.view(np.uint32))
    assert np.array_equal(perm.reshape(H, N).cpu().numpy(), op)
    assert vc.last_device_error() == 0


# -------------------------------------------------------------------- prep
PREP_KEYS = ("q8", "k8", "r8t", "q_scale", "k_scale", "v_scale", "k_mean", "v_mean", "qmu")


@pytest.mark.parametrize("N", [1, 63, 64, 65, 127, 129, 777, 1024])
def test_prep_bit_exact(vc, orc, N):
    H = 2
    Q, K, V = _inputs(1, H, N, 8, 200 + N)
    labels, perm = vc.group(V, 8, 2)
    pp = vc.prep(Q, K, V, perm)
    torch.cuda.synchronize()
    Qb, Kb, Vb = _bits(Q), _bits(K), _bits(V)
    op = orc.stable_sort(orc.kmeans(Vb, 8, 2)[0], 8)
    assert np.array_equal(perm.reshape(H, N).cpu().numpy(), op)
    ref = orc.prep(Qb, Kb, Vb, op)
    got = {k: v.cpu().numpy() for k, v in pp.views().items()}
    for key in PREP_KEYS:
        g, r = got[key], ref[key]
        if g.dtype == np.float32:
            g, r = g.view(np.uint32), r.view(np.uint32)
        bad = np.nonzero(g != r)
        assert bad[0].size == 0, "%s differs at %d places, first %s" % (key, bad[0].size,
                                                                      [b[:3] for b in bad])
    assert vc.last_device_error() == 0


@pytest.mark.parametrize("N", [1, 63, 65, 129, 777, 2049])
def test_prep_hadamard_bit_exact(vc, orc, N):
    """The QK Hadamard rotation (vcattn_prep_ex): every prepped tensor equal
    to the oracle's rotated preprocessing, bit for bit (the butterfly's FP32
    order is part of the definition), also for a strided (B, N, H, D) input."""
    H = 2
    Q, K, V = _inputs(1, H, N, 8, 220 + N)
    _, perm = vc.group(V, 8, 2)
    pp = vc.prep(Q, K, V, perm, hadamard=True)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    op = perm.reshape(H, N).cpu().numpy()
    ref = orc.prep(_bits(Q), _bits(K), _bits(V), op, flags=orc.PREP_QK_HADAMARD)
    got = {k: v.cpu().numpy() for k, v in pp.views().items()}
    for key in PREP_KEYS:
        g, r = got[key], ref[key]
        if g.dtype == np.float32:
            g, r = g.view(np.uint32), r.view(np.uint32)
        bad = np.nonzero(g != r)
        assert bad[0].size == 0, "%s differs at %d places, first %s" % (key, bad[0].size,
                                                                      [b[:3] for b in bad])
    Qs, Ks, Vs = (t.transpose(1, 2).contiguous().transpose(1, 2) for t in (Q, K, V))
    pps = vc.prep(Qs, Ks, Vs, perm, hadamard=True)
    for key, val in pp.views().items():
        assert torch.equal(pps.views()[key], val), key


def test_attn_with_hadamard_prep(vc, orc):
    """Attention on the rotated preprocessing meets both bars (against the
    oracle's rotated pipeline and against exact attention on the inputs)."""
    N, H, k = 1500, 2, 8
    Q, K, V = _inputs(1, H, N, k, 230)
    _, perm = vc.group(V, k, 5)
    pp = vc.prep(Q, K, V, perm, hadamard=True)
    O32, L = vc.attn(pp, SM, out_f32=True)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    Qb, Kb, Vb = _bits(Q), _bits(K), _bits(V)
    op = perm.reshape(H, N).cpu().numpy()
    opp = orc.prep(Qb, Kb, Vb, op, flags=orc.PREP_QK_HADAMARD)
    for h in range(H):
        Oe, Le = orc.attn_emul(opp, h, N, SM, tau8=TAU8)
        Od, _ = orc.attn_dense(Qb[h], Kb[h], Vb[h], SM)
        g = O32[0, h].cpu().numpy()
        rel, mx, _ = _metrics(g, Oe)
        assert rel <= REL_EMUL and mx <= ABS_EMUL, (rel, mx)
        assert np.abs(L[0, h].cpu().numpy() - Le).max() <= LSE_EMUL
        rel_d, _, cos_d = _metrics(g, Od)
        assert rel_d <= REL_DENSE and cos_d >= COS_DENSE, (rel_d, cos_d)


def test_prep_out_of_range_perm_is_reported_not_read(vc):
    """Permutation entries outside [0, N) (a stale or corrupt perm) are never
    dereferenced: the preprocessing reads those rows as zeros and reports a
    device-side error; the context stays usable."""
    N, H = 700, 2
    Q, K, V = _inputs(1, H, N, 8, 210)
    perm = torch.arange(N, dtype=torch.int32, device="cuda").repeat(1, H, 1).contiguous()
    perm[0, 0, 5] = N + 5
    perm[0, 1, 17] = -1
    perm[0, 1, 690] = 1 << 30
    pp = vc.prep(Q, K, V, perm)
    torch.cuda.synchronize()
    assert vc.last_device_error() == vc.ERR_DEVICE
    assert vc.last_device_error() == 0
    v = pp.views()
    assert torch.isfinite(v["k_mean"]).all() and torch.isfinite(v["v_scale"]).all()
    pp = vc.prep(Q, K, V, None)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0


def test_prep_identity_perm_and_zero_blocks(vc, orc):
    N = 200
    Q = torch.zeros(1, 1, N, 128, dtype=torch.bfloat16, device="cuda")
    K = torch.zeros_like(Q)
    V = torch.full_like(Q, 2.0)
    pp = vc.prep(Q, K, V, None)
    ref = orc.prep(_bits(Q), _bits(K), _bits(V), None)
    got = {k: v.cpu().numpy() for k, v in pp.views().items()}
    for key in PREP_KEYS:
        assert np.array_equal(got[key], ref[key]), key
    assert np.all(got["v_scale"] == 1.0) and np.all(got["r8t"] == 0)


@pytest.mark.parametrize("N,H,k,n,m", [(3000, 2, 16, 2, 3), (777, 1, 5, 1, 1), (2049, 1, 64, 3, 2)])
def test_group_warm_start(vc, orc, N, H, k, n, m):
    """vcattn_group_warm: bit-exact against the oracle's warm start, and n
    iterations followed by m warm-started ones equal n + m iterations (also
    with the centroids updated in place)."""
    Q, K, V = _inputs(1, H, N, k, 900 + N)
    _, _, c_n = vc.group(V, k, n, centroids=True)
    l_w, p_w, c_w = vc.group(V, k, m, centroids=True, init=c_n)
    l_c, p_c, c_c = vc.group(V, k, n + m, centroids=True)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    assert torch.equal(l_w, l_c) and torch.equal(p_w, p_c) and torch.equal(c_w, c_c)
    Vb = _bits(V)
    _, oc_n = orc.kmeans(Vb, k, n)
    assert np.array_equal(c_n.reshape(H, k, 128).cpu().numpy(), oc_n)
    ol, oc = orc.kmeans(Vb, k, m, init=oc_n)
    assert np.array_equal(l_w.reshape(H, N).cpu().numpy(), ol)
    assert np.array_equal(p_w.reshape(H, N).cpu().numpy(), orc.stable_sort(ol, k))
    assert np.array_equal(c_w.reshape(H, k, 128).cpu().numpy(), oc)
    # in place: the output centroid buffer is the starting one
    c_in = c_n.clone()
    s = vc._shape(V)
    lab = torch.empty(1, H, N, dtype=torch.int32, device="cuda")
    prm = torch.empty_like(lab)
    nb = vc.lib().vcattn_group_workspace_bytes(ctypes.byref(s), k)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    assert vc.lib().vcattn_group_warm(ctypes.byref(s), vc._ptr(V), k, m, vc._ptr(c_in), vc._ptr(lab),
                                      vc._ptr(prm), vc._ptr(c_in), vc._ptr(ws), nb,
                                      vc._stream(None)) == 0
    torch.cuda.synchronize()
    assert torch.equal(c_in, c_w) and torch.equal(lab, l_w)


# --------------------------------------------------------------- attention
def _attn_case(vc, orc, N, H, k, seed, mask=None, tau8=TAU8, qidx=None, off=8, keep_prep=False):
    Q, K, V = _inputs(1, H, N, k, seed)
    labels, perm = vc.group(V, k, 5)
    pp = vc.prep(Q, K, V, perm)
    mt = None if mask is None else torch.from_numpy(mask).cuda()
    O32, L = vc.attn(pp, SM, mask=mt, off=off, tau8=tau8, out_f32=True)
    O16, _ = vc.attn(pp, SM, mask=mt, off=off, tau8=tau8)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    Qb, Kb, Vb = _bits(Q), _bits(K), _bits(V)
    _, _, op, opp = _oracle_pipeline(orc, Qb, Kb, Vb, k, 5)
    assert np.array_equal(perm.reshape(H, N).cpu().numpy(), op)
    qidx = np.arange(N) if qidx is None else qidx
    res = []
    for h in range(H):
        mh = None if mask is None else mask[0, h]
        Oe, Le = orc.attn_emul(opp, h, N, SM, qidx=qidx, off=off, tau8=tau8, mask=mh)
        Od, Ld = orc.attn_dense(Qb[h], Kb[h], Vb[h], SM, qidx=qidx, mask=mh, perm=op[h])
        g32 = O32[0, h].cpu().numpy()[qidx]
        g16 = O16[0, h].float().cpu().numpy()[qidx]
        gl = L[0, h].cpu().numpy()[qidx]
        res.append((g32, g16, gl, Oe, Le, Od, Ld))
    if keep_prep:
        return res, opp, qidx
    return res


def _score_tie_rows(orc, opp, h, qidx, g32, Oe, N):
    """Rows whose output is off the emulating oracle by more than the max-abs
    bar may be waived only at a rounding tie (the method's waiver: mismatches
    only at counted ties).  The tensor core accumulates a score in FP32 in
    its own order, the oracle rounds the exact sum to nearest even; where the
    exact score is halfway between two FP32 values the two can differ by one
    ulp, and an ExpCast argument that lands on a code boundary then gives a
    code one step apart.  A row qualifies when its deviation lies along one
    key's dequantised value row minus the output (|cos| >= 0.9999) and that
    key's exact score is an FP32 tie.  Returns the rows waived; fails on any
    other row over the bar."""
    over = np.where(np.abs(g32 - Oe).max(axis=1) > ABS_EMUL)[0]
    if over.size == 0:
        return []
    Npad = opp["k8"].shape[1]
    vdec = (orc.e4m3_decode(opp["r8t"][h]).T * opp["v_scale"][h][None, :] +
            opp["v_mean"][h][np.arange(Npad) // 64])[:N]
    qd, kd = orc.e4m3_decode(opp["q8"][h]), orc.e4m3_decode(opp["k8"][h])
    waived = []
    for r in over:
        d = g32[r] - Oe[r]
        u = vdec - Oe[r][None, :]
        cos = (u @ d) / (np.linalg.norm(u, axis=1) * np.linalg.norm(d) + 1e-300)
        j = int(np.argmax(np.abs(cos)))
        x = float(qd[qidx[r]] @ kd[j])            # exact: E4M3 products summed in FP64
        x32 = float(np.float32(x))
        half = float(np.spacing(np.float32(abs(x)))) / 2
        tie = x32 != x and abs(abs(x - x32) - half) == 0.0
        assert abs(cos[j]) >= 0.9999 and tie, (h, int(qidx[r]), j, float(cos[j]), x)
        waived.append(int(qidx[r]))
    return waived


def _check_attn(res):
    for g32, g16, gl, Oe, Le, Od, Ld in res:
        rel, mx, _ = _metrics(g32, Oe)
        assert rel <= REL_EMUL and mx <= ABS_EMUL, (rel, mx)
        fin = np.isfinite(Le)
        assert np.array_equal(np.isfinite(gl), fin)
        if fin.any():
            assert np.abs(gl[fin] - Le[fin]).max() <= LSE_EMUL
        rel_d, _, cos_d = _metrics(g32, Od)
        assert rel_d <= REL_DENSE and cos_d >= COS_DENSE, (rel_d, cos_d)
        # bf16 output: the f32 value rounded to nearest even
        half_ulp = np.abs(Oe) * 2.0 ** -8 + 1e-30
        assert np.all(np.abs(g16 - Oe) <= ABS_EMUL + half_ulp)
        assert np.array_equal(g16, torch.from_numpy(g32).bfloat16().float().numpy())


@pytest.mark.parametrize("N,H,k", [(1024, 2, 8), (777, 2, 8), (129, 1, 4), (1, 1, 1), (63, 1, 2),
                                   (256, 1, 8), (2500, 1, 16)])
def test_attn_dense_parity(vc, orc, N, H, k):
    _check_attn(_attn_case(vc, orc, N, H, k, 300 + N))


@pytest.mark.parametrize("tau8", [0.0, 4.0])
def test_attn_rescale_threshold_parity(vc, orc, tau8):
    """tau8 = 0 is the exact running max; other thresholds rescale lazily."""
    _check_attn(_attn_case(vc, orc, 900, 1, 8, 401, tau8=tau8))


def test_attn_mask_parity(vc, orc):
    N, H = 1000, 2
    nq = (N + 63) // 64
    nbp = vc.npad(N) // 64
    mask = np.asarray(W.make_tile_mask(1, H, N, 555, keep_frac=0.3), np.uint8).copy()
    mask[0, 0, 3, :] = 0                   # an empty selection
    mask[0, 1, :, :] = 0
    mask[0, 1, np.arange(nq), np.arange(nq)] = 1   # diagonal only
    assert mask.shape == (1, H, nq, nbp)
    res = _attn_case(vc, orc, N, H, 8, 402, mask=mask)
    _check_attn(res)
    g32 = res[0][0]
    assert np.all(g32[192:256] == 0) and np.all(np.isneginf(res[0][2][192:256]))


@pytest.mark.parametrize("masked", [False, True])
@pytest.mark.parametrize("off,tau8", [(0, 0.0), (4, 6.0), (8, 6.0)])
def test_attn_exponent_offset_parity(vc, orc, masked, off, tau8):
    """The ExpCast exponent offset (the byte encodes 2^off p): off = 0, 4 and
    the default 8 against the emulating oracle with the same offset, dense and
    block-sparse.  With off = 0 the probabilities below 2^-6 of the row
    maximum flush to zero, so the exact FP64 attention is not a fair reference
    there; the emulating oracle is.  These inputs hold one score that is an
    exact FP32 rounding tie on a key whose code lands on a boundary (at
    off = 4 and 8): that row is waived as a counted tie and reported."""
    N, H = 1000, 2
    mask = np.asarray(W.make_tile_mask(1, H, N, 558, keep_frac=0.4), np.uint8).copy() if masked else None
    res, opp, qidx = _attn_case(vc, orc, N, H, 8, 407, mask=mask, tau8=tau8, off=off, keep_prep=True)
    for h, (g32, g16, gl, Oe, Le, Od, Ld) in enumerate(res):
        rel, _, _ = _metrics(g32, Oe)
        assert rel <= REL_EMUL, rel
        waived = _score_tie_rows(orc, opp, h, qidx, g32, Oe, N)
        if waived:
            print("off=%d head %d: rows %s off by one code at an FP32 score tie" % (off, h, waived))
        fin = np.isfinite(Le)
        assert np.array_equal(np.isfinite(gl), fin)
        if fin.any():
            assert np.abs(gl[fin] - Le[fin]).max() <= LSE_EMUL


@pytest.mark.parametrize("tau8", [0.0, 4.0])
def test_attn_mask_rescale_threshold_parity(vc, orc, tau8):
    """The block-sparse kernel with the exact running maximum (tau8 = 0,
    every rising maximum rescales O and l) and a lower lazy threshold: its
    rescale path (each of a row's two threads rescales its half of O) against
    the oracle replaying the same rule."""
    N, H = 1500, 2
    mask = np.asarray(W.make_tile_mask(1, H, N, 557, keep_frac=0.4), np.uint8).copy()
    _check_attn(_attn_case(vc, orc, N, H, 8, 406, mask=mask, tau8=tau8))


def test_attn_mask_empty_slot(vc, orc):
    """Both query tiles of one 128-row slot keep no block (that slot has no
    KV tile at all) while the other slot of the same CTA, and other CTAs,
    have work: the empty rows get O = 0 and lse2 = -inf, the rest matches
    the oracle."""
    N, H = 1000, 1
    nq, nbp = (N + 63) // 64, vc.npad(N) // 64
    mask = np.asarray(W.make_tile_mask(1, H, N, 404, keep_frac=0.3), np.uint8).copy()
    mask[0, 0, 6:8, :] = 0                 # CTA 1, slot 1: query tiles 6 and 7
    res = _attn_case(vc, orc, N, H, 8, 405, mask=mask)
    _check_attn(res)
    g32, gl = res[0][0], res[0][2]
    assert np.all(g32[384:512] == 0) and np.all(np.isneginf(gl[384:512]))
    assert np.all(np.isfinite(gl[256:384]))


@pytest.mark.parametrize("kind", ["even", "odd", "one", "ones"])
def test_attn_mask_structures(vc, orc, kind):
    """Masks whose kept blocks pair up differently from the dense tiles: every
    other block (the odd ones include the partial last block), a single block
    (an odd tile count with an empty second half), and every block."""
    N, H = 1000, 1
    nq, nbp = (N + 63) // 64, vc.npad(N) // 64
    mask = np.zeros((1, H, nq, nbp), np.uint8)
    if kind == "even":
        mask[..., 0::2] = 1
    elif kind == "odd":
        mask[..., 1::2] = 1
    elif kind == "one":
        mask[..., 5] = 1
    else:
        mask[:] = 1
    _check_attn(_attn_case(vc, orc, N, H, 8, 403, mask=mask))


def test_fwd_equals_prep_then_attn(vc):
    N, H = 700, 2
    Q, K, V = _inputs(1, H, N, 8, 501)
    _, perm = vc.group(V, 8, 5)
    O1, L1 = vc.fwd(Q, K, V, perm, SM)
    pp = vc.prep(Q, K, V, perm)
    O2, L2 = vc.attn(pp, SM)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


@pytest.mark.parametrize("B,H,N,chunk,masked,dual", [(1, 5, 1000, 2, True, True), (2, 3, 777, 0, False, True),
                                                     (1, 1, 63, 0, False, True), (1, 4, 2500, 3, False, False),
                                                     (1, 6, 900, 1, True, False)])
def test_fwd_host_equals_device_path(vc, B, H, N, chunk, masked, dual):
    """vcattn_fwd_host (host Q, K, V in, host O and lse2 out, copies
    overlapped chunk by chunk) gives the device path's O and lse2 bit for bit,
    including a last chunk with fewer heads and a mask sliced per chunk."""
    k = 8
    Q, K, V = W.make_qkv(B, H, N, k, 600 + N, device="cuda")
    mask = None
    if masked:
        mask = W.make_tile_mask(B, H, N, 601, keep_frac=0.3).cuda()
    _, perm = vc.group(V, k, 5)
    O_ref, L_ref = vc.fwd(Q, K, V, perm, SM, mask=mask)
    hQ, hK, hV = (t.cpu().pin_memory() for t in (Q, K, V))
    hO = torch.zeros(Q.shape, dtype=torch.bfloat16).pin_memory()
    hL = torch.zeros(Q.shape[:3], dtype=torch.float32).pin_memory()
    pipe = vc.HostPipeline((B, H, N, 128), k, 5, chunk_heads=chunk, dual=dual)
    pipe(hQ, hK, hV, SM, mask=mask, hO=hO, hlse2=hL)
    pipe.stream.synchronize()
    assert vc.last_device_error() == 0
    assert torch.equal(hO, O_ref.cpu())
    assert torch.equal(hL, L_ref.cpu())
    # a second call through the same workspace and streams gives the same
    hO2, _ = pipe(hQ, hK, hV, SM, mask=mask)
    pipe.stream.synchronize()
    assert torch.equal(hO2, hO)


def test_fwd_host_back_to_back_calls_share_the_workspace(vc):
    """Two calls with different inputs, enqueued back to back on one
    workspace with no synchronisation between them: the second call waits
    for the first (its last chunk uses the slot the second call fills
    first), so both outputs match the device path."""
    B, H, N, k = 1, 5, 1000, 8
    pipe = vc.HostPipeline((B, H, N, 128), k, 5, chunk_heads=2)
    outs, refs = [], []
    for seed in (700, 701):
        Q, K, V = W.make_qkv(B, H, N, k, seed, device="cuda")
        _, perm = vc.group(V, k, 5)
        refs.append(vc.fwd(Q, K, V, perm, SM)[0].cpu())
        hQ, hK, hV = (t.cpu().pin_memory() for t in (Q, K, V))
        outs.append((hQ, hK, hV))
    torch.cuda.synchronize()
    hO = [torch.zeros((B, H, N, 128), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    for (hQ, hK, hV), o in zip(outs, hO):
        pipe(hQ, hK, hV, SM, hO=o)
    pipe.stream.synchronize()
    assert vc.last_device_error() == 0
    assert torch.equal(hO[0], refs[0]) and torch.equal(hO[1], refs[1])


@pytest.mark.parametrize("B,H,N,masked", [(2, 3, 1000, False), (1, 4, 777, True)])
def test_strided_bnhd_inputs_and_output(vc, orc, B, H, N, masked):
    """Q, K, V stored as (B, N, H, D) and passed as strided (B, H, N, D) views
    give the labels, permutation, centroids, prepped bytes and output of
    contiguous copies, bit for bit; O can be written back in the (B, N, H, D)
    layout too (bf16 and f32), and that output meets the bars against both
    oracles directly."""
    k = 8
    # the workload generator's tensors, stored as (B, N, H, D)
    x = [t.transpose(1, 2).contiguous() for t in W.make_qkv(B, H, N, k, 800 + N, device="cuda")]
    Qv, Kv, Vv = (t.transpose(1, 2) for t in x)          # strided views
    Qc, Kc, Vc = (t.contiguous() for t in (Qv, Kv, Vv))
    assert not Vv.is_contiguous()
    l_v, p_v, c_v = vc.group(Vv, k, 3, centroids=True)
    l_c, p_c, c_c = vc.group(Vc, k, 3, centroids=True)
    assert torch.equal(l_v, l_c) and torch.equal(p_v, p_c) and torch.equal(c_v, c_c)
    l_w, _, c_w = vc.group(Vv, k, 1, centroids=True, init=c_c)
    l_w2, _, c_w2 = vc.group(Vc, k, 1, centroids=True, init=c_c)
    assert torch.equal(l_w, l_w2) and torch.equal(c_w, c_w2)
    pp_v = vc.prep(Qv, Kv, Vv, p_c)
    pp_c = vc.prep(Qc, Kc, Vc, p_c)
    for key, val in pp_c.views().items():
        assert torch.equal(pp_v.views()[key], val), key
    mask = W.make_tile_mask(B, H, N, 801, keep_frac=0.3).cuda() if masked else None
    for out_f32 in (False, True):
        dt = torch.float32 if out_f32 else torch.bfloat16
        O_c, L_c = vc.attn(pp_c, SM, mask=mask, out_f32=out_f32)
        O_bnhd = torch.zeros(B, N, H, 128, dtype=dt, device="cuda")
        _, L_v = vc.attn(pp_c, SM, mask=mask, out_f32=out_f32, O=O_bnhd.transpose(1, 2))
        torch.cuda.synchronize()
        assert vc.last_device_error() == 0
        assert torch.equal(O_bnhd.transpose(1, 2), O_c) and torch.equal(L_v, L_c)
        if out_f32:
            # the strided output against both oracles, directly
            Qb, Kb, Vb = _bits(Qc), _bits(Kc), _bits(Vc)
            op = p_c.reshape(B * H, N).cpu().numpy()
            opp = orc.prep(Qb, Kb, Vb, op)
            Ob = O_bnhd.cpu().numpy()
            m_np = None if mask is None else mask.cpu().numpy().reshape(B * H, *mask.shape[2:])
            for bh in range(B * H):
                b, h = divmod(bh, H)
                mh = None if m_np is None else m_np[bh]
                Oe, Le = orc.attn_emul(opp, bh, N, SM, tau8=TAU8, mask=mh)
                Od, _ = orc.attn_dense(Qb[bh], Kb[bh], Vb[bh], SM, mask=mh, perm=op[bh])
                got = Ob[b, :, h, :]
                rel, mx, _ = _metrics(got, Oe)
                assert rel <= REL_EMUL and mx <= ABS_EMUL, (bh, rel, mx)
                keep = np.linalg.norm(Od, axis=1) > 0
                rel_d, _, cos_d = _metrics(got[keep], Od[keep])
                assert rel_d <= REL_DENSE and cos_d >= COS_DENSE, (bh, rel_d, cos_d)


# ------------------------------------------------- the bench configuration
def test_live_workload_all_heads(vc, orc):
    """The 32,626-token workload in the launch configuration the benchmark
    times (all 56 heads in one call): labels, permutation and every prepped
    tensor (bytes, scales, means, k_mean, qmu) bit-exact on every head; 64
    evenly spaced queries of every head against both oracles.  The rounding
    ties are counted and reported: E4M3 quantiser inputs exactly halfway
    between two codes (where the bytes still agree, both sides rounding half
    to even), and tokens whose last k-means assignment has two equal best
    scores (where the labels still agree, the lower cluster winning)."""
    w = W.WORKLOADS["live"]
    sm = float(np.float32(w.sm_scale))
    Q, K, V = W.make_workload(w, device="cuda")
    labels, perm = vc.group(V, w.k, w.iters)
    pp = vc.prep(Q, K, V, perm)
    O32, L = vc.attn(pp, w.sm_scale, out_f32=True)   # library default tau8
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    qidx = W.evenly_spaced_queries(w.N)
    views = {k: v.cpu().numpy() for k, v in pp.views().items()}
    Qa, Ka, Va = (W.bf16_bits(t).reshape(w.H, w.N, 128) for t in (Q, K, V))
    ol, _ = orc.kmeans(Va, w.k, w.iters)
    op = orc.stable_sort(ol, w.k)
    assert np.array_equal(labels[0].cpu().numpy(), ol)
    assert np.array_equal(perm[0].cpu().numpy(), op)
    opp = orc.prep(Qa, Ka, Va, op, count_ties=True)
    for key in PREP_KEYS:
        g, r = views[key], opp[key]
        if g.dtype == np.float32:
            g, r = g.view(np.uint32), r.view(np.uint32)
        assert np.array_equal(g, r), key
    ties = opp["ties"].sum(axis=0)
    # the last assignment scores each token against the centroids of the
    # iteration before it
    _, cprev = orc.kmeans(Va, w.k, w.iters - 1)
    score_ties = 0
    for h in range(w.H):
        sc = orc.kmeans_scores(Va[h], cprev[h])
        best = sc.max(axis=1, keepdims=True)
        tied = (sc == best).sum(axis=1) > 1
        score_ties += int(tied.sum())
        # a tied token goes to the lowest tied cluster
        assert np.array_equal(ol[h][tied], np.argmax(sc[tied] == best[tied], axis=1))
    print("live, all 56 heads: E4M3 rounding ties Q %d, K %d, V residual %d (bytes equal at all); "
          "k-means score ties %d (labels equal at all)" % (ties[0], ties[1], ties[2], score_ties))
    O32h, Lh = O32[0].cpu().numpy(), L[0].cpu().numpy()
    worst = 0.0
    for h in range(w.H):
        Oe, Le = orc.attn_emul(opp, h, w.N, sm, qidx=qidx, tau8=TAU8)
        Od, _ = orc.attn_dense(Qa[h], Ka[h], Va[h], sm, qidx=qidx)
        g = O32h[h][qidx]
        rel, mx, _ = _metrics(g, Oe)
        assert rel <= REL_EMUL and mx <= ABS_EMUL, (h, rel, mx)
        assert np.abs(Lh[h][qidx] - Le).max() <= LSE_EMUL
        rel_d, _, cos_d = _metrics(g, Od)
        assert rel_d <= REL_DENSE and cos_d >= COS_DENSE, (h, rel_d, cos_d)
        worst = max(worst, rel)
    print("live, all 56 heads: worst rel-L2 vs the emulating oracle %.2e" % worst)
