"""GPU parity on the remaining workload configurations, at full size, in the
launch configuration the benchmark uses (all heads in one call):

* mid (8 heads, N = 8192, k = 32): full output, every query, two heads;
* schedule (40 heads, N = 32760, 50 denoising steps): grouping on steps
  0..12, the step-12 permutation reused on steps 13..49; per-step output
  against exact attention on 64 queries of two heads, and against the
  emulating oracle on the last step;
* sparse (56 heads, N = 115328, 20% of 64x64 tiles kept, one query tile per
  head with the diagonal only): labels, permutation and bytes bit-exact and
  64 queries against both oracles on two heads, restricted to the kept tiles.
"""
import math

import numpy as np
import pytest
import torch

from bit_smoothed_attention_gb300 import workloads as W

pytestmark = pytest.mark.gpu

REL_EMUL, ABS_EMUL = 2e-3, 4e-3
REL_DENSE, COS_DENSE = 0.05, 0.998
LSE_EMUL = 1e-3
TAU8 = 6.0


@pytest.fixture(scope="module")
def vc():
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    return vcattn


def _metrics(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    cos = (got * ref).sum() / max(np.linalg.norm(got) * np.linalg.norm(ref), 1e-30)
    return rel, np.abs(got - ref).max(), cos


def _head_bits(t, h):
    return W.bf16_bits(t[:, h:h + 1]).reshape(1, t.shape[-2], 128)


def _check_head(orc, O32, L, Qb, Kb, Vb, opp, sm, qidx, mask_h=None, perm_h=None):
    Oe, Le = orc.attn_emul(opp, 0, Qb.shape[1], sm, qidx=qidx, tau8=TAU8, mask=mask_h)
    Od, _ = orc.attn_dense(Qb[0], Kb[0], Vb[0], sm, qidx=qidx, mask=mask_h, perm=perm_h)
    g = O32[qidx]
    rel, mx, _ = _metrics(g, Oe)
    assert rel <= REL_EMUL and mx <= ABS_EMUL, (rel, mx)
    fin = np.isfinite(Le)
    assert np.array_equal(np.isfinite(L[qidx]), fin)
    if fin.any():
        assert np.abs(L[qidx][fin] - Le[fin]).max() <= LSE_EMUL
    keep = np.linalg.norm(Od, axis=1) > 0
    rel_d, _, cos_d = _metrics(g[keep], Od[keep])
    assert rel_d <= REL_DENSE and cos_d >= COS_DENSE, (rel_d, cos_d)
    return rel_d


def test_mid_full_output(vc, orc):
    w = W.WORKLOADS["mid"]
    sm = float(np.float32(w.sm_scale))
    Q, K, V = W.make_workload(w, device="cuda")
    labels, perm = vc.group(V, w.k, w.iters)
    pp = vc.prep(Q, K, V, perm)
    O32, L = vc.attn(pp, sm, out_f32=True)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    views = pp.views()
    for h in (0, 7):
        Qb, Kb, Vb = (_head_bits(t, h) for t in (Q, K, V))
        ol, _ = orc.kmeans(Vb, w.k, w.iters)
        op = orc.stable_sort(ol, w.k)
        assert np.array_equal(labels[0, h].cpu().numpy(), ol[0])
        assert np.array_equal(perm[0, h].cpu().numpy(), op[0])
        opp = orc.prep(Qb, Kb, Vb, op)
        for key in ("q8", "k8", "r8t", "q_scale", "k_scale", "v_scale", "v_mean"):
            assert np.array_equal(views[key][h].cpu().numpy(), opp[key][0]), key
        _check_head(orc, O32[0, h].cpu().numpy(), L[0, h].cpu().numpy(), Qb, Kb, Vb, opp, sm,
                    np.arange(w.N))


def test_schedule_regroup_then_reuse(vc, orc):
    """Parity with the emulating oracle on every checked step.  Against exact
    attention the bar of 0.05 holds while the drift is small (steps 0..13);
    late in the schedule the inputs carry drift of up to 2.45 standard
    deviations, the logits grow accordingly and the method itself (the
    emulating oracle) moves away from exact attention, so there the GPU's
    error against exact attention must equal the oracle's; the oracle grouped
    afresh on the late step does only slightly better than the frozen
    permutation."""
    w = W.WORKLOADS["schedule"]
    sm = float(np.float32(w.sm_scale))
    Q0, K0, V0 = W.make_workload(w, device="cuda")
    qidx = W.evenly_spaced_queries(w.N)
    heads = (0, 39)
    checked = (0, 12, 13, 30, 49)
    regroup_steps = 13                      # steps 0..12, the first quarter of 50
    perm = None
    operm = {}
    times = []
    for t in range(w.steps):
        Q, K, V = (W.drift(x, t, w.seed + j) for j, x in enumerate((Q0, K0, V0)))
        if t < regroup_steps:
            _, perm = vc.group(V, w.k, w.iters)
        pp = vc.prep(Q, K, V, perm)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        O32, L = vc.attn(pp, sm, out_f32=True)
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
        assert vc.last_device_error() == 0
        if t not in checked:
            continue
        for h in heads:
            Qb, Kb, Vb = (_head_bits(x, h) for x in (Q, K, V))
            if t < regroup_steps:
                ol, _ = orc.kmeans(Vb, w.k, w.iters)
                operm[h] = orc.stable_sort(ol, w.k)
                assert np.array_equal(perm[0, h].cpu().numpy(), operm[h][0])
            opp = orc.prep(Qb, Kb, Vb, operm[h])
            Oe, Le = orc.attn_emul(opp, 0, w.N, sm, qidx=qidx, tau8=TAU8)
            Od, _ = orc.attn_dense(Qb[0], Kb[0], Vb[0], sm, qidx=qidx)
            g = O32[0, h].cpu().numpy()[qidx]
            rel, mx, _ = _metrics(g, Oe)
            assert rel <= REL_EMUL and mx <= ABS_EMUL, (t, h, rel, mx)
            assert np.abs(L[0, h].cpu().numpy()[qidx] - Le).max() <= LSE_EMUL
            rel_d, _, cos_d = _metrics(g, Od)
            rel_m, _, _ = _metrics(Oe, Od)
            print("schedule step %2d head %2d: rel-L2 vs exact %.4f (oracle %.4f), cosine %.5f"
                  % (t, h, rel_d, rel_m, cos_d))
            if t <= regroup_steps:
                assert rel_d <= REL_DENSE and cos_d >= COS_DENSE, (t, h, rel_d, cos_d)
            else:
                assert abs(rel_d - rel_m) <= 0.1 * rel_m + 1e-3, (t, h, rel_d, rel_m)
                # The same pipeline grouped afresh on this step's V: its
                # error against exact attention is nearly as large, so most
                # of the late loss comes from the drifted inputs (larger
                # logits), and at most 30% from the permutation frozen at
                # step 12.
                fl, _ = orc.kmeans(Vb, w.k, w.iters)
                fpp = orc.prep(Qb, Kb, Vb, orc.stable_sort(fl, w.k))
                Of, _ = orc.attn_emul(fpp, 0, w.N, sm, qidx=qidx, tau8=TAU8)
                rel_f, _, _ = _metrics(Of, Od)
                print("schedule step %2d head %2d: oracle with a fresh grouping %.4f" % (t, h, rel_f))
                assert rel_f >= 0.7 * rel_m, (t, h, rel_m, rel_f)
    print("schedule: attention ms per step, median %.3f (min %.3f, max %.3f)"
          % (float(np.median(times[1:])), min(times[1:]), max(times[1:])))


def test_schedule_warm_start_regrouping(vc, orc):
    """Cheaper regrouping on the schedule: step 0 groups from the seeds
    (5 iterations), steps 1..12 start from the previous step's centroids and
    run one iteration (vcattn_group_warm).  On two heads the labels, the
    permutation and the centroids equal the oracle's own warm chain at every
    regrouping step; attention on steps 0, 6, 12 and 13 meets the bars."""
    w = W.WORKLOADS["schedule"]
    sm = float(np.float32(w.sm_scale))
    Q0, K0, V0 = W.make_workload(w, device="cuda")
    qidx = W.evenly_spaced_queries(w.N)
    heads = (0, 39)
    cent, ocent, operm = None, {}, {}
    t_warm, t_cold = [], []
    for t in range(14):
        Q, K, V = (W.drift(x, t, w.seed + j) for j, x in enumerate((Q0, K0, V0)))
        if t < 13:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record()
            if t == 0:
                labels, perm, cent = vc.group(V, w.k, w.iters, centroids=True)
            else:
                labels, perm, cent = vc.group(V, w.k, 1, centroids=True, init=cent)
            e[1].record()
            if t > 0:
                e[2].record()
                vc.group(V, w.k, w.iters)
                e[3].record()
            torch.cuda.synchronize()
            if t > 0:
                t_warm.append(e[0].elapsed_time(e[1]))
                t_cold.append(e[2].elapsed_time(e[3]))
            for h in heads:
                Vb = _head_bits(V, h)
                if t == 0:
                    ol, oc = orc.kmeans(Vb, w.k, w.iters)
                else:
                    ol, oc = orc.kmeans(Vb, w.k, 1, init=ocent[h])
                ocent[h], operm[h] = oc, orc.stable_sort(ol, w.k)
                assert np.array_equal(labels[0, h].cpu().numpy(), ol[0]), (t, h)
                assert np.array_equal(perm[0, h].cpu().numpy(), operm[h][0]), (t, h)
                assert np.array_equal(cent[0, h].cpu().numpy(), oc[0]), (t, h)
        if t in (0, 6, 12, 13):
            pp = vc.prep(Q, K, V, perm)
            O32, L = vc.attn(pp, sm, out_f32=True)
            torch.cuda.synchronize()
            assert vc.last_device_error() == 0
            for h in heads:
                Qb, Kb, Vb = (_head_bits(x, h) for x in (Q, K, V))
                opp = orc.prep(Qb, Kb, Vb, operm[h])
                rel_d = _check_head(orc, O32[0, h].cpu().numpy(), L[0, h].cpu().numpy(), Qb, Kb, Vb,
                                    opp, sm, qidx, perm_h=operm[h][0])
                print("warm schedule step %2d head %2d: rel-L2 vs exact %.4f" % (t, h, rel_d))
    print("warm regrouping: %.3f ms per step (median of steps 1-12), cold 5 iterations %.3f ms"
          % (float(np.median(t_warm)), float(np.median(t_cold))))


def test_sparse_full_size(vc, orc):
    w = W.WORKLOADS["sparse"]
    sm = float(np.float32(w.sm_scale))
    Q, K, V = W.make_workload(w, device="cuda")
    mask = W.make_tile_mask(w.B, w.H, w.N, w.seed + 7)
    labels, perm = vc.group(V, w.k, w.iters)
    pp = vc.prep(Q, K, V, perm)
    O32, L = vc.attn(pp, sm, mask=mask.cuda(), out_f32=True)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    qidx = W.evenly_spaced_queries(w.N)
    views = pp.views()
    m = mask.numpy()
    for h in (0, 31):
        Qb, Kb, Vb = (_head_bits(t, h) for t in (Q, K, V))
        ol, _ = orc.kmeans(Vb, w.k, w.iters)
        op = orc.stable_sort(ol, w.k)
        assert np.array_equal(labels[0, h].cpu().numpy(), ol[0])
        assert np.array_equal(perm[0, h].cpu().numpy(), op[0])
        opp = orc.prep(Qb, Kb, Vb, op)
        for key in ("k8", "r8t", "k_scale", "v_scale", "v_mean"):
            assert np.array_equal(views[key][h].cpu().numpy(), opp[key][0]), key
        _check_head(orc, O32[0, h].cpu().numpy(), L[0, h].cpu().numpy(), Qb, Kb, Vb, opp, sm, qidx,
                    mask_h=m[0, h], perm_h=op[0])


def test_sparse_beyond_kept_bitmask(vc, orc):
    """A sequence longer than the kernel's shared-memory bitmask of kept
    blocks (112 words per query tile, 3584 blocks): blocks past it are read
    from the mask itself.  One query tile keeps only blocks past the bitmask
    (among them the partial last block of the sequence), one only blocks
    before it, one straddles it; the sampled rows of every kind match both
    oracles."""
    N, H, k = 245000, 1, 64
    w = W.WORKLOADS["sparse"]
    sm = float(np.float32(w.sm_scale))
    Q, K, V = W.make_qkv(1, H, N, k, 1450, device="cuda")
    nq, nbp = (N + 63) // 64, vc.npad(N) // 64
    assert nbp > 32 * 112
    mask = W.make_tile_mask(1, H, N, 1451)
    m = mask.numpy()
    m[0, 0, 1, :] = 0
    m[0, 0, 1, [3600, 3650, 3700, (N - 1) // 64]] = 1   # only past the bitmask; the last block is partial
    m[0, 0, 2, :] = 0
    m[0, 0, 2, [5, 700, 3583]] = 1                       # only before it
    m[0, 0, 3, :] = 0
    m[0, 0, 3, [3000, 3583, 3584, 3800]] = 1             # across it
    mask = torch.from_numpy(m)
    labels, perm = vc.group(V, k, 5)
    pp = vc.prep(Q, K, V, perm)
    O32, L = vc.attn(pp, sm, mask=mask.cuda(), out_f32=True)
    torch.cuda.synchronize()
    assert vc.last_device_error() == 0
    qidx = np.unique(np.concatenate([W.evenly_spaced_queries(N), [64, 100, 127, 128, 191, 192, 255]]))
    Qb, Kb, Vb = (_head_bits(t, 0) for t in (Q, K, V))
    ol, _ = orc.kmeans(Vb, k, 5)
    op = orc.stable_sort(ol, k)
    assert np.array_equal(perm[0, 0].cpu().numpy(), op[0])
    opp = orc.prep(Qb, Kb, Vb, op)
    _check_head(orc, O32[0, 0].cpu().numpy(), L[0, 0].cpu().numpy(), Qb, Kb, Vb, opp, sm, qidx,
                mask_h=m[0, 0], perm_h=op[0])
