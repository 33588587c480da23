"""CPU checks of the error bounds that make the tensor-core k-means assignment
exact (csrc/km_tc.cu).

The assignment keeps every cluster whose approximate score T_c is within E of
the best one, with E = (2^-13 + 2^-21)(|v| max|c| + max|h|), and decides among
several survivors with FP32 sums in eight interleaved partials, bound E2 =
2^-15 (|v| max|c| + max|h|), before the exact fmaf chains.  Both filters are
exact as long as every approximation is within half its bound of the FP32
chain score.  Here the tensor core's accumulation is modelled at its worst:
the 272 exact products added one by one in FP32, in an adversarial order,
with every add rounded toward zero (or to nearest).  The chain and the
eight-partial sums are emulated exactly (FP64 products, FP32 rounding after
each fma)."""
import numpy as np
import pytest

D = 128
E_COEF = 2.0 ** -13 + 2.0 ** -21
E2_COEF = 2.0 ** -15


def f32(x):
    return np.float32(x)


def fma32(a, b, c):
    # a*b is exact in float64 (two 24-bit mantissas); the sum is rounded once
    # to float32, the double rounding through float64 is far below the bounds
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def bf16(x):
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16  # round to nearest even
    return r.astype(np.uint32).view(np.float32)


def chain_dot(v, c):
    acc = np.float32(0.0)
    for d in range(D):
        acc = fma32(v[d], c[d], acc)
    return acc


def tree8_dot(v, c):
    a = [np.float32(0.0)] * 8
    for d in range(D):
        a[d & 7] = fma32(v[d], c[d], a[d & 7])
    return f32(f32(f32(a[0] + a[1]) + f32(a[2] + a[3])) + f32(f32(a[4] + a[5]) + f32(a[6] + a[7])))


def fp32_add(acc, p, toward_zero):
    s = np.float64(acc) + np.float64(p)
    r = np.float32(s)
    if toward_zero and abs(np.float64(r)) > abs(s):
        r = np.nextafter(r, np.float32(0.0), dtype=np.float32)
    return r


def tc_worst(v, c, h, toward_zero, order):
    hi = bf16(c)
    lo = bf16(c - hi)
    h1 = bf16(np.float32(h))
    h2 = bf16(np.float32(h - h1))
    h3 = bf16(np.float32(h - h1 - h2))
    terms = np.concatenate([v.astype(np.float64) * hi, v.astype(np.float64) * lo, -np.array([h1, h2, h3], np.float64)])
    if order == "ascending":
        terms = terms[np.argsort(np.abs(terms))]
    elif order == "descending":
        terms = terms[np.argsort(-np.abs(terms))]
    acc = np.float32(0.0)
    for p in terms:
        acc = fp32_add(acc, p, toward_zero)
    return acc


def _case(seed, scale_v, scale_c, k=16):
    rng = np.random.default_rng(seed)
    v = bf16(rng.standard_normal(D).astype(np.float32) * scale_v)
    cent = (rng.standard_normal((k, D)) * scale_c).astype(np.float32)
    cent[1] = cent[0]                       # an exact tie
    cent[3] = cent[2] + np.float32(1e-3)     # a near tie
    cent[5] = bf16(v)                        # the token itself
    h = np.array([np.float32(0.5) * chain_dot(cc, cc) for cc in cent], np.float32)
    return v, cent, h


@pytest.mark.parametrize("seed,scale_v,scale_c", [(1, 1.0, 1.0), (2, 3.0, 0.5), (3, 0.01, 40.0), (4, 200.0, 200.0)])
def test_tensor_core_score_within_half_bound(seed, scale_v, scale_c):
    v, cent, h = _case(seed, scale_v, scale_c)
    vn = float(np.sqrt(np.sum(v.astype(np.float64) ** 2)))
    cmax = max(float(np.sqrt(np.sum(cc.astype(np.float64) ** 2))) for cc in cent)
    hmax = float(np.max(np.abs(h)))
    E = E_COEF * (vn * cmax + hmax)
    E2 = E2_COEF * (vn * cmax + hmax)
    for ci, cc in enumerate(cent):
        score = f32(chain_dot(v, cc) - h[ci])
        for tz in (True, False):
            for order in ("given", "ascending", "descending"):
                T = tc_worst(v, cc, h[ci], tz, order)
                assert abs(np.float64(T) - np.float64(score)) <= E / 2, (ci, tz, order)
        s8 = f32(tree8_dot(v, cc) - h[ci])
        assert abs(np.float64(s8) - np.float64(score)) <= E2 / 2, ci


def test_filter_keeps_the_winner():
    """With T within E/2 of the chain score, the chain's winner (lowest index
    among equal scores) always survives the threshold max T - E."""
    for seed in range(20):
        v, cent, h = _case(100 + seed, 1.0 + seed, 1.0)
        scores = np.array([f32(chain_dot(v, cc) - h[i]) for i, cc in enumerate(cent)])
        win = int(np.argmax(scores))  # first maximal index, the oracle's rule
        T = np.array([tc_worst(v, cc, h[i], True, "ascending") for i, cc in enumerate(cent)])
        vn = float(np.sqrt(np.sum(v.astype(np.float64) ** 2)))
        cmax = max(float(np.sqrt(np.sum(cc.astype(np.float64) ** 2))) for cc in cent)
        E = E_COEF * (vn * cmax + float(np.max(np.abs(h))))
        survivors = np.nonzero(T >= T.max() - E)[0]
        assert win in survivors
        assert 0 in survivors and 1 in survivors or win not in (0, 1)  # the exact tie survives together
