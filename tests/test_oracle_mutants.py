"""Planted mistakes in the CPU oracle must fail its pins.

Each mutant below is a copy of oracle/vcattn_oracle.c with one plausible slip
(a dropped term, a wrong sign, constant, divisor, order or index), compiled
here with gcc like the oracle itself.  The fast pins of
tests/test_oracle_pins.py then run against it in a child process, and at
least one of them has to fail.  This checks that the pins would notice such a
mistake in the oracle; it runs on the CPU only and loads nothing of the CUDA
path.  The slow Proposition 3.1 pins are left out of the child runs to keep
the suite short; every mutant here is caught without them.
"""
import concurrent.futures as cf
import os
import subprocess
import sys

import pytest

from oracle import build as ob

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")
FAST = "not prop31"

# (name, text in the oracle source, its replacement); each text occurs once.
MUTANTS = [
    # E4M3 codec
    ("decode exponent bias", "v = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("encode rounds half up", "double r = rint(mant * 8.0);",
     "double r = floor(mant * 8.0 + 0.5);"),
    ("encode subnormal step", "double q = rint(a * 512.0);", "double q = rint(a * 256.0);"),
    ("tie detector", "double q = (ldexp(a, -e) - 1.0) * 8.0;\n  return q - floor(q) == 0.5;",
     "double q = (ldexp(a, -e) - 1.0) * 8.0;\n  return q - floor(q) == 0.25;"),
    # ExpCast
    ("expcast flush threshold", "if (!(k >= 8.0f)) return 0;", "if (!(k >= 7.0f)) return 0;"),
    ("expcast clip", "if (k > 126.0f) k = 126.0f;", "if (k > 127.0f) k = 127.0f;"),
    ("expcast centring constant", "return (log2(1.5) - 0.5) / 2.0;", "return (log2(1.5) - 0.5);"),
    ("expcast rounds half up", "float k = rintf(t);", "float k = floorf(t + 0.5f);"),
    # k-means
    ("kmeans tie to highest cluster", "if (sc > bs) { bs = sc; best = c; }",
     "if (sc >= bs) { bs = sc; best = c; }"),
    ("kmeans full norm", "    h[c] = 0.5f * acc;\n  }\n  for (int64_t j = 0; j < N; ++j) {\n    const float* vj",
     "    h[c] = acc;\n  }\n  for (int64_t j = 0; j < N; ++j) {\n    const float* vj"),
    ("kmeans mean divisor", "cent[c * ORC_D + d] = total[c * ORC_D + d] / n;",
     "cent[c * ORC_D + d] = total[c * ORC_D + d] / (n + 1.0f);"),
    ("kmeans empty cluster divides", "if (count[c] == 0) continue;", "if (count[c] < 0) continue;"),
    ("kmeans seed index", "int64_t j = ((int64_t)c * N) / k;", "int64_t j = ((int64_t)c * (N - 1)) / k;"),
    # stable sort
    ("sort not stable", "for (int64_t j = 0; j < N; ++j) p[start[lab[j]]++] = (int32_t)j;",
     "for (int64_t j = N - 1; j >= 0; --j) p[start[lab[j]]++] = (int32_t)j;"),
    # preprocessing
    ("K centred with the wrong sign", "xf[j * ORC_D + d] = bf16_to_f32(kk[src * ORC_D + d]) - km[d];",
     "xf[j * ORC_D + d] = bf16_to_f32(kk[src * ORC_D + d]) + km[d];"),
    ("K mean divisor", "km[d] = tree_sum_f32(tmp, P) / (float)N;", "km[d] = tree_sum_f32(tmp, P) / (float)(N + 1);"),
    ("V block mean over a full block", "vm[b * ORC_D + d] = tree_sum_f32(col, ORC_BLK) / (float)rows;",
     "vm[b * ORC_D + d] = tree_sum_f32(col, ORC_BLK) / (float)ORC_BLK;"),
    ("V residual not demeaned",
     "xf[j * ORC_D + d] = xf[j * ORC_D + d] - vm[(j / ORC_BLK) * ORC_D + d];",
     "xf[j * ORC_D + d] = xf[j * ORC_D + d] - 0.0f * vm[(j / ORC_BLK) * ORC_D + d];"),
    ("V gathered without the permutation",
     "for (int d = 0; d < ORC_D; ++d) xf[j * ORC_D + d] = bf16_to_f32(vv[src * ORC_D + d]);",
     "for (int d = 0; d < ORC_D; ++d) xf[j * ORC_D + d] = bf16_to_f32(vv[j * ORC_D + d]);"),
    ("quantiser scale", "*scale = amax / 448.0f;", "*scale = amax / 240.0f;"),
    ("qmu sign", "acc = fmaf(xf[j * ORC_D + d], km[d], acc);", "acc = fmaf(xf[j * ORC_D + d], -km[d], acc);"),
    # emulating attention
    ("rank-one mean term dropped", "for (int d = 0; d < ORC_D; ++d) acc[d] += lh[h] * (double)mu[d];",
     "for (int d = 0; d < ORC_D; ++d) acc[d] += 0.0 * lh[h] * (double)mu[d];"),
    ("rescale exponent", "exp2(((double)m_run - (double)m_tile) / 8.0)",
     "exp2(((double)m_run - (double)m_tile) / 4.0)"),
    ("row sum of one half only", "l += lh[0] + lh[1];", "l += lh[0];"),
    ("tile max without the coefficient", "if (kept[h]) m_tile = fmaxf(m_tile, A[h] * mx[h]);",
     "if (kept[h]) m_tile = fmaxf(m_tile, mx[h]);"),
    ("mask ignored", "if (mask == NULL || (qt < nq64 && mask[qt * nbp + b] != 0)) own[no++] = b;",
     "if (1) own[no++] = b;"),
    ("lse2 offset sign", "lse2[qi] = (double)m_run / 8.0 - off + log2(l)",
     "lse2[qi] = (double)m_run / 8.0 + off + log2(l)"),
    ("lse2 without the query mean term",
     "+ (double)qmu[i] * (double)sm_scale * 1.4426950408889634;",
     "+ 0.0 * (double)qmu[i] * (double)sm_scale * 1.4426950408889634;"),
    # dense attention
    ("dense without the softmax scale", "s[j] = dot * (double)sm_scale;", "s[j] = dot;"),
    ("dense mask transposed", "mask[(i / ORC_BLK) * nbp + p / ORC_BLK]", "mask[(p / ORC_BLK) * nbp + i / ORC_BLK]"),
    ("dense LSE in natural log", "lse2[qi] = (mx + log(l)) * 1.4426950408889634;", "lse2[qi] = (mx + log(l));"),
    ("emulated ExpCast constant", "const float C = (float)(56.0 + 8.0 * off - 8.0 * orc_expcast_cstar());",
     "const float C = (float)(56.0 + 8.0 * off + 8.0 * orc_expcast_cstar());"),
    ("score coefficient without the softmax scale",
     "const float c0 = (float)(8.0 * 1.4426950408889634 * (double)sm_scale);",
     "const float c0 = (float)(8.0 * 1.4426950408889634);"),
    ("keys past N kept", "valid[jj] = kept[h] && (j < N);", "valid[jj] = kept[h];"),
    ("empty row LSE", "lse2[qi] = -INFINITY;\n    }\n  }\n  return 0;", "lse2[qi] = 0.0;\n    }\n  }\n  return 0;"),
    # tree sums, k-means partials, zero-block rule
    ("tree sum reads the first half twice", "float b = tree_sum_f32(x + h, h);", "float b = tree_sum_f32(x, h);"),
    ("chunk partials not reset", "memset(part, 0, (size_t)k * ORC_D * sizeof(float));", ";"),
    ("zero-block rule dropped", "if (!(amax >= AMAX_FLOOR)) {\n    for (int64_t r",
     "if (!(amax >= 0.0f)) {\n    for (int64_t r"),
    # QK Hadamard
    ("butterfly sign", "x[i + h] = a - b;", "x[i + h] = b - a;"),
    ("K rotation scale", "xf[j * ORC_D + d] *= 0.125f;", "xf[j * ORC_D + d] *= 0.0625f;"),
    ("Q rotation scale", "for (int d = 0; d < ORC_D; ++d) xf[j * ORC_D + d] *= 0.0625f;",
     "for (int d = 0; d < ORC_D; ++d) xf[j * ORC_D + d] *= 0.125f;"),
]


def _run_pins(lib):
    env = dict(os.environ, OMP_NUM_THREADS="1", OMP_WAIT_POLICY="passive")
    env[ob.ENV_LIB] = lib
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider", "-k", FAST],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-2000:]


@pytest.fixture(scope="module")
def libs(tmp_path_factory):
    """The unmodified source and every mutant, compiled side by side."""
    d = tmp_path_factory.mktemp("oracle_mutants")
    src = open(ob.SRC).read()
    jobs = [("original", src)]
    for name, old, new in MUTANTS:
        assert src.count(old) == 1, name
        jobs.append((name, src.replace(old, new)))

    def compile_one(i_job):
        i, (name, text) = i_job
        c = os.path.join(str(d), "m%02d.c" % i)
        so = os.path.join(str(d), "m%02d.so" % i)
        with open(c, "w") as f:
            f.write(text)
        ob.compile_oracle(c, so)
        return name, so

    with cf.ThreadPoolExecutor(8) as ex:
        return dict(ex.map(compile_one, enumerate(jobs)))


def test_unmodified_oracle_passes_the_fast_pins(libs):
    rc, out = _run_pins(libs["original"])
    assert rc == 0, out


def test_every_planted_mistake_fails_a_pin(libs):
    names = [m[0] for m in MUTANTS]
    with cf.ThreadPoolExecutor(max(2, min(8, os.cpu_count() or 2))) as ex:
        results = dict(zip(names, ex.map(lambda n: _run_pins(libs[n]), names)))
    # exit status 1: tests ran and at least one failed (not a crash or an
    # error in collecting them)
    survivors = {n: out for n, (rc, out) in results.items() if rc != 1}
    assert not survivors, "\n\n".join("%s (exit %d):\n%s" % (n, results[n][0], o) for n, o in survivors.items())
