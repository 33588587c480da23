"""CPU oracle for the smoothed FP8 attention forward (test infrastructure).

A plain, slow implementation in C (``vcattn_oracle.c``) of what the GPU path
computes, plus this ctypes wrapper.  Only ``tests/``, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py`` may import it; the product path never
does.  It shares no code with the CUDA path.

bf16 tensors cross this interface as ``numpy.uint16`` bit patterns with shape
``[BH, N, 128]``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _L():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_float
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [f32]
        lib.orc_e4m3_encode_n.argtypes = [P, P, i64]
        lib.orc_e4m3_decode_n.argtypes = [P, P, i64]
        lib.orc_e4m3_is_tie.argtypes = [f32]
        lib.orc_e4m3_is_tie.restype = i32
        lib.orc_expcast_cstar.restype = ctypes.c_double
        lib.orc_expcast_n.argtypes = [P, f32, f32, P, i64]
        lib.orc_expcast_v.argtypes = [P, P, P, P, i64]
        lib.orc_tree_sum.argtypes = [P, i64]
        lib.orc_tree_sum.restype = f32
        lib.orc_kmeans.argtypes = [P, i64, i64, i32, i32, P, P]
        lib.orc_kmeans_from.argtypes = [P, i64, i64, i32, i32, P, P, P]
        lib.orc_kmeans_scores.argtypes = [P, i64, P, i32, P]
        lib.orc_stable_sort.argtypes = [P, i64, i64, i32, P]
        lib.orc_prep.argtypes = [P, P, P, P, i64, i64] + [P] * 9
        lib.orc_prep_ex.argtypes = [P, P, P, P, i64, i64, i32] + [P] * 9
        lib.orc_prep_ties.argtypes = [P, P, P, P, i64, i64, i32] + [P] * 10
        lib.orc_hadamard128.argtypes = [P, P, i64]
        lib.orc_attn_emul.argtypes = [P] * 8 + [i64, f32, i32, f32, P, P, i64, i32, P, P]
        lib.orc_attn_dense.argtypes = [P, P, P, i64, f32, P, P, P, i64, P, P]
        _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


NPAD_TILE = 128
BLOCK = 64
D = 128


def npad(n):
    return ((n + NPAD_TILE - 1) // NPAD_TILE) * NPAD_TILE


def e4m3_encode(x):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _L().orc_e4m3_encode_n(_p(x), _p(out), x.size)
    return out


def e4m3_decode(c):
    c = _c(c, np.uint8)
    out = np.empty(c.shape, np.float64)
    _L().orc_e4m3_decode_n(_p(c), _p(out), c.size)
    return out


def e4m3_is_tie(x):
    x = _c(x, np.float32).ravel()
    return np.array([_L().orc_e4m3_is_tie(float(v)) for v in x], dtype=bool)


def cstar():
    """Minimax centring constant of the ExpCast byte (in log2 units)."""
    return _L().orc_expcast_cstar()


def expcast_C(off):
    """Constant term C = 56 + 8*off - 8*c*, rounded to FP32."""
    return float(np.float32(56.0 + 8.0 * off - 8.0 * cstar()))


def expcast(x, A, B):
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _L().orc_expcast_n(_p(x), float(A), float(B), _p(out), x.size)
    return out


def expcast_v(x, A, B):
    """ExpCast bytes with a coefficient A[i] and constant B[i] per score."""
    x, A, B = (_c(t, np.float32) for t in (x, A, B))
    if not (x.shape == A.shape == B.shape):
        raise ValueError("x, A and B must have one shape")
    out = np.empty(x.shape, np.uint8)
    _L().orc_expcast_v(_p(x), _p(A), _p(B), _p(out), x.size)
    return out


def tree_sum(x):
    x = _c(x, np.float32)
    return np.float32(_L().orc_tree_sum(_p(x), x.size))


def kmeans(V, k, iters, init=None):
    """V: uint16 [BH, N, 128] -> labels int32 [BH, N], centroids f32 [BH, k, 128].
    init: None (c_c = v[floor(c N / k)]) or starting centroids f32 [BH, k, 128]."""
    V = _c(V, np.uint16)
    BH, N, _ = V.shape
    labels = np.empty((BH, N), np.int32)
    cent = np.empty((BH, k, D), np.float32)
    ini = None if init is None else _c(init, np.float32)
    if ini is not None and ini.shape != (BH, k, D):
        raise ValueError("init must be [BH, k, 128]")
    rc = _L().orc_kmeans_from(_p(V), BH, N, k, iters, _p(ini), _p(labels), _p(cent))
    if rc:
        raise ValueError("orc_kmeans: bad arguments")
    return labels, cent


def kmeans_scores(V_head, cent_head):
    V_head = _c(V_head, np.uint16)
    cent_head = _c(cent_head, np.float32)
    N, k = V_head.shape[0], cent_head.shape[0]
    out = np.empty((N, k), np.float32)
    _L().orc_kmeans_scores(_p(V_head), N, _p(cent_head), k, _p(out))
    return out


def stable_sort(labels, k):
    labels = _c(labels, np.int32)
    BH, N = labels.shape
    perm = np.empty((BH, N), np.int32)
    if _L().orc_stable_sort(_p(labels), BH, N, k, _p(perm)):
        raise ValueError("orc_stable_sort: label out of range")
    return perm


PREP_QK_HADAMARD = 1


def hadamard128(x):
    """The fixed-order FP32 butterfly of the QK rotation, row by row:
    float32 [rows, 128] -> x H (H the 128-point Sylvester-Hadamard matrix)."""
    x = _c(x, np.float32).reshape(-1, D)
    y = np.empty_like(x)
    _L().orc_hadamard128(_p(x), _p(y), x.shape[0])
    return y


def prep(Q, K, V, perm=None, flags=0, count_ties=False):
    """Preprocessing of all heads.  Returns a dict of numpy arrays:
    q8, k8 [BH, Npad, 128] u8; r8t [BH, 128, Npad] u8; q_scale, k_scale
    [BH, Npad/64]; v_scale, k_mean [BH, 128]; v_mean [BH, Npad/64, 128]; qmu [BH, N].
    flags & PREP_QK_HADAMARD: Q and centred K rotated by the Hadamard transform
    before their quantisers.  count_ties: also "ties" [BH, 3] int64, the E4M3
    rounding ties among the quantiser inputs of Q, K and the V residual."""
    Q, K, V = (_c(t, np.uint16) for t in (Q, K, V))
    BH, N, _ = Q.shape
    Np = npad(N)
    nbp = Np // BLOCK
    out = dict(
        q8=np.empty((BH, Np, D), np.uint8), k8=np.empty((BH, Np, D), np.uint8),
        r8t=np.empty((BH, D, Np), np.uint8),
        q_scale=np.empty((BH, nbp), np.float32), k_scale=np.empty((BH, nbp), np.float32),
        v_scale=np.empty((BH, D), np.float32), k_mean=np.empty((BH, D), np.float32),
        v_mean=np.empty((BH, nbp, D), np.float32), qmu=np.empty((BH, N), np.float32))
    if perm is not None:
        perm = _c(perm, np.int32)
    args = (_p(Q), _p(K), _p(V), _p(perm), BH, N, int(flags),
            _p(out["q8"]), _p(out["k8"]), _p(out["r8t"]),
            _p(out["q_scale"]), _p(out["k_scale"]), _p(out["v_scale"]),
            _p(out["k_mean"]), _p(out["v_mean"]), _p(out["qmu"]))
    if count_ties:
        out["ties"] = np.zeros((BH, 3), np.int64)
        rc = _L().orc_prep_ties(*args, _p(out["ties"]))
    else:
        rc = _L().orc_prep_ex(*args)
    if rc:
        raise ValueError("orc_prep: bad arguments")
    return out


def attn_emul(pp, h, N, sm_scale, qidx=None, off=8, tau8=0.0, mask=None, flags=0):
    """Emulating attention for head h of a prep() result.  Returns
    (O [nq, 128] f64, lse2 [nq] f64)."""
    qidx = np.arange(N, dtype=np.int64) if qidx is None else _c(qidx, np.int64)
    nq = qidx.size
    O = np.empty((nq, D), np.float64)
    lse = np.empty(nq, np.float64)
    hs = {k: np.ascontiguousarray(v[h]) for k, v in pp.items()}
    m = None if mask is None else _c(mask, np.uint8)
    _L().orc_attn_emul(_p(hs["q8"]), _p(hs["k8"]), _p(hs["r8t"]), _p(hs["q_scale"]),
                       _p(hs["k_scale"]), _p(hs["v_scale"]), _p(hs["v_mean"]), _p(hs["qmu"]),
                       N, float(sm_scale), int(off), float(tau8), _p(m), _p(qidx), nq, int(flags),
                       _p(O), _p(lse))
    return O, lse


def attn_dense(Qh, Kh, Vh, sm_scale, qidx=None, mask=None, perm=None):
    """Exact FP64 attention for one head (uint16 [N, 128] each)."""
    Qh, Kh, Vh = (_c(t, np.uint16) for t in (Qh, Kh, Vh))
    N = Qh.shape[0]
    qidx = np.arange(N, dtype=np.int64) if qidx is None else _c(qidx, np.int64)
    nq = qidx.size
    O = np.empty((nq, D), np.float64)
    lse = np.empty(nq, np.float64)
    m = None if mask is None else _c(mask, np.uint8)
    p = None if perm is None else _c(perm, np.int32)
    _L().orc_attn_dense(_p(Qh), _p(Kh), _p(Vh), N, float(sm_scale), _p(m), _p(p), _p(qidx), nq,
                        _p(O), _p(lse))
    return O, lse


def threads():
    """OpenMP threads the oracle uses (OMP_NUM_THREADS or the core count)."""
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v else (os.cpu_count() or 1)
