"""Python binding of libvcattn.so (ctypes; argument marshalling only).

Every step of the path runs in the library's CUDA kernels; this module only
allocates the caller-side buffers with PyTorch, passes pointers and the
current CUDA stream, and turns status codes into exceptions.  There is no
fallback: if the library is missing or the device is not sm_103a, calls fail.

Names follow the C ABI in include/vcattn.h: ``group``, ``prep``, ``attn``,
``fwd``, ``last_device_error``.
"""
import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = _build.LIB

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(6)


class VcattnError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        msg = "%s: %s (status %d)" % (what, _lib().vcattn_status_string(status).decode(), status)
        if status == ERR_CUDA:
            msg += ": " + _lib().vcattn_last_cuda_error().decode()
        super().__init__(msg)


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("H", ctypes.c_int64), ("N", ctypes.c_int64),
                ("D", ctypes.c_int64)]


class Strides(ctypes.Structure):
    """vcattn_strides: element strides of the batch, head and token dims."""
    _fields_ = [("b", ctypes.c_int64), ("h", ctypes.c_int64), ("n", ctypes.c_int64)]


class PreppedStruct(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("q8", "k8", "r8t", "q_scale", "k_scale", "v_scale", "k_mean", "v_mean", "qmu",
                 "vmu_op")]


_L = None


def _lib():
    global _L
    if _L is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libvcattn.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        P, SP, sz, st = ctypes.c_void_p, ctypes.POINTER(Shape), ctypes.c_size_t, ctypes.c_int
        PP = ctypes.POINTER(PreppedStruct)
        lib.vcattn_npad.restype = ctypes.c_int64
        lib.vcattn_npad.argtypes = [ctypes.c_int64]
        lib.vcattn_group_workspace_bytes.restype = sz
        lib.vcattn_group_workspace_bytes.argtypes = [SP, ctypes.c_int]
        lib.vcattn_group.restype = st
        lib.vcattn_group.argtypes = [SP, P, ctypes.c_int, ctypes.c_int, P, P, P, P, sz, P]
        lib.vcattn_group_warm.restype = st
        lib.vcattn_group_warm.argtypes = [SP, P, ctypes.c_int, ctypes.c_int, P, P, P, P, P, sz, P]
        SS = ctypes.POINTER(Strides)
        lib.vcattn_group_strided.restype = st
        lib.vcattn_group_strided.argtypes = [SP, P, SS, ctypes.c_int, ctypes.c_int, P, P, P, P, P, sz, P]
        lib.vcattn_prep_strided.restype = st
        lib.vcattn_prep_strided.argtypes = [SP, P, SS, P, SS, P, SS, P, ctypes.POINTER(PreppedStruct), P, sz, P]
        lib.vcattn_attn_strided.restype = st
        lib.vcattn_attn_strided.argtypes = [SP, ctypes.POINTER(PreppedStruct), ctypes.c_float, ctypes.c_int,
                                            ctypes.c_float, ctypes.c_int, P, P, SS, P, P]
        lib.vcattn_prep_ex.restype = st
        lib.vcattn_prep_ex.argtypes = [SP, P, SS, P, SS, P, SS, P, ctypes.c_int, ctypes.POINTER(PreppedStruct),
                                       P, sz, P]
        lib.vcattn_prepped_bytes.restype = sz
        lib.vcattn_prepped_bytes.argtypes = [SP]
        lib.vcattn_prepped_carve.restype = st
        lib.vcattn_prepped_carve.argtypes = [SP, P, sz, PP]
        lib.vcattn_prep_workspace_bytes.restype = sz
        lib.vcattn_prep_workspace_bytes.argtypes = [SP]
        lib.vcattn_prep.restype = st
        lib.vcattn_prep.argtypes = [SP, P, P, P, P, PP, P, sz, P]
        lib.vcattn_attn.restype = st
        lib.vcattn_attn.argtypes = [SP, PP, ctypes.c_float, P, P, P, P]
        lib.vcattn_attn_ex.restype = st
        lib.vcattn_attn_ex.argtypes = [SP, PP, ctypes.c_float, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                       P, P, P, P]
        lib.vcattn_fwd_workspace_bytes.restype = sz
        lib.vcattn_fwd_workspace_bytes.argtypes = [SP]
        lib.vcattn_fwd.restype = st
        lib.vcattn_fwd.argtypes = [SP, P, P, P, P, ctypes.c_float, P, P, P, P, sz, P]
        lib.vcattn_fwd_host_workspace_bytes.restype = sz
        lib.vcattn_fwd_host_workspace_bytes.argtypes = [SP, ctypes.c_int, ctypes.c_int]
        lib.vcattn_fwd_host.restype = st
        lib.vcattn_fwd_host.argtypes = [SP, P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_float, P, P, P,
                                        ctypes.c_int, P, sz, ctypes.POINTER(P)]
        lib.vcattn_last_device_error.restype = st
        lib.vcattn_last_device_error.argtypes = [P]
        lib.vcattn_status_string.restype = ctypes.c_char_p
        lib.vcattn_status_string.argtypes = [st]
        lib.vcattn_last_cuda_error.restype = ctypes.c_char_p
        lib.vcattn_last_cuda_error.argtypes = []
        _L = lib
    return _L


def lib():
    """The loaded ctypes library (raw C ABI)."""
    return _lib()


def _check(status, what):
    if status != OK:
        raise VcattnError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _shape(x):
    B, H, N, D = x.shape
    return Shape(B, H, N, D)


def _req(x, dtype, name):
    if not (x.is_cuda and x.dtype == dtype and x.is_contiguous()):
        raise ValueError("%s must be a contiguous CUDA %s tensor" % (name, dtype))


def _req_mask(mask, B, H, N):
    """A tile mask is u8 [B, H, ceil(N/64), Npad/64] on the GPU, contiguous."""
    _req(mask, torch.uint8, "mask")
    want = (int(B), int(H), (int(N) + 63) // 64, npad(int(N)) // 64)
    if tuple(mask.shape) != want:
        raise ValueError("mask must have shape %s, got %s" % (want, tuple(mask.shape)))


def _rows(x, dtype, name):
    """None for a contiguous [B,H,N,128] tensor, else its Strides (channels
    contiguous, e.g. a (B,N,H,D) tensor viewed as (B,H,N,D) by transpose(1, 2))."""
    if not (x.is_cuda and x.dtype == dtype and x.dim() == 4 and x.shape[-1] == 128):
        raise ValueError("%s must be a CUDA %s tensor [B, H, N, 128]" % (name, dtype))
    if x.is_contiguous():
        return None
    if x.stride(3) != 1:
        raise ValueError("%s: the 128 channels must be contiguous" % name)
    return Strides(x.stride(0), x.stride(1), x.stride(2))


def npad(N):
    return int(_lib().vcattn_npad(N))


def group(V, k, iters=5, centroids=False, stream=None, init=None):
    """k-means labels and the stable-sort permutation of V [B,H,N,128] bf16.
    Returns (labels, perm[, centroids]) as int32 [B,H,N] (and f32 [B,H,k,128]).
    init: starting centroids f32 [B,H,k,128] (vcattn_group_warm) instead of
    the evenly spaced seeds."""
    sv = _rows(V, torch.bfloat16, "V")
    if init is not None:
        _req(init, torch.float32, "init")
        if tuple(init.shape) != (V.shape[0], V.shape[1], k, 128):
            raise ValueError("init must be [B, H, k, 128]")
    s = _shape(V)
    B, H, N, _ = V.shape
    labels = torch.empty(B, H, N, dtype=torch.int32, device=V.device)
    perm = torch.empty_like(labels)
    cent = torch.empty(B, H, k, 128, dtype=torch.float32, device=V.device) if centroids else None
    nbytes = _lib().vcattn_group_workspace_bytes(ctypes.byref(s), k)
    if nbytes == 0:
        raise ValueError("unsupported grouping shape or k")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=V.device)
    if sv is not None:
        _check(_lib().vcattn_group_strided(ctypes.byref(s), _ptr(V), ctypes.byref(sv), k, iters, _ptr(init),
                                           _ptr(labels), _ptr(perm), _ptr(cent), _ptr(ws), nbytes,
                                           _stream(stream)), "vcattn_group_strided")
    elif init is None:
        _check(_lib().vcattn_group(ctypes.byref(s), _ptr(V), k, iters, _ptr(labels), _ptr(perm),
                                   _ptr(cent), _ptr(ws), nbytes, _stream(stream)), "vcattn_group")
    else:
        _check(_lib().vcattn_group_warm(ctypes.byref(s), _ptr(V), k, iters, _ptr(init), _ptr(labels),
                                        _ptr(perm), _ptr(cent), _ptr(ws), nbytes, _stream(stream)),
               "vcattn_group_warm")
    return (labels, perm, cent) if centroids else (labels, perm)


class Prepped:
    """Owner of the prepped buffer (one torch allocation) plus views of its parts."""

    def __init__(self, shape_tuple, device):
        B, H, N, D = shape_tuple
        self.shape = Shape(B, H, N, D)
        self.nbytes = _lib().vcattn_prepped_bytes(ctypes.byref(self.shape))
        if self.nbytes == 0:
            raise ValueError("unsupported shape")
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)
        self.struct = PreppedStruct()
        _check(_lib().vcattn_prepped_carve(ctypes.byref(self.shape), _ptr(self.buf), self.nbytes,
                                           ctypes.byref(self.struct)), "vcattn_prepped_carve")

    def views(self):
        """Torch views of the prepped tensors (for tests)."""
        B, H, N = self.shape.B, self.shape.H, self.shape.N
        Np = npad(N)
        nbp = Np // 64
        base = self.buf.data_ptr()

        def v(name, shape, dtype):
            off = getattr(self.struct, name) - base
            n = 1
            for d in shape:
                n *= d
            esz = torch.empty((), dtype=dtype).element_size()
            return self.buf[off:off + n * esz].view(dtype).view(*shape)

        return dict(
            q8=v("q8", (B * H, Np, 128), torch.uint8), k8=v("k8", (B * H, Np, 128), torch.uint8),
            r8t=v("r8t", (B * H, 128, Np), torch.uint8),
            q_scale=v("q_scale", (B * H, nbp), torch.float32),
            k_scale=v("k_scale", (B * H, nbp), torch.float32),
            v_scale=v("v_scale", (B * H, 128), torch.float32),
            k_mean=v("k_mean", (B * H, 128), torch.float32),
            v_mean=v("v_mean", (B * H, nbp, 128), torch.float32),
            qmu=v("qmu", (B * H, N), torch.float32),
            vmu_op=v("vmu_op", (B * H, nbp, 128, 4), torch.float32))


PREP_QK_HADAMARD = 1


def prep(Q, K, V, perm=None, out=None, stream=None, hadamard=False):
    """Fused K mean, gather by perm, V block demean and Q/K/V quantisers.
    Q, K, V may be strided views (channels contiguous).  hadamard=True
    rotates Q and centred K by the 128-point Hadamard transform before their
    quantisers (vcattn_prep_ex with VCATTN_PREP_QK_HADAMARD)."""
    rows = [_rows(t, torch.bfloat16, n) for t, n in ((Q, "Q"), (K, "K"), (V, "V"))]
    if perm is not None:
        _req(perm, torch.int32, "perm")
    pp = out if out is not None else Prepped(tuple(Q.shape), Q.device)
    s = _shape(Q)
    nbytes = _lib().vcattn_prep_workspace_bytes(ctypes.byref(s))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=Q.device)
    if hadamard:
        st = [None if r is None else ctypes.byref(r) for r in rows]
        _check(_lib().vcattn_prep_ex(ctypes.byref(s), _ptr(Q), st[0], _ptr(K), st[1], _ptr(V), st[2],
                                     _ptr(perm), PREP_QK_HADAMARD, ctypes.byref(pp.struct), _ptr(ws), nbytes,
                                     _stream(stream)), "vcattn_prep_ex")
    elif all(r is None for r in rows):
        _check(_lib().vcattn_prep(ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V), _ptr(perm),
                                  ctypes.byref(pp.struct), _ptr(ws), nbytes, _stream(stream)),
               "vcattn_prep")
    else:
        B, H, N, D = Q.shape
        st = [r if r is not None else Strides(H * N * D, N * D, D) for r in rows]
        _check(_lib().vcattn_prep_strided(ctypes.byref(s), _ptr(Q), ctypes.byref(st[0]), _ptr(K),
                                          ctypes.byref(st[1]), _ptr(V), ctypes.byref(st[2]), _ptr(perm),
                                          ctypes.byref(pp.struct), _ptr(ws), nbytes, _stream(stream)),
               "vcattn_prep_strided")
    return pp


def attn(pp, sm_scale, mask=None, off=8, tau8=6.0, out_f32=False, O=None, lse2=None, want_lse=True,
         stream=None):
    """Attention forward from prepped tensors.  Returns (O [B,H,N,128] bf16, or f32 with
    out_f32, and lse2 f32 [B,H,N])."""
    B, H, N = pp.shape.B, pp.shape.H, pp.shape.N
    dev = pp.buf.device
    if O is None:
        O = torch.empty(B, H, N, 128, dtype=torch.float32 if out_f32 else torch.bfloat16, device=dev)
    if lse2 is None and want_lse:
        lse2 = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    if mask is not None:
        _req_mask(mask, B, H, N)
    so = _rows(O, torch.float32 if out_f32 else torch.bfloat16, "O")
    if so is None:
        _check(_lib().vcattn_attn_ex(ctypes.byref(pp.shape), ctypes.byref(pp.struct), float(sm_scale),
                                     int(off), float(tau8), int(bool(out_f32)), _ptr(mask), _ptr(O),
                                     _ptr(lse2),
                                     _stream(stream)), "vcattn_attn")
    else:
        _check(_lib().vcattn_attn_strided(ctypes.byref(pp.shape), ctypes.byref(pp.struct), float(sm_scale),
                                          int(off), float(tau8), int(bool(out_f32)), _ptr(mask), _ptr(O),
                                          ctypes.byref(so), _ptr(lse2), _stream(stream)), "vcattn_attn_strided")
    return O, lse2


def fwd(Q, K, V, perm, sm_scale, mask=None, O=None, lse2=None, ws=None, stream=None):
    """vcattn_fwd: prep into a workspace + attention, one call (contiguous
    tensors; strided ones go through prep() and attn())."""
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _req(t, torch.bfloat16, n)
    if perm is not None:
        _req(perm, torch.int32, "perm")
    if O is not None:
        _req(O, torch.bfloat16, "O")
    s = _shape(Q)
    if mask is not None:
        _req_mask(mask, s.B, s.H, s.N)
    nbytes = _lib().vcattn_fwd_workspace_bytes(ctypes.byref(s))
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=Q.device)
    if O is None:
        O = torch.empty_like(Q)
    if lse2 is None:
        lse2 = torch.empty(Q.shape[:3], dtype=torch.float32, device=Q.device)
    _check(_lib().vcattn_fwd(ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V), _ptr(perm), float(sm_scale),
                             _ptr(mask), _ptr(O), _ptr(lse2), _ptr(ws), ws.numel(), _stream(stream)),
           "vcattn_fwd")
    return O, lse2


class HostPipeline:
    """vcattn_fwd_host with its device workspace and three streams kept
    across calls: grouping, preprocessing and attention of host-resident
    Q, K, V (bf16 [B,H,N,128], ideally pinned) into host O (and lse2), the
    copies overlapped with the computation chunk by chunk."""

    def __init__(self, shape, k, iters=5, chunk_heads=0, device=None, dual=True):
        self.shape = Shape(*shape)
        self.k, self.iters, self.chunk_heads = int(k), int(iters), int(chunk_heads)
        self.device = torch.device("cuda") if device is None else torch.device(device)
        nbytes = _lib().vcattn_fwd_host_workspace_bytes(ctypes.byref(self.shape), self.k, self.chunk_heads)
        if nbytes == 0:
            raise VcattnError(ERR_INVALID_ARG, "vcattn_fwd_host_workspace_bytes")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        # compute 0, compute 1 (the same stream unless dual), copy in, copy out
        st = [torch.cuda.Stream(device=self.device) for _ in range(4 if dual else 3)]
        self.streams = [st[0], st[1] if dual else st[0]] + st[-2:]
        self._sp = (ctypes.c_void_p * 4)(*[s.cuda_stream for s in self.streams])

    @property
    def stream(self):
        """The stream that completes the call (synchronise it, or wait on it)."""
        return self.streams[0]

    def __call__(self, hQ, hK, hV, sm_scale, mask=None, hO=None, hlse2=None):
        for t, n in ((hQ, "hQ"), (hK, "hK"), (hV, "hV")):
            if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
                raise ValueError("%s must be a contiguous host bf16 tensor" % n)
        if hO is None:
            hO = torch.empty(hQ.shape, dtype=torch.bfloat16, pin_memory=True)
        if mask is not None:
            _req_mask(mask, self.shape.B, self.shape.H, self.shape.N)
        # the compute streams start after the caller's pending work
        for s in self.streams[:2]:
            s.wait_stream(torch.cuda.current_stream(self.device))
        _check(_lib().vcattn_fwd_host(ctypes.byref(self.shape), ctypes.c_void_p(hQ.data_ptr()),
                                      ctypes.c_void_p(hK.data_ptr()), ctypes.c_void_p(hV.data_ptr()),
                                      self.k, self.iters, float(sm_scale), _ptr(mask),
                                      ctypes.c_void_p(hO.data_ptr()),
                                      None if hlse2 is None else ctypes.c_void_p(hlse2.data_ptr()),
                                      self.chunk_heads, _ptr(self.ws), self.ws.numel(), self._sp),
               "vcattn_fwd_host")
        return hO, hlse2


def fwd_workspace_bytes(shape_tuple):
    s = Shape(*shape_tuple)
    return int(_lib().vcattn_fwd_workspace_bytes(ctypes.byref(s)))


def test_attn_stalled(pp, sm_scale, stream=None):
    """Failure-path test hook: attention with the K/V loader switched off, so
    every bounded wait in the kernel runs out; last_device_error() then
    reports ERR_TIMEOUT."""
    B, H, N = pp.shape.B, pp.shape.H, pp.shape.N
    O = torch.empty(B, H, N, 128, dtype=torch.bfloat16, device=pp.buf.device)
    lse2 = torch.empty(B, H, N, dtype=torch.float32, device=pp.buf.device)
    f = _lib().vcattn_test_attn_stalled
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(PreppedStruct), ctypes.c_float, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    _check(f(ctypes.byref(pp.shape), ctypes.byref(pp.struct), float(sm_scale), _ptr(O), _ptr(lse2),
             _stream(stream)), "vcattn_test_attn_stalled")
    return O, lse2


def test_attn_stalled_after(pp, sm_scale, steps, mask=None, stream=None):
    """Failure-path test hook: the K/V loader stops after `steps` KV tiles, so
    the kernel gives up with copies and MMAs already issued and must drain
    them before it exits; last_device_error() then reports ERR_TIMEOUT.
    `mask` (u8 [B,H,ceil(N/64),Npad/64], as for attn) selects the block-sparse
    kernel."""
    B, H, N = pp.shape.B, pp.shape.H, pp.shape.N
    if mask is not None:
        _req_mask(mask, B, H, N)
    O = torch.empty(B, H, N, 128, dtype=torch.bfloat16, device=pp.buf.device)
    lse2 = torch.empty(B, H, N, dtype=torch.float32, device=pp.buf.device)
    f = _lib().vcattn_test_attn_stalled_after
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(PreppedStruct), ctypes.c_float, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    _check(f(ctypes.byref(pp.shape), ctypes.byref(pp.struct), float(sm_scale), _ptr(mask), int(steps), _ptr(O),
             _ptr(lse2), _stream(stream)), "vcattn_test_attn_stalled_after")
    return O, lse2


def test_expcast(x, A, B, stream=None):
    """The attention kernel's ExpCast bytes (test hook): x f32 [n] (n a
    multiple of 4), A and B f32 [n/4] on the GPU; returns uint8 [n]."""
    for t, n in ((x, "x"), (A, "A"), (B, "B")):
        _req(t, torch.float32, n)
    if x.numel() % 4 or A.numel() != x.numel() // 4 or B.numel() != A.numel():
        raise ValueError("x needs 4*m scores and A, B m values each")
    codes = torch.empty(x.numel(), dtype=torch.uint8, device=x.device)
    f = _lib().vcattn_test_expcast
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int64, ctypes.c_void_p]
    _check(f(_ptr(x), _ptr(A), _ptr(B), _ptr(codes), x.numel(), _stream(stream)), "vcattn_test_expcast")
    return codes


def last_device_error(stream=None):
    """Synchronise and return (and clear) the device error status."""
    return _lib().vcattn_last_device_error(_stream(stream))


def prep_noalloc(Q, K, V, perm=None, out=None, stream=None):
    """vcattn_prep without a caller workspace: for callers that cannot
    allocate device memory at call time.  The scratch is a 16 MiB array owned
    by the library (shared by all calls on a device; overlapping calls race)."""
    f = _lib().vcattn_prep_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.POINTER(Shape), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.POINTER(PreppedStruct), ctypes.c_void_p]
    for t, n in ((Q, "Q"), (K, "K"), (V, "V")):
        _req(t, torch.bfloat16, n)
    pp = out if out is not None else Prepped(tuple(Q.shape), Q.device)
    s = _shape(Q)
    _check(f(ctypes.byref(s), _ptr(Q), _ptr(K), _ptr(V), _ptr(perm), ctypes.byref(pp.struct),
             _stream(stream)), "vcattn_prep_noalloc")
    return pp
