"""Seeded synthetic workloads (inputs only; none of the method's arithmetic).

These stand in for the captured video-DiT Q/K/V named on the pages (MiniMax-H3
at its live shape (1, 32626, 56, 128); Wan2.2, HunyuanVideo-1.5, LongCat-Video),
which are not available.  The recipe:

* Q, K ~ N(0, 1); K gets a per-channel offset ~ N(0, 2) (variance 2) drawn per
  head, so K centring has something to remove.
* V = centroid[label] + N(0, 1), with ``k_lat`` latent centroids per head drawn
  from N(0, 3) (variance 3) and labels uniform; then each entry is multiplied
  by 20 with probability 0.001 (value outliers).
* Everything is rounded to bf16 (round to nearest even).
* Block-sparse mask (config ``sparse``): per (head, query 64-tile) keep
  round(0.2 * nb) KV 64-blocks, the diagonal always, the rest uniform without
  replacement; one query tile per head keeps the diagonal only.
* Denoising drift (config ``schedule``): step t adds t * N(0, 0.05^2) noise,
  fresh per step, to each of Q, K and V.

The same generator serves the GPU path and the oracle; tests copy the
generated tensors to the host for the oracle.
"""
from dataclasses import dataclass
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    k_lat: int      # latent V clusters of the generator
    k: int          # k-means clusters
    iters: int = 5  # Lloyd iterations
    sparse: bool = False
    steps: int = 1
    seed: int = 1000
    D: int = 128

    @property
    def sm_scale(self):
        return 1.0 / math.sqrt(self.D)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 1024, 8, 8, seed=1000),
    "mid": Workload("mid", 1, 8, 8192, 32, 32, seed=1001),
    "live": Workload("live", 1, 56, 32626, 64, 64, seed=1002),
    # 8 of the live workload's heads (inputs still larger than L2): the size
    # the kernel profiles are captured at
    "live_h8": Workload("live_h8", 1, 8, 32626, 64, 64, seed=1002),
    "schedule": Workload("schedule", 1, 40, 32760, 64, 64, steps=50, seed=1003),
    "sparse": Workload("sparse", 1, 56, 115328, 64, 64, sparse=True, seed=1004),
    # 4 of the sparse workload's heads: the size the masked kernel's profile
    # is captured at
    "sparse_h4": Workload("sparse_h4", 1, 4, 115328, 64, 64, sparse=True, seed=1004),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_qkv(B, H, N, k_lat, seed, device="cpu", D=128, outlier_p=1e-3, outlier_mul=20.0):
    """Q, K, V as bf16 [B, H, N, D] on ``device``, generated head by head."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    Q = torch.empty(B, H, N, D, dtype=torch.bfloat16, device=dev)
    K = torch.empty_like(Q)
    V = torch.empty_like(Q)
    for b in range(B):
        for h in range(H):
            q = torch.randn(N, D, generator=g, device=dev)
            Q[b, h] = q.to(torch.bfloat16)
            k = torch.randn(N, D, generator=g, device=dev)
            k += torch.randn(1, D, generator=g, device=dev) * math.sqrt(2.0)
            K[b, h] = k.to(torch.bfloat16)
            cent = torch.randn(k_lat, D, generator=g, device=dev) * math.sqrt(3.0)
            lab = torch.randint(0, k_lat, (N,), generator=g, device=dev)
            v = cent[lab] + torch.randn(N, D, generator=g, device=dev)
            out = torch.rand(N, D, generator=g, device=dev) < outlier_p
            v = torch.where(out, v * outlier_mul, v)
            V[b, h] = v.to(torch.bfloat16)
    return Q, K, V


def make_workload(w: Workload, device="cpu"):
    return make_qkv(w.B, w.H, w.N, w.k_lat, w.seed, device=device, D=w.D)


def drift(x0, t, seed, device=None, sigma=0.05):
    """Step-t input of the denoising schedule: x0 + t * N(0, sigma^2)."""
    dev = x0.device if device is None else torch.device(device)
    g = _gen(dev, seed * 1000 + t)
    eps = torch.randn(x0.shape, generator=g, device=dev) * sigma
    return (x0.float() + t * eps).to(torch.bfloat16)


def make_tile_mask(B, H, N, seed, keep_frac=0.2, device="cpu"):
    """uint8 [B, H, ceil(N/64), Npad/64] tile mask (query 64-tiles in the
    original order x KV 64-blocks in the permuted order)."""
    nq = (N + 63) // 64
    nb = nq
    npad_blocks = ((N + 127) // 128) * 2
    keep = max(1, int(round(keep_frac * nb)))
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    M = torch.zeros(B, H, nq, npad_blocks, dtype=torch.uint8)
    for b in range(B):
        for h in range(H):
            lone = int(torch.randint(0, nq, (1,), generator=g))
            for i in range(nq):
                M[b, h, i, i] = 1
                if i == lone or keep <= 1:
                    continue
                cand = torch.randperm(nb - 1, generator=g)[: keep - 1]
                cand = cand + (cand >= i).to(cand.dtype)   # skip the diagonal
                M[b, h, i, cand] = 1
    return M.to(device)


def bf16_bits(t):
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def evenly_spaced_queries(N, n=64):
    """Query positions i*(N-1)/(n-1), rounded half to even."""
    import numpy as np
    return np.array([int(np.rint(i * (N - 1) / (n - 1))) for i in range(n)], dtype=np.int64)
