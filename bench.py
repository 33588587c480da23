"""Benchmark of the FP8 smoothed attention forward hot path on GB300.

One step = the whole path over one batch of synthetic input: k-means grouping
(5 Lloyd iterations + stable label sort), fused preprocessing, and the FP8
attention forward, on the 32,626-token video-DiT workload
(B=1, H=56, N=32626, D=128; k=64).  The headline metric is attention TFLOPS,
4*N^2*D*H per step divided by the step time, whole job over all ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) the heads are split across the
ranks; the path has no exchange step, so the only collectives are the timing
barrier and the max-over-ranks reduction.

`--impl reference` times the CPU oracle (plain C, OpenMP) on a bounded sample
of the same workload on the host cores and reports it in the same unit.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from bit_smoothed_attention_gb300 import workloads as W  # noqa: E402

WORKLOAD = "live"
E2E_CHUNK_HEADS = 8   # heads per chunk of the host pipeline (end-to-end arm)
METRIC = "FP8 smoothed attn fwd TFLOPS (4·N²·D·H/s) and % of GB300 FP8 dense peak"
FP8_OVER_BF16 = 2.0   # nominal dense ratio (4.5 vs 2.25 PFLOP/s)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def attn_traffic():
    """DRAM bytes per 56-head attention launch from the committed ncu summary,
    or None when the kernel source has changed since those counters were
    taken (the summary records the source hash)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "attn_fwd_live_h8.md")
    src = os.path.join(ROOT, "bit_smoothed_attention_gb300", "csrc", "attn.cu")
    try:
        text = open(path).read()
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    except OSError:
        return None
    rec = {}
    for ln in text.splitlines():
        if ":" in ln and ln.split(":")[0].strip() in ("kernel_source_sha256", "traffic_bytes_per_launch"):
            k, v = ln.split(":", 1)
            rec[k.strip()] = v.strip().split()[0]
    if rec.get("kernel_source_sha256") != h or "traffic_bytes_per_launch" not in rec:
        return None
    return int(rec["traffic_bytes_per_launch"])


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def head_range(H, world, rank):
    """Contiguous split of H heads over `world` ranks (first ranks take the extra)."""
    base, extra = divmod(H, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def max_over_ranks(x, device):
    """The largest of the ranks' values of x (the job's time is the slowest
    rank's)."""
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def workload_config(w, world):
    """The `config` object of the JSON line (the same keys in both arms)."""
    qkv_gb = 3 * w.B * w.H * w.N * 128 * 2 / 1e9
    return {"workload": "%s: B=%d H=%d N=%d D=128, k-means k=%d x%d iters, 64-token blocks%s"
                        % (w.name, w.B, w.H, w.N, w.k, w.iters, ", block-sparse" if w.sparse else ""),
            "B": w.B, "H": w.H, "N": w.N, "D": 128, "k": w.k, "iters": w.iters,
            "step": "vcattn_group + vcattn_prep + vcattn_attn",
            "l2": "inputs (%.2f GB bf16 Q/K/V) exceed the 129 MB L2" % qkv_gb,
            "parallelism": "heads split over %d rank(s), no collective in the path" % world}


# --------------------------------------------------------------------- ours
def run_ours(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()

    w = W.WORKLOADS[args.workload]
    h0, h1 = head_range(w.H, world, rank)
    Hl = h1 - h0
    Q, K, V = W.make_workload(w, device=dev)
    Q, K, V = (t[:, h0:h1].contiguous() for t in (Q, K, V))
    torch.cuda.synchronize()
    mask = None
    if w.sparse:
        mask = W.make_tile_mask(w.B, w.H, w.N, w.seed + 7)[:, h0:h1].contiguous().to(dev)
    sm_scale = float(np.float32(w.sm_scale))
    kept_frac = 1.0 if mask is None else float(mask.float().mean().item()) * (
        mask.shape[-1] / mask.shape[-2])

    B, N = w.B, w.N
    labels = torch.empty(B, Hl, N, dtype=torch.int32, device=dev)
    perm = torch.empty_like(labels)
    gshape = vcattn.Shape(B, Hl, N, 128)
    import ctypes
    L = vcattn.lib()
    gws_n = L.vcattn_group_workspace_bytes(ctypes.byref(gshape), w.k)
    gws = torch.empty(gws_n, dtype=torch.uint8, device=dev)
    pp = vcattn.Prepped((B, Hl, N, 128), dev)
    pws_n = L.vcattn_prep_workspace_bytes(ctypes.byref(gshape))
    pws = torch.empty(pws_n, dtype=torch.uint8, device=dev)
    O = torch.empty(B, Hl, N, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Hl, N, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    sptr = ctypes.c_void_p(stream.cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    mptr = None if mask is None else P(mask)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        st = L.vcattn_group(ctypes.byref(gshape), P(V), w.k, w.iters, P(labels), P(perm), None, P(gws),
                            gws_n, sptr)
        if ev:
            ev[1].record(stream)
        st |= L.vcattn_prep(ctypes.byref(gshape), P(Q), P(K), P(V), P(perm), ctypes.byref(pp.struct),
                            P(pws), pws_n, sptr)
        if ev:
            ev[2].record(stream)
        st |= L.vcattn_attn(ctypes.byref(gshape), ctypes.byref(pp.struct), ctypes.c_float(sm_scale), mptr,
                            P(O), P(lse), sptr)
        if ev:
            ev[3].record(stream)
        if st:
            raise RuntimeError("vcattn call failed with status %d" % st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if vcattn.last_device_error() != 0:
        raise RuntimeError("device-side error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if world == 1 else local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    if vcattn.last_device_error() != 0:
        raise RuntimeError("device-side error during the timed region")
    ms = t_start.elapsed_time(t_end)
    if world > 1:
        ms = max_over_ranks(ms, dev)
    ms_step = ms / args.steps
    t_group = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    t_prep = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    t_attn = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)

    flops_step = 4.0 * N * N * 128 * w.H * B * kept_frac    # whole job
    value = flops_step / (ms_step * 1e-3) / 1e12
    flops_attn_local = 4.0 * N * N * 128 * Hl * B * kept_frac
    attn_tflops = flops_attn_local / (t_attn * 1e-3) / 1e12
    pk = peaks()
    # The attention launch (about 16 ms) runs at the full SM clock inside a
    # sub-second timed region, so its denominator is the burst bf16 rate (the
    # sustained rate was measured power-capped at a lower clock).
    fp8_peak = pk["bf16"] * FP8_OVER_BF16
    Np = vcattn.npad(N)
    prep_bytes = B * Hl * (3 * N * 128 * 2 + 3 * Np * 128 + N * 4 * 2 + (Np // 64) * 128 * 4 +
                           (Np // 128) * 4096)
    prep_gbs = prep_bytes / (t_prep * 1e-3) / 1e9
    kmeans_flop = 2.0 * N * w.k * 128 * w.iters * Hl * B
    # k-means: init, per iteration assign + fix-up + chunk sums + finalize,
    # two sort kernels; preprocessing: 3; attention: 1
    launches_per_step = (1 + 4 * w.iters + 2) + 3 + 1

    e2e = run_e2e(args, w, vcattn, dev, Q, K, V, mask, sm_scale, flops_step, world)
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3",
        "data": "synthetic (seeded generator standing in for captured video-DiT Q/K/V)",
        "config": workload_config(w, world),
        "breakdown_ms": {"group": round(t_group, 4), "prep": round(t_prep, 4), "attn": round(t_attn, 4)},
        "attn_tflops": round(attn_tflops, 2),
        "prep_gbs": round(prep_gbs, 1),
        "prep_hbm_frac": round(prep_gbs / pk["hbm"], 4),
        "kmeans_tflops": round(kmeans_flop / (t_group * 1e-3) / 1e12, 2),
        "group_pct_of_attn": round(100 * t_group / t_attn, 2),
        "roofline": {"bound": "tensor", "kernel": "attn_sparse" if w.sparse else "attn_fwd",
                     "achieved": round(attn_tflops, 2),
                     "peak": round(fp8_peak, 1), "unit": "TFLOP/s",
                     "frac": round(attn_tflops / fp8_peak, 4),
                     "peak_source": "%s bf16 burst x %.0f (nominal FP8/bf16 ratio)" % (pk["src"], FP8_OVER_BF16),
                     "traffic": attn_traffic() if (args.workload == "live" and world == 1) else None,
                     "traffic_unit": "bytes per launch (ncu dram read + write)"},
        "gpu_launches": launches_per_step * args.steps,
        "e2e": e2e,
        "clocks": clock_info,
    }
    if rank == 0 and world == 1 and not args.skip_cpu:
        out["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_e2e(args, w, vcattn, dev, Q, K, V, mask, sm_scale, flops_step, world):
    """Same metric through the public API with pinned host buffers: every
    step is one vcattn_fwd_host call, which copies Q, K, V host->device and
    O device->host inside the timed region, overlapped with the grouping,
    preprocessing and attention of the other head chunks."""
    hQ, hK, hV = (t.cpu().pin_memory() for t in (Q, K, V))
    hO = torch.empty(Q.shape, dtype=torch.bfloat16).pin_memory()
    B, H, N, D = Q.shape
    pipe = vcattn.HostPipeline((B, H, N, D), w.k, w.iters, chunk_heads=E2E_CHUNK_HEADS, device=dev)
    steps = max(1, min(args.steps, 5))

    def one():
        pipe(hQ, hK, hV, sm_scale, mask=mask, hO=hO)

    for _ in range(2):  # warm-up calls
        one()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / steps
    if world > 1:
        dt = max_over_ranks(dt, dev)
    return {"value": round(flops_step / dt / 1e12, 2), "unit": "TFLOPS",
            "h2d_bytes_per_step": int(3 * Q.numel() * 2) * world,
            "d2h_bytes_per_step": int(Q.numel() * 2) * world,
            "ms_per_step": round(dt * 1e3, 3), "steps": steps,
            "api": "vcattn_fwd_host, %d-head chunks, copies overlapped with compute" % pipe_chunk(H * B)}


def pipe_chunk(bh):
    return min(bh, E2E_CHUNK_HEADS if E2E_CHUNK_HEADS > 0 else 8)


# ------------------------------------------------------------ CPU baseline
def cpu_sample(w, heads, nq, seed_offset=0):
    """Oracle on a bounded sample: full grouping + preprocessing of `heads`
    heads and the emulated attention of `nq` evenly spaced queries per head.
    Returns (seconds, attention-equivalent FLOPs of the full heads)."""
    import oracle
    Q, K, V = W.make_qkv(1, heads, w.N, w.k_lat, w.seed + 17 + seed_offset)
    Qb, Kb, Vb = (W.bf16_bits(t).reshape(heads, w.N, 128) for t in (Q, K, V))
    qidx = W.evenly_spaced_queries(w.N, nq)
    t0 = time.perf_counter()
    labels, _ = oracle.kmeans(Vb, w.k, w.iters)
    perm = oracle.stable_sort(labels, w.k)
    pp = oracle.prep(Qb, Kb, Vb, perm)
    t1 = time.perf_counter()
    for h in range(heads):
        oracle.attn_emul(pp, h, w.N, float(np.float32(w.sm_scale)), qidx=qidx)
    t2 = time.perf_counter()
    # extrapolate the per-query attention time to all N queries
    t_full = (t1 - t0) + (t2 - t1) * (w.N / nq)
    flops = 4.0 * w.N * w.N * 128 * heads
    return t_full, flops, (t1 - t0), (t2 - t1)


def cpu_baseline(w, budget_s=30.0):
    import oracle
    cores = oracle.threads()
    heads = max(1, min(cores, w.H))
    nq = 64
    t_full, flops, tg, ta = cpu_sample(w, heads, nq)
    return {"value": round(flops / t_full / 1e12, 6), "unit": "TFLOPS", "cores": cores,
            "kind": "oracle",
            "sample": ("%d of %d heads: full k-means + sort + prep (%.1f s), emulated attention for "
                       "%d evenly spaced queries per head (%.1f s), attention time extrapolated to all "
                       "%d queries" % (heads, w.H, tg, nq, ta, w.N))}


def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is the bounded
    sample `cpu_baseline` also times (as many heads as cores, grouped and
    prepped in full, emulated attention of 64 evenly spaced queries per head).
    `ms_per_step` is the measured time of that sample; `value` is the
    oracle's attention throughput on the full workload, with the attention
    time extrapolated from the sampled queries to all of them (the
    extrapolated full-step time is reported beside it)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build.build()
    w = W.WORKLOADS[args.workload]
    cores = oracle.threads()
    heads = max(1, min(cores, w.H))
    nq = 64
    for i in range(args.warmup):
        cpu_sample(w, heads, nq, seed_offset=i)
    full, measured, tg, ta = [], [], 0.0, 0.0
    for i in range(args.steps):
        t_full, flops, g, a = cpu_sample(w, heads, nq, seed_offset=100 + i)
        full.append(t_full)
        measured.append(g + a)
        tg += g
        ta += a
    t_full = sum(full) / len(full)
    t_meas = sum(measured) / len(measured)
    value = 4.0 * w.N * w.N * 128 * heads / t_full / 1e12
    sample = ("per step: %d of %d heads, full k-means + sort + prep (%.2f s), emulated attention of %d "
              "evenly spaced queries per head (%.2f s); attention time extrapolated to all %d queries"
              % (heads, w.H, tg / args.steps, nq, ta / args.steps, w.N))
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(t_meas * 1e3, 2), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "e4m3 (emulated in software)", "data": "synthetic",
           "config": workload_config(w, world),
           "extrapolated": {"full_step_ms_for_sampled_heads": round(t_full * 1e3, 2),
                            "heads": heads, "queries_run_per_head": nq,
                            "note": "value = 4*N^2*D*heads / this extrapolated time"},
           "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def profile_case(workload):
    """One grouping, one preprocessing and two attention calls on `workload`
    (with the bench's tile mask if it is block-sparse), untimed: the launch
    sequence the committed ncu summaries capture (``-k regex:<kernel> -s <n>
    -c <m>``)."""
    from bit_smoothed_attention_gb300 import build, vcattn
    build.build()
    w = W.WORKLOADS[workload]
    Q, K, V = W.make_workload(w, device="cuda")
    _, perm = vcattn.group(V, w.k, w.iters)
    pp = vcattn.prep(Q, K, V, perm)
    pp = vcattn.prep(Q, K, V, perm, out=pp)
    sm = float(np.float32(w.sm_scale))
    # the bench's mask for a block-sparse workload
    mask = W.make_tile_mask(w.B, w.H, w.N, w.seed + 7).to(Q.device) if w.sparse else None
    O, L = vcattn.attn(pp, sm, mask=mask)
    vcattn.attn(pp, sm, mask=mask, O=O, lse2=L)
    torch.cuda.synchronize()
    st = vcattn.last_device_error()
    if st != 0:
        raise RuntimeError("device error status %d" % st)
    print("profile case %s done" % workload)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--skip-cpu", action="store_true", help="omit the CPU-baseline leg")
    ap.add_argument("--cpu-budget", type=float, default=30.0)
    ap.add_argument("--profile-case", default=None, choices=sorted(W.WORKLOADS),
                    help="run one untimed pass of the path for an ncu capture and exit")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
