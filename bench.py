"""Attention forward benchmark: TFLOP/s on one GB300 and the fraction of the dense
bf16 tensor-core peak.

Default workload: long-sequence causal self-attention, B=2, h=16, n=8192,
d_k=d_v=64, bf16 inputs N(0,1) x 0.5 (the pages' O(n^2 d) scaling case). One step
is one attn_fwd call over the whole batch (all steps of the hot path: Q/K/V
tiles in, QK^T, scale, mask, online softmax, PV, normalisation and the bf16 /
lse stores). FLOPs are algorithmic: 2 (d_k + d_v) per legal query-key pair.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-cpu-baseline] [--grad]

--mha times the whole multi-head attention layer instead (one attn_mha_fwd call per
step: the Q, K, V projections in one launch, the attention on the projections'
[B, n, h*d] layout and the output projection; d_model = h*d, random weights resident
on the device);
FLOPs are algorithmic: 2 d_model h d per projected row for each of the four
projections plus the attention's.

--grad times the gradients instead (one attn_bwd call per step, attn_bwd_local for
the local-window workload: D = rowsum(dO*O), the dK/dV kernel and the dQ kernel),
given the forward's output and lse computed once before the timed region; FLOPs are algorithmic, 2 (3 d_k + 2 d_v) per legal
pair (the five products of the backward pass).

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU (independent shards of B*h, no collective on the data path; weak scaling),
the timed region is bracketed by a barrier and a synchronize on both sides, and
the time is the maximum over ranks. Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on bounded row samples of the same
workload (rank 0 only; other ranks exit without work).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from transformer_scaled_dot_mha_gb300 import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "long_causal_b2_h16_n8192_d64"
L2_FLUSH_BYTES = 512 << 20
L2_NOTE = (f"flushed between timed steps: a {L2_FLUSH_BYTES >> 20} MiB memset, then a read of the same buffer "
           "(L2 holds none of the step's data and no dirty lines whose write-back the step would pay for)")
L2_WARM_NOTE = ("warm: no flush between timed steps; every step reads the same inputs, which stay in L2 "
                "when they fit (129 MB), so this line is a tensor-roofline view, not an HBM one")


class L2Flush:
    """Evicts the 129 MB L2 between timed steps, outside the events. The memset alone
    leaves up to an L2 of dirty lines, and the next step would pay for their write-back
    to HBM (about 12 us of a 75 us decode step); reading the buffer afterwards moves
    that write-back before the step."""

    def __init__(self, dev):
        import torch

        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.words = self.buf.view(torch.int64)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self):
        self.buf.zero_()
        self.sink.copy_(self.words.sum())


FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic per launch of the dominant kernel from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by the workload and the
# sha256 of that kernel's own sources; reported only while those sources match.
KERNEL_SOURCES = {
    "attn_fwd_tc_kernel": ("attn_fwd_tc.cu", "ptx_sm103.cuh"),
    "attn_decode_split_kernel": ("attn_decode.cu", "ptx_sm103.cuh"),
    "attn_decode_warp_kernel": ("attn_decode.cu", "ptx_sm103.cuh"),
    "attn_bwd_tc_kernel": ("attn_bwd.cu", "ptx_sm103.cuh"),
}
NCU_TRAFFIC = {
    ("long_causal_b2_h16_n8192_d64", "attn_fwd_tc_kernel", "dd287655676f270e"): 153654016,
    ("long_none_b2_h16_n8192_d64", "attn_fwd_tc_kernel", "dd287655676f270e"): 114852352,
    ("long_causal_b2_h16_n8192_d128", "attn_fwd_tc_kernel", "dd287655676f270e"): 572768256,
    ("long_none_b2_h16_n8192_d128", "attn_fwd_tc_kernel", "dd287655676f270e"): 1066685952,
    ("long_cross_pad_b2_h16_q4096_k8192_d64", "attn_fwd_tc_kernel", "dd287655676f270e"): 76273152,
    ("long_cross_pad_b2_h16_q4096_k8192_d128", "attn_fwd_tc_kernel", "dd287655676f270e"): 529536512,
    ("local_causal_b2_h16_n8192_d64_w511", "attn_fwd_tc_kernel", "dd287655676f270e"): 110697472,
    # the warp kernel only (the merge kernel is not counted)
    ("decode_b16_h16_q1_k8192_d64", "attn_decode_warp_kernel", "15a9265a513b2001"): 424486400,
    # the fused d = 64 kernel (the local-window workload: its LOCAL instantiation)
    ("long_causal_b2_h16_n8192_d64", "attn_bwd_tc_kernel", "0aab31e7fb26f9cd"): 291646464,
    ("local_causal_b2_h16_n8192_d64_w511", "attn_bwd_tc_kernel", "0aab31e7fb26f9cd"): 290630656,
}


_C_COMMENT = re.compile(r'"(?:\\.|[^"\\])*"|//[^\n]*|/\*.*?\*/', re.S)


def _code_only(src: str) -> str:
    """C++ source without its comments, blank lines and the whitespace at either end of a
    line (string literals kept): DRAM traffic depends on the code, so a comment or
    indentation edit must not invalidate a capture."""
    s = _C_COMMENT.sub(lambda m: m.group(0) if m.group(0).startswith('"') else "", src)
    return "\n".join(line.strip() for line in s.splitlines() if line.strip())


def kernel_source_hash(kernel: str = "attn_fwd_tc_kernel") -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "transformer_scaled_dot_mha_gb300", "csrc", f)) as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_seed(w, rank: int) -> int:
    """Each rank draws its own shard of (b, h) problems; rank 0 keeps the workload's seed."""
    return w.seed + 1000 * rank


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a per-rank scalar over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_tflops(flops_per_rank_step: float, steps: int, max_total_ms: float, world: int) -> float:
    """Whole-job throughput: the work of every rank over the slowest rank's time."""
    return world * flops_per_rank_step * steps / (max_total_ms / 1e3) / 1e12


def mask_name(mode):
    names = {1: "causal", 2: "key_padding", 4: "decode", 8: "window"}
    return "+".join(v for k, v in names.items() if mode & k) or "none"


def config_of(w, extra=None):
    cfg = {"workload": w.name, "B": w.B, "h": w.H, "n_q": w.n_q, "n_k": w.n_k, "d_k": w.d_k, "d_v": w.d_v,
           "mask": mask_name(w.mask_mode), "inputs": f"N(0,1) x {w.input_scale}, seed {w.seed}",
           **({"window": w.window} if w.mask_mode & W.MASK_WINDOW else {}),
           "flops": "algorithmic: 2*(d_k+d_v) per legal (query, key) pair"}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for ln in out.splitlines():
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) == 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        # samples arrive every 100 ms; keep the loaded ones (the timed region is short)
        loaded = [r for r in rows if float(r[3]) > 200.0] or rows
        sm = [float(r[1]) for r in loaded]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in loaded:
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(float(r[2]) for r in rows),
                "reasons": sorted(reasons), "samples": len(loaded), "power_w_max": max(float(r[3]) for r in loaded)}


# ---------------------------------------------------------------- CPU oracle leg
def sample_row_ids(w, rng_seed=7):
    """Row ids spread over all heads and positions of the workload."""
    rng = np.random.Generator(np.random.PCG64(rng_seed))
    return rng.permutation(w.B * w.H * w.n_q).astype(np.int64)


def oracle_rows_flops(w, ids, key_lens):
    i = ids % w.n_q
    b = ids // (w.H * w.n_q)
    lim = np.full(ids.shape, w.n_k, np.int64)
    if w.mask_mode & W.MASK_KEY_PADDING:
        lim = np.minimum(lim, key_lens[b])
    if w.mask_mode & W.MASK_CAUSAL:
        lim = np.minimum(lim, i + 1)
    lo = np.zeros_like(lim)
    if w.mask_mode & W.MASK_WINDOW:
        lim = np.minimum(lim, i + w.window + 1)
        lo = np.maximum(lo, i - w.window)
    if w.mask_mode & W.MASK_DECODE:
        lim = np.minimum(lim, key_lens[b] - w.n_q + i + 1)
    return float(2 * (w.d_k + w.d_v) * np.maximum(lim - lo, 0).sum())


def time_oracle(w, inputs, ids, threads):
    import oracle

    if not os.path.exists(oracle.LIB):
        oracle.build()
    orc = oracle.Oracle()
    q, k, v, kl = inputs
    t0 = time.perf_counter()
    orc.attention_rows(q, k, v, w.scale, ids, w.mask_mode, kl, n_threads=threads, window=max(w.window, 0))
    return time.perf_counter() - t0


def cpu_baseline(w, inputs, target_s=12.0):
    """The oracle as it stands, on a bounded sample of rows of the same workload."""
    threads = os.cpu_count() or 1
    ids_all = sample_row_ids(w)
    n = max(threads, 16)
    dt = time_oracle(w, inputs, ids_all[:n], threads)
    while dt < 0.5 and n < ids_all.size:
        n = min(ids_all.size, n * 4)
        dt = time_oracle(w, inputs, ids_all[:n], threads)
    n = int(min(ids_all.size, max(n, n * target_s / max(dt, 1e-9))))
    ids = ids_all[:n]
    dt = time_oracle(w, inputs, ids, threads)
    flops = oracle_rows_flops(w, ids, inputs[3])
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n} query rows drawn uniformly from all {w.B * w.H * w.n_q} rows of the workload "
                      f"({flops / 1e9:.2f} GFLOP algorithmic), fp64 C oracle, {dt:.2f} s wall"}


# ---------------------------------------------------------------- our arm
def run_ours(args, w):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    from transformer_scaled_dot_mha_gb300 import attn

    attn.lib()
    q, k, v, kl = W.make_inputs(w, shard_seed(w, rank))
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    kld = torch.from_numpy(kl).to(dev)
    out = torch.empty((w.B, w.H, w.n_q, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.n_q), dtype=torch.float32, device=dev)
    flush = (lambda: None) if args.warm_l2 else L2Flush(dev)
    stream = torch.cuda.current_stream()
    key_lens = kld if w.mask_mode & W.MASK_KEY_PADDING else None
    decode = bool(w.mask_mode & W.MASK_DECODE)
    if decode:
        ws = torch.empty(attn.attn_decode_workspace_size(w.B, w.H, w.n_q, w.n_k, w.d_k), dtype=torch.uint8,
                         device=dev)

    def step():
        if decode:
            attn.attn_decode(qd, kd, vd, out, kld, ws, lse, w.scale, stream)
        elif w.mask_mode & W.MASK_WINDOW:
            attn.attn_fwd_local(qd, kd, vd, out, w.window, lse, w.scale, w.mask_mode & ~W.MASK_WINDOW, key_lens,
                                stream)
        else:
            attn.attn_fwd(qd, kd, vd, out, lse, w.scale, w.mask_mode, key_lens, stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    st, code = attn.attn_fault_status(stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel fault record {code:#x} during warm-up")

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for e0, e1 in evs:
        flush()  # L2 flush between timed steps, outside the events
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop() if rank == 0 else None
    times_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(sum(times_ms), dev)
    st, code = attn.attn_fault_status(stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel fault record {code:#x} in the timed region")

    flops_step = w.algorithmic_flops(kl)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_tflops(flops_step, args.steps, total_ms, world)

    # ---- end to end through the public call: pinned host buffers in, result out
    e2e = run_e2e(args, w, q, k, v, kl, dev, stream, attn, flops_step, world)

    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    kernel = ("attn_decode_warp_kernel" if w.n_q == 1 else "attn_decode_split_kernel") if decode else "attn_fwd_tc_kernel"
    src_hash = kernel_source_hash(kernel)
    traffic = NCU_TRAFFIC.get((w.name, kernel, src_hash))
    if decode:  # HBM-bound: one read of the used cache rows dominates
        roof = {"bound": "hbm", "achieved": round(w.algorithmic_bytes(kl) / (ms_per_step / 1e3) / 1e9, 1),
                "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
                "algorithmic_bytes": w.algorithmic_bytes(kl), "peak_source": f"hbm_gbs of {peak_src}",
                "kernel": f"attn_decode ({kernel} + merge kernel, timed together)"}
    else:
        achieved = flops_step / (ms_per_step / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": float(peaks["bf16_tflops"]),
                "unit": "TFLOP/s", "peak_source": f"bf16_tflops (burst) of {peak_src}",
                "kernel": "attn_fwd_tc_kernel"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = traffic
    roof["kernel_source"] = src_hash
    line = {
        "metric": "attention fwd TFLOP/s on 1 GB300 and % of dense bf16 tensor peak",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, {"l2": L2_WARM_NOTE if args.warm_l2 else L2_NOTE,
                                "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU",
                                "dense_equivalent_tflops": round(world * w.dense_flops() * args.steps /
                                                                 (total_ms / 1e3) / 1e12, 2)}),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": args.steps * (2 if decode else 1),
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
    }
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, (q, k, v, kl))
    return line


def run_e2e(args, w, q, k, v, kl, dev, stream, attn, flops_step, world):
    """Same metric from pinned host buffers, all inside the events: H2D of Q/K/V (and
    key lengths), the kernel, D2H of the output. Full forward workloads go through
    attn_fwd_host (chunked copies overlapping the kernels); decoding and the local
    window copy around the device entry point."""
    import torch

    pin = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).pin_memory()
    qh, kh, vh = pin(q), pin(k), pin(v)
    klh = torch.from_numpy(kl).pin_memory()
    outh = torch.empty((w.B, w.H, w.n_q, w.d_v), dtype=torch.bfloat16).pin_memory()
    qd, kd, vd = (torch.empty_like(t, device=dev) for t in (qh, kh, vh))
    kld = torch.empty_like(klh, device=dev)
    out = torch.empty_like(outh, device=dev)
    decode = bool(w.mask_mode & W.MASK_DECODE)
    use_kl = bool(w.mask_mode & (W.MASK_KEY_PADDING | W.MASK_DECODE))
    host = not decode and not (w.mask_mode & W.MASK_WINDOW)
    steps = max(3, min(args.steps, 50))
    if host:
        hws = torch.empty(attn.attn_fwd_host_workspace_size(w.B, w.H, w.n_q, w.n_k, w.d_k, w.mask_mode), dtype=torch.uint8,
                          device=dev)
    if decode:
        # a serving step: the key/value cache stays resident in HBM; the new queries
        # and the cache lengths come from the host, the output goes back
        kd.copy_(kh)
        vd.copy_(vh)
        ws = torch.empty(attn.attn_decode_workspace_size(w.B, w.H, w.n_q, w.n_k, w.d_k), dtype=torch.uint8,
                         device=dev)

    def step():
        if host:
            attn.attn_fwd_host(qh, kh, vh, outh, hws, None, w.scale, w.mask_mode, klh if use_kl else None, stream)
            return
        qd.copy_(qh, non_blocking=True)
        if not decode:
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
        if use_kl:
            kld.copy_(klh, non_blocking=True)
        if decode:
            attn.attn_decode(qd, kd, vd, out, kld, ws, None, w.scale, stream)
        elif w.mask_mode & W.MASK_WINDOW:
            attn.attn_fwd_local(qd, kd, vd, out, w.window, None, w.scale, w.mask_mode & ~W.MASK_WINDOW,
                                kld if use_kl else None, stream)
        else:
            attn.attn_fwd(qd, kd, vd, out, None, w.scale, w.mask_mode, kld if use_kl else None, stream)
        outh.copy_(out, non_blocking=True)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, dev)
    h2d = sum(t.numel() * t.element_size() for t in ((qh,) if decode else (qh, kh, vh))) + \
        (klh.numel() * 4 if use_kl else 0)
    d2h = outh.numel() * outh.element_size()
    how = "pinned host buffers, copies and kernel on one stream, CUDA events"
    if host:
        how = ("attn_fwd_host on pinned host buffers: chunked H2D / kernel / D2H overlapped on three streams, "
               "CUDA events on the caller's stream")
    if decode:
        how += "; key/value cache resident on the device"
    return {"value": round(weak_scaling_tflops(flops_step, 1, ms, world), 2), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(ms, 4),
            "steps": steps, "how": how}


# ---------------------------------------------------------------- gradients
def cpu_baseline_grad(w, inputs, dout):
    """The oracle's gradients, as they stand, on a bounded sample: whole heads of
    the workload (one host thread per head)."""
    import oracle

    if not os.path.exists(oracle.LIB):
        oracle.build()
    orc = oracle.Oracle()
    q, k, v, kl = inputs
    threads = os.cpu_count() or 1
    hs = max(1, min(threads, w.H))
    sl = lambda a: np.ascontiguousarray(a[:1, :hs])
    kl1 = kl[:1] if w.mask_mode & W.MASK_KEY_PADDING else None
    window = w.window if w.mask_mode & W.MASK_WINDOW else 0
    t0 = time.perf_counter()
    orc.attention_bwd(sl(q), sl(k), sl(v), sl(dout), w.scale, w.mask_mode, kl1, window=window, n_threads=hs)
    dt = time.perf_counter() - t0
    if w.mask_mode & W.MASK_WINDOW:
        pairs = W.legal_pairs_window(1, hs, w.n_q, w.mask_mode, w.window, kl1)
    else:
        pairs = W.legal_pairs(1, hs, w.n_q, w.n_k, w.mask_mode, kl1)
    flops = 2.0 * (3 * w.d_k + 2 * w.d_v) * pairs
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": hs, "kind": "oracle",
            "sample": f"{hs} whole heads (batch 0) of the workload, fp64 C oracle gradients, {dt:.2f} s wall"}


def run_ours_grad(args, w):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    from transformer_scaled_dot_mha_gb300 import attn

    attn.lib()
    seed = shard_seed(w, rank)
    q, k, v, kl = W.make_inputs(w, seed)
    dout = W.make_grad_output(w, seed)
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    qd, kd, vd, gd = to_dev(q), to_dev(k), to_dev(v), to_dev(dout)
    kld = torch.from_numpy(kl).to(dev)
    key_lens = kld if w.mask_mode & W.MASK_KEY_PADDING else None
    out = torch.empty((w.B, w.H, w.n_q, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.n_q), dtype=torch.float32, device=dev)
    local_window = bool(w.mask_mode & W.MASK_WINDOW)
    base_mask = w.mask_mode & ~W.MASK_WINDOW
    if local_window:
        attn.attn_fwd_local(qd, kd, vd, out, w.window, lse, w.scale, base_mask, key_lens)
    else:
        attn.attn_fwd(qd, kd, vd, out, lse, w.scale, w.mask_mode, key_lens)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(attn.attn_bwd_workspace_size(w.B, w.H, w.n_q, w.d_k), dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def step():
        if local_window:
            attn.attn_bwd_local(qd, kd, vd, out, gd, lse, dq, dk, dv, ws, w.window, w.scale, base_mask, key_lens,
                                stream)
        else:
            attn.attn_bwd(qd, kd, vd, out, gd, lse, dq, dk, dv, ws, w.scale, w.mask_mode, key_lens, stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    st, code = attn.attn_fault_status(stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel fault record {code:#x} during warm-up")
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop() if rank == 0 else None
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), dev)
    st, code = attn.attn_fault_status(stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel fault record {code:#x} in the timed region")
    flops_step = w.algorithmic_bwd_flops(kl)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_tflops(flops_step, args.steps, total_ms, world)

    # end to end: pinned host Q, K, V, O, dO, lse in; dQ, dK, dV out
    pin = lambda t: t.cpu().pin_memory()
    hosts = [pin(t) for t in (qd, kd, vd, out, gd, lse)]
    klh = torch.from_numpy(kl).pin_memory()
    grads_h = [torch.empty_like(t, device="cpu").pin_memory() for t in (dq, dk, dv)]
    e2e_steps = max(3, min(args.steps, 20))

    if local_window:  # copies around attn_bwd_local on one stream
        devs = (qd, kd, vd, out, gd, lse)

        def e2e_step():
            for dst, src in zip(devs, hosts):
                dst.copy_(src, non_blocking=True)
            if key_lens is not None:
                kld.copy_(klh, non_blocking=True)
            step()
            for dst, src in zip(grads_h, (dq, dk, dv)):
                dst.copy_(src, non_blocking=True)
    else:
        hws = torch.empty(attn.attn_bwd_host_workspace_size(w.B, w.H, w.n_q, w.n_k, w.d_k, w.mask_mode),
                          dtype=torch.uint8, device=dev)

        def e2e_step():
            attn.attn_bwd_host(*hosts[:5], hosts[5], *grads_h, hws, w.scale, w.mask_mode,
                               klh if key_lens is not None else None, stream)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    h2d = sum(t.numel() * t.element_size() for t in hosts) + (klh.numel() * 4 if key_lens is not None else 0)
    d2h = sum(t.numel() * t.element_size() for t in grads_h)
    e2e = {"value": round(weak_scaling_tflops(flops_step, 1, e2e_ms, world), 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
           "steps": e2e_steps,
           "how": ("pinned host buffers copied in, attn_bwd_local, gradients copied out, one stream"
                   if local_window else
                   "attn_bwd_host on pinned host buffers: chunked H2D / gradient kernels / D2H overlapped on the "
                   "library's streams, CUDA events on the caller's stream")}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    achieved = flops_step / (ms_per_step / 1e3) / 1e12
    fused = w.d_k == 64
    src_hash = kernel_source_hash("attn_bwd_tc_kernel")
    roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": float(peaks["bf16_tflops"]),
            "unit": "TFLOP/s", "peak_source": f"bf16_tflops (burst) of {peak_src}",
            "kernel": ("attn_bwd fused schedule (memset, dot kernel, fused dK/dV/dQ kernel, dQ conversion; "
                       "timed together)" if fused else
                       "attn_bwd (dot kernel + dK/dV kernel + dQ kernel, timed together)"),
            "traffic": NCU_TRAFFIC.get((w.name, "attn_bwd_tc_kernel", src_hash)) if fused else None,
            "kernel_source": src_hash}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    line = {
        "metric": "attention bwd TFLOP/s on 1 GB300 and % of dense bf16 tensor peak",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, {"pass": "gradients (attn_bwd_local)" if local_window else "gradients (attn_bwd)",
                                "schedule": ("fused: five products once, dQ by TMA reduce-add" if fused else
                                             "deterministic: dK/dV kernel + dQ kernel, seven products"),
                                "flops": "algorithmic: 2*(3*d_k+2*d_v) per legal (query, key) pair",
                                "l2": L2_NOTE,
                                "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU"}),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": args.steps * 3,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
    }
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_grad(w, (q, k, v, kl), dout)
    return line


# ---------------------------------------------------------------- multi-head layer
def mha_flops(w, key_lens):
    hd, d_model = w.H * w.d_k, w.H * w.d_k
    proj = 2.0 * d_model * hd * w.B * (2 * w.n_q + 2 * w.n_k)
    return proj + w.algorithmic_flops(key_lens)


def cpu_baseline_mha(w, target_s=12.0):
    """The oracle's multi-head layer, as it stands, on a bounded sample: one batch
    row of the same layer (d_model, h, d, mask) with a shortened sequence, grown
    until it takes about ``target_s`` seconds."""
    import oracle

    if not os.path.exists(oracle.LIB):
        oracle.build()
    orc = oracle.Oracle()
    threads = os.cpu_count() or 1
    n = 16
    while True:
        inp = W.make_mha_inputs(w, B=1, n_q=n, n_k=n if w.n_q == w.n_k else 2 * n)
        kl = np.minimum(inp["key_lens"], inp["x_kv"].shape[1])
        t0 = time.perf_counter()
        orc.mha(inp["x_q"], inp["x_kv"], inp["w_q"], inp["w_k"], inp["w_v"], inp["w_o"], w.H, w.scale, w.mask_mode,
                kl, b_q=inp["b_q"], b_k=inp["b_k"], b_v=inp["b_v"], b_o=inp["b_o"], n_threads=threads)
        dt = time.perf_counter() - t0
        if dt > target_s / 4 or 2 * n > w.n_q:
            break
        n *= 2
    n_k = inp["x_kv"].shape[1]
    sub = W.Workload(w.name, 1, w.H, n, n_k, w.d_k, w.d_v, w.dtype, w.mask_mode, w.key_len_range, w.input_scale,
                     w.index, w.window)
    flops = mha_flops(sub, kl)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"one batch row of the same layer with n_q = {n}, n_k = {n_k} (d_model {w.H * w.d_k}, h {w.H}), "
                      f"fp64 C oracle (projections single-threaded, attention on {threads} threads), {dt:.2f} s wall"}


def run_ours_weights(args, w):
    """attn_weights: the softmax weight matrix [B, h, n_q, n_k] (fp32) from q, k and the
    forward's lse. HBM-bound on its write; value = algorithmic bytes per second."""
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from transformer_scaled_dot_mha_gb300 import attn

    attn.lib()
    q, k, v, kl = W.make_inputs(w, shard_seed(w, rank))
    to_dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    kld = torch.from_numpy(kl).to(dev)
    key_lens = kld if w.mask_mode & W.MASK_KEY_PADDING else None
    out = torch.empty((w.B, w.H, w.n_q, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.n_q), dtype=torch.float32, device=dev)
    attn.attn_fwd(qd, kd, vd, out, lse, w.scale, w.mask_mode, key_lens)
    wts = torch.empty((w.B, w.H, w.n_q, w.n_k), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def step():
        attn.attn_weights(qd, kd, lse, wts, w.scale, w.mask_mode, key_lens, stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    st, code = attn.attn_fault_status(stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel fault record {code:#x} during warm-up")
    clocks = ClockSampler(local)
    clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    st, code = attn.attn_fault_status(stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel fault record {code:#x} in the timed region")
    total_ms = sum(a.elapsed_time(b) for a, b in evs)
    ms = total_ms / args.steps
    nbytes = w.B * w.H * (w.n_q * w.n_k * 4 + (w.n_q + w.n_k) * w.d_k * 2 + w.n_q * 4)
    peaks, peak_src = load_peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": float(peaks["hbm_gbs"]), "unit": "GB/s",
            "peak_source": f"hbm_gbs of {peak_src}", "kernel": "attn_weights_kernel", "algorithmic_bytes": nbytes,
            "frac": round(achieved / float(peaks["hbm_gbs"]), 4), "traffic": None}
    return {
        "metric": "attention weights (softmax matrix) GB/s on 1 GB300 and % of measured HBM bandwidth",
        "value": round(achieved, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": config_of(w, {"l2": L2_NOTE, "pass": "attn_weights (fp32 weights from q, k and lse)",
                                "parallelism": "single GPU"}),
        "roofline": roof,
        "e2e": None,
        "gpu_launches": args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
    }


def run_ours_mha(args, w):
    import torch

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    from transformer_scaled_dot_mha_gb300 import attn

    attn.lib()
    inp = W.make_mha_inputs(w, shard_seed(w, rank))
    self_attn = w.n_q == w.n_k
    to_dev = lambda a: None if a is None else torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    xq = to_dev(inp["x_q"])
    xkv = xq if self_attn else to_dev(inp["x_kv"])
    wts = {k: to_dev(inp[k]) for k in ("w_q", "w_k", "w_v", "w_o", "b_q", "b_k", "b_v", "b_o")}
    kl = inp["key_lens"]
    kld = torch.from_numpy(kl).to(dev)
    key_lens = kld if w.mask_mode & W.MASK_KEY_PADDING else None
    d_model = w.H * w.d_k
    out = torch.empty((w.B, w.n_q, d_model), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(attn.attn_mha_workspace_size(w.B, w.n_q, w.n_k, d_model, w.H, w.d_k), dtype=torch.uint8,
                     device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def layer(x_q, x_kv):
        attn.attn_mha_fwd(x_q, x_kv, wts["w_q"], wts["w_k"], wts["w_v"], wts["w_o"], out, w.H, ws, wts["b_q"],
                          wts["b_k"], wts["b_v"], wts["b_o"], w.scale, w.mask_mode, key_lens, stream)

    for _ in range(args.warmup):
        flush()
        layer(xq, xkv)
    torch.cuda.synchronize()
    st, code = attn.attn_fault_status(stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel fault record {code:#x} during warm-up")
    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        layer(xq, xkv)
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop() if rank == 0 else None
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in evs), dev)
    st, code = attn.attn_fault_status(stream)
    if st != attn.ATTN_OK:
        raise RuntimeError(f"kernel fault record {code:#x} in the timed region")
    flops_step = mha_flops(w, kl)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_tflops(flops_step, args.steps, total_ms, world)

    # end to end: the layer's inputs from pinned host memory, its output back; the
    # weights are the model's parameters and stay on the device
    xqh = xq.cpu().pin_memory()
    xkvh = xqh if self_attn else xkv.cpu().pin_memory()
    klh = torch.from_numpy(kl).pin_memory()
    outh = torch.empty_like(out, device="cpu").pin_memory()
    xq2 = torch.empty_like(xq)
    xkv2 = xq2 if self_attn else torch.empty_like(xkv)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        xq2.copy_(xqh, non_blocking=True)
        if not self_attn:
            xkv2.copy_(xkvh, non_blocking=True)
        if key_lens is not None:
            kld.copy_(klh, non_blocking=True)
        layer(xq2, xkv2)
        outh.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)
    h2d = xqh.numel() * 2 + (0 if self_attn else xkvh.numel() * 2) + (klh.numel() * 4 if key_lens is not None else 0)
    e2e = {"value": round(weak_scaling_tflops(flops_step, 1, e2e_ms, world), 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(outh.numel() * 2), "ms_per_step": round(e2e_ms, 4),
           "steps": e2e_steps, "how": "pinned host x in, y out, copies and kernels on one stream, CUDA events; "
                                     "weights resident on the device"}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return None
    peaks, peak_src = load_peaks()
    achieved = flops_step / (ms_per_step / 1e3) / 1e12
    roof = {"bound": "tensor", "achieved": round(achieved, 2), "peak": float(peaks["bf16_tflops"]),
            "unit": "TFLOP/s", "peak_source": f"bf16_tflops (burst) of {peak_src}",
            "kernel": ("attn_mha_fwd (the Q/K/V projection launch, the attention kernel and the output "
                       "projection launch, timed together)"), "traffic": None}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    line = {
        "metric": "multi-head attention layer TFLOP/s on 1 GB300 and % of dense bf16 tensor peak",
        "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_of(w, {"pass": "multi-head layer (attn_mha_fwd)", "d_model": d_model,
                                "inputs": f"x N(0,1), W N(0,1/rows), b N(0,1) x 0.1, seed {w.seed + 2}",
                                "flops": "algorithmic: four projections 2*d_model*h*d per row + attention",
                                "l2": L2_NOTE,
                                "parallelism": f"independent replicas x{world}" if world > 1 else "single GPU"}),
        "roofline": roof,
        "e2e": e2e,
        "gpu_launches": args.steps * 3,
        "clocks": clk,
        "wall_s_timed_region": round(wall, 3),
    }
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_mha(w)
    return line


# ---------------------------------------------------------------- reference arm
def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    threads = os.cpu_count() or 1
    inputs = W.make_inputs(w)
    ids_all = sample_row_ids(w)
    # per-step sample sized so warm-up + steps take about a minute in total
    budget_s = 60.0 / max(1, args.steps + args.warmup)
    n = threads
    dt = time_oracle(w, inputs, ids_all[:n], threads)
    n = int(max(1, min(ids_all.size // max(1, args.steps + args.warmup), n * budget_s / max(dt, 1e-9))))
    pos = 0
    for _ in range(args.warmup):
        time_oracle(w, inputs, ids_all[pos:pos + n], threads)
        pos = (pos + n) % max(1, ids_all.size - n)
    total_s, total_flops = 0.0, 0.0
    for _ in range(args.steps):
        ids = ids_all[pos:pos + n]
        total_s += time_oracle(w, inputs, ids, threads)
        total_flops += oracle_rows_flops(w, ids, inputs[3])
        pos = (pos + n) % max(1, ids_all.size - n)
    value = total_flops / total_s / 1e12
    sample = (f"each step: {n} query rows drawn uniformly from all {w.B * w.H * w.n_q} rows of the workload, "
              f"fp64 C oracle on {threads} host threads")
    return {"impl": "reference", "metric": "attention fwd TFLOP/s on 1 GB300 and % of dense bf16 tensor peak",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_s / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--grad", action="store_true", help="time the gradients (attn_bwd) instead of the forward")
    ap.add_argument("--mha", action="store_true", help="time the multi-head layer (attn_mha_fwd) instead")
    ap.add_argument("--weights", action="store_true",
                    help="time attn_weights (the fp32 softmax weight matrix) instead of the forward")
    ap.add_argument("--warm-l2", dest="warm_l2", action="store_true",
                    help="forward only: no L2 flush between timed steps, so a workload that fits in L2 is "
                         "read from it (the tensor-roofline view of a short shape; not the default line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = W.WORKLOADS[args.workload]
    if w.dtype != "bf16":
        ap.error("the benchmark times the bf16 tensor-core path; pick a bf16 workload")
    world, rank, _ = dist_env()
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            ap.error("--gpus N > 1 must be launched with torchrun (one process per GPU)")
    if args.weights:
        if args.mha or args.grad or args.impl == "reference" or w.mask_mode & (W.MASK_DECODE | W.MASK_WINDOW):
            ap.error("--weights times attn_weights alone (--impl ours) on the full-attention workloads")
        line = run_ours_weights(args, w)
    elif args.mha:
        if args.grad or w.mask_mode & (W.MASK_DECODE | W.MASK_WINDOW):
            ap.error("--mha covers the forward of the full-attention workloads")
        if args.impl == "reference":
            ap.error("--mha is measured for --impl ours; its line carries the oracle's cpu_baseline")
        line = run_ours_mha(args, w)
    elif args.grad:
        if w.mask_mode & W.MASK_DECODE:
            ap.error("--grad covers the full-attention and local-window workloads (no decode)")
        if args.impl == "reference":
            ap.error("--grad is measured for --impl ours; its line carries the oracle's cpu_baseline")
        line = run_ours_grad(args, w)
    else:
        line = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
