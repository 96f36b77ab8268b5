"""Benchmark of the Ulysses sequence-parallel hot path on GB300.

One step = the whole per-layer attention path for all sp simulated ranks of one
GPU: seq->head swap of Q, K, V; causal packed attention forward; head->seq of O;
seq->head of dO; attention backward; head->seq of dQ, dK, dV. By default the swaps
are fused into the attention kernels (usp_ulysses_attn_fwd / _bwd read and write the
seq-sharded layout); --unfused runs them as separate re-layout kernels. The metric
is algorithmic attention TFLOP/s (4*D FLOPs per allowed (query, key) pair per query
head forward, 10*D backward), plus the stand-alone re-layout kernels' GB/s against HBM.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl usp|reference]
       [--workload llama|tiny|packed|gqa|long]
Under torchrun (N > 1) every rank runs the same per-GPU workload on its own GPU
(weak scaling, no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "local attn fwd+bwd TFLOP/s & % GB300 bf16 peak; re-layout GB/s vs HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# DRAM bytes (read + write) of one attn_bwd_kernel launch from an ncu capture of this
# bench's own command, keyed by workload, path and the kernel source they were taken on;
# any change to the kernel source makes the figure stale and it is reported as null.
MEASURED_BWD_TRAFFIC = {
    ("llama", True): ("fa020faed73a5828", 404870656 + 222942208),
}


def bwd_traffic(w, fused):
    import hashlib
    entry = MEASURED_BWD_TRAFFIC.get((w.name, fused))
    if entry is None:
        return None
    with open(os.path.join(ROOT, "ulysses_sequence_seq_gb300", "csrc", "attn_bwd.cu"), "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    return entry[1] if digest == entry[0] else None


def workload_desc(w):
    kind = "packed" if w.num_seqs > 1 else "single sequence"
    return (f"{w.name}: {w.total_tokens} tokens ({kind}, {w.num_seqs} samples), sp={w.sp}, hq={w.hq}, "
            f"hkv={w.hkv}, D={w.head_dim}, causal, bf16 N(0,1), fwd+bwd, all sp ranks' heads in one launch")


def attention_flops(w):
    pairs = w.allowed_pairs()
    return 4.0 * w.head_dim * pairs * w.hq, 10.0 * w.head_dim * pairs * w.hq


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [l.strip().split(", ") for l in self.file.read().splitlines() if l.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest `value` over all ranks (timing is reported for the slowest rank)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample_step(w, tokens: int, heads: int = 1):
    """The oracle's fwd+bwd on the first `heads` query heads (MHA: each with its own
    key/value head) over the first `tokens` tokens of the workload's first sample;
    returns (seconds, algorithmic FLOPs credited, threads, tokens)."""
    import numpy as np

    import oracle
    from ulysses_sequence_seq_gb300.synth import head_bits
    L = min(tokens, w.lengths[0])
    hs = range(heads)
    q = np.stack([head_bits(w, "q", h)[:L] for h in hs])
    k = np.stack([head_bits(w, "k", h % w.hkv)[:L] for h in hs])
    v = np.stack([head_bits(w, "v", h % w.hkv)[:L] for h in hs])
    do = np.stack([head_bits(w, "do", h)[:L] for h in hs])
    cu = np.array([0, L], dtype=np.int32)
    t0 = time.perf_counter()
    oracle.attn_fwd(q, k, v, cu)
    oracle.attn_bwd(q, k, v, do, cu)
    dt = time.perf_counter() - t0
    pairs = L * (L + 1) // 2
    return dt, 14.0 * w.head_dim * pairs * heads, oracle.num_threads(), L


def run_reference(args, w):
    """The CPU oracle as the reference arm (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle.build import build_oracle
    build_oracle()
    tokens = args.ref_tokens
    for _ in range(args.warmup):
        oracle_sample_step(w, min(tokens, 256))
    times, flops = [], 0.0
    for _ in range(args.steps):
        dt, fl, threads, L = oracle_sample_step(w, tokens)
        times.append(dt)
        flops = fl
    mean = sum(times) / len(times)
    value = flops / mean / 1e12
    sample = (f"one query head, causal fwd+bwd over the first {L} tokens of sample 0 of the {w.name} "
              f"workload per step (float64 C oracle)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(w), "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_usp(args, w):
    import numpy as np
    import torch

    import ulysses_sequence_seq_gb300 as usp
    from ulysses_sequence_seq_gb300.synth import packed_labels, seq_sharded_bits

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    usp.load()
    dev = torch.device("cuda", local_rank)
    T, H, HKV, D, sp = w.total_tokens, w.hq, w.hkv, w.head_dim, w.sp

    f16 = args.dtype == "f16"
    if f16 and args.unfused:
        raise SystemExit("fp16 activations run on the fused path only")
    act_dtype = torch.float16 if f16 else torch.bfloat16
    grad_code = usp.USP_FP16 if f16 else usp.USP_BF16

    def to_host_pinned(bits):
        t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(act_dtype)
        return t.pin_memory()

    hq_, hk_, hv_, hdo_ = (to_host_pinned(seq_sharded_bits(w, t, dtype=args.dtype)) for t in ("q", "k", "v", "do"))
    xq, xk, xv, xdo = (t.to(dev) for t in (hq_, hk_, hv_, hdo_))
    cu = torch.from_numpy(w.cu_seqlens()).to(dev)
    fused = not args.unfused
    layer = usp.UlyssesAttention(T, w.num_seqs, H, HKV, D, sp, causal=True, device=dev, fused=fused, dtype=act_dtype)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)   # > L2 (129 MB)
    stream = torch.cuda.current_stream(dev)

    # events: 0 start | 1 after the seq->head swaps (unfused) | 2 after the forward |
    #         3 after the O / dO swaps (unfused) | 4 after the backward | 5 end
    def step(ev=None):
        if ev is None:
            layer.forward(xq, xk, xv, cu)
            layer.backward(xdo, cu)
            return
        ev[0].record(stream)
        if fused:
            ev[1].record(stream)
            usp.ulysses_attn_fwd(xq, xk, xv, layer.o_seq, layer.lse, cu, layer.B, T, sp, H, HKV, D, layer.scale,
                                 True, layer.ws, layer.ws_bytes)
            ev[2].record(stream)
            ev[3].record(stream)
            usp.ulysses_attn_bwd(xq, xk, xv, layer.o_seq, layer.lse, xdo, layer.dq_seq, layer.dk_seq, layer.dv_seq,
                                 grad_code, cu, layer.B, T, sp, H, HKV, D, layer.scale, True, layer.ws,
                                 layer.ws_bytes)
            ev[4].record(stream)
            ev[5].record(stream)
            return
        usp.seq_to_head(xq, layer.q_h, sp)
        usp.seq_to_head(xk, layer.k_h, sp)
        usp.seq_to_head(xv, layer.v_h, sp)
        ev[1].record(stream)
        usp.attn_fwd_varlen(layer.q_h, layer.k_h, layer.v_h, layer.o_h, layer.lse, cu, layer.B, T, H, HKV, D,
                            layer.scale, True, layer.ws, layer.ws_bytes)
        ev[2].record(stream)
        usp.head_to_seq(layer.o_h, layer.o_seq, sp)
        usp.seq_to_head(xdo, layer.do_h, sp)
        ev[3].record(stream)
        usp.attn_bwd_varlen(layer.q_h, layer.k_h, layer.v_h, layer.o_h, layer.lse, layer.do_h, layer.dq_h,
                            layer.dk_h, layer.dv_h, usp.USP_BF16, cu, layer.B, T, H, HKV, D, layer.scale, True,
                            layer.ws, layer.ws_bytes)
        ev[4].record(stream)
        usp.head_to_seq(layer.dq_h, layer.dq_seq, sp)
        usp.head_to_seq(layer.dk_h, layer.dk_seq, sp)
        usp.head_to_seq(layer.dv_h, layer.dv_seq, sp)
        ev[5].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if layer.device_status() != usp.USP_OK:
        raise RuntimeError(f"device status {usp.status_string(layer.device_status())} after warm-up")

    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()                          # evict L2 between timed steps (outside the events)
        step(evs[i])
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ck = clocks.stop() if clocks else None
    if layer.device_status() != usp.USP_OK:
        raise RuntimeError(f"device status {usp.status_string(layer.device_status())} after timing")

    step_ms = [e[0].elapsed_time(e[5]) for e in evs]
    fwd_ms = [e[1].elapsed_time(e[2]) for e in evs]
    bwd_ms = [e[3].elapsed_time(e[4]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    ms_per_step = total_ms / args.steps
    fwd_fl, bwd_fl = attention_flops(w)
    value = (fwd_fl + bwd_fl) * world / (ms_per_step * 1e-3) / 1e12

    # ---- the stand-alone layout swaps (usp_seq_to_head / usp_head_to_seq) on this workload's
    # eight tensors, L2 flushed before each: the metric's re-layout GB/s against HBM
    rel_bufs = [(xq, H), (xk, HKV), (xv, HKV), (xdo, H)]
    rel_tmp = {hh: torch.empty(T * hh * D, dtype=torch.bfloat16, device=dev) for hh in {H, HKV}}
    rel_back = {hh: torch.empty(T * hh * D, dtype=torch.bfloat16, device=dev) for hh in {H, HKV}}
    rel_ms = []
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for it in range(args.steps + 1):
        tot = 0.0
        for to_head in (True, False):          # a layer swaps Q, K, V (and dO) together
            flush.zero_()
            r0.record(stream)
            for x, hh in rel_bufs:
                if to_head:
                    usp.seq_to_head(x, rel_tmp[hh].view(sp, hh // sp, T, D), sp)
                else:
                    usp.head_to_seq(rel_tmp[hh].view(sp, hh // sp, T, D), rel_back[hh].view(sp, T // sp, hh, D), sp)
            r1.record(stream)
            r1.synchronize()
            tot += r0.elapsed_time(r1)
        if it > 0:                             # the first pass is a warm-up
            rel_ms.append(tot)
    relayout_bytes = sum(2 * 2 * T * hh * D for _, hh in rel_bufs) * 2   # read + write, both directions

    # ---- sample and loss bookkeeping on the device: cu_seqlens -> position_ids ->
    # cu_seqlens (padded to 2x the samples), label shift with per-rank good-token counts,
    # weighted loss over the sp ranks; L2 flushed before each pass
    max_seqs = 2 * w.num_seqs
    pos_d = torch.empty(T, dtype=torch.int64, device=dev)
    cu_pad = torch.empty(max_seqs + 1, dtype=torch.int32, device=dev)
    nseq_d = torch.empty(1, dtype=torch.int32, device=dev)
    pws_bytes = usp.position_ids_workspace_size(T)
    pws = torch.zeros(pws_bytes, dtype=torch.uint8, device=dev)
    labels_d = torch.from_numpy(packed_labels(w.cu_seqlens(), vocab=32000, seed=1000 * w.index + 50)).to(dev)
    shifted_d = torch.empty(T, dtype=torch.int64, device=dev)
    good_d = torch.empty(sp, dtype=torch.int64, device=dev)
    rank_loss_d = torch.rand(sp, dtype=torch.float32, device=dev) * 4
    loss_d = torch.empty((), dtype=torch.float32, device=dev)
    book_ms = []
    for it in range(args.steps + 1):
        flush.zero_()
        r0.record(stream)
        usp.cu_seqlens_to_position_ids(cu, w.num_seqs, T, pos_d)
        usp.position_ids_to_cu_seqlens(pos_d, T, cu_pad, max_seqs, nseq_d, pws, pws_bytes)
        usp.shift_labels(labels_d, cu_pad, max_seqs, T, sp, shifted_d, good_d)
        usp.sp_weighted_loss(rank_loss_d, good_d, sp, loss_d)
        r1.record(stream)
        r1.synchronize()
        if it > 0:
            book_ms.append(r0.elapsed_time(r1))
    if usp.get_device_status(pws) != usp.USP_OK or int(nseq_d.item()) != w.num_seqs:
        raise RuntimeError("position_ids -> cu_seqlens failed on the bench workload")
    book_bytes = 8 * T + 8 * T + 16 * T     # write ids; read ids; read labels + write shifted

    # ---- end to end through the public API: pinned host inputs in, results back to host
    out_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for t in (layer.o_seq, layer.dq_seq, layer.dk_seq, layer.dv_seq)]
    h2d = sum(t.numel() * t.element_size() for t in (hq_, hk_, hv_, hdo_))
    d2h = sum(t.numel() * t.element_size() for t in out_host)

    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)

    def e2e_step():
        # Every copy of the step is inside the timed region; they overlap the compute they do
        # not feed: Q, K, V come in first on a copy stream, dO arrives while the forward runs,
        # and O goes out while the backward runs.
        h2d_stream.wait_stream(stream)
        with torch.cuda.stream(h2d_stream):
            dq_, dk_, dv_ = (t.to(dev, non_blocking=True) for t in (hq_, hk_, hv_))
            qkv_in = torch.cuda.Event()
            qkv_in.record(h2d_stream)
            ddo_ = hdo_.to(dev, non_blocking=True)
            do_in = torch.cuda.Event()
            do_in.record(h2d_stream)
        for t in (dq_, dk_, dv_, ddo_):
            t.record_stream(stream)
        stream.wait_event(qkv_in)
        o = layer.forward(dq_, dk_, dv_, cu)
        d2h_stream.wait_stream(stream)
        with torch.cuda.stream(d2h_stream):
            out_host[0].copy_(o, non_blocking=True)
        stream.wait_event(do_in)
        g = layer.backward(ddo_, cu)
        for dst, src in zip(out_host[1:], g):
            dst.copy_(src, non_blocking=True)
        stream.wait_stream(d2h_stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for _ in range(args.steps):
        flush.zero_()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_value = (fwd_fl + bwd_fl) * world / (statistics.mean(e2e_ms) * 1e-3) / 1e12

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    peaks, peak_src = load_peaks()
    bwd_mean = statistics.mean(bwd_ms)
    fwd_mean = statistics.mean(fwd_ms)
    bwd_tflops = bwd_fl / (bwd_mean * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    rel_gbs = relayout_bytes / (statistics.mean(rel_ms) * 1e-3) / 1e9
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        from oracle.build import build_oracle
        build_oracle()
        dt1, _, _, _ = oracle_sample_step(w, args.cpu_tokens)          # calibration: one head
        nh = max(1, min(w.hq, math.ceil(12.0 / max(dt1, 1e-3))))         # about 12 s of oracle work
        dt, fl, threads, L = oracle_sample_step(w, args.cpu_tokens, nh)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{nh} query heads, causal fwd+bwd over the first {L} tokens of sample 0 "
                         f"({dt:.1f} s of float64 C oracle work)"}
    # fused: schedule + attn_fwd | bwd_prep + schedule + attn_bwd + dq_convert;
    # unfused adds the eight re-layout launches
    launches_per_step = 6 if fused else 14
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": workload_desc(w), "seq_len": T, "heads": H, "kv_heads": HKV, "head_dim": D,
                   "sp": sp, "parallelism": f"replicas x{world} (sp={sp} simulated per GPU)",
                   "path": "fused layout swaps (usp_ulysses_attn_fwd/bwd)" if fused else
                           "separate re-layout kernels around usp_attn_fwd/bwd_varlen",
                   "l2": "flushed between timed steps (512 MB write outside the events)",
                   "fwd_ms": fwd_mean, "bwd_ms": bwd_mean,
                   "fwd_tflops": fwd_fl / (fwd_mean * 1e-3) / 1e12, "bwd_tflops": bwd_tflops},
        "roofline": {"bound": "tensor",
                     "kernel": ("usp_ulysses_attn_bwd" if fused else "usp_attn_bwd_varlen") +
                               " call: attn_bwd_kernel + bwd_prep + schedule + dq_convert",
                     "achieved": bwd_tflops, "peak": peak, "unit": "TFLOP/s", "frac": bwd_tflops / peak,
                     "peak_source": f"{peak_src} bf16 burst", "traffic": bwd_traffic(w, fused),
                     "traffic_of": "attn_bwd_kernel, DRAM read+write bytes per launch (ncu)"},
        "relayout": {"achieved_gbs": rel_gbs, "peak_gbs": hbm, "frac": rel_gbs / hbm,
                     "peak_source": f"{peak_src} hbm copy", "bytes": relayout_bytes,
                     "what": "usp_seq_to_head on Q, K, V, dO back to back, then usp_head_to_seq on the four; "
                             "L2 flushed before each batch",
                     "ms": statistics.mean(rel_ms)},
        "sp_bookkeeping": {"ms": statistics.mean(book_ms), "bytes": book_bytes,
                           "achieved_gbs": book_bytes / (statistics.mean(book_ms) * 1e-3) / 1e9,
                           "what": "usp_cu_seqlens_to_position_ids, usp_position_ids_to_cu_seqlens (padded), "
                                   "usp_shift_labels (+ good tokens per rank), usp_sp_weighted_loss; "
                                   "7 launches, L2 flushed before each pass; latency-bound at this T"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": ck,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="usp", choices=["usp", "reference"])
    ap.add_argument("--workload", default="llama", choices=["tiny", "llama", "packed", "gqa", "long"])
    ap.add_argument("--ref-tokens", type=int, default=2048)
    ap.add_argument("--cpu-tokens", type=int, default=4096)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused", action="store_true", help="time separate re-layout kernels around the attention")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f16"],
                    help="activation type (fp32 accumulation and softmax either way)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    from ulysses_sequence_seq_gb300.synth import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_usp(args, w)


if __name__ == "__main__":
    main()
