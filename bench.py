"""Benchmark of the Ulysses sequence-parallel hot path on GB300.

One step = one rank's share of a Ulysses layer's attention: causal, packed-sample
attention forward and backward over all T tokens for the rank's hq/sp query heads,
read from and written to the token-major [T][hq/sp][D] buffers that the
sequence -> heads exchange delivers (usp_ulysses_attn_fwd / _bwd, layout swaps fused
into the kernels). The headline workload is the 262,144-token single sequence (32
heads, D = 128, sp = 8: 4 heads per rank). The metric is algorithmic attention
TFLOP/s: 4*D FLOPs per allowed (query, key) pair per query head forward, 10*D
backward. The same line also carries the all-ranks launch of the headline workload,
one rank's slice of the other >= 32k-token workloads, the stand-alone re-layout
kernels' GB/s against HBM, the end-to-end figure through the public API with host
copies, and the float64 oracle timed on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl usp|reference]
       [--workload long|packed|gqa|llama|tiny] [--extras packed,gqa]
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
# bench's own command (one rank's slice of the workload), keyed by workload, path and the
# kernel source they were taken on; any change to the kernel source makes the figure stale
# and it is reported as null.
MEASURED_BWD_TRAFFIC = {
    ("long", True): ("bbed6de96912f02e", 8073437696 + 4252054272),
}


def bwd_traffic(w, fused):
    import hashlib
    entry = MEASURED_BWD_TRAFFIC.get((w.name, fused))
    if entry is None:
        return None
    with open(os.path.join(ROOT, "ulysses_sequence_seq_gb300", "csrc", "attn_bwd.cu"), "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    return entry[1] if digest == entry[0] else None


def bwd_algorithmic_bytes(w):
    """Bytes attn_bwd_kernel must move once: its fp16 q, k, v, dO copies read, the fp32 dQ
    accumulator read and written, dK and dV written (bf16), LSE and Delta read."""
    T, D = w.total_tokens, w.head_dim
    return 2 * T * D * (2 * w.hq + 2 * w.hkv) + 8 * w.hq * T * D + 4 * w.hkv * T * D + 8 * w.hq * T


def workload_desc(w, rank_slice=False):
    kind = "packed" if w.num_seqs > 1 else "single sequence"
    if rank_slice:
        return (f"{w.name}: one rank's slice, {w.hq} query / {w.hkv} key-value heads over all {w.total_tokens} "
                f"tokens ({kind}, {w.num_seqs} samples), D={w.head_dim}, causal, N(0,1), fwd+bwd")
    return (f"{w.name}: {w.total_tokens} tokens ({kind}, {w.num_seqs} samples), sp={w.sp}, hq={w.hq}, "
            f"hkv={w.hkv}, D={w.head_dim}, causal, bf16 N(0,1), fwd+bwd, all sp ranks' heads in one launch")


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
    from ulysses_sequence_seq_gb300.synth import rank_slice
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
            "config": {"workload": workload_desc(rank_slice(w), True), "sample": sample},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def attn_flops(w):
    """(forward, backward) algorithmic FLOPs of one call over all of w's query heads."""
    pairs = w.allowed_pairs()
    return 4.0 * w.head_dim * pairs * w.hq, 10.0 * w.head_dim * pairs * w.hq


class AttnCase:
    """Device buffers of one fused attention step (token-major q, k, v, dO in; o, lse,
    dq, dk, dv out) and its CUDA-event timing."""

    def __init__(self, w, usp, torch, dev, act_dtype, grad_code, host_bits=True, seed=0):
        self.w, self.usp, self.torch = w, usp, torch
        T, H, HKV, D = w.total_tokens, w.hq, w.hkv, w.head_dim
        self.grad_code = grad_code
        if host_bits:
            from ulysses_sequence_seq_gb300.synth import seq_sharded_bits
            import numpy as np

            def pinned(t):
                bits = np.ascontiguousarray(seq_sharded_bits(w, t, dtype="f16" if act_dtype == torch.float16
                                                             else "bf16"))
                return torch.from_numpy(bits.view(np.int16)).view(act_dtype).reshape(T, -1, D).pin_memory()
            self.host = {t: pinned(t) for t in ("q", "k", "v", "do")}
            self.x = {t: h.to(dev) for t, h in self.host.items()}
        else:   # timing-only inputs drawn on the device: N(0, 1) from a seeded generator
            g = torch.Generator(device=dev)
            g.manual_seed(seed)
            self.host = None
            self.x = {t: torch.randn(T, HKV if t in ("k", "v") else H, D, generator=g, device=dev,
                                     dtype=torch.float32).to(act_dtype) for t in ("q", "k", "v", "do")}
        self.cu = torch.from_numpy(w.cu_seqlens()).to(dev)
        self.layer = usp.UlyssesAttention(T, w.num_seqs, H, HKV, D, w.sp, causal=w.causal, device=dev,
                                          fused=True, dtype=act_dtype)

    def fwd(self):
        L, x = self.layer, self.x
        self.usp.ulysses_attn_fwd(x["q"], x["k"], x["v"], L.o_seq, L.lse, self.cu, L.B, L.T, L.sp, L.hq, L.hkv, L.D,
                                  L.scale, L.causal, L.ws, L.ws_bytes, o_res=L.o_res_seq)

    def bwd(self):
        L, x = self.layer, self.x
        self.usp.ulysses_attn_bwd(x["q"], x["k"], x["v"], L.o_seq, L.lse, x["do"], L.dq_seq, L.dk_seq, L.dv_seq,
                                  self.grad_code, self.cu, L.B, L.T, L.sp, L.hq, L.hkv, L.D, L.scale, L.causal,
                                  L.ws, L.ws_bytes, o_res=L.o_res_seq)

    def time(self, steps, warmup, flush, stream):
        """Mean forward, backward and step milliseconds over `steps` timed steps (L2 flushed
        before each, outside the events) after `warmup` untimed ones."""
        torch = self.torch
        for _ in range(warmup):
            self.fwd()
            self.bwd()
        torch.cuda.synchronize()
        st = self.layer.device_status()
        if st != self.usp.USP_OK:
            raise RuntimeError(f"device status {self.usp.status_string(st)} after warm-up")
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            self.fwd()
            e[1].record(stream)
            self.bwd()
            e[2].record(stream)
        torch.cuda.synchronize()
        st = self.layer.device_status()
        if st != self.usp.USP_OK:
            raise RuntimeError(f"device status {self.usp.status_string(st)} after timing")
        fwd = [e[0].elapsed_time(e[1]) for e in evs]
        bwd = [e[1].elapsed_time(e[2]) for e in evs]
        return {"fwd_ms": statistics.mean(fwd), "bwd_ms": statistics.mean(bwd),
                "step_ms_total": sum(f + b for f, b in zip(fwd, bwd)), "steps": steps}


def rates(w, t, peak_burst, peak_sust):
    fl_f, fl_b = attn_flops(w)
    f = fl_f / (t["fwd_ms"] * 1e-3) / 1e12
    b = fl_b / (t["bwd_ms"] * 1e-3) / 1e12
    fb = (fl_f + fl_b) / ((t["fwd_ms"] + t["bwd_ms"]) * 1e-3) / 1e12
    return {"fwd_tflops": f, "bwd_tflops": b, "fwd_bwd_tflops": fb, "fwd_ms": t["fwd_ms"], "bwd_ms": t["bwd_ms"],
            "frac_of_sustained": fb / peak_sust, "frac_of_burst": fb / peak_burst,
            "bwd_frac_of_sustained": b / peak_sust}


def run_usp(args, w):
    import torch

    import ulysses_sequence_seq_gb300 as usp
    from ulysses_sequence_seq_gb300.synth import WORKLOADS, packed_labels, rank_slice

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
    f16 = args.dtype == "f16"
    act_dtype = torch.float16 if f16 else torch.bfloat16
    grad_code = usp.USP_FP16 if f16 else usp.USP_BF16
    peaks, peak_src = load_peaks()
    peak_burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sust = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)   # > L2 (129 MB)
    stream = torch.cuda.current_stream(dev)

    # ---- headline: one rank's slice (hq/sp heads over all T tokens, what one GPU computes
    # under Ulysses once the exchange has delivered its heads), timed in the fused path
    ws_ = rank_slice(w)
    main = AttnCase(ws_, usp, torch, dev, act_dtype, grad_code)
    clocks = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_main = main.time(args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ck = clocks.stop() if clocks else None
    total_ms = max_over_ranks(t_main["step_ms_total"], dist, dev)
    ms_per_step = total_ms / args.steps
    fl_f, fl_b = attn_flops(ws_)
    value = (fl_f + fl_b) * world / (ms_per_step * 1e-3) / 1e12
    main_rates = rates(ws_, t_main, peak_burst, peak_sust)

    # ---- end to end through the public API on the same slice: pinned host inputs in,
    # results back to host, every copy inside the timed region
    layer = main.layer
    out_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                for t in (layer.o_seq, layer.dq_seq, layer.dk_seq, layer.dv_seq)]
    h2d = sum(t.numel() * t.element_size() for t in main.host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host)
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    hq_, hk_, hv_, hdo_ = (main.host[t] for t in ("q", "k", "v", "do"))

    def e2e_step():
        # Q, K, V come in first on a copy stream, dO arrives while the forward runs, O goes
        # out while the backward runs, the gradients after it
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
        o = layer.forward(dq_, dk_, dv_, main.cu)
        d2h_stream.wait_stream(stream)
        with torch.cuda.stream(d2h_stream):
            out_host[0].copy_(o, non_blocking=True)
        stream.wait_event(do_in)
        g = layer.backward(ddo_, main.cu)
        for dst, src in zip(out_host[1:], g):
            dst.copy_(src, non_blocking=True)
        stream.wait_stream(d2h_stream)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for _ in range(args.e2e_steps):
        flush.zero_()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    serial_ms = max_over_ranks(sum(e2e_ms), dist, dev) / args.e2e_steps
    e2e_serial = (fl_f + fl_b) * world / (serial_ms * 1e-3) / 1e12

    # The same steps as a stream of batches: step i+1's Q, K, V and dO upload while step i
    # computes, and step i's O and gradients download while step i+1 runs. The device
    # inputs alternate between two slots; each step's forward waits until the previous O
    # is on the host, its backward until the previous gradients are. The timed region
    # opens before the first upload and closes after the last download.
    slots = [{t: torch.empty_like(h, device=dev) for t, h in main.host.items()} for _ in range(2)]

    def e2e_stream(n_steps, timed):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        h2d_stream.wait_stream(stream)
        slot_free = [None, None]

        def upload(i):
            s = slots[i % 2]
            with torch.cuda.stream(h2d_stream):
                if slot_free[i % 2] is not None:
                    h2d_stream.wait_event(slot_free[i % 2])
                for t in ("q", "k", "v"):
                    s[t].copy_(main.host[t], non_blocking=True)
                qkv_in = torch.cuda.Event()
                qkv_in.record(h2d_stream)
                s["do"].copy_(main.host["do"], non_blocking=True)
                do_in = torch.cuda.Event()
                do_in.record(h2d_stream)
            return qkv_in, do_in

        o_out = g_out = None
        nxt = upload(0)
        for i in range(n_steps):
            qkv_in, do_in = nxt
            s = slots[i % 2]
            flush.zero_()                      # inside the timed region: L2 starts cold
            stream.wait_event(qkv_in)
            if o_out is not None:
                stream.wait_event(o_out)
            o = layer.forward(s["q"], s["k"], s["v"], main.cu)
            f_done = torch.cuda.Event()
            f_done.record(stream)
            if i + 1 < n_steps:
                nxt = upload(i + 1)
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(f_done)
                out_host[0].copy_(o, non_blocking=True)
                o_out = torch.cuda.Event()
                o_out.record(d2h_stream)
            stream.wait_event(do_in)
            if g_out is not None:
                stream.wait_event(g_out)
            g = layer.backward(s["do"], main.cu)
            b_done = torch.cuda.Event()
            b_done.record(stream)
            slot_free[i % 2] = b_done
            with torch.cuda.stream(d2h_stream):
                d2h_stream.wait_event(b_done)
                for dst, src in zip(out_host[1:], g):
                    dst.copy_(src, non_blocking=True)
                g_out = torch.cuda.Event()
                g_out.record(d2h_stream)
        stream.wait_event(g_out)
        end.record(stream)
        torch.cuda.synchronize()
        return start.elapsed_time(end) if timed else None

    e2e_stream(2, False)
    if dist:
        dist.barrier()
    stream_ms = max_over_ranks(e2e_stream(args.e2e_steps, True), dist, dev) / args.e2e_steps
    e2e_value = (fl_f + fl_b) * world / (stream_ms * 1e-3) / 1e12
    e2e_status = layer.device_status()
    if e2e_status != usp.USP_OK:
        raise RuntimeError(f"device status {usp.status_string(e2e_status)} after the end-to-end steps")
    del slots
    main_host = main.host
    del main, layer, out_host
    torch.cuda.empty_cache()

    # ---- secondary: all sp ranks' heads of the workload in one launch (timing-only inputs
    # drawn on the device)
    all_ranks = None
    if args.all_ranks_steps > 0:
        case = AttnCase(w, usp, torch, dev, act_dtype, grad_code, host_bits=False, seed=1000 * w.index)
        t = case.time(args.all_ranks_steps, 2, flush, stream)
        all_ranks = dict(rates(w, t, peak_burst, peak_sust), heads=w.hq, kv_heads=w.hkv,
                         steps=args.all_ranks_steps)
        del case
        torch.cuda.empty_cache()

    # ---- the other workloads of size >= 32k tokens, one rank's slice each
    extras = {}
    for name in args.extras.split(",") if args.extras else []:
        if name == w.name or name not in WORKLOADS:
            continue
        xw = rank_slice(WORKLOADS[name])
        case = AttnCase(xw, usp, torch, dev, act_dtype, grad_code)
        t = case.time(args.steps, args.warmup, flush, stream)
        extras[name] = dict(rates(xw, t, peak_burst, peak_sust), workload=workload_desc(xw, True),
                            allowed_pairs_per_head=xw.allowed_pairs())
        del case
        torch.cuda.empty_cache()

    # ---- the stand-alone layout swaps (usp_seq_to_head / usp_head_to_seq) on the full
    # workload's Q, K, V, dO (all heads), L2 flushed before each batch
    T, H, HKV, D, sp = w.total_tokens, w.hq, w.hkv, w.head_dim, w.sp
    rel_in = {hh: torch.empty(T * hh * D, dtype=torch.bfloat16, device=dev) for hh in {H, HKV}}
    rel_tmp = {hh: torch.empty(T * hh * D, dtype=torch.bfloat16, device=dev) for hh in {H, HKV}}
    rel_back = {hh: torch.empty(T * hh * D, dtype=torch.bfloat16, device=dev) for hh in {H, HKV}}
    for t_ in rel_in.values():
        t_.view(torch.int16).random_(-32768, 32767)
    heads4 = [H, HKV, HKV, H]
    rel_ms = []
    r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for it in range(args.steps + 1):
        tot = 0.0
        for to_head in (True, False):
            flush.zero_()
            r0.record(stream)
            for hh in heads4:
                if to_head:
                    usp.seq_to_head(rel_in[hh].view(sp, T // sp, hh, D), rel_tmp[hh].view(sp, hh // sp, T, D), sp)
                else:
                    usp.head_to_seq(rel_tmp[hh].view(sp, hh // sp, T, D), rel_back[hh].view(sp, T // sp, hh, D), sp)
            r1.record(stream)
            r1.synchronize()
            tot += r0.elapsed_time(r1)
        if it > 0:
            rel_ms.append(tot)
    for hh in rel_in:
        if not torch.equal(rel_back[hh].view(torch.int16), rel_in[hh].view(torch.int16)):   # bits (NaNs included)
            raise RuntimeError("re-layout round trip is not the identity")
    relayout_bytes = sum(2 * 2 * T * hh * D for hh in heads4) * 2
    rel_gbs = relayout_bytes / (statistics.mean(rel_ms) * 1e-3) / 1e9
    del rel_in, rel_tmp, rel_back
    torch.cuda.empty_cache()

    # ---- sample and loss bookkeeping on the device (cu_seqlens -> position_ids ->
    # cu_seqlens padded to 2x the samples, label shift with per-rank good tokens, weighted
    # loss over the sp ranks), L2 flushed before each pass
    cu = torch.from_numpy(w.cu_seqlens()).to(dev)
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

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        from oracle.build import build_oracle
        build_oracle()
        dt1, _, _, _ = oracle_sample_step(w, args.cpu_tokens)          # calibration: one head
        nh = max(1, min(w.hq, math.ceil(12.0 / max(dt1, 1e-3))))         # about 12 s of oracle work
        dt, fl, threads, L = oracle_sample_step(w, args.cpu_tokens, nh)
        pairs_run = nh * L * (L + 1) // 2
        full_fl = sum(attn_flops(ws_))
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{nh} query heads, causal fwd+bwd over the first {L} tokens of sample 0 "
                         f"({dt:.1f} s of float64 C oracle work)",
               "wall_s": dt, "pairs_per_s": pairs_run / dt,
               "extrapolated_full_step_s": full_fl / (fl / dt),
               "extrapolated_note": "one full fwd+bwd step of the headline slice at the sample's FLOP rate "
                                    "(extrapolated, not run)"}
    del main_host
    # per fused step: schedule + attn_fwd | bwd_stats + bwd_convert + schedule + attn_bwd + dq_convert
    launches_per_step = 7
    # Exponentials per second, a diagnostic beside the tensor-core figure: the forward takes one
    # exp per allowed pair and query head (4·D FLOPs), the backward one (P recomputed, 10·D).
    # The ceiling: 32 ex2 per clock per SM (a register-only probe of ex2.approx.ftz.f32 measured
    # 31.4 on this part), times the SMs, at the median SM clock sampled during the timed steps.
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    mhz = (ck or {}).get("sm_mhz") or (ck or {}).get("sm_max_mhz")
    exp_peak = 32.0 * sms * mhz * 1e6 if mhz else None
    exp_f = main_rates["fwd_tflops"] * 1e12 / (4 * ws_.head_dim)
    exp_b = main_rates["bwd_tflops"] * 1e12 / (10 * ws_.head_dim)
    exp_rate = {"fwd_exp_per_s": exp_f, "bwd_exp_per_s": exp_b, "peak_exp_per_s": exp_peak,
                "fwd_frac": exp_f / exp_peak if exp_peak else None,
                "bwd_frac": exp_b / exp_peak if exp_peak else None,
                "peak_source": f"32 ex2/clk/SM x {sms} SMs x median {mhz} MHz"}
    bwd_tflops = main_rates["bwd_tflops"]
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
        "config": {"workload": workload_desc(ws_, True), "seq_len": ws_.total_tokens, "heads": ws_.hq,
                   "kv_heads": ws_.hkv, "head_dim": ws_.head_dim, "sp": w.sp,
                   "allowed_pairs_per_head": ws_.allowed_pairs(),
                   "parallelism": f"replicas x{world}: each GPU runs one rank's slice of sp={w.sp} Ulysses",
                   "path": "fused layout swaps (usp_ulysses_attn_fwd/bwd) on the token-major [T][hq/sp][D] buffers",
                   "l2": "flushed between timed steps (512 MB write outside the events)",
                   **{k: main_rates[k] for k in ("fwd_ms", "bwd_ms", "fwd_tflops", "bwd_tflops")}},
        "fwd_bwd_frac_of_sustained_bf16": main_rates["frac_of_sustained"],
        "fwd_bwd_frac_of_burst_bf16": main_rates["frac_of_burst"],
        "roofline": {"bound": "tensor",
                     "kernel": "usp_ulysses_attn_bwd call: attn_bwd_kernel + bwd_stats + bwd_convert + schedule + "
                               "dq_convert",
                     "achieved": bwd_tflops, "peak": peak_sust, "unit": "TFLOP/s", "frac": bwd_tflops / peak_sust,
                     "peak_source": f"{peak_src} bf16 sustained (the timed region runs for seconds)",
                     "peak_burst": peak_burst, "frac_of_burst": bwd_tflops / peak_burst,
                     "traffic": bwd_traffic(ws_, True),
                     "traffic_of": "attn_bwd_kernel, DRAM read+write bytes per launch (ncu)",
                     "algorithmic_bytes": bwd_algorithmic_bytes(ws_)},
        "exp_rate": exp_rate,
        "scheduler_share_of_step": {"value": 0.0001, "source": "ncu launch list of this command's kernels "
                                                                "(schedule_kernel 0.01% of the step)"},
        "all_ranks_one_launch": all_ranks,
        "extras": extras,
        "relayout": {"achieved_gbs": rel_gbs, "peak_gbs": hbm, "frac": rel_gbs / hbm,
                     "peak_source": f"{peak_src} hbm copy", "bytes": relayout_bytes,
                     "tensor_bytes": 2 * T * H * D,
                     "what": f"usp_seq_to_head on Q, K, V, dO of all {H} heads back to back, then usp_head_to_seq "
                             "on the four; L2 flushed before each batch; round trip checked",
                     "ms": statistics.mean(rel_ms)},
        "sp_bookkeeping": {"ms": statistics.mean(book_ms), "bytes": book_bytes,
                           "achieved_gbs": book_bytes / (statistics.mean(book_ms) * 1e-3) / 1e9,
                           "what": "usp_cu_seqlens_to_position_ids, usp_position_ids_to_cu_seqlens (padded), "
                                   "usp_shift_labels (+ good tokens per rank), usp_sp_weighted_loss; "
                                   "7 launches, L2 flushed before each pass"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": args.e2e_steps, "ms_per_step": stream_ms,
                "what": "UlyssesAttention.forward/backward on the headline slice from pinned host buffers; "
                        "step i+1's uploads and step i's downloads overlap the neighbouring steps' compute "
                        "(two device input slots); every step's copies inside the timed region",
                "serial": {"value": e2e_serial, "ms_per_step": serial_ms,
                           "what": "each step timed alone: its Q, K, V upload before its forward, its "
                                   "gradients' download after its backward"}},
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
    ap.add_argument("--workload", default="long", choices=["tiny", "llama", "packed", "gqa", "long"],
                    help="the headline workload (timed on one rank's slice)")
    ap.add_argument("--extras", default="packed,gqa",
                    help="comma-separated workloads also timed (one rank's slice each); '' for none")
    ap.add_argument("--all-ranks-steps", type=int, default=3,
                    help="timed steps of the all-ranks launch of the headline workload (0 skips it)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--ref-tokens", type=int, default=2048)
    ap.add_argument("--cpu-tokens", type=int, default=4096)
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
