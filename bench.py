"""Throughput of the GQA attention hot path on GB300.

Default run (N=1): the Llama-3-8B-shaped prefill (B=4, L=2048, H=32, Hkv=8,
D=128, rope_theta 5e5 with the Llama 3 ramp, causal). One step is the whole
prefill path through the C ABI: RoPE on q, the fused K RoPE + cache append,
and the prefill attention. value = attention FLOP per step / step time.

The same line carries the decode half of the metric, measured on the
64-row batched decode (cached lengths U{512..8192}, H=32, Hkv=8, D=128): one
step is RoPE on q, the append of the new token and the split-KV decode;
GB/s = K/V cache bytes read per step / step time.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torchrun: each rank runs the same workload on its own
GPU (the path needs no exchange between GPUs), value sums all ranks' work over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill attn TFLOP/s (% TC peak); decode KV-cache GB/s (% of 8 TB/s HBM)"
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25        # dense TF32 vs dense BF16 nominal rates
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--decode-steps", type=int, default=200)
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--workload", default="llama3_8b_prefill",
                    choices=["llama3_8b_prefill", "gemma2_window"],
                    help="prefill workload of the timed step")
    ap.add_argument("--no-chunked", action="store_true",
                    help="skip the chunked prefill continuing a cached prefix")
    ap.add_argument("--no-long-decode", action="store_true",
                    help="skip the carried-cache decode (1024 steps after a 1024-token prefill)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the steps as eager launches instead of CUDA graph replays")
    ap.add_argument("--separate-append", action="store_true",
                    help="time kv_cache_append + gqa_attn_v_transpose + gqa_attn_prefill_rope_vt "
                         "as the step instead of the fused gqa_attn_prefill_step")
    ap.add_argument("--unfused-q-rope", action="store_true",
                    help="time attn_rope_apply on q + gqa_attn_prefill instead of the fused call")
    ap.add_argument("--no-gemma", action="store_true",
                    help="skip the Gemma-2-shaped window prefill key")
    ap.add_argument("--no-block", action="store_true",
                    help="skip the decoder block and projection (attn_linear) keys")
    ap.add_argument("--no-identical", action="store_true",
                    help="skip the identical-numeric-mode timings")
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="rows of the batched decode (default: the workload's 64; smaller "
                         "values are for profiling captures)")
    return ap.parse_args()


def peaks():
    p = {"hbm_gbs": 6669.5, "bf16_tflops": 1926.5, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        p.update({"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                  "source": "measured"})
    p["tf32_tflops"] = p["bf16_tflops"] * NOMINAL_TF32_OVER_BF16
    return p


# DRAM bytes (read + write) per launch from the committed ncu captures of the
# current kernels (profiles/); None where no capture of the timed kernel exists.
# The decode capture ran on 16 of the 64 rows; its traffic scales with the
# algorithmic bytes processed (ratio below).
NCU_PREFILL_TRAFFIC = {("llama3_8b_prefill", "fused"): 347.001088e6 + 96.9472e6,
                       ("gemma2_window", "fused"): 1915.213e6 + 244.01664e6}
NCU_DECODE_TRAFFIC_PER_ALG_BYTE = (585.903872e6 + 4.77312e6) / 585572352.0
# gemm_tc2_kernel (the CTA-pair projection kernel) at the down projection's shape (T=8192, N=4096, K=14336), one launch.
NCU_GEMM_TRAFFIC = 2422.774e6 + 122.948352e6


def measure_tf32_peak(dev):
    """Dense TF32 matmul rate of this GPU, measured the same way as the bf16
    figure: cuBLAS fp32 8192^3 with TF32 allowed, best of 10 (CUDA events)."""
    import torch
    n = 8192
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        gen = torch.Generator(device=dev).manual_seed(0)
        a = torch.randn(n, n, device=dev, generator=gen)
        b = torch.randn(n, n, device=dev, generator=gen)
        c = torch.empty(n, n, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = float("inf")
        for _ in range(10):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            e1.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b, c
        torch.cuda.empty_cache()
        return 2.0 * n ** 3 / (best * 1e-3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() in ("active", "yes", "1"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def reduce_max(ms, dist):
    """The largest of the ranks' timings, returned on every rank (ms itself with no group).
    The reduction runs on the GPU under NCCL and on the host under gloo."""
    if not dist:
        return ms
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def timed(fn, steps, warmup, dist, events_for=None):
    """Run fn() warmup + steps times; device time of the timed steps (ms, max over ranks)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    if dist:
        ms = reduce_max(ms, dist)
        dist.barrier()
    torch.cuda.synchronize()
    return ms


def kernel_median(fn, iters=50, warm=10):
    """Device time of one call of fn (ms): warm-up calls, then the median of `iters`
    calls each bracketed by CUDA events on the launching stream."""
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    evs = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs)


KERNEL_ITERS, KERNEL_WARM = 50, 10


def graph_of(fn, warm=3):
    """fn's launches captured once into a CUDA graph (warmed up on a side stream
    first); replaying it takes the per-call host work out of the step."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        fn()
    torch.cuda.synchronize()
    return gr


def visible_pairs(L, window):
    """Number of (query, key) pairs the causal (or windowed) mask admits in one row."""
    if window <= 0 or window >= L:
        return L * (L + 1) // 2
    return window * (window + 1) // 2 + (L - window) * window


def prefill_flops(w, B=None, H=None):
    B = w.B if B is None else B
    H = w.H if H is None else H
    return 4.0 * B * H * w.D * visible_pairs(w.L, w.window)


def prefill_bytes(w):
    """Bytes the prefill step touches: q, k, v, out and both cache buffers."""
    cap = w.window if w.window else w.capacity
    return 4 * (2 * w.B * w.H * w.L * w.D + 2 * w.B * w.Hkv * w.L * w.D
                + 2 * w.B * w.Hkv * cap * w.D)


def bench_prefill(w, args, dist, dev, rank, steps=None, e2e=True):
    import torch
    import gqa_causal_attention_gb300 as g
    from gqa_causal_attention_gb300 import synthetic as syn

    steps = args.steps if steps is None else steps
    inp = syn.prefill_inputs(w)
    rp = g.RopeParams.make(theta=w.theta, rope_dim=w.rope_dim, max_positions=w.max_positions,
                           scaling=w.scaling)
    table = g.rope_table(rp, w.D, dev)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    qn = None if inp["q_norm_w"] is None else inp["q_norm_w"].to(dev)
    kn = None if inp["k_norm_w"] is None else inp["k_norm_w"].to(dev)
    cap = w.window if w.window else w.capacity
    kc = torch.zeros(w.B, w.Hkv, cap, w.D, device=dev)
    vc = torch.zeros_like(kc)
    out = torch.empty_like(q)
    start = torch.zeros(w.B, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pws = torch.empty(max(4, g.gqa_attn_prefill_rope_workspace_size(w.B, w.H, w.Hkv, w.L, w.D,
                                                                    rp) // 4), device=dev)
    vt = torch.empty(w.B * w.Hkv * w.D * g.gqa_attn_vt_pitch(w.L), device=dev)
    vws = torch.empty(max(4, g.gqa_attn_prefill_rope_vt_workspace_size(w.B, w.H, w.L, w.D, rp)
                          // 4), device=dev)
    sws = torch.empty(max(4, g.gqa_attn_prefill_step_workspace_size(w.B, w.H, w.Hkv, w.L, w.D,
                                                                    w.window, rp) // 4),
                      device=dev)
    # q's RMSNorm/RoPE runs inside the attention kernel when the kernel takes it (no
    # workspace needed), else as a pass over q inside the call
    q_fused = g.gqa_attn_prefill_rope_vt_workspace_size(w.B, w.H, w.L, w.D, rp) <= 16
    separate = args.separate_append or args.unfused_q_rope

    def step():
        if not separate:
            # one call: k RMSNorm/RoPE into the cache, v into the cache and transposed
            # (one memory pass over k and v), then attention with q's RMSNorm/RoPE fused,
            # reading the rotated keys from the cache
            g.gqa_attn_prefill_step(q, k, v, out, kc, vc, rp, table, qn, kn, w.norm_eps,
                                    w.window, w.softcap, 0.0, workspace=sws, status=status)
            return
        # k: RMSNorm + RoPE in place and into the cache; v transposed for the tensor cores;
        # q: RMSNorm + RoPE inside the attention kernel (or a pass inside the call)
        g.kv_cache_append(k, v, start, 0, rp, table, kn, w.norm_eps, kc, vc, w.window, status)
        if args.unfused_q_rope:
            g.attn_rope_apply(q, start, 0, rp, table, qn, w.norm_eps, status)
            g.gqa_attn_prefill(q, k, v, out, w.window, w.softcap, 0.0, workspace=pws,
                               status=status)
        else:
            g.gqa_attn_v_transpose(v, vt)
            g.gqa_attn_prefill_rope_vt(q, k, vt, out, start, 0, rp, table, qn, w.norm_eps,
                                       w.window, w.softcap, 0.0, workspace=vws, status=status)

    ms_eager = timed(step, steps, args.warmup, dist)
    launches_per_step = (2 if not separate else 3) + (0 if q_fused or args.unfused_q_rope
                                                      else 1)
    # The step as a CUDA graph: the whole-step time.
    with ClockSampler(torch.cuda.current_device()) as clk:
        if args.no_graph:
            ms = timed(step, steps, args.warmup, dist)
        else:
            gr = graph_of(step)
            ms = timed(gr.replay, steps, args.warmup, dist)
    torch.cuda.synchronize()
    # The attention kernel alone (the roofline): rotated keys and V^T prepared once; with
    # q rotated in the kernel, the call itself; otherwise q rotated once beforehand and
    # the call without RoPE.
    if not separate:
        krot = k.clone()
        g.kv_cache_append(krot, v, start, 0, rp, table, kn, w.norm_eps, kc, vc, w.window,
                          status)
        g.gqa_attn_v_transpose(v, vt)
    else:
        krot = k
    if args.unfused_q_rope:
        qrot = q
    elif q_fused:
        qrot = None
    else:
        qrot = q.clone()
        g.attn_rope_apply(qrot, start, 0, rp, table, qn, w.norm_eps, status)

    def attention():
        if args.unfused_q_rope:
            g.gqa_attn_prefill(qrot, krot, v, out, w.window, w.softcap, 0.0, workspace=pws,
                               status=status)
        elif q_fused:
            g.gqa_attn_prefill_rope_vt(q, krot, vt, out, start, 0, rp, table, qn, w.norm_eps,
                                       w.window, w.softcap, 0.0, workspace=vws, status=status)
        else:
            g.gqa_attn_prefill_rope_vt(qrot, krot, vt, out, None, 0, None, None, None,
                                       w.norm_eps, w.window, w.softcap, 0.0, status=status)

    kern_ms = kernel_median(attention, KERNEL_ITERS, KERNEL_WARM)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    kernel_launches = (2 if args.unfused_q_rope else 1) * (KERNEL_ITERS + KERNEL_WARM)
    res = {"ms": ms / steps, "ms_eager": ms_eager / steps, "kernel_ms": kern_ms,
           "clocks": clk.summary(), "launches_per_step": launches_per_step,
           "q_fused": q_fused,
           "launches": launches_per_step * 2 * steps + kernel_launches}
    del qrot, krot

    if e2e and not args.no_e2e:
        hq, hk, hv = (inp[n].pin_memory() for n in ("q", "k", "v"))
        hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        cap = kc.shape[2]
        hws = torch.empty(max(4, g.gqa_attn_prefill_from_host_workspace_size(
            w.B, w.H, w.Hkv, w.L, w.D, cap, rp) // 4), device=dev)

        def e2e_step():
            # one C-ABI call from pinned host buffers: row chunks of q, k, v in, append and
            # attention, out back, copies and kernels of different chunks overlapped
            g.gqa_attn_prefill_from_host(hq, hk, hv, hout, q, k, v, out, kc, vc, start, 0, rp,
                                         table, qn, kn, w.norm_eps, w.window, w.softcap, 0.0,
                                         workspace=hws, status=status)

        def e2e_serial_step():
            # the same step with the copies and the kernels one after another on one stream
            q.copy_(hq, non_blocking=True)
            k.copy_(hk, non_blocking=True)
            v.copy_(hv, non_blocking=True)
            step()
            hout.copy_(out, non_blocking=True)

        e_steps = max(3, min(args.steps, 50))
        ems = timed(e2e_step, e_steps, 3, dist)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item())}"
        res["e2e_ms"] = ems / e_steps
        res["e2e_serial_ms"] = timed(e2e_serial_step, e_steps, 3, dist) / e_steps
        if w.B >= 16:                           # the call's chunks (at most 16)
            chunks = -(-w.B // -(-w.B // 16))
        else:
            per_row = -(-w.Hkv // -(-w.Hkv // (16 // w.B)))
            chunks = w.B * per_row
        res["e2e_launches"] = 3 * chunks * e_steps + res["launches_per_step"] * e_steps
        res["launches"] += res["e2e_launches"]
        res["e2e_chunks"] = chunks
        res["h2d"] = sum(t.numel() * 4 for t in (hq, hk, hv))
        res["d2h"] = hout.numel() * 4
    return res


def bench_decode(w, args, dist, dev):
    import torch
    import gqa_causal_attention_gb300 as g
    from gqa_causal_attention_gb300 import synthetic as syn

    n = syn.cache_lengths(w.seed, w.B, *w.cache_len_range)
    gen = torch.Generator(device=dev).manual_seed(w.seed)
    kc = torch.randn(w.B, w.Hkv, w.capacity, w.D, device=dev, generator=gen)
    vc = torch.randn(w.B, w.Hkv, w.capacity, w.D, device=dev, generator=gen)
    tok = syn.decode_token_inputs(w, 0)
    q, k, v = (tok[x].to(dev) for x in ("q", "k", "v"))
    rp = g.RopeParams.make(theta=w.theta, rope_dim=w.rope_dim, max_positions=w.max_positions,
                           scaling=w.scaling)
    table = g.rope_table(rp, w.D, dev)
    pos = n.to(dev)
    cl = (n + 1).to(dev)
    maxlen = int(n.max()) + 1
    ws = torch.empty(max(4, g.gqa_attn_decode_workspace_size(w.B, w.H, w.Hkv, w.D, maxlen,
                                                             w.window) // 4), device=dev)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    sws = torch.empty(g.gqa_attn_decode_step_workspace_size(w.B, w.H, w.Hkv, w.D, maxlen - 1,
                                                            w.window) // 4 + 4, device=dev)
    qrot = q.clone()
    g.attn_rope_apply(qrot, pos, maxlen - 1, rp, table, None, w.norm_eps, status)

    def step():
        # one call: q and k rotated at position n_b, k and v appended, then the split-KV
        # decode and the combine of its splits
        g.gqa_attn_decode_step(q, k, v, out, pos, maxlen - 1, kc, vc, rp, table, None, None,
                               w.norm_eps, w.window, w.softcap, 0.0, workspace=sws,
                               status=status)

    steps = args.decode_steps
    ms_eager = timed(step, steps, args.warmup, dist)
    with ClockSampler(torch.cuda.current_device()) as clk:
        if args.no_graph:
            ms = timed(step, steps, args.warmup, dist)
        else:
            gr = graph_of(step)
            ms = timed(gr.replay, steps, args.warmup, dist)
    kern_ms = kernel_median(
        lambda: g.gqa_attn_decode(qrot, kc, vc, cl, maxlen, out, 0, w.softcap, 0.0, ws, status),
        KERNEL_ITERS, KERNEL_WARM)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    nbytes = 2.0 * w.Hkv * w.D * 4 * float((n + 1).sum())
    ksplit = 2 if g.gqa_attn_decode_workspace_size(w.B, w.H, w.Hkv, w.D, maxlen, w.window) > 16 \
        else 1
    per_step = decode_step_launches(w, maxlen)
    return {"ms": ms / steps, "ms_eager": ms_eager / steps, "kernel_ms": kern_ms, "bytes": nbytes,
            "clocks": clk.summary(),
            "launches_per_step": per_step,
            "launches": per_step * 2 * steps + ksplit * (KERNEL_ITERS + KERNEL_WARM)}


def decode_step_launches(w, cache_len):
    """Kernels of one gqa_attn_decode_step over cache_len positions, as the library
    reports them: the RoPE/append pass unless the decode kernel does it, the decode
    kernel, and the combine of a row's splits unless a cluster merges them."""
    import gqa_causal_attention_gb300 as g
    return g.gqa_attn_decode_launches(w.B, w.H, w.Hkv, w.D, cache_len, w.window, w.R)


def bench_long_decode(w, args, dist, dev):
    """The carried-cache decode workload: a cache filled by a 1024-token prefill's
    append, then 1024 single-token steps (q RoPE, k RoPE + append, decode over the
    growing cache), all 1024 captured in one CUDA graph and replayed."""
    import torch
    import gqa_causal_attention_gb300 as g

    gen = torch.Generator(device=dev).manual_seed(w.seed)
    rp = g.RopeParams.make(theta=w.theta, rope_dim=w.rope_dim, max_positions=w.max_positions,
                           scaling=w.scaling)
    table = g.rope_table(rp, w.D, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    kc = torch.zeros(w.B, w.Hkv, w.capacity, w.D, device=dev)
    vc = torch.zeros_like(kc)
    k0 = torch.randn(w.B, w.Hkv, w.L, w.D, device=dev, generator=gen)
    v0 = torch.randn(w.B, w.Hkv, w.L, w.D, device=dev, generator=gen)
    zero = torch.zeros(w.B, dtype=torch.int32, device=dev)
    g.kv_cache_append(k0, v0, zero, 0, rp, table, None, w.norm_eps, kc, vc, 0, status)
    n = w.decode_steps
    qs = torch.randn(n, w.B, w.H, 1, w.D, device=dev, generator=gen)
    ks = torch.randn(n, w.B, w.Hkv, 1, w.D, device=dev, generator=gen)
    vs = torch.randn(n, w.B, w.Hkv, 1, w.D, device=dev, generator=gen)
    out = torch.empty(w.B, w.H, 1, w.D, device=dev)
    pos = torch.arange(w.L, w.L + n, dtype=torch.int32, device=dev).repeat(w.B, 1).t().contiguous()
    cl = (pos + 1).contiguous()
    ws = torch.empty(max(4, g.gqa_attn_decode_step_workspace_size(w.B, w.H, w.Hkv, w.D,
                                                                   w.L + n - 1, 0) // 4),
                     device=dev)

    def steps():
        for t in range(n):
            p = w.L + t
            g.gqa_attn_decode_step(qs[t], ks[t], vs[t], out, pos[t], p, kc, vc, rp, table, None,
                                   None, w.norm_eps, 0, 0.0, 0.0, workspace=ws, status=status)

    gr = graph_of(steps, warm=1)
    with ClockSampler(torch.cuda.current_device()) as clk:
        ms = timed(gr.replay, 1, 2, dist)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    nbytes = 2.0 * w.Hkv * w.D * 4 * w.B * sum(w.L + t + 1 for t in range(n))
    launches = sum(decode_step_launches(w, w.L + t + 1) for t in range(n))
    return {"steps": n, "ms_per_step": ms / n, "us_per_token_step": 1e3 * ms / n,
            "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9, "launches": launches,
            "clocks": clk.summary()}


CHUNKED = {"B": 1, "H": 32, "Hkv": 8, "D": 128, "prefix": 6144, "L": 2048, "theta": 5e5}


def bench_chunked_prefill(args, dist, dev):
    """A 2048-token chunk continuing a 6144-token cache (Llama-3-8B attention shape):
    gqa_attn_prefill_cached with q's RoPE fused; the call gathers the kept prefix and
    the chunk, then runs the persistent tensor-core kernel."""
    import torch
    import gqa_causal_attention_gb300 as g

    c = CHUNKED
    B, H, Hkv, D, P, L = c["B"], c["H"], c["Hkv"], c["D"], c["prefix"], c["L"]
    gen = torch.Generator(device=dev).manual_seed(5)
    rp = g.RopeParams.make(theta=c["theta"], max_positions=P + L)
    table = g.rope_table(rp, D, dev)
    kc = torch.randn(B, Hkv, P + L, D, device=dev, generator=gen)
    vc = torch.randn(B, Hkv, P + L, D, device=dev, generator=gen)
    q = torch.randn(B, H, L, D, device=dev, generator=gen)
    k = torch.randn(B, Hkv, L, D, device=dev, generator=gen)
    v = torch.randn(B, Hkv, L, D, device=dev, generator=gen)
    out = torch.empty_like(q)
    st = torch.full((B,), P, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(g.gqa_attn_prefill_cached_workspace_size(B, H, Hkv, L, D, P, 0, rp) // 4 + 4,
                     device=dev)

    def call():
        g.gqa_attn_prefill_cached(q, k, v, kc, vc, out, st, P, rp, table, workspace=ws,
                                  status=status)

    steps = max(3, min(args.steps, 100))
    ms = timed(call, steps, max(3, args.warmup), dist) / steps
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    flops = 4.0 * B * H * D * sum(P + l + 1 for l in range(L))
    return {"config": dict(c), "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "flops": flops,
            "launches": 2}


BLOCK = {"B": 4, "L": 2048, "H": 32, "Hkv": 8, "D": 128, "IT": 14336, "theta": 5e5}


def block_flops(c):
    """Projection FLOP (q, k, v, o, gate, up, down) plus attention FLOP of one block."""
    T, dm, kw = c["B"] * c["L"], c["H"] * c["D"], c["Hkv"] * c["D"]
    proj = 2.0 * T * dm * (dm + 2 * kw + dm + 3 * c["IT"])
    attn = 4.0 * c["B"] * c["H"] * c["D"] * visible_pairs(c["L"], 0)
    return proj, attn


def bench_block(args, dist, dev):
    """The Llama-3-8B-shaped decoder block (gqa_block_forward: norms, the seven
    projections on the tcgen05 GEMM kernel, RoPE, attention, SwiGLU, residuals) on
    4 x 2048 tokens, and the projection kernel alone (attn_linear) at the down
    projection's shape."""
    import torch
    import gqa_causal_attention_gb300 as g

    c = BLOCK
    B, L, H, Hkv, D, IT = c["B"], c["L"], c["H"], c["Hkv"], c["D"], c["IT"]
    dm, kw, T = H * D, Hkv * D, B * L
    gen = torch.Generator(device=dev).manual_seed(11)

    def mat(rows, cols, gain=0.5):
        return torch.randn(rows, cols, device=dev, generator=gen) * (gain / cols ** 0.5)

    w = {"input_layernorm.weight": 1 + 0.1 * torch.randn(dm, device=dev, generator=gen),
         "post_attention_layernorm.weight": 1 + 0.1 * torch.randn(dm, device=dev, generator=gen),
         "q_proj.weight": mat(dm, dm, 1.0), "k_proj.weight": mat(kw, dm, 1.0),
         "v_proj.weight": mat(kw, dm), "o_proj.weight": mat(dm, dm),
         "gate_proj.weight": mat(IT, dm), "up_proj.weight": mat(IT, dm),
         "down_proj.weight": mat(dm, IT)}
    x = torch.randn(B, L, dm, device=dev, generator=gen)
    out = torch.empty_like(x)
    rp = g.RopeParams.make(theta=c["theta"], max_positions=8192,
                           scaling=("llama3", 8.0, 1.0, 4.0, 8192))
    table = g.rope_table(rp, D, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(g.gqa_block_forward_workspace_size(B, L, H, Hkv, D, IT, rp) // 4 + 4,
                     device=dev)

    def block():
        g.gqa_block_forward(x, out, w, H, Hkv, rp, table, workspace=ws, status=status)

    iters = 20
    with ClockSampler(torch.cuda.current_device()) as clk:
        block_ms = kernel_median(block, iters, 3)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    del w, x, out, ws
    torch.cuda.empty_cache()
    # the projection kernel alone at the down projection's shape
    xl = torch.randn(T, IT, device=dev, generator=gen)
    wl = mat(dm, IT)
    yl = torch.empty(T, dm, device=dev)
    lin_ms = kernel_median(lambda: g.attn_linear(xl, wl, yl), KERNEL_ITERS, KERNEL_WARM)
    del xl, wl, yl
    torch.cuda.empty_cache()
    proj, attn = block_flops(c)
    return {"config": dict(c), "ms": block_ms, "proj_flops": proj, "attn_flops": attn,
            "clocks": clk.summary(), "linear_ms": lin_ms,
            "linear_shape": {"T": T, "N": dm, "K": IT},
            "linear_flops": 2.0 * T * dm * IT,
            # kernels per block: 2 RMSNorm, 4 projection launches, k RoPE, V^T, attention
            "launches": 9 * (iters + 3) + KERNEL_ITERS + KERNEL_WARM}


def bench_identical(args, dist, dev):
    """The identical numeric mode's two calls on the Llama-3-8B-shaped prefill and on the
    batched decode (CUDA cores, fixed summation order): what reproducibility costs."""
    import torch
    import gqa_causal_attention_gb300 as g
    from gqa_causal_attention_gb300 import synthetic as syn

    w = syn.WORKLOADS["llama3_8b_prefill"]
    gen = torch.Generator(device=dev).manual_seed(13)
    q = torch.randn(w.B, w.H, w.L, w.D, device=dev, generator=gen)
    k = torch.randn(w.B, w.Hkv, w.L, w.D, device=dev, generator=gen)
    v = torch.randn(w.B, w.Hkv, w.L, w.D, device=dev, generator=gen)
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pre_ms = kernel_median(lambda: g.gqa_attn_prefill_identical(q, k, v, out, status=status),
                           5, 1)
    del q, k, v, out
    wd = syn.WORKLOADS["batched_decode"]
    n = syn.cache_lengths(wd.seed, wd.B, *wd.cache_len_range)
    kc = torch.randn(wd.B, wd.Hkv, wd.capacity, wd.D, device=dev, generator=gen)
    vc = torch.randn(wd.B, wd.Hkv, wd.capacity, wd.D, device=dev, generator=gen)
    qd = torch.randn(wd.B, wd.H, 1, wd.D, device=dev, generator=gen)
    od = torch.empty_like(qd)
    cl = (n + 1).to(dev)
    maxlen = int(n.max()) + 1
    dec_ms = kernel_median(lambda: g.gqa_attn_decode_identical(qd, kc, vc, cl, maxlen, od,
                                                               status=status), 5, 1)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    del kc, vc
    torch.cuda.empty_cache()
    return {"prefill_ms": pre_ms, "prefill_flops": prefill_flops(w),
            "decode_ms": dec_ms, "decode_bytes": 2.0 * wd.Hkv * wd.D * 4 * float((n + 1).sum()),
            "launches": 12}


def cpu_baseline_prefill(w, budget_s=20.0, min_s=10.0):
    """The oracle, as it stands, on the host cores: the whole prefill workload when it fits
    the budget (run again until about min_s seconds have been timed), else a sample of
    whole KV-head groups of batch row 0 at full length."""
    import oracle
    from gqa_causal_attention_gb300 import synthetic as syn

    def cfg(B, H, Hkv):
        return oracle.Cfg(B=B, H=H, Hkv=Hkv, L=w.L, D=w.D, rope_dim=w.R, theta=w.theta,
                          scaling=w.scaling, norm_eps=w.norm_eps, window=w.window,
                          softcap=w.softcap)

    inp = syn.prefill_inputs(w, B=1)
    # calibrate on one KV head and its query group of row 0
    t0 = time.perf_counter()
    oracle.prefill(inp["q"][:, :w.G], inp["k"][:, :1], inp["v"][:, :1], [0], cfg(1, w.G, 1),
                   inp["q_norm_w"], inp["k_norm_w"])
    t1 = time.perf_counter() - t0
    if t1 * w.B * w.Hkv <= budget_s:
        full = syn.prefill_inputs(w)
        runs, dt = 0, 0.0
        while runs == 0 or (dt < min_s and dt * (runs + 1) / runs <= budget_s):
            t0 = time.perf_counter()
            oracle.prefill(full["q"], full["k"], full["v"], [0] * w.B, cfg(w.B, w.H, w.Hkv),
                           full["q_norm_w"], full["k_norm_w"])
            dt += time.perf_counter() - t0
            runs += 1
        fl = prefill_flops(w)
        return {"value": fl * runs / dt / 1e12, "unit": "TFLOP/s",
                "cores": oracle.num_threads(), "kind": "oracle",
                "sample": f"the whole {w.name} prefill (B={w.B}, H={w.H}, L={w.L}), "
                          f"{fl:.3e} FLOP, run {runs} times in {dt:.1f} s"}
    groups = max(1, min(w.Hkv, int(budget_s / max(t1, 1e-3))))
    H2, Hkv2 = groups * w.G, groups
    t0 = time.perf_counter()
    oracle.prefill(inp["q"][:, :H2], inp["k"][:, :Hkv2], inp["v"][:, :Hkv2], [0],
                   cfg(1, H2, Hkv2), inp["q_norm_w"], inp["k_norm_w"])
    dt = time.perf_counter() - t0
    fl = prefill_flops(w, B=1, H=H2)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"batch row 0, heads 0..{H2 - 1} ({Hkv2} KV heads) of the {w.name} "
                      f"prefill, full L={w.L}: {fl:.3e} FLOP in {dt:.2f} s"}


def reference_arm(args, w, rank):
    """The oracle, as it stands, timed on the host cores over a bounded sample per step."""
    if rank != 0:
        return
    import oracle
    from gqa_causal_attention_gb300 import synthetic as syn

    oracle.build()
    per_step = max(0.2, 150.0 / max(1, args.steps + args.warmup))   # whole run within minutes
    inp = syn.prefill_inputs(w, B=1)
    cfg = oracle.Cfg(B=1, H=w.G, Hkv=1, L=w.L, D=w.D, rope_dim=w.R, theta=w.theta,
                     scaling=w.scaling, norm_eps=w.norm_eps, window=w.window,
                     softcap=w.softcap)
    # one KV head with its query group at full length, trimmed until it fits the step budget
    L = w.L
    while True:
        sub = oracle.Cfg(**{**cfg.__dict__, "L": L})
        t0 = time.perf_counter()
        oracle.prefill(inp["q"][:, :w.G, :L], inp["k"][:, :1, :L], inp["v"][:, :1, :L], [0], sub,
                       inp["q_norm_w"], inp["k_norm_w"])
        dt = time.perf_counter() - t0
        if dt <= per_step or L <= 128:
            break
        L = max(128, L // 2)

    def one():
        oracle.prefill(inp["q"][:, :w.G, :L], inp["k"][:, :1, :L], inp["v"][:, :1, :L], [0], sub,
                       inp["q_norm_w"], inp["k_norm_w"])

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = (time.perf_counter() - t0) / args.steps
    fl = 4.0 * w.G * w.D * visible_pairs(L, w.window)
    val = fl / dt / 1e12
    sample = (f"batch row 0, KV head 0 with its {w.G} query heads, first {L} tokens of the "
              f"{w.name} prefill ({fl:.3e} FLOP per step)")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "Hkv": w.Hkv,
                       "D": w.D},
            "cpu_baseline": {"value": val, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    from gqa_causal_attention_gb300 import synthetic as syn
    w = syn.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, w, rank)
        return

    import torch
    import torch.distributed as tdist
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        tdist.init_process_group("nccl", device_id=dev)
        dist = tdist
    import gqa_causal_attention_gb300 as g
    g.load()
    pk = peaks()
    pk["tf32_derived"] = pk["tf32_tflops"]
    pk["tf32_tflops"] = measure_tf32_peak(dev)

    pre = bench_prefill(w, args, dist, dev, rank)
    fl = prefill_flops(w)
    value = world * fl / (pre["ms"] * 1e-3) / 1e12
    kern_tflops = fl / (pre["kernel_ms"] * 1e-3) / 1e12
    q_fused = pre["q_fused"]
    gem = None
    if not args.no_gemma and w.name != "gemma2_window":
        gem = bench_prefill(syn.WORKLOADS["gemma2_window"], args, dist, dev, rank,
                            steps=max(5, min(args.steps, 50)), e2e=False)
    dec = None
    if not args.no_decode:
        wd = syn.WORKLOADS["batched_decode"]
        if args.decode_batch:
            import dataclasses
            wd = dataclasses.replace(wd, B=args.decode_batch)
        dec = bench_decode(wd, args, dist, dev)
    chk = None if args.no_chunked else bench_chunked_prefill(args, dist, dev)
    lng = None
    if not args.no_decode and not args.no_long_decode:
        lng = bench_long_decode(syn.WORKLOADS["long_decode"], args, dist, dev)
    blk = None if args.no_block else bench_block(args, dist, dev)
    idn = None if args.no_identical else bench_identical(args, dist, dev)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": pre["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "tf32" if g.load() and w.D % 4 == 0 else "f32", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "L": w.L, "H": w.H, "Hkv": w.Hkv, "D": w.D,
                   "rope": f"theta {w.theta:g}" + (f", {w.scaling[0]} {tuple(w.scaling[1:])}"
                                                   if w.scaling else ""),
                   "mask": f"window {w.window}" if w.window else "causal",
                   "softcap": w.softcap, "qk_norm": w.qk_norm,
                   "step": ((("kv_cache_append (k RMSNorm/RoPE + cache) + "
                              + ("attn_rope_apply (q) + gqa_attn_prefill (V^T pre-pass inside)"
                                 if args.unfused_q_rope
                                 else "gqa_attn_v_transpose + gqa_attn_prefill_rope_vt"))
                             if args.separate_append or args.unfused_q_rope else
                             "gqa_attn_prefill_step: one pass writes rotated k and v into the "
                             "cache and V^T, then the attention kernel reads k from the cache")
                            + (" (q RMSNorm/RoPE fused into the attention kernel)" if q_fused
                               else " (q RMSNorm/RoPE as a pass over q inside the call)")
                            + ("" if args.no_graph else "; timed as CUDA graph replays")),
                   "ms_per_step_eager": pre["ms_eager"],
                   "l2": f"inputs larger than L2 ({prefill_bytes(w) / 2**20:.0f} MiB per step)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": kern_tflops, "peak": pk["tf32_tflops"],
                     "unit": "TFLOP/s", "frac": kern_tflops / pk["tf32_tflops"],
                     "traffic": NCU_PREFILL_TRAFFIC.get(
                         (w.name, "unfused" if args.unfused_q_rope else "fused")),
                     "traffic_note": "ncu dram bytes of prefill_tq_kernel (one launch)",
                     "kernel": ("gqa_attn_prefill (V^T pre-pass + attention)"
                                if args.unfused_q_rope else
                                "gqa_attn_prefill_rope_vt (the attention kernel alone)"),
                     "kernel_ms": pre["kernel_ms"],
                     "kernel_timing": f"median of {KERNEL_ITERS} calls after {KERNEL_WARM} "
                                      "warm-ups, CUDA events on the launching stream",
                     "peak_note": "dense TF32 measured in this run: cuBLAS fp32 8192^3 "
                                  "with TF32 allowed, best of 10",
                     "frac_of_tf32_nominal_ratio_peak": kern_tflops / pk["tf32_derived"],
                     "frac_of_bf16_peak": kern_tflops / pk["bf16_tflops"]},
        "gpu_launches": pre["launches"],
        "clocks": pre["clocks"],
    }
    if "e2e_ms" in pre:
        line["e2e"] = {"value": world * fl / (pre["e2e_ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": pre["h2d"], "d2h_bytes_per_step": pre["d2h"],
                       "ms_per_step": pre["e2e_ms"],
                       "call": "gqa_attn_prefill_from_host (pinned host q, k, v in, out back; "
                               f"{pre['e2e_chunks']} chunks overlap copies and kernels)",
                       "serial_ms_per_step": pre["e2e_serial_ms"]}

    if dec is not None:
        gbs = dec["bytes"] / (dec["ms"] * 1e-3) / 1e9
        kgbs = dec["bytes"] / (dec["kernel_ms"] * 1e-3) / 1e9
        line["decode"] = {
            "workload": "batched_decode", "value": world * gbs, "unit": "GB/s",
            "ms_per_step": dec["ms"], "ms_per_step_eager": dec["ms_eager"],
            "bytes_per_step": dec["bytes"],
            "frac_of_8tbs": gbs / NOMINAL_HBM_GBS,
            "step": "gqa_attn_decode_step: q, k RMSNorm/RoPE at n_b + append (one pass), then "
                    "the split-KV decode and its combine; CUDA graph replays",
            "roofline": {"bound": "hbm", "achieved": kgbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": kgbs / pk["hbm_gbs"],
                         "traffic": (NCU_DECODE_TRAFFIC_PER_ALG_BYTE * dec["bytes"]
                                     if NCU_DECODE_TRAFFIC_PER_ALG_BYTE else None),
                         "kernel": "gqa_attn_decode", "kernel_ms": dec["kernel_ms"]},
            "gpu_launches": dec["launches"],
            "clocks": dec["clocks"]}
        line["gpu_launches"] += line["decode"]["gpu_launches"]
    if chk is not None:
        line["chunked_prefill"] = {
            "workload": "chunked_prefill", "config": chk["config"], "value": world * chk["tflops"],
            "unit": "TFLOP/s", "ms_per_step": chk["ms"], "flops_per_step": chk["flops"],
            "frac_of_tf32_peak": chk["tflops"] / pk["tf32_tflops"],
            "step": "gqa_attn_prefill_cached (gather of the cached prefix + chunk, then the "
                    "persistent kernel with q RoPE fused)",
            "gpu_launches": chk["launches"] * max(3, min(args.steps, 100))}
        line["gpu_launches"] += line["chunked_prefill"]["gpu_launches"]
    if lng is not None:
        wl = syn.WORKLOADS["long_decode"]
        line["long_decode"] = {
            "workload": "long_decode", "config": {"B": wl.B, "H": wl.H, "Hkv": wl.Hkv,
                                                   "D": wl.D, "rope_dim": wl.rope_dim,
                                                   "prefill": wl.L, "steps": wl.decode_steps},
            "value": world * lng["gbs"], "unit": "GB/s",
            "us_per_step": lng["us_per_token_step"], "bytes_total": lng["bytes"],
            "step": "gqa_attn_decode_step (q, k RoPE and the append folded into the split-KV "
                    "kernel; one cluster per (row, KV head) merges its splits in distributed "
                    "shared memory, or a combine pass when the groups do not fit at once), "
                    "1024 steps in one CUDA graph",
            "note": "the cache (134 MB) is about L2-sized; part of each step's reads hit L2",
            "gpu_launches": lng["launches"], "clocks": lng["clocks"]}
        line["gpu_launches"] += lng["launches"]
    if gem is not None:
        wg = syn.WORKLOADS["gemma2_window"]
        gfl = prefill_flops(wg)
        gk = gfl / (gem["kernel_ms"] * 1e-3) / 1e12
        line["gemma2_window"] = {
            "workload": "gemma2_window",
            "config": {"B": wg.B, "L": wg.L, "H": wg.H, "Hkv": wg.Hkv, "D": wg.D,
                       "window": wg.window, "softcap": wg.softcap, "qk_norm": wg.qk_norm,
                       "rope": f"theta {wg.theta:g}", "cache": f"ring of {wg.window}"},
            "value": world * gfl / (gem["ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": gem["ms"], "ms_per_step_eager": gem["ms_eager"],
            "flops_per_step": gfl,
            "step": "gqa_attn_prefill_step: one pass writes rotated k (ring + a rotated copy), "
                    "v and V^T; q RMSNorm/RoPE as a pass; then the attention kernel; "
                    "CUDA graph replays",
            "roofline": {"bound": "tensor", "achieved": gk, "peak": pk["tf32_tflops"],
                         "unit": "TFLOP/s", "frac": gk / pk["tf32_tflops"],
                         "traffic": NCU_PREFILL_TRAFFIC.get(("gemma2_window", "fused")),
                         "kernel": "the attention kernel alone (q rotated beforehand; "
                                   "gqa_attn_prefill_rope_vt without RoPE)",
                         "kernel_ms": gem["kernel_ms"],
                         "frac_of_bf16_peak": gk / pk["bf16_tflops"]},
            "gpu_launches": gem["launches"], "clocks": gem["clocks"]}
        line["gpu_launches"] += gem["launches"]
    if blk is not None:
        btot = blk["proj_flops"] + blk["attn_flops"]
        lt = blk["linear_flops"] / (blk["linear_ms"] * 1e-3) / 1e12
        line["block"] = {
            "workload": "llama3_8b_block", "config": blk["config"],
            "value": world * btot / (blk["ms"] * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": blk["ms"], "flops_per_step": btot,
            "proj_flops": blk["proj_flops"], "attn_flops": blk["attn_flops"],
            "step": "gqa_block_forward: RMSNorm, q/k/v projections (one launch, head-major "
                    "out), k RoPE, V^T + attention (q RoPE fused), o_proj + residual, "
                    "RMSNorm, gate/up with SwiGLU epilogue, down_proj + residual; "
                    "median of 20 calls",
            "roofline": {"bound": "tensor", "achieved": lt, "peak": pk["tf32_tflops"],
                         "unit": "TFLOP/s", "frac": lt / pk["tf32_tflops"],
                         "traffic": NCU_GEMM_TRAFFIC,
                         "traffic_note": "ncu dram bytes of gemm_tc2_kernel (one launch)",
                         "kernel": "attn_linear (gemm_tc2_kernel) at the down projection's "
                                   f"shape T={blk['linear_shape']['T']} "
                                   f"N={blk['linear_shape']['N']} K={blk['linear_shape']['K']}",
                         "kernel_ms": blk["linear_ms"]},
            "gpu_launches": blk["launches"], "clocks": blk["clocks"]}
        line["gpu_launches"] += blk["launches"]
    if idn is not None:
        line["identical"] = {
            "prefill": {"workload": "llama3_8b_prefill",
                        "value": world * idn["prefill_flops"] / (idn["prefill_ms"] * 1e-3) / 1e12,
                        "unit": "TFLOP/s", "ms": idn["prefill_ms"],
                        "call": "gqa_attn_prefill_identical (median of 5)"},
            "decode": {"workload": "batched_decode",
                       "value": world * idn["decode_bytes"] / (idn["decode_ms"] * 1e-3) / 1e9,
                       "unit": "GB/s", "ms": idn["decode_ms"],
                       "call": "gqa_attn_decode_identical (median of 5)"},
            "gpu_launches": idn["launches"]}
        line["gpu_launches"] += idn["launches"]
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_prefill(w)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
