"""Benchmark of the KDA core on GB300: prefill and decode tokens/s against the rooflines.

One JSON line on rank 0.  The headline `value` is chunked-prefill throughput on the
Kimi-K3-shaped prefill workload (B=1, T=8192, H=96, d=128, chunk 64, zero initial
state) with inputs resident in HBM; `decode` reports the one-token decode step
(B=256, H=96, d=128, fp32 state 1.6 GB updated in place, sigmoid-gated RMSNorm
fused).  `e2e` repeats the prefill through the public API with pinned host
inputs, the host->device copies and the read-back of o and the final state inside
the timed region.  `cpu_baseline` times the fp64 oracle on a bounded sample of the
same workload on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs its own replica (the (sequence, head) units
are independent, there is no exchange step); value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s & decode tokens/s (H=96,d=128) vs tensor/HBM roofline"
PREFILL_BYTES_PER_TH = 3 * 256 + 512 + 4 + 512   # q,k,v bf16 + g fp32 + beta + o fp32 = 1796
PREFILL_FLOP_PER_TH = 10 * 64 * 128 + 6 * 128 * 128 + (2 * 64 * 64) // 3  # 182,955 at C=64, d=128
STATE_BYTES = 128 * 128 * 4
DECODE_BYTES_PER_UNIT = 2 * STATE_BYTES + 3 * 256 + 512 + 4 + 256 + 512  # + gate bf16, y fp32
# the decode step with the q, k, v short convolutions fused: + three histories of W-1 = 3
# rows of 128 fp32 channels read and written per unit; the filters (3 x 128 x W fp32 per
# head) are counted once per call
DECODE_CONV_BYTES_PER_UNIT = DECODE_BYTES_PER_UNIT + 2 * 3 * 3 * 128 * 4
PREFILL_LOGITS_BYTES_PER_TH = 3 * 256 + 256 + 2 + 512  # q,k,v bf16 + g logits bf16 + beta logit bf16 + o fp32
PREFILL_NORM_BYTES_PER_TH = 3 * 256 + 512 + 4 + 256 + 256  # q,k,v bf16 + g fp32 + beta + gate bf16 + y bf16
PREFILL_LONG_BYTES_PER_TH = 3 * 256 + 512 + 4 + 256 + 512  # q,k,v bf16 + g fp32 + beta + gate bf16 + y fp32

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per unit of work from one
# ncu capture summarised under profiles/, valid only for the kernel source it was
# taken on: `traffic` is reported as null as soon as that source file changes.
MEASURED_TRAFFIC = {
    # B=1 T=2048 H=96 capture, mean of two launches: (328.410112 MB - 6.29 MB of final state)
    # / (2048 * 96) token-heads
    "prefill_fused": {"source": "kimi_delta_attention_gated_gb300/csrc/kda_chunk_tc.cu",
                      "sha256": "78a254e0b521b659e9c1ca535b80449b1df1bcbe1f85ecc50bf4286205bef4eb",
                      "bytes_per_unit": (328.410112e6 - 6.291456e6) / (2048 * 96),
                      "capture": "ncu, B=1 T=2048 H=96, g and beta given"},
    # the same kernel with gates from bf16 logits, B=1 T=2048 H=96 capture, mean of two
    # launches: (274.22208 MB - 6.29 MB of final state) / (2048 * 96) token-heads
    "prefill_logits": {"source": "kimi_delta_attention_gated_gb300/csrc/kda_chunk_tc.cu",
                       "sha256": "78a254e0b521b659e9c1ca535b80449b1df1bcbe1f85ecc50bf4286205bef4eb",
                       "bytes_per_unit": (274.22208e6 - 6.291456e6) / (2048 * 96),
                       "capture": "ncu, B=1 T=2048 H=96, bf16 logits"},
    # the same kernel with the fused gated norm (bf16 gate in, bf16 y out), B=1 T=2048 H=96
    # capture, mean of two launches: (342.155648 MB - 6.29 MB of final state) / (2048 * 96)
    "prefill_norm": {"source": "kimi_delta_attention_gated_gb300/csrc/kda_chunk_tc.cu",
                     "sha256": "78a254e0b521b659e9c1ca535b80449b1df1bcbe1f85ecc50bf4286205bef4eb",
                     "bytes_per_unit": (342.155648e6 - 6.291456e6) / (2048 * 96),
                     "capture": "ncu, B=1 T=2048 H=96, fused gated norm"},
    # B=64 capture: mean of two launches, 754.667264 MB / (64 * 96) (sequence, head) units
    # (part of the state written back stays in L2 at the kernel's end: below the algorithmic bytes)
    "decode": {"source": "kimi_delta_attention_gated_gb300/csrc/kda_recurrent.cu",
               "sha256": "5b652beb9f24e8ee12b996eb18914cbb7bf46a2a94542e35fbb00fcbfeea303b",
               "bytes_per_unit": 754.667264e6 / (64 * 96),
               "capture": "ncu, decode B=64 H=96"},
    # the decode step with the short convolutions fused, B=64 capture: mean of two launches,
    # 814.222592 MB / (64 * 96) units
    "decode_conv": {"source": "kimi_delta_attention_gated_gb300/csrc/kda_recurrent.cu",
                    "sha256": "5b652beb9f24e8ee12b996eb18914cbb7bf46a2a94542e35fbb00fcbfeea303b",
                    "bytes_per_unit": 814.222592e6 / (64 * 96),
                    "capture": "ncu, decode B=64 H=96, short convolutions fused"},
    # full-size captures: mean of two launches per (token, channel) element
    "conv_prefill": {"source": "kimi_delta_attention_gated_gb300/csrc/kda_short_conv.cu",
                     "sha256": "5455c4ca65aa3564cc58dfe31e882936cc835e7c78b214ec91bc918376e0107f",
                     "bytes_per_unit": 1180.691584e6 / (8192 * 36864),
                     "capture": "ncu, full size"},
    "conv_decode": {"source": "kimi_delta_attention_gated_gb300/csrc/kda_short_conv.cu",
                    "sha256": "5455c4ca65aa3564cc58dfe31e882936cc835e7c78b214ec91bc918376e0107f",
                    "bytes_per_unit": 204.401152e6 / (256 * 36864),
                    "capture": "ncu, full size"},
}


def sources_sha256(sources):
    """SHA-256 over the named source files, concatenated in order."""
    import hashlib
    h = hashlib.sha256()
    for src in sources:
        with open(os.path.join(ROOT, src), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kind: str, units: float, fixed: float = 0.0):
    """Traffic of one launch (or one call's launches) scaled from the capture, or None if
    a kernel source changed since the counters were taken."""
    m = MEASURED_TRAFFIC.get(kind)
    if m is None:
        return None
    srcs = m["sources"] if "sources" in m else [m["source"]]
    try:
        if sources_sha256(srcs) != m["sha256"]:
            return None
    except OSError:
        return None
    return m["bytes_per_unit"] * units + fixed


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        os.remove(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_steps(fn, steps, warmup, world, clocks_index=None):
    """Warm up, then time `steps` calls with CUDA events on the current stream; an event
    pair around every call gives the per-call device time of what it launched."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(clocks_index) if clocks_index is not None else None
    if sampler:
        sampler.__enter__()
    torch.cuda.synchronize()
    n0 = kda.launch_count()
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    launches = kda.launch_count() - n0
    if sampler:
        sampler.__exit__(None, None, None)
    barrier(world)
    total_ms = start.elapsed_time(end)
    per_call = [a.elapsed_time(b) for a, b in ev]
    return {"ms_per_step": max_over_ranks(total_ms / steps, world), "call_ms": statistics.mean(per_call),
            "launches": launches, "clocks": sampler.summary() if sampler else None}


def prefill_inputs(device, T=None):
    from kimi_delta_attention_gated_gb300.inputs import make_inputs
    return make_inputs("prefill", device=device, T=T)


def bench_prefill(args, world, rank, peaks, form="fused"):
    """The prefill workload through one tensor-core form: "fused" (one kernel per (sequence,
    head), no workspace), "concurrent" (the fused kernel with the pre-pass beside it on the
    idle SMs, a workspace given) or "split" (the pre-pass over all chunks and heads, then
    the per-head chain kernel).  `kernel_ms` is the device time of the whole call, every
    kernel of it together (CUDA events around the call on the caller's stream, which the
    concurrent form's second stream joins)."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    d = prefill_inputs("cuda", args.prefill_T)
    B, T, H, K, V = d["B"], d["T"], d["H"], d["K"], d["V"]
    o = torch.empty((B, T, H, V), device="cuda", dtype=torch.float32)
    fs = torch.empty((B, H, K, V), device="cuda", dtype=torch.float32)
    ws = None if form == "fused" else torch.empty(kda.workspace_size(B, T, H), dtype=torch.uint8, device="cuda")
    mode = "split" if form == "split" else args.mode
    fn = lambda: kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, scale=d["scale"], chunk=64,
                               o=o, final_state=fs, mode=mode, workspace=ws)
    if form == "concurrent":
        kda.prepass_hits()
    r = time_steps(fn, args.steps, args.warmup, world,
                   clocks_index=torch.cuda.current_device() if form == args.headline else None)
    hits = kda.prepass_hits() if form == "concurrent" else None
    th = B * T * H
    kernel_ms = r["call_ms"]
    algo_bytes = th * PREFILL_BYTES_PER_TH + B * H * STATE_BYTES
    algo_flop = th * PREFILL_FLOP_PER_TH
    achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
    tflops = algo_flop / (kernel_ms * 1e-3) / 1e12
    kernels = {"fused": "chunk_tc_kernel", "concurrent": "chunk_tc_kernel + chunk_prep_kernel beside it, one call",
               "split": "chunk_prep_kernel + chunk_chain_kernel, one call"}[form]
    out = {
        "value": world * B * T / (r["ms_per_step"] * 1e-3),
        "ms_per_step": r["ms_per_step"],
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"],
                     "traffic": measured_traffic("prefill_fused", th, B * H * STATE_BYTES) if form == "fused" else None,
                     "algorithmic_bytes_per_launch": algo_bytes, "kernel_ms": kernel_ms, "kernels": kernels,
                     "launches_per_call": max(1, r["launches"] // args.steps), "peak_source": peaks["source"]},
        "roofline_tensor": {"achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                            "frac": tflops / peaks["bf16_tflops"], "algorithmic_flop_per_launch": algo_flop},
        "config": {"workload": f"prefill B={B} T={T} H={H} d={K} chunk=64 zero initial state",
                   "B": B, "T": T, "H": H, "d": K, "chunk": 64, "mode": args.mode, "form": form,
                   "l2_flush": "inputs larger than L2 (1.42 GB read+written per step vs 129 MB L2)",
                   "parallelism": f"replicas x{world}"},
    }
    if hits is not None:
        n_chunks = B * H * ((T + 63) // 64) * (args.warmup + args.steps)
        out["prepass_share"] = hits / n_chunks  # chunks whose grams and UT transform came from the pre-pass
    return out, d


def bench_prefill_workload(args, world, peaks, name):
    """A full-size prefill workload timed in the launch configuration its parity test uses:
    "varlen" = 8 packed sequences, lengths log-uniform in [512, 16384], each with an fp32
    initial state N(0, 0.02^2) and its own final state, fp32 o; "long" = B=2, T=65536 with
    the fused sigmoid-gated RMSNorm (bf16 gate in, fp32 y out, o not written) and the
    final states."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    from kimi_delta_attention_gated_gb300.inputs import make_inputs
    d = make_inputs(name, device="cuda")
    B, T, H, K, V, N = d["B"], d["T"], d["H"], d["K"], d["V"], d["N"]
    fs = torch.empty((N, H, K, V), device="cuda", dtype=torch.float32)
    th = B * T * H
    if name == "varlen":
        o = torch.empty((B, T, H, V), device="cuda", dtype=torch.float32)
        cu = d["cu_seqlens"]
        fn = lambda: kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["initial_state"], scale=d["scale"],
                                   chunk=64, cu_seqlens=cu, o=o, final_state=fs, mode=args.mode)
        per_th, state_bytes = PREFILL_BYTES_PER_TH, 2 * N * H * STATE_BYTES
        lens = (cu[1:] - cu[:-1]).tolist()
        workload = f"varlen prefill, {N} packed sequences of {lens} tokens ({T} total), H={H} d={K}, fp32 initial " \
                   "and final states, fp32 o"
        traffic = measured_traffic("prefill_fused", th, state_bytes)
    else:
        y = torch.empty((B, T, H * V), device="cuda", dtype=torch.float32)
        fn = lambda: kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, scale=d["scale"], chunk=64,
                                   gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"], return_o=False, y=y,
                                   final_state=fs, mode=args.mode)
        per_th, state_bytes = PREFILL_LONG_BYTES_PER_TH, N * H * STATE_BYTES
        workload = f"long prefill B={B} T={T} H={H} d={K} + fused sigmoid-gated RMSNorm (bf16 gate, fp32 y, o not " \
                   "written), final states"
        traffic = None
    steps = max(3, args.steps // (4 if name == "long" else 1))
    r = time_steps(fn, steps, args.warmup, world)
    kernel_ms = r["call_ms"]  # the call's device time (both kernels of the split form)
    algo_bytes = th * per_th + state_bytes
    achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
    tflops = th * PREFILL_FLOP_PER_TH / (kernel_ms * 1e-3) / 1e12
    return {"metric": "KDA prefill tokens/s", "value": world * B * T / (r["ms_per_step"] * 1e-3), "unit": "tokens/s",
            "ms_per_step": r["ms_per_step"], "steps": steps, "gpu_launches": r["launches"],
            "config": {"workload": workload, "l2_flush": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                         "algorithmic_bytes_per_launch": algo_bytes, "kernel_ms": kernel_ms,
                         "peak_source": peaks["source"]},
            "roofline_tensor": {"achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                "frac": tflops / peaks["bf16_tflops"]}}


def bench_decode(args, world, peaks):
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    from kimi_delta_attention_gated_gb300.inputs import make_inputs
    d = make_inputs("decode", device="cuda", B=args.decode_B)
    sq = lambda t: t.squeeze(1).contiguous()
    q, k, v, g, beta, gate = (sq(d[n]) for n in ("q", "k", "v", "g", "beta", "gate"))
    state = d["initial_state"]
    B, H, K, V = state.shape
    y = torch.empty((B, H * V), device="cuda", dtype=torch.float32)
    fn = lambda: kda.recurrent_step(q, k, v, g, beta, state, state_out=state, gate=gate, norm_w=d["norm_w"],
                                    eps=d["eps"], y=y, return_o=False)
    r = time_steps(fn, max(args.steps, 20), args.warmup, world)
    kernel_ms = r["call_ms"] / max(1, r["launches"] // max(args.steps, 20))
    algo_bytes = B * H * DECODE_BYTES_PER_UNIT
    achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
    return {"metric": "KDA decode tokens/s", "value": world * B / (r["ms_per_step"] * 1e-3), "unit": "tokens/s",
            "ms_per_step": r["ms_per_step"], "gpu_launches": r["launches"],
            "config": {"workload": f"decode B={B} H={H} d={K} fp32 state in place + fused sigmoid-gated RMSNorm",
                       "l2_flush": "state 1.61 GB > L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic("decode", B * H),
                         "algorithmic_bytes_per_launch": algo_bytes, "kernel_ms": kernel_ms,
                         "peak_source": peaks["source"]}}


def bench_decode_conv(args, world, peaks):
    """The decode step with the q, k, v short convolutions (+ SiLU) fused ahead of it
    (kda_recurrent_step_conv): raw bf16 projections in, state and the three histories
    updated in place, the gated norm fused, y fp32 out."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    from kimi_delta_attention_gated_gb300.inputs import make_decode_conv_inputs
    B = args.decode_B or 256
    d = make_decode_conv_inputs(B=B, H=96, W=4, device="cuda")
    state = d["initial_state"]
    _, H, K, V = state.shape
    y = torch.empty((B, H * V), device="cuda", dtype=torch.float32)
    conv = (d["conv_weight"], d["conv_state"], d["conv_state"])
    fn = lambda: kda.recurrent_step(d["q"], d["k"], d["v"], d["g"], d["beta"], state, state_out=state,
                                    gate=d["gate"], norm_w=d["norm_w"], eps=d["eps"], y=y, return_o=False,
                                    conv=conv)
    r = time_steps(fn, max(args.steps, 20), args.warmup, world)
    kernel_ms = r["call_ms"] / max(1, r["launches"] // max(args.steps, 20))
    algo_bytes = B * H * DECODE_CONV_BYTES_PER_UNIT + H * 3 * 128 * d["W"] * 4
    achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
    return {"metric": "KDA decode tokens/s, short convolutions fused", "value": world * B / (r["ms_per_step"] * 1e-3),
            "unit": "tokens/s", "ms_per_step": r["ms_per_step"], "gpu_launches": r["launches"],
            "config": {"workload": f"decode B={B} H={H} d={K} W=4: raw q/k/v projections through the fused short "
                                   "convolutions, fp32 state and histories in place, fused sigmoid-gated RMSNorm",
                       "l2_flush": "state 1.61 GB > L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"], "traffic": measured_traffic("decode_conv", B * H),
                         "algorithmic_bytes_per_launch": algo_bytes, "kernel_ms": kernel_ms,
                         "peak_source": peaks["source"]}}


def bench_prefill_logits(args, world, peaks):
    """The same prefill with g and beta computed in the kernel from bf16 logits
    (kda_chunk_fwd_logits), sharing the prefill's shapes and q, k, v."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    from kimi_delta_attention_gated_gb300.inputs import make_logit_inputs
    d = make_logit_inputs("prefill", device="cuda", T=args.prefill_T)
    B, T, H, K, V = d["B"], d["T"], d["H"], d["K"], d["V"]
    o = torch.empty((B, T, H, V), device="cuda", dtype=torch.float32)
    fs = torch.empty((B, H, K, V), device="cuda", dtype=torch.float32)
    fn = lambda: kda.chunk_fwd_logits(d["q"], d["k"], d["v"], d["g_logits"], d["beta_logits"], d["A_log"], None,
                                      dt_bias=d["dt_bias"], g_lower_bound=d["g_lower_bound"], scale=d["scale"],
                                      mode=args.mode, o=o, final_state=fs)
    r = time_steps(fn, args.steps, args.warmup, world)
    kernel_ms = r["call_ms"]  # the call's device time (both kernels of the split form)
    th = B * T * H
    algo_bytes = th * PREFILL_LOGITS_BYTES_PER_TH + B * H * STATE_BYTES
    achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
    return {"metric": "KDA prefill tokens/s, gates from logits", "value": world * B * T / (r["ms_per_step"] * 1e-3),
            "unit": "tokens/s", "ms_per_step": r["ms_per_step"], "gpu_launches": r["launches"],
            "config": {"workload": f"prefill B={B} T={T} H={H} d={K}, bf16 g/beta logits + A_log + dt_bias, "
                                   "lower bound -5", "l2_flush": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": measured_traffic("prefill_logits", th, B * H * STATE_BYTES),
                         "algorithmic_bytes_per_launch": algo_bytes, "kernel_ms": kernel_ms,
                         "peak_source": peaks["source"]}}


def bench_prefill_norm(args, world, peaks):
    """The same prefill with the fused sigmoid-gated RMSNorm: bf16 gate in, y = the layer's
    normed output in bf16 out (o itself is not written), sharing the prefill's q, k, v, g,
    beta; gate ~ N(0, 1), norm weight 1 + N(0, 0.1^2), eps 1e-5."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    from kimi_delta_attention_gated_gb300.inputs import make_inputs
    d = make_inputs("prefill", device="cuda", T=args.prefill_T)
    B, T, H, K, V = d["B"], d["T"], d["H"], d["K"], d["V"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(20_000)
    gate = torch.randn((B, T, H, V), generator=gen, device="cuda").to(torch.bfloat16)
    norm_w = 1 + 0.1 * torch.randn(V, generator=gen, device="cuda")
    y = torch.empty((B, T, H * V), device="cuda", dtype=torch.bfloat16)
    fs = torch.empty((B, H, K, V), device="cuda", dtype=torch.float32)
    fn = lambda: kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, scale=d["scale"], mode=args.mode,
                               gate=gate, norm_w=norm_w, eps=1e-5, out_dtype=torch.bfloat16, return_o=False, y=y,
                               final_state=fs)
    r = time_steps(fn, args.steps, args.warmup, world)
    kernel_ms = r["call_ms"]  # the call's device time (both kernels of the split form)
    th = B * T * H
    algo_bytes = th * PREFILL_NORM_BYTES_PER_TH + B * H * STATE_BYTES
    achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
    return {"metric": "KDA prefill tokens/s, fused gated RMSNorm output", "value": world * B * T / (r["ms_per_step"] * 1e-3),
            "unit": "tokens/s", "ms_per_step": r["ms_per_step"], "gpu_launches": r["launches"],
            "config": {"workload": f"prefill B={B} T={T} H={H} d={K}, bf16 gate in, bf16 y out (sigmoid-gated "
                                   "RMSNorm), o not written", "l2_flush": "inputs larger than L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": measured_traffic("prefill_norm", th, B * H * STATE_BYTES),
                         "algorithmic_bytes_per_launch": algo_bytes, "kernel_ms": kernel_ms,
                         "peak_source": peaks["source"]}}


def bench_short_conv(args, world, peaks):
    """The q/k/v short convolution (causal depthwise, 4 taps, SiLU): one 8192-token prompt
    (state out) and one decode step of 256 sequences (state updated in place), each over
    the 3 x 12288 channels of q, k and v side by side."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    from kimi_delta_attention_gated_gb300.inputs import make_conv_inputs
    out = {}
    for name in ("conv_prefill", "conv_decode"):
        d = make_conv_inputs(name, device="cuda")
        B, T, D, W, N = d["B"], d["T"], d["D"], d["W"], d["N"]
        y = torch.empty_like(d["x"])
        st = d["conv_state"]
        sf = st if st is not None else torch.empty((N, W - 1, D), device="cuda")
        fn = lambda: kda.short_conv(d["x"], d["weight"], None, st, y=y, final_state=sf)
        steps = max(args.steps, 20)
        r = time_steps(fn, steps, args.warmup, world)
        kernel_ms = r["call_ms"] / max(1, r["launches"] // steps)
        state_bytes = N * (W - 1) * D * 4 * (2 if st is not None else 1)
        algo_bytes = B * T * D * (2 + 2) + state_bytes + D * W * 4
        achieved = algo_bytes / (kernel_ms * 1e-3) / 1e9
        out[name] = {
            "metric": "short-conv tokens/s", "value": world * B * T / (r["ms_per_step"] * 1e-3), "unit": "tokens/s",
            "ms_per_step": r["ms_per_step"], "gpu_launches": r["launches"],
            "config": {"workload": f"{name} B={B} T={T} D={D} (q, k, v) W={W} SiLU bf16 in/out",
                       "l2_flush": "inputs + outputs larger than L2"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / peaks["hbm_gbs"],
                         "traffic": measured_traffic(name, B * T * D),
                         "algorithmic_bytes_per_launch": algo_bytes, "kernel_ms": kernel_ms,
                         "peak_source": peaks["source"]}}
    return out


def bench_o_proj(args, world, peaks):
    """The output projection (12288 -> 7168, bf16 in/out, fp32 accumulation) for the decode
    batch (weight-bandwidth bound) and the 8192-token prompt (tensor bound)."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    out = {}
    K, N = 96 * 128, 7168
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    w = (torch.randn((N, K), generator=g, device="cuda") * K ** -0.5).to(torch.bfloat16)
    legs = (("decode", 256), ("prefill", 8192)) if not args.oproj_rows else \
        (("decode" if args.oproj_rows <= 256 else "prefill", args.oproj_rows),)
    for name, rows in legs:
        y = torch.randn((rows, K), generator=g, device="cuda").to(torch.bfloat16)
        o = torch.empty((rows, N), device="cuda", dtype=torch.bfloat16)
        fn = lambda: kda.o_proj(y, w, out=o)
        steps = max(args.steps, 20)
        r = time_steps(fn, steps, args.warmup, world)
        kernel_ms = r["call_ms"] / max(1, r["launches"] // steps)
        flop = 2.0 * rows * N * K
        byts = (N * K + rows * K + rows * N) * 2
        if name == "decode":
            ach = byts / (kernel_ms * 1e-3) / 1e9
            roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": ach / peaks["hbm_gbs"], "traffic": None, "algorithmic_bytes_per_launch": byts}
        else:
            ach = flop / (kernel_ms * 1e-3) / 1e12
            roof = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                    "frac": ach / peaks["bf16_tflops"], "traffic": None, "algorithmic_flop_per_launch": flop}
        roof.update(kernel_ms=kernel_ms, peak_source=peaks["source"])
        # context only: the same product through torch (cuBLAS) on the same device and inputs
        lib_fn = lambda: torch.matmul(y, w.t(), out=o)
        lib_ms = time_steps(lib_fn, steps, args.warmup, world)["call_ms"]
        out[name] = {"metric": "o_proj tokens/s", "value": world * rows / (r["ms_per_step"] * 1e-3), "unit": "tokens/s",
                     "ms_per_step": r["ms_per_step"], "gpu_launches": r["launches"],
                     "config": {"workload": f"o_proj rows={rows} 12288->7168 bf16 (tcgen05 GEMM)"}, "roofline": roof,
                     "torch_cublas_ms_same_inputs": lib_ms}
    return out


def bench_e2e(args, world, d):
    """Same prefill through the public call with pinned host inputs and host outputs."""
    import torch
    import kimi_delta_attention_gated_gb300 as kda
    host = {n: d[n].cpu().pin_memory() for n in ("q", "k", "v", "g", "beta")}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    B, T, H, V = d["B"], d["T"], d["H"], d["V"]
    o_h = torch.empty((B, T, H, V), dtype=torch.float32).pin_memory()
    s_h = torch.empty((B, H, d["K"], V), dtype=torch.float32).pin_memory()
    d2h = o_h.numel() * 4 + s_h.numel() * 4
    fn = lambda: kda.chunk_fwd(host["q"], host["k"], host["v"], host["g"], host["beta"], None, scale=d["scale"],
                               chunk=64, mode=args.mode, o=o_h, final_state=s_h)
    steps = max(2, min(args.steps, 5))
    for _ in range(max(1, min(args.warmup, 2))):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        o, s = fn()  # returns host tensors: the read-back is synchronous
    torch.cuda.synchronize()
    dt = max_over_ranks((time.perf_counter() - t0) / steps, world)
    return {"value": world * B * T / dt, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": dt * 1e3, "steps": steps,
            "path": f"chunk_fwd on pinned host tensors -> the C entry kda_chunk_fwd_host: {kda.HOST_SEGMENT}-token "
                    "segments, 2-D copies in / fused kernel / copies out on three streams"}


def cpu_baseline(d, heads: int):
    """The fp64 oracle, as it stands, on the first `heads` heads of the prefill workload."""
    import numpy as np
    import oracle
    f = lambda t: np.ascontiguousarray(t[:, :, :heads].float().cpu().numpy())
    q, k, v, g, beta = (f(d[n]) for n in ("q", "k", "v", "g", "beta"))
    threads = oracle.default_threads()
    oracle.build()
    t0 = time.perf_counter()
    oracle.recurrent(q, k, v, g, beta, scale=d["scale"], n_threads=threads)
    dt = time.perf_counter() - t0
    frac = heads / d["H"]
    return {"value": d["B"] * d["T"] * frac / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"{heads} of {d['H']} heads x {d['T']} tokens (all chunks) of the prefill workload; "
                      f"tokens/s scaled by {heads}/{d['H']}; {dt:.2f} s wall"}


def cpu_baseline_decode_one_core(units: int = 2048):
    """The fp64 oracle on one host core for the decode step (B=256, H=96): a sample of
    `units` (sequence, head) units, tokens/s scaled to the whole batch."""
    import numpy as np
    import torch
    import oracle
    from kimi_delta_attention_gated_gb300.inputs import make_inputs
    d = make_inputs("decode", device="cpu")
    B, H = d["B"], d["H"]
    f = lambda t: np.ascontiguousarray(t.float().numpy())
    n = min(units, B * H)
    flat = lambda t: t.reshape((B * H, 1, 1) + tuple(t.shape[3:]))[:n]  # each unit its own sequence
    q, k, v, g = (f(flat(d[x])) for x in ("q", "k", "v", "g"))
    beta = f(d["beta"].reshape(B * H, 1, 1)[:n])
    s0 = f(d["initial_state"].reshape((B * H, 1) + tuple(d["initial_state"].shape[2:]))[:n])
    oracle.build()
    t0 = time.perf_counter()
    oracle.recurrent(q, k, v, g, beta, s0, scale=d["scale"], n_threads=1)
    dt = time.perf_counter() - t0
    return {"value": B * (n / (B * H)) / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{n} of {B * H} (sequence, head) units of the decode step B={B} H={H}; tokens/s scaled "
                      f"by {n}/{B * H}; {dt:.2f} s wall (the gated norm epilogue not included)"}


def run_reference(args, world, rank):
    """The reference arm: the fp64 oracle on the host cores, a bounded sample per step."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from kimi_delta_attention_gated_gb300.inputs import make_inputs
    oracle.build()
    heads = args.ref_heads
    d = make_inputs("prefill", device="cpu", H=heads)
    f = lambda t: np.ascontiguousarray(t.float().numpy())
    q, k, v, g, beta = (f(d[n]) for n in ("q", "k", "v", "g", "beta"))
    threads = oracle.default_threads()
    run = lambda: oracle.recurrent(q, k, v, g, beta, scale=d["scale"], n_threads=threads)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = d["B"] * d["T"] * heads / 96 / dt
    sample = f"{heads} of 96 heads x 8192 tokens of the prefill workload per step; tokens/s scaled by {heads}/96"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill B=1 T=8192 H=96 d=128 chunk=64 zero initial state",
                   "B": 1, "T": 8192, "H": 96, "d": 128, "chunk": 64, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["auto", "tensor", "fp32"], default="auto")
    ap.add_argument("--cpu-heads", type=int, default=96, help="heads of the prefill workload the oracle baseline runs")
    ap.add_argument("--ref-heads", type=int, default=8, help="heads per step of the reference arm")
    ap.add_argument("--only", choices=["all", "prefill", "concurrent", "decode", "decode_conv", "conv", "kernels",
                                       "logits", "norm", "varlen", "long", "oproj"], default="all",
                    help="profiling runs: time one workload only")
    ap.add_argument("--prefill-T", type=int, default=None, help="shorter prefill (profiling cases only)")
    ap.add_argument("--oproj-rows", type=int, default=None,
                    help="with --only oproj: one o_proj leg of this many rows (profiling cases only)")
    ap.add_argument("--headline", choices=["fused", "concurrent"], default="fused",
                    help="the prefill form timed as the headline value (the other is reported beside it)")
    ap.add_argument("--decode-B", type=int, default=None, help="smaller decode batch (profiling cases only)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-conv", action="store_true")
    ap.add_argument("--no-logits", action="store_true")
    ap.add_argument("--no-norm", action="store_true")
    ap.add_argument("--no-oproj", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the varlen and long prefill workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import torch
    from kimi_delta_attention_gated_gb300 import build as kbuild
    kbuild.build()
    peaks = load_peaks()
    if args.only in ("concurrent", "decode", "decode_conv", "conv", "kernels", "logits", "norm", "varlen", "long",
                     "oproj"):
        if args.only == "concurrent":  # the prefill's concurrent form alone (profiling runs)
            res = bench_prefill(args, world, rank, peaks, form="concurrent")[0]
        elif args.only == "oproj":
            res = bench_o_proj(args, world, peaks)
        elif args.only in ("varlen", "long"):
            res = bench_prefill_workload(args, world, peaks, args.only)
        elif args.only == "kernels":  # decode step + short convolution (profiling runs)
            res = {"decode": bench_decode(args, world, peaks), "short_conv": bench_short_conv(args, world, peaks)}
        elif args.only == "logits":  # the prefill with gates from logits alone (profiling runs)
            res = bench_prefill_logits(args, world, peaks)
        elif args.only == "norm":  # the prefill with the fused gated norm alone (profiling runs)
            res = bench_prefill_norm(args, world, peaks)
        elif args.only == "decode_conv":
            res = bench_decode_conv(args, world, peaks)
        else:
            res = bench_decode(args, world, peaks) if args.only == "decode" else bench_short_conv(args, world, peaks)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    pre, d = bench_prefill(args, world, rank, peaks, form=args.headline)
    other_form = "fused" if args.headline == "concurrent" else "concurrent"
    other = None if args.only == "prefill" else bench_prefill(args, world, rank, peaks, form=other_form)[0]
    split = None if args.only == "prefill" else bench_prefill(args, world, rank, peaks, form="split")[0]
    dec = None if (args.no_decode or args.only == "prefill") else bench_decode(args, world, peaks)
    if dec is not None:
        dec["fused_short_conv"] = bench_decode_conv(args, world, peaks)
    conv = None if (args.no_conv or args.only == "prefill") else bench_short_conv(args, world, peaks)
    logits = None if (args.no_logits or args.only == "prefill") else bench_prefill_logits(args, world, peaks)
    norm = None if (args.no_norm or args.only == "prefill") else bench_prefill_norm(args, world, peaks)
    oproj = None if (args.no_oproj or args.only == "prefill") else bench_o_proj(args, world, peaks)
    varlen = long_ = None
    if not (args.no_workloads or args.only == "prefill"):
        varlen = bench_prefill_workload(args, world, peaks, "varlen")
        long_ = bench_prefill_workload(args, world, peaks, "long")
    e2e = None if (args.no_e2e or args.only == "prefill") else bench_e2e(args, world, d)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.only == "all":
        cpu = cpu_baseline(d, args.cpu_heads)
        if dec is not None:
            dec["cpu_baseline_one_core"] = cpu_baseline_decode_one_core()
    if rank != 0:
        return
    dtype = "f32" if args.mode == "fp32" else "bf16 hi/lo split operands, f32 accumulate and state"
    line = {
        "metric": METRIC, "value": pre["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": pre["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic", "config": pre["config"],
        "roofline": pre["roofline"], "roofline_tensor": pre["roofline_tensor"], "cpu_baseline": cpu,
        "e2e": e2e, "gpu_launches": pre["gpu_launches"], "clocks": pre["clocks"], "decode": dec,
        "short_conv": conv, "prefill_gate_logits": logits, "prefill_gated_norm": norm, "o_proj": oproj,
        "prefill_varlen": varlen, "prefill_long_norm": long_, "gpu": torch.cuda.get_device_name(),
        "prefill_split_two_kernels": None if split is None else {
            "value": split["value"], "ms_per_step": split["ms_per_step"], "roofline": split["roofline"]},
        f"prefill_{other_form}": None if other is None else {
            "value": other["value"], "ms_per_step": other["ms_per_step"], "roofline": other["roofline"],
            "prepass_share": other.get("prepass_share")},
    }
    if pre.get("prepass_share") is not None:
        line["prepass_share"] = pre["prepass_share"]
    line["summary"] = summary(pre, dec, varlen, long_, logits, norm, conv, oproj, split, other, other_form)
    print(json.dumps(line), flush=True)


def summary(pre, dec, varlen, long_, logits, norm, conv, oproj, split=None, other=None, other_form=None):
    """Every timed workload in a few numbers, last on the line so that a reader of the
    line's tail sees all of them: kernel ms per launch, throughput and the fraction of
    the binding roofline (of the measured peak)."""
    def row(r, unit_scale, unit):
        if r is None:
            return None
        f = r["roofline"]
        return {"kernel_ms": round(f["kernel_ms"], 4), unit: round(r["value"] / unit_scale, 3),
                "frac": round(f["frac"], 4), "bound": f["bound"]}
    out = {"prefill_T8192": row(pre, 1e6, "Mtok_s"), "prefill_varlen": row(varlen, 1e6, "Mtok_s"),
           "prefill_long_norm": row(long_, 1e6, "Mtok_s"), "decode_B256": row(dec, 1e3, "Ktok_s"),
           "prefill_logits": row(logits, 1e6, "Mtok_s"), "prefill_norm_bf16": row(norm, 1e6, "Mtok_s"),
           "prefill_T8192_split": row(split, 1e6, "Mtok_s")}
    if other is not None:
        out[f"prefill_T8192_{other_form}"] = row(other, 1e6, "Mtok_s")
    for r, key in ((pre, "prefill_T8192"), (other, f"prefill_T8192_{other_form}")):
        if r is not None and r.get("prepass_share") is not None:
            out[key]["prepass_share"] = round(r["prepass_share"], 3)
    if dec and dec.get("fused_short_conv"):
        out["decode_conv_B256"] = row(dec["fused_short_conv"], 1e3, "Ktok_s")
    if conv:
        out["conv_prefill"] = row(conv["conv_prefill"], 1e6, "Mtok_s")
        out["conv_decode"] = row(conv["conv_decode"], 1e6, "Mtok_s")
    if oproj:
        out["o_proj_256"] = row(oproj["decode"], 1e6, "Mtok_s")
        out["o_proj_8192"] = row(oproj["prefill"], 1e6, "Mtok_s")
        for k, n in (("o_proj_256", "decode"), ("o_proj_8192", "prefill")):
            out[k]["cublas_ms"] = round(oproj[n]["torch_cublas_ms_same_inputs"], 4)
    return {k: v for k, v in out.items() if v is not None}


if __name__ == "__main__":
    main()
