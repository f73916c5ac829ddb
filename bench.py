#!/usr/bin/env python3
"""Benchmark of the routed-expert FP4 MoE layer on GB300.

Default workload: one MoE layer at the pages' shape (d=5120, f=2304, E=384 experts, top-k 6,
every expert resident in a 7.22 GB arena behind a permuted expert->slot table), decode with
T=1 token per call.  A step is 1000 fresh synthetic tokens processed one call at a time
(each call = router + top-k + slot lookup + gate/up SwiGLU + down + fixed-order combine),
replayed from a CUDA graph.  Metric: MoE-layer tokens/s.  The arena (7.2 GB) is far larger
than L2, so no L2 flush is inserted between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 (torchrun, one process per GPU) every rank runs an independent replica of the
layer (the path has no exchange step); value = all ranks' tokens / the slowest rank's time.
--impl reference times the CPU oracle (plain C, one host core) on a bounded sample of the
same workload.  Two more measurements ride on the same line (rank 0): "prefill" (one T=4096
chunk) and "cb3" (the decode workload with the experts in the 3-bit codebook format).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

D, F, E, K = 5120, 2304, 384, 6
TOKENS = 1000
SCALE = (-10, -6)
EXPERT_BYTES = 18_800_640
ROUTER_BYTES = E * D * 2
# per token: 6 experts' full FP4 weights + scales, the router matrix, x in and y out
ALG_BYTES_PER_TOKEN = K * EXPERT_BYTES + ROUTER_BYTES + 2 * D * 2
# dominant kernel, the expert FFN (one launch per decode call: gate/up + SwiGLU + down +
# combine): the 6 chosen experts' three FP4 matrices (codes + UE8M0 scales) + x in + y out
FFN_BYTES = K * EXPERT_BYTES + 2 * D * 2
METRIC = "MoE-layer tokens/s (T=1 decode, d=5120 f=2304 E=384 k=6)"
CONFIG = {"workload": "decode T=1, one MoE layer, d=5120 f=2304 E=384 top-k=6, 384 resident experts (7.22 GB arena, "
                      "permuted slot table), 1000 fresh tokens per step",
          "tokens_per_step": TOKENS, "l2": "inputs larger than L2 (7.22 GB arena), no flush"}


def max_over_ranks(v: float, dist=None, device=None) -> float:
    """The slowest rank's time: all-reduce MAX over the process group (identity without one)."""
    if dist is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's step time."""
    return world * units_per_rank / (ms_per_step / 1e3)


def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


FFN_SOURCES = ("fp4_routed_expert_gb300/csrc/mxf4_decode.cu", "fp4_routed_expert_gb300/csrc/mxf4_common.cuh",
               "fp4_routed_expert_gb300/csrc/moe_internal.cuh", "fp4_routed_expert_gb300/csrc/route_select.cuh")
FFN_KERNEL = "mxf4_decode_kernel"
TRAFFIC_RECORD = "profiles/traffic_expert_ffn_decode_T1_d5120_f2304_E384_k6.json"


def sources_digest(files) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return h.hexdigest()[:16]


def ffn_traffic():
    """DRAM bytes per FFN launch from the committed traffic record (written by --record-traffic
    from an ncu capture), if it was taken on the current kernel source, else None."""
    try:
        rec = json.load(open(os.path.join(ROOT, TRAFFIC_RECORD)))
        if rec.get("digest") == sources_digest(FFN_SOURCES):
            return int(rec["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


def record_traffic(csv_path: str, kernel_regex: str, out_path: str, command: str) -> dict:
    """Write the traffic record of one kernel from ncu's raw page (ncu -i REP --page raw --csv
    --print-units base): the mean of dram__bytes_read.sum + dram__bytes_write.sum over the
    captured launches whose name matches kernel_regex, with the digest of the FFN sources."""
    import csv
    import re
    rows = list(csv.reader(open(csv_path)))
    head = rows[0]
    ki = head.index("Kernel Name")
    ri, wi = head.index("dram__bytes_read.sum"), head.index("dram__bytes_write.sum")
    vals = []
    for r in rows[1:]:
        if len(r) <= max(ki, ri, wi) or not re.search(kernel_regex, r[ki]):
            continue
        try:
            vals.append(float(r[ri].replace(",", "")) + float(r[wi].replace(",", "")))
        except ValueError:
            continue            # the units row
    if not vals:
        raise SystemExit("no launch of %r with DRAM counters in %s" % (kernel_regex, csv_path))
    rec = {"kernel": kernel_regex, "launches": len(vals), "dram_bytes_per_launch": int(statistics.mean(vals)),
           "digest": sources_digest(FFN_SOURCES), "sources": list(FFN_SOURCES), "command": command}
    with open(os.path.join(ROOT, out_path), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            return json.load(open(p)), "measured"
        except Exception:
            pass
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.path = None

    def start(self):
        import tempfile
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks_bench_%d_" % self.gpu, suffix=".csv")
            self.f = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            lines = fh.readlines()
        os.unlink(self.path)
        for line in lines:
            p = [s.strip() for s in line.split(",")]
            if len(p) < 8:
                continue
            try:
                sm.append(float(p[0]))
                mx.append(float(p[1]))
            except ValueError:
                continue
            for n, v in zip(names, p[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- workload

def build_workload(device):
    import torch
    import fp4_routed_expert_gb300 as moe
    from fp4_routed_expert_gb300.layer import Arena, MoeLayer
    from synth import gpu as sgpu
    from synth import tensors as syn
    dims = moe.moe_dims(D, F, E, K)
    table = syn.permuted_slot_table(0, 0, E)
    arena = Arena(dims, E, device)
    stage = sgpu.ExpertStaging(D, F, device)
    for e in range(E):
        arena.pack(int(table[e]), stage.fill(0, 0, e, *SCALE))
    torch.cuda.synchronize()
    del stage
    x_bits = syn.activations(0, 0, TOKENS, D, stream=7)
    wr_bits = syn.router_weight(0, 0, E, D)
    def to_dev(b):
        return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).to(device).view(torch.bfloat16)
    x = to_dev(x_bits)
    wr = to_dev(wr_bits)
    tab = torch.from_numpy(table).to(device)
    layer = MoeLayer(D, F, E, K, 1, arena, device)
    y = torch.empty((TOKENS, D), dtype=torch.bfloat16, device=device)
    return dict(layer=layer, arena=arena, x=x, wr=wr, tab=tab, y=y, x_bits=x_bits, wr_bits=wr_bits, table=table)


def token_calls(w, i, stream=None, split=False):
    """One decode call of token i: routing and experts in one request (the router hands its
    key records to the expert kernel), or as the two separate calls."""
    layer = w["layer"]
    if split:
        layer.route(w["x"][i:i + 1], w["wr"], w["tab"], None, T=1, stream=stream)
        layer.experts(w["x"][i:i + 1], T=1, stream=stream, y=w["y"][i:i + 1])
    else:
        layer.decode(w["x"][i:i + 1], w["wr"], w["tab"], None, T=1, stream=stream, y=w["y"][i:i + 1])


class CudaRt:
    """Event record nodes inside a captured graph (external events) for per-kernel timing."""

    def __init__(self):
        self.rt = None
        for name in ("libcudart.so.13", "libcudart.so"):
            try:
                self.rt = ctypes.CDLL(name)
                break
            except OSError:
                continue

    def ok(self):
        return self.rt is not None

    def event(self):
        ev = ctypes.c_void_p()
        if self.rt.cudaEventCreate(ctypes.byref(ev)) != 0:
            raise RuntimeError("cudaEventCreate failed")
        return ev

    def record_external(self, ev, stream_handle):
        # cudaEventRecordExternal = 1: an event record node when the stream is capturing
        return self.rt.cudaEventRecordWithFlags(ev, ctypes.c_void_p(stream_handle), 1)

    def elapsed_ms(self, a, b):
        ms = ctypes.c_float()
        if self.rt.cudaEventElapsedTime(ctypes.byref(ms), a, b) != 0:
            return None
        return ms.value


def run_ours(args, rank, world, local_rank):
    import torch
    import fp4_routed_expert_gb300 as moe
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    w = build_workload(device)
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()
    # eager warm-up (sets kernel attributes before capture)
    with torch.cuda.stream(stream):
        for i in range(4):
            token_calls(w, i, split=(i % 2 == 1))
    torch.cuda.synchronize()
    # graph of one step; every 10th token runs the routing and expert calls separately, its
    # expert-FFN kernel bracketed by external event nodes (the other calls are single requests,
    # with no host-visible point between their two kernels)
    rt = CudaRt()
    probes = []
    g = torch.cuda.CUDAGraph()
    launches_before = moe.moe_kernel_launches()
    with torch.cuda.graph(g, stream=stream):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(TOKENS):
            layer = w["layer"]
            probe = rt.ok() and i % 10 == 5
            if not probe:
                token_calls(w, i)
                continue
            layer.route(w["x"][i:i + 1], w["wr"], w["tab"], None, T=1)
            a, b = rt.event(), rt.event()
            rt.record_external(a, h)
            layer.experts(w["x"][i:i + 1], T=1, y=w["y"][i:i + 1])
            rt.record_external(b, h)
            probes.append((a, b))
    launches_per_step = moe.moe_kernel_launches() - launches_before   # kernels in one replay
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kernel_ms = []
    with torch.cuda.stream(stream):
        ev0.record()
        for _ in range(args.steps):
            g.replay()
        ev1.record()
    torch.cuda.synchronize()
    if probes:
        # the probe events hold the last replay's times
        kernel_ms = [rt.elapsed_ms(a, b) for a, b in probes]
        kernel_ms = [v for v in kernel_ms if v is not None]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), dist, device)
    ms_per_step = total_ms / args.steps
    value = job_throughput(TOKENS, world, ms_per_step)
    # end-to-end through the public API with host buffers: pinned x in, y out, every step
    x_host = torch.empty((TOKENS, D), dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(w["x"].cpu())
    y_host = torch.empty((TOKENS, D), dtype=torch.bfloat16, pin_memory=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(args.steps):
            w["x"].copy_(x_host, non_blocking=True)
            g.replay()
            y_host.copy_(w["y"], non_blocking=True)
        e1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, device)
    status = int(w["layer"].status.item())
    peaks, peak_kind = measured_peaks()
    out = None
    if rank == 0:
        k_ms = statistics.mean(kernel_ms) if kernel_ms else None
        achieved = (FFN_BYTES / (k_ms * 1e-3) / 1e9) if k_ms else None
        peak = float(peaks["hbm_gbs"])
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "fp4 (e2m1 x e2m1 block-scaled tcgen05 MMA, UE8M0/32, activations as 4 MXFP4 terms; fp32 accumulate)",
            "data": "synthetic (seeded Philox FP4 experts, N(0,1) bf16 tokens, N(0,0.02) bf16 router)",
            "config": dict(CONFIG, parallelism="replicas" if world > 1 else "single GPU"),
            "roofline": {"bound": "hbm", "kernel": FFN_KERNEL + " (expert FFN: gate/up + SwiGLU + down + combine, T=1)",
                         "achieved": round(achieved, 1) if achieved else None, "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4) if achieved else None, "traffic": ffn_traffic(),
                         "bytes_per_launch": FFN_BYTES, "launch_ms": round(k_ms, 5) if k_ms else None,
                         "launches_timed": "one call in ten, whose routing runs as a separate call so that events "
                                           "can bracket this kernel; the other nine are single requests whose "
                                           "expert kernel selects from the router's key records",
                         "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_kind if peak_kind == "measured" else "fallback 6.8 TB/s"},
            "layer_roofline": {"bytes_per_token": ALG_BYTES_PER_TOKEN,
                               "achieved_gbs": round(ALG_BYTES_PER_TOKEN * value / world / 1e9, 1),
                               "frac": round(ALG_BYTES_PER_TOKEN * value / world / 1e9 / peak, 4)},
            "e2e": {"value": round(job_throughput(TOKENS, world, e2e_ms), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": TOKENS * D * 2, "d2h_bytes_per_step": TOKENS * D * 2},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
            "device_status": status,
        }
    return out, w


# ---------------------------------------------------------------------------- prefill chunk

PREFILL_T = 4096
PREFILL_BIAS = (1.2, 0.04)   # Zipf s, beta of the per-expert score bias


def run_prefill(w, args, device, resident=None):
    """One prefill chunk at the pages' shape: T=4096 tokens of N(0,1) bf16, Zipf(1.2)-skewed
    score bias, every expert resident; route -> permute -> expert FFN -> combine, graph-replayed.
    resident = n keeps only the first n experts routable (the rest masked): the diagnostic
    compute-bound case (n = 12: about 2,048 tokens per expert, above the ridge point).
    Returns the measurement object added to the JSON line."""
    import torch
    from fp4_routed_expert_gb300.layer import MoeLayer
    from synth import tensors as syn
    T = PREFILL_T
    xb = syn.activations(0, 0, T, D, stream=9)
    bias = torch.from_numpy(syn.zipf_score_bias(0, 0, E, *PREFILL_BIAS)).to(device)
    x = torch.from_numpy(np.ascontiguousarray(xb).view(np.int16)).to(device).view(torch.bfloat16)
    layer = MoeLayer(D, F, E, K, T, w["arena"], device)
    y = torch.empty((T, D), dtype=torch.bfloat16, device=device)
    tab = w["tab"]
    if resident is not None:
        keep = np.full(E, -1, np.int32)
        keep[:resident] = w["table"][:resident]
        tab = torch.from_numpy(keep).to(device)
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        layer.route(x, w["wr"], tab, bias)
        layer.experts(x, fused_prefill=True, y=y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer.route(x, w["wr"], tab, bias)
        layer.experts(x, fused_prefill=True, y=y)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g.replay()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    ids = layer.ids[:T].cpu().numpy()
    used = int(np.unique(ids[ids >= 0]).size)
    # per-call breakdown: the same kernels in a second graph with event probes around each call
    # (the combine issued as its own call, as the fused call launches it)
    import fp4_routed_expert_gb300 as moe
    rt = CudaRt()

    def probed(probe):
        with probe("route"):
            layer.route(x, w["wr"], tab, bias)
        with probe("permute"):
            moe.moe_permute(layer.dims, T, layer.ids, layer.offsets, layer.row_src, layer.row_dst, layer.ws)
        with probe("ffn (plan + A quantise + gate/up + down)"):
            moe.moe_expert_ffn_fp4(layer.dims, layer.arena.c, T, x, layer.ids, layer.slots, layer.w, layer.offsets,
                                   layer.row_src, layer.row_dst, 0, layer.rows, None, layer.status, layer.ws)
        with probe("combine"):
            moe.moe_combine(layer.dims, T, layer.rows, layer.row_dst, layer.w, y)

    g2, probes = _probe_graph(stream, probed, rt)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g2.replay()
    torch.cuda.synchronize()
    pk = _probe_ms(rt, probes)
    peaks, kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    fp4 = float(peaks["bf16_tflops"]) * (13.5 / 2.25)   # FP4 dense peak = measured bf16 x nominal ratio
    bytes_ = used * EXPERT_BYTES + ROUTER_BYTES + 2 * T * D * 2
    flops = 6.0 * T * K * D * F                          # gate, up, down: 2 flops per multiply-add
    what = ("all experts resident" if resident is None else
            "DIAGNOSTIC (not a workload of the pages): only experts 0..%d routable, ~%d tokens per expert"
            % (resident - 1, T * K // resident))
    return {"workload": "prefill chunk T=%d, d=%d f=%d E=%d top-k=%d, Zipf(s=%.1f, beta=%.2f) score bias, %s; "
                        "route + permute + expert FFN + combine" % (T, D, F, E, K, *PREFILL_BIAS, what),
            "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_chunk": round(ms, 4),
            "experts_used": used, "status": int(layer.status.item()),
            "roofline_hbm": {"bound": "hbm", "achieved": round(bytes_ / (ms * 1e-3) / 1e9, 1), "peak": hbm,
                             "unit": "GB/s", "frac": round(bytes_ / (ms * 1e-3) / 1e9 / hbm, 4), "bytes": bytes_},
            "roofline_fp4": {"bound": "tensor", "achieved": round(flops / (ms * 1e-3) / 1e12, 2), "peak": round(fp4, 1),
                             "unit": "TFLOP/s", "frac": round(flops / (ms * 1e-3) / 1e12 / fp4, 4),
                             "peak_source": "measured bf16 x 6 (nominal fp4/bf16 dense ratio)" if kind == "measured"
                             else "fallback bf16 x 6"},
            "breakdown_ms": {n: round(statistics.mean(v), 4) for n, v in pk.items()},
            "breakdown_note": "event-bracketed calls of one replay of a second graph (the combine as its own call); "
                              "the ffn call's own kernels (plan, quantise, FFN) are split in the ncu launch list"}


# ---------------------------------------------------------------------------- 40-layer keep-set workloads

KS_DECODE_STEPS = 20          # fresh tokens (T=1) or verify batches (T=16) per replay
LONG_T, LONG_CHUNKS = 8192, 4  # a 32,768-token sequence in four chunks
LONG_BIAS = (1.1, 0.04)       # Zipf s, beta of the fresh per-layer score bias
NORM_EPS = 1e-6


def _probe_graph(stream, body, rt):
    """Capture body(probe) into a graph; probe(name) returns a context that brackets the calls
    inside it with external event record nodes.  Returns (graph, {name: [(a, b), ...]})."""
    import contextlib
    import torch
    probes = {}

    @contextlib.contextmanager
    def probe(name, on=True):
        if not (on and rt.ok()):
            yield
            return
        h = torch.cuda.current_stream().cuda_stream
        a, b = rt.event(), rt.event()
        rt.record_external(a, h)
        yield
        rt.record_external(b, h)
        probes.setdefault(name, []).append((a, b))

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body(probe)
    return g, probes


def _probe_ms(rt, probes):
    out = {}
    for name, pairs in probes.items():
        v = [rt.elapsed_ms(a, b) for a, b in pairs]
        v = [x for x in v if x is not None]
        if v:
            out[name] = v
    return out


def _fractions(bytes_, flops, ms, peaks, kind):
    hbm = float(peaks["hbm_gbs"])
    fp4 = float(peaks["bf16_tflops"]) * (13.5 / 2.25)
    gbs = bytes_ / (ms * 1e-3) / 1e9
    tfs = flops / (ms * 1e-3) / 1e12
    return ({"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
             "bytes": int(bytes_), "peak_source": "%s hbm_gbs" % kind},
            {"bound": "tensor", "achieved": round(tfs, 3), "peak": round(fp4, 1), "unit": "TFLOP/s",
             "frac": round(tfs / fp4, 5), "flops": float(flops),
             "peak_source": "%s bf16 x 6 (nominal fp4/bf16 dense ratio)" % kind})


def run_keepset_decode(ks, T, args, device):
    """One 40-layer decode (T=1) or DSpark-verify (T=16) step per fresh input, KS_DECODE_STEPS
    of them per graph replay: each layer routes over its 154 resident experts (the rest masked),
    runs the expert FFN with the combine fused, and the next layer's input is
    bf16(RMSNorm(x + y)) computed on the device.  Distinct experts per layer (U) are counted
    from an eager pass over the same inputs, which is also the warm-up."""
    import torch
    import fp4_routed_expert_gb300 as moe
    from fp4_routed_expert_gb300.layer import MoeLayer
    from synth import tensors as syn
    from synth.keepset import LAYERS, KEEP, bits_to_device
    S = KS_DECODE_STEPS
    layer = MoeLayer(D, F, E, K, T, ks.arena, device)
    xs = bits_to_device(syn.activations(0, 0, S * T, D, stream=15 if T == 1 else 14), device).view(S, T, D)
    x = torch.empty((T, D), dtype=torch.bfloat16, device=device)
    y = torch.empty((T, D), dtype=torch.bfloat16, device=device)
    ids_log = torch.empty((S, LAYERS, T, K), dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device)

    def step(s, probe=None, log=False):
        x.copy_(xs[s])
        for l in range(LAYERS):
            on = probe is not None and s == S // 2
            # routing and experts as two calls: between layers the RMSNorm step (a plain
            # launch) ends the overlap of consecutive calls, and then the router's last block
            # selecting while the expert kernel's CTAs start measured faster than every CTA
            # selecting (the single request of moe_layer_decode_fp4)
            with (probe("route", on) if on else _null()):
                layer.route(x, ks.wr[l], ks.tab_dev[l], None, T=T)
            if log:
                ids_log[s, l].copy_(layer.ids[:T])
            with (probe("ffn", on) if on else _null()):
                layer.experts(x, T=T, y=y)
            with (probe("norm", on) if on else _null()):
                moe.moe_residual_rmsnorm(T, D, x, y, NORM_EPS, x)

    with torch.cuda.stream(stream):
        for s in range(S):
            step(s, log=True)
    torch.cuda.synchronize()
    ids = ids_log.cpu().numpy()
    U = np.array([[np.unique(ids[s, l][ids[s, l] >= 0]).size for l in range(LAYERS)] for s in range(S)])
    rt = CudaRt()
    before = moe.moe_kernel_launches()
    g, probes = _probe_graph(stream, lambda probe: [step(s, probe) for s in range(S)], rt)
    launches = moe.moe_kernel_launches() - before
    ms = _replay_ms(g, stream, args)
    pk = _probe_ms(rt, probes)
    status = int(layer.status.item())
    peaks, kind = measured_peaks()
    per_layer_io = 2 * T * D * 2 + KEEP * D * 2          # x in, y out, the resident router rows
    bytes_ = float(U.sum()) * EXPERT_BYTES + S * LAYERS * per_layer_io
    flops = 6.0 * S * LAYERS * T * K * D * F
    hbm, fp4 = _fractions(bytes_, flops, ms, peaks, kind)
    out = {"workload": "40-layer keep-set %s: d=%d f=%d E=%d (154 resident per layer, 6,160 slots, %.1f GB arena, "
                       "Zipf(1.1) keep-sets, non-resident experts masked), top-k=%d, T=%d; %d fresh %s per replay, "
                       "layers chained by bf16(RMSNorm(x + y)) on the device"
                       % ("decode" if T == 1 else "DSpark verify", D, F, E, ks.arena.num_slots * EXPERT_BYTES / 1e9,
                          K, T, S, "tokens" if T == 1 else "16-token batches"),
           "value": round(S * T / (ms * 1e-3), 2), "unit": "tokens/s (through all 40 layers)",
           "ms_per_step": round(ms / S, 4), "layer_tokens_per_s": round(S * T * LAYERS / (ms * 1e-3), 1),
           "distinct_experts_per_layer": {"mean": round(float(U.mean()), 2), "min": int(U.min()), "max": int(U.max())},
           "roofline_hbm": hbm, "roofline_fp4": fp4, "status": status, "gpu_launches_per_replay": launches,
           "l2": "inputs larger than L2 (115.8 GB arena; each layer streams U experts), no flush"}
    if "ffn" in pk:
        s_mid = S // 2
        fb = float(U[s_mid].sum()) * EXPERT_BYTES + LAYERS * 2 * T * D * 2
        f_ms = sum(pk["ffn"])
        out["ffn_roofline"] = {"bound": "hbm", "kernel": "expert FFN + fused combine (one call per layer)",
                               "achieved": round(fb / (f_ms * 1e-3) / 1e9, 1), "peak": float(peaks["hbm_gbs"]),
                               "unit": "GB/s", "frac": round(fb / (f_ms * 1e-3) / 1e9 / float(peaks["hbm_gbs"]), 4),
                               "launch_us_mean": round(1e3 * f_ms / len(pk["ffn"]), 2)}
        out["breakdown_us_per_layer"] = {n: round(1e3 * statistics.mean(v), 2) for n, v in pk.items()}
        out["breakdown_note"] = ("event-bracketed calls of the middle step of one replay: route = router + top-k + "
                                 "slot lookup, ffn = expert FFN + combine, norm = the chaining step")
    return out


class _null:
    def __enter__(self):
        return None

    def __exit__(self, *a):
        return False


def _replay_ms(g, stream, args, reps=None):
    import torch
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g.replay()
    torch.cuda.synchronize()
    reps = reps or max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def run_long_prefill(ks, args, device):
    """A 32,768-token sequence as four 8,192-token chunks through the 40 keep-set layers, a fresh
    Zipf(1.1) score bias per layer, layers chained by bf16(RMSNorm(x + y)) on the device.  One
    graph holds one chunk's 40 layers; a step copies each chunk's input in and replays it.  The
    first pass (eager) logs the routing for U and warms up; a second graph with event probes
    and the combine issued as its own call gives the per-call breakdown of one chunk."""
    import torch
    import fp4_routed_expert_gb300 as moe
    from fp4_routed_expert_gb300.layer import MoeLayer
    from synth import tensors as syn
    from synth.keepset import LAYERS, KEEP, bits_to_device
    T = LONG_T
    layer = MoeLayer(D, F, E, K, T, ks.arena, device)
    xs = [bits_to_device(syn.activations(0, 0, T, D, start_token=c * T, stream=13), device) for c in range(LONG_CHUNKS)]
    bias = [torch.from_numpy(syn.zipf_score_bias(0, l, E, *LONG_BIAS)).to(device) for l in range(LAYERS)]
    x = torch.empty((T, D), dtype=torch.bfloat16, device=device)
    y = torch.empty((T, D), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.Stream(device)
    U = np.zeros((LONG_CHUNKS, LAYERS), np.int64)
    with torch.cuda.stream(stream):
        for c in range(LONG_CHUNKS):
            x.copy_(xs[c])
            for l in range(LAYERS):
                layer.route(x, ks.wr[l], ks.tab_dev[l], bias[l])
                ids = layer.ids[:T].cpu().numpy()
                U[c, l] = np.unique(ids[ids >= 0]).size
                layer.experts(x, fused_prefill=True, y=y)
                moe.moe_residual_rmsnorm(T, D, x, y, NORM_EPS, x)
    torch.cuda.synchronize()

    def chunk(probe):
        for l in range(LAYERS):
            layer.route(x, ks.wr[l], ks.tab_dev[l], bias[l])
            layer.experts(x, fused_prefill=True, y=y)
            moe.moe_residual_rmsnorm(T, D, x, y, NORM_EPS, x)

    rt = CudaRt()
    before = moe.moe_kernel_launches()
    g, _ = _probe_graph(stream, chunk, rt)
    launches = moe.moe_kernel_launches() - before
    with torch.cuda.stream(stream):
        for c in range(LONG_CHUNKS):       # warm replays
            x.copy_(xs[c])
            g.replay()
    torch.cuda.synchronize()
    reps = 1 if args.steps < 10 else 2
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            for c in range(LONG_CHUNKS):
                x.copy_(xs[c])
                g.replay()
        e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    status = int(layer.status.item())

    # per-call breakdown of one chunk: the same kernels, the combine issued as its own call
    def chunk_probed(probe):
        for l in range(LAYERS):
            with probe("route"):
                layer.route(x, ks.wr[l], ks.tab_dev[l], bias[l])
            with probe("permute"):
                moe.moe_permute(layer.dims, T, layer.ids, layer.offsets, layer.row_src, layer.row_dst, layer.ws)
            with probe("ffn (plan + A quantise + gate/up + down)"):
                moe.moe_expert_ffn_fp4(layer.dims, layer.arena.c, T, x, layer.ids, layer.slots, layer.w,
                                       layer.offsets, layer.row_src, layer.row_dst, 0, layer.rows, None,
                                       layer.status, layer.ws)
            with probe("combine"):
                moe.moe_combine(layer.dims, T, layer.rows, layer.row_dst, layer.w, y)
            with probe("norm"):
                moe.moe_residual_rmsnorm(T, D, x, y, NORM_EPS, x)

    g2, probes = _probe_graph(stream, chunk_probed, rt)
    with torch.cuda.stream(stream):
        x.copy_(xs[0])
        g2.replay()
        x.copy_(xs[0])
        g2.replay()
    torch.cuda.synchronize()
    pk = _probe_ms(rt, probes)
    peaks, kind = measured_peaks()
    per_layer_io = 2 * T * D * 2 + KEEP * D * 2
    bytes_ = float(U.sum()) * EXPERT_BYTES + LONG_CHUNKS * LAYERS * per_layer_io
    flops = 6.0 * LONG_CHUNKS * LAYERS * T * K * D * F
    hbm, fp4 = _fractions(bytes_, flops, ms, peaks, kind)
    out = {"workload": "long prefill: 32,768 tokens as 4 x 8,192-token chunks through 40 keep-set layers (154 resident "
                       "of 384 per layer, 6,160 slots), d=%d f=%d top-k=%d, fresh Zipf(s=%.1f, beta=%.2f) score bias "
                       "per layer, layers chained by bf16(RMSNorm(x + y)) on the device; route + permute + expert FFN "
                       "+ combine per chunk-layer" % (D, F, K, *LONG_BIAS),
           "value": round(LONG_CHUNKS * T / (ms * 1e-3), 1), "unit": "tokens/s (through all 40 layers)",
           "ms_per_sequence": round(ms, 3), "ms_per_chunk_layer": round(ms / (LONG_CHUNKS * LAYERS), 4),
           "layer_tokens_per_s": round(LONG_CHUNKS * T * LAYERS / (ms * 1e-3), 1),
           "distinct_experts_per_chunk_layer": {"mean": round(float(U.mean()), 2), "min": int(U.min()),
                                                "max": int(U.max())},
           "roofline_hbm": hbm, "roofline_fp4": fp4, "status": status, "gpu_launches_per_chunk": launches,
           "timed": "%d pass(es) over the whole sequence after one eager and one graph warm-up pass" % reps}
    if pk:
        tot = sum(sum(v) for v in pk.values())
        out["breakdown_ms_per_chunk"] = {n: round(sum(v), 3) for n, v in pk.items()}
        out["breakdown_share"] = {n: round(sum(v) / tot, 4) for n, v in pk.items()}
        out["breakdown_note"] = ("one chunk (40 layers) of a second graph with event probes around each call; "
                                 "the combine runs as its own call there (the same kernel the fused call launches)")
    return out


def run_keepset(args, device):
    import torch
    from synth.keepset import KeepSetArena
    t0 = time.perf_counter()
    ks = KeepSetArena(device)
    build_s = time.perf_counter() - t0
    out = {"arena": {"slots": ks.arena.num_slots, "gb": round(ks.arena.num_slots * EXPERT_BYTES / 1e9, 2),
                     "build_s": round(build_s, 1)}}
    out["keepset_decode"] = run_keepset_decode(ks, 1, args, device)
    out["keepset_verify"] = run_keepset_decode(ks, 16, args, device)
    if not args.no_long_prefill:
        out["long_prefill"] = run_long_prefill(ks, args, device)
    ks.release()
    del ks
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------- cb3 experts

CB3_SLOT_BYTES = 13_426_688
SM_COUNT, SM_MAX_MHZ, FP32_LANES_PER_SM = 152, 2070, 128


def run_cb3(w, args, device):
    """The same decode workload with the experts in the cb3 format (3-bit per-row codebook,
    packed on the device from the FP4 arena): route + cb3 expert FFN per token, graph-replayed,
    events around every 10th token's FFN.  Also the output's distance from the FP4 layer on
    the same tokens (the approximation's cost).  Returns the object added to the JSON line."""
    import torch
    import fp4_routed_expert_gb300 as moe
    from fp4_routed_expert_gb300.layer import Cb3Arena
    dims = moe.moe_dims(D, F, E, K)
    cb = Cb3Arena(dims, E, device)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    t0 = time.perf_counter()
    for s_ in range(E):
        cb.pack_from(w["arena"], s_, s_, st)
    torch.cuda.synchronize()
    pack_s = time.perf_counter() - t0
    layer = w["layer"]
    y = torch.empty_like(w["y"])
    stream = torch.cuda.Stream(device)
    with torch.cuda.stream(stream):
        for i in range(4):
            layer.route(w["x"][i:i + 1], w["wr"], w["tab"], None, T=1)
            layer.experts_cb3(cb, w["x"][i:i + 1], T=1, y=y[i:i + 1])
    torch.cuda.synchronize()
    rt = CudaRt()
    probes = []
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(TOKENS):
            layer.route(w["x"][i:i + 1], w["wr"], w["tab"], None, T=1)
            probe = rt.ok() and i % 10 == 5
            if probe:
                a, b = rt.event(), rt.event()
                rt.record_external(a, h)
            layer.experts_cb3(cb, w["x"][i:i + 1], T=1, y=y[i:i + 1])
            if probe:
                rt.record_external(b, h)
                probes.append((a, b))
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g.replay()
    torch.cuda.synchronize()
    reps = max(3, min(args.steps, 10))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    k_ms = [rt.elapsed_ms(a, b) for a, b in probes]
    k_ms = statistics.mean([v for v in k_ms if v is not None]) if k_ms else None
    # distance from the FP4 layer (w["y"] holds the FP4 path's outputs for the same tokens)
    yc, yf = y.float(), w["y"].float()
    rel = ((yc - yf).abs().amax(dim=1) / yf.abs().amax(dim=1).clamp_min(1e-30)).cpu().numpy()
    peaks, kind = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    prods = 3 * K * D * F                                  # weight x activation products per token
    peak_alu = SM_COUNT * FP32_LANES_PER_SM * SM_MAX_MHZ * 1e6 / 1e12
    bytes_ = K * CB3_SLOT_BYTES + 2 * D * 2
    out = {"workload": "decode T=1 as above, experts in the cb3 format (8 bf16 levels per row, 3-bit indices; "
                       "%d B per expert, %.1f%% of FP4)" % (CB3_SLOT_BYTES, 100.0 * CB3_SLOT_BYTES / EXPERT_BYTES),
           "value": round(TOKENS / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 4),
           "pack_s": round(pack_s, 3), "experts_packed": E, "status": int(st.item()) | int(layer.status.item()),
           "vs_fp4_row_rel_err": {"median": float(np.median(rel)), "max": float(rel.max())}}
    if k_ms:
        out["ffn_launch_ms"] = round(k_ms, 5)
        out["roofline_alu"] = {"bound": "alu", "achieved": round(prods / (k_ms * 1e-3) / 1e12, 3), "peak": round(peak_alu, 2),
                               "unit": "T weight-products/s", "frac": round(prods / (k_ms * 1e-3) / 1e12 / peak_alu, 4),
                               "peak_source": "152 SMs x 128 FP32 lanes x 2070 MHz: one instruction per product"}
        out["roofline_hbm"] = {"bound": "hbm", "achieved": round(bytes_ / (k_ms * 1e-3) / 1e9, 1), "peak": hbm,
                               "unit": "GB/s", "frac": round(bytes_ / (k_ms * 1e-3) / 1e9 / hbm, 4), "bytes": bytes_}
    del cb
    return out


# ---------------------------------------------------------------------------- oracle timing

def oracle_sample(n_tokens, time_budget_s=None, x_bits=None, wr_bits=None, table=None, start_token=0):
    """Time the oracle on tokens [start_token, start_token + n_tokens) of the same workload;
    expert tensors are generated beforehand (outside the timing)."""
    import oracle
    from synth import tensors as syn
    if x_bits is None:
        x_bits = syn.activations(0, 0, n_tokens, D, start_token=start_token, stream=7)
        wr_bits = syn.router_weight(0, 0, E, D)
        table = syn.permuted_slot_table(0, 0, E)
    r = oracle.route_topk(x_bits[:n_tokens], wr_bits, None, table, K)
    inv = {int(s): e for e, s in enumerate(table)}
    cache = {}
    for t in range(n_tokens):
        for s in r["slots"][t]:
            if int(s) not in cache:
                cache[int(s)] = syn.expert_tensors(0, 0, inv[int(s)], D, F, *SCALE)
    t0 = time.perf_counter()
    done = 0
    for t in range(n_tokens):
        rr = oracle.route_topk(x_bits[t:t + 1], wr_bits, None, table, K)
        z = np.zeros((K, D), np.float32)
        for j in range(K):
            _, z[j] = oracle.expert_ffn_f32(x_bits[t], cache[int(rr["slots"][0, j])])
        oracle.combine_f32(z, rr["weights"][0])
        done += 1
        if time_budget_s and time.perf_counter() - t0 > time_budget_s:
            break
    el = time.perf_counter() - t0
    return done, el


def _oracle_shard(start_token):
    """One host core's share of the sharded oracle timing (a spawned process)."""
    return oracle_sample(2, start_token=start_token)


def cpu_baseline_block():
    """The oracle timed on the host: one core on the first tokens (about 15 s), then the same
    plain routine token-sharded over every host core, each process on its own two tokens
    (processes are spawned: the parent has already used the GPU)."""
    import multiprocessing as mp
    n, el = oracle_sample(24, time_budget_s=15.0)
    single = n / el
    cores = os.cpu_count() or 1
    try:
        with mp.get_context("spawn").Pool(cores) as pool:
            res = pool.map(_oracle_shard, [100 + 2 * i for i in range(cores)])
        tokens = sum(r[0] for r in res)
        value = tokens / max(r[1] for r in res)
        sample = ("%d tokens on %d host cores, token-sharded (2 per process, the slowest process's time), "
                  "plus %d tokens on 1 core (%.4f tokens/s, %.1f s); full layer per token: exact router over 384 "
                  "experts, 6 experts' SwiGLU FFN in sequential fp32, fixed-order combine; plain single-threaded C per process"
                  % (tokens, cores, n, single, el))
        return {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
                "single_core_value": round(single, 4)}
    except Exception as exc:   # the single-core figure still stands
        return {"value": round(single, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": "%d tokens of the same workload on 1 core, %.1f s (sharded run failed: %s)" % (n, el, exc)}


def _oracle_token_layer(x_row, seed_layer, table, bias):
    """Time the oracle on one token through one layer (exact router over the 384 experts, the
    chosen experts' fp32 SwiGLU FFNs, fixed-order combine); expert tensors are generated
    beforehand, outside the timing.  Returns seconds."""
    import oracle
    from synth import tensors as syn
    r = oracle.route_topk(x_row[None], _WR_CACHE.setdefault(seed_layer, syn.router_weight(0, seed_layer, E, D)),
                          bias, table, K)
    experts = {int(e): syn.expert_tensors(0, seed_layer, int(e), D, F, *SCALE) for e in r["ids"][0] if e >= 0}
    t0 = time.perf_counter()
    rr = oracle.route_topk(x_row[None], _WR_CACHE[seed_layer], bias, table, K)
    z = np.zeros((K, D), np.float32)
    for j in range(K):
        e = int(rr["ids"][0, j])
        if e >= 0:
            _, z[j] = oracle.expert_ffn_f32(x_row, experts[e])
    oracle.combine_f32(z, rr["weights"][0])
    return time.perf_counter() - t0


_WR_CACHE = {}


def _oracle_configs_shard(i):
    """One host core's sample for the multi-layer and prefill workloads (a spawned process):
    one token-layer each of the keep-set decode, the T=4096 prefill chunk and the long
    prefill, teacher-forced (each layer's input is a fresh synthetic token; the oracle's cost
    does not depend on the values)."""
    from synth import tensors as syn
    from synth.keepset import KEEP, LAYERS, ZIPF_S
    tabs = syn.keepset_slot_tables(0, LAYERS, E, KEEP, ZIPF_S)
    l = (7 * i + 3) % LAYERS
    out = {}
    x = syn.activations(0, 0, 1, D, start_token=i, stream=15)
    out["keepset"] = _oracle_token_layer(x[0], l, tabs[l], None)
    x = syn.activations(0, 0, 1, D, start_token=(97 * i) % PREFILL_T, stream=9)
    out["prefill"] = _oracle_token_layer(x[0], 0, syn.permuted_slot_table(0, 0, E),
                                         syn.zipf_score_bias(0, 0, E, *PREFILL_BIAS))
    c = i % LONG_CHUNKS
    x = syn.activations(0, 0, 1, D, start_token=c * LONG_T + (131 * i) % LONG_T, stream=13)
    out["long"] = _oracle_token_layer(x[0], l, tabs[l], syn.zipf_score_bias(0, l, E, *LONG_BIAS))
    return out


def config_cpu_baselines():
    """The oracle's host throughput for the keep-set decode/verify, the prefill chunk and the
    long prefill: every host core (spawned processes) times one token-layer of each; a
    workload's rate is the sampled token-layers over the slowest process's time, divided by
    the layers a token passes through.  The full workloads (20 steps x 40 layers, 4,096
    tokens, 4 x 8,192 tokens x 40 layers) would take hours on the host: these figures are
    linear extrapolations from the sample and say so."""
    import multiprocessing as mp
    cores = os.cpu_count() or 1
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_oracle_configs_shard, range(cores))
    out = {}
    for key, layers, name in (("keepset", 40, "keepset_decode"), ("prefill", 1, "prefill"), ("long", 40, "long_prefill")):
        t = [r[key] for r in res]
        rate = len(t) / max(t)                       # token-layers per second over all cores
        out[name] = {"value": round(rate / layers, 5), "unit": "tokens/s (through all %d layer%s)"
                     % (layers, "s" if layers > 1 else ""), "cores": cores, "kind": "oracle",
                     "extrapolated": True,
                     "sample": "%d token-layers, one per host core in parallel (median %.2f s each, slowest %.2f s); "
                               "rate = token-layers / slowest time / %d layers, extrapolated linearly to the whole "
                               "workload" % (len(t), statistics.median(t), max(t), layers)}
    out["keepset_verify"] = dict(out["keepset_decode"])     # same per-token-layer work in the oracle
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return None
    per_step = 2
    for _ in range(args.warmup):
        oracle_sample(per_step)
    times = []
    for _ in range(args.steps):
        n, el = oracle_sample(per_step)
        times.append(el / n)
    tps = 1.0 / statistics.mean(times)
    return {"metric": METRIC, "value": round(tps, 4), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * per_step / tps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 (oracle FFN: sequential fp32 sums), exact-then-fp32 router",
            "data": "synthetic", "config": dict(CONFIG, parallelism="single host core"), "impl": "reference",
            "cpu_baseline": {"value": round(tps, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": "%d tokens per step of the same workload" % per_step},
            "e2e": {"value": round(tps, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--experts", type=int, default=384,
                    help="experts resident in the arena (profiling runs use fewer; the metric is defined at 384)")
    ap.add_argument("--tokens", type=int, default=1000, help="tokens per step")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill-chunk measurement")
    ap.add_argument("--no-cb3", action="store_true", help="skip the cb3-format decode measurement")
    ap.add_argument("--no-keepset", action="store_true",
                    help="skip the 40-layer keep-set measurements (they need a 115.8 GB arena)")
    ap.add_argument("--no-long-prefill", action="store_true", help="skip the 4 x 8,192-token long prefill")
    ap.add_argument("--record-traffic", metavar="RAW_CSV",
                    help="write the decode FFN traffic record from ncu's raw page (--print-units base) and exit")
    ap.add_argument("--traffic-command", default="", help="the ncu command the raw page came from (recorded)")
    ap.add_argument("--keepset-only", action="store_true",
                    help="measure only the 40-layer keep-set workloads (profiling runs)")
    ap.add_argument("--cb3-only", action="store_true",
                    help="measure only the cb3-format decode leg (profiling runs; the FP4 layer runs once, eagerly, "
                         "for the comparison)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="measure only the prefill chunk (profiling runs; with --experts the arena holds fewer experts)")
    ap.add_argument("--prefill-resident", type=int, default=None,
                    help="with --prefill-only: only the first N experts routable (the compute-bound diagnostic)")
    args = ap.parse_args()
    global E, TOKENS, ROUTER_BYTES, ALG_BYTES_PER_TOKEN
    E, TOKENS = args.experts, args.tokens
    ROUTER_BYTES = E * D * 2
    ALG_BYTES_PER_TOKEN = K * EXPERT_BYTES + ROUTER_BYTES + 2 * D * 2
    if E != 384 or TOKENS != 1000:
        CONFIG["workload"] = "PROFILING VARIANT (not the metric's workload): E=%d experts, %d tokens per step" % (E, TOKENS)
        CONFIG["tokens_per_step"] = TOKENS
        CONFIG["l2"] = "arena of %.2f GB (each call streams 6 experts, 112.8 MB, more than L2), no flush" % (
            E * EXPERT_BYTES / 1e9)
    rank, world, local_rank = env_rank()
    if args.record_traffic:
        print(json.dumps(record_traffic(args.record_traffic, FFN_KERNEL, TRAFFIC_RECORD, args.traffic_command)))
        return 0
    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return 0
    import fp4_routed_expert_gb300 as moe
    moe.lib()
    if args.prefill_only:
        if rank == 0:
            import torch
            torch.cuda.set_device(local_rank)
            dev = torch.device("cuda", local_rank)
            out = {"metric": "prefill chunk tokens/s", "impl": "ours", "config": dict(CONFIG),
                   "prefill": run_prefill(build_workload(dev), args, dev, resident=args.prefill_resident)}
            print(json.dumps(out), flush=True)
        return 0
    if args.keepset_only:
        if rank == 0:
            import torch
            torch.cuda.set_device(local_rank)
            dev = torch.device("cuda", local_rank)
            out = {"metric": "40-layer keep-set tokens/s", "impl": "ours"}
            out.update(run_keepset(args, dev))
            print(json.dumps(out), flush=True)
        return 0
    if args.cb3_only:
        if rank == 0:
            import torch
            torch.cuda.set_device(local_rank)
            dev = torch.device("cuda", local_rank)
            w = build_workload(dev)
            for i in range(TOKENS):
                token_calls(w, i)
            out = {"metric": "cb3 decode tokens/s", "impl": "ours", "config": dict(CONFIG), "cb3": run_cb3(w, args, dev)}
            print(json.dumps(out), flush=True)
        return 0
    out, w = run_ours(args, rank, world, local_rank)
    if rank == 0 and out is not None and not args.no_prefill and E == 384:
        import torch
        out["prefill"] = run_prefill(w, args, torch.device("cuda", local_rank))
        out["prefill_diagnostic_12_experts"] = run_prefill(w, args, torch.device("cuda", local_rank), resident=12)
    if rank == 0 and out is not None and not args.no_cb3 and E == 384:
        import torch
        out["cb3"] = run_cb3(w, args, torch.device("cuda", local_rank))
    if rank == 0 and out is not None and not args.no_keepset and E == 384:
        import torch
        del w["arena"], w["layer"]
        torch.cuda.empty_cache()
        out.update(run_keepset(args, torch.device("cuda", local_rank)))
    if rank == 0 and out is not None:
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline_block()
            if E == 384:
                for name, blk in config_cpu_baselines().items():
                    if isinstance(out.get(name), dict):
                        out[name]["cpu_baseline"] = blk
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
