"""Throughput of the low-bit decode GEMV path on GB300 (one JSON line on rank 0).

A step is one decode pass (batch 1) over the large-shape workload: CQ-W4A8 GEMV
(``a8_quantize`` -> ``cq_gemv``, which rotates the activations in its prologue) and Q4_0
GEMV (``q4_0_gemv``) on the four matrices [8192, 8192], [28672, 8192], [8192, 28672] and
the lm_head [128256, 4096]
(1.15 GB of packed weights per step, far larger than L2, so no flush is needed).
Weights are encoded once before timing (offline, as the format intends); the timed
region holds only the decode work (K replays of the step captured as a CUDA graph, one
event pair around them; the per-kernel
times behind ``roofline`` come from a second pass of the same steps with events around
each launch).  ``value`` is algorithmic GB/s: packed indices +
norms (CQ) or Q4_0 blocks, plus activations and outputs, divided by the step time.

The line also reports every other workload of the path:
  * ``prefill``: the grouped prefill GEMM of the 20-layer model, TFLOP/s and the
    fraction of the bf16 peak as flat keys per M;
  * ``batched`` (the large-shape decode at batches 2, 8, 32): ``cq_gemv`` at 4 bits, ``q4_0_gemv`` (B = 2)
    and ``q4_0_gemm`` (B >= 8), GB/s, each call timed alone after an L2 flush;
  * ``mixed``: ``cq_gemv`` at b = 1..4 on [4096, 4096] and [11008, 4096] with
    outliers, batches 1 / 4 / 16;
  * ``small``: CQ-W4A8 512 x 512 and one Minueza Q4_0 layer, each as
    single-call latency and as streamed GB/s over weight copies spanning 4x the L2;
  * ``narrow``: batch-1 decode of 1-bit, 2-bit and ternary rows through ``cq_gemv`` and the
    table-lookup ``cq_gemv_lut`` (timed in a child process after everything else);
  * ``cpu_baseline``: the oracle timed on the host cores, on sampled rows of the timed
    step's own encoded weights, with its outputs checked against the GPU's (``parity``);
  * ``summary`` (last): the headline number of every workload as flat keys.

``--impl reference`` times the CPU oracle as it stands on a bounded sample of the same
workload.  ``--gpus N`` (under torchrun) runs N independent replicas, one per GPU:
the path needs no exchange, so there is no collective beyond the timing barrier.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("decode GEMV GB/s & Gweights/s (frac of HBM); prefill GEMM TFLOP/s "
          "(frac of TC peak)")
WORKLOAD = ("large-shape decode, batch 1: CQ-W4A8 GEMV (4-bit, group 128, int8 per-token "
            "activations) and Q4_0 GEMV on [8192,8192], [28672,8192], [8192,28672], "
            "lm_head [128256,4096]")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def load_codebook():
    """The committed Lloyd-Max table (cb2 | cb3 | cb4 as float32 bit patterns)."""
    with open(os.path.join(ROOT, "tests", "golden", "codebook_seed0.json")) as f:
        d = json.load(f)
    hexes = d["cb2_f32_hex"] + d["cb3_f32_hex"] + d["cb4_f32_hex"]
    return np.array([int(h, 16) for h in hexes], dtype=np.uint32).view(np.float32)


def kernel_source_hash():
    """Hash of the sources the batch-1 decode kernels of the timed step are built from (the
    4-bit integer-codeword GEMV and the Q4_0 GEMV, with their shared header and dispatch);
    the recorded DRAM traffic is valid only for the sources it was captured on."""
    h = hashlib.sha256()
    for name in ("gemv.cu", "gemv_fx.cu", "gemv_pipe.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "gemm_cq_gemv_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, alg_bytes_per_launch):
    """DRAM bytes per launch for ``kernel``, scaled from the committed ncu capture.

    The capture covers one matrix of the workload (``profiles/traffic.json``); its
    DRAM-bytes / algorithmic-bytes ratio is applied to this run's algorithmic bytes per
    launch.  None when the kernel source changed since the counters were taken.
    """
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(kernel)
    if not rec or rec.get("source_hash") != kernel_source_hash():
        return None
    return int(round(rec["traffic_over_algorithmic"] * alg_bytes_per_launch))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        with open(self.out.name) as f:
            rows = [r.strip().split(",") for r in f if r.strip()]
        os.unlink(self.out.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[3:7]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------
# The GPU arm
# ------------------------------------------------------------------------------------
def build_workload(dev, cb, torch, cq, synth, only=None):
    """Encode the large-shape weights once (device) and allocate every step buffer.  The
    step's activations are views into one device buffer and its outputs into another
    (``xbuf``, ``ybuf`` of every entry), so the end-to-end leg moves each with one copy."""
    sel = [(i, m) for i, m in enumerate(synth.LARGE) if not only or m.name in only]
    xbuf = torch.empty((sum(m.K for _, m in sel),), dtype=torch.float32, device=dev)
    ybuf = torch.empty((sum(2 * m.N for _, m in sel),), dtype=torch.float32, device=dev)
    xo = yo = 0
    mats = []
    for i, m in sel:
        g = torch.Generator(device=dev)
        g.manual_seed(synth.weight_seed(4, i))
        W = torch.randn((m.N, m.K), device=dev, generator=g) * 0.02
        packed, norms = cq.cq_encode(W, 4, cb)
        blocks = cq.q4_0_quantize(W)
        del W
        gx = torch.Generator(device=dev)
        gx.manual_seed(synth.activation_seed(4, 1) + i)
        X = xbuf[xo:xo + m.K].view(1, m.K)   # K, N are multiples of 4: 16-byte aligned views
        X.copy_(torch.randn((1, m.K), device=dev, generator=gx))
        xo += m.K
        mats.append(dict(
            m=m, packed=packed, norms=norms, blocks=blocks, X=X,
            Xq=torch.empty((1, m.K), dtype=torch.int8, device=dev),
            s=torch.empty((1,), dtype=torch.float32, device=dev),
            ws=torch.empty((cq.cq_gemv_workspace_bytes(1, m.K),), dtype=torch.uint8, device=dev),
            Ycq=ybuf[yo:yo + m.N].view(1, m.N),
            Yq4=ybuf[yo + m.N:yo + 2 * m.N].view(1, m.N),
            xbuf=xbuf, ybuf=ybuf))
        yo += 2 * m.N
    torch.cuda.synchronize()
    torch.cuda.empty_cache()   # release the float32 weights before anything is timed
    return mats


def twin_buffers(mats, torch):
    """A second set of the step's device inputs and outputs (``xbuf``/``ybuf`` and their
    per-matrix views at the same offsets), sharing the weights and scratch of ``mats``."""
    xbuf = torch.empty_like(mats[0]["xbuf"]).copy_(mats[0]["xbuf"])
    ybuf = torch.empty_like(mats[0]["ybuf"])
    xo = yo = 0
    out = []
    for d in mats:
        m = d["m"]
        e = dict(d)
        e["X"] = xbuf[xo:xo + m.K].view(1, m.K)
        e["Ycq"] = ybuf[yo:yo + m.N].view(1, m.N)
        e["Yq4"] = ybuf[yo + m.N:yo + 2 * m.N].view(1, m.N)
        e["xbuf"], e["ybuf"] = xbuf, ybuf
        xo += m.K
        yo += 2 * m.N
        out.append(e)
    return out


def step_bytes(mats):
    cq_b = sum(d["packed"].numel() + 2 * d["norms"].numel() + d["m"].K + 4 + 4 * d["m"].N
               for d in mats)
    q4_b = sum(d["blocks"].numel() + 4 * d["m"].K + 4 * d["m"].N for d in mats)
    weights = sum(2 * d["m"].N * d["m"].K for d in mats)
    return cq_b, q4_b, weights


def run_step(mats, cb, cq, events=None, kinds=("cq", "q4_0")):
    """One decode pass.  With ``events``, brackets each GEMV launch for per-kernel time."""
    for d in mats:
        m = d["m"]
        if "cq" in kinds:
            cq.a8_quantize(d["X"], Xq=d["Xq"], scale=d["s"])
            if events is not None:
                events["cq_gemv"][0].append(_ev())
            cq.cq_gemv(d["packed"], d["norms"], m.N, m.K, 4, cb, d["Xq"], d["s"], Y=d["Ycq"],
                       workspace=d["ws"])
            if events is not None:
                events["cq_gemv"][1].append(_ev())
        if "q4_0" in kinds:
            if events is not None:
                events["q4_0_gemv"][0].append(_ev())
            cq.q4_0_gemv(d["blocks"], m.N, m.K, d["X"], Y=d["Yq4"])
            if events is not None:
                events["q4_0_gemv"][1].append(_ev())


def reduce_max(x, dist, device):
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _ev():
    import torch
    e = torch.cuda.Event(enable_timing=True)
    e.record()
    return e


def build_prefill(dev, cb, torch, cq, synth, M):
    """The 20-layer synthetic 45M-parameter model (layer-major), encoded 4-bit on device."""
    gx = torch.Generator(device=dev)
    gx.manual_seed(synth.activation_seed(3, M))
    acts = {K: cq.a8_quantize(torch.randn((M, K), device=dev, generator=gx)) for K in (512, 1536)}
    items, flops = [], 0
    for i, (layer, m) in enumerate(synth.prefill_matrices()):
        g = torch.Generator(device=dev)
        g.manual_seed(synth.weight_seed(3, i))
        W = torch.randn((m.N, m.K), device=dev, generator=g) * 0.02
        packed, norms = cq.cq_encode(W, 4, cb)
        q, s = acts[m.K]
        items.append((packed, norms, m.N, m.K, q, s,
                      torch.empty((M, m.N), dtype=torch.bfloat16, device=dev)))
        flops += 2 * M * m.N * m.K
    probs = cq.make_gemm_problems(items)
    ws = torch.empty((cq.cq_gemm_grouped_workspace_bytes(probs, M),), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    return dict(items=items, probs=probs, ws=ws, flops=flops, M=M)


def time_prefill(pf, cb, cq, torch, steps, warmup):
    """Device time of the grouped prefill GEMM (rotation + tcgen05 GEMM): the call captured
    as a CUDA graph, `steps` replays between CUDA events."""
    f = lambda: cq.cq_gemm_grouped(pf["probs"], pf["M"], 4, cb, workspace=pf["ws"])
    for _ in range(warmup):
        f()
    torch.cuda.synchronize()
    cq.cq_device_error()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        f()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        graph.replay()   # one untimed replay
        e0.record(cap)
        for _ in range(steps):
            graph.replay()
        e1.record(cap)
    torch.cuda.synchronize()
    cq.cq_device_error()
    return e0.elapsed_time(e1) / steps


def prefill_report(dev, cb, torch, cq, synth, steps, warmup, peaks, kind):
    """The grouped prefill GEMM of the 20-layer model at each M, as flat scalar
    keys (``M512_tflops``, ``M512_frac``, ...) so that every number sits one level deep."""
    peak = float(peaks["bf16_tflops"])
    out = {"workload": "20-layer 45M-parameter model (q,o 512x512; k,v 128x512; up 1536x512; "
                       "down 512x1536), CQ-W4A8, one grouped launch of 120 matrices",
           "dtype": "fp16 MMA operands, fp32 accumulate, bf16 out",
           "kernel": "cq_gemm_kernel", "bound": "tensor", "unit": "TFLOP/s", "peak_tflops": peak,
           "peak_source": f"{kind} bf16_tflops (burst; the GEMM is timed alone; fp16 and bf16 "
                          "have the same nominal dense rate, ratio 1)"}
    for M in synth.PREFILL_TOKENS:
        pf = build_prefill(dev, cb, torch, cq, synth, M)
        ms = time_prefill(pf, cb, cq, torch, steps, warmup)
        tf = pf["flops"] / (ms * 1e-3) / 1e12
        out[f"M{M}_ms"] = round(ms, 4)
        out[f"M{M}_gflop"] = round(pf["flops"] / 1e9, 2)
        out[f"M{M}_tflops"] = round(tf, 1)
        out[f"M{M}_frac"] = round(tf / peak, 4)
        del pf
        torch.cuda.empty_cache()
    return out


def flushed_call_ms(torch, flush, fn, steps, warmup):
    """Median device time of ``fn`` over ``steps`` calls (after ``warmup``), each call alone
    between CUDA events with the L2 flushed (``flush`` larger than the L2 is zeroed) first."""
    for _ in range(warmup):
        fn()
    ts = []
    for _ in range(steps):
        flush.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def batched_report(mats, cb, torch, cq, synth, dev, steps, warmup, batches=(2, 8, 32),
                   kinds=("cq", "q4_0"), hbm=None):
    """The large-shape decode at batches above 1: ``cq_gemv`` at 4 bits (B >= 3 takes the tcgen05 path, B = 2
    one two-token CUDA-core pass) and, for Q4_0, ``q4_0_gemv`` at B = 2 and ``q4_0_gemm`` on
    the tensor cores at larger batches; per large matrix, each call timed alone with CUDA
    events after an L2 flush (the [8192, 8192] weights would otherwise stay in the 129 MB L2).
    GB/s counts the algorithmic bytes (weights once, activations and outputs)."""
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
    out = {"workload": "large-shape decode batches, weights read once per call for all tokens",
           "dtype": "B=2: fp32 (CUDA cores); B>=8: fp16 MMA operands, fp32 accumulate, fp32 out",
           "timing": "per call, CUDA events, L2 flushed before each call"}

    def one(fn):
        ms = flushed_call_ms(torch, flush, fn, steps, warmup)
        cq.cq_device_error()
        return ms

    for B in batches:
        q4_name = "q4_0_gemv" if B <= 2 else "q4_0_gemm"
        res = {k: {"us": {}, "bytes": 0, "ms": 0.0} for k in kinds}
        for i, d in enumerate(mats):
            m = d["m"]
            g = torch.Generator(device=dev)
            g.manual_seed(synth.activation_seed(4, B) + i)
            X = torch.randn((B, m.K), device=dev, generator=g)
            Y = torch.empty((B, m.N), dtype=torch.float32, device=dev)
            if "cq" in kinds:
                Xq, sc = cq.a8_quantize(X)
                ws = torch.empty((cq.cq_gemv_workspace_bytes(B, m.K),), dtype=torch.uint8, device=dev)
                ms = one(lambda: cq.cq_gemv(d["packed"], d["norms"], m.N, m.K, 4, cb, Xq, sc, Y=Y,
                                            workspace=ws))
                r = res["cq"]
                r["us"][m.name] = round(ms * 1e3, 1)
                r["ms"] += ms
                r["bytes"] += d["packed"].numel() + 2 * d["norms"].numel() + B * m.K + 4 * B * (1 + m.N)
            if "q4_0" in kinds:
                if B <= 2:
                    ms = one(lambda: cq.q4_0_gemv(d["blocks"], m.N, m.K, X, Y=Y))
                else:
                    ws = torch.empty((max(cq.q4_0_gemm_workspace_bytes(B, m.K), 256),), dtype=torch.uint8,
                                     device=dev)
                    ms = one(lambda: cq.q4_0_gemm(d["blocks"], m.N, m.K, X, Y=Y, workspace=ws))
                r = res["q4_0"]
                r["us"][m.name] = round(ms * 1e3, 1)
                r["ms"] += ms
                r["bytes"] += d["blocks"].numel() + 4 * B * m.K + 4 * B * m.N
        rep = {}
        for k, v in res.items():
            gbps = v["bytes"] / (v["ms"] * 1e-3) / 1e9
            e = {"us": v["us"], "GBps": round(gbps, 1)}
            if hbm:
                e["frac_of_hbm"] = round(gbps / hbm, 4)
            rep["cq_gemv" if k == "cq" else q4_name] = e
        out[f"B{B}"] = rep
    del flush
    torch.cuda.empty_cache()
    return out


def mixed_report(dev, cb, torch, cq, synth, steps, warmup, hbm):
    """The mixed-width sweep: CQ at every width b = 1..4 on [4096, 4096] and [11008, 4096] (weights with
    1 % x10 outliers), batches 1 / 4 / 16, each measured twice: one ``cq_gemv`` call timed
    alone after an L2 flush (``<matrix>_b<b>_B<B>_{us,GBps,Gwps,frac}``), and streamed:
    one CUDA graph of back-to-back calls over distinct copies of the weights spanning 4x
    the L2, per call (``..._streamed_{us,GBps,frac}``).  GB/s counts packed indices,
    norms, activations, scales and outputs."""
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)
    l2 = l2_bytes(torch, dev)
    out = {"workload": "CQ mixed widths: [4096,4096] (sq) and [11008,4096] (up), b=1..4, "
                       "batch 1/4/16, 1% x10 outliers",
           "timing": "per call, CUDA events, L2 flushed before each call; streamed: one graph "
                     "over distinct weight copies spanning 4x L2, per call",
           "peak_hbm_gbs": hbm}
    for i, m in enumerate(synth.CQ_MIXED):
        g = torch.Generator(device=dev)
        g.manual_seed(synth.weight_seed(2, i))
        W = torch.randn((m.N, m.K), device=dev, generator=g) * 0.02
        W = torch.where(torch.rand((m.N, m.K), device=dev, generator=g) < 0.01, W * 10.0, W)
        for b in synth.CQ_MIXED_BITS:
            packed, norms = cq.cq_encode(W, b, cb)
            for B in synth.CQ_MIXED_BATCHES:
                gx = torch.Generator(device=dev)
                gx.manual_seed(synth.activation_seed(2, B) + i)
                Xq, sc = cq.a8_quantize(torch.randn((B, m.K), device=dev, generator=gx))
                ws = torch.empty((cq.cq_gemv_workspace_bytes(B, m.K),), dtype=torch.uint8, device=dev)
                Y = torch.empty((B, m.N), dtype=torch.float32, device=dev)
                ms = flushed_call_ms(torch, flush, lambda: cq.cq_gemv(packed, norms, m.N, m.K, b, cb, Xq, sc,
                                                                      Y=Y, workspace=ws), steps, warmup)
                nbytes = packed.numel() + 2 * norms.numel() + B * m.K + 4 * B + 4 * B * m.N
                gbps = nbytes / (ms * 1e-3) / 1e9
                key = f"{m.name}_b{b}_B{B}"
                out[key + "_us"] = round(ms * 1e3, 1)
                out[key + "_GBps"] = round(gbps, 1)
                out[key + "_Gwps"] = round(m.N * m.K / (ms * 1e-3) / 1e9, 1)
                out[key + "_frac"] = round(gbps / hbm, 4)
                wbytes = packed.numel() + 2 * norms.numel()
                copies = -(-4 * l2 // wbytes)
                P = copies_of(torch, dev, packed, copies)
                Q = copies_of(torch, dev, norms, copies)
                ms_s = streamed_ms(torch, lambda: [cq.cq_gemv(P[c], Q[c], m.N, m.K, b, cb, Xq, sc, Y=Y,
                                                             workspace=ws) for c in range(copies)]) / copies
                gbps_s = nbytes / (ms_s * 1e-3) / 1e9
                out[key + "_streamed_us"] = round(ms_s * 1e3, 2)
                out[key + "_streamed_GBps"] = round(gbps_s, 1)
                out[key + "_streamed_frac"] = round(gbps_s / hbm, 4)
                del P, Q
            del packed, norms
        del W
        torch.cuda.empty_cache()
    cq.cq_device_error()
    del flush
    torch.cuda.empty_cache()
    return out


def _capture(torch, fn):
    """``fn``'s launches captured as a CUDA graph (replayed on the current stream)."""
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fn()
    torch.cuda.synchronize()
    return g


def streamed_ms(torch, fn, reps=3):
    """Device time of one replay of ``fn`` captured as a CUDA graph (after one untimed
    replay), averaged over ``reps`` back-to-back replays."""
    g = _capture(torch, fn)
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def copies_of(torch, dev, t, n):
    """``n`` copies of ``t`` in one buffer, each starting at a 256-byte boundary (distinct
    memory, so that streaming them reads every copy from HBM)."""
    per = t.numel() * t.element_size()
    stride = -(-per // 256) * 256
    flat = torch.empty((n * stride,), dtype=torch.uint8, device=dev)
    src = t.contiguous().view(torch.uint8).reshape(-1)
    views = []
    for c in range(n):
        v = flat[c * stride:c * stride + per]
        v.copy_(src)
        views.append(v.view(t.dtype).view(t.shape))
    return views


def l2_bytes(torch, dev):
    props = torch.cuda.get_device_properties(dev)
    return int(getattr(props, "L2_cache_size", 0) or (129 << 20))


def small_report(dev, cb, torch, cq, synth, steps, warmup):
    """The CQ 512 x 512 call and the Minueza Q4_0 layer, each reported twice: the latency
    of one call, replayed as a CUDA graph after an L2 flush, and the streamed throughput
    of back-to-back calls over distinct copies of the weights spanning 4x the L2 (one
    graph of all copies).  The calls are the fused decode chain (``cq_gemv_layer``: int8
    quantization, rotation and GEMV in one launch; ``q4_0_gemv_layer``: every matrix of the
    layer in one launch); the per-matrix launches of the unfused path are timed beside
    them (``unfused_latency_us``)."""
    l2 = l2_bytes(torch, dev)
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)

    def latency(fn):
        return flushed_call_ms(torch, flush, _capture(torch, fn).replay, steps, warmup)

    def streamed(fn, reps=3):
        return streamed_ms(torch, fn, reps)

    def copies_of_(t, n):
        return copies_of(torch, dev, t, n)

    def gen(shape, seed):
        g = torch.Generator(device=dev)
        g.manual_seed(seed)
        return torch.randn(shape, device=dev, generator=g)

    tiny = torch.empty((1,), dtype=torch.float32, device=dev)
    floor_us = latency(lambda: tiny.zero_()) * 1e3   # one trivial kernel, timed the same way
    out = {"timing": "latency: one call as a CUDA graph after an L2 flush, median; streamed: "
                     "one graph over distinct weight copies spanning 4x L2",
           "launch_floor_us": round(floor_us, 1),
           "launch_floor": "latency of one trivial kernel (a 1-element fill) measured the same way",
           "path": "fused decode chain: cq_gemv_layer (a8 + rotation + GEMV, one launch), "
                   "q4_0_gemv_layer (all matrices of the layer, one launch)",
           "l2_bytes": l2}
    # CQ-W4A8 512 x 512, batch 1: float32 activations in, one launch
    N = K = 512
    packed, norms = cq.cq_encode(gen((N, K), synth.weight_seed(0, 0)) * 0.02, 4, cb)
    X = gen((1, K), synth.activation_seed(0, 1))
    Y = torch.empty((1, N), dtype=torch.float32, device=dev)
    ws = torch.empty((cq.cq_gemv_workspace_bytes(1, K),), dtype=torch.uint8, device=dev)
    Xq = torch.empty((1, K), dtype=torch.int8, device=dev)
    sc = torch.empty((1,), dtype=torch.float32, device=dev)
    nbytes = packed.numel() + 2 * norms.numel() + 4 * K + 4 * N
    one = cq.make_gemv_layer([(packed, norms, N, K, X, Y)])
    us = latency(lambda: cq.cq_gemv_layer(one, 4, cb)) * 1e3

    def unfused():
        cq.a8_quantize(X, Xq=Xq, scale=sc)
        cq.cq_gemv(packed, norms, N, K, 4, cb, Xq, sc, Y=Y, workspace=ws)

    us_unfused = latency(unfused) * 1e3
    copies = -(-4 * l2 // nbytes)
    P = copies_of_(packed, copies)
    Q = copies_of_(norms, copies)
    calls = [cq.make_gemv_layer([(P[c], Q[c], N, K, X, Y)]) for c in range(copies)]
    ms = streamed(lambda: [cq.cq_gemv_layer(c1, 4, cb) for c1 in calls])
    per = cq.LAYER_MAX_PROBLEMS
    groups = [cq.make_gemv_layer([(P[c], Q[c], N, K, X, Y) for c in range(c0, min(c0 + per, copies))])
              for c0 in range(0, copies, per)]
    ms16 = streamed(lambda: [cq.cq_gemv_layer(g1, 4, cb) for g1 in groups])
    out["cq_w4a8_512x512"] = {
        "latency_us": round(us, 1), "unfused_latency_us": round(us_unfused, 1),
        "launches": 1, "unfused_launches": 2, "bytes_per_call": nbytes, "copies": copies,
        "streamed_us_per_call": round(ms * 1e3 / copies, 2),
        "streamed_GBps": round(copies * nbytes / (ms * 1e-3) / 1e9, 1),
        "streamed_Gweights_per_s": round(copies * N * K / (ms * 1e-3) / 1e9, 2),
        "streamed_16_per_launch_GBps": round(copies * nbytes / (ms16 * 1e-3) / 1e9, 1)}
    del P, Q, calls, groups, packed, norms
    # one Minueza layer in Q4_0 (8 matrices with the tied lm_head), batch 1
    layer = []
    xs = {}
    for i, m in enumerate(synth.MINUEZA_LAYER):
        blocks = cq.q4_0_quantize(gen((m.N, m.K), synth.weight_seed(1, i)) * 0.02)
        if m.K not in xs:
            xs[m.K] = gen((1, m.K), synth.activation_seed(1, 1) + m.K)
        layer.append((m, blocks, torch.empty((1, m.N), dtype=torch.float32, device=dev)))
    lbytes = sum(b.numel() + 4 * m.K + 4 * m.N for m, b, _ in layer)
    lweights = sum(m.N * m.K for m, _, _ in layer)
    fused = cq.make_q4_0_layer([(b, m.N, m.K, xs[m.K], y) for m, b, y in layer])
    us = latency(lambda: cq.q4_0_gemv_layer(fused)) * 1e3

    def one_layer():
        for m, b, y in layer:
            cq.q4_0_gemv(b, m.N, m.K, xs[m.K], Y=y)

    us_unfused = latency(one_layer) * 1e3
    copies = -(-4 * l2 // lbytes)
    reps = [(m, copies_of_(b, copies), y) for m, b, y in layer]
    lcalls = [cq.make_q4_0_layer([(b[c], m.N, m.K, xs[m.K], y) for m, b, y in reps]) for c in range(copies)]
    ms = streamed(lambda: [cq.q4_0_gemv_layer(c1) for c1 in lcalls])
    out["minueza_q4_0_layer"] = {"latency_us": round(us, 1), "unfused_latency_us": round(us_unfused, 1),
                                 "launches": 1, "unfused_launches": len(layer),
                                 "bytes_per_layer": lbytes, "copies": copies,
                                 "streamed_us_per_layer": round(ms * 1e3 / copies, 2),
                                 "streamed_GBps": round(copies * lbytes / (ms * 1e-3) / 1e9, 1),
                                 "streamed_Gweights_per_s": round(copies * lweights / (ms * 1e-3) / 1e9, 2)}
    cq.cq_device_error()
    del reps, layer, lcalls, flush
    torch.cuda.empty_cache()
    return out


def narrow_report(dev, cb, torch, cq, synth, steps, warmup, case=None, codes=None):
    """Batch-1 decode of 1-bit, 2-bit and ternary rows on the large shapes: ``cq_gemv``
    against the table-lookup ``cq_gemv_lut``, each call timed alone after an L2 flush, plus
    the largest relative difference between the two outputs (both compute the same product).
    ``case`` and ``codes`` restrict the matrices and the codes (profiling runs)."""
    flush = torch.empty((256 << 20,), dtype=torch.uint8, device=dev)

    def one(fn):
        return flushed_call_ms(torch, flush, fn, steps, warmup)

    peaks, kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    out = {"workload": "large-shape decode, batch 1, 1-bit / 2-bit / ternary CQ rows",
           "peak": {"hbm_gbs": hbm, "source": f"{kind} (hbm_gbs)"},
           "timing": "per call, CUDA events, L2 flushed before each call",
           "unit": "us per call; GB/s of algorithmic bytes over the four matrices"}
    for b, name in ((1, "b1"), (2, "b2"), (cq.CQ_TERNARY, "ternary")):
        if codes and name not in codes:
            continue
        res = {"cq_gemv": {"us": {}, "ms": 0.0}, "cq_gemv_lut": {"us": {}, "ms": 0.0}}
        nbytes = 0
        diff = 0.0
        for i, m in enumerate(synth.LARGE):
            if case and m.name not in case:
                continue
            g = torch.Generator(device=dev)
            g.manual_seed(synth.weight_seed(4, i))
            W = torch.randn((m.N, m.K), device=dev, generator=g) * 0.02
            packed, norms = cq.cq_encode(W, b, cb)
            del W
            gx = torch.Generator(device=dev)
            gx.manual_seed(synth.activation_seed(4, 1) + i)
            Xq, sc = cq.a8_quantize(torch.randn((1, m.K), device=dev, generator=gx))
            ws = torch.empty((cq.cq_gemv_workspace_bytes(1, m.K),), dtype=torch.uint8, device=dev)
            Yg = torch.empty((1, m.N), dtype=torch.float32, device=dev)
            Yl = torch.empty((1, m.N), dtype=torch.float32, device=dev)
            for key, fn in (("cq_gemv", lambda: cq.cq_gemv(packed, norms, m.N, m.K, b, cb, Xq, sc, Y=Yg,
                                                           workspace=ws)),
                            ("cq_gemv_lut", lambda: cq.cq_gemv_lut(packed, norms, m.N, m.K, b, cb, Xq, sc,
                                                                   Y=Yl))):
                ms = one(fn)
                res[key]["us"][m.name] = round(ms * 1e3, 1)
                res[key]["ms"] += ms
            nbytes += packed.numel() + 2 * norms.numel() + m.K + 4 + 4 * m.N
            den = float(Yg.abs().max())
            diff = max(diff, float((Yl - Yg).abs().max()) / (den if den > 0 else 1.0))
            del packed, norms
            torch.cuda.empty_cache()
        out[name] = {k: {"us": v["us"], "GBps": round(nbytes / (v["ms"] * 1e-3) / 1e9, 1),
                         "frac_of_hbm": round(nbytes / (v["ms"] * 1e-3) / 1e9 / hbm, 4)}
                     for k, v in res.items()}
        out[name]["max_rel_diff"] = float(f"{diff:.3g}")
    cq.cq_device_error()
    del flush
    torch.cuda.empty_cache()
    return out


def narrow_child(args, local_rank):
    """Runs narrow_report in a child process, so that a failure of the newer kernel can
    only cost this entry, never the rest of the line.  The child is a single-rank run on
    this process's GPU (no process group)."""
    cmd = [sys.executable, os.path.abspath(__file__), "--narrow-only", "--warmup", str(args.warmup)]
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK=str(local_rank))
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env)
    except subprocess.TimeoutExpired:
        return {"error": "timed out after 600 s"}
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    if r.returncode != 0 or not lines:
        tail = (r.stderr or r.stdout).strip().splitlines()[-3:]
        return {"error": f"exit {r.returncode}: " + " | ".join(tail)}
    try:
        return json.loads(lines[-1])
    except ValueError as e:
        return {"error": f"unreadable report: {e}"[:300]}


def gpu_arm(args, rank, world, local_rank):
    import torch
    import gemm_cq_gemv_gb300 as cq
    from gemm_cq_gemv_gb300 import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    cb = cq.make_codebook(load_codebook())
    if args.narrow_only:
        steps = args.steps if args.narrow_codes or args.case else 10
        print(json.dumps(narrow_report(dev, cb, torch, cq, synth, steps, args.warmup, case=args.case,
                                       codes=args.narrow_codes)), flush=True)
        return
    if args.small_only:
        print(json.dumps(small_report(dev, cb, torch, cq, synth, 10, args.warmup)), flush=True)
        return
    if args.mixed_only:
        peaks, _ = load_peaks()
        print(json.dumps(mixed_report(dev, cb, torch, cq, synth, 10, args.warmup,
                                      float(peaks["hbm_gbs"]))), flush=True)
        return
    if args.prefill_only:
        pf = build_prefill(dev, cb, torch, cq, synth, args.prefill_m)
        ms = time_prefill(pf, cb, cq, torch, args.steps, args.warmup)
        if rank == 0:
            print(json.dumps({"prefill_M": args.prefill_m, "ms": ms,
                              "tflops": pf["flops"] / (ms * 1e-3) / 1e12}), flush=True)
        return
    mats = build_workload(dev, cb, torch, cq, synth, only=args.case)
    kinds = tuple(args.kernels)
    if args.batched_only:
        rep_ = batched_report(mats, cb, torch, cq, synth, dev, args.steps, args.warmup,
                              batches=(args.batch,), kinds=kinds)
        if rank == 0:
            print(json.dumps(rep_), flush=True)
        return
    cq_b, q4_b, weights = step_bytes(mats)
    cq_b = cq_b if "cq" in kinds else 0
    q4_b = q4_b if "q4_0" in kinds else 0
    weights = weights // 2 * len(kinds)
    total_b = cq_b + q4_b

    for _ in range(args.warmup):
        run_step(mats, cb, cq, kinds=kinds)
    torch.cuda.synchronize()
    # one decode step captured as a CUDA graph (same launches, same buffers); the timed
    # region replays it K times
    cap = torch.cuda.Stream(device=dev)
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        run_step(mats, cb, cq, kinds=kinds)
    torch.cuda.synchronize()

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.4)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(cap):
        t0.record(cap)
        for _ in range(args.steps):
            graph.replay()
        t1.record(cap)
    torch.cuda.synchronize()
    cq.cq_device_error()
    if dist:
        dist.barrier()
    ms = reduce_max(t0.elapsed_time(t1) / args.steps, dist, dev)
    # per-kernel durations for the roofline: the same steps again with an event pair
    # around every launch (kept out of the step timing above: event records between
    # launches serialise the stream and cost ~40 us per step)
    events = {"cq_gemv": ([], []), "q4_0_gemv": ([], [])}
    for _ in range(args.steps):
        run_step(mats, cb, cq, events, kinds=kinds)
    torch.cuda.synchronize()
    clocks = sampler.stop() if sampler else None

    per_kernel = {}
    for k, (a, b) in events.items():
        if a:
            tot = sum(x.elapsed_time(y) for x, y in zip(a, b))
            per_kernel[k] = {"ms_total": tot, "launches": len(a)}
    if args.no_e2e:
        if rank == 0:
            print(json.dumps({"ms_per_step": ms, "kernels": per_kernel,
                              "GBps": total_b / (ms * 1e-3) / 1e9}), flush=True)
        if dist:
            dist.destroy_process_group()
        return

    # end to end through the public API with host buffers: every step copies its
    # activations from pinned host memory and reads its outputs back (every matrix's
    # activations in one buffer and its outputs in another: one copy each way).  The
    # copies run on a copy stream against two device sets of inputs and outputs, so
    # step i's read-back and step i+1's upload overlap step i's and i+1's neighbours'
    # compute; the timed region ends after the last read-back.
    sets = [mats, twin_buffers(mats, torch)]
    host_x = torch.empty(mats[0]["xbuf"].shape, dtype=torch.float32, pin_memory=True).copy_(mats[0]["xbuf"])
    host_y = torch.empty(mats[0]["ybuf"].shape, dtype=torch.float32, pin_memory=True)
    h2d = host_x.numel() * 4
    d2h = host_y.numel() * 4
    comp = torch.cuda.current_stream()
    copy = torch.cuda.Stream(device=dev)

    def e2e_run(n):
        done = [None, None]     # per set: its last step's compute finished
        up = [None, None]       # per set: its inputs uploaded
        def upload(k):
            with torch.cuda.stream(copy):
                if done[k] is not None:
                    copy.wait_event(done[k])   # the set's previous step no longer reads them
                sets[k][0]["xbuf"].copy_(host_x, non_blocking=True)
                up[k] = torch.cuda.Event()
                up[k].record(copy)
        upload(0)
        for i in range(n):
            k = i & 1
            if i + 1 < n:
                upload(k ^ 1)
            comp.wait_event(up[k])
            run_step(sets[k], cb, cq, kinds=kinds)
            done[k] = torch.cuda.Event()
            done[k].record(comp)
            with torch.cuda.stream(copy):
                copy.wait_event(done[k])
                host_y.copy_(sets[k][0]["ybuf"], non_blocking=True)
        comp.wait_stream(copy)

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    a = time.perf_counter()
    e2e_run(args.steps)
    torch.cuda.synchronize()
    e2e_ms = reduce_max((time.perf_counter() - a) * 1e3 / args.steps, dist, dev)

    if rank == 0:
        peaks, kind = load_peaks()
        hbm = float(peaks["hbm_gbs"])
        dom = max(per_kernel, key=lambda k: per_kernel[k]["ms_total"])
        dom_bytes = cq_b if dom == "cq_gemv" else q4_b
        dk = per_kernel[dom]
        achieved = dom_bytes * args.steps / (dk["ms_total"] * 1e-3) / 1e9
        value = world * total_b / (ms * 1e-3) / 1e9
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations)",
            "config": {"workload": WORKLOAD, "batch": 1, "group": 128, "cq_bits": 4,
                       "bytes_per_step": total_b, "weights_per_step": weights,
                       "l2": "inputs larger than L2 (1.15 GB of weights per step)",
                       "parallelism": f"replicas x{world}"},
            "gweights_per_s": round(world * weights / (ms * 1e-3) / 1e9, 2),
            "frac_of_hbm": round(value / world / hbm, 4),
            "kernels": {k: {"launches": v["launches"], "ms_total": round(v["ms_total"], 4),
                            "GBps": round((cq_b if k == "cq_gemv" else q4_b) * args.steps /
                                          (v["ms_total"] * 1e-3) / 1e9, 1)}
                        for k, v in per_kernel.items()},
            "kernel_timing": "a second pass of the same steps with CUDA events around each launch",
            "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1),
                         "peak": hbm, "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "peak_source": f"{kind} (MEASURED_PEAKS.json hbm_gbs)" if kind == "measured"
                         else "fallback 6.8 TB/s",
                         "algorithmic_bytes_per_launch": dom_bytes // len(mats),
                         "traffic": recorded_traffic(dom, dom_bytes // len(mats))},
            "e2e": {"value": round(world * total_b / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * len(mats) * (2 * ("cq" in kinds) + ("q4_0" in kinds)),
            "gpu_launches_note": "per decode step: a8_quantize and cq_gemv (which rotates the "
                                 "activations in its prologue at batch 1) per CQ matrix, one "
                                 "q4_0_gemv kernel per Q4_0 matrix",
            "clocks": clocks,
        }
        # host copies of sampled rows of the timed step (encoded bytes, activations, the
        # GPU's outputs) for the oracle check of the CPU-baseline leg below
        sample = (gpu_sample(mats, args.cpu_rows)
                  if not args.no_cpu_baseline and world == 1 and set(kinds) == {"cq", "q4_0"} else None)
        if not args.no_prefill:
            line["prefill"] = prefill_report(dev, cb, torch, cq, synth, max(3, args.steps // 5),
                                             args.warmup, peaks, kind)
        if not args.no_batched:
            line["batched"] = batched_report(mats, cb, torch, cq, synth, dev, 10, 3, kinds=kinds, hbm=hbm)
        if not args.no_mixed and world == 1 and "cq" in kinds:
            try:
                line["mixed"] = mixed_report(dev, cb, torch, cq, synth, 10, 3, hbm)
            except Exception as e:   # report, never lose the line
                line["mixed"] = {"error": f"{type(e).__name__}: {e}"[:300]}
        if not args.no_small and world == 1:
            try:
                line["small"] = small_report(dev, cb, torch, cq, synth, 10, 3)
            except Exception as e:   # report, never lose the line
                line["small"] = {"error": f"{type(e).__name__}: {e}"[:300]}
        if not args.no_narrow and world == 1:
            line["narrow"] = narrow_child(args, local_rank)
        if not args.no_cpu_baseline and world == 1:   # the oracle is timed at N = 1 only
            try:
                line["cpu_baseline"] = cpu_baseline_report(args.cpu_rows, sample=sample)
            except Exception as e:   # report, never lose the line
                line["cpu_baseline"] = {"error": f"{type(e).__name__}: {e}"[:300], "kind": "oracle"}
        line["summary"] = summary_of(line, hbm)   # last, so that it ends the printed line
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def summary_of(line, hbm):
    """Every workload's headline numbers as flat scalar keys, each named by its workload:
    ``cq512_*`` and ``minueza_q4_0_layer_*`` the small workloads (latency, streamed GB/s
    and its fraction of HBM), ``mixed_*`` the mixed-width sweep's fractions, ``prefill_*``
    the prefill GEMM, ``decode_B<B>_*`` the large-shape decode at each batch, plus the
    oracle check."""
    out = {}
    sm = line.get("small") or {}
    for key, name in (("cq512", "cq_w4a8_512x512"), ("minueza_q4_0_layer", "minueza_q4_0_layer")):
        r = sm.get(name)
        if isinstance(r, dict):
            out[f"{key}_latency_us"] = r.get("latency_us")
            out[f"{key}_streamed_GBps"] = r.get("streamed_GBps")
            if r.get("streamed_GBps"):
                out[f"{key}_streamed_frac"] = round(r["streamed_GBps"] / hbm, 4)
    mx = line.get("mixed") or {}
    for k, v in mx.items():
        if k.endswith("_frac"):
            out["mixed_" + k] = v
    pf = line.get("prefill") or {}
    for k in ("M512_tflops", "M512_frac", "M2048_tflops", "M2048_frac"):
        if k in pf:
            out["prefill_" + k] = pf[k]
    for k, v in (line.get("kernels") or {}).items():
        out[f"decode_B1_{k}_GBps"] = v.get("GBps")
        if v.get("GBps"):
            out[f"decode_B1_{k}_frac"] = round(v["GBps"] / hbm, 4)
    for bk, rep in (line.get("batched") or {}).items():
        if bk.startswith("B") and isinstance(rep, dict):
            for kern, v in rep.items():
                if isinstance(v, dict) and "GBps" in v:
                    out[f"decode_{bk}_{kern}_GBps"] = v["GBps"]
                    out[f"decode_{bk}_{kern}_frac"] = round(v["GBps"] / hbm, 4)
    par = (line.get("cpu_baseline") or {}).get("parity")
    if par:
        out["oracle_check_ok"] = par["ok"]
        out["oracle_check_cq"] = par["cq_gemv_max_rel_err"]
        out["oracle_check_q4_0"] = par["q4_0_gemv_max_rel_err"]
    return out


# ------------------------------------------------------------------------------------
# The oracle arm (CPU): the oracle as it stands, on a bounded sample of the workload
# ------------------------------------------------------------------------------------
def oracle_sample_step(rows, cb, synth, oracle, state, outputs=None):
    """Oracle GEMV of ``rows`` rows of every large matrix (both formats); returns bytes.
    With ``outputs`` (a list), appends each matrix's (cq, q4_0) oracle outputs to it."""
    nbytes = 0
    for d in state:
        m = d["m"]
        nbytes += d["p"].nbytes + d["n"].nbytes + m.K + 4 + 4 * rows
        ycq = oracle.cq_gemv_ref(d["p"], d["n"], 4, cb, d["q"], d["s"])
        nbytes += d["b"].nbytes + 4 * m.K + 4 * rows
        yq4 = oracle.q4_0_gemv_ref(d["b"], m.K, d["X"])
        if outputs is not None:
            outputs.append((ycq, yq4))
    return nbytes


def oracle_state(rows, cb, synth, oracle):
    state = []
    for i, m in enumerate(synth.LARGE):
        W = synth.weights(rows, m.K, seed=synth.weight_seed(4, i))
        X = synth.activations(1, m.K, seed=synth.activation_seed(4, 1) + i)
        p, n = oracle.cq_encode(W, 4, cb)
        q, s = oracle.a8_quantize(X)
        state.append(dict(m=m, p=p, n=n, q=q, s=s, X=X, b=oracle.q4_0_quantize(W)))
    return state


def gpu_sample(mats, rows):
    """Host copies of the first ``rows`` rows of every matrix of the timed decode step: the
    encoded weights the GPU streamed, the step's activations and the GPU's outputs for those
    rows (taken after the timed region; no arithmetic)."""
    out = []
    for d in mats:
        r = min(rows, d["m"].N)
        out.append(dict(m=d["m"], p=d["packed"][:r].cpu().numpy(),
                        n=d["norms"][:r].cpu().numpy().view("uint16"),
                        b=d["blocks"][:r].cpu().numpy(), q=d["Xq"].cpu().numpy(),
                        s=d["s"].cpu().numpy(), X=d["X"].cpu().numpy(),
                        y_cq=d["Ycq"][:, :r].cpu().numpy(), y_q4=d["Yq4"][:, :r].cpu().numpy()))
    return out


def _max_rel(y, ref):
    """max |y - ref| / max |ref| over one output vector (the sampled rows of it)."""
    y = np.asarray(y, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    den = float(np.max(np.abs(ref)))
    return float(np.max(np.abs(y - ref)) / (den if den > 0 else 1.0))


_BLAS_THREAD_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def blas_threads():
    """Threads NumPy's BLAS runs with: the pinning variable if one is set, else every core
    (the OpenBLAS default)."""
    for v in _BLAS_THREAD_VARS:
        if os.environ.get(v, "").isdigit():
            return int(os.environ[v])
    return os.cpu_count()


def cpu_baseline(rows, seconds=10.0, sample=None):
    """The oracle as it stands, timed on ``rows`` rows of each large matrix (both formats).

    With ``sample`` (``gpu_sample`` of the timed decode step) the oracle runs on exactly the
    bytes the GPU streamed, and its outputs are compared with the GPU's for those rows
    (``parity``: the float32-accumulation tolerance 1e-3 of the GEMV parity tests).
    Without it (the one-thread child, the reference arm) the sample is drawn and encoded
    here from the same seeds."""
    import oracle
    from gemm_cq_gemv_gb300 import synth
    cb = load_codebook()
    t0 = time.perf_counter()
    state = sample if sample is not None else oracle_state(rows, cb, synth, oracle)
    t1 = time.perf_counter()
    for d in state:
        oracle.cq_reconstruct(d["p"], d["n"], 4, cb)
        oracle.q4_0_dequantize(d["b"], d["m"].K)
    t2 = time.perf_counter()
    outputs = []
    oracle_sample_step(rows, cb, synth, oracle, state, outputs)
    # repeat the sample for about ten seconds of CPU work
    reps, nbytes = 0, 0
    a = time.perf_counter()
    while reps == 0 or time.perf_counter() - a < seconds:
        nbytes += oracle_sample_step(rows, cb, synth, oracle, state)
        reps += 1
    dt = time.perf_counter() - a
    out = {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": blas_threads(),
           "kind": "oracle",
           "sample": f"{reps} x {rows} rows of each large matrix, CQ-W4A8 and Q4_0, batch 1 "
                     f"(float64 reconstruction + product), {dt:.1f} s",
           "phases_s": {("copy_sample" if sample is not None else "draw_and_encode"): round(t1 - t0, 3),
                        "reconstruct": round(t2 - t1, 3),
                        "note": f"once over the same {rows}-row sample, both formats"}}
    if sample is not None:
        e_cq = max(_max_rel(d["y_cq"], o[0]) for d, o in zip(state, outputs))
        e_q4 = max(_max_rel(d["y_q4"], o[1]) for d, o in zip(state, outputs))
        out["parity"] = {"rows_per_matrix": rows, "cq_gemv_max_rel_err": float(f"{e_cq:.3g}"),
                         "q4_0_gemv_max_rel_err": float(f"{e_q4:.3g}"), "tol": 1e-3,
                         "ok": bool(e_cq < 1e-3 and e_q4 < 1e-3),
                         "what": "the timed step's outputs for these rows against the oracle "
                                 "on the same encoded bytes and activations"}
    return out


def cpu_baseline_report(rows, sample=None):
    """The oracle timed twice: with BLAS on every core (this process, on ``sample`` when
    given) and pinned to one thread (a child process, since BLAS reads its thread count
    when NumPy loads)."""
    out = cpu_baseline(rows, sample=sample)
    env = dict(os.environ, **{v: "1" for v in _BLAS_THREAD_VARS})
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-only", "--cpu-rows", str(rows)]
    try:
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
        lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
        out["one_thread"] = (json.loads(lines[-1]) if r.returncode == 0 and lines
                             else {"error": f"exit {r.returncode}"})
    except subprocess.TimeoutExpired:
        out["one_thread"] = {"error": "timed out after 300 s"}
    except ValueError as e:
        out["one_thread"] = {"error": f"unreadable report: {e}"[:300]}
    return out


def reference_arm(args, rank, world):
    if rank != 0:
        return
    import oracle
    from gemm_cq_gemv_gb300 import synth
    cb = load_codebook()
    rows = args.cpu_rows
    state = oracle_state(rows, cb, synth, oracle)
    for _ in range(args.warmup):
        oracle_sample_step(rows, cb, synth, oracle, state)
    a = time.perf_counter()
    nbytes = 0
    for _ in range(args.steps):
        nbytes += oracle_sample_step(rows, cb, synth, oracle, state)
    dt = time.perf_counter() - a
    value = nbytes / dt / 1e9
    ms = dt * 1e3 / args.steps
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) activations)",
        "config": {"workload": WORKLOAD, "batch": 1, "group": 128, "cq_bits": 4,
                   "parallelism": "cpu oracle, rank 0"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"{rows} rows of each large matrix per step, both formats"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-rows", type=int, default=256,
                    help="rows per matrix in the oracle sample (CPU baseline / reference arm)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-baseline-only", action="store_true",
                    help="print only the CPU oracle timing (the one-thread child of a full run)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="time the device step only and print a short line (profiling runs)")
    ap.add_argument("--case", nargs="*", default=None,
                    help="restrict to these large matrices (sq8k up28k down28k lm_head)")
    ap.add_argument("--kernels", nargs="*", default=["cq", "q4_0"], choices=["cq", "q4_0"])
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill GEMM report")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the grouped prefill GEMM (profiling runs)")
    ap.add_argument("--prefill-m", type=int, default=2048)
    ap.add_argument("--no-batched", action="store_true", help="skip the decode-batch report")
    ap.add_argument("--no-mixed", action="store_true", help="skip the mixed-width CQ sweep")
    ap.add_argument("--batched-only", action="store_true",
                    help="time only the tensor-core decode batch of --batch tokens (profiling runs)")
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--no-small", action="store_true",
                    help="skip the small-workload report (CQ 512x512, one Minueza Q4_0 layer)")
    ap.add_argument("--no-narrow", action="store_true",
                    help="skip the 1-bit / 2-bit / ternary decode report (cq_gemv vs cq_gemv_lut)")
    ap.add_argument("--mixed-only", action="store_true",
                    help="print only the mixed-width CQ report")
    ap.add_argument("--small-only", action="store_true",
                    help="print only the small-workload report (profiling runs)")
    ap.add_argument("--narrow-codes", nargs="*", default=None, choices=["b1", "b2", "ternary"],
                    help="restrict the narrow-code report to these codes (profiling runs)")
    ap.add_argument("--narrow-only", action="store_true",
                    help="print only that report (the child process the full run starts)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.cpu_baseline_only:
        print(json.dumps(cpu_baseline(args.cpu_rows)), flush=True)
    elif args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        gpu_arm(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
