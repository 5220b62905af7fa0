#!/usr/bin/env python
"""Benchmark: decode attention over the packed KV cache, and KV compression.

Default workload (w5 at batch 32 x context 65536, 2.1M cached tokens per layer):
Mistral-Nemo-12B-shaped KV cache, 40 layers x 8 KV heads x 128, 32 query heads,
keys 3-bit (symmetric grid) and values 3-bit (Gaussian Lloyd-Max), 128 fp16
sink tokens per sequence.  One step is one decode step of the whole model: the
query of every layer attends to its sinks and its packed tokens (prep, split-K
and combine kernels over all 40 layers, 70.3 GB of cache read per step, far
more than L2, so no flush is needed between steps).  Inputs are synthetic
(seeded N(0,1) with 4 outlier channels per head x10), compressed once by the
library and resident in HBM before timing.

`value` is decode-attention throughput in algorithmic GB/s (cache bytes read
plus q and output bytes, per step) over all ranks; `compress` reports KV
compression in Mtok/s (one token = K and V of all 8 heads of one layer);
`roofline` is the packed split-K kernel alone.  `also` holds the decode figures
of the other large workloads (unless --no-extra): w2 (Llama-3-8B shape, K8V3,
sinks and 64-token chunks), w3 at batch 8 (age tiers fp16 / K4V4 / K3V2 / K2V1
over 131072 positions, 1.05M tokens) and w4 at batch 32 (per-head widths 1-8
with QJL sketches, 1.05M tokens).

    python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--workload wN]

Other workloads (`--workload w1|w2|w3|w4|w5`, with `--batch`/`--context` for the
w5 sweep) make the main line instead.  Under torchrun each rank runs an
independent replica (weak scaling); the time is the max over ranks.
`--impl reference` times the CPU oracle instead on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rotated_quantized_kv_gb300 import workloads as W  # noqa: E402

METRIC = "decode-attn HBM GB/s (% of ~8 TB/s) over packed KV; KV compress Mtok/s"
NOMINAL_HBM_GBS = 8000.0
DECODE_SRCS = ("tq_decode_packed.cuh", "tq_decode_common.cuh", "tq_decode.cu", "tq_decode_geometry.h")


def measured_tensor_peak():
    """Dense fp16/bf16 tensor peak in TFLOP/s: the measured cuBLAS bf16 burst
    figure (fp16 runs at the same nominal rate), else the fallback."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        for k in ("bf16_tflops", "bf16_dense_tflops"):
            if k in d and d[k]:
                return float(d[k]), "measured"
    except (OSError, ValueError):
        pass
    return 1900.0, "fallback"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# --------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.path = None
        try:
            bus = torch.cuda.get_device_properties(device).pci_bus_id
            sel = ["-i", bus] if bus else []
        except Exception:
            sel = []
        self.sel = sel

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for ln in open(self.path):
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        except Exception:
            pass
        if self.path and os.path.exists(self.path):
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


def traffic_for(workload: str, packed_bytes: int, head_dim: int = 128):
    """DRAM bytes per launch of the packed kernel from an ncu capture taken on
    the current kernel sources (null otherwise): the captured bytes when the
    capture had this launch's size, else the captured traffic per algorithmic
    byte times this launch's algorithmic bytes (captures of the large
    workloads are taken at a smaller batch).  Captures at another head_dim
    carry a _d<head_dim> suffix."""
    suffix = "" if head_dim == 128 else f"_d{head_dim}"
    path = os.path.join(ROOT, "profiles", f"decode_packed_{workload}{suffix}_traffic.json")
    if not os.path.exists(path):
        return None
    t = json.load(open(path))
    if t.get("source_sha256") != kernel_sha():
        return None
    if t.get("algorithmic_bytes_per_launch") == packed_bytes and "traffic_bytes_per_launch" in t:
        return t["traffic_bytes_per_launch"]
    return int(round(t["traffic_ratio"] * packed_bytes)) if "traffic_ratio" in t else None


def kernel_sha() -> str:
    h = hashlib.sha256()
    for f in DECODE_SRCS:
        h.update(open(os.path.join(ROOT, "rotated_quantized_kv_gb300", "csrc", f), "rb").read())
    return h.hexdigest()


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time: every rank's timed region covers the same
    per-rank work, so the job finishes when the slowest replica does."""
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank: int, ms_max: float) -> float:
    """Weak scaling: all replicas' bytes over the slowest replica's time."""
    return world * bytes_per_rank / (ms_max * 1e-3) / 1e9


def timed_region(tq, step, nbytes, K, Wm, world, dev, sample_clocks=True):
    """Warm-up, then K timed steps between a barrier and a synchronize on both
    sides (the whole-job value).  Then K more steps with the packed split-K
    launches of each step bracketed by their own CUDA events on the launching
    stream (the dominant kernel's duration for the roofline): events between
    the call's kernels keep them from overlapping, so the value's steps run
    without them.  step(i) runs step i and returns its launches;
    nbytes(i) -> (packed, total)."""
    for s in range(Wm):
        step(s)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:  # torch creates the CUDA event at its first record; the library re-records it
        a.record()
        b.record()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches, total_bytes, packed_bytes = 0, 0, []
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(dev) as clk:
        torch.cuda.synchronize()
        start.record()
        for i in range(K):
            launches += step(Wm + i)
            total_bytes += nbytes(Wm + i)[1]
        stop.record()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        ms = start.elapsed_time(stop)
        # the dominant kernel alone, K further steps
        for i in range(K):
            s = Wm + K + i
            tq.tq_set_decode_kernel_events(*ev[i])
            step(s)
            packed_bytes.append(nbytes(s)[0])
        tq.tq_set_decode_kernel_events(None, None)
        torch.cuda.synchronize()
        # a short timed region sees few 200 ms clock samples: keep the same
        # steps running for ~1.5 s so the samples see the GPU under this load
        t_end = time.time() + (1.5 if sample_clocks else 0.0)
        s = Wm + 2 * K
        while time.time() < t_end:
            for _ in range(4):
                step(s)
                s += 1
            torch.cuda.synchronize()
    return {"ms": max_over_ranks(ms, world, "cuda"),
            "kern_ms": [a.elapsed_time(b) for a, b in ev], "launches": launches,
            "total_bytes": total_bytes, "packed_bytes": packed_bytes, "clocks": clk.summary()}


def time_compress(tq, jobs, reps=3):
    """Mean ms of one pass over `jobs` (callables that each launch one compress)."""
    for j in jobs:
        j()
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record()
    for _ in range(reps):
        for j in jobs:
            j()
    c1.record()
    torch.cuda.synchronize()
    return c0.elapsed_time(c1) / reps


def result_line(args, world, m, t, e2e, comp, config, workload):
    peak, peak_kind = measured_peaks()
    K = args.steps
    value = whole_job_gbs(world, t["total_bytes"], t["ms"])
    kern_avg_ms = float(np.mean(t["kern_ms"]))
    achieved = float(np.mean(t["packed_bytes"])) / (kern_avg_ms * 1e-3) / 1e9
    return {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(t["ms"] / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": config,
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "tokens_per_s": round(world * m.B * K / (t["ms"] * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": decode_kernel_name(m.d, m.Hq // m.H),
                     "achieved": round(achieved, 1),
                     "timing": "CUDA events around the packed launches of K further steps",
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic_for(workload, int(np.mean(t["packed_bytes"])), m.d),
                     "bytes_per_launch": int(np.mean(t["packed_bytes"])),
                     "avg_launch_ms": round(kern_avg_ms, 5)},
        "compress": {"value": round(comp["mtok"], 1), "unit": "Mtok/s", "ms_per_layer": round(comp["ms"], 4),
                     "tokens_per_layer": comp["tokens"],
                     "achieved_gbs": round(comp["bytes"] / (comp["ms"] * 1e-3) / 1e9, 1),
                     "frac_of_peak": round(comp["bytes"] / (comp["ms"] * 1e-3) / 1e9 / peak, 4),
                     **({"dense_rotation": comp["dense"]} if "dense" in comp else {})},
        "e2e": {"value": round(world * e2e["bytes"] / (e2e["ms"] * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": e2e["bi"], "d2h_bytes_per_step": e2e["bo"]},
        "gpu_launches": t["launches"],
        "clocks": t["clocks"],
    }


def run_w2(args, rank, world, tq):
    from rotated_quantized_kv_gb300.model_cache import ChunkedDecodeCache
    dev = torch.cuda.current_device()
    m = ChunkedDecodeCache()
    K, Wm = args.steps, args.warmup
    torch.cuda.synchronize()
    t = timed_region(tq, m.step, lambda s: (lambda pb, ob: (pb, pb + ob))(*m.step_bytes(s)), K, Wm, world, dev)

    # ---- e2e: each step's q and new-token K/V as one pinned host block (one
    # host-to-device copy), the output back to host (one copy)
    steps = m.steps_cap
    qh = m.qpool.cpu().reshape(steps, -1)
    # the new token's K and V of every layer, [steps][L][B][H][d] on the host
    newk = m.pool_k_all.permute(3, 0, 1, 2, 4).contiguous().cpu().reshape(steps, -1)
    newv = m.pool_v_all.permute(3, 0, 1, 2, 4).contiguous().cpu().reshape(steps, -1)
    nq, nk = qh.shape[1], newk.shape[1]
    blk_h = torch.cat([qh, newk, newv], dim=1).pin_memory()   # [steps][q | k | v] fp16
    blk_d = torch.empty(blk_h.shape[1], dtype=torch.float16, device="cuda")
    qdev = blk_d[:nq].view(m.q.shape)
    kstage = blk_d[nq:nq + nk].view(m.pool_k_all[:, :, :, 0].shape)
    vstage = blk_d[nq + nk:].view(m.pool_v_all[:, :, :, 0].shape)
    outh = torch.empty(m.out.shape, dtype=torch.float32).pin_memory()
    e2e = {"bi": blk_d.numel() * 2, "bo": m.out.numel() * 4, "bytes": 0}
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        s = (Wm + i) % m.steps_cap
        blk_d.copy_(blk_h[s], non_blocking=True)
        m.pool_k_all[:, :, :, s].copy_(kstage)
        m.pool_v_all[:, :, :, s].copy_(vstage)
        m.step(s, q=qdev)
        outh.copy_(m.out, non_blocking=True)
        pb, ob = m.step_bytes(s)
        e2e["bytes"] += pb + ob
    e1.record()
    torch.cuda.synchronize()
    e2e["ms"] = e0.elapsed_time(e1)

    # ---- compress throughput: re-compress every layer's prompt (one pass = 32 calls)
    nsrc = 8  # distinct inputs cycled: 8 x 66 MB, more than L2
    src = [W.kv_block(m.w, l, m.B, m.n_prompt_packed, 1002, device="cuda", token_offset=777)
           for l in range(nsrc)]
    scratch = [tq.PackedSegment(m.packed[l].layout) for l in range(nsrc)]
    jobs = [(lambda l=l: tq.tq_compress(scratch[l % nsrc], m.rots[l], *src[l % nsrc])) for l in range(m.L)]
    ms = time_compress(tq, jobs) / m.L
    tokens = m.n_prompt_packed * m.B
    comp = {"ms": ms, "tokens": tokens, "mtok": tokens / (ms * 1e-3) / 1e6,
            "bytes": tokens * m.H * (m.d * 2 * 2 + 16 * (m.w.kbits + m.w.vbits) + 8)}
    # ---- the same compression with a dense Haar rotation per layer (tensor cores)
    qd = [tq.tq_make_haar_rotation(m.d, 42 + l).cuda() for l in range(m.L)]
    drot = [tq.dense_rotation(m.rots[l], qd[l]) for l in range(m.L)]
    djobs = [(lambda l=l: tq.tq_compress(scratch[l % nsrc], drot[l], *src[l % nsrc])) for l in range(m.L)]
    tq.tq_compress_error_flag(reset=True)
    dms = time_compress(tq, djobs) / m.L
    assert tq.tq_compress_error_flag() == 0
    peak, _ = measured_peaks()
    tpeak, tkind = measured_tensor_peak()
    vec = tokens * m.H * 2                      # K and V vectors per layer
    dflops = vec * 2 * m.d * m.d                # y = Q x: 2 d^2 per vector (the kernel issues twice that: hi + lo)
    comp["dense"] = {"value": round(tokens / (dms * 1e-3) / 1e6, 1), "unit": "Mtok/s", "ms_per_layer": round(dms, 4),
                     "achieved_gbs": round(comp["bytes"] / (dms * 1e-3) / 1e9, 1),
                     "frac_of_peak": round(comp["bytes"] / (dms * 1e-3) / 1e9 / peak, 4),
                     "tensor_tflops": round(dflops / (dms * 1e-3) / 1e12, 1),
                     "tensor_issued_tflops": round(2 * dflops / (dms * 1e-3) / 1e12, 1),
                     "tensor_peak": tpeak, "tensor_peak_kind": tkind,
                     "tensor_frac_issued": round(2 * dflops / (dms * 1e-3) / 1e12 / tpeak, 4),
                     "rotation": "Haar (QR) per layer, fp16 hi + lo on tcgen05"}
    del qd, drot, djobs
    config = {"workload": m.w.name, "layers": m.L, "batch": m.B, "context": m.T, "kv_heads": m.H,
              "q_heads": m.Hq, "head_dim": m.d, "kbits": m.w.kbits, "vbits": m.w.vbits,
              "sinks": m.sinks, "chunk": m.chunk, "l2": "inputs larger than L2 (~0.8 GB read per step)",
              "parallelism": f"replicas x{world}"}
    return result_line(args, world, m, t, e2e, comp, config, "w2")


def run_static(args, rank, world, tq):
    from rotated_quantized_kv_gb300.model_cache import StaticCache
    dev = torch.cuda.current_device()
    w = W.WORKLOADS[args.workload]
    if args.head_dim:
        w = dataclasses.replace(w, head_dim=args.head_dim)
    seed = 1000 + int(args.workload[1:])
    m = StaticCache(w, batch=args.batch, context=args.context, seed=seed, rotation=args.rotation)
    K, Wm = args.steps, args.warmup
    nq = 4
    qpool = W.query_pool(w, nq, m.B, seed, device="cuda")
    pb, ob = m.step_bytes()
    torch.cuda.synchronize()

    def step(s):  # returns the kernel launches the library reports for the call
        m.decode(qpool[s % nq])
        return tq.tq_decode_last_launches()
    t = timed_region(tq, step, lambda s: (pb, pb + ob), K, Wm, world, dev)

    # ---- e2e: queries from pinned host memory, output back to host
    qh = qpool.cpu().pin_memory()
    outh = torch.empty(m.out.shape, dtype=torch.float32).pin_memory()
    qdev = torch.empty_like(qpool[0])
    e2e = {"bi": qdev.numel() * 2, "bo": m.out.numel() * 4, "bytes": 0}
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(K):
        qdev.copy_(qh[i % nq], non_blocking=True)
        m.decode(qdev)
        outh.copy_(m.out, non_blocking=True)
        e2e["bytes"] += pb + ob
    e1.record()
    torch.cuda.synchronize()
    e2e["ms"] = e0.elapsed_time(e1)

    # ---- compress throughput: each layer's packed segments from its fp16
    # prompt, cycling distinct layers' inputs until they exceed 4x L2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    layer_in = 2 * m.B * m.H * m.T * m.d * 2
    nsrc = max(1, min(m.L, -(-4 * l2 // layer_in)))
    if layer_in * nsrc > 24 * (1 << 30):
        nsrc = 1
    src = [W.kv_block(w, l, m.B, m.T, seed + 7, device="cuda") for l in range(nsrc)]
    scr, calls = {}, []
    for l in range(m.L):
        Kx, Vx = src[l % nsrc]
        for si in m.layers[l]:
            if not si.packed:
                continue
            # one scratch segment per distinct layout (the layer's own widths)
            lay = si.seg.layout
            key = (si.pos0, tuple(lay.kbits), tuple(lay.vbits), tuple(lay.qjl))
            if key not in scr:
                scr[key] = tq.PackedSegment(si.seg.layout)
            calls.append(lambda Kx=Kx, Vx=Vx, si=si, sg=scr[key], rot=m.rots[l]: tq.tq_compress(
                sg, rot, Kx[:, :, si.pos0:si.pos0 + si.n], Vx[:, :, si.pos0:si.pos0 + si.n],
                qjl_S=m.qjl_S if any(si.qjl) else None))
    ms = time_compress(tq, calls) / m.L
    tokens = m.packed_tokens() // m.L
    cbytes = sum(m.B * si.n * (m.H * m.d * 4 + si.bytes_per_token(m.d)) for si in m.layers[0] if si.packed)
    comp = {"ms": ms, "tokens": tokens, "mtok": tokens / (ms * 1e-3) / 1e6, "bytes": cbytes}
    del src, scr, calls
    rq = None
    if w.tiers:
        # tier demotion: every layer's K4V4 (warm) tier re-quantised to K3V2 (cold)
        warm = [[si for si in segs if si.packed and si.kbits[0] == 4][0] for segs in m.layers]
        n = warm[0].n
        dst = [tq.PackedSegment(tq.make_layout(m.B, m.H, m.d, warm[0].seg.layout.capacity, 3, 2))
               for _ in range(2)]
        rcalls = [(lambda l=l: tq.tq_requantize(warm[l].seg, 0, n, dst[l % 2], 0)) for l in range(m.L)]
        rms = time_compress(tq, rcalls) / m.L
        rbytes = m.B * m.H * n * ((16 * 8 + 8) + (16 * 5 + 8))
        peak, _ = measured_peaks()
        rq = {"from": "K4V4", "to": "K3V2", "tokens_per_layer": n * m.B, "ms_per_layer": round(rms, 4),
              "value": round(rbytes / (rms * 1e-3) / 1e9, 1), "unit": "GB/s",
              "frac_of_peak": round(rbytes / (rms * 1e-3) / 1e9 / peak, 4),
              "mtok_per_s": round(n * m.B / (rms * 1e-3) / 1e6, 1)}
        del dst, rcalls
    mass = None
    if w.tiers:
        # attention mass of every cached token (the demotion signal): the same
        # decode with a mass buffer on every segment; the difference is the
        # mass kernel (it runs after the merges)
        views, bufs = [], []
        for l, segs in enumerate(m.layers):
            for si in segs:
                si.seg.attn_mass = torch.empty(m.B, m.H, si.seg.layout.capacity, device="cuda")
                bufs.append(si.seg.attn_mass)
            views.append(tq.layer_view(m.rots[l], [si.seg for si in segs]))
            for si in segs:
                si.seg.attn_mass = None
        arr = tq.views_array(views)
        ws2 = torch.empty(tq.tq_decode_workspace_size(views, m.B, m.H, m.Hq, m.d), dtype=torch.uint8, device="cuda")
        out2 = torch.empty_like(m.out)
        call = (lambda s: tq.tq_decode_attention(None, qpool[s % nq], out2, ws2, m.H, qjl_S=m.qjl_S, views=arr))
        for s in range(3):
            call(s)
        torch.cuda.synchronize()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for s in range(K):
            call(s)
        a1.record()
        torch.cuda.synchronize()
        ms_mass = a0.elapsed_time(a1) / K
        ms_plain = t["ms"] / K
        # bytes the mass kernel reads and writes: key records + scales, fp16 keys, one float out
        mbytes = 0
        for segs in m.layers:
            for si in segs:
                if si.packed:  # key record + scale (+ QJL signs and norm) + the mass
                    mbytes += m.B * si.n * sum(16 * si.kbits[h] + 4 + (20 if si.qjl[h] else 0) + 4
                                               for h in range(m.H))
                else:  # fp16 key + the mass
                    mbytes += m.B * si.n * m.H * (2 * m.d + 4)
        peak, _ = measured_peaks()
        extra = ms_mass - ms_plain
        resolved = extra > 0.01 * ms_plain  # below 1% of the step the difference is timing noise
        mass = {"ms_per_step_with_mass": round(ms_mass, 4), "ms_per_step_without": round(ms_plain, 4),
                "extra_ms": round(extra, 4), "bytes": int(mbytes),
                "kernel_gbs_est": round(mbytes / (extra * 1e-3) / 1e9, 1) if resolved else None,
                "frac_of_peak_est": round(mbytes / (extra * 1e-3) / 1e9 / peak, 4) if resolved else None,
                "timing": "difference of two decode-call timings (CUDA events, K steps each)"}
        del views, bufs, arr, ws2, out2
    vq = None
    if w.qjl_max_bits and args.rotation == "srht":
        # QJL on values: the same cache with the key-sketched heads also sketching
        # their values; the decode call adds the correction pass
        m2 = StaticCache(w, batch=args.batch, context=args.context, seed=seed, value_qjl=True)
        for s in range(3):
            m2.decode(qpool[s % nq])
        torch.cuda.synchronize()
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        v0.record()
        for s in range(K):
            m2.decode(qpool[s % nq])
        v1.record()
        torch.cuda.synchronize()
        ms_v = v0.elapsed_time(v1) / K
        sk = sum(m2.B * si.n * 20 for segs in m2.layers for si in segs if si.packed for h in range(m2.H)
                 if si.qjl[h])
        vq = {"ms_per_step": round(ms_v, 4), "ms_per_step_without": round(t["ms"] / K, 4),
              "extra_ms": round(ms_v - t["ms"] / K, 4), "sketch_bytes": int(sk),
              "heads": "every head with a key sketch (widths <= 2) also sketches its values",
              "launches_per_step": tq.tq_decode_last_launches()}
        del m2
        torch.cuda.empty_cache()
    plan = [(si.pos0, si.n, sorted(set(zip(si.kbits, si.vbits, si.qjl)))) for si in m.layers[0]]
    config = {"workload": w.name, "layers": m.L, "batch": m.B, "context": m.T, "kv_heads": m.H,
              "q_heads": m.Hq, "head_dim": m.d,
              "segments_layer0": [{"pos0": p, "n": n, "k_v_qjl": [list(x) for x in kb]} for p, n, kb in plan],
              "rotation": args.rotation,
              "l2": f"inputs larger than L2 ({(pb + ob) / 1e9:.2f} GB read per step)",
              "parallelism": f"replicas x{world}"}
    res = result_line(args, world, m, t, e2e, comp, config, args.workload)
    if rq is not None:
        res["requantize"] = rq
    if mass is not None:
        res["attention_mass"] = mass
    if vq is not None:
        res["value_qjl"] = vq
    return res


def decode_kernel_name(d, gqa):
    """The split-K kernel runs head_dim 128, and 64 / 256 / 512 at GQA 1, 2 or 4
    (token pairs / 128-dim sub-records); other shapes run the generic kernel."""
    return "decode_packed_kernel" if d == 128 or (d in (64, 256, 512) and gqa in (1, 2, 4)) else "gen_decode_kernel"


# (workload, batch, context, head_dim): w2, the mixed-tier points of >= 1M cached
# tokens per layer, and the w5 shape at head_dim 256 and 64 (the other head dims' kernels)
EXTRA_POINTS = (("w2", None, None, None), ("w3", 8, None, None), ("w4", 32, None, None), ("w5", 8, 16384, 256),
                ("w5", 8, 16384, 64))


def decode_point(tq, name, batch, context, K, Wm, world, dev, head_dim=None):
    """Decode figures of one more workload (compact): whole-step GB/s over K
    steps and the split-K kernel alone (CUDA events on its stream)."""
    from rotated_quantized_kv_gb300.model_cache import ChunkedDecodeCache, StaticCache
    w = W.WORKLOADS[name]
    if head_dim:
        w = dataclasses.replace(w, head_dim=head_dim)
    if name == "w2":
        m = ChunkedDecodeCache()
        step = m.step
        nbytes = lambda s: (lambda pb, ob: (pb, pb + ob))(*m.step_bytes(s))  # noqa: E731
        B, T = m.B, m.T
    else:
        seed = 1000 + int(name[1:])
        m = StaticCache(w, batch=batch, context=context, seed=seed)
        qpool = W.query_pool(w, 4, m.B, seed, device="cuda")
        pb, ob = m.step_bytes()

        def step(s):
            m.decode(qpool[s % 4])
            return tq.tq_decode_last_launches()
        nbytes = lambda s: (pb, pb + ob)  # noqa: E731
        B, T = m.B, m.T
    torch.cuda.synchronize()
    t = timed_region(tq, step, nbytes, K, Wm, world, dev, sample_clocks=False)
    peak, peak_kind = measured_peaks()
    value = whole_job_gbs(world, t["total_bytes"], t["ms"])
    kern_ms = float(np.mean(t["kern_ms"]))
    achieved = float(np.mean(t["packed_bytes"])) / (kern_ms * 1e-3) / 1e9
    res = {"workload": w.name, "batch": B, "context": T, "tokens": B * T, "layers": w.layers, "head_dim": w.head_dim,
           "kernel": decode_kernel_name(w.head_dim, w.q_heads // w.kv_heads),
           "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(t["ms"] / K, 5),
           "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
           "kernel_gbs": round(achieved, 1), "kernel_frac": round(achieved / peak, 4), "peak": peak,
           "peak_kind": peak_kind, "kernel_ms": round(kern_ms, 5),
           "bytes_per_step": int(t["total_bytes"] / K), "gpu_launches": t["launches"]}
    if head_dim and head_dim != 128:
        # compression at this head_dim: every layer's packed prompt again, from
        # one fresh fp16 input per layer position
        src = W.kv_block(w, 0, m.B, m.T, 1007, device="cuda")
        calls, scr = [], {}
        for l in range(m.L):
            for si in m.layers[l]:
                if si.packed:
                    key = (tuple(si.seg.layout.kbits), tuple(si.seg.layout.vbits), si.pos0)
                    if key not in scr:
                        scr[key] = tq.PackedSegment(si.seg.layout)
                    calls.append(lambda si=si, sg=scr[key], rot=m.rots[l]: tq.tq_compress(
                        sg, rot, src[0][:, :, si.pos0:si.pos0 + si.n], src[1][:, :, si.pos0:si.pos0 + si.n]))
        cms = time_compress(tq, calls) / m.L
        ctok = sum(si.n for si in m.layers[0] if si.packed) * m.B
        cbytes = sum(m.B * si.n * (m.H * m.d * 4 + si.bytes_per_token(m.d)) for si in m.layers[0] if si.packed)
        res["compress"] = {"value": round(ctok / (cms * 1e-3) / 1e6, 1), "unit": "Mtok/s",
                           "ms_per_layer": round(cms, 4), "achieved_gbs": round(cbytes / (cms * 1e-3) / 1e9, 1),
                           "frac_of_peak": round(cbytes / (cms * 1e-3) / 1e9 / peak, 4),
                           "kernel": "compress_rows_kernel" if m.d in (64, 256, 512) else "gen_compress_kernel"}
        del src, calls, scr
    del m
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_ours(args, rank, world):
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq
    if args.workload == "w2":
        if args.rotation != "srht":
            raise SystemExit("--rotation haar applies to the static workloads (w1, w3, w5)")
        res = run_w2(args, rank, world, tq)
        wl = W.WORKLOADS["w2"]
    else:
        res = run_static(args, rank, world, tq)
        wl = W.WORKLOADS[args.workload]
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if (not args.no_extra and args.workload == "w5" and args.batch is None and args.context is None
            and args.head_dim is None):
        dev = torch.cuda.current_device()
        res["also"] = [decode_point(tq, n, b, c, args.steps, args.warmup, world, dev, head_dim=hd)
                       for n, b, c, hd in EXTRA_POINTS]
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(wl, seconds=args.cpu_seconds)
    return res


# --------------------------------------------------------------------- oracle arm
def oracle_plan(w, context):
    """Layer 0's segments as (pos0, n, kbits[H], vbits[H], qjl[H]), planned on
    the oracle side (its own tier ranges; the seeded bit-width draw)."""
    from oracle import oracle as O
    H = w.kv_heads
    if w.tiers:
        return [(s, e - s, [W.tier_bits(t)[0]] * H, [W.tier_bits(t)[1]] * H, [0] * H)
                for t, s, e in O.tier_ranges(context)]
    if w.per_head_bits:
        kb = [int(b) for b in W.draw_head_bits(w.layers, H)[0]]
        return [(0, context, kb, list(kb), [int(b <= w.qjl_max_bits) for b in kb])]
    out = [(0, w.sinks, [16] * H, [16] * H, [0] * H)] if w.sinks else []
    return out + [(w.sinks, context - w.sinks, [w.kbits] * H, [w.vbits] * H, [0] * H)]


def oracle_sample(w, budget_tokens=4096, seed=1002, layer=0):
    """A bounded sample of a workload for the CPU oracle: one layer (default 0),
    batch element 0, each segment of the layer's plan cut to its share of
    `budget_tokens` positions (fp16 segments of <= 128 positions kept whole).
    Returns (segments, sign, q, S, algorithmic bytes, description)."""
    from oracle import oracle as O
    H, d = w.kv_heads, w.head_dim
    plan = oracle_plan(w, w.context)
    total = sum(n for _, n, *_ in plan)
    cut = []
    for pos0, n, kb, vb, qj in plan:
        m = n if (kb[0] == 16 and n <= 128) else max(16, min(n, round(n * budget_tokens / total)))
        cut.append((pos0, m, kb, vb, qj))
    span = max(p + m for p, m, *_ in cut)
    K, V = W.kv_block(w, layer, 1, span, seed)
    sign = O.signs(d, W.ROTATION_SEED + layer)
    S = O.qjl_matrix(128, d, W.QJL_SEED) if w.qjl_max_bits else None
    segs, nbytes = [], w.q_heads * d * 6
    for pos0, m, kb, vb, qj in cut:
        if kb[0] == 16:
            sg = O.Fp16Segment(1, H, d, m, n_tokens=m)
            sg.k16[:] = K[:, :, pos0:pos0 + m].numpy().view(np.uint16).ravel()
            sg.v16[:] = V[:, :, pos0:pos0 + m].numpy().view(np.uint16).ravel()
            nbytes += m * H * d * 4
        else:
            sg = O.PackedSegment(1, H, d, ((m + 15) // 16) * 16, kb, vb, qj)
            O.compress(sg, K[:, :, pos0:pos0 + m].numpy().view(np.uint16),
                       V[:, :, pos0:pos0 + m].numpy().view(np.uint16), sign, S)
            sg.n_tokens = m
            nbytes += m * sum(d // 8 * (a + b) + 8 + (20 if q else 0) for a, b, q in zip(kb, vb, qj))
        segs.append(sg)
    q = W.queries(w, layer, 1, seed).numpy()
    desc = (f"{w.name} layer {layer}, batch element 0: " +
            " + ".join(f"{m} {'fp16' if kb[0] == 16 else 'packed'}" for _, m, kb, _, _ in cut) +
            f" tokens, {w.q_heads} query heads")
    return segs, sign, q, S, nbytes, desc


def cpu_baseline(w, seconds=10.0):
    """The oracle as it stands, timed on the host cores: one thread on one
    layer's sample, then one thread per allowed core, each on its own layer's
    sample (the oracle's C call releases the GIL, so the threads run in
    parallel over independent (layer) units).  The all-core figure is the
    line's value; the single-thread one is kept beside it."""
    import concurrent.futures as cf
    from oracle import oracle as O
    segs, sign, q, S, nbytes, desc = oracle_sample(w)
    reps, t = 0, 0.0
    while t < seconds / 2 or reps == 0:
        t0 = time.perf_counter()
        O.decode_attention(segs, q, sign, w.kv_heads, S=S)
        t += time.perf_counter() - t0
        reps += 1
    single = reps * nbytes / t / 1e9
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    samples = [(segs, sign, q, S, nbytes)] + [oracle_sample(w, layer=l % w.layers)[:5] for l in range(1, cores)]
    done = [0] * cores
    t_stop = [0.0]

    def worker(i):
        sg, sn, qq, SS, _ = samples[i]
        while True:
            O.decode_attention(sg, qq, sn, w.kv_heads, S=SS)
            done[i] += 1
            if time.perf_counter() >= t_stop[0]:
                return

    t0 = time.perf_counter()
    t_stop[0] = t0 + seconds / 2
    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(worker, range(cores)))
    dt = time.perf_counter() - t0
    allb = sum(done[i] * samples[i][4] for i in range(cores))
    return {"value": round(allb / dt / 1e9, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "single_thread": {"value": round(single, 6), "unit": "GB/s", "cores": 1, "repetitions": reps,
                              "seconds": round(t, 2)},
            "sample": f"{desc}; all-core run: {cores} threads, thread i on layer i's sample of the same "
                      f"shape, {sum(done)} calls in {dt:.1f} s; single thread: {reps} calls in {t:.1f} s "
                      f"(plain scalar C)"}


def run_reference(args, rank, world):
    """The oracle as it stands on the host cores: one thread per allowed core,
    thread i on layer i's bounded sample; a step is one call on every thread."""
    if rank != 0:
        return None
    import concurrent.futures as cf
    from oracle import oracle as O
    w = W.WORKLOADS[args.workload]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    samples = [oracle_sample(w, budget_tokens=1024, layer=l % w.layers) for l in range(cores)]
    desc = samples[0][5]
    nbytes = sum(smp[4] for smp in samples)

    def one(i):
        sg, sn, qq, SS = samples[i][:4]
        O.decode_attention(sg, qq, sn, w.kv_heads, S=SS)

    with cf.ThreadPoolExecutor(max_workers=cores) as ex:
        for _ in range(args.warmup):
            list(ex.map(one, range(cores)))
        t0 = time.perf_counter()
        for _ in range(args.steps):
            list(ex.map(one, range(cores)))
        dt = time.perf_counter() - t0
    v = args.steps * nbytes / dt / 1e9
    desc += f" (CPU oracle, {cores} threads, thread i on layer i's sample of the same shape)"
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "layers": w.layers, "batch": w.batch, "context": w.context,
                       "kv_heads": w.kv_heads, "q_heads": w.q_heads, "head_dim": w.head_dim, "kbits": w.kbits,
                       "vbits": w.vbits, "sinks": w.sinks, "chunk": w.chunk, "sample": desc},
            "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="w5", choices=sorted(W.WORKLOADS),
                    help="w5 (default, batch 32 x 65536): the largest single-GPU workload; "
                         "w2: chunked decode with sinks; w1, w3, w4: decode steps over a prompt "
                         "compressed once")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decode figures of w2, w3 (batch 8) and w4 (batch 32)")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (w1, w3-w5)")
    ap.add_argument("--rotation", default="srht", choices=["srht", "haar"],
                    help="haar: a dense Haar rotation per layer (tensor-core compressor; w1, w3, w5)")
    ap.add_argument("--context", type=int, default=None, help="override the workload's context (w1, w3-w5)")
    ap.add_argument("--head-dim", type=int, default=None,
                    help="override the workload's head_dim (w1, w3-w5; a power of two 16..1024)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl")
    res = run_ours(args, rank, world)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
