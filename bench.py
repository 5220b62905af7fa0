#!/usr/bin/env python
"""Benchmark: decode attention over the packed KV cache, and KV compression.

Default workload (w2): Llama-3-8B-shaped KV cache, 32 layers x 8 KV heads x 128,
32 query heads, batch 1, context 16384; keys 8-bit, values 3-bit; 128 fp16 sink
tokens; new tokens buffered in fp16 and compressed 64 at a time.  One step is
one decode step of the whole model: the query of every layer attends to its
sinks, its packed tokens and its fp16 buffer (prep, split-K and combine kernels
over all 32 layers), and every 64th step the 64 buffered tokens of each layer
are compressed into the packed segment.  Inputs are synthetic (seeded N(0,1)
with per-channel log-normal scales), resident in HBM before timing; each step
reads ~0.8 GB, more than L2, so no flush is needed between steps.

`value` is decode-attention throughput in algorithmic GB/s (cache bytes read
plus q and output bytes, per step) over all ranks; `compress` reports KV
compression in Mtok/s (one token = K and V of all 8 heads of one layer).

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun each rank runs an independent replica (weak scaling); the time
is the max over ranks.  `--impl reference` times the CPU oracle instead on a
bounded sample of the same workload (rank 0 only).
"""
from __future__ import annotations

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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rotated_quantized_kv_gb300 import workloads as W  # noqa: E402

METRIC = json.load(open(os.path.join(ROOT, "BASELINE.json")))["metric"] if os.path.exists(
    os.path.join(ROOT, "BASELINE.json")) else "decode-attn HBM GB/s over packed KV; KV compress Mtok/s"
NOMINAL_HBM_GBS = 8000.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_packed_w2_traffic.json")
DECODE_SRC = os.path.join(ROOT, "rotated_quantized_kv_gb300", "csrc", "tq_decode.cu")


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


# --------------------------------------------------------------------- w2 model
class W2:
    """The w2 cache on one GPU: per layer an fp16 sink segment, a packed segment
    (capacity for the prompt plus the decode steps) and an fp16 buffer segment
    that views a pool of the decode tokens."""

    def __init__(self, tq, steps_cap=256, device="cuda", seed=1002):
        self.tq = tq
        w = self.w = W.WORKLOADS["w2"]
        self.L, self.B, self.H, self.Hq, self.d = w.layers, w.batch, w.kv_heads, w.q_heads, w.head_dim
        self.T, self.sinks, self.chunk = w.context, w.sinks, w.chunk
        self.steps_cap = steps_cap
        self.n_prompt_packed = self.T - self.sinks
        cap = ((self.n_prompt_packed + steps_cap + 15) // 16) * 16
        self.rots, self.sink, self.packed = [], [], []
        # decode tokens of every layer: [L][B][H][steps][d], one tensor so that a
        # step's new token of all layers is one strided slice
        self.pool_k_all = torch.empty(self.L, self.B, self.H, steps_cap, self.d, dtype=torch.float16, device=device)
        self.pool_v_all = torch.empty_like(self.pool_k_all)
        for l in range(self.L):
            rot = tq.tq_make_rotation(self.d, W.ROTATION_SEED + l)
            K, V = W.kv_block(w, l, self.B, self.T, seed, device=device)
            s = tq.Fp16Segment(self.B, self.H, self.d, self.sinks, n_tokens=self.sinks,
                               k=K[:, :, :self.sinks].contiguous(), v=V[:, :, :self.sinks].contiguous())
            p = tq.PackedSegment(tq.make_layout(self.B, self.H, self.d, cap, w.kbits, w.vbits))
            tq.tq_compress(p, rot, K[:, :, self.sinks:], V[:, :, self.sinks:], t_begin=0)
            p.n_tokens = self.n_prompt_packed
            pk, pv = W.kv_block(w, l, self.B, steps_cap, seed, device=device, token_offset=self.T)
            self.pool_k_all[l].copy_(pk)
            self.pool_v_all[l].copy_(pv)
            self.rots.append(rot)
            self.sink.append(s)
            self.packed.append(p)
            del K, V, pk, pv
        self.pool_k = [self.pool_k_all[l] for l in range(self.L)]
        self.pool_v = [self.pool_v_all[l] for l in range(self.L)]
        self.qpool = W.query_pool(w, steps_cap, self.B, seed, device=device)  # [steps][L][B][Hq][d]
        self.q = self.qpool[0]
        self.buf = [tq.Fp16Segment(self.B, self.H, self.d, steps_cap, n_tokens=1, k=self.pool_k[l],
                                   v=self.pool_v[l]) for l in range(self.L)]
        self.views = [tq.layer_view(self.rots[l], [self.sink[l], self.packed[l], self.buf[l]])
                      for l in range(self.L)]
        self.arr = tq.views_array(self.views)
        self.out = torch.empty(self.L, self.B, self.Hq, self.d, device=device)
        self.ws = torch.empty(self.max_workspace(), dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

    def max_workspace(self):
        best = 0
        for s in (0, self.steps_cap - 1):
            self.set_step(s)
            best = max(best, self.tq.tq_decode_workspace_size(list(self.arr), self.B, self.H, self.Hq, self.d))
        return best + (1 << 20)

    def set_step(self, s):
        """Point the segment views at decode step s (0-based within the pool)."""
        s %= self.steps_cap
        w0 = (s // self.chunk) * self.chunk
        esz = self.pool_k[0].element_size()
        for l in range(self.L):
            seg = self.arr[l].seg
            seg[1].n_tokens = self.n_prompt_packed + w0
            seg[2].n_tokens = s - w0 + 1
            seg[2].k16 = self.pool_k[l].data_ptr() + w0 * self.d * esz
            seg[2].v16 = self.pool_v[l].data_ptr() + w0 * self.d * esz
        return w0

    def compress_window(self, s):
        """At the first step of a new 64-token window, compress the previous one."""
        s %= self.steps_cap
        if s == 0 or s % self.chunk:
            return 0
        w0 = s - self.chunk
        for l in range(self.L):
            self.tq.tq_compress(self.packed[l], self.rots[l], self.pool_k[l][:, :, w0:s],
                                self.pool_v[l][:, :, w0:s], t_begin=self.n_prompt_packed + w0)
        return self.L

    def step(self, s, q=None):
        launches = self.compress_window(s)
        self.set_step(s)
        qq = self.qpool[s % self.steps_cap] if q is None else q
        self.tq.tq_decode_attention(None, qq, self.out, self.ws, self.H, views=self.arr)
        return launches + 2  # split-K over fp16 segments, split-K over packed segments

    def step_bytes(self, s):
        s %= self.steps_cap
        w0 = (s // self.chunk) * self.chunk
        per_tok_packed = self.H * (16 * (self.w.kbits + self.w.vbits) + 8)
        per_tok_fp16 = self.H * self.d * 2 * 2
        packed = self.L * (self.n_prompt_packed + w0) * per_tok_packed * self.B
        fp16 = self.L * (self.sinks + s - w0 + 1) * per_tok_fp16 * self.B
        qo = self.L * self.B * self.Hq * self.d * (2 + 4)
        return packed, fp16 + qo


def run_ours(args, rank, world):
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq
    dev = torch.cuda.current_device()
    m = W2(tq)
    K, Wm = args.steps, args.warmup
    for s in range(Wm):
        m.step(s)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev:  # torch creates the CUDA event at its first record; the library re-records it
        a.record()
        b.record()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    total_bytes = 0
    packed_bytes = []
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(dev) as clk:
        torch.cuda.synchronize()
        start.record()
        for i in range(K):
            s = Wm + i
            tq.tq_set_decode_kernel_events(*ev[i])
            launches += m.step(s)
            pb, ob = m.step_bytes(s)
            packed_bytes.append(pb)
            total_bytes += pb + ob
        stop.record()
        tq.tq_set_decode_kernel_events(None, None)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        # the timed region lasts milliseconds, shorter than the 200 ms sampling
        # period: keep the same steps running for ~1.5 s so the clock samples
        # see the GPU under this load
        t_end = time.time() + 1.5
        s = Wm + K
        while time.time() < t_end:
            for _ in range(20):
                m.step(s)
                s += 1
            torch.cuda.synchronize()
    ms = start.elapsed_time(stop)
    ms_all = torch.tensor([ms], device="cuda")
    if world > 1:
        torch.distributed.all_reduce(ms_all, op=torch.distributed.ReduceOp.MAX)
    ms_max = float(ms_all.item())
    kern_ms = [a.elapsed_time(b) for a, b in ev]
    clocks = clk.summary()

    # ---- e2e: q and the new token's K/V from pinned host memory, output back to host
    qh = m.qpool.cpu().pin_memory()
    # the new token's K and V of every layer, [steps][L][B][H][d] on the host
    newk = m.pool_k_all.permute(3, 0, 1, 2, 4).contiguous().cpu().pin_memory()
    newv = m.pool_v_all.permute(3, 0, 1, 2, 4).contiguous().cpu().pin_memory()
    kstage = torch.empty(newk.shape[1:], dtype=torch.float16, device="cuda")
    vstage = torch.empty_like(kstage)
    outh = torch.empty(m.out.shape, dtype=torch.float32).pin_memory()
    qdev = torch.empty_like(m.q)
    bi = m.q.numel() * 2 + kstage.numel() * 2 * 2
    bo = m.out.numel() * 4
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_bytes = 0
    e0.record()
    for i in range(K):
        s = (Wm + i) % m.steps_cap
        qdev.copy_(qh[s], non_blocking=True)
        kstage.copy_(newk[s], non_blocking=True)
        vstage.copy_(newv[s], non_blocking=True)
        m.pool_k_all[:, :, :, s].copy_(kstage)
        m.pool_v_all[:, :, :, s].copy_(vstage)
        m.step(s, q=qdev)
        outh.copy_(m.out, non_blocking=True)
        pb, ob = m.step_bytes(s)
        e2e_bytes += pb + ob
    e1.record()
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)

    # ---- compress throughput: re-compress every layer's prompt (one step = 32 calls)
    comp_tokens = m.n_prompt_packed * m.L * m.B
    nsrc = 8  # distinct inputs cycled: 8 x 66 MB, more than L2
    src = [W.kv_block(m.w, l, m.B, m.n_prompt_packed, 1002, device="cuda", token_offset=777)
           for l in range(nsrc)]
    scratch = [tq.PackedSegment(m.packed[l].layout) for l in range(nsrc)]
    for l in range(m.L):  # warm-up
        tq.tq_compress(scratch[l % nsrc], m.rots[l], *src[l % nsrc])
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    creps = 3
    c0.record()
    for _ in range(creps):
        for l in range(m.L):
            tq.tq_compress(scratch[l % nsrc], m.rots[l], *src[l % nsrc])
    c1.record()
    torch.cuda.synchronize()
    cms = c0.elapsed_time(c1) / creps
    c_mtok = comp_tokens / (cms * 1e-3) / 1e6
    c_bytes = comp_tokens * m.H * (m.d * 2 * 2 + 16 * (m.w.kbits + m.w.vbits) + 8)
    peak, peak_kind = measured_peaks()

    value = world * total_bytes / (ms_max * 1e-3) / 1e9
    kern_avg_ms = float(np.mean(kern_ms))
    achieved = float(np.mean(packed_bytes)) / (kern_avg_ms * 1e-3) / 1e9
    traffic = None
    if os.path.exists(TRAFFIC_FILE):
        t = json.load(open(TRAFFIC_FILE))
        h = hashlib.sha256(open(DECODE_SRC, "rb").read()).hexdigest()
        if t.get("source_sha256") == h:
            traffic = t.get("traffic_bytes_per_launch")
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": Wm,
        "ms_per_step": round(ms_max / K, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": m.w.name, "layers": m.L, "batch": m.B, "context": m.T, "kv_heads": m.H,
                   "q_heads": m.Hq, "head_dim": m.d, "kbits": m.w.kbits, "vbits": m.w.vbits,
                   "sinks": m.sinks, "chunk": m.chunk, "l2": "inputs larger than L2 (~0.8 GB read per step)",
                   "parallelism": f"replicas x{world}"},
        "pct_of_nominal_8tbs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "tokens_per_s": round(world * m.B * K / (ms_max * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": "decode_packed_kernel", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": traffic, "bytes_per_launch": int(np.mean(packed_bytes)),
                     "avg_launch_ms": round(kern_avg_ms, 5)},
        "compress": {"value": round(c_mtok, 1), "unit": "Mtok/s", "ms_per_model": round(cms, 4),
                     "achieved_gbs": round(c_bytes / (cms * 1e-3) / 1e9, 1),
                     "frac_of_peak": round(c_bytes / (cms * 1e-3) / 1e9 / peak, 4)},
        "e2e": {"value": round(world * e2e_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(seconds=args.cpu_seconds)
    return result


# --------------------------------------------------------------------- oracle arm
def oracle_sample(layers=1, packed_tokens=4096, seed=1002):
    """A bounded sample of w2 for the CPU oracle: `layers` layers with the 128
    sinks, the first `packed_tokens` packed tokens and a 1-token buffer.
    Returns (list of (segments, sign), queries, algorithmic bytes)."""
    from oracle import oracle as O
    w = W.WORKLOADS["w2"]
    H, d = w.kv_heads, w.head_dim
    out, nbytes = [], 0
    for l in range(layers):
        K, V = W.kv_block(w, l, 1, w.sinks + packed_tokens, seed)
        sign = O.signs(d, W.ROTATION_SEED + l)
        sink = O.Fp16Segment(1, H, d, w.sinks, n_tokens=w.sinks)
        sink.k16[:] = K[:, :, :w.sinks].numpy().view(np.uint16).ravel()
        sink.v16[:] = V[:, :, :w.sinks].numpy().view(np.uint16).ravel()
        cap = ((packed_tokens + 15) // 16) * 16
        seg = O.PackedSegment(1, H, d, cap, [w.kbits] * H, [w.vbits] * H)
        O.compress(seg, K[:, :, w.sinks:].numpy().view(np.uint16), V[:, :, w.sinks:].numpy().view(np.uint16),
                   sign)
        q = W.queries(w, l, 1, seed).numpy()
        out.append(([sink, seg], sign, q))
        nbytes += packed_tokens * H * (16 * (w.kbits + w.vbits) + 8) + w.sinks * H * d * 4 + w.q_heads * d * 6
    return out, nbytes


def cpu_baseline(seconds=10.0):
    from oracle import oracle as O
    sample, nbytes = oracle_sample(layers=1, packed_tokens=4096)
    reps, t = 0, 0.0
    while t < seconds or reps == 0:
        t0 = time.perf_counter()
        for segs, sign, q in sample:
            O.decode_attention(segs, q, sign, W.KV_HEADS)
        t += time.perf_counter() - t0
        reps += 1
    return {"value": round(reps * nbytes / t / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"w2 layer 0: 128 fp16 sinks + 4096 packed K8/V3 tokens, 32 query heads; "
                      f"{reps} repetitions, {t:.1f} s of single-threaded C"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from oracle import oracle as O
    sample, nbytes = oracle_sample(layers=1, packed_tokens=1024)
    for _ in range(args.warmup):
        for segs, sign, q in sample:
            O.decode_attention(segs, q, sign, W.KV_HEADS)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        for segs, sign, q in sample:
            O.decode_attention(segs, q, sign, W.KV_HEADS)
    dt = time.perf_counter() - t0
    v = args.steps * nbytes / dt / 1e9
    w = W.WORKLOADS["w2"]
    desc = "w2 layer 0: 128 fp16 sinks + 1024 packed K8/V3 tokens, 32 query heads (CPU oracle, 1 thread)"
    return {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "layers": w.layers, "batch": w.batch, "context": w.context,
                       "kv_heads": w.kv_heads, "q_heads": w.q_heads, "head_dim": w.head_dim, "kbits": w.kbits,
                       "vbits": w.vbits, "sinks": w.sinks, "chunk": w.chunk, "sample": desc},
            "cpu_baseline": {"value": round(v, 6), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": desc},
            "e2e": {"value": round(v, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
