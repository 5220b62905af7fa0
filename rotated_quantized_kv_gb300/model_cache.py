"""Whole-model KV caches on one GPU in the segment layouts of the five workloads.

Host orchestration only: every byte of a cache is written by the library's
compress kernel (tq_compress) or copied verbatim (fp16 segments), and decode
runs through tq_decode_attention.  The segment plans follow the pages:

  sinks     the first 128 positions stay fp16 ("turboquant-mlx", "FP16
            Attention Sinks").
  tiers     by token age: < 1K fp16, 1K-8K K4V4, 8K-64K K3V2, >= 64K K2V1
            ("TurboMOQ", "Progressive temporal tiering").
  chunking  decode tokens are buffered in fp16 and compressed 64 at a time
            ("turboquant-mlx", "Dynamic Chunk Buffering").

`StaticCache` builds workloads 1, 3, 4 and 5 (a prompt compressed once, then
decode steps against it); `ChunkedDecodeCache` builds workload 2 (sinks, a
packed prompt, and an fp16 buffer of decode tokens that is compressed every
64 steps).  Both expose `views` (ctypes layer views), `decode(q)` and the
algorithmic bytes a decode step reads.
"""
from __future__ import annotations

from dataclasses import dataclass

import ctypes

import numpy as np
import torch

from . import tq as T
from . import workloads as W

AGE_BOUNDS = (1024, 8192, 65536)


def _cap16(n: int) -> int:
    return max(16, ((n + 15) // 16) * 16)


@dataclass
class SegInfo:
    """One segment of a layer: its library object, first position, token count
    and per-head widths (16 = fp16)."""
    seg: object
    pos0: int
    n: int
    kbits: list
    vbits: list
    qjl: list

    @property
    def packed(self) -> bool:
        return self.kbits[0] != 16

    def bytes_per_token(self, d: int) -> int:
        """Algorithmic bytes of one position over all heads (records + scales
        [+ QJL signs and norm]); fp16: K and V verbatim."""
        if not self.packed:
            return len(self.kbits) * d * 4
        return sum(d // 8 * (kb + vb) + 8 + (20 if q else 0)
                   for kb, vb, q in zip(self.kbits, self.vbits, self.qjl))


def plan_segments(w: W.Workload, context: int, layer: int):
    """(pos0, n, kbits[H], vbits[H], qjl[H]) of one layer's segments, in position order."""
    H = w.kv_heads
    if w.tiers:
        out = []
        tiers = T.tq_age_tiers(context, list(AGE_BOUNDS))
        for tier in range(len(tiers) - 1, -1, -1):  # oldest positions first
            s, e = tiers[tier]
            if e > s:
                kb, vb = W.tier_bits(tier)
                out.append((s, e - s, [kb] * H, [vb] * H, [0] * H))
        return out
    if w.per_head_bits:
        bits = W.draw_head_bits(w.layers, H)[layer]
        kb = [int(b) for b in bits]
        qj = [int(b <= w.qjl_max_bits) for b in bits]
        return [(0, context, kb, list(kb), qj)]
    out = []
    if w.sinks:
        out.append((0, w.sinks, [16] * H, [16] * H, [0] * H))
    out.append((w.sinks, context - w.sinks, [w.kbits] * H, [w.vbits] * H, [0] * H))
    return out


class StaticCache:
    """A prompt of `context` positions compressed once per layer (workloads 1, 3, 4, 5)."""

    def __init__(self, w: W.Workload, batch: int | None = None, context: int | None = None, seed: int = 1000,
                 device="cuda", sample_inputs=None, rotation: str = "srht", value_qjl: bool = False):
        """sample_inputs(layer, K, V), if given, sees each layer's fp16 inputs
        ([B][H][T][d] CUDA tensors) before they are dropped.  rotation: "srht"
        (D H D / sqrt(d)) or "haar" (a dense Haar matrix per layer, seed + l;
        no QJL heads).  value_qjl: the heads with a key sketch also sketch
        their value residuals."""
        assert rotation in ("srht", "haar")
        if rotation == "haar" and w.qjl_max_bits:
            raise ValueError("the dense-rotation compressor takes no QJL heads")
        self.w = w
        self.L, self.H, self.Hq, self.d = w.layers, w.kv_heads, w.q_heads, w.head_dim
        self.B = batch or w.batch
        self.T = context or w.context
        self.seed = seed
        self.qjl_S = T.tq_make_qjl(self.d, 128, W.QJL_SEED).to(device) if w.qjl_max_bits else None
        self.rots, self.layers, self.views, self.dense_q = [], [], [], []
        for l in range(self.L):
            rot = T.tq_make_rotation(self.d, W.ROTATION_SEED + l)
            if rotation == "haar":
                self.dense_q.append(T.tq_make_haar_rotation(self.d, W.ROTATION_SEED + l).to(device))
                rot = T.dense_rotation(rot, self.dense_q[-1])
            K, V = W.kv_block(w, l, self.B, self.T, seed, device=device)
            segs = []
            for pos0, n, kb, vb, qj in plan_segments(w, self.T, l):
                if kb[0] == 16:
                    s = T.Fp16Segment(self.B, self.H, self.d, n, n_tokens=n,
                                      k=K[:, :, pos0:pos0 + n].contiguous(), v=V[:, :, pos0:pos0 + n].contiguous())
                else:
                    s = T.PackedSegment(T.make_layout(self.B, self.H, self.d, _cap16(n), kb, vb, qj,
                                                      qjl_v=qj if value_qjl else None), device=device)
                    T.tq_compress(s, rot, K[:, :, pos0:pos0 + n], V[:, :, pos0:pos0 + n], t_begin=0,
                                  qjl_S=self.qjl_S if any(qj) else None)
                segs.append(SegInfo(s, pos0, n, kb, vb, qj))
            if sample_inputs is not None:
                sample_inputs(l, K, V)
            del K, V
            self.rots.append(rot)
            self.layers.append(segs)
            self.views.append(T.layer_view(rot, [si.seg for si in segs]))
        self.arr = T.views_array(self.views)
        self.out = torch.empty(self.L, self.B, self.Hq, self.d, device=device)
        self.ws = torch.empty(T.tq_decode_workspace_size(self.views, self.B, self.H, self.Hq, self.d),
                              dtype=torch.uint8, device=device)

    def decode(self, q: torch.Tensor, out: torch.Tensor | None = None):
        """One decode step of every layer: q fp16 [L][B][Hq][d] -> out fp32 [L][B][Hq][d]."""
        o = self.out if out is None else out
        T.tq_decode_attention(None, q, o, self.ws, self.H, qjl_S=self.qjl_S, views=self.arr)
        return o

    def step_bytes(self):
        """(packed-segment bytes, other bytes) read or written by one decode step."""
        packed = other = 0
        for segs in self.layers:
            for si in segs:
                b = self.B * si.n * si.bytes_per_token(self.d)
                if si.packed:
                    packed += b
                else:
                    other += b
        other += self.L * self.B * self.Hq * self.d * (2 + 4)
        return packed, other

    def packed_tokens(self) -> int:
        return sum(si.n for segs in self.layers for si in segs if si.packed) * self.B


class ChunkedDecodeCache:
    """Workload 2 on one GPU: per layer an fp16 sink segment, a packed segment
    (capacity for the prompt plus the decode steps) and an fp16 buffer segment
    that views a pool of the decode tokens; every 64th step compresses the
    previous 64 buffered tokens of each layer into the packed segment."""

    def __init__(self, w: W.Workload | None = None, steps_cap=256, device="cuda", seed=1002):
        w = self.w = w or W.WORKLOADS["w2"]
        self.L, self.B, self.H, self.Hq, self.d = w.layers, w.batch, w.kv_heads, w.q_heads, w.head_dim
        self.T, self.sinks, self.chunk = w.context, w.sinks, w.chunk
        self.steps_cap = steps_cap
        self.n_prompt_packed = self.T - self.sinks
        cap = _cap16(self.n_prompt_packed + steps_cap)
        self.rots, self.sink, self.packed = [], [], []
        # decode tokens of every layer: [L][B][H][steps][d], one tensor so that a
        # step's new token of all layers is one strided slice
        self.pool_k_all = torch.empty(self.L, self.B, self.H, steps_cap, self.d, dtype=torch.float16, device=device)
        self.pool_v_all = torch.empty_like(self.pool_k_all)
        for l in range(self.L):
            rot = T.tq_make_rotation(self.d, W.ROTATION_SEED + l)
            K, V = W.kv_block(w, l, self.B, self.T, seed, device=device)
            s = T.Fp16Segment(self.B, self.H, self.d, self.sinks, n_tokens=self.sinks,
                              k=K[:, :, :self.sinks].contiguous(), v=V[:, :, :self.sinks].contiguous())
            p = T.PackedSegment(T.make_layout(self.B, self.H, self.d, cap, w.kbits, w.vbits))
            T.tq_compress(p, rot, K[:, :, self.sinks:], V[:, :, self.sinks:], t_begin=0)
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
        self.buf = [T.Fp16Segment(self.B, self.H, self.d, steps_cap, n_tokens=1, k=self.pool_k[l],
                                  v=self.pool_v[l]) for l in range(self.L)]
        self.views = [T.layer_view(self.rots[l], [self.sink[l], self.packed[l], self.buf[l]])
                      for l in range(self.L)]
        self.arr = T.views_array(self.views)
        self._bind_step_fields()
        self.out = torch.empty(self.L, self.B, self.Hq, self.d, device=device)
        self.ws = torch.empty(self.max_workspace(), dtype=torch.uint8, device=device)

    def _bind_step_fields(self):
        """numpy views of the four per-step fields of every layer's view (packed
        n_tokens, buffer n_tokens, buffer K and V pointers) inside the ctypes
        array, so that a step updates all layers with four array stores."""
        lv, sg = T.tq_layer_view, T.tq_segment
        base = ctypes.addressof(self.arr)
        raw = (ctypes.c_char * (ctypes.sizeof(lv) * self.L)).from_address(base)

        def field(seg_i, fld, dtype):
            off = lv.seg.offset + seg_i * ctypes.sizeof(sg) + getattr(sg, fld).offset
            return np.ndarray((self.L,), dtype=dtype, buffer=raw, offset=off, strides=(ctypes.sizeof(lv),))
        self._n_packed = field(1, "n_tokens", np.int32)
        self._n_buf = field(2, "n_tokens", np.int32)
        self._k_buf = field(2, "k16", np.uint64)
        self._v_buf = field(2, "v16", np.uint64)
        self._k_base = np.array([self.pool_k[l].data_ptr() for l in range(self.L)], np.uint64)
        self._v_base = np.array([self.pool_v[l].data_ptr() for l in range(self.L)], np.uint64)
        self._tok_bytes = self.d * self.pool_k[0].element_size()

    def max_workspace(self):
        best = 0
        for s in (0, self.steps_cap - 1):
            self.set_step(s)
            best = max(best, T.tq_decode_workspace_size(list(self.arr), self.B, self.H, self.Hq, self.d))
        return best + (1 << 20)

    def set_step(self, s):
        """Point the segment views at decode step s (0-based within the pool)."""
        s %= self.steps_cap
        w0 = (s // self.chunk) * self.chunk
        self._n_packed[:] = self.n_prompt_packed + w0
        self._n_buf[:] = s - w0 + 1
        self._k_buf[:] = self._k_base + np.uint64(w0 * self._tok_bytes)
        self._v_buf[:] = self._v_base + np.uint64(w0 * self._tok_bytes)
        return w0

    def compress_window(self, s):
        """At the first step of a new 64-token window, compress the previous one."""
        s %= self.steps_cap
        if s == 0 or s % self.chunk:
            return 0
        w0 = s - self.chunk
        for l in range(self.L):
            T.tq_compress(self.packed[l], self.rots[l], self.pool_k[l][:, :, w0:s],
                          self.pool_v[l][:, :, w0:s], t_begin=self.n_prompt_packed + w0)
        return self.L

    def step(self, s, q=None, out=None):
        """Decode step s (into `out`, default self.out); returns the number of
        kernel launches it made."""
        launches = self.compress_window(s)
        self.set_step(s)
        qq = self.qpool[s % self.steps_cap] if q is None else q
        T.tq_decode_attention(None, qq, self.out if out is None else out, self.ws, self.H, views=self.arr)
        return launches + T.tq_decode_last_launches()

    def step_bytes(self, s):
        s %= self.steps_cap
        w0 = (s // self.chunk) * self.chunk
        per_tok_packed = self.H * (16 * (self.w.kbits + self.w.vbits) + 8)
        per_tok_fp16 = self.H * self.d * 2 * 2
        packed = self.L * (self.n_prompt_packed + w0) * per_tok_packed * self.B
        fp16 = self.L * (self.sinks + s - w0 + 1) * per_tok_fp16 * self.B
        qo = self.L * self.B * self.Hq * self.d * (2 + 4)
        return packed, fp16 + qo

    def layer_segments(self, l, s):
        """SegInfo list of layer l as decode step s sees it."""
        s %= self.steps_cap
        w0 = (s // self.chunk) * self.chunk
        H = self.H
        return [SegInfo(self.sink[l], 0, self.sinks, [16] * H, [16] * H, [0] * H),
                SegInfo(self.packed[l], self.sinks, self.n_prompt_packed + w0, [self.w.kbits] * H,
                        [self.w.vbits] * H, [0] * H),
                SegInfo(None, self.T + w0, s - w0 + 1, [16] * H, [16] * H, [0] * H)]


def record_offsets(seg: T.PackedSegment, which: str, b: int, h: int, t: np.ndarray) -> np.ndarray:
    """Byte offsets of the records of positions t of (batch b, head h) in the
    kcodes ('k') or vcodes ('v') buffer: [B][head blocks of capacity x record]."""
    L = seg.layout
    bits = [L.kbits[i] if which == "k" else L.vbits[i] for i in range(L.n_heads)]
    r = [L.head_dim * x // 8 for x in bits]
    return b * L.capacity * sum(r) + L.capacity * sum(r[:h]) + np.asarray(t, np.int64) * r[h]
