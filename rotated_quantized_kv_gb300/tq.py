"""Thin Python binding of the C ABI in ``include/tq.h`` (libtq.so).

Argument marshalling only: every step of compression and attention runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  Importing
this module loads libtq.so and raises ImportError when it is missing or fails
to load; there is no fallback path.

Functions keep the C names: ``tq_make_rotation``, ``tq_fit_codebook``,
``tq_make_qjl``, ``tq_packed_size``, ``tq_compress``, ``tq_dequantize``,
``tq_age_tiers``, ``tq_decode_workspace_size``, ``tq_decode_attention``.
Errors come back as ``TQError`` carrying the status and its message.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libtq.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"libtq.so not found at {_LIB_PATH}; build it with "
        "`python -m rotated_quantized_kv_gb300.build` (needs nvcc)")
try:
    _lib = ctypes.CDLL(_LIB_PATH)
except OSError as e:  # pragma: no cover - depends on the machine
    raise ImportError(f"cannot load {_LIB_PATH}: {e}") from e

LIB_PATH = _LIB_PATH

TQ_MAX_HEADS = 16
TQ_MAX_SEGMENTS = 8
TQ_MAX_HEAD_DIM = 1024
TQ_SEG_PACKED = 0
TQ_SEG_FP16 = 1
TQ_VALUE_LAW_GAUSS = 0
TQ_VALUE_LAW_SPHERE = 1
TQ_QJL_UNBIASED = 0
TQ_QJL_SIGN_PAIR = 1
TQ_ERR_TIMEOUT = -6
TQ_WAIT_POLLS_DEFAULT = 1 << 20

STATUS = {0: "TQ_OK", -1: "TQ_ERR_ARG", -2: "TQ_ERR_UNSUPPORTED", -3: "TQ_ERR_ALIGN",
          -4: "TQ_ERR_SIZE", -5: "TQ_ERR_CUDA", -6: "TQ_ERR_TIMEOUT"}

EXPORTED = ["tq_status_string", "tq_last_cuda_error", "tq_version", "tq_make_rotation",
            "tq_fit_codebook", "tq_make_qjl", "tq_packed_size", "tq_compress", "tq_dequantize",
            "tq_age_tiers", "tq_decode_workspace_size", "tq_decode_attention",
            "tq_set_decode_kernel_events", "tq_decode_attention_static", "tq_decode_error_flag",
            "tq_requantize", "tq_fit_codebook_sphere", "tq_make_haar_rotation", "tq_compress_error_flag", "tq_decode_last_launches",
            "tq_set_decode_wait_polls", "tq_value_code_table"]


class TQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.tq_status_string(status).decode()
        if status == -5:
            msg += f" (cudaError {_lib.tq_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


class tq_rotation(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int), ("seed", ctypes.c_uint64),
                ("sign_bits", ctypes.c_uint32 * (TQ_MAX_HEAD_DIM // 32)), ("dense", ctypes.c_void_p)]


class tq_segment_layout(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("n_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("capacity", ctypes.c_int), ("jl_dim", ctypes.c_int),
                ("kbits", ctypes.c_uint8 * TQ_MAX_HEADS), ("vbits", ctypes.c_uint8 * TQ_MAX_HEADS),
                ("qjl", ctypes.c_uint8 * TQ_MAX_HEADS), ("value_law", ctypes.c_uint8),
                ("qjl_v", ctypes.c_uint8 * TQ_MAX_HEADS)]


class tq_packed_sizes(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("kcode_bytes", "vcode_bytes", "kscale_bytes",
                                                "vscale_bytes", "qjl_sign_bytes", "qjl_norm_bytes",
                                                "vqjl_sign_bytes", "vqjl_norm_bytes")]


class tq_packed_bufs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("kcodes", "vcodes", "kscale", "vscale",
                                                "qjl_signs", "qjl_norm", "vqjl_signs", "vqjl_norm")]


class tq_segment(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("n_tokens", ctypes.c_int), ("layout", tq_segment_layout),
                ("packed", tq_packed_bufs), ("k16", ctypes.c_void_p), ("v16", ctypes.c_void_p),
                ("attn_mass", ctypes.c_void_p)]


class tq_layer_view(ctypes.Structure):
    _fields_ = [("rot", tq_rotation), ("n_segments", ctypes.c_int),
                ("seg", tq_segment * TQ_MAX_SEGMENTS), ("qjl_estimator", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_lib.tq_status_string.restype = ctypes.c_char_p
_lib.tq_status_string.argtypes = [_I]
_lib.tq_last_cuda_error.restype = _I
_lib.tq_version.restype = _I
_lib.tq_decode_last_launches.restype = _I
_lib.tq_decode_last_launches.argtypes = []
_lib.tq_make_rotation.argtypes = [_I, ctypes.c_uint64, ctypes.POINTER(tq_rotation)]
_lib.tq_fit_codebook.argtypes = [_I, _P, _P]
_lib.tq_fit_codebook_sphere.argtypes = [_I, _I, _P, _P]
_lib.tq_value_code_table.argtypes = [_I, _P, _P]
_lib.tq_make_haar_rotation.argtypes = [_I, ctypes.c_uint64, _P]
_lib.tq_compress_error_flag.argtypes = [ctypes.POINTER(ctypes.c_int), _I]
_lib.tq_make_qjl.argtypes = [_I, _I, ctypes.c_uint64, _P]
_lib.tq_packed_size.argtypes = [ctypes.POINTER(tq_segment_layout), ctypes.POINTER(tq_packed_sizes)]
_lib.tq_compress.argtypes = [ctypes.POINTER(tq_segment_layout), ctypes.POINTER(tq_rotation), _P, _P, _P,
                             _I, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _I,
                             ctypes.POINTER(tq_packed_bufs), _P]
_lib.tq_dequantize.argtypes = [ctypes.POINTER(tq_segment_layout), ctypes.POINTER(tq_packed_bufs),
                               ctypes.POINTER(tq_rotation), _I, _I, _P, _P, _P, _P, _P]
_lib.tq_requantize.argtypes = [ctypes.POINTER(tq_segment_layout), ctypes.POINTER(tq_packed_bufs), _I,
                               ctypes.POINTER(tq_segment_layout), ctypes.POINTER(tq_packed_bufs), _I, _I, _P]
_lib.tq_age_tiers.argtypes = [_I, _I, _P, _P, _P]
_lib.tq_decode_workspace_size.argtypes = [ctypes.POINTER(tq_layer_view), _I, _I, _I, _I, _I,
                                          ctypes.POINTER(ctypes.c_size_t)]
_lib.tq_decode_attention.argtypes = [ctypes.POINTER(tq_layer_view), _I, _I, _I, _I, _I, _P, _I, _P, _P,
                                     _P, ctypes.c_size_t, _P]
_lib.tq_set_decode_kernel_events.argtypes = [_P, _P]
_lib.tq_decode_error_flag.argtypes = [_P, ctypes.POINTER(ctypes.c_int), _P]
_lib.tq_set_decode_wait_polls.argtypes = [_I]
_lib.tq_decode_attention_static.argtypes = [ctypes.POINTER(tq_layer_view), _I, _I, _I, _I, _I, _P, _I, _P,
                                            _P, _P]
TQ_STATIC_WORKSPACE_BYTES = 16 << 20
for _n in EXPORTED:
    if _n not in ("tq_status_string", "tq_last_cuda_error", "tq_version", "tq_decode_last_launches"):
        getattr(_lib, _n).restype = _I


def _check(status: int, where: str):
    if status != 0:
        raise TQError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


# ----------------------------------------------------------------- host calls
def tq_version() -> int:
    return _lib.tq_version()


def tq_make_rotation(head_dim: int, seed: int) -> tq_rotation:
    rot = tq_rotation()
    _check(_lib.tq_make_rotation(head_dim, seed, ctypes.byref(rot)), "tq_make_rotation")
    return rot


def tq_fit_codebook(bits: int):
    """(centroids, thresholds) as float32 CPU tensors."""
    c = torch.zeros(1 << bits, dtype=torch.float32)
    t = torch.zeros(max((1 << bits) - 1, 1), dtype=torch.float32)
    _check(_lib.tq_fit_codebook(bits, c.data_ptr(), t.data_ptr()), "tq_fit_codebook")
    return c, t[: (1 << bits) - 1]


def tq_value_code_table(bits: int, thresholds) -> np.ndarray:
    """The compressor's value-code lookup table (2048 uint32) for 1-4 bits and
    an ascending binary32 threshold set (see include/tq.h)."""
    t = np.ascontiguousarray(np.asarray(thresholds, dtype=np.float32))
    out = np.zeros(2048, dtype=np.uint32)
    _check(_lib.tq_value_code_table(bits, t.ctypes.data, out.ctypes.data), "tq_value_code_table")
    return out


def tq_fit_codebook_sphere(bits: int, head_dim: int = 128):
    """(centroids, thresholds) of the sphere-coordinate law, float32 CPU tensors."""
    c = torch.zeros(1 << bits, dtype=torch.float32)
    t = torch.zeros(max((1 << bits) - 1, 1), dtype=torch.float32)
    _check(_lib.tq_fit_codebook_sphere(bits, head_dim, c.data_ptr(), t.data_ptr()), "tq_fit_codebook_sphere")
    return c, t[: (1 << bits) - 1]


def tq_make_haar_rotation(head_dim: int, seed: int) -> torch.Tensor:
    """Haar-random rotation Q (float32 CPU tensor [d][d], y = Q x)."""
    Q = torch.zeros(head_dim, head_dim, dtype=torch.float32)
    _check(_lib.tq_make_haar_rotation(head_dim, seed, Q.data_ptr()), "tq_make_haar_rotation")
    return Q


def dense_rotation(rot: tq_rotation, Q: torch.Tensor) -> tq_rotation:
    """A copy of ``rot`` that rotates with the dense matrix Q (a float32 CUDA
    tensor [d][d] the caller keeps alive) instead of the SRHT."""
    r = tq_rotation()
    ctypes.pointer(r)[0] = rot
    assert Q.dtype == torch.float32 and Q.is_contiguous() and tuple(Q.shape) == (rot.head_dim, rot.head_dim)
    r.dense = Q.data_ptr()
    return r


def tq_compress_error_flag(reset: bool = False) -> int:
    """The dense compressor's timeout flag (0: none); the call's TQ_ERR_TIMEOUT
    status is returned as the flag, not raised."""
    f = ctypes.c_int(0)
    st = _lib.tq_compress_error_flag(ctypes.byref(f), int(reset))
    if st != TQ_ERR_TIMEOUT:
        _check(st, "tq_compress_error_flag")
    return f.value


def tq_make_qjl(head_dim: int, jl_dim: int, seed: int) -> torch.Tensor:
    """QJL projection S (float32 CPU tensor [jl_dim][head_dim])."""
    S = torch.zeros(jl_dim, head_dim, dtype=torch.float32)
    _check(_lib.tq_make_qjl(head_dim, jl_dim, seed, S.data_ptr()), "tq_make_qjl")
    return S


def make_layout(batch, n_heads, head_dim, capacity, kbits, vbits, qjl=None, jl_dim=128, value_law=0, qjl_v=None):
    L = tq_segment_layout()
    L.batch, L.n_heads, L.head_dim, L.capacity, L.jl_dim = batch, n_heads, head_dim, capacity, jl_dim
    L.value_law = value_law
    kb = [int(kbits)] * n_heads if isinstance(kbits, int) else [int(x) for x in kbits]
    vb = [int(vbits)] * n_heads if isinstance(vbits, int) else [int(x) for x in vbits]
    qj = [0] * n_heads if qjl is None else [int(bool(x)) for x in qjl]
    qv = [0] * n_heads if qjl_v is None else [int(bool(x)) for x in qjl_v]
    for h in range(n_heads):
        L.kbits[h], L.vbits[h], L.qjl[h], L.qjl_v[h] = kb[h], vb[h], qj[h], qv[h]
    return L


def tq_packed_size(layout: tq_segment_layout) -> tq_packed_sizes:
    s = tq_packed_sizes()
    _check(_lib.tq_packed_size(ctypes.byref(layout), ctypes.byref(s)), "tq_packed_size")
    return s


def tq_age_tiers(n_tokens: int, age_bounds):
    b = (ctypes.c_int * max(len(age_bounds), 1))(*age_bounds)
    start = (ctypes.c_int * (len(age_bounds) + 1))()
    end = (ctypes.c_int * (len(age_bounds) + 1))()
    _check(_lib.tq_age_tiers(n_tokens, len(age_bounds), b, start, end), "tq_age_tiers")
    return list(zip(start, end))


# ----------------------------------------------------------------- segments
class PackedSegment:
    """Device buffers of one packed segment, allocated with torch from the sizes
    tq_packed_size reports."""

    kind = TQ_SEG_PACKED
    attn_mass = None  # optional float tensor [B][H][capacity]: written by tq_decode_attention

    def __init__(self, layout: tq_segment_layout, device="cuda", n_tokens: int = 0):
        self.layout = layout
        self.n_tokens = n_tokens
        s = tq_packed_size(layout)
        u8 = dict(dtype=torch.uint8, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.kcodes = torch.zeros(max(s.kcode_bytes, 16), **u8)
        self.vcodes = torch.zeros(max(s.vcode_bytes, 16), **u8)
        self.kscale = torch.zeros(max(s.kscale_bytes // 4, 4), **f32)
        self.vscale = torch.zeros(max(s.vscale_bytes // 4, 4), **f32)
        self.qjl_signs = torch.zeros(max(s.qjl_sign_bytes, 16), **u8) if s.qjl_sign_bytes else None
        self.qjl_norm = torch.zeros(max(s.qjl_norm_bytes // 4, 4), **f32) if s.qjl_norm_bytes else None
        self.vqjl_signs = torch.zeros(max(s.vqjl_sign_bytes, 16), **u8) if s.vqjl_sign_bytes else None
        self.vqjl_norm = torch.zeros(max(s.vqjl_norm_bytes // 4, 4), **f32) if s.vqjl_norm_bytes else None

    def bufs(self) -> tq_packed_bufs:
        b = tq_packed_bufs()
        b.kcodes, b.vcodes = _ptr(self.kcodes), _ptr(self.vcodes)
        b.kscale, b.vscale = _ptr(self.kscale), _ptr(self.vscale)
        b.qjl_signs, b.qjl_norm = _ptr(self.qjl_signs), _ptr(self.qjl_norm)
        b.vqjl_signs, b.vqjl_norm = _ptr(self.vqjl_signs), _ptr(self.vqjl_norm)
        return b

    def segment(self) -> tq_segment:
        s = tq_segment()
        s.kind, s.n_tokens, s.layout, s.packed = TQ_SEG_PACKED, self.n_tokens, self.layout, self.bufs()
        s.attn_mass = _ptr(self.attn_mass)
        return s

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.kcodes, self.vcodes, self.kscale, self.vscale, self.qjl_signs, self.qjl_norm,
                    self.vqjl_signs, self.vqjl_norm)
                   if t is not None)


class Fp16Segment:
    """Tokens kept verbatim in fp16: [B][H][capacity][d] K and V."""

    kind = TQ_SEG_FP16
    attn_mass = None  # optional float tensor [B][H][capacity]: written by tq_decode_attention

    def __init__(self, batch, n_heads, head_dim, capacity, device="cuda", n_tokens=0, k=None, v=None):
        self.layout = make_layout(batch, n_heads, head_dim, capacity, 1, 1)
        self.n_tokens = n_tokens
        shape = (batch, n_heads, capacity, head_dim)
        self.k = k if k is not None else torch.zeros(shape, dtype=torch.float16, device=device)
        self.v = v if v is not None else torch.zeros(shape, dtype=torch.float16, device=device)

    def segment(self) -> tq_segment:
        s = tq_segment()
        s.kind, s.n_tokens, s.layout = TQ_SEG_FP16, self.n_tokens, self.layout
        s.k16, s.v16 = _ptr(self.k), _ptr(self.v)
        s.attn_mass = _ptr(self.attn_mass)
        return s


def layer_view(rot: tq_rotation, segments, qjl_estimator: int = TQ_QJL_UNBIASED) -> tq_layer_view:
    """A layer's segments; a segment's attn_mass tensor (if set) receives the
    attention mass of its tokens at the next decode call."""
    lv = tq_layer_view()
    lv.rot = rot
    lv.qjl_estimator = qjl_estimator
    lv.n_segments = len(segments)
    for i, s in enumerate(segments):
        lv.seg[i] = s.segment()
    return lv


# ----------------------------------------------------------------- device calls
def tq_compress(seg: PackedSegment, rot: tq_rotation, K: torch.Tensor, V: torch.Tensor, t_begin: int = 0,
                qjl_S: torch.Tensor | None = None, stream=None):
    """Compress K, V (fp16 CUDA tensors [B][H][T][d], unit stride in d) into
    positions [t_begin, t_begin + T) of ``seg``."""
    B, H, T, d = K.shape
    assert V.shape == K.shape and V.stride() == K.stride() and K.dtype == torch.float16
    sb, sh, st, si = K.stride()
    assert si == 1
    _check(_lib.tq_compress(ctypes.byref(seg.layout), ctypes.byref(rot), _ptr(qjl_S), _ptr(K), _ptr(V), T,
                            sb, sh, st, t_begin, ctypes.byref(seg.bufs()), _stream(stream)), "tq_compress")
    seg.n_tokens = max(seg.n_tokens, t_begin + T)


def tq_requantize(src: PackedSegment, src_t_begin: int, n_tokens: int, dst: PackedSegment, dst_t_begin: int,
                  stream=None):
    """Tier demotion: tokens [src_t_begin, src_t_begin + n) of src re-quantised
    in the rotated space with dst's widths into [dst_t_begin, dst_t_begin + n)."""
    _check(_lib.tq_requantize(ctypes.byref(src.layout), ctypes.byref(src.bufs()), src_t_begin,
                              ctypes.byref(dst.layout), ctypes.byref(dst.bufs()), dst_t_begin, n_tokens,
                              _stream(stream)), "tq_requantize")
    dst.n_tokens = max(dst.n_tokens, dst_t_begin + n_tokens)


def tq_dequantize(seg: PackedSegment, t_begin: int, n_tokens: int, rot: tq_rotation | None = None,
                  rotated: bool = True, original: bool = False, stream=None):
    """(k_rot, v_rot, k_orig, v_orig) float32 [B][H][n][d] CUDA tensors (None where not asked)."""
    L = seg.layout
    shape = (L.batch, L.n_heads, n_tokens, L.head_dim)
    dev = seg.kcodes.device
    mk = (lambda: torch.empty(shape, dtype=torch.float32, device=dev))
    kr, vr = (mk(), mk()) if rotated else (None, None)
    ko, vo = (mk(), mk()) if original else (None, None)
    _check(_lib.tq_dequantize(ctypes.byref(L), ctypes.byref(seg.bufs()),
                              ctypes.byref(rot) if rot is not None else None, t_begin, n_tokens,
                              _ptr(kr), _ptr(vr), _ptr(ko), _ptr(vo), _stream(stream)), "tq_dequantize")
    return kr, vr, ko, vo


def _views(layers):
    arr = (tq_layer_view * len(layers))()
    for i, lv in enumerate(layers):
        arr[i] = lv
    return arr


def tq_decode_workspace_size(layers, batch, n_heads, q_heads, head_dim) -> int:
    n = ctypes.c_size_t()
    _check(_lib.tq_decode_workspace_size(_views(layers), len(layers), batch, n_heads, q_heads, head_dim,
                                         ctypes.byref(n)), "tq_decode_workspace_size")
    return n.value


def tq_decode_attention(layers, q: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                        n_heads: int, qjl_S: torch.Tensor | None = None, jl_dim: int = 128, stream=None,
                        views=None):
    """out[l][b][j] = attention of q[l][b][j] (fp16) over layer l's segments.
    ``layers`` is a list of tq_layer_view; ``views`` may pass a prebuilt ctypes array."""
    L, B, Hq, d = q.shape
    arr = views if views is not None else _views(layers)
    _check(_lib.tq_decode_attention(arr, L, B, n_heads, Hq, d, _ptr(qjl_S), jl_dim, _ptr(q), _ptr(out),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)), "tq_decode_attention")
    return out


def tq_decode_last_launches() -> int:
    """Kernel launches this thread's last decode call made."""
    return _lib.tq_decode_last_launches()


def tq_set_decode_kernel_events(start=None, stop=None):
    """Time the packed split-K kernel alone: pass two torch.cuda.Event objects
    (created with enable_timing=True), or None, None to stop."""
    sp = start.cuda_event if start is not None else None
    ep = stop.cuda_event if stop is not None else None
    _check(_lib.tq_set_decode_kernel_events(sp, ep), "tq_set_decode_kernel_events")


def tq_decode_attention_static(layers, q: torch.Tensor, out: torch.Tensor, n_heads: int,
                               qjl_S: torch.Tensor | None = None, jl_dim: int = 128, stream=None, views=None):
    """tq_decode_attention without a workspace argument: the library's fixed
    TQ_STATIC_WORKSPACE_BYTES device array is the scratch, so the call allocates
    nothing (for callers that may not allocate device memory while running).
    Calls share that array: keep them ordered on one stream."""
    L, B, Hq, d = q.shape
    arr = views if views is not None else _views(layers)
    _check(_lib.tq_decode_attention_static(arr, L, B, n_heads, Hq, d, _ptr(qjl_S), jl_dim, _ptr(q), _ptr(out),
                                           _stream(stream)), "tq_decode_attention_static")
    return out


def tq_decode_error_flag(workspace: torch.Tensor | None, stream=None) -> int:
    """Non-zero if a decode call on this workspace stopped a CTA after a bounded
    wait for its own copies (never expected); synchronises the stream.  None:
    the static scratch array of tq_decode_attention_static.  The call's
    TQ_ERR_TIMEOUT status is returned as the flag, not raised."""
    f = ctypes.c_int()
    st = _lib.tq_decode_error_flag(_ptr(workspace), ctypes.byref(f), _stream(stream))
    if st != TQ_ERR_TIMEOUT:
        _check(st, "tq_decode_error_flag")
    return f.value


def tq_set_decode_wait_polls(polls: int):
    """Failure-path hook for tests: polls of a split-K CTA's wait for its own
    copies before it gives up (default 2^20; 0 = give up at once)."""
    _check(_lib.tq_set_decode_wait_polls(polls), "tq_set_decode_wait_polls")


def views_array(layers):
    """Prebuilt ctypes array of layer views (reuse across calls to skip marshalling)."""
    return _views(layers)
