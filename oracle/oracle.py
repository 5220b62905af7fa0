"""CPU oracle for rotated + quantized KV compression and decode attention.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The product path (the CUDA
library and its Python binding) never imports this module, and this module
never imports the product package.

The arithmetic lives in ``tq_oracle.c`` (plain scalar C, binary32 where the
compressed format fixes binary32, binary64 elsewhere).  This wrapper only moves
numpy arrays in and out and holds the packed-segment layout, which is a byte
format both sides implement independently:

* record sizes ``rk(h) = d*kbits[h]/8`` and ``rv(h) = d*vbits[h]/8`` bytes;
* key/value codes of (b, h, t) at byte ``b*cap*sum(r) + cap*sum(r[:h]) + t*r[h]``;
* scales (float32) at ``(b*H + h)*cap + t``;
* QJL sign records (``jl/8`` bytes) and norms at ``(b*nq + rank(h))*cap + t``
  where ``rank(h)`` counts the QJL heads before ``h``;
* fp16 segments: ``((b*H + h)*cap + t)*d`` elements.

Pages cited (title and section): "turboquant-mlx" (TurboQuant-MLX v2.0 README),
sections "Walsh-Hadamard Rotation", "FP16 Attention Sinks", "Dynamic Chunk
Buffering"; "TurboMOQ", sections "Architecture", "Progressive temporal tiering",
"QJL residual correction (sub-2-bit)".
"""
from __future__ import annotations

import ctypes
import functools
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libtq_oracle.so")

GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (no FMA contraction) if it is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *GCC_FLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_P = ctypes.c_void_p
_I = ctypes.c_int
_U64 = ctypes.c_uint64
_LL = ctypes.c_longlong


class _Segment(ctypes.Structure):
    _fields_ = [
        ("kind", _I), ("n_tokens", _I), ("capacity", _I),
        ("kbits", _P), ("vbits", _P), ("qjl", _P),
        ("kcodes", _P), ("vcodes", _P), ("kscale", _P), ("vscale", _P),
        ("qjl_signs", _P), ("qjl_norm", _P), ("k16", _P), ("v16", _P), ("value_law", _I),
        ("qjl_v", _P), ("vqjl_signs", _P), ("vqjl_norm", _P),
    ]


@functools.lru_cache(maxsize=None)
def lib() -> ctypes.CDLL:
    L = ctypes.CDLL(build())
    L.tqo_splitmix64.argtypes = [_U64, _I, _P]
    L.tqo_signs.argtypes = [_I, _U64, _P]
    L.tqo_half_to_double.argtypes = [ctypes.c_uint16]
    L.tqo_half_to_double.restype = ctypes.c_double
    L.tqo_rotate_f32.argtypes = [_I, _P, _P, _P]
    L.tqo_rotate_f64.argtypes = [_I, _P, _P, _P]
    L.tqo_lloyd_max.argtypes = [_I, _P, _P, _I]
    L.tqo_lloyd_max.restype = _I
    L.tqo_lloyd_max_sphere.argtypes = [_I, _I, _P, _P, _I]
    L.tqo_lloyd_max_sphere.restype = _I
    L.tqo_quant_key.argtypes = [_I, _I, _P, _P, _P]
    L.tqo_key_level.argtypes = [_I, _I]
    L.tqo_key_level.restype = ctypes.c_double
    L.tqo_quant_value.argtypes = [_I, _I, _P, _P, _P, _P]
    L.tqo_pack.argtypes = [_I, _I, _P, _P]
    L.tqo_unpack.argtypes = [_I, _I, _P, _P]
    L.tqo_qjl_matrix.argtypes = [_I, _I, _U64, _P]
    L.tqo_qjl_project.argtypes = [_I, _I, _P, _P, _P]
    L.tqo_qjl_sketch.argtypes = [_I, _I, _P, _P, _P, _P, _P]
    L.tqo_compress.argtypes = [_I, _I, _I, _I, _P, _P, _LL, _LL, _LL, _P, _P, _P, _I,
                               ctypes.POINTER(_Segment), _I, _P, _P]
    L.tqo_rotate_dense_f32.argtypes = [_I, _P, _P, _P]
    L.tqo_dequant.argtypes = [_I, _I, ctypes.POINTER(_Segment), _I, _I, _I, _I, _P, _P, _P]
    L.tqo_decode_attention.argtypes = [_I, _I, _I, _I, _I, ctypes.POINTER(_Segment), _P, _P,
                                       _P, _I, _I, _P, _P, _P, _P]
    L.tqo_requantize.argtypes = [_I, _I, _I, ctypes.POINTER(_Segment), _I, _I, _P, _P,
                                 ctypes.POINTER(_Segment), _I]
    return L


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------- #
# primitives
# --------------------------------------------------------------------------- #
def splitmix64(seed: int, n: int) -> np.ndarray:
    out = np.zeros(n, np.uint64)
    lib().tqo_splitmix64(seed, n, _ptr(out))
    return out


def signs(d: int, seed: int) -> np.ndarray:
    """Sign diagonal D (int8, +-1) of the layer rotation seeded with ``seed``."""
    out = np.zeros(d, np.int8)
    lib().tqo_signs(d, seed, _ptr(out))
    return out


def half_to_double(bits: np.ndarray) -> np.ndarray:
    f = lib().tqo_half_to_double
    flat = np.asarray(bits, np.uint16).ravel()
    return np.array([f(int(h)) for h in flat], np.float64).reshape(np.shape(bits))


def rotate_f32(x: np.ndarray, sign: np.ndarray) -> np.ndarray:
    """y = R x in the binary32 order of the compressed format; x is [..., d] float32."""
    x = _c(x, np.float32)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    y = np.empty_like(flat)
    s = _c(sign, np.int8)
    L = lib()
    for i in range(flat.shape[0]):
        L.tqo_rotate_f32(d, _ptr(s), _ptr(flat[i]), _ptr(y[i]))
    return y.reshape(x.shape)


def rotate_f64(x: np.ndarray, sign: np.ndarray) -> np.ndarray:
    x = _c(x, np.float64)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    y = np.empty_like(flat)
    s = _c(sign, np.int8)
    L = lib()
    for i in range(flat.shape[0]):
        L.tqo_rotate_f64(d, _ptr(s), _ptr(flat[i]), _ptr(y[i]))
    return y.reshape(x.shape)


@functools.lru_cache(maxsize=None)
def haar_rotation(d: int, seed: int) -> np.ndarray:
    """Dense Haar-random rotation ("TurboMOQ", "Stable QR Rotation": QR of a
    Gaussian matrix through LAPACK).  G = the N(0,1) matrix of qjl_matrix(d, d,
    seed) (Box-Muller on SplitMix64, binary32); G = Q R by numpy.linalg.qr in
    binary64, the columns of Q multiplied by the signs of diag(R) so that R has a
    positive diagonal (Q is then Haar-distributed, Mezzadri 2007); Q rounded to
    binary32.  y = Q x is the rotation."""
    G = qjl_matrix(d, d, seed).astype(np.float64)
    Qm, R = np.linalg.qr(G)
    sgn = np.where(np.diag(R) < 0, -1.0, 1.0)
    return (Qm * sgn[None, :]).astype(np.float32)


def rotate_dense_f32(x: np.ndarray, Q: np.ndarray) -> np.ndarray:
    """Binary32 rotated vector y = Q x (the exact product rounded once)."""
    xx = _c(np.asarray(x, np.float32), np.float32)
    y = np.zeros(Q.shape[0], np.float32)
    lib().tqo_rotate_dense_f32(Q.shape[0], _ptr(_c(Q, np.float32)), _ptr(xx), _ptr(y))
    return y


def lloyd_max(bits: int, max_iter: int = 1_000_000):
    """Gaussian Lloyd-Max codebook in binary64: (centroids, thresholds, sweeps)."""
    n = 1 << bits
    c = np.zeros(n, np.float64)
    t = np.zeros(max(n - 1, 1), np.float64)
    it = lib().tqo_lloyd_max(bits, _ptr(c), _ptr(t), max_iter)
    if it < 0:
        raise ValueError(f"bad bit width {bits}")
    c.setflags(write=False)
    t.setflags(write=False)
    return c, t[: n - 1], it


@functools.lru_cache(maxsize=None)
def lloyd_max_sphere(bits: int, d: int = 128, max_iter: int = 1_000_000):
    """binary64 (centroids, thresholds, sweeps) of the Lloyd-Max quantizer for
    sqrt(d) times a coordinate of a uniform unit d-vector (the sphere-coordinate
    value codebook)."""
    n = 1 << bits
    c = np.zeros(n)
    t = np.zeros(max(n - 1, 1))
    it = lib().tqo_lloyd_max_sphere(bits, d, _ptr(c), _ptr(t), max_iter)
    assert it > 0
    return c, t[: n - 1], it


def codebook_f32(bits: int):
    """The binary32 centroids and thresholds the format stores."""
    c, t, _ = lloyd_max(bits)
    return c.astype(np.float32), t.astype(np.float32)


def codebook_sphere_f32(bits: int, d: int = 128):
    """The binary32 centroids and thresholds of the sphere-coordinate codebook."""
    c, t, _ = lloyd_max_sphere(bits, d)
    return c.astype(np.float32), t.astype(np.float32)


@functools.lru_cache(maxsize=None)
def _cent_thr_tables():
    """binary32 centroid and threshold tables of widths 1..8 for both value
    codebook laws (index law * 9 + bits; law 0 Gaussian, 1 sphere coordinate
    for d = 128) and C pointer arrays to them (cached: the arrays must outlive
    every call that uses the pointers)."""
    cents = ([np.zeros(1, np.float32)] + [codebook_f32(b)[0] for b in range(1, 9)] +
             [np.zeros(1, np.float32)] + [codebook_sphere_f32(b)[0] for b in range(1, 9)])
    thrs = ([np.zeros(1, np.float32)] + [codebook_f32(b)[1] for b in range(1, 9)] +
            [np.zeros(1, np.float32)] + [codebook_sphere_f32(b)[1] for b in range(1, 9)])
    cp = (ctypes.c_void_p * 18)(*[c.ctypes.data for c in cents])
    tp = (ctypes.c_void_p * 18)(*[t.ctypes.data for t in thrs])
    return cents, thrs, cp, tp


def quant_key(y: np.ndarray, bits: int):
    """Key codes (uint8 [..., d]) and scales m (float32 [...]) of rotated vectors."""
    y = _c(y, np.float32)
    d = y.shape[-1]
    flat = y.reshape(-1, d)
    codes = np.empty(flat.shape, np.uint8)
    scales = np.empty(flat.shape[0], np.float32)
    L = lib()
    for i in range(flat.shape[0]):
        L.tqo_quant_key(d, bits, _ptr(flat[i]), _ptr(codes[i]), _ptr(scales[i:i + 1]))
    return codes.reshape(y.shape), scales.reshape(y.shape[:-1])


def key_levels(bits: int) -> np.ndarray:
    f = lib().tqo_key_level
    return np.array([f(bits, k) for k in range(1 << bits)], np.float64)


def quant_value(y: np.ndarray, bits: int):
    """Value codes (uint8 [..., d]) and scales sigma (float32 [...])."""
    y = _c(y, np.float32)
    d = y.shape[-1]
    flat = y.reshape(-1, d)
    thr = _c(codebook_f32(bits)[1], np.float32)
    codes = np.empty(flat.shape, np.uint8)
    scales = np.empty(flat.shape[0], np.float32)
    L = lib()
    for i in range(flat.shape[0]):
        L.tqo_quant_value(d, bits, _ptr(flat[i]), _ptr(thr), _ptr(codes[i]), _ptr(scales[i:i + 1]))
    return codes.reshape(y.shape), scales.reshape(y.shape[:-1])


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    d = codes.shape[-1]
    flat = codes.reshape(-1, d)
    out = np.zeros((flat.shape[0], d * bits // 8), np.uint8)
    L = lib()
    for i in range(flat.shape[0]):
        L.tqo_pack(d, bits, _ptr(flat[i]), _ptr(out[i]))
    return out.reshape(codes.shape[:-1] + (d * bits // 8,))


def unpack(rec: np.ndarray, bits: int, d: int) -> np.ndarray:
    rec = _c(rec, np.uint8)
    flat = rec.reshape(-1, d * bits // 8)
    out = np.zeros((flat.shape[0], d), np.uint8)
    L = lib()
    for i in range(flat.shape[0]):
        L.tqo_unpack(d, bits, _ptr(flat[i]), _ptr(out[i]))
    return out.reshape(rec.shape[:-1] + (d,))


def qjl_matrix(jl: int, d: int, seed: int) -> np.ndarray:
    S = np.zeros((jl, d), np.float32)
    lib().tqo_qjl_matrix(jl, d, seed, _ptr(S))
    return S


def qjl_project(S: np.ndarray, r: np.ndarray) -> np.ndarray:
    S = _c(S, np.float32)
    r = _c(r, np.float32)
    p = np.zeros(S.shape[0], np.float64)
    lib().tqo_qjl_project(S.shape[0], S.shape[1], _ptr(S), _ptr(r), _ptr(p))
    return p


def qjl_sketch(S: np.ndarray, y: np.ndarray, yhat: np.ndarray):
    S = _c(S, np.float32)
    y = _c(y, np.float32)
    yhat = _c(yhat, np.float32)
    jl, d = S.shape
    signs_ = np.zeros(jl // 8, np.uint8)
    rho = np.zeros(1, np.float32)
    lib().tqo_qjl_sketch(jl, d, _ptr(S), _ptr(y), _ptr(yhat), _ptr(signs_), _ptr(rho))
    return signs_, float(rho[0])


# --------------------------------------------------------------------------- #
# packed segments
# --------------------------------------------------------------------------- #
class PackedSegment:
    """Host buffers of one packed segment in the documented byte layout."""

    kind = 0

    def __init__(self, B, H, d, capacity, kbits, vbits, qjl=None, jl=128, n_tokens=0, law=0, qjl_v=None):
        self.B, self.H, self.d, self.capacity, self.jl = B, H, d, capacity, jl
        self.law = law  # value codebook: 0 Gaussian, 1 sphere coordinate (d = 128)
        assert law in (0, 1) and (law == 0 or d == 128)
        self.kbits = _c(kbits, np.uint8)
        self.vbits = _c(vbits, np.uint8)
        self.qjl = _c(np.zeros(H) if qjl is None else qjl, np.uint8)
        self.n_tokens = n_tokens
        rk = int(sum(d * int(b) // 8 for b in self.kbits))
        rv = int(sum(d * int(b) // 8 for b in self.vbits))
        nq = int(self.qjl.astype(bool).sum())
        self.nq = nq
        self.kcodes = np.zeros(B * capacity * rk, np.uint8)
        self.vcodes = np.zeros(B * capacity * rv, np.uint8)
        self.kscale = np.zeros(B * H * capacity, np.float32)
        self.vscale = np.zeros(B * H * capacity, np.float32)
        self.qjl_signs = np.zeros(max(B * nq * capacity * (jl // 8), 1), np.uint8)
        self.qjl_norm = np.zeros(max(B * nq * capacity, 1), np.float32)
        # QJL on values: the value residual's sketch, heads ranked like the keys'
        self.qjl_v = _c(np.zeros(H) if qjl_v is None else qjl_v, np.uint8)
        nv = int(self.qjl_v.astype(bool).sum())
        self.nv = nv
        self.vqjl_signs = np.zeros(max(B * nv * capacity * (jl // 8), 1), np.uint8)
        self.vqjl_norm = np.zeros(max(B * nv * capacity, 1), np.float32)

    def code_offset(self, which: str, b: int, h: int, t: int) -> int:
        bits = self.kbits if which == "k" else self.vbits
        r = [self.d * int(x) // 8 for x in bits]
        return b * self.capacity * sum(r) + self.capacity * sum(r[:h]) + t * r[h]

    def qjl_rank(self, h: int) -> int:
        return int(self.qjl[:h].astype(bool).sum())

    def vqjl_rank(self, h: int) -> int:
        return int(self.qjl_v[:h].astype(bool).sum())

    def c_struct(self) -> _Segment:
        s = _Segment()
        s.kind, s.n_tokens, s.capacity = 0, self.n_tokens, self.capacity
        s.kbits, s.vbits, s.qjl = _ptr(self.kbits), _ptr(self.vbits), _ptr(self.qjl)
        s.kcodes, s.vcodes = _ptr(self.kcodes), _ptr(self.vcodes)
        s.kscale, s.vscale = _ptr(self.kscale), _ptr(self.vscale)
        s.qjl_signs, s.qjl_norm = _ptr(self.qjl_signs), _ptr(self.qjl_norm)
        s.k16 = s.v16 = None
        s.value_law = self.law
        s.qjl_v, s.vqjl_signs, s.vqjl_norm = _ptr(self.qjl_v), _ptr(self.vqjl_signs), _ptr(self.vqjl_norm)
        return s


class Fp16Segment:
    """Tokens kept verbatim in fp16 (sinks, the newest tier, the chunk buffer)."""

    kind = 1

    def __init__(self, B, H, d, capacity, n_tokens=0):
        self.B, self.H, self.d, self.capacity, self.n_tokens = B, H, d, capacity, n_tokens
        self.k16 = np.zeros(B * H * capacity * d, np.uint16)
        self.v16 = np.zeros(B * H * capacity * d, np.uint16)

    def c_struct(self) -> _Segment:
        s = _Segment()
        s.kind, s.n_tokens, s.capacity = 1, self.n_tokens, self.capacity
        s.k16, s.v16 = _ptr(self.k16), _ptr(self.v16)
        return s


def compress(seg: PackedSegment, K: np.ndarray, V: np.ndarray, sign: np.ndarray,
             S: np.ndarray | None = None, t_begin: int = 0, Q: np.ndarray | None = None) -> None:
    """Compress fp16 K, V ([B][H][T][d] arrays of fp16 values or uint16 bit
    patterns) into positions [t_begin, t_begin + T) of ``seg``; Q (binary32
    d x d) replaces the SRHT of ``sign`` by the dense rotation y = Q x."""
    Kb = _c(np.asarray(K).view(np.uint16) if np.asarray(K).dtype == np.float16 else K, np.uint16)
    Vb = _c(np.asarray(V).view(np.uint16) if np.asarray(V).dtype == np.float16 else V, np.uint16)
    B, H, T, d = Kb.shape
    assert (B, H, d) == (seg.B, seg.H, seg.d) and t_begin + T <= seg.capacity
    _, _, cp, tp = _cent_thr_tables()
    s = _c(sign, np.int8)
    Sm = None if S is None else _c(S, np.float32)
    cs = seg.c_struct()
    Qm = None if Q is None else _c(Q, np.float32)
    lib().tqo_compress(B, H, d, T, _ptr(Kb), _ptr(Vb), H * T * d, T * d, d, _ptr(s), tp,
                       _ptr(Sm), seg.jl, ctypes.byref(cs), t_begin, _ptr(Qm), cp)
    seg.n_tokens = max(seg.n_tokens, t_begin + T)


def dequant(seg: PackedSegment, b: int, h: int, t0: int, n: int):
    """Rotated-space dequantized keys and values (float32 [n][d]) of (b, h)."""
    cents, _, cp, _ = _cent_thr_tables()
    kh = np.zeros((n, seg.d), np.float32)
    vh = np.zeros((n, seg.d), np.float32)
    cs = seg.c_struct()
    lib().tqo_dequant(seg.H, seg.d, ctypes.byref(cs), b, h, t0, n, cp, _ptr(kh), _ptr(vh))
    return kh, vh


def requantize(src: PackedSegment, src_t0: int, n: int, dst: PackedSegment, dst_t0: int) -> None:
    """Tier demotion: tokens [src_t0, src_t0 + n) of src, dequantized in the
    rotated space, compressed again with dst's widths into [dst_t0, dst_t0 + n)
    of dst (no QJL on dst)."""
    assert (src.B, src.H, src.d) == (dst.B, dst.H, dst.d)
    assert src_t0 + n <= src.capacity and dst_t0 + n <= dst.capacity and not dst.qjl.any() and not dst.qjl_v.any()
    _, _, cp, tp = _cent_thr_tables()
    ss, ds = src.c_struct(), dst.c_struct()
    lib().tqo_requantize(src.B, src.H, src.d, ctypes.byref(ss), src_t0, n, cp, tp, ctypes.byref(ds), dst_t0)
    dst.n_tokens = max(dst.n_tokens, dst_t0 + n)


def decode_attention(segments, q: np.ndarray, sign: np.ndarray, H: int,
                     S: np.ndarray | None = None, jl: int = 128, estimator: int = 0,
                     with_mass: bool = False, Q: np.ndarray | None = None):
    """Binary64 attention of q ([B][Hq][d], fp16) over a layer's segments.

    estimator: 0 = QJL residual estimate added to the key ("QJL residual
    correction (sub-2-bit)"); 1 = sign-pair estimate added to the score ("RaBitQ
    vs QJL correction").  with_mass: also return, per segment, the attention
    mass [B][H][n_tokens] of each token: its softmax weight averaged over the
    query heads of its KV head.  Q: the layer's dense rotation (binary32 d x d)
    instead of the SRHT of ``sign``."""
    qb = _c(np.asarray(q).view(np.uint16) if np.asarray(q).dtype == np.float16 else q, np.uint16)
    B, Hq, d = qb.shape
    cents, _, cp, _ = _cent_thr_tables()
    arr = (_Segment * max(len(segments), 1))(*[s.c_struct() for s in segments])
    out = np.zeros((B, Hq, d), np.float64)
    s = _c(sign, np.int8)
    Sm = None if S is None else _c(S, np.float32)
    total = sum(int(sg.n_tokens) for sg in segments)
    mass = np.zeros((B, H, max(total, 1)), np.float64) if with_mass else None
    Qm = None if Q is None else _c(Q, np.float32)
    lib().tqo_decode_attention(B, H, Hq, d, len(segments), arr, _ptr(s), cp, _ptr(Sm), jl, estimator,
                               _ptr(qb), _ptr(out), _ptr(mass), _ptr(Qm))
    if not with_mass:
        return out
    per_seg, n = [], 0
    for sg in segments:
        per_seg.append(mass[:, :, n:n + int(sg.n_tokens)].copy())
        n += int(sg.n_tokens)
    return out, per_seg


# --------------------------------------------------------------------------- #
# host planning steps of the method
# --------------------------------------------------------------------------- #
def tier_ranges(T: int, age_bounds=(1024, 8192, 65536)):
    """Progressive tiers by token age ("TurboMOQ", "Progressive temporal tiering":
    Active 0-1K fp16, Warm 1K-8K K4V4, Cold 8K-64K K3V2, Archive 64K+ K2V1).
    Age of position p is T-1-p.  Returns [(tier, start, end)] for non-empty tiers,
    tier 0 = newest, in ascending position order."""
    out = []
    edges = [0, *age_bounds, None]
    for tier in range(len(edges) - 1, 0, -1):
        lo_age = edges[tier - 1]
        hi_age = edges[tier]
        # positions with lo_age <= T-1-p < hi_age
        start = 0 if hi_age is None else max(0, T - hi_age)
        end = max(0, T - lo_age)
        if end > start:
            out.append((tier - 1, start, end))
    return out


def chunk_schedule(T: int, sinks: int = 128, chunk: int = 64):
    """Sinks stay fp16 ("FP16 Attention Sinks": first 128 tokens); the rest is
    compressed in whole chunks of 64 ("Dynamic Chunk Buffering"); the remainder
    waits in an fp16 buffer.  Returns (sink_count, [chunk starts], buffered)."""
    s = min(T, sinks)
    n_chunks = (T - s) // chunk
    starts = [s + i * chunk for i in range(n_chunks)]
    return s, starts, T - s - n_chunks * chunk
