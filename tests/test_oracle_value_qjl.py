"""Pins of QJL on values (the second half of the QJL row: "TurboMOQ", "QJL
residual correction (sub-2-bit)" applied to the value residual as to the key
one).  The value residual r = y - sigma c[code] is sketched as sign(S r),
||r||; attention adds sqrt(pi/2)/jl ||r|| S^T s to each packed value.

Pinned by: brute-force sign bits (numpy), the unbiasedness of the
reconstruction (its mean over projections is r, so a one-token cache returns
the original vector on average), and no effect when no head asks for it."""
import math

import numpy as np

from oracle import oracle as O


def _one(seed_s, x, sign, vb=1):
    d = x.size
    seg = O.PackedSegment(1, 1, d, 16, [8], [vb], jl=d, qjl_v=[1])
    S = O.qjl_matrix(d, d, seed_s)
    X = x.astype(np.float16)[None, None, None]
    O.compress(seg, X, X, sign, S)
    seg.n_tokens = 1
    q = np.ones((1, 1, d), np.float16)
    return O.decode_attention([seg], q, sign, 1, S=S, jl=d)[0, 0], seg, S


def test_value_sketch_matches_brute_force():
    d, H, T = 32, 3, 9
    rng = np.random.default_rng(4)
    sign = O.signs(d, 3)
    S = O.qjl_matrix(d, d, 77)
    V = rng.standard_normal((1, H, T, d)).astype(np.float16)
    seg = O.PackedSegment(1, H, d, 16, [2] * H, [1, 2, 3], jl=d, qjl_v=[1, 0, 1])
    O.compress(seg, V, V, sign, S)
    Sd = S.astype(np.float64)
    checked = 0
    for h in (0, 2):
        vb = int(seg.vbits[h])
        c32, _ = O.codebook_f32(vb)
        for t in range(T):
            y = O.rotate_f32(V[0, h, t].astype(np.float32), sign)
            codes, sg = O.quant_value(y[None], vb)
            r = (y - (np.float32(sg[0]) * c32[codes[0]]).astype(np.float32)).astype(np.float32)
            p = Sd @ r.astype(np.float64)
            qi = seg.vqjl_rank(h) * seg.capacity + t
            bits = np.unpackbits(seg.vqjl_signs[qi * (d // 8):(qi + 1) * (d // 8)], bitorder="little")
            sure = np.abs(p) > 1e-9 * np.linalg.norm(r)
            assert np.array_equal(bits[sure], (p[sure] >= 0).astype(np.uint8))
            assert abs(float(seg.vqjl_norm[qi]) - np.linalg.norm(r.astype(np.float64))) <= 1e-6 * np.linalg.norm(r)
            checked += 1
    assert checked == 2 * T
    assert seg.nv == 2 and not seg.vqjl_signs[2 * 16 * (d // 8):].any()


def test_value_reconstruction_is_unbiased():
    # one token: the output is R^T vhat; E over projections of vhat is y, so the
    # mean output is the rotated-back binary32 vector (the fp16 input, to rounding)
    d = 16
    rng = np.random.default_rng(9)
    sign = O.signs(d, 5)
    x = rng.standard_normal(d).astype(np.float16).astype(np.float64)
    n = 1500
    outs = np.array([_one(3000 + i, x, sign)[0] for i in range(n)])
    mean, sd = outs.mean(0), outs.std(0) / math.sqrt(n)
    assert np.all(np.abs(mean - x) < 5 * sd + 1e-6), (np.abs(mean - x) / sd).max()
    # and without the correction the one-token output is the 1-bit reconstruction, far from x
    plain = O.PackedSegment(1, 1, d, 16, [8], [1], jl=d)
    X = x.astype(np.float16)[None, None, None]
    O.compress(plain, X, X, sign, None)
    plain.n_tokens = 1
    out0 = O.decode_attention([plain], np.ones((1, 1, d), np.float16), sign, 1)[0, 0]
    assert np.abs(out0 - x).max() > 20 * sd.max()


def test_no_value_sketch_no_change():
    d, H, T = 16, 2, 7
    rng = np.random.default_rng(2)
    sign = O.signs(d, 1)
    S = O.qjl_matrix(d, d, 5)
    K = rng.standard_normal((1, H, T, d)).astype(np.float16)
    V = rng.standard_normal((1, H, T, d)).astype(np.float16)
    q = rng.standard_normal((1, 4, d)).astype(np.float16)
    outs = []
    for qv in (None, [0, 0]):
        seg = O.PackedSegment(1, H, d, 16, [2, 3], [1, 2], qjl=[1, 0], jl=d, qjl_v=qv)
        O.compress(seg, K, V, sign, S)
        outs.append(O.decode_attention([seg], q, sign, H, S=S, jl=d))
    assert np.array_equal(outs[0], outs[1])
