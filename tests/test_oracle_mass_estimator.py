"""Pins of two decode-side outputs of the oracle.

Attention mass ("TurboMOQ", "Attention-weighted tier demotion": tiers follow
the real attention weights of each decode step): the softmax weight of every
cached token, averaged over the query heads that read its KV head.  Pinned by
the probability axioms, by torch.softmax over keys rebuilt through an explicit
Hadamard matrix, and by the attention output itself (one-hot values turn the
output into the weights).

Sign-pair QJL estimator ("turboquant-mlx", "RaBitQ vs QJL correction": pi/2
times both scales times the sign agreement): pinned by Sheppard's formula
E[sign(<s, a>) sign(<s, b>)] = 1 - 2 theta / pi for Gaussian s, so the
correction averages ||q'|| ||r|| (pi/2 - theta) over projections.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import torch

from oracle import oracle as O


def _R(d, sign):
    H = scipy.linalg.hadamard(d).astype(np.float64)
    D = np.diag(sign.astype(np.float64))
    return D @ H @ D / math.sqrt(d)


def _keys_by_definition(seg, sign, b, h):
    """Key vectors of a packed segment (no QJL) in the original space, from
    numpy bit unpacking and the explicit rotation matrix."""
    d, kb = seg.d, int(seg.kbits[h])
    R = _R(d, sign)
    out = []
    for t in range(seg.n_tokens):
        o = seg.code_offset("k", b, h, t)
        bits = np.unpackbits(seg.kcodes[o:o + d * kb // 8], bitorder="little").reshape(d, kb)
        c = (bits.astype(np.int64) << np.arange(kb)).sum(1)
        m = float(seg.kscale[(b * seg.H + h) * seg.capacity + t])
        out.append(R @ (m * ((c + 0.5) * 2.0 ** (1 - kb) - 1)))
    return np.array(out)


def _case(seed, d=16, H=2, Hq=4, T_sink=5, T_pack=9, kb=3, vb=2):
    rng = np.random.default_rng(seed)
    sign = O.signs(d, 42)
    sink = O.Fp16Segment(1, H, d, T_sink, n_tokens=T_sink)
    Ks = rng.standard_normal((1, H, T_sink, d)).astype(np.float16)
    Vs = rng.standard_normal((1, H, T_sink, d)).astype(np.float16)
    sink.k16[:] = Ks.ravel().view(np.uint16)
    sink.v16[:] = Vs.ravel().view(np.uint16)
    seg = O.PackedSegment(1, H, d, 16, [kb] * H, [vb] * H, jl=d)
    K = (2 * rng.standard_normal((1, H, T_pack, d))).astype(np.float16)
    V = rng.standard_normal((1, H, T_pack, d)).astype(np.float16)
    O.compress(seg, K, V, sign, None)
    seg.n_tokens = T_pack
    q = (1.5 * rng.standard_normal((1, Hq, d))).astype(np.float16)
    return sign, sink, Ks, seg, q


def test_mass_is_a_distribution_over_all_segments():
    for seed in range(4):
        sign, sink, Ks, seg, q = _case(seed)
        _, mass = O.decode_attention([sink, seg], q, sign, 2, with_mass=True)
        total = mass[0].sum(axis=2) + mass[1].sum(axis=2)
        assert np.allclose(total, 1.0, atol=1e-14)
        assert all((m >= 0).all() for m in mass)


def test_mass_matches_torch_softmax_of_rebuilt_keys():
    d, H, Hq = 16, 2, 4
    g = Hq // H
    sign, sink, Ks, seg, q = _case(7, d=d, H=H, Hq=Hq)
    _, mass = O.decode_attention([sink, seg], q, sign, H, with_mass=True)
    for h in range(H):
        keys = np.concatenate([Ks[0, h].astype(np.float64), _keys_by_definition(seg, sign, 0, h)])
        qs = torch.tensor(q[0, h * g:(h + 1) * g].astype(np.float64))
        p = torch.softmax(qs @ torch.tensor(keys).T / math.sqrt(d), dim=1).mean(0).numpy()
        assert np.allclose(mass[0][0, h], p[:sink.n_tokens], rtol=1e-12, atol=0)
        assert np.allclose(mass[1][0, h], p[sink.n_tokens:], rtol=1e-12, atol=0)


def test_mass_equals_output_under_one_hot_values():
    # one query head per KV head and values e_t: out[t] = p(t) = mass[t]
    d, H, T = 16, 3, 11
    rng = np.random.default_rng(3)
    sign = O.signs(d, 5)
    seg = O.Fp16Segment(1, H, d, T, n_tokens=T)
    K = rng.standard_normal((1, H, T, d)).astype(np.float16)
    V = np.zeros((1, H, T, d), np.float16)
    for t in range(T):
        V[0, :, t, t] = 1.0
    seg.k16[:] = K.ravel().view(np.uint16)
    seg.v16[:] = V.ravel().view(np.uint16)
    q = rng.standard_normal((1, H, d)).astype(np.float16)
    out, mass = O.decode_attention([seg], q, sign, H, with_mass=True)
    assert np.allclose(out[0, :, :T], mass[0][0], rtol=1e-13, atol=0)
    # a dominant key takes (almost) all the mass
    K[0, 1, 4] = (40 * q[0, 1] / np.linalg.norm(q[0, 1].astype(np.float64))).astype(np.float16)
    seg.k16[:] = K.ravel().view(np.uint16)
    _, mass = O.decode_attention([seg], q, sign, H, with_mass=True)
    assert mass[0][0, 1, 4] > 0.999


def test_sign_pair_estimator_leaves_heads_without_sketch_alone():
    sign, sink, Ks, seg, q = _case(11)
    a = O.decode_attention([sink, seg], q, sign, 2, S=O.qjl_matrix(16, 16, 1), jl=16, estimator=0)
    b = O.decode_attention([sink, seg], q, sign, 2, S=O.qjl_matrix(16, 16, 1), jl=16, estimator=1)
    assert np.array_equal(a, b)


def _packed_score_correction(estimator, S, d, k, q, sign, qk_sink):
    """The QJL term the oracle adds to q.k of one 1-bit QJL key, read back from
    the attention mass against an fp16 sink token whose score is exact."""
    seg = O.PackedSegment(1, 1, d, 16, [1], [1], qjl=[1], jl=d)
    O.compress(seg, k[None, None, None], np.zeros((1, 1, 1, d), np.float16), sign, S)
    seg.n_tokens = 1
    sink = O.Fp16Segment(1, 1, d, 1, n_tokens=1)
    sink.k16[:] = qk_sink.view(np.uint16)
    _, mass = O.decode_attention([sink, seg], q[None, None], sign, 1, S=S, jl=d, estimator=estimator,
                                 with_mass=True)
    s_sink = float(q.astype(np.float64) @ qk_sink.astype(np.float64)) / math.sqrt(d)
    s_pack = s_sink + math.log(mass[1][0, 0, 0] / mass[0][0, 0, 0])
    base = float(q.astype(np.float64) @ _keys_by_definition(seg, sign, 0, 0)[0])
    return s_pack * math.sqrt(d) - base


def test_sign_pair_estimator_mean_follows_sheppard():
    d = 16
    rng = np.random.default_rng(21)
    sign = O.signs(d, 9)
    k = rng.standard_normal(d).astype(np.float16)
    # the residual of the 1-bit key code, computed as the compressor does (binary32)
    y = O.rotate_f32(k.astype(np.float32), sign)
    codes, m = O.quant_key(y, 1)
    r = (y - (m * O.key_levels(1)[codes]).astype(np.float32)).astype(np.float64)
    rho = np.linalg.norm(r)
    # a query whose rotated image makes an angle well below 90 degrees with r
    R = _R(d, sign)
    q = (R @ (2.0 * r / rho + 0.12 * rng.standard_normal(d))).astype(np.float16)
    qr = R @ q.astype(np.float64)
    theta = math.acos(qr @ r / np.linalg.norm(qr) / rho)
    sink = rng.standard_normal(d).astype(np.float16)
    n = 1500
    vals = [_packed_score_correction(1, O.qjl_matrix(d, d, 5000 + i), d, k, q, sign, sink) for i in range(n)]
    mean, sd = np.mean(vals), np.std(vals) / math.sqrt(n)
    want = np.linalg.norm(qr) * rho * (math.pi / 2 - theta)
    assert abs(mean - want) < 5 * sd, (mean, want, sd)
    # and not the plain inner product (the two differ by far more than the noise here)
    assert abs(want - qr @ r) > 10 * sd
    # the unbiased estimator's mean is the inner product itself
    vals0 = [_packed_score_correction(0, O.qjl_matrix(d, d, 5000 + i), d, k, q, sign, sink) for i in range(n)]
    assert abs(np.mean(vals0) - qr @ r) < 5 * np.std(vals0) / math.sqrt(n)


def test_sign_pair_estimator_is_invariant_to_projection_scale():
    # the sign agreement and ||q'|| do not see the scale of S; the unbiased estimator does
    d = 16
    rng = np.random.default_rng(4)
    sign = O.signs(d, 9)
    k = rng.standard_normal(d).astype(np.float16)
    q = rng.standard_normal(d).astype(np.float16)
    sink = rng.standard_normal(d).astype(np.float16)
    S = O.qjl_matrix(d, d, 77)
    a = _packed_score_correction(1, S, d, k, q, sign, sink)
    b = _packed_score_correction(1, (4 * S).astype(np.float32), d, k, q, sign, sink)
    assert abs(a - b) < 1e-9 * max(1.0, abs(a))
    a0 = _packed_score_correction(0, S, d, k, q, sign, sink)
    b0 = _packed_score_correction(0, (4 * S).astype(np.float32), d, k, q, sign, sink)
    assert abs(b0 - 4 * a0) < 1e-6 * max(1.0, abs(a0))
