"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Compression: codes bit-exact; scales bit-exact (the binary32 order is part of
the format); QJL sign bits exact except where |(S r)_j| <= 1e-6 ||S_j|| rho
(counted, < 1e-5 of all bits).  Dequantization: rotated values bit-exact,
original-space values within 1e-5 max(1, |x|).  Attention: per query head,
max|o - o_ref| / max|o_ref| <= 2e-3 against the binary64 oracle over the same
packed cache (the oracle's own compression of the same input, uploaded)."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as O
from rotated_quantized_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3


@pytest.fixture(scope="module")
def tq():
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq as T
    return T


def _kv(B, H, T, seed, law="outliers"):
    w = W.Workload("t", layers=1, batch=B, context=T, kv_heads=H, law=law)
    return W.kv_block(w, 0, B, T, seed)


def _oracle_segment(B, H, cap, kb, vb, qjl, K, V, sign, S, t_begin=0, law=0, qjl_v=None):
    seg = O.PackedSegment(B, H, 128, cap, kb, vb, qjl, jl=128, law=law, qjl_v=qjl_v)
    O.compress(seg, K.numpy().view(np.uint16), V.numpy().view(np.uint16), sign, S, t_begin=t_begin)
    return seg


def _upload(tq, oseg, layout, n_tokens):
    g = tq.PackedSegment(layout, n_tokens=n_tokens)
    g.kcodes.copy_(torch.from_numpy(oseg.kcodes))
    g.vcodes.copy_(torch.from_numpy(oseg.vcodes))
    g.kscale.copy_(torch.from_numpy(oseg.kscale))
    g.vscale.copy_(torch.from_numpy(oseg.vscale))
    if g.qjl_signs is not None:
        g.qjl_signs.copy_(torch.from_numpy(oseg.qjl_signs))
        g.qjl_norm.copy_(torch.from_numpy(oseg.qjl_norm))
    if g.vqjl_signs is not None:
        g.vqjl_signs.copy_(torch.from_numpy(oseg.vqjl_signs))
        g.vqjl_norm.copy_(torch.from_numpy(oseg.vqjl_norm))
    return g


def _qjl_window_ok(oseg, gseg_signs, K, sign, S, B, H, T, t_begin):
    """Sign-bit mismatches must sit in the 1e-6 window around zero."""
    got = gseg_signs.cpu().numpy()
    bad = np.flatnonzero(got != oseg.qjl_signs)
    if bad.size == 0:
        return 0
    Sd = S.astype(np.float64)
    rown = np.linalg.norm(Sd, axis=1)
    mism = 0
    for byte in bad:
        rec = byte // 16
        pos = rec % oseg.capacity
        bq = rec // oseg.capacity
        b, q = divmod(bq, oseg.nq)
        h = [hh for hh in range(H) if oseg.qjl[hh] and oseg.qjl_rank(hh) == q][0]
        x = K[b, h, pos - t_begin].float().numpy()
        y = O.rotate_f32(x, sign)
        codes, m = O.quant_key(y, int(oseg.kbits[h]))
        yh = (m * O.key_levels(int(oseg.kbits[h]))[codes]).astype(np.float32)
        r = (y - yh).astype(np.float32)
        p = Sd @ r.astype(np.float64)
        rho = np.linalg.norm(r.astype(np.float64))
        diff = got[byte] ^ oseg.qjl_signs[byte]
        for bit in range(8):
            if (diff >> bit) & 1:
                j = (byte % 16) * 8 + bit
                assert abs(p[j]) <= 1e-6 * rown[j] * rho, (b, h, pos, j, p[j])
                mism += 1
    return mism


COMPRESS_CASES = [
    # B, H, T, t_begin, kbits, vbits, qjl, value codebook law
    (2, 8, 200, 0, [1, 2, 3, 4, 5, 6, 7, 8], [8, 7, 6, 5, 4, 3, 2, 1], None, 0),
    (1, 8, 64, 16, [4] * 8, [4] * 8, None, 0),
    (3, 4, 77, 32, [1, 2, 2, 3], [1, 3, 2, 4], [1, 1, 0, 0], 0),
    (1, 8, 130, 0, [8, 3, 2, 1, 5, 7, 6, 4], [3, 1, 8, 2, 6, 4, 5, 7], [0, 0, 1, 1, 0, 0, 0, 1], 0),
    (2, 8, 150, 16, [4, 4, 3, 3, 2, 2, 1, 8], [1, 2, 3, 4, 5, 6, 7, 8], [0, 0, 0, 0, 1, 0, 0, 0], 1),
    (1, 4, 90, 0, [1, 2, 1, 2], [3, 2, 3, 5], [1, 1, 1, 1], 0),  # every head sketched
    # no sketches: the one-thread-per-vector kernels, every width, both codebook laws
    (2, 8, 150, 16, [2, 4, 6, 8, 1, 3, 5, 7], [1, 2, 3, 4, 5, 6, 7, 8], None, 1),
    (3, 2, 33, 7, [3, 3], [3, 3], None, 0),
]


@pytest.mark.parametrize("B,H,T,t_begin,kb,vb,qjl,law", COMPRESS_CASES)
def test_compress_bit_exact(tq, B, H, T, t_begin, kb, vb, qjl, law):
    K, V = _kv(B, H, T, seed=11 + T)
    cap = ((t_begin + T + 15) // 16) * 16
    sign = O.signs(128, 42)
    S = O.qjl_matrix(128, 128, 42 + 1000) if qjl else None
    oseg = _oracle_segment(B, H, cap, kb, vb, qjl, K, V, sign, S, t_begin, law=law)
    layout = tq.make_layout(B, H, 128, cap, kb, vb, qjl, value_law=law)
    g = tq.PackedSegment(layout)
    rot = tq.tq_make_rotation(128, 42)
    Sd = torch.from_numpy(S).cuda() if qjl else None
    tq.tq_compress(g, rot, K.cuda(), V.cuda(), t_begin=t_begin, qjl_S=Sd)
    torch.cuda.synchronize()
    assert np.array_equal(g.kcodes.cpu().numpy(), oseg.kcodes)
    assert np.array_equal(g.vcodes.cpu().numpy(), oseg.vcodes)
    assert np.array_equal(g.kscale.cpu().numpy().view(np.uint32), oseg.kscale.view(np.uint32))
    assert np.array_equal(g.vscale.cpu().numpy().view(np.uint32), oseg.vscale.view(np.uint32))
    if qjl:
        n = _qjl_window_ok(oseg, g.qjl_signs, K, sign, S, B, H, T, t_begin)
        assert n <= 1e-5 * oseg.qjl_signs.size * 8
        assert np.allclose(g.qjl_norm.cpu().numpy(), oseg.qjl_norm, rtol=1e-5, atol=0)


VALUE_SKETCH_CASES = [
    # B, H, T, t_begin, kbits, vbits, key qjl, value qjl
    (2, 4, 90, 16, [2, 1, 3, 2], [1, 2, 1, 3], [1, 0, 0, 1], [1, 1, 0, 1]),
    (1, 8, 130, 0, [1] * 8, [1, 2, 3, 4, 5, 6, 7, 8], None, [1, 0, 1, 0, 1, 0, 1, 1]),
]


def _value_window_ok(oseg, gsigns, V, sign, S, B, H, t_begin):
    """Value-sketch sign mismatches must sit in the 1e-6 window around zero."""
    got = gsigns.cpu().numpy()
    bad = np.flatnonzero(got != oseg.vqjl_signs)
    Sd = S.astype(np.float64)
    rown = np.linalg.norm(Sd, axis=1)
    n = 0
    for byte in bad:
        rec = byte // 16
        pos = rec % oseg.capacity
        b, v = divmod(rec // oseg.capacity, oseg.nv)
        h = [hh for hh in range(H) if oseg.qjl_v[hh] and oseg.vqjl_rank(hh) == v][0]
        y = O.rotate_f32(V[b, h, pos - t_begin].float().numpy(), sign)
        codes, sg = O.quant_value(y[None], int(oseg.vbits[h]))
        c32, _ = O.codebook_f32(int(oseg.vbits[h]))
        r = (y - (np.float32(sg[0]) * c32[codes[0]]).astype(np.float32)).astype(np.float64)
        p = Sd @ r
        diff = got[byte] ^ oseg.vqjl_signs[byte]
        for bit in range(8):
            if (diff >> bit) & 1:
                j = (byte % 16) * 8 + bit
                assert abs(p[j]) <= 1e-6 * rown[j] * np.linalg.norm(r), (b, h, pos, j)
                n += 1
    return n


@pytest.mark.parametrize("B,H,T,t_begin,kb,vb,qjl,qjl_v", VALUE_SKETCH_CASES)
def test_compress_value_sketch(tq, B, H, T, t_begin, kb, vb, qjl, qjl_v):
    K, V = _kv(B, H, T, seed=70 + T)
    cap = ((t_begin + T + 15) // 16) * 16
    sign = O.signs(128, 42)
    S = O.qjl_matrix(128, 128, 42 + 1000)
    oseg = _oracle_segment(B, H, cap, kb, vb, qjl, K, V, sign, S, t_begin, qjl_v=qjl_v)
    g = tq.PackedSegment(tq.make_layout(B, H, 128, cap, kb, vb, qjl, qjl_v=qjl_v))
    tq.tq_compress(g, tq.tq_make_rotation(128, 42), K.cuda(), V.cuda(), t_begin=t_begin,
                   qjl_S=torch.from_numpy(S).cuda())
    torch.cuda.synchronize()
    assert np.array_equal(g.vcodes.cpu().numpy(), oseg.vcodes)
    assert np.array_equal(g.vscale.cpu().numpy().view(np.uint32), oseg.vscale.view(np.uint32))
    n = _value_window_ok(oseg, g.vqjl_signs, V, sign, S, B, H, t_begin)
    assert n <= 1e-5 * oseg.vqjl_signs.size * 8
    assert np.allclose(g.vqjl_norm.cpu().numpy(), oseg.vqjl_norm, rtol=1e-5, atol=0)


def test_compress_edge_vectors(tq):
    # all-zero vectors, one-hot vectors (exact +-absmax), huge fp16 values
    B, H, T = 1, 8, 70
    K = torch.zeros(B, H, T, 128, dtype=torch.float16)
    V = torch.zeros(B, H, T, 128, dtype=torch.float16)
    K[0, :, 1, 5] = 1.0
    V[0, :, 1, 5] = -2.0
    K[0, :, 2] = 60000.0
    V[0, :, 2, ::2] = -60000.0
    K[0, :, 3:] = torch.randn(H, T - 3, 128).half()
    V[0, :, 3:] = torch.randn(H, T - 3, 128).half()
    kb = [1, 2, 3, 4, 5, 6, 7, 8]
    sign = O.signs(128, 42 + 3)
    oseg = _oracle_segment(B, H, 80, kb, kb[::-1], None, K, V, sign, None)
    layout = tq.make_layout(B, H, 128, 80, kb, kb[::-1])
    g = tq.PackedSegment(layout)
    tq.tq_compress(g, tq.tq_make_rotation(128, 42 + 3), K.cuda(), V.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(g.kcodes.cpu().numpy(), oseg.kcodes)
    assert np.array_equal(g.vcodes.cpu().numpy(), oseg.vcodes)
    assert np.array_equal(g.kscale.cpu().numpy(), oseg.kscale)
    assert np.array_equal(g.vscale.cpu().numpy(), oseg.vscale)


def test_compress_chunked_equals_one_shot(tq):
    # "Dynamic Chunk Buffering": compressing 64 tokens at a time gives the same bytes
    B, H, T = 1, 8, 256
    K, V = _kv(B, H, T, seed=5)
    layout = tq.make_layout(B, H, 128, T, 8, 3)
    rot = tq.tq_make_rotation(128, 42)
    a, c = tq.PackedSegment(layout), tq.PackedSegment(layout)
    Kc, Vc = K.cuda(), V.cuda()
    tq.tq_compress(a, rot, Kc, Vc)
    for t0 in range(0, T, 64):
        tq.tq_compress(c, rot, Kc[:, :, t0:t0 + 64], Vc[:, :, t0:t0 + 64], t_begin=t0)
    torch.cuda.synchronize()
    for x, y in ((a.kcodes, c.kcodes), (a.vcodes, c.vcodes), (a.kscale, c.kscale), (a.vscale, c.vscale)):
        assert torch.equal(x, y)


def test_compress_strided_input(tq):
    # K, V viewed from a [B][T][H][d] tensor (token-major layout)
    B, H, T = 2, 8, 100
    base = torch.randn(2, B, T, H, 128).half()
    K = base[0].permute(0, 2, 1, 3)
    V = base[1].permute(0, 2, 1, 3)
    sign = O.signs(128, 42)
    oseg = _oracle_segment(B, H, 112, [3] * 8, [3] * 8, None, K.contiguous(), V.contiguous(), sign, None)
    g = tq.PackedSegment(tq.make_layout(B, H, 128, 112, 3, 3))
    bc = base.cuda()
    tq.tq_compress(g, tq.tq_make_rotation(128, 42), bc[0].permute(0, 2, 1, 3), bc[1].permute(0, 2, 1, 3))
    torch.cuda.synchronize()
    assert np.array_equal(g.kcodes.cpu().numpy(), oseg.kcodes)
    assert np.array_equal(g.vcodes.cpu().numpy(), oseg.vcodes)


@pytest.mark.parametrize("law", [0, 1])
def test_dequantize(tq, law):
    B, H, T = 2, 8, 90
    kb = [1, 2, 3, 4, 5, 6, 7, 8]
    vb = [2, 3, 4, 5, 6, 7, 8, 1]
    K, V = _kv(B, H, T, seed=3)
    sign = O.signs(128, 42)
    oseg = _oracle_segment(B, H, 96, kb, vb, None, K, V, sign, None, law=law)
    layout = tq.make_layout(B, H, 128, 96, kb, vb, value_law=law)
    g = _upload(tq, oseg, layout, T)
    rot = tq.tq_make_rotation(128, 42)
    kr, vr, ko, vo = tq.tq_dequantize(g, 5, T - 5, rot=rot, rotated=True, original=True)
    torch.cuda.synchronize()
    for b in range(B):
        for h in range(H):
            ok, ov = O.dequant(oseg, b, h, 5, T - 5)
            assert np.array_equal(kr[b, h].cpu().numpy(), ok)
            assert np.array_equal(vr[b, h].cpu().numpy(), ov)
            for got, y in ((ko, ok), (vo, ov)):
                x = O.rotate_f64(y.astype(np.float64), sign)
                err = np.abs(got[b, h].cpu().numpy() - x)
                assert np.all(err <= 1e-5 * np.maximum(1.0, np.abs(x)))


def _max_rel(out, ref):
    o = out.reshape(-1, out.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    return (np.abs(o - r).max(axis=1) / np.maximum(np.abs(r).max(axis=1), 1e-30)).max()


MASS_RTOL = 1e-4  # binary32 scores: |ds| ~ 1e-5 in log units at these magnitudes


def _attention_case(tq, L, B, H, Hq, spec, seed, qjl_any=False, estimator=0, mass=False):
    """spec: list of segments per layer: ('fp16', T) or ('packed', T, kb, vb, qjl[, law[, qjl_v]]).
    mass: every segment gets an attention-mass buffer, checked against the oracle's."""
    rng = np.random.default_rng(seed)
    S = O.qjl_matrix(128, 128, 42 + 1000) if qjl_any else None
    Sd = torch.from_numpy(S).cuda() if qjl_any else None
    views, oracle_layers, keep = [], [], []
    for l in range(L):
        sign = O.signs(128, 42 + l)
        rot = tq.tq_make_rotation(128, 42 + l)
        osegs, gsegs = [], []
        for si, sp in enumerate(spec):
            T = sp[1]
            cap = max(16, ((T + 15) // 16) * 16)
            K, V = _kv(B, H, max(T, 1), seed=seed * 100 + l * 10 + si)
            if sp[0] == "fp16":
                o = O.Fp16Segment(B, H, 128, cap, n_tokens=T)
                kk = np.zeros((B, H, cap, 128), np.float16)
                vv = np.zeros((B, H, cap, 128), np.float16)
                kk[:, :, :T] = K.numpy()[:, :, :T]
                vv[:, :, :T] = V.numpy()[:, :, :T]
                o.k16[:] = kk.ravel().view(np.uint16)
                o.v16[:] = vv.ravel().view(np.uint16)
                g = tq.Fp16Segment(B, H, 128, cap, n_tokens=T, k=torch.from_numpy(kk).cuda(),
                                   v=torch.from_numpy(vv).cuda())
            else:
                kb, vb, qj = sp[2:5]
                law = sp[5] if len(sp) > 5 else 0
                qv = sp[6] if len(sp) > 6 else None
                o = O.PackedSegment(B, H, 128, cap, kb, vb, qj, jl=128, law=law, qjl_v=qv)
                if T:
                    O.compress(o, K.numpy().view(np.uint16), V.numpy().view(np.uint16), sign, S)
                o.n_tokens = T
                g = _upload(tq, o, tq.make_layout(B, H, 128, cap, kb, vb, qj, value_law=law, qjl_v=qv), T)
            if mass:  # -1 marks entries the call must leave alone
                g.attn_mass = torch.full((B, H, cap), -1.0, device="cuda")
            osegs.append(o)
            gsegs.append(g)
        keep.append(gsegs)
        views.append(tq.layer_view(rot, gsegs, qjl_estimator=estimator))
        oracle_layers.append((osegs, sign))
    q = torch.from_numpy(rng.standard_normal((L, B, Hq, 128)).astype(np.float16))
    out = torch.empty(L, B, Hq, 128, device="cuda")
    ws = torch.empty(tq.tq_decode_workspace_size(views, B, H, Hq, 128), dtype=torch.uint8, device="cuda")
    tq.tq_decode_attention(views, q.cuda(), out, ws, H, qjl_S=Sd)
    assert tq.tq_decode_error_flag(ws) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    worst = 0.0
    for l in range(L):
        osegs, sign = oracle_layers[l]
        if estimator == 1 and S is not None:
            # the query's sign decisions must be unique: no |(S q')_j| inside the
            # binary32 error bound of the kernels' q' and S q' (~(7 + 128) 2^-24
            # relative) around zero; the seed is chosen so that none is
            Sd = S.astype(np.float64)
            qr = np.stack([O.rotate_f64(x.astype(np.float64), sign) for x in q[l].numpy().reshape(-1, 128)])
            t = qr @ Sd.T
            rel = np.abs(t) / np.linalg.norm(Sd, axis=1)[None] / np.linalg.norm(qr, axis=1)[:, None]
            assert rel.min() > 1e-5, rel.min()
        ref = O.decode_attention(osegs, q[l].numpy(), sign, H, S=S, estimator=estimator, with_mass=mass)
        if mass:
            ref, ref_mass = ref
            for g, rm in zip(keep[l], ref_mass):
                gm = g.attn_mass.cpu().numpy()
                n = g.n_tokens
                assert np.all(gm[:, :, n:] == -1.0)
                err = np.abs(gm[:, :, :n] - rm)
                assert np.all(err <= MASS_RTOL * rm + 1e-30), (err / np.maximum(rm, 1e-30)).max()
        if all(s.n_tokens == 0 for s in osegs):
            assert np.all(got[l] == 0)
            continue
        worst = max(worst, _max_rel(got[l], ref))
    return worst


ATTN_CASES = [
    # L, B, H, Hq, segments
    (1, 1, 8, 32, [("packed", 1024, [4] * 8, [4] * 8, None)]),
    (2, 2, 2, 8, [("fp16", 10), ("packed", 300, [3, 5], [2, 8], None), ("fp16", 7)]),
    (1, 2, 4, 8, [("packed", 200, [1, 2, 3, 4], [1, 2, 3, 4], None), ("packed", 129, [5, 6, 7, 8], [8, 7, 6, 5], None)]),
    (1, 1, 8, 8, [("packed", 333, [8, 3, 2, 1, 5, 7, 6, 4], [3, 1, 8, 2, 6, 4, 5, 7], None)]),
    (2, 1, 4, 16, [("fp16", 64), ("packed", 190, [2, 1, 4, 3], [3, 4, 1, 2], [1, 1, 0, 0])]),
    # both value codebook laws in one call: same widths, separate decode classes
    (1, 2, 4, 8, [("packed", 260, [4, 3, 2, 8], [1, 2, 3, 4], None, 1),
                  ("packed", 140, [4, 3, 2, 8], [1, 2, 3, 4], None, 0), ("fp16", 5)]),
    (1, 1, 8, 32, [("packed", 500, [3] * 8, [1, 3, 5, 6, 7, 8, 2, 4], [1, 0, 0, 0, 0, 0, 0, 1], 1)]),
]


@pytest.mark.parametrize("L,B,H,Hq,spec", ATTN_CASES)
def test_decode_attention_matches_oracle(tq, L, B, H, Hq, spec):
    qjl_any = any(s[0] == "packed" and s[4] and any(s[4]) for s in spec)
    worst = _attention_case(tq, L, B, H, Hq, spec, seed=len(spec) * 7 + L, qjl_any=qjl_any)
    assert worst <= ATTN_TOL, worst


MASS_CASES = [
    # L, B, H, Hq, segments
    (2, 2, 2, 8, [("fp16", 10), ("packed", 300, [3, 5], [2, 8], None), ("fp16", 7)]),
    (1, 3, 4, 8, [("packed", 200, [1, 2, 3, 4], [1, 2, 3, 4], [1, 1, 0, 0]),
                  ("packed", 129, [5, 6, 7, 8], [8, 7, 6, 5], None), ("fp16", 0)]),
    (1, 1, 8, 8, [("packed", 333, [8, 3, 2, 1, 5, 7, 6, 4], [3, 1, 8, 2, 6, 4, 5, 7], None, 1)]),
    (1, 2, 8, 16, [("fp16", 1100), ("packed", 2100, [3] * 8, [3] * 8, None), ("fp16", 37)]),
]


@pytest.mark.parametrize("L,B,H,Hq,spec", MASS_CASES)
def test_attention_mass_matches_oracle(tq, L, B, H, Hq, spec):
    qjl_any = any(s[0] == "packed" and s[4] and any(s[4]) for s in spec)
    worst = _attention_case(tq, L, B, H, Hq, spec, seed=40 + len(spec), qjl_any=qjl_any, mass=True)
    assert worst <= ATTN_TOL, worst


@pytest.mark.parametrize("spec", [
    [("packed", 190, [2, 1, 4, 3], [3, 4, 1, 2], [1, 1, 0, 0]), ("fp16", 20)],
    [("packed", 260, [1] * 4, [2] * 4, [1] * 4), ("packed", 70, [2] * 4, [1] * 4, [1, 0, 1, 0])],
])
def test_decode_attention_sign_pair_estimator(tq, spec):
    # same sketch, the sign-pair score term; the mass kernel follows it too
    w = _attention_case(tq, 1, 2, 4, 16, spec, seed=67, qjl_any=True, estimator=1, mass=True)
    assert w <= ATTN_TOL, w


@pytest.mark.parametrize("L,B,H,Hq,spec", [
    (1, 2, 4, 16, [("packed", 300, [2, 1, 2, 1], [1, 1, 2, 1], [1, 1, 0, 0], 0, [1, 1, 1, 0]), ("fp16", 9)]),
    (2, 1, 8, 32, [("packed", 1500, [1] * 8, [1] * 8, [1] * 8, 0, [1] * 8),
                   ("packed", 200, [3] * 8, [2] * 8, None, 1, [0, 1, 0, 1, 0, 1, 0, 1])]),
])
def test_decode_attention_value_sketch(tq, L, B, H, Hq, spec):
    # QJL on values: the correction pass adds R (sqrt(pi/2)/jl S^T z) to the output
    w = _attention_case(tq, L, B, H, Hq, spec, seed=90 + L, qjl_any=True, mass=True)
    assert w <= ATTN_TOL, w


def test_decode_attention_empty_and_single_token(tq):
    # a layer with no tokens gives zeros; a single token returns its value
    assert _attention_case(tq, 1, 1, 2, 8, [("fp16", 0), ("packed", 0, [3, 3], [3, 3], None)], seed=1) == 0.0
    w = _attention_case(tq, 1, 1, 2, 8, [("packed", 1, [4, 4], [4, 4], None)], seed=2)
    assert w <= ATTN_TOL
    w = _attention_case(tq, 1, 2, 2, 2, [("fp16", 1)], seed=3)
    assert w <= ATTN_TOL


def test_decode_attention_tiers(tq):
    # progressive tiers on a short context: fp16 newest, then K4V4, K3V2, K2V1
    T = 3000
    tiers = tq.tq_age_tiers(T, [256, 1024, 2048])
    spec = []
    for tier, (s, e) in enumerate(tiers):
        if e > s:
            kb, vb = W.tier_bits(tier)
            spec.append(("fp16", e - s) if kb == 16 else ("packed", e - s, [kb] * 8, [vb] * 8, None))
    assert _attention_case(tq, 1, 1, 8, 32, spec, seed=9) <= ATTN_TOL


REQUANT_CASES = [
    # B, H, T, src kbits, src vbits, dst kbits, dst vbits
    (2, 4, 70, [4, 4, 4, 4], [4, 4, 4, 4], [3, 3, 3, 3], [2, 2, 2, 2]),   # warm -> cold tier
    (1, 8, 45, [3] * 8, [2] * 8, [2] * 8, [1] * 8),                       # cold -> archive tier
    (1, 8, 33, [8, 7, 6, 5, 4, 3, 2, 1], [1, 2, 3, 4, 5, 6, 7, 8], [1, 2, 3, 4, 5, 6, 7, 8],
     [8, 7, 6, 5, 4, 3, 2, 1]),                                            # every width pair shape
    (2, 2, 16, [5, 5], [5, 5], [5, 5], [5, 5]),                            # same widths
]

REQUANT_LAW_CASES = [
    # B, H, T, src kbits, src vbits, dst kbits, dst vbits, src law, dst law
    (2, 4, 70, [4] * 4, [4] * 4, [3] * 4, [2] * 4, 1, 1),
    (1, 4, 40, [4, 3, 2, 8], [4, 6, 1, 8], [2, 2, 1, 5], [3, 1, 1, 7], 0, 1),
    (1, 4, 40, [4, 3, 2, 8], [4, 6, 1, 8], [2, 2, 1, 5], [3, 1, 1, 7], 1, 0),
]


@pytest.mark.parametrize("B,H,T,skb,svb,dkb,dvb", REQUANT_CASES)
def test_requantize_bit_exact(tq, B, H, T, skb, svb, dkb, dvb):
    K, V = _kv(B, H, T, seed=300 + T)
    sign = O.signs(128, 42)
    scap = ((T + 20 + 15) // 16) * 16
    osrc = _oracle_segment(B, H, scap, skb, svb, None, K, V, sign, None, 20)
    gsrc = _upload(tq, osrc, tq.make_layout(B, H, 128, scap, skb, svb), 20 + T)
    dcap = ((T + 7 + 15) // 16) * 16
    odst = O.PackedSegment(B, H, 128, dcap, dkb, dvb)
    O.requantize(osrc, 20, T, odst, 7)
    gdst = tq.PackedSegment(tq.make_layout(B, H, 128, dcap, dkb, dvb))
    tq.tq_requantize(gsrc, 20, T, gdst, 7)
    torch.cuda.synchronize()
    assert np.array_equal(gdst.kcodes.cpu().numpy()[:odst.kcodes.size], odst.kcodes)
    assert np.array_equal(gdst.vcodes.cpu().numpy()[:odst.vcodes.size], odst.vcodes)
    assert np.array_equal(gdst.kscale.cpu().numpy()[:odst.kscale.size].view(np.uint32), odst.kscale.view(np.uint32))
    assert np.array_equal(gdst.vscale.cpu().numpy()[:odst.vscale.size].view(np.uint32), odst.vscale.view(np.uint32))


@pytest.mark.parametrize("B,H,T,skb,svb,dkb,dvb,slaw,dlaw", REQUANT_LAW_CASES)
def test_requantize_across_codebook_laws(tq, B, H, T, skb, svb, dkb, dvb, slaw, dlaw):
    K, V = _kv(B, H, T, seed=500 + T + slaw)
    sign = O.signs(128, 42)
    scap = ((T + 3 + 15) // 16) * 16
    osrc = _oracle_segment(B, H, scap, skb, svb, None, K, V, sign, None, 3, law=slaw)
    gsrc = _upload(tq, osrc, tq.make_layout(B, H, 128, scap, skb, svb, value_law=slaw), 3 + T)
    dcap = ((T + 15) // 16) * 16
    odst = O.PackedSegment(B, H, 128, dcap, dkb, dvb, law=dlaw)
    O.requantize(osrc, 3, T, odst, 0)
    gdst = tq.PackedSegment(tq.make_layout(B, H, 128, dcap, dkb, dvb, value_law=dlaw))
    tq.tq_requantize(gsrc, 3, T, gdst, 0)
    torch.cuda.synchronize()
    for got, ref in ((gdst.kcodes, odst.kcodes), (gdst.vcodes, odst.vcodes)):
        assert np.array_equal(got.cpu().numpy()[:ref.size], ref)
    for got, ref in ((gdst.kscale, odst.kscale), (gdst.vscale, odst.vscale)):
        assert np.array_equal(got.cpu().numpy()[:ref.size].view(np.uint32), ref.view(np.uint32))


def test_decode_reports_its_launches(tq):
    # query prep + one grid per packed class + the fp16 kernel (+ mass pass)
    B, H, Hq = 1, 2, 8
    rot = tq.tq_make_rotation(128, 42)
    K, V = _kv(B, H, 70, seed=5)
    segs = []
    for kb, vb in ((3, 3), (4, 2)):
        o = _oracle_segment(B, H, 80, [kb] * H, [vb] * H, None, K, V, O.signs(128, 42), None)
        o.n_tokens = 70
        segs.append(_upload(tq, o, tq.make_layout(B, H, 128, 80, [kb] * H, [vb] * H), 70))
    f16 = tq.Fp16Segment(B, H, 128, 16, n_tokens=9, k=torch.zeros(B, H, 16, 128, dtype=torch.float16, device="cuda"),
                         v=torch.zeros(B, H, 16, 128, dtype=torch.float16, device="cuda"))
    q = torch.randn(1, B, Hq, 128, device="cuda").half()
    out = torch.empty(1, B, Hq, 128, device="cuda")
    views = [tq.layer_view(rot, segs + [f16])]
    ws = torch.empty(tq.tq_decode_workspace_size(views, B, H, Hq, 128), dtype=torch.uint8, device="cuda")
    tq.tq_decode_attention(views, q, out, ws, H)
    assert tq.tq_decode_last_launches() == 1 + 2 + 1
    f16.attn_mass = torch.zeros(B, H, 16, device="cuda")
    views = [tq.layer_view(rot, segs + [f16])]
    ws = torch.empty(tq.tq_decode_workspace_size(views, B, H, Hq, 128), dtype=torch.uint8, device="cuda")
    tq.tq_decode_attention(views, q, out, ws, H)
    assert tq.tq_decode_last_launches() == 1 + 2 + 1 + 1
    torch.cuda.synchronize()
