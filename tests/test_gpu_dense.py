"""GPU parity of the dense Haar rotation ("TurboMOQ", "Stable QR Rotation"):
the tensor-core compression, dequantization through Q^T and decode attention
over dense-rotation layers, against the oracle given the same binary32 Q.

Compression tolerance (the method's own): codes equal the oracle's except at
coordinates within 1e-6 of a decision boundary, those counted; the tensor cores
add the 256 products of a coordinate (Q split in two fp16 parts) in an order
of their own, so y carries ~1e-7 relative error, which can move a coordinate
that sits on a boundary.  Scales follow y: within 4e-6 relative."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from rotated_quantized_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3
WINDOW = 1e-6       # distance to a decision boundary, in units of the normalised coordinate
SCALE_RTOL = 4e-6


@pytest.fixture(scope="module")
def tq():
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq as T
    return T


def _kv(B, H, T, seed, law="outliers"):
    w = W.Workload("t", layers=1, batch=B, context=T, kv_heads=H, law=law)
    return W.kv_block(w, 0, B, T, seed)


def _codes(rec, bits):
    return O.unpack(rec, bits, 128).astype(np.int64)


def _check_codes(gseg, oseg, K, V, Q, t_begin, T):
    """Codes of every (b, h, token) vector: equal, or the oracle's coordinate
    is within WINDOW of the boundary between the two codes.  Returns (mismatches, codes)."""
    kc, vc = gseg.kcodes.cpu().numpy(), gseg.vcodes.cpu().numpy()
    ks, vs = gseg.kscale.cpu().numpy(), gseg.vscale.cpu().numpy()
    B, H = oseg.B, oseg.H
    bad = total = 0
    for b in range(B):
        for h in range(H):
            kb, vb = int(oseg.kbits[h]), int(oseg.vbits[h])
            _, thr = O.codebook_sphere_f32(vb) if oseg.law else O.codebook_f32(vb)
            for t in range(T):
                pos = t_begin + t
                idx = (b * H + h) * oseg.capacity + pos
                for which, X, bits, codes_g, codes_o, sc_g, sc_o in (
                        ("k", K, kb, kc, oseg.kcodes, ks, oseg.kscale),
                        ("v", V, vb, vc, oseg.vcodes, vs, oseg.vscale)):
                    o = oseg.code_offset(which, b, h, pos)
                    cg = _codes(codes_g[o:o + 16 * bits], bits)
                    co = _codes(codes_o[o:o + 16 * bits], bits)
                    assert abs(float(sc_g[idx]) - float(sc_o[idx])) <= SCALE_RTOL * abs(float(sc_o[idx])), \
                        (which, b, h, t, sc_g[idx], sc_o[idx])
                    total += 128
                    diff = np.nonzero(cg != co)[0]
                    if diff.size == 0:
                        continue
                    y = O.rotate_dense_f32(X[b, h, t].float().numpy(), Q).astype(np.float64)
                    s = float(sc_o[idx])
                    for i in diff:
                        assert abs(cg[i] - co[i]) == 1, (which, b, h, t, i)
                        edge = max(cg[i], co[i])  # boundary between codes edge - 1 and edge
                        if which == "k":
                            u = y[i] / s
                            dist = abs(u - (edge * 2.0 ** (1 - bits) - 1.0))
                        else:
                            u = y[i] / s
                            dist = abs(u - float(thr[edge - 1]))
                        assert dist <= WINDOW, (which, b, h, t, i, dist)
                        bad += 1
    return bad, total


COMPRESS_CASES = [
    # B, H, T, t_begin, kbits, vbits, value law
    (2, 8, 300, 0, [1, 2, 3, 4, 5, 6, 7, 8], [8, 7, 6, 5, 4, 3, 2, 1], 0),
    (1, 4, 77, 16, [3, 3, 4, 2], [3, 2, 4, 1], 1),
    (3, 2, 129, 0, [4, 4], [4, 4], 0),
]


@pytest.mark.parametrize("B,H,T,t_begin,kb,vb,law", COMPRESS_CASES)
def test_dense_compress_matches_oracle(tq, B, H, T, t_begin, kb, vb, law):
    K, V = _kv(B, H, T, seed=900 + T)
    Q = O.haar_rotation(128, 42)
    cap = ((t_begin + T + 15) // 16) * 16
    oseg = O.PackedSegment(B, H, 128, cap, kb, vb, law=law)
    O.compress(oseg, K.numpy().view(np.uint16), V.numpy().view(np.uint16), O.signs(128, 42), None,
               t_begin=t_begin, Q=Q)
    Qd = torch.from_numpy(Q).cuda()
    rot = tq.dense_rotation(tq.tq_make_rotation(128, 42), Qd)
    g = tq.PackedSegment(tq.make_layout(B, H, 128, cap, kb, vb, value_law=law))
    tq.tq_compress_error_flag(reset=True)
    tq.tq_compress(g, rot, K.cuda(), V.cuda(), t_begin=t_begin)
    torch.cuda.synchronize()
    assert tq.tq_compress_error_flag() == 0
    bad, total = _check_codes(g, oseg, K, V, Q, t_begin, T)
    # bounded count at the widths in use; 8-bit grids have 255 boundaries per coordinate range
    assert bad <= max(2, 1e-4 * total), (bad, total)


def test_dense_compress_rejects_qjl_heads(tq):
    Q = torch.from_numpy(O.haar_rotation(128, 1)).cuda()
    rot = tq.dense_rotation(tq.tq_make_rotation(128, 1), Q)
    g = tq.PackedSegment(tq.make_layout(1, 2, 128, 16, [1, 2], [1, 2], [1, 0]))
    K = torch.zeros(1, 2, 4, 128, dtype=torch.float16, device="cuda")
    S = torch.from_numpy(O.qjl_matrix(128, 128, 5)).cuda()
    with pytest.raises(tq.TQError) as e:
        tq.tq_compress(g, rot, K, K, qjl_S=S)
    assert e.value.status == -2


def test_dense_dequantize_original_space(tq):
    B, H, T = 2, 4, 70
    kb, vb = [1, 3, 5, 8], [2, 4, 6, 7]
    K, V = _kv(B, H, T, seed=5)
    Q = O.haar_rotation(128, 9)
    oseg = O.PackedSegment(B, H, 128, 80, kb, vb)
    O.compress(oseg, K.numpy().view(np.uint16), V.numpy().view(np.uint16), O.signs(128, 9), None, Q=Q)
    g = tq.PackedSegment(tq.make_layout(B, H, 128, 80, kb, vb), n_tokens=T)
    for name in ("kcodes", "vcodes", "kscale", "vscale"):
        getattr(g, name).copy_(torch.from_numpy(getattr(oseg, name)))
    Qd = torch.from_numpy(Q).cuda()
    rot = tq.dense_rotation(tq.tq_make_rotation(128, 9), Qd)
    kr, vr, ko, vo = tq.tq_dequantize(g, 3, T - 3, rot=rot, rotated=True, original=True)
    torch.cuda.synchronize()
    Q64 = Q.astype(np.float64)
    for b in range(B):
        for h in range(H):
            ok, ov = O.dequant(oseg, b, h, 3, T - 3)
            assert np.array_equal(kr[b, h].cpu().numpy(), ok)
            assert np.array_equal(vr[b, h].cpu().numpy(), ov)
            for got, y in ((ko, ok), (vo, ov)):
                x = y.astype(np.float64) @ Q64  # rows: Q^T y
                err = np.abs(got[b, h].cpu().numpy() - x)
                assert np.all(err <= 1e-5 * np.maximum(1.0, np.abs(x)))


def _dense_attention_case(tq, B, H, Hq, spec, seed, dense_layers, mass=False):
    """Layers of `spec` segments; layers in dense_layers use a Haar rotation."""
    rng = np.random.default_rng(seed)
    L = len(dense_layers)
    views, keep, oracle_layers, Qs = [], [], [], []
    for l in range(L):
        sign = O.signs(128, 42 + l)
        rot = tq.tq_make_rotation(128, 42 + l)
        Q = O.haar_rotation(128, 100 + l) if dense_layers[l] else None
        if Q is not None:
            Qdev = torch.from_numpy(Q).cuda()
            Qs.append(Qdev)
            rot = tq.dense_rotation(rot, Qdev)
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
                _, _, kb, vb = sp
                o = O.PackedSegment(B, H, 128, cap, kb, vb)
                O.compress(o, K.numpy().view(np.uint16), V.numpy().view(np.uint16), sign, None, Q=Q)
                o.n_tokens = T
                g = tq.PackedSegment(tq.make_layout(B, H, 128, cap, kb, vb), n_tokens=T)
                for name in ("kcodes", "vcodes", "kscale", "vscale"):
                    getattr(g, name).copy_(torch.from_numpy(getattr(o, name)))
            if mass:
                g.attn_mass = torch.full((B, H, cap), -1.0, device="cuda")
            osegs.append(o)
            gsegs.append(g)
        keep.append(gsegs)
        views.append(tq.layer_view(rot, gsegs))
        oracle_layers.append((osegs, sign, Q))
    q = torch.from_numpy(rng.standard_normal((L, B, Hq, 128)).astype(np.float16))
    out = torch.empty(L, B, Hq, 128, device="cuda")
    ws = torch.empty(tq.tq_decode_workspace_size(views, B, H, Hq, 128), dtype=torch.uint8, device="cuda")
    tq.tq_decode_attention(views, q.cuda(), out, ws, H)
    assert tq.tq_decode_error_flag(ws) == 0
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    worst = 0.0
    for l in range(L):
        osegs, sign, Q = oracle_layers[l]
        ref = O.decode_attention(osegs, q[l].numpy(), sign, H, Q=Q, with_mass=mass)
        if mass:
            ref, rmass = ref
            for g, rm in zip(keep[l], rmass):
                gm = g.attn_mass.cpu().numpy()[:, :, :g.n_tokens]
                assert np.all(np.abs(gm - rm) <= 1e-4 * rm + 1e-30)
        o = got[l].reshape(-1, 128)
        r = ref.reshape(-1, 128)
        worst = max(worst, (np.abs(o - r).max(axis=1) / np.abs(r).max(axis=1)).max())
    return worst


@pytest.mark.parametrize("B,H,Hq,spec,dense", [
    (2, 4, 16, [("packed", 300, [3, 4, 2, 8], [3, 2, 4, 1])], [True]),
    (1, 8, 32, [("fp16", 40), ("packed", 700, [3] * 8, [3] * 8), ("fp16", 9)], [True, False]),
    (3, 2, 4, [("packed", 129, [1, 5], [6, 1]), ("packed", 64, [4, 4], [4, 4])], [False, True, True]),
])
def test_dense_decode_attention_matches_oracle(tq, B, H, Hq, spec, dense):
    w = _dense_attention_case(tq, B, H, Hq, spec, seed=B * 7 + H, dense_layers=dense, mass=True)
    assert w <= ATTN_TOL, w
