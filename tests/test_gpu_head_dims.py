"""Head dimensions other than 128 (powers of two 16..1024) against the CPU oracle.

The rotation of "turboquant-mlx" (TurboQuant-MLX v2.0 README), "Walsh-Hadamard
Rotation" takes any power-of-two head_dim (WalshHadamardRotation(head_dim,
seed)); the format is the same binary32 sequence as at 128 dimensions, so codes
and scales must match the oracle bit for bit.  Dequantized rotated values are
bit-exact, original-space ones within 1e-5 max(1, |x|); decode attention within
2e-3 max relative error per query-head vector against the binary64 oracle over
the same packed cache (the oracle's own compression, uploaded)."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from rotated_quantized_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ATTN_TOL = 2e-3
DIMS = [16, 32, 64, 256, 512, 1024]


@pytest.fixture(scope="module")
def tq():
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq as T
    return T


def _kv(B, H, T, d, seed):
    w = W.Workload("t", layers=1, batch=B, context=T, kv_heads=H, head_dim=d, law="outliers",
                   outlier_channels=min(4, d))
    return W.kv_block(w, 0, B, T, seed)


def _widths(H, d, salt):
    kb = [(salt + 3 * h + d // 16) % 8 + 1 for h in range(H)]
    vb = [(salt + 5 * h + 1) % 8 + 1 for h in range(H)]
    return kb, vb


@pytest.mark.parametrize("d", DIMS)
def test_compress_bit_exact_other_dims(tq, d):
    B, H, T, t_begin = 2, 3, 45, 3
    cap = 64
    kb, vb = _widths(H, d, 1)
    K, V = _kv(B, H, T, d, seed=d + 1)
    sign = O.signs(d, 42)
    oseg = O.PackedSegment(B, H, d, cap, kb, vb)
    O.compress(oseg, K.numpy().view(np.uint16), V.numpy().view(np.uint16), sign, t_begin=t_begin)
    g = tq.PackedSegment(tq.make_layout(B, H, d, cap, kb, vb))
    tq.tq_compress(g, tq.tq_make_rotation(d, 42), K.cuda(), V.cuda(), t_begin=t_begin)
    torch.cuda.synchronize()
    assert np.array_equal(g.kcodes.cpu().numpy(), oseg.kcodes)
    assert np.array_equal(g.vcodes.cpu().numpy(), oseg.vcodes)
    assert np.array_equal(g.kscale.cpu().numpy().view(np.uint32), oseg.kscale.view(np.uint32))
    assert np.array_equal(g.vscale.cpu().numpy().view(np.uint32), oseg.vscale.view(np.uint32))


@pytest.mark.parametrize("t_begin,T", [(0, 45), (4, 46), (2, 1), (0, 600)])
def test_compress_bit_exact_token_pairs(tq, t_begin, T):
    # head_dim 64 from an even position: two tokens per thread (an odd count
    # leaves the last token unpaired); odd positions take the team kernel
    d, B, H = 64, 2, 4
    cap = ((t_begin + T + 15) // 16) * 16
    kb, vb = [1, 3, 4, 8], [2, 3, 5, 7]
    K, V = _kv(B, H, T, d, seed=T + t_begin)
    sign = O.signs(d, 44)
    oseg = O.PackedSegment(B, H, d, cap, kb, vb)
    O.compress(oseg, K.numpy().view(np.uint16), V.numpy().view(np.uint16), sign, t_begin=t_begin)
    g = tq.PackedSegment(tq.make_layout(B, H, d, cap, kb, vb))
    tq.tq_compress(g, tq.tq_make_rotation(d, 44), K.cuda(), V.cuda(), t_begin=t_begin)
    torch.cuda.synchronize()
    assert np.array_equal(g.kcodes.cpu().numpy(), oseg.kcodes)
    assert np.array_equal(g.vcodes.cpu().numpy(), oseg.vcodes)
    assert np.array_equal(g.kscale.cpu().numpy().view(np.uint32), oseg.kscale.view(np.uint32))
    assert np.array_equal(g.vscale.cpu().numpy().view(np.uint32), oseg.vscale.view(np.uint32))


@pytest.mark.parametrize("d", [16, 64, 256, 1024])
def test_compress_edge_vectors_other_dims(tq, d):
    # zeros, one-hot and fp16 extremes: the scale-0 and clamp paths
    B, H, T = 1, 2, 16
    K = torch.zeros(B, H, T, d, dtype=torch.float16)
    V = torch.zeros(B, H, T, d, dtype=torch.float16)
    K[0, 0, 1, 3] = 1.0
    V[0, 1, 2, 0] = -2.0
    K[0, 1, 3] = 65504.0
    V[0, 0, 4] = -65504.0
    K[0, 0, 5, ::2] = 1e-7
    kb, vb = [1, 8], [8, 2]
    sign = O.signs(d, 7)
    oseg = O.PackedSegment(B, H, d, 16, kb, vb)
    O.compress(oseg, K.numpy().view(np.uint16), V.numpy().view(np.uint16), sign)
    g = tq.PackedSegment(tq.make_layout(B, H, d, 16, kb, vb))
    tq.tq_compress(g, tq.tq_make_rotation(d, 7), K.cuda(), V.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(g.kcodes.cpu().numpy(), oseg.kcodes)
    assert np.array_equal(g.vcodes.cpu().numpy(), oseg.vcodes)
    assert np.array_equal(g.kscale.cpu().numpy().view(np.uint32), oseg.kscale.view(np.uint32))
    assert np.array_equal(g.vscale.cpu().numpy().view(np.uint32), oseg.vscale.view(np.uint32))


@pytest.mark.parametrize("d", [32, 256])
def test_dequantize_other_dims(tq, d):
    B, H, T = 2, 2, 40
    kb, vb = _widths(H, d, 2)
    K, V = _kv(B, H, T, d, seed=5 * d)
    sign = O.signs(d, 43)
    rot = tq.tq_make_rotation(d, 43)
    g = tq.PackedSegment(tq.make_layout(B, H, d, 48, kb, vb), n_tokens=T)
    tq.tq_compress(g, rot, K.cuda(), V.cuda())
    kr, vr, ko, vo = tq.tq_dequantize(g, 0, T, rot=rot, original=True)
    torch.cuda.synchronize()
    oseg = O.PackedSegment(B, H, d, 48, kb, vb)
    O.compress(oseg, K.numpy().view(np.uint16), V.numpy().view(np.uint16), sign)
    for b in range(B):
        for h in range(H):
            ky, vy = O.dequant(oseg, b, h, 0, T)
            assert np.array_equal(kr[b, h].cpu().numpy(), ky)
            assert np.array_equal(vr[b, h].cpu().numpy(), vy)
            kx = np.stack([O.rotate_f64(r.astype(np.float64), sign) for r in ky])
            vx = np.stack([O.rotate_f64(r.astype(np.float64), sign) for r in vy])
            assert np.all(np.abs(ko[b, h].cpu().numpy() - kx) <= 1e-5 * np.maximum(1.0, np.abs(kx)))
            assert np.all(np.abs(vo[b, h].cpu().numpy() - vx) <= 1e-5 * np.maximum(1.0, np.abs(vx)))


def _max_rel(out, ref):
    o = out.reshape(-1, out.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    return (np.abs(o - r).max(axis=1) / np.maximum(np.abs(r).max(axis=1), 1e-30)).max()


def _attention(tq, d, L, B, H, Hq, spec, seed):
    """spec per layer: ('fp16', T) or ('packed', T, kb[H], vb[H])."""
    rng = np.random.default_rng(seed)
    views, oracle_layers, keep = [], [], []
    for l in range(L):
        sign = O.signs(d, 42 + l)
        rot = tq.tq_make_rotation(d, 42 + l)
        osegs, gsegs = [], []
        for si, sp in enumerate(spec):
            T = sp[1]
            cap = max(16, ((T + 15) // 16) * 16)
            K, V = _kv(B, H, max(T, 1), d, seed=seed * 100 + l * 10 + si)
            if sp[0] == "fp16":
                o = O.Fp16Segment(B, H, d, cap, n_tokens=T)
                kk = np.zeros((B, H, cap, d), np.float16)
                vv = np.zeros((B, H, cap, d), np.float16)
                kk[:, :, :T] = K.numpy()[:, :, :T]
                vv[:, :, :T] = V.numpy()[:, :, :T]
                o.k16[:] = kk.ravel().view(np.uint16)
                o.v16[:] = vv.ravel().view(np.uint16)
                g = tq.Fp16Segment(B, H, d, cap, n_tokens=T, k=torch.from_numpy(kk).cuda(),
                                   v=torch.from_numpy(vv).cuda())
            else:
                kb, vb = sp[2], sp[3]
                o = O.PackedSegment(B, H, d, cap, kb, vb)
                if T:
                    O.compress(o, K.numpy().view(np.uint16), V.numpy().view(np.uint16), sign)
                o.n_tokens = T
                g = tq.PackedSegment(tq.make_layout(B, H, d, cap, kb, vb), n_tokens=T)
                g.kcodes.copy_(torch.from_numpy(o.kcodes))
                g.vcodes.copy_(torch.from_numpy(o.vcodes))
                g.kscale.copy_(torch.from_numpy(o.kscale))
                g.vscale.copy_(torch.from_numpy(o.vscale))
            osegs.append(o)
            gsegs.append(g)
        keep.append(gsegs)
        views.append(tq.layer_view(rot, gsegs))
        oracle_layers.append((osegs, sign))
    q = torch.from_numpy(rng.standard_normal((L, B, Hq, d)).astype(np.float16))
    out = torch.full((L, B, Hq, d), float("nan"), device="cuda")
    ws = torch.empty(tq.tq_decode_workspace_size(views, B, H, Hq, d), dtype=torch.uint8, device="cuda")
    tq.tq_decode_attention(views, q.cuda(), out, ws, H)
    assert tq.tq_decode_error_flag(ws) == 0
    got = out.cpu().numpy()
    worst = 0.0
    for l in range(L):
        osegs, sign = oracle_layers[l]
        if all(s.n_tokens == 0 for s in osegs):
            assert np.all(got[l] == 0)
            continue
        ref = O.decode_attention(osegs, q[l].numpy(), sign, H)
        worst = max(worst, _max_rel(got[l], ref))
    return worst


ATTN_CASES = [
    # d, L, B, H, Hq, segments
    (64, 2, 2, 4, 16, [("fp16", 10), ("packed", 300, [3, 5, 1, 8], [2, 8, 4, 3]), ("fp16", 7)]),
    (256, 2, 2, 2, 8, [("fp16", 33), ("packed", 290, [3, 4], [3, 1])]),
    (256, 1, 1, 8, 32, [("packed", 700, [3] * 8, [3] * 8)]),
    (16, 1, 2, 4, 8, [("packed", 200, [1, 2, 3, 4], [4, 3, 2, 1]), ("fp16", 3)]),
    (32, 1, 1, 2, 2, [("packed", 100, [8, 7], [6, 5])]),
    (512, 1, 1, 2, 8, [("fp16", 20), ("packed", 150, [2, 6], [5, 2])]),
    (1024, 1, 1, 1, 4, [("packed", 60, [4], [4]), ("fp16", 18)]),
    (64, 1, 1, 4, 12, [("packed", 0, [3] * 4, [3] * 4), ("fp16", 0)]),  # GQA 3, empty cache
    # head_dim 256 / 512 on the split-K kernels (GQA 1, 2, 4): every key and
    # value width, several stages per group, ragged tails, multi-chunk fp16
    (256, 1, 3, 8, 8, [("packed", 333, [1, 2, 3, 4, 5, 6, 7, 8], [8, 7, 6, 5, 4, 3, 2, 1]), ("fp16", 150)]),
    (256, 2, 2, 4, 8, [("fp16", 64), ("packed", 1000, [2, 3, 4, 5], [5, 4, 3, 2]),
                       ("packed", 77, [8, 8, 1, 1], [1, 8, 1, 8])]),
    (512, 1, 2, 2, 8, [("packed", 640, [3, 5], [4, 3]), ("fp16", 70)]),
    (512, 1, 1, 4, 4, [("packed", 129, [1, 2, 7, 8], [8, 7, 2, 1])]),
    (256, 2, 1, 2, 8, [("packed", 0, [3, 3], [3, 3]), ("fp16", 5)]),  # fp16 tokens only
    (256, 1, 1, 2, 8, [("packed", 0, [3, 3], [3, 3]), ("fp16", 0)]),  # empty cache
    (256, 1, 1, 2, 6, [("packed", 100, [3, 3], [3, 3]), ("fp16", 9)]),  # GQA 3: the generic kernel
    # head_dim 64 on the split-K kernels (token pairs read as 128-dim records):
    # every width, odd token counts (an unpaired last token), GQA 1, 2, 4
    (64, 1, 3, 8, 8, [("packed", 333, [1, 2, 3, 4, 5, 6, 7, 8], [8, 7, 6, 5, 4, 3, 2, 1]), ("fp16", 151)]),
    (64, 2, 2, 4, 8, [("fp16", 64), ("packed", 2049, [2, 3, 4, 5], [5, 4, 3, 2]),
                      ("packed", 77, [8, 8, 1, 1], [1, 8, 1, 8])]),
    (64, 1, 1, 2, 8, [("packed", 1, [3, 3], [3, 3]), ("fp16", 0)]),  # a single (unpaired) token
    (64, 1, 2, 2, 8, [("packed", 0, [3, 3], [3, 3]), ("fp16", 33)]),  # fp16 tokens only
]


@pytest.mark.parametrize("d,L,B,H,Hq,spec", ATTN_CASES)
def test_decode_attention_other_dims(tq, d, L, B, H, Hq, spec):
    worst = _attention(tq, d, L, B, H, Hq, spec, seed=d + L + len(spec))
    assert worst <= ATTN_TOL, worst


def test_chunked_compress_then_decode_256(tq):
    # 64-token chunks appended one after another equal one-shot compression,
    # and decode reads the appended cache ("turboquant-mlx", "Dynamic Chunk Buffering")
    d, B, H, T = 256, 1, 2, 192
    K, V = _kv(B, H, T, d, seed=77)
    rot = tq.tq_make_rotation(d, 42)
    one = tq.PackedSegment(tq.make_layout(B, H, d, T, [3, 3], [3, 3]))
    tq.tq_compress(one, rot, K.cuda(), V.cuda())
    chunked = tq.PackedSegment(tq.make_layout(B, H, d, T, [3, 3], [3, 3]))
    for c in range(0, T, 64):
        tq.tq_compress(chunked, rot, K[:, :, c:c + 64].contiguous().cuda(), V[:, :, c:c + 64].contiguous().cuda(),
                       t_begin=c)
    torch.cuda.synchronize()
    assert torch.equal(one.kcodes, chunked.kcodes) and torch.equal(one.vcodes, chunked.vcodes)
    assert torch.equal(one.kscale, chunked.kscale) and torch.equal(one.vscale, chunked.vscale)


def test_unsupported_features_other_dims(tq):
    d, B, H = 64, 1, 2
    K, V = _kv(B, H, 16, d, seed=3)
    # QJL heads, the sphere codebook and dense rotations stay at 128 dimensions
    g = tq.PackedSegment(tq.make_layout(B, H, d, 16, [2, 2], [2, 2], qjl=[1, 0]))
    S = tq.tq_make_qjl(d, 128, 9).cuda()
    with pytest.raises(tq.TQError) as e:
        tq.tq_compress(g, tq.tq_make_rotation(d, 1), K.cuda(), V.cuda(), qjl_S=S)
    assert e.value.status == -2
    g2 = tq.PackedSegment(tq.make_layout(B, H, d, 16, [2, 2], [2, 2], value_law=1))
    with pytest.raises(tq.TQError) as e:
        tq.tq_compress(g2, tq.tq_make_rotation(d, 1), K.cuda(), V.cuda())
    assert e.value.status == -2
