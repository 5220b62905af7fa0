"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something the pages or the mathematics fix:
published PRNG outputs, the Sylvester Hadamard matrix (scipy), closed forms,
numerical integration (scipy.integrate.quad), brute force over all cells,
numpy.unpackbits, PyTorch's scaled_dot_product_attention in float64, and the
tables printed on the pages (tests/golden/).
"""
import math
import os

import numpy as np
import pytest
import scipy.integrate
import scipy.linalg
import scipy.stats
import torch

from oracle import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


# --------------------------------------------------------------------------- PRNG
def test_splitmix64_published_outputs():
    for seed, *vals in _rows("splitmix64.txt"):
        got = O.splitmix64(int(seed), len(vals))
        assert [int(v, 16) for v in vals] == [int(x) for x in got]


def test_signs_are_top_bits_of_the_stream():
    words = O.splitmix64(42, 128)
    s = O.signs(128, 42)
    assert set(np.unique(s)) <= {-1, 1}
    assert np.array_equal(s == -1, (words >> np.uint64(63)) == 1)
    # roughly balanced, and per-layer seeds differ
    assert 40 < (s == -1).sum() < 88
    assert not np.array_equal(O.signs(128, 42), O.signs(128, 43))


# ----------------------------------------------------------------------- rotation
def _explicit_R(d, sign):
    H = scipy.linalg.hadamard(d).astype(np.float64)
    D = np.diag(sign.astype(np.float64))
    return D @ H @ D / math.sqrt(d)


@pytest.mark.parametrize("d", [16, 64, 128, 256])
def test_unscaled_transform_is_sylvester_hadamard(d):
    # Butterflies of the basis vectors with D = I reproduce scipy's Hadamard
    # matrix column by column, so H H^T = d I.
    ones = np.ones(d, np.int8)
    cols = O.rotate_f64(np.eye(d), ones) * math.sqrt(d)
    H = scipy.linalg.hadamard(d)
    assert np.array_equal(np.rint(cols).astype(int), H.T)
    assert np.allclose(cols @ cols.T, d * np.eye(d), atol=1e-9)


@pytest.mark.parametrize("d", [16, 128, 256])
def test_rotation_matches_explicit_matrix(d):
    sign = O.signs(d, 7)
    R = _explicit_R(d, sign)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((20, d)).astype(np.float16).astype(np.float64)
    y64 = O.rotate_f64(x, sign)
    assert np.allclose(y64, x @ R.T, rtol=0, atol=1e-12)
    y32 = O.rotate_f32(x.astype(np.float32), sign).astype(np.float64)
    err = np.abs(y32 - x @ R.T).max(axis=1) / np.linalg.norm(x, axis=1)
    assert err.max() < 2e-6
    # R is symmetric and an involution: R R = I
    assert np.allclose(R, R.T) and np.allclose(R @ R, np.eye(d), atol=1e-12)


def test_norm_preservation_and_exact_inverse():
    rng = np.random.default_rng(1)
    for d in (64, 256):  # 1/sqrt(d) is a power of two: every step is exact in binary64
        sign = O.signs(d, 3)
        x = rng.standard_normal((50, d)).astype(np.float16).astype(np.float64)
        y = O.rotate_f64(x, sign)
        assert np.allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-14)
        assert np.array_equal(O.rotate_f64(y, sign), x)


def test_rotation_gaussianizes_outliers():
    # "turboquant-mlx", "How It Works / Pipeline": kurtosis drops to about 3.
    rng = np.random.default_rng(2)
    d, n = 128, 4000
    x = rng.standard_normal((n, d))
    x[:, [3, 50, 77, 100]] *= 10.0
    x = x.astype(np.float16).astype(np.float32)
    y = O.rotate_f32(x, O.signs(d, 42)).astype(np.float64)
    k_before = scipy.stats.kurtosis(x.ravel(), fisher=False)
    k_after = scipy.stats.kurtosis(y.ravel(), fisher=False)
    assert k_before > 15 and abs(k_after - 3.0) < 0.15


# --------------------------------------------------------------------- codebooks
def test_lloyd_max_matches_printed_and_textbook_levels():
    for row in _rows("lloyd_max_gaussian.txt"):
        if row[0].startswith("D"):
            continue
        bits, _, tol = int(row[0]), row[1], float(row[2])
        want = np.array([float(v) for v in row[3:]])
        c, t, _ = O.lloyd_max(bits)
        assert np.allclose(c[len(c) // 2:], want, atol=tol), (bits, c)
        assert np.array_equal(c, -c[::-1])
        assert t[len(t) // 2] == 0.0


def test_lloyd_max_closed_forms_and_integrals():
    c1, _, _ = O.lloyd_max(1)
    assert abs(c1[1] - math.sqrt(2 / math.pi)) < 1e-12
    # centroid condition by numerical integration of x phi(x) over each cell,
    # and the distortion against Max's table
    dist = {int(r[0][1:]): float(r[1]) for r in _rows("lloyd_max_gaussian.txt") if r[0].startswith("D")}
    for bits in range(1, 7):
        c, t, _ = O.lloyd_max(bits)
        edges = np.concatenate([[-np.inf], t, [np.inf]])
        mse = 0.0
        for k in range(len(c)):
            a, b = edges[k], edges[k + 1]
            p = scipy.stats.norm.cdf(b) - scipy.stats.norm.cdf(a)
            m1 = scipy.integrate.quad(lambda x: x * scipy.stats.norm.pdf(x), a, b, epsabs=1e-14)[0]
            assert abs(m1 / p - c[k]) < 1e-8
            mse += scipy.integrate.quad(lambda x: (x - c[k]) ** 2 * scipy.stats.norm.pdf(x), a, b,
                                        epsabs=1e-14)[0]
        if bits in dist:
            assert abs(mse - dist[bits]) < 2e-4 * max(1.0, dist[bits] / 0.01)
        # thresholds are midpoints (nearest-centroid cells)
        assert np.allclose(t, 0.5 * (c[:-1] + c[1:]), atol=1e-15)


def test_lloyd_max_8bit_is_monotone_and_converged():
    c, t, sweeps = O.lloyd_max(8)
    assert np.all(np.diff(c) > 0) and np.all(np.diff(t) > 0)
    assert sweeps < 1_000_000
    assert 4.4 < c[-1] < 4.8


# ---------------------------------------------------------------------- keys
@pytest.mark.parametrize("bits", range(1, 9))
def test_key_codes_are_nearest_cell_centres(bits):
    rng = np.random.default_rng(bits)
    y = rng.standard_normal((64, 128)).astype(np.float32)
    codes, m = O.quant_key(y, bits)
    assert np.allclose(m, np.abs(y).max(axis=1))
    lev = O.key_levels(bits)
    v = y.astype(np.float64) / m[:, None].astype(np.float64)
    brute = np.abs(v[..., None] - lev).argmin(axis=-1)
    # away from cell edges (where v*2^(b-1) is an integer) the nearest centre wins
    edge_dist = np.abs((v + 1) * 2 ** (bits - 1) - np.rint((v + 1) * 2 ** (bits - 1)))
    far = edge_dist > 1e-5
    assert np.array_equal(codes[far], brute[far])
    # symmetry: negating a vector mirrors its codes away from edges
    cneg, _ = O.quant_key(-y, bits)
    assert np.array_equal(cneg[far], ((1 << bits) - 1 - codes)[far])


def test_key_edges_ties_and_zero():
    b = 3
    # exact cell edges: v = -1 + k/4 for k = 0..8; ties go to the upper cell,
    # v = +1 to the top cell
    m = 2.0
    y = np.array([m * (-1 + k / 4) for k in range(9)] + [0.0] * 119, np.float32)
    codes, scale = O.quant_key(y[None], b)
    assert scale[0] == m
    assert codes[0, :9].tolist() == [0, 1, 2, 3, 4, 5, 6, 7, 7]
    z, sz = O.quant_key(np.zeros((1, 128), np.float32), b)
    assert sz[0] == 0 and np.all(z == 4)


def test_key_8bit_cosine():
    rng = np.random.default_rng(5)
    y = rng.standard_normal((200, 128)).astype(np.float32)
    codes, m = O.quant_key(y, 8)
    yh = m[:, None] * O.key_levels(8)[codes]
    cos = (yh * y).sum(1) / np.linalg.norm(yh, axis=1) / np.linalg.norm(y, axis=1)
    assert cos.min() > 0.9999


# ---------------------------------------------------------------------- values
@pytest.mark.parametrize("bits", range(1, 9))
def test_value_codes_are_nearest_centroids(bits):
    rng = np.random.default_rng(100 + bits)
    y = rng.standard_normal((64, 128)).astype(np.float32)
    codes, sigma = O.quant_value(y, bits)
    rms = np.sqrt((y.astype(np.float64) ** 2).mean(axis=1))
    assert np.allclose(sigma, rms, rtol=1e-6)
    c, t, _ = O.lloyd_max(bits)
    u = y.astype(np.float64) / sigma[:, None]
    brute = np.abs(u[..., None] - c).argmin(axis=-1)
    far = np.abs(u[..., None] - t).min(axis=-1) > 1e-5 if len(t) else np.ones_like(u, bool)
    assert np.array_equal(codes[far], brute[far])


def test_value_ties_go_low_and_sigma_is_rms_of_input():
    b = 2
    _, t32 = O.codebook_f32(b)
    sig = 1.0
    # a vector whose RMS is exactly 1 with coordinates at the thresholds
    y = np.zeros(128, np.float32)
    y[0], y[1], y[2] = t32[0], t32[1], t32[2]
    rest = np.float32(math.sqrt((128 - float(t32[0]) ** 2 - float(t32[1]) ** 2 - float(t32[2]) ** 2) / 125))
    y[3:] = rest
    codes, sigma = O.quant_value(y[None], b)
    u = y / sigma[0]
    for i in range(3):
        want = int((t32 < u[i]).sum())
        assert codes[0, i] == want
    # orthogonal rotation keeps the norm: sigma = ||x|| / sqrt(d)
    rng = np.random.default_rng(9)
    x = rng.standard_normal((30, 128)).astype(np.float16).astype(np.float32)
    y = O.rotate_f32(x, O.signs(128, 42))
    _, s = O.quant_value(y, 4)
    assert np.allclose(s, np.linalg.norm(x.astype(np.float64), axis=1) / math.sqrt(128), rtol=2e-6)
    assert sig == 1.0


def test_value_cosine_follows_distortion():
    # cosine of a Lloyd-Max reconstruction of N(0,1) coordinates ~ sqrt(1 - D_b);
    # 1 bit gives ~0.798 ("TurboMOQ", QJL section: 1-bit base cosine 0.796).
    rng = np.random.default_rng(11)
    y = rng.standard_normal((400, 128)).astype(np.float32)
    for bits, D in [(1, 1 - 2 / math.pi), (2, 0.1175), (3, 0.03454), (4, 0.009497)]:
        codes, s = O.quant_value(y, bits)
        c32, _ = O.codebook_f32(bits)
        yh = s[:, None] * c32[codes]
        cos = ((yh * y).sum(1) / np.linalg.norm(yh, axis=1) / np.linalg.norm(y, axis=1)).mean()
        assert abs(cos - math.sqrt(1 - D)) < 0.004, (bits, cos)


# ---------------------------------------------------------------------- packing
@pytest.mark.parametrize("bits", range(1, 9))
def test_packing_is_lsb_first_bitstream(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(10, 128)).astype(np.uint8)
    rec = O.pack(codes, bits)
    assert rec.shape == (10, 16 * bits)
    stream = np.unpackbits(rec, axis=1, bitorder="little").reshape(10, 128, bits)
    rebuilt = (stream.astype(np.int64) << np.arange(bits)).sum(axis=2)
    assert np.array_equal(rebuilt, codes)
    assert np.array_equal(O.unpack(rec, bits, 128), codes)


def test_packed_size_matches_printed_3bit_table():
    # codes take b/16 of the fp16 bytes; 3 bits: 1024 MB -> 192 MB (5.3x)
    seg = O.PackedSegment(B=1, H=8, d=128, capacity=4096, kbits=[3] * 8, vbits=[3] * 8)
    fp16 = 1 * 8 * 4096 * 128 * 2 * 2
    code_bytes = seg.kcodes.nbytes + seg.vcodes.nbytes
    assert code_bytes * 16 == fp16 * 3
    for ctx, mb16, mb3, ratio in _rows("memory_3bit.txt"):
        mb16, mb3 = float(mb16), float(mb3)
        assert mb16 * 3 / 16 == mb3
        assert abs(mb16 / mb3 - float(ratio)) < 0.05


# ---------------------------------------------------------------------- QJL
def test_qjl_matrix_is_standard_normal():
    S = O.qjl_matrix(128, 128, 42 + 1000).ravel().astype(np.float64)
    assert abs(S.mean()) < 0.02 and abs(S.std() - 1) < 0.02
    assert scipy.stats.kstest(S, "norm").pvalue > 1e-3


def test_qjl_inner_product_is_unbiased_over_seeds():
    # E_S[sqrt(pi/2)/m * rho * <S q, sign(S r)>] = <q, r> for Gaussian S
    rng = np.random.default_rng(3)
    d = jl = 64
    q = rng.standard_normal(d).astype(np.float32)
    r = rng.standard_normal(d).astype(np.float32)
    est = []
    for seed in range(1500):
        S = O.qjl_matrix(jl, d, 10_000 + seed)
        sb, rho = O.qjl_sketch(S, r, np.zeros(d, np.float32))
        s = np.where(np.unpackbits(sb, bitorder="little")[:jl] == 1, 1.0, -1.0)
        est.append(math.sqrt(math.pi / 2) / jl * rho * float((S.astype(np.float64) @ q) @ s))
    est = np.array(est)
    truth = float(q.astype(np.float64) @ r.astype(np.float64))
    se = est.std(ddof=1) / math.sqrt(len(est))
    assert abs(est.mean() - truth) < 3.5 * se, (est.mean(), truth, se)
    # the same estimator without the pi/2 correction is biased by 2/pi
    assert abs(est.mean() * 2 / math.pi - truth) > 3.5 * se


def test_qjl_improves_one_bit_keys():
    # "TurboMOQ", QJL section: 1-bit cosine 0.796 -> 0.827 with the residual
    # sketch.  Cosine is a vector-reconstruction measure, so the sketch is decoded
    # here with the MSE-optimal scale: with s = sign(S r), E<r, S^T s> =
    # m sqrt(2/pi) rho and E||S^T s||^2 = m d + m (m-1) 2/pi, giving
    # alpha = sqrt(2/pi) rho / (d + (m-1) 2/pi).  (Scores use the unbiased scale
    # sqrt(pi/2)/m rho instead; see the test above.)
    rng = np.random.default_rng(4)
    d = m = 128
    S = O.qjl_matrix(m, d, 42 + 1000).astype(np.float64)
    y = rng.standard_normal((300, d)).astype(np.float32)
    codes, mx = O.quant_key(y, 1)
    yh = (mx[:, None] * O.key_levels(1)[codes]).astype(np.float32)
    base, corr = [], []
    for i in range(len(y)):
        sb, rho = O.qjl_sketch(S.astype(np.float32), y[i], yh[i])
        s = np.where(np.unpackbits(sb, bitorder="little") == 1, 1.0, -1.0)
        alpha = math.sqrt(2 / math.pi) * rho / (d + (m - 1) * 2 / math.pi)
        for acc, v in ((base, yh[i].astype(np.float64)), (corr, yh[i] + alpha * (S.T @ s))):
            acc.append(v @ y[i] / np.linalg.norm(v) / np.linalg.norm(y[i]))
    assert abs(np.mean(base) - 0.796) < 0.01
    assert np.mean(corr) > np.mean(base) + 0.02


# ---------------------------------------------------------------------- attention
def _tiny_case(d=16, H=2, Hq=4, T=7, kb=3, vb=2, qjl=None, seed=0):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((1, H, T, d)).astype(np.float16)
    V = rng.standard_normal((1, H, T, d)).astype(np.float16)
    q = rng.standard_normal((1, Hq, d)).astype(np.float16)
    sign = O.signs(d, 42)
    seg = O.PackedSegment(1, H, d, T, [kb] * H, [vb] * H, qjl=qjl, jl=d)
    S = O.qjl_matrix(d, d, 1042) if qjl is not None else None
    O.compress(seg, K, V, sign, S)
    return K, V, q, sign, seg, S


def _dequant_by_definition(seg, sign, b, h, d, S=None):
    """Unpack with numpy and rebuild khat, vhat in the original space by the
    explicit matrix R; an independent route to the attention inputs."""
    R = _explicit_R(d, sign)
    T = seg.n_tokens
    ks, vs = [], []
    for t in range(T):
        kb, vb = int(seg.kbits[h]), int(seg.vbits[h])
        o = seg.code_offset("k", b, h, t)
        bits = np.unpackbits(seg.kcodes[o:o + d * kb // 8], bitorder="little").reshape(d, kb)
        kc = (bits.astype(np.int64) << np.arange(kb)).sum(1)
        o = seg.code_offset("v", b, h, t)
        bits = np.unpackbits(seg.vcodes[o:o + d * vb // 8], bitorder="little").reshape(d, vb)
        vc = (bits.astype(np.int64) << np.arange(vb)).sum(1)
        idx = (b * seg.H + h) * seg.capacity + t
        yk = float(seg.kscale[idx]) * ((kc + 0.5) * 2.0 ** (1 - kb) - 1)
        if seg.qjl[h]:
            qi = (b * seg.nq + seg.qjl_rank(h)) * seg.capacity + t
            sb = seg.qjl_signs[qi * (seg.jl // 8):(qi + 1) * (seg.jl // 8)]
            s = np.where(np.unpackbits(sb, bitorder="little") == 1, 1.0, -1.0)
            yk = yk + math.sqrt(math.pi / 2) / seg.jl * float(seg.qjl_norm[qi]) * (S.astype(np.float64).T @ s)
        c32, _ = O.codebook_f32(vb)
        yv = float(seg.vscale[idx]) * c32[vc].astype(np.float64)
        ks.append(R @ yk)
        vs.append(R @ yv)
    return np.array(ks), np.array(vs)


@pytest.mark.parametrize("kb,vb,qjl", [(3, 2, None), (1, 1, [1, 0]), (8, 4, [0, 1])])
def test_attention_matches_torch_sdpa_on_tiny_inputs(kb, vb, qjl):
    d, H, Hq = 16, 2, 4
    K, V, q, sign, seg, S = _tiny_case(d=d, H=H, Hq=Hq, kb=kb, vb=vb, qjl=qjl)
    out = O.decode_attention([seg], q, sign, H, S=S, jl=d)
    g = Hq // H
    for j in range(Hq):
        kh, vh = _dequant_by_definition(seg, sign, 0, j // g, d, S)
        qq = torch.tensor(q[0, j].astype(np.float64))[None, None, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, torch.tensor(kh)[None, None], torch.tensor(vh)[None, None])
        assert np.allclose(out[0, j], ref[0, 0, 0].numpy(), atol=1e-12)


def test_attention_rotation_invariance_and_special_cases():
    d = 16
    sign = O.signs(d, 42)
    R = _explicit_R(d, sign)
    rng = np.random.default_rng(8)
    q = rng.standard_normal(d)
    yk = rng.standard_normal(d)
    assert abs(q @ (R @ yk) - (R @ q) @ yk) < 1e-12
    # identical keys -> the output is the mean of the values
    H, T = 1, 5
    seg = O.Fp16Segment(1, H, d, T, n_tokens=T)
    k = rng.standard_normal(d).astype(np.float16)
    V = rng.standard_normal((T, d)).astype(np.float16)
    seg.k16[:] = np.tile(k, T).view(np.uint16)
    seg.v16[:] = V.ravel().view(np.uint16)
    qh = rng.standard_normal((1, 1, d)).astype(np.float16)
    out = O.decode_attention([seg], qh, sign, H)
    assert np.allclose(out[0, 0], V.astype(np.float64).mean(0), atol=1e-12)
    # empty cache -> zero output
    empty = O.Fp16Segment(1, H, d, 4, n_tokens=0)
    assert np.all(O.decode_attention([empty], qh, sign, H) == 0)


def test_fp16_and_packed_segments_concatenate():
    # attention over [sinks fp16 | packed] equals one softmax over all tokens
    d, H, Hq = 16, 1, 2
    K, V, q, sign, seg, S = _tiny_case(d=d, H=H, Hq=Hq, T=6, kb=4, vb=4)
    rng = np.random.default_rng(12)
    sink = O.Fp16Segment(1, H, d, 3, n_tokens=3)
    Ks = rng.standard_normal((3, d)).astype(np.float16)
    Vs = rng.standard_normal((3, d)).astype(np.float16)
    sink.k16[:] = Ks.ravel().view(np.uint16)
    sink.v16[:] = Vs.ravel().view(np.uint16)
    out = O.decode_attention([sink, seg], q, sign, H)
    for j in range(Hq):
        kh, vh = _dequant_by_definition(seg, sign, 0, 0, d)
        kk = np.concatenate([Ks.astype(np.float64), kh])
        vv = np.concatenate([Vs.astype(np.float64), vh])
        s = kk @ q[0, j].astype(np.float64) / math.sqrt(d)
        p = np.exp(s - s.max())
        p /= p.sum()
        assert np.allclose(out[0, j], p @ vv, atol=1e-12)


# ---------------------------------------------------------------------- host steps
def test_tiers_follow_the_printed_table():
    rows = _rows("tiers.txt")
    T = 131072
    got = O.tier_ranges(T)
    ages = [(int(r[1]), None if r[2] == "inf" else int(r[2])) for r in rows]
    # tier i covers ages [lo, hi) -> positions (T-1-hi, T-1-lo]
    for tier, start, end in got:
        lo, hi = ages[tier]
        assert T - 1 - (end - 1) == lo or tier == 0 and end == T
        if hi is not None:
            assert T - 1 - start == hi - 1 or start == 0
    sizes = {tier: end - start for tier, start, end in got}
    assert sizes == {0: 1024, 1: 7168, 2: 57344, 3: 65536}
    # bytes per layer (8 heads, d=128): fp16 512 B, else 16(kb+vb) + 8 B per token-head
    per = {0: 512, 1: 16 * 8 + 8, 2: 16 * 5 + 8, 3: 16 * 3 + 8}
    total = sum(sizes[t] * 8 * per[t] for t in sizes)
    assert abs(total / 1e6 - 81.72) < 0.01
    assert O.tier_ranges(500) == [(0, 0, 500)]


def test_chunk_schedule():
    s, starts, buf = O.chunk_schedule(16384)
    assert s == 128 and len(starts) == 254 and buf == 0 and starts[0] == 128
    s, starts, buf = O.chunk_schedule(16384 + 100)
    assert len(starts) == 255 and buf == 36
