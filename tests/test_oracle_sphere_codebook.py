"""Pins of the oracle's sphere-coordinate Lloyd-Max codebook (the value
codebook variant: "TurboMOQ", "Head-to-Head Comparison" lists a Beta-CDF
codebook beside the Lloyd-Max one; "Project Structure": Beta-distribution
codebooks).  The law is sqrt(d) times a coordinate of a uniform unit d-vector:
u = sqrt(d) (2 B - 1) with B ~ Beta((d-1)/2, (d-1)/2)."""
import math

import numpy as np
import pytest
from scipy import integrate, stats

from oracle import oracle as O


def _law(d):
    a = 0.5 * (d - 1)
    rd = math.sqrt(d)
    beta = stats.beta(a, a)
    return (lambda u: beta.pdf(0.5 * (u / rd + 1.0)) / (2.0 * rd)), rd


@pytest.mark.parametrize("d", [16, 128, 1024])
def test_one_bit_is_the_half_mean(d):
    # one bit: +-E|u| = +-sqrt(d) Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2))
    c, t, _ = O.lloyd_max_sphere(1, d)
    want = math.sqrt(d) * math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
    assert c[1] == pytest.approx(want, rel=1e-12)
    assert c[0] == -c[1] and t[0] == 0.0


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_centroid_condition_by_quadrature(bits):
    # each centroid is the conditional mean of its cell under the Beta law
    # (integrated here by scipy, not by the oracle's quadrature)
    d = 128
    f, rd = _law(d)
    c, t, _ = O.lloyd_max_sphere(bits, d)
    edges = np.concatenate([[-rd], t, [rd]])
    for k in range(len(c)):
        lo, hi = edges[k], edges[k + 1]
        m0 = integrate.quad(f, lo, hi, epsabs=0, epsrel=1e-13, limit=200)[0]
        m1 = integrate.quad(lambda u: u * f(u), lo, hi, epsabs=0, epsrel=1e-13, limit=200)[0]
        assert c[k] == pytest.approx(m1 / m0, rel=1e-9, abs=1e-12)
    assert np.allclose(t, 0.5 * (c[1:] + c[:-1]), rtol=0, atol=1e-15)


def test_symmetric_and_ordered():
    for bits in range(1, 6):
        c, t, _ = O.lloyd_max_sphere(bits, 128)
        assert np.all(np.diff(c) > 0) and np.all(np.diff(t) > 0)
        assert np.array_equal(c, -c[::-1])


def test_tends_to_the_gaussian_codebook():
    # the law tends to N(0,1) as d grows: the distance to the Gaussian codebook
    # shrinks roughly like 1/d
    for bits in (2, 3):
        g = O.lloyd_max(bits)[0]
        e = [np.abs(O.lloyd_max_sphere(bits, d)[0] - g).max() for d in (64, 512, 4096)]
        assert e[0] > e[1] > e[2] and e[2] < 1e-3 and e[1] / e[2] > 4


def test_segments_with_the_sphere_law_use_its_thresholds():
    # compress through a law-1 segment: every value code is the count of sphere
    # thresholds below y / sigma (brute force), and dequantization uses its centroids
    rng = np.random.default_rng(5)
    K = rng.standard_normal((1, 2, 24, 128)).astype(np.float16)
    V = (rng.standard_normal((1, 2, 24, 128)) * 3).astype(np.float16)
    sign = O.signs(128, 42)
    seg = O.PackedSegment(1, 2, 128, 32, [3, 3], [3, 4], law=1)
    O.compress(seg, K, V, sign)
    for h, vb in enumerate([3, 4]):
        c, t = O.codebook_sphere_f32(vb)
        for tok in range(24):
            y = O.rotate_f32(V[0, h, tok].astype(np.float32), sign)
            s = seg.vscale[h * 32 + tok]
            u = (y * np.float32(np.float32(1.0) / s)).astype(np.float32)
            off = seg.code_offset("v", 0, h, tok)
            codes = O.unpack(seg.vcodes[off:off + 16 * vb], vb, 128)
            assert np.array_equal(codes, (t[None, :] < u[:, None]).sum(axis=1))
            _, vh = O.dequant(seg, 0, h, tok, 1)
            assert np.array_equal(vh[0], (s * c[codes]).astype(np.float32))
