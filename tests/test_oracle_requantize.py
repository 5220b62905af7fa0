"""Pins of the oracle's tier demotion (re-quantisation of packed tokens in the
rotated space, "TurboMOQ", "Progressive temporal tiering").

Requantisation compresses the rotated-space reconstruction again, so its
result is fixed by the source codes alone: these tests derive the destination
codes and scales in binary64 from the source codes (a route that never forms
the reconstructed vectors) and compare, allowing only coordinates within 1e-6
of a decision boundary to differ."""
import numpy as np
import pytest

from oracle import oracle as O

D = 128


def _packed(B, H, T, kb, vb, seed):
    rng = np.random.default_rng(seed)
    K = (rng.standard_normal((B, H, T, D)) * rng.uniform(0.2, 5.0, (B, H, 1, 1))).astype(np.float16)
    V = (rng.standard_normal((B, H, T, D)) * rng.uniform(0.2, 5.0, (B, H, 1, 1))).astype(np.float16)
    seg = O.PackedSegment(B, H, D, ((T + 15) // 16) * 16, kb, vb)
    O.compress(seg, K, V, O.signs(D, 42))
    return seg


def _codes(seg, which, b, h, t):
    bits = int((seg.kbits if which == "k" else seg.vbits)[h])
    buf = seg.kcodes if which == "k" else seg.vcodes
    off = seg.code_offset(which, b, h, t)
    return O.unpack(buf[off:off + D * bits // 8], bits, D).astype(np.int64)


def _key_closed_form(k_src, b1, b2):
    lev = (k_src + 0.5) * 2.0 ** (1 - b1) - 1.0   # cell centres in units of m
    mx = np.abs(lev).max()
    u = (lev / mx + 1.0) * 2.0 ** (b2 - 1)
    return np.clip(np.floor(u), 0, 2 ** b2 - 1).astype(np.int64), u, mx


@pytest.mark.parametrize("b1", range(1, 9))
def test_same_width_keys_are_unchanged(b1):
    src = _packed(1, 2, 40, [b1, b1], [3, 3], seed=b1)
    dst = O.PackedSegment(1, 2, D, 48, [b1, b1], [3, 3])
    O.requantize(src, 0, 40, dst, 0)
    for h in range(2):
        for t in range(40):
            k0 = _codes(src, "k", 0, h, t)
            assert np.array_equal(_codes(dst, "k", 0, h, t), k0)
            m0 = src.kscale[h * src.capacity + t]
            lev_max = np.abs((k0 + 0.5) * 2.0 ** (1 - b1) - 1.0).max()
            assert dst.kscale[h * dst.capacity + t] == np.float32(m0 * np.float32(lev_max))


@pytest.mark.parametrize("b1,b2", [(8, 4), (8, 1), (4, 3), (4, 2), (3, 2), (2, 1), (6, 5)])
def test_key_demotion_matches_code_closed_form(b1, b2):
    src = _packed(2, 3, 33, [b1] * 3, [2] * 3, seed=10 * b1 + b2)
    dst = O.PackedSegment(2, 3, D, 48, [b2] * 3, [1] * 3)
    O.requantize(src, 0, 33, dst, 5)
    near = total = 0
    for b in range(2):
        for h in range(3):
            for t in range(33):
                want, u, _ = _key_closed_form(_codes(src, "k", b, h, t), b1, b2)
                got = _codes(dst, "k", b, h, t + 5)
                edge = np.abs(u - np.round(u)) <= 1e-6 * 2 ** (b2 - 1)
                assert np.array_equal(got[~edge], want[~edge])
                near += int((got != want).sum())
                total += D
    assert near <= 1e-5 * total + 1


@pytest.mark.parametrize("b1,b2", [(8, 3), (4, 4), (4, 2), (3, 2), (3, 1), (2, 1)])
def test_value_demotion_matches_code_closed_form(b1, b2):
    src = _packed(1, 4, 29, [4] * 4, [b1] * 4, seed=100 + 10 * b1 + b2)
    dst = O.PackedSegment(1, 4, D, 32, [2] * 4, [b2] * 4)
    O.requantize(src, 0, 29, dst, 0)
    c1 = O.lloyd_max(b1)[0]                    # binary64 centroids
    c1 = c1.astype(np.float32).astype(np.float64)
    t2 = O.codebook_f32(b2)[1].astype(np.float64)
    for h in range(4):
        for t in range(29):
            y = c1[_codes(src, "v", 0, h, t)]  # reconstruction in units of the source sigma
            u = y / np.sqrt(np.mean(y * y))
            want = (t2[None, :] < u[:, None]).sum(axis=1)
            got = _codes(dst, "v", 0, h, t)
            edge = (np.abs(u[:, None] - t2[None, :]) <= 1e-6 * np.maximum(1.0, np.abs(t2))).any(axis=1)
            assert np.array_equal(got[~edge], want[~edge])
            s_src = np.float64(src.vscale[h * src.capacity + t])
            assert dst.vscale[h * dst.capacity + t] == pytest.approx(s_src * np.sqrt(np.mean(y * y)), rel=1e-6)


def test_requantize_writes_only_its_range():
    src = _packed(1, 2, 20, [4, 4], [4, 4], seed=7)
    dst = O.PackedSegment(1, 2, D, 64, [2, 3], [1, 2])
    before = dst.kcodes.copy()
    O.requantize(src, 3, 10, dst, 40)
    for h, rk in enumerate([32, 48]):
        base = dst.code_offset("k", 0, h, 0)
        changed = np.nonzero(dst.kcodes[base:base + 64 * rk] != before[base:base + 64 * rk])[0] // rk
        assert changed.size == 0 or (changed.min() >= 40 and changed.max() < 50)
    assert dst.n_tokens == 50
