"""The compressor's value-code lookup tables (tq_value_code_table), on the CPU.

The code of a value quotient u is the number of thresholds below it,
#{j : t_j < u} ("TurboMOQ", "Architecture": nearest Lloyd-Max level of the
value codebook).  The one-thread-per-vector compressor takes it from a table
indexed by the top bits of u's binary32 pattern; these tests decode with the
same arithmetic the kernels use (written out below from the table's
documented layout) and compare with the count itself, over every bucket edge,
every threshold and its neighbouring floats, signed zeros, a dense grid and
random bit patterns, for both codebook laws at 1-4 bits."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def tq():
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq as T
    return T


def _decode(table, bits, u):
    """The kernels' table decode of the float32 quotients u."""
    p = u.view(np.uint32)
    if bits <= 3:
        i = (p >> 22).astype(np.int64)
        t = table.view(np.float32)[2 * i]
        k = table[2 * i + 1]
        return k + (t < u).astype(np.uint32)
    e = table[(p >> 21).astype(np.int64)]
    low = np.uint32(0x1FFFFF)
    x = (p & low) ^ np.where(p >> 31 != 0, low, np.uint32(0)).astype(np.uint32)
    return (e >> 21) + ((e & low) < x).astype(np.uint32)


def _probes(thr):
    """Bit patterns of finite floats: bucket edges (11- and 10-bit) +-3, every
    threshold +-5 ulps, both zeros, a grid over [-4, 4], random patterns."""
    edges = (np.arange(2048, dtype=np.int64) << 21)[:, None] + np.arange(-3, 4)[None]
    tb = thr.astype(np.float32).view(np.uint32).astype(np.int64)[:, None] + np.arange(-5, 6)[None]
    grid = np.arange(-4.0, 4.0, 1.0 / 4096, dtype=np.float32).view(np.uint32).astype(np.int64)
    rnd = np.random.default_rng(7).integers(0, 1 << 32, size=1 << 20, dtype=np.int64)
    p = np.concatenate([edges.ravel(), tb.ravel(), [0, 1 << 31], grid, rnd]) & 0xFFFFFFFF
    u = p.astype(np.uint32).view(np.float32)
    return u[np.isfinite(u)]


@pytest.mark.parametrize("law", ["gaussian", "sphere"])
@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_table_decode_counts_thresholds_below(tq, bits, law):
    thr = (tq.tq_fit_codebook(bits) if law == "gaussian" else tq.tq_fit_codebook_sphere(bits, 128))[1]
    thr = np.asarray(thr, dtype=np.float32)
    table = tq.tq_value_code_table(bits, thr)
    u = _probes(thr)
    want = np.searchsorted(thr, u, side="left").astype(np.uint32)  # #{j : t_j < u}
    got = _decode(table, bits, u)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, (u[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_table_with_negative_zero_threshold(tq):
    # a middle threshold of -0.0 must decode like +0.0: [t < u] is u > 0 for both
    thr = np.asarray(tq.tq_fit_codebook(4)[1], dtype=np.float32).copy()
    thr[7] = np.float32(-0.0)
    table = tq.tq_value_code_table(4, thr)
    u = _probes(thr)
    want = np.searchsorted(np.where(thr == 0, np.float32(0.0), thr), u, side="left").astype(np.uint32)
    assert np.array_equal(_decode(table, 4, u), want)


def test_table_rejects_bad_arguments_and_shared_buckets(tq):
    with pytest.raises(tq.TQError) as e:
        tq.tq_value_code_table(5, np.zeros(31, np.float32))
    assert e.value.status == -1  # TQ_ERR_ARG
    with pytest.raises(tq.TQError) as e:
        tq.tq_value_code_table(0, np.zeros(1, np.float32))
    assert e.value.status == -1
    # two thresholds inside [1, 1.25): one 11-bit bucket
    thr = np.array([-2.0, -1.0, -0.5, -0.25, 0.0, 0.25, 0.5, 1.0, 1.1, 1.5, 2.0, 2.5, 3.0, 3.5, 4.0],
                   dtype=np.float32)
    with pytest.raises(tq.TQError) as e:
        tq.tq_value_code_table(4, thr)
    assert e.value.status == -2  # TQ_ERR_UNSUPPORTED
