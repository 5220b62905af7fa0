"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/tq.h declares, its host-side functions agree with the oracle, and bad
arguments are rejected on the host before anything is launched."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from oracle import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def tq():
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq as T
    return T


def test_header_symbols_are_exported(tq):
    hdr = open(os.path.join(ROOT, "include", "tq.h")).read()
    declared = set(re.findall(r"^\s*(?:const\s+)?[a-z_]+\s*\*?\s*(tq_[a-z_0-9]+)\s*\(", hdr, re.M))
    assert len(declared) >= 12
    lib = ctypes.CDLL(tq.LIB_PATH)
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert declared <= set(tq.EXPORTED)


def test_rotation_signs_match_oracle(tq):
    for seed in (0, 42, 42 + 39):
        rot = tq.tq_make_rotation(128, seed)
        bits = np.array([(rot.sign_bits[i >> 5] >> (i & 31)) & 1 for i in range(128)])
        assert np.array_equal(np.where(bits == 1, -1, 1), O.signs(128, seed))
    with pytest.raises(tq.TQError):
        tq.tq_make_rotation(100, 1)


@pytest.mark.parametrize("bits", range(1, 9))
def test_codebook_matches_oracle(tq, bits):
    c, t = tq.tq_fit_codebook(bits)
    oc, ot = O.codebook_f32(bits)
    assert np.array_equal(c.numpy(), oc)
    assert np.array_equal(t.numpy(), ot)


@pytest.mark.parametrize("bits", range(1, 8))
def test_sphere_codebook_matches_oracle(tq, bits):
    # the host fit and the oracle's are separate programs of the same iteration;
    # the 8-bit fit (~15 s on each side) is covered by the GPU parity tests
    c, t = tq.tq_fit_codebook_sphere(bits, 128)
    oc, ot = O.codebook_sphere_f32(bits)
    assert np.array_equal(c.numpy().view(np.uint32), np.asarray(oc, np.float32).view(np.uint32))
    assert np.array_equal(t.numpy().view(np.uint32), np.asarray(ot, np.float32).view(np.uint32))


@pytest.mark.parametrize("d,seed", [(16, 3), (64, 7), (128, 42), (128, 1043)])
def test_haar_rotation_matches_oracle(tq, d, seed):
    # Householder QR here, LAPACK's through numpy in the oracle: both round the
    # binary64 factor to binary32; allow one ulp where the two land on either
    # side of a rounding boundary
    Q = tq.tq_make_haar_rotation(d, seed).numpy()
    Qo = O.haar_rotation(d, seed)
    ulps = np.abs(Q.astype(np.float64) - Qo) / np.spacing(np.abs(Qo))
    assert ulps.max() <= 1 and (ulps > 0).sum() <= 2


def test_qjl_matrix_matches_oracle(tq):
    S = tq.tq_make_qjl(128, 128, 1042).numpy()
    assert np.array_equal(S, O.qjl_matrix(128, 128, 1042))


def test_packed_sizes_match_layout(tq):
    kb = [1, 2, 3, 4, 5, 6, 7, 8]
    vb = [8, 7, 6, 5, 4, 3, 2, 1]
    qj = [1, 0, 1, 0, 0, 0, 0, 1]
    L = tq.make_layout(3, 8, 128, 96, kb, vb, qj)
    s = tq.tq_packed_size(L)
    seg = O.PackedSegment(3, 8, 128, 96, kb, vb, qj)
    assert s.kcode_bytes == seg.kcodes.nbytes and s.vcode_bytes == seg.vcodes.nbytes
    assert s.kscale_bytes == seg.kscale.nbytes and s.vscale_bytes == seg.vscale.nbytes
    assert s.qjl_sign_bytes == seg.qjl_signs.nbytes and s.qjl_norm_bytes == seg.qjl_norm.nbytes
    assert s.vqjl_sign_bytes == 0 and s.vqjl_norm_bytes == 0
    qv = [0, 1, 1, 0, 0, 0, 0, 1]
    sv = tq.tq_packed_size(tq.make_layout(3, 8, 128, 96, kb, vb, qj, qjl_v=qv))
    segv = O.PackedSegment(3, 8, 128, 96, kb, vb, qj, qjl_v=qv)
    assert sv.vqjl_sign_bytes == segv.vqjl_signs.nbytes and sv.vqjl_norm_bytes == segv.vqjl_norm.nbytes
    bad_v = tq.make_layout(1, 8, 128, 16, 3, 3)
    bad_v.qjl_v[0] = 2
    with pytest.raises(tq.TQError):  # flags are 0/1
        tq.tq_packed_size(bad_v)
    # 3 bits: codes are 3/16 of the fp16 bytes (1024 MB -> 192 MB)
    s3 = tq.tq_packed_size(tq.make_layout(1, 8, 128, 65536, 3, 3))
    assert (s3.kcode_bytes + s3.vcode_bytes) * 16 == 65536 * 8 * 128 * 2 * 2 * 3


def test_age_tiers_match_oracle(tq):
    for T in (0, 1, 500, 1024, 1025, 8192, 9000, 131072, 200000):
        got = tq.tq_age_tiers(T, [1024, 8192, 65536])
        want = {tier: (s, e) for tier, s, e in O.tier_ranges(T)}
        for tier, (s, e) in enumerate(got):
            if s == e:
                assert tier not in want
            else:
                assert want[tier] == (s, e)


def test_host_side_argument_errors(tq):
    bad = tq.make_layout(1, 8, 128, 64, 9, 3)
    with pytest.raises(tq.TQError) as e:
        tq.tq_packed_size(bad)
    assert e.value.status == -1
    with pytest.raises(tq.TQError) as e:  # value codebook law outside {0, 1}
        tq.tq_packed_size(tq.make_layout(1, 8, 128, 64, 3, 3, value_law=2))
    assert e.value.status == -1
    with pytest.raises(tq.TQError):
        tq.tq_fit_codebook_sphere(0, 128)
    L = tq.make_layout(1, 8, 128, 64, 3, 3)
    b = tq.tq_packed_bufs()
    rot = tq.tq_make_rotation(128, 42)
    lib = ctypes.CDLL(tq.LIB_PATH)
    lib.tq_compress.restype = ctypes.c_int
    # NULL inputs
    st = lib.tq_compress(ctypes.byref(L), ctypes.byref(rot), None, None, None, 8, 0, 0, 128, 0,
                         ctypes.byref(b), None)
    assert st == -1
    # capacity exceeded (checked before pointers are touched)
    fake = tq.tq_packed_bufs(16, 16, 16, 16, None, None)
    st = lib.tq_compress(ctypes.byref(L), ctypes.byref(rot), None, ctypes.c_void_p(16), ctypes.c_void_p(16),
                         65, 0, 0, 128, 0, ctypes.byref(fake), None)
    assert st == -4
    # misaligned pointer
    st = lib.tq_compress(ctypes.byref(L), ctypes.byref(rot), None, ctypes.c_void_p(18), ctypes.c_void_p(16),
                         8, 0, 0, 128, 0, ctypes.byref(fake), None)
    assert st == -3
    # a feature the head dims other than 128 do not take (QJL sketches)
    L64 = tq.make_layout(1, 8, 64, 64, 3, 3, qjl=[1] + [0] * 7)
    rot64 = tq.tq_make_rotation(64, 42)
    st = lib.tq_compress(ctypes.byref(L64), ctypes.byref(rot64), ctypes.c_void_p(16), ctypes.c_void_p(16),
                         ctypes.c_void_p(16), 8, ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(64),
                         0, ctypes.byref(tq.tq_packed_bufs(16, 16, 16, 16, 16, 16)), None)
    assert st == -2
    # decode: GQA 8 unsupported, bad head counts rejected
    seg = tq.Fp16Segment(1, 2, 128, 16, device="cpu", n_tokens=4)
    lv = tq.layer_view(rot, [seg])
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_workspace_size([lv], 1, 2, 16, 128)
    assert e.value.status == -2
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_workspace_size([lv], 1, 2, 3, 128)
    assert e.value.status == -1
    assert tq.tq_decode_workspace_size([lv], 1, 2, 8, 128) > 0
    with pytest.raises(tq.TQError) as e:  # unknown QJL estimator
        tq.tq_decode_workspace_size([tq.layer_view(rot, [seg], qjl_estimator=2)], 1, 2, 8, 128)
    assert e.value.status == -1
    # an attention-mass buffer adds the merged (max, sum) table to the workspace
    seg.attn_mass = torch.zeros(1, 2, 16)
    assert tq.tq_decode_workspace_size([tq.layer_view(rot, [seg])], 1, 2, 8, 128) >= \
        tq.tq_decode_workspace_size([lv], 1, 2, 8, 128)
    seg.attn_mass = None
    # packed capacity must keep scale rows 16-byte aligned
    P = tq.PackedSegment(tq.make_layout(1, 2, 128, 40, 3, 3), device="cpu", n_tokens=10)
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_workspace_size([tq.layer_view(rot, [P])], 1, 2, 8, 128)
    assert e.value.status == -3
    with pytest.raises(tq.TQError):
        tq.tq_age_tiers(10, [5, 3])
    # head_dim 64 / 256 / 512: GQA 1-4 plan (1, 2, 4 on the split-K kernels, 3
    # on the generic one); QJL keys and attention-mass outputs stay at 128
    for d in (64, 256, 512):
        rotd = tq.tq_make_rotation(d, 42)
        Pd = tq.PackedSegment(tq.make_layout(1, 2, d, 48, 3, 3), device="cpu", n_tokens=40)
        for hq in (2, 4, 6, 8):
            assert tq.tq_decode_workspace_size([tq.layer_view(rotd, [Pd])], 1, 2, hq, d) > 0
        Pq = tq.PackedSegment(tq.make_layout(1, 2, d, 48, 2, 3, qjl=[1, 0]), device="cpu", n_tokens=40)
        with pytest.raises(tq.TQError) as e:
            tq.tq_decode_workspace_size([tq.layer_view(rotd, [Pq])], 1, 2, 8, d)
        assert e.value.status == -2
        Pd.attn_mass = torch.zeros(1, 2, 48)
        with pytest.raises(tq.TQError) as e:
            tq.tq_decode_workspace_size([tq.layer_view(rotd, [Pd])], 1, 2, 8, d)
        assert e.value.status == -2


def test_requantize_argument_errors(tq):
    lib = tq._lib
    fake = tq.tq_packed_bufs(16, 16, 16, 16, None, None)
    src = tq.make_layout(2, 4, 128, 64, 4, 4)

    def call(dst_layout, s0=0, d0=0, n=8, src_layout=src):
        return lib.tq_requantize(ctypes.byref(src_layout), ctypes.byref(fake), s0, ctypes.byref(dst_layout),
                                 ctypes.byref(fake), d0, n, None)
    assert call(tq.make_layout(2, 2, 128, 64, 3, 2)) == -1           # head counts differ
    assert call(tq.make_layout(1, 4, 128, 64, 3, 2)) == -1           # batch differs
    assert call(tq.make_layout(2, 4, 128, 64, 2, 2, qjl=[1, 0, 0, 0])) == -2  # QJL on the destination
    assert call(tq.make_layout(2, 4, 128, 32, 3, 2), d0=30) == -4    # destination range past capacity
    assert call(tq.make_layout(2, 4, 128, 64, 3, 2), s0=60) == -4    # source range past capacity
    assert call(tq.make_layout(2, 4, 128, 64, 9, 2)) == -1           # width outside 1..8
    assert call(tq.make_layout(2, 4, 128, 64, 3, 2), n=0) == 0       # nothing to do
    odd = tq.tq_packed_bufs(18, 16, 16, 16, None, None)
    assert lib.tq_requantize(ctypes.byref(src), ctypes.byref(odd), 0,
                             ctypes.byref(tq.make_layout(2, 4, 128, 64, 3, 2)), ctypes.byref(fake), 0, 8,
                             None) == -3                                # misaligned buffer


def test_product_binding_has_no_fallback():
    # the binding refuses to import without the library rather than falling back
    src = open(os.path.join(ROOT, "rotated_quantized_kv_gb300", "tq.py")).read()
    assert "raise ImportError" in src and "oracle" not in src.lower().replace("no fallback", "")
