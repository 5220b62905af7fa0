"""The decode kernels' bounded waits, made to run out on purpose.

A split-K CTA that waits too long for a stage of its own bulk copies stops: it
lets the copies it issued land (that drain keeps the full bound), leaves the
(layer, batch, KV head) groups it touched unmerged, and sets the workspace's
error flag, which tq_decode_error_flag reports as TQ_ERR_TIMEOUT.  The test
shortens the consumer wait to zero polls through the library's failure-path
hook, so every wait gives up at once: no copy is lost, no address is invalid,
nothing spins.  It then checks the flag, that the output was left unwritten,
that the next call clears the flag, and that a normal call afterwards still
matches a call that never timed out, bit for bit."""
import numpy as np
import pytest
import torch

from rotated_quantized_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq as T
    return T


def _packed_cache(tq, L, B, H, T, seed, d=128):
    w = W.Workload("t", layers=L, batch=B, context=T, kv_heads=H, head_dim=d, law="outliers")
    keep, views = [], []
    for l in range(L):
        rot = tq.tq_make_rotation(d, 42 + l)
        K, V = W.kv_block(w, l, B, T, seed)
        seg = tq.PackedSegment(tq.make_layout(B, H, d, T, [3] * H, [3] * H))
        tq.tq_compress(seg, rot, K.cuda(), V.cuda())
        keep.append(seg)
        views.append(tq.layer_view(rot, [seg]))
    return keep, tq.views_array(views)


@pytest.mark.parametrize("d", [128, 256, 64])  # 256: 128-dim sub-records; 64: token pairs
def test_decode_wait_timeout_sets_flag_and_clears(tq, d):
    L, B, H, Hq, T = 2, 2, 4, 16, 1024
    keep, arr = _packed_cache(tq, L, B, H, T, seed=5, d=d)
    ws = torch.empty(tq.tq_decode_workspace_size(list(arr), B, H, Hq, d), dtype=torch.uint8, device="cuda")
    q = torch.randn(L, B, Hq, d, generator=torch.Generator().manual_seed(3)).half().cuda()
    ref = torch.empty(L, B, Hq, d, device="cuda")
    tq.tq_decode_attention(None, q, ref, ws, H, views=arr)
    assert tq.tq_decode_error_flag(ws) == 0

    out = torch.full((L, B, Hq, d), float("nan"), device="cuda")
    try:
        tq.tq_set_decode_wait_polls(0)
        tq.tq_decode_attention(None, q, out, ws, H, views=arr)
        flag = tq.tq_decode_error_flag(ws)
    finally:
        tq.tq_set_decode_wait_polls(tq.TQ_WAIT_POLLS_DEFAULT)
    assert flag != 0
    # every group's CTAs gave up before their merge: nothing was written
    assert torch.isnan(out).all()
    # the status the C call returns with the flag set
    import ctypes
    f = ctypes.c_int()
    assert tq._lib.tq_decode_error_flag(ws.data_ptr(), ctypes.byref(f), None) == tq.TQ_ERR_TIMEOUT
    assert f.value != 0

    # the next call clears the flag and computes the same bits as before
    out2 = torch.full_like(out, float("nan"))
    tq.tq_decode_attention(None, q, out2, ws, H, views=arr)
    assert tq.tq_decode_error_flag(ws) == 0
    assert torch.equal(out2, ref)


def test_wait_polls_hook_rejects_out_of_range(tq):
    for bad in (-1, (1 << 20) + 1):
        with pytest.raises(tq.TQError) as e:
            tq.tq_set_decode_wait_polls(bad)
        assert e.value.status == -1
