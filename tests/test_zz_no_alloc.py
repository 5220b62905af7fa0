"""tq_decode_attention_static: decode attention for callers that may not allocate
device memory while they run (serving loops that reserve all device memory at
start-up, or hosts whose device memory belongs to another allocator).  Its
scratch is the library's fixed device array instead of a caller workspace.

Checked through the C ABI against tq_decode_attention (caller workspace) on two
calls in a row.  The array keeps the previous call's contents, so the second
call has another shape (fewer layers, another batch, QJL heads with their
projection matrix): its plan tables, counters and partial records sit at other
offsets, and a stale read of the first call's scratch would change its result.
Both entry points run the same kernels on the same inputs in the same order,
so the outputs must agree bit for bit.  Collected last on purpose; runs alone
too."""
import ctypes

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


def _cache(tq, L, B, H, seed, qjl_S=None):
    w = W.Workload("t", layers=L, batch=B, context=600, kv_heads=H, law="outliers")
    keep, views = [], []
    for l in range(L):
        rot = tq.tq_make_rotation(128, 42 + l)
        K, V = W.kv_block(w, l, B, 600, seed)
        sink = tq.Fp16Segment(B, H, 128, 32, n_tokens=32, k=K[:, :, :32].contiguous().cuda(),
                              v=V[:, :, :32].contiguous().cuda())
        kb = [(3 + h + l) % 8 + 1 for h in range(H)]
        vb = [(5 + 2 * h + l) % 8 + 1 for h in range(H)]
        qjl = [int(h % 2 == 0) for h in range(H)] if qjl_S is not None else None
        seg = tq.PackedSegment(tq.make_layout(B, H, 128, 576, kb, vb, qjl))
        tq.tq_compress(seg, rot, K[:, :, 32:].cuda(), V[:, :, 32:].cuda(),
                       qjl_S=qjl_S if qjl and any(qjl) else None)
        keep.append((sink, seg))
        views.append(tq.layer_view(rot, [sink, seg]))
    return keep, views


def test_static_workspace_matches_caller_workspace_twice(tq):
    lib = ctypes.CDLL(tq.LIB_PATH)
    lib.tq_decode_attention_static.restype = ctypes.c_int
    lib.tq_decode_attention_static.argtypes = tq._lib.tq_decode_attention_static.argtypes
    lib.tq_decode_error_flag.restype = ctypes.c_int
    lib.tq_decode_error_flag.argtypes = tq._lib.tq_decode_error_flag.argtypes
    stream = torch.cuda.current_stream().cuda_stream
    S = tq.tq_make_qjl(128, 128, W.QJL_SEED).cuda()
    # call 1: three layers, batch 2, no QJL; call 2: two layers, batch 3, QJL heads
    shapes = [(3, 2, 4, 16, None), (2, 3, 4, 16, S)]
    for call, (L, B, H, Hq, qjl_S) in enumerate(shapes):
        keep, views = _cache(tq, L, B, H, seed=31 + call, qjl_S=qjl_S)
        if qjl_S is not None:
            assert any(v for _, seg in keep for v in seg.layout.qjl[:H])
        arr = tq.views_array(views)
        ws = torch.empty(tq.tq_decode_workspace_size(views, B, H, Hq, 128), dtype=torch.uint8, device="cuda")
        q = torch.randn(L, B, Hq, 128, generator=torch.Generator().manual_seed(call)).half().cuda()
        ref = torch.full((L, B, Hq, 128), float("nan"), device="cuda")
        out = torch.full((L, B, Hq, 128), float("nan"), device="cuda")
        tq.tq_decode_attention(None, q, ref, ws, H, qjl_S=qjl_S, views=arr)
        st = lib.tq_decode_attention_static(arr, L, B, H, Hq, 128, None if qjl_S is None else qjl_S.data_ptr(),
                                            128, q.data_ptr(), out.data_ptr(), stream)
        assert st == 0, tq._lib.tq_status_string(st)
        flag = ctypes.c_int(-1)
        assert lib.tq_decode_error_flag(None, ctypes.byref(flag), stream) == 0
        assert flag.value == 0
        torch.cuda.synchronize()
        r, o = ref.cpu().numpy(), out.cpu().numpy()
        assert np.all(np.isfinite(r))
        assert np.array_equal(o, r), f"call {call}: static and caller-workspace outputs differ"


def test_static_workspace_rejects_oversized_calls(tq):
    # 2048 sequences x 8 KV heads: one split-K partial each, more scratch than
    # the fixed array holds
    B, H, Hq = 2048, 8, 32
    seg = tq.Fp16Segment(B, H, 128, 16, n_tokens=1)
    views = [tq.layer_view(tq.tq_make_rotation(128, 42), [seg])]
    assert tq.tq_decode_workspace_size(views, B, H, Hq, 128) > tq.TQ_STATIC_WORKSPACE_BYTES
    q = torch.zeros(1, B, Hq, 128, dtype=torch.float16, device="cuda")
    out = torch.zeros(1, B, Hq, 128, device="cuda")
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention_static(views, q, out, H)
    assert e.value.status == -4
    # argument errors come before the size check, as for tq_decode_attention
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention_static(views, q[:, :, :, 1:], out, H)
    assert e.value.status in (-1, -3)
