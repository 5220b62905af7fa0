"""Host logic of the chunked decode cache: the per-step update of the layer
views writes, for every layer, the same fields as setting them one by one."""
import torch

from rotated_quantized_kv_gb300 import model_cache as MC


def test_step_fields_update_every_layer():
    from rotated_quantized_kv_gb300 import build
    build.build()
    from rotated_quantized_kv_gb300 import tq as T

    class Views(MC.ChunkedDecodeCache):
        def __init__(self):  # the view plumbing only, host tensors
            self.L, self.B, self.H, self.d = 3, 1, 2, 128
            self.n_prompt_packed, self.chunk, self.steps_cap = 1000, 64, 256
            self.pool_k = [torch.zeros(1, 2, 256, 128, dtype=torch.float16) for _ in range(3)]
            self.pool_v = [torch.zeros(1, 2, 256, 128, dtype=torch.float16) for _ in range(3)]
            rot = T.tq_make_rotation(128, 1)
            segs = [[T.Fp16Segment(1, 2, 128, 16, device="cpu", n_tokens=4),
                     T.PackedSegment(T.make_layout(1, 2, 128, 16, 3, 3), device="cpu"),
                     T.Fp16Segment(1, 2, 128, 256, device="cpu", n_tokens=1, k=self.pool_k[l], v=self.pool_v[l])]
                    for l in range(3)]
            self.arr = T.views_array([T.layer_view(rot, sg) for sg in segs])
            self._bind_step_fields()

    v = Views()
    for s, w0 in ((130, 128), (5, 0), (255, 192)):
        v.set_step(s)
        for l in range(3):
            sg = v.arr[l].seg
            assert sg[1].n_tokens == 1000 + w0 and sg[2].n_tokens == s - w0 + 1
            assert sg[2].k16 == v.pool_k[l].data_ptr() + w0 * 256
            assert sg[2].v16 == v.pool_v[l].data_ptr() + w0 * 256
            assert sg[0].n_tokens == 4 and v.arr[l].n_segments == 3
