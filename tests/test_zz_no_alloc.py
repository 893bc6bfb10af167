"""The verify entry point that allocates nothing, for callers that cannot call
cudaMalloc (a plugin whose host framework owns all device memory, or a decode
loop that must not risk cudaMalloc's device synchronisation).

It runs the same kernel on the same inputs as vegas_verify_attn_capture with a
caller workspace, so its outputs and captured scores must be bit-identical to
that call's, on two calls in a row (the fixed scratch array is shared between
calls and keeps the previous call's contents).  This file is collected last.
"""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import self_speculative_sparse_paged_gb300 as vg  # noqa: E402
from vegas_case import Case  # noqa: E402
from workload import configs  # noqa: E402

pytestmark = pytest.mark.gpu


def _noalloc(c: Case):
    w = c.w
    out = torch.full_like(c.qv, float("nan"))
    scores = torch.full((w.batch, w.hkv, c.stride), float("nan"), device="cuda")
    vg.vegas_verify_attn_capture_noalloc(c.kv, c.qv, out, scores, c.stride, c.lens_t, w.batch,
                                         w.gamma, 0, w.gamma, c.scale)
    vg.vegas_read_device_status()
    return out, scores


# Shapes whose split-KV merge goes through the scratch: 44 query rows at
# head_dim 128 (the mma.sync kernel), and 160 (sequence, KV head) units (more
# than the SMs: the tcgen05 kernel's last-arriving-CTA merge).
@pytest.mark.parametrize("w", [
    configs.QWEN3_8B_B8_48K_64K.with_(batch=3, ctx_lo=3000, ctx_hi=9000, gamma=10),
    configs.QWEN3_8B_B8_48K_64K.with_(batch=20, ctx_lo=250, ctx_hi=300),
], ids=["qwen_b3_gamma10", "qwen_b20_160_units"])
def test_noalloc_matches_workspace_entry_point_twice(w):
    c = Case(w, device_gen=True)
    assert 0 < vg.vegas_verify_workspace_size(c.kv, w.batch, w.gamma) <= \
        vg.vegas_verify_noalloc_max_scratch_bytes()
    ref_out, ref_scores = c.verify()
    for _ in range(2):
        out, scores = _noalloc(c)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), \
            "no-alloc verify output differs from the workspace call"
        for b in range(w.batch):
            L = int(c.lens[b])
            got, exp = scores[b, :, :L].cpu().numpy(), ref_scores[b, :, :L].cpu().numpy()
            np.testing.assert_array_equal(got.view(np.uint32), exp.view(np.uint32))


def test_noalloc_rejects_shapes_beyond_the_scratch():
    """512 sequences x 8 KV heads: the partials of 4096 units exceed the fixed
    array.  Every buffer is real and sized for the shape (one cache page that all
    block-table entries name, ten-token prefixes), so the call could run safely
    even if the size check were missing; it must refuse instead."""
    big = configs.QWEN3_8B_B8_48K_64K.with_(batch=512, ctx_lo=4000, ctx_hi=4000)
    B, T, d = big.batch, big.gamma + 1, big.head_dim
    k = torch.zeros((1, big.hkv, 16, d), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    bt = torch.zeros((B, 256), dtype=torch.int32, device="cuda")
    kv = vg.paged_kv(k, v, bt, big.hq)
    q = torch.zeros((B, T, big.hq, d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lens = torch.full((B,), 10, dtype=torch.int32, device="cuda")
    assert vg.vegas_verify_workspace_size(kv, B, big.gamma) > \
        vg.vegas_verify_noalloc_max_scratch_bytes()
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_capture_noalloc(kv, q, out, None, 1, lens, B, big.gamma, 0,
                                             big.gamma, 0.1)
    assert ei.value.status == 3
    torch.cuda.synchronize()
