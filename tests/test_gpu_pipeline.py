"""One decode iteration over a stack of layers through vegas_decode_iteration:
every layer's verify, scores, indices and draft outputs against the oracle's
iteration of that layer, with select(l) pipelined against verify(l + 1) on a
second stream and serially (both orders give bit-identical results)."""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import self_speculative_sparse_paged_gb300 as vg  # noqa: E402
from vegas_case import (DEV, Case, assert_attention_close, bf16_to_f64, score_bound,  # noqa: E402
                        tie_band_ok, to_dev)
from workload import configs, gen  # noqa: E402

pytestmark = pytest.mark.gpu


class Stack:
    """`layers` layers of one workload, host-generated (the oracle sees the same bits)."""

    def __init__(self, w, layers):
        self.w = w
        self.cases = [Case(w, layer=l) for l in range(layers)]
        c0 = self.cases[0]
        self.lens_t, self.kps_t = c0.lens_t, c0.kps_t
        self.stride, self.k_max, self.scale = c0.stride, c0.k_max, c0.scale
        tails = np.array([[gen.tail_len(w, j)] * w.batch for j in range(w.gamma)], np.int32)
        self.tails_t = to_dev(tails)
        self.max_tail = int(tails.max())
        self.out_v = [torch.empty_like(c.qv) for c in self.cases]
        self.out_d = [torch.empty_like(c.qd) for c in self.cases]
        self.scores = [torch.empty((w.batch, w.hkv, self.stride), device=DEV) for _ in self.cases]
        self.idx = [torch.empty((w.batch, w.hkv, self.k_max), dtype=torch.int32, device=DEV)
                    for _ in self.cases]
        nb = vg.vegas_verify_workspace_size(c0.kv, w.batch, w.gamma)
        self.ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device=DEV)

    def run(self, side=None):
        for t in self.out_v + self.out_d:
            t.fill_(float("nan"))
        for t in self.idx:
            t.fill_(-7)
        w = self.w
        layers = [vg.layer(c.kv, c.qv, ov, c.qd, od, s, i) for c, ov, od, s, i in
                  zip(self.cases, self.out_v, self.out_d, self.scores, self.idx)]
        vg.vegas_decode_iteration(layers, self.lens_t, self.kps_t, self.tails_t, self.max_tail,
                                  w.batch, w.gamma, self.stride, self.k_max, self.scale, self.ws,
                                  self.ws.numel(), select_stream=side)
        vg.vegas_read_device_status()
        return ([o.clone() for o in self.out_v], [o.clone() for o in self.out_d],
                [s.clone() for s in self.scores], [i.clone() for i in self.idx])


def _check_layer_against_oracle(c: Case, out_v, out_d, scores, idx):
    w = c.w
    kf, vf = c.caches_f64()
    res = oracle.iteration(c.qv_f64(), c.qd_f64(), kf, vf, c.pm.block_table, c.lens, c.kps,
                           c.scale)
    assert_attention_close(bf16_to_f64(out_v), res["o_verify"], f"layer {c.layer} verify")
    got_idx = idx.cpu().numpy()
    s32 = scores.cpu().numpy().astype(np.float64)
    G = w.group
    for b in range(w.batch):
        L, k = int(c.lens[b]), int(c.kps[b])
        for g in range(w.hkv):
            pos = np.arange(L)
            K = oracle.gather_rows(kf, c.pm.block_table[b], g, pos)
            qr = c.qv_f64()[b][[0, w.gamma]][:, g * G:(g + 1) * G].reshape(-1, w.head_dim)
            assert np.all(np.abs(s32[b, g, :L] - res["scores"][b, g, :L])
                          <= score_bound(qr, K, c.scale)), f"layer {c.layer} scores ({b},{g})"
            np.testing.assert_array_equal(got_idx[b, g, :k], oracle.select_topk(s32[b, g, :L], k))
            ok, msg = tie_band_ok(got_idx[b, g, :k], res["idx"][b, g, :k],
                                  res["scores"][b, g, :L], k)
            assert ok, f"layer {c.layer}: {msg}"
    for j in range(w.gamma):
        ref = oracle.sparse_decode(c.qd_f64()[j], kf, vf, c.pm.block_table, got_idx, c.kps,
                                   c.lens, np.full(w.batch, gen.tail_len(w, j)), c.scale)
        assert_attention_close(bf16_to_f64(out_d[j]), ref, f"layer {c.layer} draft {j}")


@pytest.mark.parametrize("w,layers", [
    (configs.TINY, 3),
    (configs.QWEN3_8B_B8_48K_64K.with_(batch=2, ctx_lo=3000, ctx_hi=6000), 3),
], ids=["tiny_3_layers", "qwen_b2_3k_6k_3_layers"])
def test_layer_pipelined_iteration_matches_the_oracle_per_layer(w, layers):
    st = Stack(w, layers)
    side = torch.cuda.Stream(device=DEV)
    pip = st.run(side)
    ser = st.run(None)
    for a, b in zip(pip[0] + pip[1], ser[0] + ser[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(pip[2] + pip[3], ser[2] + ser[3]):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    for li, c in enumerate(st.cases):
        _check_layer_against_oracle(c, pip[0][li], pip[1][li], pip[2][li], pip[3][li])


def test_layer_pipelined_iteration_in_a_cuda_graph():
    """The call joins its select stream back, so it captures and replays as one graph."""
    w = configs.TINY
    st = Stack(w, 2)
    side = torch.cuda.Stream(device=DEV)
    ref = st.run(side)                     # first call creates the events
    s = torch.cuda.Stream(device=DEV)
    layers = [vg.layer(c.kv, c.qv, ov, c.qd, od, sc, i) for c, ov, od, sc, i in
              zip(st.cases, st.out_v, st.out_d, st.scores, st.idx)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        vg.vegas_decode_iteration(layers, st.lens_t, st.kps_t, st.tails_t, st.max_tail, w.batch,
                                  w.gamma, st.stride, st.k_max, st.scale, st.ws, st.ws.numel(),
                                  stream=s, select_stream=side)
    for t in st.out_d:
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    vg.vegas_read_device_status()
    for a, b in zip(ref[1], st.out_d):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
