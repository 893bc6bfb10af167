"""Whole iterations (verify + capture -> top-k -> gamma draft steps) on the GPU.

Small workloads are compared element by element with the oracle's iteration.
The full-size workloads (the Qwen3-8B / gpt-oss-20b layer shapes at 32K-128K
and the 36-layer stack) are compared on sampled (sequence, KV head) units that
the oracle recomputes one by one from the generator.
"""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
from vegas_case import (Case, assert_attention_close, bf16_to_f64, score_bound,  # noqa: E402
                        tie_band_ok)
from workload import configs, gen  # noqa: E402

pytestmark = pytest.mark.gpu


def _gpu_iteration(c: Case):
    out_v, scores = c.verify()
    idx = c.select(scores)
    drafts = [c.sparse(j, idx) for j in range(c.w.gamma)]
    return out_v, scores, idx, drafts


@pytest.mark.parametrize("w", [
    configs.TINY,
    configs.QWEN3_8B_B8_48K_64K.with_(batch=2, ctx_lo=3000, ctx_hi=5000),
    configs.GPTOSS_20B_B4_128K.with_(batch=2, ctx_lo=6000, ctx_hi=6000),
    configs.QWEN3_8B_B1_32K.with_(hq=16, hkv=8, gamma=15, ctx_lo=2000, ctx_hi=2000),
], ids=["tiny", "qwen_b2", "gptoss_b2", "qwen_gamma15_g2"])
def test_small_iteration_matches_oracle(w):
    c = Case(w)
    out_v, scores, idx, drafts = _gpu_iteration(c)
    kf, vf = c.caches_f64()
    res = oracle.iteration(c.qv_f64(), c.qd_f64(), kf, vf, c.pm.block_table, c.lens, c.kps,
                           c.scale)
    assert_attention_close(bf16_to_f64(out_v), res["o_verify"], "verify")
    got_idx = idx.cpu().numpy()
    s32 = scores.cpu().numpy().astype(np.float64)
    for b in range(w.batch):
        L, k = int(c.lens[b]), int(c.kps[b])
        for g in range(w.hkv):
            # bit-exact on identical (GPU fp32) scores
            np.testing.assert_array_equal(got_idx[b, g, :k], oracle.select_topk(s32[b, g, :L], k))
            ok, msg = tie_band_ok(got_idx[b, g, :k], res["idx"][b, g, :k], res["scores"][b, g, :L], k)
            assert ok, msg
    for j in range(w.gamma):
        ref = oracle.sparse_decode(c.qd_f64()[j], kf, vf, c.pm.block_table, got_idx, c.kps,
                                   c.lens, np.full(w.batch, w.gamma + 2 + j), c.scale)
        assert_attention_close(bf16_to_f64(drafts[j]), ref, f"draft {j}")


def _check_sampled_unit(c: Case, b: int, g: int, out_v, scores, idx, drafts):
    w = c.w
    L, k, G = int(c.lens[b]), int(c.kps[b]), w.group
    K, V = c.unit_rows(b, g, L + 2 * w.gamma + 1)
    qv, qd = c.qv_f64(), c.qd_f64()
    heads = range(g * G, (g + 1) * G)
    got_o = bf16_to_f64(out_v[b])
    ref_o = np.stack([[oracle.attention_row(qv[b, t, h], K[:L + t + 1], V[:L + t + 1], c.scale)
                       for h in heads] for t in range(w.gamma + 1)])
    assert_attention_close(got_o[:, g * G:(g + 1) * G], ref_o, f"verify unit ({b},{g})")
    rows = (0, w.gamma) if w.gamma > 0 else (0,)
    ref_s = sum(oracle.logits_row(qv[b, t, h], K[:L], c.scale) for t in rows for h in heads)
    got_s = scores[b, g, :L].cpu().numpy().astype(np.float64)
    qr = np.concatenate([qv[b, t, g * G:(g + 1) * G] for t in rows])
    assert np.all(np.abs(got_s - ref_s) <= score_bound(qr, K[:L], c.scale)), "captured scores"
    got_idx = idx[b, g].cpu().numpy()
    np.testing.assert_array_equal(got_idx[:k], oracle.select_topk(got_s, k))
    ok, msg = tie_band_ok(got_idx[:k], oracle.select_topk(ref_s, k), ref_s, k)
    assert ok, msg
    for j in range(w.gamma):
        pos = oracle.sparse_positions(got_idx, k, L, w.gamma + 2 + j)
        ref = np.stack([oracle.attention_row(qd[j, b, h], K[pos], V[pos], c.scale) for h in heads])
        assert_attention_close(bf16_to_f64(drafts[j][b, g * G:(g + 1) * G]), ref,
                               f"draft {j} unit ({b},{g})")


@pytest.mark.parametrize("w", [configs.QWEN3_8B_B1_32K, configs.QWEN3_8B_B8_48K_64K,
                               configs.GPTOSS_20B_B4_128K],
                         ids=["qwen3_8b_b1_32k", "qwen3_8b_b8_48k_64k", "gptoss_20b_b4_128k"])
def test_full_size_sampled_units(w):
    c = Case(w, device_gen=True)
    out_v, scores, idx, drafts = _gpu_iteration(c)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w.seed)
    units = {(0, 0), (w.batch - 1, w.hkv - 1)}
    units.add((int(rng.integers(w.batch)), int(rng.integers(w.hkv))))
    for b, g in sorted(units):
        _check_sampled_unit(c, b, g, out_v, scores, idx, drafts)


@pytest.mark.parametrize("gamma,pct", [(2, 3), (8, 10)])
def test_stack_full_size_sampled_layers(gamma, pct):
    """36-layer Qwen3-8B stack at 96K-120K: two layers (first and last) at full size."""
    w = configs.QWEN3_8B_36L_B4_96K_120K.with_(gamma=gamma, k_pct=pct)
    for layer in (0, w.layers - 1):
        c = Case(w, layer=layer, device_gen=True)
        out_v, scores, idx, drafts = _gpu_iteration(c)
        torch.cuda.synchronize()
        _check_sampled_unit(c, layer % w.batch, (3 * layer) % w.hkv, out_v, scores, idx, drafts)
        del c, out_v, scores, idx, drafts
        torch.cuda.empty_cache()
