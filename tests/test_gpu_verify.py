"""Verify attention + Collect-2-Query capture on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import self_speculative_sparse_paged_gb300 as vg  # noqa: E402
from vegas_case import Case, assert_attention_close, bf16_to_f64, score_bound  # noqa: E402
from workload import configs  # noqa: E402

pytestmark = pytest.mark.gpu

T, C2, C3, C4 = (configs.TINY, configs.QWEN3_8B_B1_32K, configs.QWEN3_8B_B8_48K_64K,
                 configs.GPTOSS_20B_B4_128K)

SMALL = {
    "tiny": T,
    "qwen_b1_ragged": C2.with_(ctx_lo=3001, ctx_hi=3001),
    "qwen_b3_var": C3.with_(batch=3, ctx_lo=900, ctx_hi=2100),
    "gptoss_b2": C4.with_(batch=2, ctx_lo=2500, ctx_hi=2500),
    "gamma0": C2.with_(gamma=0, ctx_lo=37, ctx_hi=37),
    "len1": T.with_(ctx_lo=1, ctx_hi=1, k_abs=1),
    "len0": T.with_(ctx_lo=0, ctx_hi=0, k_abs=0),
    "qwen_gamma8": C2.with_(gamma=8, ctx_lo=1500, ctx_hi=1500),     # 36 rows, Q in smem
    "qwen_gamma10": C2.with_(gamma=10, ctx_lo=700, ctx_hi=700),     # 44 rows + 2 capture
    "gptoss_gamma6_g9": C4.with_(batch=1, hq=72, hkv=8, gamma=5, ctx_lo=900, ctx_hi=900),  # 54 rows
    "mha_g1": T.with_(hq=4, hkv=4, gamma=3, ctx_lo=600, ctx_hi=600),
    "odd_rows_g3": C4.with_(batch=1, hq=24, hkv=8, gamma=4, ctx_lo=500, ctx_hi=500),
    "long_split": C2.with_(ctx_lo=20000, ctx_hi=20000, hkv=2, hq=8),       # 16-CTA clusters
    "cluster3_ragged": C2.with_(ctx_lo=400, ctx_hi=400),                   # 3 splits of 9, 9, 8 pages
    "qwen_b2_mixed": C3.with_(batch=2, ctx_lo=150, ctx_hi=6000),           # one short, one long
    "tc_ticket_b13": C3.with_(batch=13, ctx_lo=600, ctx_hi=900),           # 104 units: workspace merge
    "gptoss_b5_ragged": C4.with_(batch=5, ctx_lo=3000, ctx_hi=9000),      # 40 units, 3-CTA clusters
    "gptoss_b3_short": C4.with_(batch=3, ctx_lo=1, ctx_hi=700),           # a few tiles a unit
    "gamma15_g2": C2.with_(hq=16, hkv=8, gamma=15, ctx_lo=1000, ctx_hi=1000),   # largest gamma
    "gptoss_gamma15_g3": C4.with_(batch=1, hq=24, hkv=8, gamma=15, ctx_lo=900, ctx_hi=900),
    "g16_gamma1": C2.with_(hq=32, hkv=2, gamma=1, ctx_lo=1500, ctx_hi=1500),   # 16 heads a group
    "gptoss_g16_gamma2": C4.with_(batch=1, hq=32, hkv=2, gamma=2, ctx_lo=1500, ctx_hi=1500),
}


def _check_case(c: Case, rows=None, capture=True, mask=None):
    if mask is not None:
        rows = [t for t in range(c.w.gamma + 1) if (mask >> t) & 1]
    out, scores = c.verify(capture=capture, rows=rows, mask=mask)
    kf, vf = c.caches_f64()
    qv = c.qv_f64()
    ref_o = oracle.verify_attention(qv, kf, vf, c.pm.block_table, c.lens, c.scale)
    assert_attention_close(bf16_to_f64(out), ref_o, "verify output")
    if not capture:
        return out, None
    rows = rows if rows is not None else (0, c.w.gamma)
    ref_s = oracle.capture_scores(qv, kf, c.pm.block_table, c.lens, c.scale,
                                  rows=sorted(set(rows)))
    got = scores.cpu().numpy().astype(np.float64)
    G = c.w.group
    for b in range(c.w.batch):
        L = int(c.lens[b])
        for g in range(c.w.hkv):
            if L == 0:
                continue
            K = oracle.gather_rows(kf, c.pm.block_table[b], g, np.arange(L))
            qr = np.concatenate([qv[b, t, g * G:(g + 1) * G] for t in sorted(set(rows))])
            bound = score_bound(qr, K, c.scale) + 1e-30
            err = np.abs(got[b, g, :L] - ref_s[b, g, :L])
            assert np.all(err <= bound), f"score error {err.max()} > bound (b={b}, g={g})"
            # positions past L_b are never written
            assert np.all(np.isnan(got[b, g, L:])), "score written past the prefix"
    return out, scores


@pytest.mark.parametrize("name", list(SMALL))
def test_verify_capture_matches_oracle(name):
    _check_case(Case(SMALL[name]))


@pytest.mark.parametrize("w", [C2.with_(gamma=11, ctx_lo=700, ctx_hi=700),
                               C4.with_(batch=1, gamma=7, ctx_lo=900, ctx_hi=900)],
                         ids=["qwen_48rows", "gptoss_64rows"])
def test_verify_without_capture_at_the_row_limit(w):
    """(gamma+1)*G at the tile limit (48 rows at d=128, 64 at d=64) without capture."""
    _check_case(Case(w), capture=False)


def test_capture_switch_leaves_output_bit_identical():
    c = Case(SMALL["qwen_b3_var"])
    o1, _ = c.verify(capture=True)
    o2, _ = c.verify(capture=False)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


@pytest.mark.parametrize("rows", [(0, 0), (1, 4), (4, 4), (2, 3)])
def test_capture_row_choice(rows):
    _check_case(Case(T), rows=rows)


@pytest.mark.parametrize("name,mask", [("tiny", "all"), ("qwen_b1_ragged", "all"),
                                       ("gptoss_b2", "all"), ("qwen_b3_var", 0b10110),
                                       ("long_split", "all")])
def test_capture_row_mask_matches_oracle(name, mask):
    # collect-all (every window row) and an arbitrary row set, against the oracle's
    # sum over the same rows; the attention output is the two-row call's, bit for bit
    c = Case(SMALL[name])
    m = (1 << (c.w.gamma + 1)) - 1 if mask == "all" else mask
    out, _ = _check_case(c, mask=m)
    out2, _ = c.verify()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_capture_row_mask_rejects_rows_past_gamma():
    c = Case(T)
    with pytest.raises(vg.VegasError) as ei:
        c.verify(mask=1 << (c.w.gamma + 1))
    assert ei.value.status == 1
    with pytest.raises(vg.VegasError):
        c.verify(mask=0)


def test_repeat_calls_are_deterministic():
    c = Case(SMALL["gptoss_b2"])
    o1, s1 = c.verify()
    o2, s2 = c.verify()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(s1, s2)


def test_cluster_merged_shape_needs_no_workspace():
    # 64 (sequence, KV head) units at head_dim 128: one 2-CTA cluster per unit,
    # whose splits merge on chip
    c = Case(C3.with_(batch=8, ctx_lo=2000, ctx_hi=2000), device_gen=True)
    w = c.w
    assert vg.vegas_verify_workspace_size(c.kv, w.batch, w.gamma) == 0
    ref_out, ref_scores = c.verify()
    out = torch.empty_like(c.qv)
    scores = torch.full_like(ref_scores, float("nan"))
    vg.vegas_verify_attn_capture(c.kv, c.qv, out, scores, c.stride, c.lens_t, w.batch, w.gamma,
                                 0, w.gamma, c.scale, None, 0)
    vg.vegas_read_device_status()
    assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(scores[..., :2000], ref_scores[..., :2000])


def test_several_clusters_per_unit_merge_through_the_workspace():
    """Few units (2 KV heads at batch 1): each unit's splits form several
    clusters, merged on chip within a cluster and through a few workspace rows
    across clusters; repeated calls leave the tickets at zero and give identical
    results."""
    c = Case(C2.with_(ctx_lo=5000, ctx_hi=5000, hkv=2, hq=8))
    w = c.w
    nb = vg.vegas_verify_workspace_size(c.kv, w.batch, w.gamma)
    assert nb > 0
    ref_out, ref_scores = _check_case(c)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")       # one workspace, reused
    for _ in range(2):
        out = torch.empty_like(c.qv)
        scores = torch.full_like(ref_scores, float("nan"))
        vg.vegas_verify_attn_capture(c.kv, c.qv, out, scores, c.stride, c.lens_t, w.batch,
                                     w.gamma, 0, w.gamma, c.scale, ws, nb)
        vg.vegas_read_device_status()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))
        assert torch.equal(scores[..., :5000], ref_scores[..., :5000])


@pytest.mark.parametrize("name", ["tiny", "qwen_b1_ragged", "gptoss_b2", "qwen_b3_var"])
def test_raw_logits_and_their_aggregate_match_oracle(name):
    """The pages' capture: raw logits of rows {0, gamma} for every query head, then
    summed per KV head by the aggregation kernel; the attention output is the
    capture-free verify's, bit for bit."""
    c = Case(SMALL[name])
    w = c.w
    rows = sorted({0, w.gamma})
    mask = sum(1 << t for t in rows)
    R = len(rows)
    raw = torch.full((w.batch, R, w.hq, c.stride), float("nan"), device="cuda")
    out = torch.empty_like(c.qv)
    nbytes = vg.vegas_verify_workspace_size(c.kv, w.batch, w.gamma)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    vg.vegas_verify_attn_raw_logits(c.kv, c.qv, out, raw, c.stride, c.lens_t, w.batch, w.gamma,
                                    mask, c.scale, ws, ws.numel())
    scores = torch.full((w.batch, w.hkv, c.stride), float("nan"), device="cuda")
    vg.vegas_aggregate_raw_logits(raw, c.stride, c.lens_t, w.batch, R, w.hq, w.hkv,
                                  int(c.lens.max()), scores, c.stride)
    vg.vegas_read_device_status()
    plain, _ = c.verify(capture=False)
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))
    kf, _ = c.caches_f64()
    qv = c.qv_f64()
    ref_raw = oracle.raw_capture_logits(qv, kf, c.pm.block_table, c.lens, c.scale, rows)
    ref_s = oracle.capture_scores(qv, kf, c.pm.block_table, c.lens, c.scale, rows=rows)
    got_raw = raw.cpu().numpy().astype(np.float64)
    got_s = scores.cpu().numpy().astype(np.float64)
    G = w.group
    for b in range(w.batch):
        L = int(c.lens[b])
        if L == 0:
            continue
        for g in range(w.hkv):
            K = oracle.gather_rows(kf, c.pm.block_table[b], g, np.arange(L))
            for r, t in enumerate(rows):
                for h in range(g * G, (g + 1) * G):
                    bound = score_bound(qv[b, t, h][None], K, c.scale) + 1e-30
                    err = np.abs(got_raw[b, r, h, :L] - ref_raw[b, r, h, :L])
                    assert np.all(err <= bound), f"raw logit error {err.max()} (b={b} h={h})"
            qr = np.concatenate([qv[b, t, g * G:(g + 1) * G] for t in rows])
            bound = score_bound(qr, K, c.scale) + 1e-30
            err = np.abs(got_s[b, g, :L] - ref_s[b, g, :L])
            assert np.all(err <= bound), f"aggregated score error {err.max()} (b={b}, g={g})"
