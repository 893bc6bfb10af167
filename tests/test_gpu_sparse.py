"""Sparse draft-decode attention on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import self_speculative_sparse_paged_gb300 as vg  # noqa: E402
from vegas_case import Case, assert_attention_close, bf16_to_f64, to_dev  # noqa: E402
from workload import configs, gen  # noqa: E402

pytestmark = pytest.mark.gpu

T, C2, C4 = configs.TINY, configs.QWEN3_8B_B1_32K, configs.GPTOSS_20B_B4_128K

CASES = {
    "tiny": T,
    "qwen_b2": C2.with_(batch=2, ctx_lo=2999, ctx_hi=4100),
    "gptoss_b2": C4.with_(batch=2, ctx_lo=3000, ctx_hi=3000),
    "group16": T.with_(hq=32, hkv=2, ctx_lo=1200, ctx_hi=1200),
    "group16_d128": C2.with_(hq=32, hkv=2, ctx_lo=2000, ctx_hi=2000),   # two column tiles at d 128
    "k_equals_L": T.with_(ctx_lo=700, ctx_hi=700, k_abs=700),
    "big_k": C2.with_(hkv=2, hq=8, ctx_lo=30000, ctx_hi=30000, k_pct=10),
    # one query head a KV head at head_dim 64: 64 output elements over a large cluster,
    # so some CTAs own none of them and receive only the row maxima and sums
    "mha_g1_wide_cluster": T.with_(hq=4, hkv=4, ctx_lo=10000, ctx_hi=10000, k_abs=760),
}


def _oracle_idx(c: Case):
    kf, _ = c.caches_f64()
    s = oracle.capture_scores(c.qv_f64(), kf, c.pm.block_table, c.lens, c.scale)
    return oracle.select_topk_batch(s, c.lens, c.kps, c.k_max)


@pytest.mark.parametrize("name", list(CASES))
def test_sparse_matches_oracle(name):
    c = Case(CASES[name])
    idx = _oracle_idx(c)
    kf, vf = c.caches_f64()
    for j in range(c.w.gamma):
        out = c.sparse(j, to_dev(idx))
        tl = c.w.gamma + 2 + j
        ref = oracle.sparse_decode(c.qd_f64()[j], kf, vf, c.pm.block_table, idx, c.kps, c.lens,
                                   np.full(c.w.batch, tl), c.scale)
        assert_attention_close(bf16_to_f64(out), ref, f"draft step {j}")


@pytest.mark.parametrize("rows", [16384, 32768])
def test_sparse_at_the_largest_attention_sets(rows):
    """k_per_seq + tail up to the call's limit (32768 entries: sixteen CTAs with
    full row tables at the limit, 1024 entries each at half of it), on random
    distinct positions of a 33K prefix."""
    w = C2.with_(batch=1, hq=4, hkv=1, ctx_lo=33000, ctx_hi=33000)
    c = Case(w)
    tl = gen.tail_len(w, 0)
    k = rows - tl
    rng = np.random.default_rng(rows)
    idx = np.sort(rng.choice(int(c.lens[0]), size=k, replace=False)).astype(np.int32)
    idx = idx.reshape(1, 1, k)
    out = c.sparse(0, to_dev(idx), k_per_seq=[k])
    kf, vf = c.caches_f64()
    ref = oracle.sparse_decode(c.qd_f64()[0], kf, vf, c.pm.block_table, idx, np.array([k]),
                               c.lens, np.array([tl]), c.scale)
    assert_attention_close(bf16_to_f64(out), ref, f"{rows} entries")


def test_sparse_full_prefix_reduces_to_verify_rows():
    """T = [0, L_b) with tail [L_b, L_b + t + 1) attends exactly what verify row t attends."""
    c = Case(T.with_(ctx_lo=1500, ctx_hi=1500, k_abs=1500))
    out_v, _ = c.verify(capture=False)
    idx = np.tile(np.arange(1500, dtype=np.int32), (1, c.w.hkv, 1))
    for t in range(c.w.gamma + 1):
        q = c.qv[:, t].contiguous()
        o = c.sparse(0, to_dev(idx), tail_len=t + 1, q=q)
        np.testing.assert_allclose(bf16_to_f64(o), bf16_to_f64(out_v[:, t]), atol=2e-2)


def test_sparse_tail_only():
    c = Case(T.with_(ctx_lo=300, ctx_hi=300, k_abs=0))
    kf, vf = c.caches_f64()
    idx = np.zeros((1, c.w.hkv, 1), dtype=np.int32)
    out = c.sparse(1, to_dev(idx), k_per_seq=[0])
    ref = oracle.sparse_decode(c.qd_f64()[1], kf, vf, c.pm.block_table, idx, np.array([0]),
                               c.lens, np.array([c.w.gamma + 3]), c.scale)
    assert_attention_close(bf16_to_f64(out), ref, "tail only")


@pytest.mark.parametrize("name,sink,window", [("qwen_b2", 4, 200), ("gptoss_b2", 0, 96),
                                              ("tiny", 16, 4000)])
def test_sparse_over_window_selection_matches_oracle(name, sink, window):
    """The query-agnostic window set feeds the same draft kernel."""
    c = Case(CASES[name])
    w = c.w
    k_max = sink + window
    idx = torch.full((w.batch, w.hkv, k_max), -7, dtype=torch.int32, device="cuda")
    ks = torch.zeros((w.batch,), dtype=torch.int32, device="cuda")
    vg.vegas_select_window(c.lens_t, sink, window, ks, idx, w.batch, w.hkv, k_max)
    ref_idx, ref_k = oracle.window_select_batch(c.lens, sink, window, w.hkv, k_max)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    kf, vf = c.caches_f64()
    for j in range(w.gamma):
        out = c.sparse(j, idx, k_per_seq=ref_k)
        tl = w.gamma + 2 + j
        ref = oracle.sparse_decode(c.qd_f64()[j], kf, vf, c.pm.block_table, ref_idx, ref_k,
                                   c.lens, np.full(w.batch, tl), c.scale)
        assert_attention_close(bf16_to_f64(out), ref, f"window draft step {j}")
