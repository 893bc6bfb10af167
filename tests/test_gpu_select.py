"""Top-k select on the GPU: bit-exact against the oracle on identical fp32 scores."""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import self_speculative_sparse_paged_gb300 as vg  # noqa: E402
from vegas_case import DEV, Case, tie_band_ok, to_dev  # noqa: E402
from workload import configs  # noqa: E402

pytestmark = pytest.mark.gpu


def _run(scores32: np.ndarray, lens, kps, k_max, stride=None):
    B, H, S = scores32.shape
    idx = torch.full((B, H, k_max), -7, dtype=torch.int32, device=DEV)
    vg.vegas_select_topk(to_dev(scores32), S, to_dev(np.asarray(lens, np.int32)),
                         to_dev(np.asarray(kps, np.int32)), idx, B, H, k_max)
    vg.vegas_read_device_status()
    got = idx.cpu().numpy()
    ref = oracle.select_topk_batch(scores32.astype(np.float64), np.asarray(lens),
                                   np.asarray(kps), k_max)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("L,k", [(1, 1), (5, 2), (1000, 0), (1000, 1000), (1000, 37),
                                 (4097, 205), (32768, 1639), (65536, 3277), (131072, 3933),
                                 (262144, 5000), (65537, 60000), (131072, 131071),
                                 (131072, 131072), (262144, 262143)])
def test_select_random_scores(L, k):
    rng = np.random.default_rng(L + k)
    s = (rng.standard_normal((2, 3, L)) * 3).astype(np.float32)
    _run(s, [L, L], [k, k], max(k, 1) + 3)


def test_select_heavy_ties_and_signed_zero():
    rng = np.random.default_rng(1)
    s = rng.integers(-3, 3, size=(1, 4, 50000)).astype(np.float32)
    s[0, 1, ::2] = -0.0
    s[0, 1, 1::2] = 0.0
    s[0, 2, :] = 1.5
    _run(s, [50000], [777], 800)


@pytest.mark.parametrize("L,k", [(65536, 3277), (131072, 100)])
def test_select_ties_inside_the_chosen_bin(L, k):
    """About 64 equal keys per value, so the chosen value bin holds one tied
    group small enough to be resolved from its keys directly (wide chunks);
    ties go to the lower position."""
    rng = np.random.default_rng(L + 7)
    s = (rng.integers(0, L // 64, size=(2, 3, L)) * 0.25).astype(np.float32)
    _run(s, [L, L], [k, k], k + 5)


def test_select_variable_lengths_and_k():
    rng = np.random.default_rng(2)
    lens = [10, 40000, 3, 20001]
    kps = [10, 2000, 0, 1]
    s = (rng.standard_normal((4, 2, 40000)) * 10).astype(np.float32)
    _run(s, lens, kps, 2100)


def test_select_clustered_values():
    """Scores concentrated in a few float exponent bins (the radix worst case)."""
    rng = np.random.default_rng(3)
    s = (1000.0 + rng.integers(0, 64, size=(1, 8, 32768)) * 2.0 ** -10).astype(np.float32)
    _run(s, [32768], [1639], 1639)


@pytest.mark.parametrize("L,k", [(32768, 1639), (131072, 3933)])
def test_select_with_large_outliers(L, k):
    """A few logits a thousand times above (and below) the rest stretch the
    row's [min, max]: level 0's value bins then hold the bulk in one bin, and
    the search goes on by sub-bins and key bits."""
    rng = np.random.default_rng(L + 9)
    s = (rng.standard_normal((1, 4, L)) * 3).astype(np.float32)
    for h in range(4):
        pos = rng.choice(L, size=16, replace=False)
        s[0, h, pos[:8]] = 3000.0 * (1 + np.arange(8) / 16)
        s[0, h, pos[8:]] = -3000.0 * (1 + np.arange(8) / 16)
    _run(s, [L], [k], k + 3)


# ---------------------------------------------------------------- shared T (all heads)
def _run_shared(scores32: np.ndarray, lens, kps, k_max):
    B, H, S = scores32.shape
    idx = torch.full((B, H, k_max), -7, dtype=torch.int32, device=DEV)
    vg.vegas_select_topk_shared(to_dev(scores32), S, to_dev(np.asarray(lens, np.int32)),
                                to_dev(np.asarray(kps, np.int32)), idx, B, H, k_max)
    vg.vegas_read_device_status()
    # identical keys: the call's stated fp32 head-order sum, taken by both sides
    ref = oracle.select_topk_shared_batch_f32(scores32, np.asarray(lens), np.asarray(kps), k_max)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
    return idx


@pytest.mark.parametrize("L,k,H", [(1, 1, 8), (1000, 37, 8), (32768, 1639, 8),
                                   (131072, 3933, 8), (5000, 250, 1)])
def test_select_shared_random_scores(L, k, H):
    rng = np.random.default_rng(L + 7 * k + H)
    s = (rng.standard_normal((2, H, L)) * 3).astype(np.float32)
    _run_shared(s, [L, L], [k, k], k + 2)


def test_select_shared_ties_and_variable_lengths():
    rng = np.random.default_rng(5)
    s = rng.integers(-2, 3, size=(3, 4, 20000)).astype(np.float32)
    _run_shared(s, [20000, 7, 15000], [900, 7, 0], 1000)


@pytest.mark.parametrize("w", [configs.TINY,
                               configs.QWEN3_8B_B8_48K_64K.with_(batch=2, ctx_lo=3000, ctx_hi=6000)],
                         ids=["tiny", "qwen_b2_3k_6k"])
def test_select_shared_end_to_end_within_the_tie_band_of_the_exact_sum(w):
    """GPU capture then GPU shared select, against the method's definition: the
    fp64 sum over every head of the fp64 oracle's captured logits.  The sets may
    differ only at positions within the tie band of the k-th exact score."""
    c = Case(w)
    _, scores = c.verify()
    idx = torch.full((w.batch, w.hkv, c.k_max), -7, dtype=torch.int32, device=DEV)
    vg.vegas_select_topk_shared(scores, c.stride, c.lens_t, c.kps_t, idx, w.batch, w.hkv,
                                c.k_max)
    vg.vegas_read_device_status()
    got = idx.cpu().numpy()
    kf, _ = c.caches_f64()
    ref_s = oracle.capture_scores(c.qv_f64(), kf, c.pm.block_table, c.lens, c.scale)
    ref = oracle.select_topk_shared_batch(ref_s, c.lens, c.kps, c.k_max)
    for b in range(w.batch):
        L, k = int(c.lens[b]), int(c.kps[b])
        summed = oracle.summed_head_scores(ref_s, L, b)
        assert (got[b] == got[b, 0]).all(), "one T for every KV head"
        ok, msg = tie_band_ok(got[b, 0, :k], ref[b, 0, :k], summed, k)
        assert ok, msg
        assert (got[b, :, k:] == -1).all()


# ---------------------------------------------------------------- sliding window (+ sinks)
@pytest.mark.parametrize("lens,s,w", [([100, 10, 3, 0, 5000], 4, 16), ([32768], 0, 1639),
                                      ([32768, 2000], 64, 1575), ([20, 21], 4, 16)])
def test_select_window_matches_oracle(lens, s, w):
    H, k_max = 3, s + w + 5
    idx = torch.full((len(lens), H, k_max), -7, dtype=torch.int32, device=DEV)
    ks = torch.full((len(lens),), -7, dtype=torch.int32, device=DEV)
    vg.vegas_select_window(to_dev(np.asarray(lens, np.int32)), s, w, ks, idx, len(lens), H,
                           k_max)
    vg.vegas_read_device_status()
    ref, ref_k = oracle.window_select_batch(np.asarray(lens), s, w, H, k_max)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)
    np.testing.assert_array_equal(ks.cpu().numpy(), ref_k)


def test_select_window_rejects_a_short_k_max():
    lens = to_dev(np.asarray([100], np.int32))
    idx = torch.zeros((1, 1, 10), dtype=torch.int32, device=DEV)
    ks = torch.zeros((1,), dtype=torch.int32, device=DEV)
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_select_window(lens, 4, 16, ks, idx, 1, 1, 10)
    assert ei.value.status == 1
