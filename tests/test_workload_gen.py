"""Host-side checks of the seeded input generator (no method arithmetic here)."""
import numpy as np
import torch

from workload import configs, gen


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(1 << 16) * rng.choice([1e-3, 1, 1e3], 1 << 16)).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.00390625, 1.01171875]   # exact ties: round to even
    ours = gen.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_normals_moments_and_determinism():
    z = gen.normals(gen.stream_key(1, 2), np.arange(1 << 20)).astype(np.float64)
    assert abs(z.mean()) < 5e-3 and abs(z.var() - 1) < 1e-2
    assert np.abs(z).max() <= 2 * np.sqrt(3) + 1e-6
    z2 = gen.normals(gen.stream_key(1, 2), np.arange(1000, 2000)).astype(np.float64)
    np.testing.assert_array_equal(z[1000:2000], z2)


def test_splitmix64_reference_sequence():
    # SplitMix64 seeded with 0: published first outputs of the generator
    key = 0
    out = [int(v) for v in gen.draws(key, np.arange(3))]
    assert out[0] == 0xE220A8397B1DCDAF
    assert out[1] == 0x6E789E6AA1B965F4
    assert out[2] == 0x06C45D188009454F


def test_page_map_is_a_permutation():
    w = configs.QWEN3_8B_B8_48K_64K
    lens = gen.ctx_lens(w)
    assert lens.min() >= w.ctx_lo and lens.max() <= w.ctx_hi
    pm = gen.page_map(w, lens)
    used = np.concatenate([pm.block_table[b, :pm.pages[b]] for b in range(w.batch)])
    assert sorted(used.tolist()) == list(range(pm.num_pages))
    for b in range(w.batch):
        assert np.all(pm.block_table[b, pm.pages[b]:] == -1)
        lp = np.arange(pm.pages[b])
        np.testing.assert_array_equal(pm.owner[pm.block_table[b, lp]], b * pm.max_pages + lp)


def test_k_per_seq_rounds_up():
    w = configs.QWEN3_8B_B1_32K
    assert gen.k_per_seq(w, np.array([32768]))[0] == 1639
    w4 = configs.GPTOSS_20B_B4_128K
    assert gen.k_per_seq(w4, np.array([131072]))[0] == 3933
    assert gen.k_per_seq(configs.TINY, np.array([2048, 50]))[0] == 128
    assert gen.k_per_seq(configs.TINY, np.array([2048, 50]))[1] == 50


def test_heavy_rows_are_planted():
    w = configs.GPTOSS_20B_B4_128K.with_(ctx_lo=4096, ctx_hi=4096)
    pos = np.arange(4096)
    hv = gen.heavy_mask(w, 0, 1, 3, pos, 4096)
    assert hv[-512:].all()
    frac = hv[:-512].mean()
    assert 0.003 < frac < 0.02
    rows = gen.kv_rows_f32(w, 0, "k", 1, 3, pos, 4096)
    u = gen.unit_direction(w)
    proj = rows @ u
    assert proj[hv].mean() > 2.5 and abs(proj[~hv].mean()) < 0.2
