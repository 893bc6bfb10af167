"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

No test here re-types an oracle formula: each checks a closed form, an
invariant, a brute-force search over subsets, a library routine on a special
case, or a hand-worked example under tests/golden/.  Source pages: "Vegas:
Self-Speculative Decoding with Verification-Guided Sparse Attention",
gist.science technical summary (paper 2602.07223).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _paged(rows_by_head, shuffle_seed=None, extra_pages=0):
    """Build a paged cache [pages][Hkv][16][d] holding logical rows [Hkv][n][d]."""
    Hkv, n, d = rows_by_head.shape
    npages = (n + 15) // 16
    phys = np.arange(npages + extra_pages)
    if shuffle_seed is not None:
        phys = np.random.default_rng(shuffle_seed).permutation(npages + extra_pages)
    bt = phys[:npages].astype(np.int32)
    cache = np.full((npages + extra_pages, Hkv, 16, d), np.nan)
    for i in range(n):
        cache[bt[i // 16], :, i % 16, :] = rows_by_head[:, i, :]
    return cache, bt


def _rand_case(rng, B=2, Hq=4, Hkv=2, d=8, gamma=3, lens=(21, 37)):
    T = gamma + 1
    n_max = max(lens) + 2 * gamma + 1
    K = rng.standard_normal((B, Hkv, n_max, d))
    V = rng.standard_normal((B, Hkv, n_max, d))
    q = rng.standard_normal((B, T, Hq, d))
    caches_k, caches_v, bts = [], [], []
    for b in range(B):
        ck, bt = _paged(K[b], shuffle_seed=b)
        cv, _ = _paged(V[b], shuffle_seed=b)
        caches_k.append(ck)
        caches_v.append(cv)
        bts.append(bt)
    # one shared physical pool: concatenate per-sequence pools
    off = 0
    bt_all = np.zeros((B, max(len(x) for x in bts)), dtype=np.int32)
    for b in range(B):
        bt_all[b, :len(bts[b])] = bts[b] + off
        off += caches_k[b].shape[0]
    kc = np.concatenate(caches_k)
    vc = np.concatenate(caches_v)
    return q, K, V, kc, vc, bt_all, np.array(lens, dtype=np.int32)


# ---------------------------------------------------------------------------
# Selection: §2.A argmax over |T| = k
# ---------------------------------------------------------------------------

def _brute_force_best(s, k):
    """The lexicographically smallest ascending subset among those of maximal sum."""
    best, best_set = None, None
    for T in itertools.combinations(range(len(s)), k):
        tot = sum(s[i] for i in T)
        if best is None or tot > best:
            best, best_set = tot, T
    return list(best_set) if best_set is not None else []


@pytest.mark.parametrize("seed", range(40))
def test_topk_equals_brute_force_subset_search(seed):
    rng = np.random.default_rng(seed)
    L = int(rng.integers(1, 11))
    # small integers: many exact ties, sums exact in fp64
    s = rng.integers(-3, 4, size=L).astype(np.float64)
    for k in range(0, min(L, 6) + 1):
        assert list(oracle.select_topk(s, k)) == _brute_force_best(list(s), k)


def test_equation_triple_sum_brute_force():
    """§2.A: argmax over T of sum_t sum_h sum_{i in T} l, brute-forced over subsets,
    equals select(capture(all rows)); the logits come from explicit dot products."""
    rng = np.random.default_rng(7)
    gamma, Hq, Hkv, d, L = 2, 4, 2, 4, 9
    T = gamma + 1
    q = rng.integers(-2, 3, size=(1, T, Hq, d)).astype(np.float64)
    K = rng.integers(-2, 3, size=(Hkv, L + T, d)).astype(np.float64)
    kc, bt = _paged(K)
    scale = 0.5  # 1/sqrt(4)
    s = oracle.capture_scores(q, kc, bt[None], np.array([L]), scale, rows=range(T))
    G = Hq // Hkv
    for g in range(Hkv):
        def objective(Tset):
            tot = 0.0
            for t in range(T):
                for h in range(g * G, (g + 1) * G):
                    for i in Tset:
                        tot += scale * sum(q[0, t, h, j] * K[g, i, j] for j in range(d))
            return tot
        for k in (1, 3, 4):
            best = max(objective(c) for c in itertools.combinations(range(L), k))
            chosen = oracle.select_topk(s[0, g, :L], k)
            assert math.isclose(objective(chosen), best, rel_tol=0, abs_tol=1e-9)


def test_topk_special_cases():
    L = 12
    eq = np.ones(L)
    assert list(oracle.select_topk(eq, 5)) == [0, 1, 2, 3, 4]
    dec = -np.arange(L, dtype=np.float64)
    assert list(oracle.select_topk(dec, 4)) == [0, 1, 2, 3]
    inc = np.arange(L, dtype=np.float64)
    assert list(oracle.select_topk(inc, 4)) == [8, 9, 10, 11]
    assert list(oracle.select_topk(inc, L)) == list(range(L))
    assert list(oracle.select_topk(inc, 0)) == []
    z = np.array([-0.0, 0.0, -0.0, -1.0])
    assert list(oracle.select_topk(z, 2)) == [0, 1]
    with pytest.raises(ValueError):
        oracle.select_topk(np.array([1.0, np.nan]), 1)


def test_golden_topk_ties():
    gd = _golden("topk_ties.json")
    for case in gd["cases"]:
        assert list(oracle.select_topk(np.array(gd["scores"]), case["k"])) == case["T"]


def test_select_batch_pads_with_minus_one():
    s = np.array([[[3.0, 1.0, 2.0, 0.0]]])
    out = oracle.select_topk_batch(s, np.array([4]), np.array([2]), 3)
    assert out.tolist() == [[[0, 2, -1]]]


# ---------------------------------------------------------------------------
# Attention: closed forms and invariants (§2 full / sparse attention)
# ---------------------------------------------------------------------------

def test_golden_two_position_attention():
    gd = _golden("two_position_attention.json")
    scale = 1.0 / math.sqrt(gd["d"])
    K, V, q = np.array(gd["K"], float), np.array(gd["V"], float), np.array(gd["q"], float)
    np.testing.assert_allclose(oracle.logits_row(q, K, scale), gd["logits"], atol=1e-15)
    np.testing.assert_allclose(oracle.attention_row(q, K, V, scale), gd["o"], atol=1e-15)


def test_softmax_against_library_and_row_sums():
    from scipy.special import softmax as sp_softmax
    rng = np.random.default_rng(3)
    for n in (1, 2, 17, 1000):
        l = rng.standard_normal(n) * 7
        p = oracle.softmax(l)
        np.testing.assert_allclose(p, sp_softmax(l), rtol=1e-13, atol=1e-300)
        assert abs(p.sum() - 1.0) < 1e-12


def test_attention_closed_forms():
    rng = np.random.default_rng(4)
    d, n = 8, 13
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    # q = 0: uniform weights -> mean of V
    np.testing.assert_allclose(oracle.attention_row(np.zeros(d), K, V, 0.35), V.mean(0),
                               atol=1e-14)
    # one position: o = v0
    np.testing.assert_allclose(oracle.attention_row(rng.standard_normal(d), K[:1], V[:1], 0.35),
                               V[0], atol=1e-15)
    # V = 1: o = 1
    np.testing.assert_allclose(oracle.attention_row(rng.standard_normal(d), K, np.ones((n, d)),
                                                    0.35), np.ones(d), atol=1e-14)
    # large scale: weights collapse on the arg max of q.k (hard max)
    q = rng.standard_normal(d)
    i = int(np.argmax(K @ q))
    np.testing.assert_allclose(oracle.attention_row(q, K, V, 1e6), V[i], atol=1e-12)
    # two positions with logits a*b*scale and 0: a sigmoid
    a, b, sc = 1.5, 2.0, 1 / math.sqrt(d)
    q2 = np.zeros(d); q2[0] = a
    K2 = np.zeros((2, d)); K2[0, 0] = b
    V2 = rng.standard_normal((2, d))
    p0 = 1.0 / (1.0 + math.exp(-a * b * sc))
    np.testing.assert_allclose(oracle.attention_row(q2, K2, V2, sc), p0 * V2[0] + (1 - p0) * V2[1],
                               atol=1e-15)
    with pytest.raises(ValueError):
        oracle.attention_row(q, K[:0], V[:0], 1.0)


def test_verify_causality_within_window():
    rng = np.random.default_rng(5)
    q, K, V, kc, vc, bt, lens = _rand_case(rng)
    scale = 1 / math.sqrt(K.shape[-1])
    base = oracle.verify_attention(q, kc, vc, bt, lens, scale)
    gamma = q.shape[1] - 1
    for b in range(q.shape[0]):
        for t in range(gamma + 1):
            pos_after = int(lens[b]) + t + 1      # first position row t must not see
            kc2, vc2 = kc.copy(), vc.copy()
            for p in range(pos_after, int(lens[b]) + 2 * gamma + 1):
                kc2[bt[b, p // 16], :, p % 16] += 5.0
                vc2[bt[b, p // 16], :, p % 16] -= 5.0
            o2 = oracle.verify_attention(q, kc2, vc2, bt, lens, scale)
            np.testing.assert_array_equal(o2[b, t], base[b, t])
            # the row's own position is visible: perturbing it changes the row
            p = pos_after - 1
            vc3 = vc.copy()
            vc3[bt[b, p // 16], :, p % 16] += 1.0
            o3 = oracle.verify_attention(q, kc, vc3, bt, lens, scale)
            assert np.abs(o3[b, t] - base[b, t]).max() > 1e-6


def test_verify_page_placement_invariance():
    rng = np.random.default_rng(6)
    q, K, V, kc, vc, bt, lens = _rand_case(rng)
    scale = 1 / math.sqrt(K.shape[-1])
    o = oracle.verify_attention(q, kc, vc, bt, lens, scale)
    # same logical rows in identity-ordered pages
    off = 0
    kcs, vcs, bti = [], [], np.zeros_like(bt)
    for b in range(q.shape[0]):
        ck, btb = _paged(K[b])
        cv, _ = _paged(V[b])
        bti[b, :len(btb)] = btb + off
        off += ck.shape[0]
        kcs.append(ck); vcs.append(cv)
    o2 = oracle.verify_attention(q, np.concatenate(kcs), np.concatenate(vcs), bti, lens, scale)
    np.testing.assert_allclose(o2, o, atol=1e-13)


def test_verify_gqa_head_mapping():
    """V of KV head g is the constant g: query head h must return floor(h / G)."""
    rng = np.random.default_rng(8)
    q, K, V, kc, vc, bt, lens = _rand_case(rng, Hq=6, Hkv=3)
    vc = np.zeros_like(vc)
    for g in range(3):
        vc[:, g] = g
    o = oracle.verify_attention(q, kc, vc, bt, lens, 0.3)
    for h in range(6):
        np.testing.assert_allclose(o[:, :, h, :], h // 2, atol=1e-13)


# ---------------------------------------------------------------------------
# Capture: §2.A sum over rows and heads, §2.B rows {0, gamma}, §3 pre-softmax
# ---------------------------------------------------------------------------

def test_golden_collect2_scores():
    gd = _golden("collect2_scores.json")
    q = np.array(gd["q"], float)[None]
    keys = np.array(gd["keys"], float)[None]          # [Hkv=1][n][d]
    kc, bt = _paged(keys)
    L = gd["ctx_len"]
    s = oracle.capture_scores(q, kc, bt[None], np.array([L]), 1.0 / math.sqrt(gd["d"]))
    np.testing.assert_allclose(s[0, 0], gd["scores"], atol=1e-15)
    assert list(oracle.select_topk(s[0, 0], gd["k"])) == gd["T"]


def test_capture_rows_heads_linearity():
    rng = np.random.default_rng(9)
    q, K, V, kc, vc, bt, lens = _rand_case(rng, gamma=4)
    sc = 0.25
    s = oracle.capture_scores(q, kc, bt, lens, sc)
    # pre-softmax logits are linear in q (probabilities would not be)
    np.testing.assert_allclose(oracle.capture_scores(2 * q, kc, bt, lens, sc), 2 * s, atol=1e-12)
    # middle rows 1..gamma-1 do not enter
    q2 = q.copy(); q2[:, 1:-1] += 3.0
    np.testing.assert_array_equal(oracle.capture_scores(q2, kc, bt, lens, sc), s)
    # rows 0 and gamma do
    for t in (0, q.shape[1] - 1):
        q3 = q.copy(); q3[:, t] += 1.0
        assert np.abs(oracle.capture_scores(q3, kc, bt, lens, sc) - s).max() > 1e-6
    # another group's heads do not enter group 0's scores
    q4 = q.copy(); q4[:, :, 2:] *= -7.0
    np.testing.assert_array_equal(oracle.capture_scores(q4, kc, bt, lens, sc)[:, 0], s[:, 0])
    # window keys (positions >= L_b) do not enter; entries past L_b are zero
    kc5 = kc.copy()
    for b in range(q.shape[0]):
        for p in range(int(lens[b]), int(lens[b]) + 9):
            kc5[bt[b, p // 16], :, p % 16] += 11.0
    np.testing.assert_array_equal(oracle.capture_scores(q, kc5, bt, lens, sc), s)
    assert np.all(s[0, :, int(lens[0]):] == 0.0)


def test_capture_one_hot_closed_form():
    """q = e_j on row 0 of one head, zero elsewhere; k_i = i e_j -> s_i = i * scale."""
    d, L, gamma = 8, 30, 3
    q = np.zeros((1, gamma + 1, 4, d))
    q[0, 0, 1, 5] = 1.0                    # head 1 -> KV head 0 (G = 2)
    K = np.zeros((2, L + gamma + 1, d))
    K[:, :, 5] = np.arange(L + gamma + 1)[None, :]
    kc, bt = _paged(K)
    s = oracle.capture_scores(q, kc, bt[None], np.array([L]), 0.125)
    np.testing.assert_allclose(s[0, 0], 0.125 * np.arange(L), atol=1e-15)
    np.testing.assert_array_equal(s[0, 1], 0.0)


# ---------------------------------------------------------------------------
# Draft phase: sparse attention over T plus the tail
# ---------------------------------------------------------------------------

def test_sparse_with_full_prefix_equals_verify_row():
    """k = L_b with tail [L_b, L_b + t + 1) reduces to verify row t."""
    rng = np.random.default_rng(10)
    q, K, V, kc, vc, bt, lens = _rand_case(rng)
    sc = 1 / math.sqrt(8)
    o = oracle.verify_attention(q, kc, vc, bt, lens, sc)
    B = q.shape[0]
    kmax = int(lens.max())
    idx = np.full((B, 2, kmax), -1, dtype=np.int32)
    for b in range(B):
        idx[b, :, :lens[b]] = np.arange(lens[b])
    for t in range(q.shape[1]):
        od = oracle.sparse_decode(q[:, t], kc, vc, bt, idx, lens, lens,
                                  np.full(B, t + 1), sc)
        np.testing.assert_allclose(od, o[:, t], atol=1e-13)


def test_sparse_closed_forms():
    rng = np.random.default_rng(11)
    q, K, V, kc, vc, bt, lens = _rand_case(rng)
    B = q.shape[0]
    idx = np.zeros((B, 2, 4), dtype=np.int32)
    idx[:, :, :] = [2, 5, 7, 11]
    # every attended V row equal to c -> output c
    vc2 = np.zeros_like(vc) + 0.75
    o = oracle.sparse_decode(q[:, 0], kc, vc2, bt, idx, np.full(B, 4), lens, np.full(B, 3), 0.3)
    np.testing.assert_allclose(o, 0.75, atol=1e-14)
    # q = 0 -> mean of the attended V rows (T then tail)
    o = oracle.sparse_decode(np.zeros_like(q[:, 0]), kc, vc, bt, idx, np.full(B, 4), lens,
                             np.full(B, 2), 0.3)
    for b in range(B):
        pos = [2, 5, 7, 11, int(lens[b]), int(lens[b]) + 1]
        for h in range(4):
            np.testing.assert_allclose(o[b, h], V[b, h // 2, pos].mean(0), atol=1e-14)
    # k = 0: tail only
    o0 = oracle.sparse_decode(q[:, 0], kc, vc, bt, idx, np.zeros(B, int), lens, np.full(B, 1), 0.3)
    for b in range(B):
        np.testing.assert_allclose(o0[b], V[b, np.arange(4) // 2, int(lens[b])], atol=1e-14)


def test_sparse_does_not_depend_on_the_order_of_the_selected_positions():
    """T is a set (the §2.A argmax is over subsets): any order of its indices
    gives the same draft output."""
    rng = np.random.default_rng(12)
    q, K, V, kc, vc, bt, lens = _rand_case(rng)
    B = q.shape[0]
    k = 9
    idx = np.zeros((B, 2, k + 2), dtype=np.int32)
    for b in range(B):
        for g in range(2):
            idx[b, g, :k] = np.sort(rng.choice(int(lens[b]), size=k, replace=False))
    o = oracle.sparse_decode(q[:, 1], kc, vc, bt, idx, np.full(B, k), lens, np.full(B, 4), 0.4)
    perm = idx.copy()
    for b in range(B):
        for g in range(2):
            perm[b, g, :k] = rng.permutation(perm[b, g, :k])
    assert not np.array_equal(perm, idx)
    o2 = oracle.sparse_decode(q[:, 1], kc, vc, bt, perm, np.full(B, k), lens, np.full(B, 4), 0.4)
    np.testing.assert_allclose(o2, o, atol=1e-13)


def test_attention_is_affine_in_v():
    """Softmax weights are non-negative and sum to one, so replacing V by
    a * V + c maps every output o to a * o + c (verify rows and draft rows)."""
    rng = np.random.default_rng(13)
    q, K, V, kc, vc, bt, lens = _rand_case(rng)
    sc = 1 / math.sqrt(8)
    a, c = -1.75, 0.625
    o = oracle.verify_attention(q, kc, vc, bt, lens, sc)
    o2 = oracle.verify_attention(q, kc, a * vc + c, bt, lens, sc)
    np.testing.assert_allclose(o2, a * o + c, atol=1e-12)
    B = q.shape[0]
    idx = np.tile(np.arange(6, dtype=np.int32) * 3, (B, 2, 1))
    d1 = oracle.sparse_decode(q[:, 0], kc, vc, bt, idx, np.full(B, 6), lens, np.full(B, 2), sc)
    d2 = oracle.sparse_decode(q[:, 0], kc, a * vc + c, bt, idx, np.full(B, 6), lens,
                              np.full(B, 2), sc)
    np.testing.assert_allclose(d2, a * d1 + c, atol=1e-12)


def test_iteration_dense_selection_reduces_to_dense_draft():
    """r = 100%: every draft step equals dense attention over [0, L_b + gamma + 2 + j)."""
    rng = np.random.default_rng(12)
    q, K, V, kc, vc, bt, lens = _rand_case(rng, gamma=3)
    B, gamma = q.shape[0], q.shape[1] - 1
    qd = rng.standard_normal((gamma, B, 4, 8))
    sc = 1 / math.sqrt(8)
    res = oracle.iteration(q, qd, kc, vc, bt, lens, lens.copy(), sc)
    for j in range(gamma):
        for b in range(B):
            n = int(lens[b]) + gamma + 2 + j
            for h in range(4):
                ref = oracle.attention_row(qd[j, b, h], K[b, h // 2, :n], V[b, h // 2, :n], sc)
                np.testing.assert_allclose(res["o_draft"][j, b, h], ref, atol=1e-13)


# ---------------------------------------------------------------------------
# One T shared by every query head (§2.A with H = all heads of the layer)
# ---------------------------------------------------------------------------

def test_shared_selection_is_the_all_heads_triple_sum_argmax():
    """Brute force over subsets of the objective sum over ALL query heads (and the
    captured rows) of the explicit dot products equals the shared selection of the
    per-KV-head captured scores."""
    rng = np.random.default_rng(11)
    gamma, Hq, Hkv, d, L = 1, 4, 2, 4, 8
    T = gamma + 1
    q = rng.integers(-2, 3, size=(1, T, Hq, d)).astype(np.float64)
    K = rng.integers(-2, 3, size=(Hkv, L + T, d)).astype(np.float64)
    kc, bt = _paged(K)
    scale = 0.5
    s = oracle.capture_scores(q, kc, bt[None], np.array([L]), scale, rows=range(T))
    G = Hq // Hkv

    def objective(Tset):
        return sum(scale * sum(q[0, t, h, j] * K[h // G, i, j] for j in range(d))
                   for t in range(T) for h in range(Hq) for i in Tset)
    for k in (1, 2, 5):
        best = max(objective(c) for c in itertools.combinations(range(L), k))
        idx = oracle.select_topk_shared_batch(s.astype(np.float32), np.array([L]),
                                              np.array([k]), k)
        assert math.isclose(objective(list(idx[0, 0, :k])), best, rel_tol=0, abs_tol=1e-9)
        assert (idx[0] == idx[0, 0]).all()          # the same T for every KV head


@pytest.mark.parametrize("seed", range(10))
def test_shared_selection_ties_match_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    L = int(rng.integers(1, 10))
    s = rng.integers(-2, 3, size=(1, 3, L)).astype(np.float32)      # exact sums, many ties
    for k in range(0, min(L, 5) + 1):
        idx = oracle.select_topk_shared_batch(s, np.array([L]), np.array([k]), 6)
        assert list(idx[0, 0, :k]) == _brute_force_best(list(s[0].sum(axis=0)), k)
        assert (idx[0, :, k:] == -1).all()


def test_shared_selection_sums_the_heads_exactly_not_in_fp32():
    """The shared objective is the exact sum over heads: where an fp32 head-order
    sum loses a term (1e8 + 1 - 1e8 = 0 in fp32), the selection still follows the
    exact sum, brute-forced here in integers; the fp32 head-order variant (the
    library call's stated key) picks the other position."""
    s = np.array([[[1e8, 0.5, 0.0], [1.0, 0.0, 0.0], [-1e8, 0.0, 0.25]]], dtype=np.float32)
    exact = [sum(int(round(4 * float(s[0, g, i]))) for g in range(3)) for i in range(3)]
    assert exact == [4, 2, 1]
    for k in (1, 2):
        idx = oracle.select_topk_shared_batch(s, np.array([3]), np.array([k]), 3)
        assert list(idx[0, 0, :k]) == _brute_force_best(exact, k)
    f32 = oracle.select_topk_shared_batch_f32(s, np.array([3]), np.array([1]), 1)
    assert list(f32[0, 0]) == [1]          # fp32: 1e8 + 1 - 1e8 -> 0 < 0.5
    assert oracle.summed_head_scores(s, 3, 0)[0] == 1.0


@pytest.mark.parametrize("seed", range(4))
def test_shared_selection_f32_key_equals_the_exact_one_on_representable_sums(seed):
    rng = np.random.default_rng(300 + seed)
    s = (rng.integers(-512, 513, size=(2, 8, 700)) * 0.125).astype(np.float32)
    lens, ks = np.array([700, 333]), np.array([35, 17])
    np.testing.assert_array_equal(oracle.select_topk_shared_batch_f32(s, lens, ks, 40),
                                  oracle.select_topk_shared_batch(s, lens, ks, 40))


def test_shared_selection_with_one_kv_head_is_the_per_head_selection():
    rng = np.random.default_rng(12)
    s = rng.standard_normal((3, 1, 40)).astype(np.float32)
    lens, ks = np.array([40, 17, 5]), np.array([7, 17, 0])
    np.testing.assert_array_equal(oracle.select_topk_shared_batch(s, lens, ks, 20),
                                  oracle.select_topk_batch(s.astype(np.float64), lens, ks, 20))


# ---------------------------------------------------------------------------
# Query-agnostic sliding-window selector (§1 "Problem")
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L,s,w", [(100, 4, 16), (10, 4, 16), (3, 4, 16), (0, 4, 16),
                                   (100, 0, 16), (100, 4, 0), (20, 4, 16), (21, 4, 16)])
def test_window_selection_closed_forms(L, s, w):
    T = oracle.window_select(L, s, w)
    assert len(T) == min(L, s + w)
    assert list(T) == sorted(set(T.tolist()))               # ascending, no repeats
    if L <= s + w:
        assert list(T) == list(range(L))                    # everything fits
    else:
        assert list(T) == list(range(s)) + list(range(L - w, L))


def test_window_selection_over_the_whole_prefix_is_dense_drafting():
    """A window covering the prefix makes the draft step the dense decode row."""
    rng = np.random.default_rng(13)
    q, K, V, kc, vc, bt, lens = _rand_case(rng, B=1, lens=(30,))
    idx, ks = oracle.window_select_batch(lens, 0, 30, kc.shape[1], 32)
    tail = np.array([3])
    qd = rng.standard_normal((1, q.shape[2], q.shape[3]))
    o_sparse = oracle.sparse_decode(qd, kc, vc, bt, idx, ks, lens, tail, 0.3)
    full = np.arange(30)[None, None, :].repeat(kc.shape[1], axis=1).astype(np.int32)
    o_full = oracle.sparse_decode(qd, kc, vc, bt, full, np.array([30]), lens, tail, 0.3)
    np.testing.assert_allclose(o_sparse, o_full, rtol=0, atol=1e-14)


def test_raw_logits_sum_to_the_capture_and_match_dot_products():
    """§3's raw logits: explicit dot products entry by entry, and their sum over the
    rows and the group's heads is the (brute-force-pinned) capture."""
    rng = np.random.default_rng(14)
    q, K, V, kc, vc, bt, lens = _rand_case(rng, B=2, lens=(21, 37))
    rows = (0, 3)
    raw = oracle.raw_capture_logits(q, kc, bt, lens, 0.25, rows)
    G = q.shape[2] // kc.shape[1]
    for b in range(2):
        L = int(lens[b])
        for r, t in enumerate(rows):
            for h in range(q.shape[2]):
                want = [0.25 * float(np.dot(q[b, t, h], K[b, h // G, i])) for i in range(L)]
                np.testing.assert_allclose(raw[b, r, h, :L], want, rtol=0, atol=1e-12)
    s = oracle.capture_scores(q, kc, bt, lens, 0.25, rows=rows)
    agg = raw.reshape(2, len(rows), kc.shape[1], G, -1).sum(axis=(1, 3))
    np.testing.assert_allclose(agg, s, rtol=0, atol=1e-12)
