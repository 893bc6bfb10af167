"""fp64 CPU oracle for the Vegas hot path.  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this module.  The product path (the CUDA library and its Python
binding) never calls it and shares no code with it: the two meet only at the
seeded input generator in ``workload/``.

Source: "Vegas: Self-Speculative Decoding with Verification-Guided Sparse
Attention" (Yue, Xue, Huang), technical summary pages at gist.science
(paper 2602.07223), cited below by section:

* §2 "Core mechanism": the verify phase runs full attention over every KV entry
  and computes the attention logits; the selected critical entries form the
  sparse mask of the next draft phase; drafting attends only to them.
* §2.A "Aggregated attention-logit selection": the selected prefix set is
  T = argmax over T subset of P, |T| = k, of sum_t sum_{h in H} sum_{i in T} l^(h)_{ti},
  summing the logits over every drafted token (accepted and rejected) and the
  query heads.
* §2.B "Collect-2-Query": collect the logits of only the first drafted token and
  the bonus token, the two ends of the draft chain.
* §3 "Implementation": the logits are taken before softmax normalisation; the
  draft kernel is PagedAttention with one token per page, the selected token
  indices serving as page indices.

Readings taken where the pages are silent:

* Verify window: gamma + 1 query rows t = 0..gamma over positions L_b + t of the
  cache; row t attends positions [0, L_b + t] (causal inside the window).
  Row 0 produces the first drafted token's verification, row gamma produces the
  bonus token, so Collect-2-Query captures rows {0, gamma}.
* H in the equation is the group of G = Hq / Hkv query heads that share KV head
  g; query head h reads KV head floor(h / G).  Selection is per (sequence, KV head).
* P = [0, L_b), the committed prefix; the logits are the scaled dot products
  q . k / sqrt(d), not probabilities.
* Ties in the top-k go to the lower position; the output is sorted ascending.
* Draft step j attends T plus the dense tail [L_b, L_b + tail_len).

Every function has pins in ``tests/test_oracle_pins.py`` (closed forms,
invariants, brute force on tiny inputs); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

PAGE_SIZE = 16


# ----------------------------------------------------------------------------
# Paged-cache addressing (§3: PagedAttention; one physical page holds 16 tokens)
# ----------------------------------------------------------------------------

def gather_rows(cache: np.ndarray, block_table_row: np.ndarray, g: int,
                positions: np.ndarray) -> np.ndarray:
    """Rows of logical positions for KV head g.

    cache: [num_pages][Hkv][PAGE_SIZE][d]; logical position i lives in physical
    page block_table_row[i // PAGE_SIZE], slot i % PAGE_SIZE.
    """
    pos = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[pos // PAGE_SIZE]
    if pos.size and (pages.min() < 0 or pages.max() >= cache.shape[0]):
        raise ValueError("block table entry out of range")
    return np.asarray(cache[pages, g, pos % PAGE_SIZE, :], dtype=np.float64)


# ----------------------------------------------------------------------------
# Attention for one query row (§2: full attention in verify, sparse in draft)
# ----------------------------------------------------------------------------

def logits_row(q: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """Pre-softmax attention logits l_i = scale * (q . k_i) for the rows of K."""
    return (K @ np.asarray(q, dtype=np.float64)) * scale


def softmax(l: np.ndarray) -> np.ndarray:
    """p_i = exp(l_i - max l) / sum_j exp(l_j - max l)."""
    e = np.exp(l - np.max(l))
    return e / np.sum(e)


def attention_row(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """o = sum_i softmax(l)_i v_i over the given rows."""
    if K.shape[0] == 0:
        raise ValueError("attention over an empty set")
    return softmax(logits_row(q, K, scale)) @ V


# ----------------------------------------------------------------------------
# Verify phase: full attention over the window's gamma + 1 rows
# ----------------------------------------------------------------------------

def verify_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                     block_table: np.ndarray, ctx_lens: np.ndarray,
                     scale: float) -> np.ndarray:
    """Full verify attention.

    q: [B][gamma+1][Hq][d]; row t of sequence b attends logical positions
    [0, L_b + t].  Returns o with q's shape.
    """
    B, T, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, T, Hq, d), dtype=np.float64)
    for b in range(B):
        L = int(ctx_lens[b])
        pos = np.arange(L + T, dtype=np.int64)
        for g in range(Hkv):
            K = gather_rows(k_cache, block_table[b], g, pos)
            V = gather_rows(v_cache, block_table[b], g, pos)
            for h in range(g * G, (g + 1) * G):
                for t in range(T):
                    n = L + t + 1
                    out[b, t, h] = attention_row(q[b, t, h], K[:n], V[:n], scale)
    return out


# ----------------------------------------------------------------------------
# Logit capture (§2.A equation restricted to the rows of §2.B, logits of §3)
# ----------------------------------------------------------------------------

def capture_scores(q: np.ndarray, k_cache: np.ndarray, block_table: np.ndarray,
                   ctx_lens: np.ndarray, scale: float, rows=None) -> np.ndarray:
    """s[b][g][i] = sum_{t in rows} sum_{h in group g} l^(h)_{t,i}, for i in [0, L_b).

    rows defaults to Collect-2-Query's {0, gamma}; pass range(gamma + 1) for
    the all-rows sum of the §2.A equation.  Entries at i >= L_b are 0.
    """
    B, T, Hq, d = q.shape
    gamma = T - 1
    if rows is None:
        rows = (0, gamma) if gamma > 0 else (0,)
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    Lmax = int(np.max(ctx_lens)) if B else 0
    s = np.zeros((B, Hkv, Lmax), dtype=np.float64)
    for b in range(B):
        L = int(ctx_lens[b])
        pos = np.arange(L, dtype=np.int64)
        for g in range(Hkv):
            K = gather_rows(k_cache, block_table[b], g, pos)
            for t in rows:
                for h in range(g * G, (g + 1) * G):
                    s[b, g, :L] += logits_row(q[b, t, h], K, scale)
    return s


def raw_capture_logits(q: np.ndarray, k_cache: np.ndarray, block_table: np.ndarray,
                       ctx_lens: np.ndarray, scale: float, rows) -> np.ndarray:
    """§3 "Implementation": the raw pre-softmax logits the pages' verify kernel
    writes for the collected rows, raw[b][r][h][i] = l^(h)_{rows[r], i} for
    i in [0, L_b) (0 beyond), every query head h."""
    B, T, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    rows = list(rows)
    Lmax = int(np.max(ctx_lens)) if B else 0
    raw = np.zeros((B, len(rows), Hq, Lmax), dtype=np.float64)
    for b in range(B):
        L = int(ctx_lens[b])
        pos = np.arange(L, dtype=np.int64)
        for g in range(Hkv):
            K = gather_rows(k_cache, block_table[b], g, pos)
            for r, t in enumerate(rows):
                for h in range(g * G, (g + 1) * G):
                    raw[b, r, h, :L] = logits_row(q[b, t, h], K, scale)
    return raw


# ----------------------------------------------------------------------------
# Selection (§2.A): argmax over |T| = k of the summed logits
# ----------------------------------------------------------------------------

def select_topk(s: np.ndarray, k: int) -> np.ndarray:
    """The k positions of largest score, ties to the lower position, ascending.

    The objective of the §2.A equation is a sum of per-position terms, so the
    maximising set is the k largest per-position sums.  Implemented as a stable
    sort on -s (equal scores keep position order), first k, then sorted.
    """
    s = np.asarray(s)
    if np.isnan(s).any():
        raise ValueError("NaN score")
    k = int(k)
    if k < 0 or k > s.shape[0]:
        raise ValueError("k out of range")
    order = np.argsort(-s, kind="stable")
    return np.sort(order[:k]).astype(np.int64)


def select_topk_batch(scores: np.ndarray, ctx_lens: np.ndarray, k_per_seq: np.ndarray,
                      k_max: int) -> np.ndarray:
    """[B][Hkv][k_max] int32: select_topk over s[b][g][:L_b]; entries >= k_b are -1."""
    B, Hkv = scores.shape[0], scores.shape[1]
    out = np.full((B, Hkv, k_max), -1, dtype=np.int32)
    for b in range(B):
        L, k = int(ctx_lens[b]), int(k_per_seq[b])
        for g in range(Hkv):
            out[b, g, :k] = select_topk(scores[b, g, :L], k)
    return out


def summed_head_scores(scores: np.ndarray, L: int, b: int) -> np.ndarray:
    """s[i] = sum over the KV heads g of scores[b][g][i], i < L, in fp64.

    Each scores[b][g] already sums its group's query heads (capture_scores), so
    this is the §2.A triple sum with H = every query head of the layer."""
    return np.asarray(scores[b, :, :L], dtype=np.float64).sum(axis=0)


def select_topk_shared_batch(scores: np.ndarray, ctx_lens: np.ndarray,
                             k_per_seq: np.ndarray, k_max: int) -> np.ndarray:
    """§2.A with H = every query head of the layer: one T per sequence, the k_b
    positions of largest summed score sum_g s[b][g][i] (fp64), written to the
    rows of every KV head.  [B][Hkv][k_max] int32, -1 padded."""
    B, Hkv = scores.shape[0], scores.shape[1]
    out = np.full((B, Hkv, k_max), -1, dtype=np.int32)
    for b in range(B):
        L, k = int(ctx_lens[b]), int(k_per_seq[b])
        T = select_topk(summed_head_scores(scores, L, b), k)
        for g in range(Hkv):
            out[b, g, :k] = T
    return out


def summed_head_scores_f32(scores_f32: np.ndarray, L: int, b: int) -> np.ndarray:
    """The shared-T library call's stated key: sum over the KV heads of
    scores[b][g][i], added in fp32 in head order g = 0, 1, ...  Not the method's
    definition (that is summed_head_scores, fp64); it lets a test feed the
    library and this oracle the same fp32 keys and demand identical indices."""
    s = np.array(scores_f32[b, 0, :L], dtype=np.float32)
    for g in range(1, scores_f32.shape[1]):
        s = (s + np.asarray(scores_f32[b, g, :L], dtype=np.float32)).astype(np.float32)
    return s


def select_topk_shared_batch_f32(scores_f32: np.ndarray, ctx_lens: np.ndarray,
                                 k_per_seq: np.ndarray, k_max: int) -> np.ndarray:
    """select_topk_shared_batch on the fp32 head-order keys of
    summed_head_scores_f32 (the library call's stated key, for the bit-exact
    identical-keys comparison)."""
    B, Hkv = scores_f32.shape[0], scores_f32.shape[1]
    out = np.full((B, Hkv, k_max), -1, dtype=np.int32)
    for b in range(B):
        L, k = int(ctx_lens[b]), int(k_per_seq[b])
        T = select_topk(summed_head_scores_f32(scores_f32, L, b).astype(np.float64), k)
        for g in range(Hkv):
            out[b, g, :k] = T
    return out


def window_select(L: int, num_sink: int, window: int) -> np.ndarray:
    """§1 "Problem": the query-agnostic sliding-window selector, with optional
    sink positions at the start: every prefix position i in [0, L) with
    i < num_sink or i >= L - window, ascending."""
    return np.array([i for i in range(L) if i < num_sink or i >= L - window], dtype=np.int64)


def window_select_batch(ctx_lens: np.ndarray, num_sink: int, window: int, num_kv_heads: int,
                        k_max: int):
    """(idx [B][Hkv][k_max] int32 -1 padded, k [B]) of window_select per sequence,
    the same for every KV head."""
    B = len(ctx_lens)
    out = np.full((B, num_kv_heads, k_max), -1, dtype=np.int32)
    ks = np.zeros(B, dtype=np.int32)
    for b in range(B):
        T = window_select(int(ctx_lens[b]), num_sink, window)
        ks[b] = len(T)
        out[b, :, :len(T)] = T
    return out, ks


# ----------------------------------------------------------------------------
# Draft phase: sparse attention over T plus the dense tail (§2, §3)
# ----------------------------------------------------------------------------

def sparse_positions(idx_row: np.ndarray, k: int, tail_start: int, tail_len: int) -> np.ndarray:
    """The attended positions of one draft step: T (k entries) then the tail."""
    sel = np.asarray(idx_row[:k], dtype=np.int64)
    return np.concatenate([sel, np.arange(tail_start, tail_start + tail_len, dtype=np.int64)])


def sparse_decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                  block_table: np.ndarray, idx: np.ndarray, k_per_seq: np.ndarray,
                  tail_start: np.ndarray, tail_len: np.ndarray, scale: float) -> np.ndarray:
    """One draft step. q: [B][Hq][d]; idx: [B][Hkv][k_max]. Returns o [B][Hq][d]."""
    B, Hq, d = q.shape
    Hkv = k_cache.shape[1]
    G = Hq // Hkv
    out = np.zeros((B, Hq, d), dtype=np.float64)
    for b in range(B):
        for g in range(Hkv):
            pos = sparse_positions(idx[b, g], int(k_per_seq[b]), int(tail_start[b]),
                                   int(tail_len[b]))
            K = gather_rows(k_cache, block_table[b], g, pos)
            V = gather_rows(v_cache, block_table[b], g, pos)
            for h in range(g * G, (g + 1) * G):
                out[b, h] = attention_row(q[b, h], K, V, scale)
    return out


# ----------------------------------------------------------------------------
# One iteration of the path (§2: verify -> select -> gamma draft steps)
# ----------------------------------------------------------------------------

def iteration(q_verify: np.ndarray, q_draft: np.ndarray, k_cache: np.ndarray,
              v_cache: np.ndarray, block_table: np.ndarray, ctx_lens: np.ndarray,
              k_per_seq: np.ndarray, scale: float) -> dict:
    """verify + capture -> top-k -> gamma draft steps, under full acceptance.

    q_draft: [gamma][B][Hq][d]; draft step j attends T and the tail
    [L_b, L_b + gamma + 2 + j): the window, the bonus token and drafts 0..j-1,
    ending at its own position.
    """
    gamma = q_verify.shape[1] - 1
    o_verify = verify_attention(q_verify, k_cache, v_cache, block_table, ctx_lens, scale)
    s = capture_scores(q_verify, k_cache, block_table, ctx_lens, scale)
    k_max = int(np.max(k_per_seq))
    idx = select_topk_batch(s, ctx_lens, k_per_seq, k_max)
    o_draft = []
    for j in range(gamma):
        tl = np.full_like(ctx_lens, gamma + 2 + j)
        o_draft.append(sparse_decode(q_draft[j], k_cache, v_cache, block_table, idx,
                                     k_per_seq, ctx_lens, tl, scale))
    return {"o_verify": o_verify, "scores": s, "idx": idx, "o_draft": np.stack(o_draft)}
