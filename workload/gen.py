"""Seeded synthetic inputs for the Vegas hot path (host side, numpy).

This module draws the inputs that both the GPU path and the fp64 oracle consume.
It holds none of the method's arithmetic: no attention, no logit capture, no
selection.  Everything is a pure function of (seed, tensor tag, element index),
so any slice of any tensor can be regenerated on its own, and the device-side
generator in the CUDA library implements the same definition element for element.

Generator definition (the one both sides implement):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): state advances by the golden gamma
  ``0x9E3779B97F4A7C15`` and each output is the state passed through the
  ``mix64`` finaliser below.  Used counter-style: the i-th draw of a stream is
  ``mix64(key + (i + 1) * GAMMA)`` with ``key = mix64(seed + tag * GAMMA)``.
* Normal approximation: the Irwin-Hall sum of the four 16-bit fields of one
  draw, centred and scaled to unit variance:
  ``z = float32(u0 + u1 + u2 + u3 - 131070) * float32(sqrt(3) / 65536)``.
  Every step is exact integer arithmetic or one correctly rounded fp32
  multiply, so host and device agree bit for bit.  ``z`` is bounded by
  ``+-2*sqrt(3)`` and has variance ``1 - 2**-32``.
* fp32 -> bf16 is round-to-nearest-even on the bit pattern.

Workload structure (the shapes and value distribution of the pages' decode
workloads, Qwen3 / gpt-oss-20b attention layers at 32K-128K context):

* K, V, Q ~ N(0, 1) per coordinate.
* A seeded unit direction ``u`` (normalised draw of ``d`` normals).
* "Heavy hitter" prefix positions, chosen per (sequence, KV head, position) by
  a Bernoulli draw, get keys ``3*u + 0.3*z``; some workloads also key the last
  ``heavy_last`` prefix positions this way.
* Queries get ``z + 3*u``.
* Block tables map logical pages to a seeded permutation of the physical pool
  (Fisher-Yates driven by the same stream), or to the identity.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
MIX_M1 = 0xBF58476D1CE4E5B9
MIX_M2 = 0x94D049BB133111EB

# Stream tags; a layer adds LAYER_STRIDE * layer.
TAG_K = 1
TAG_V = 2
TAG_QV = 3      # verify-window queries
TAG_QD = 4      # draft-step queries
TAG_HEAVY = 5
TAG_U = 6
TAG_PERM = 7
TAG_LEN = 8
LAYER_STRIDE = 16

PAGE_SIZE = 16
UNIT_SHIFT = 24  # position field width inside a K/V element counter

# float32(sqrt(3) / 65536), the Irwin-Hall scale; bit pattern shared with CUDA.
IH_SCALE = np.float32(math.sqrt(3.0) / 65536.0)
IH_SCALE_BITS = int(np.array([IH_SCALE], dtype=np.float32).view(np.uint32)[0])
F32_THREE = np.float32(3.0)
F32_POINT3 = np.float32(0.3)


def mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * MIX_M1) & MASK64
    z = ((z ^ (z >> 27)) * MIX_M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tag: int) -> int:
    return mix64_int((seed + tag * GAMMA) & MASK64)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(MIX_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(MIX_M2)
    return z ^ (z >> np.uint64(31))


def draws(key: int, idx) -> np.ndarray:
    """uint64 draws ``mix64(key + (idx + 1) * GAMMA)`` for an array of counters."""
    i = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + (i + np.uint64(1)) * np.uint64(GAMMA))


def normals(key: int, idx) -> np.ndarray:
    """float32 Irwin-Hall(4) normal approximations for an array of counters."""
    r = draws(key, idx)
    m = np.uint64(0xFFFF)
    s = ((r & m) + ((r >> np.uint64(16)) & m) + ((r >> np.uint64(32)) & m)
         + (r >> np.uint64(48))).astype(np.int64) - 131070
    return s.astype(np.float32) * IH_SCALE


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    return ((b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


@dataclass(frozen=True)
class Workload:
    """One synthetic decode workload: the attention-layer shape and value structure."""
    name: str
    layers: int
    batch: int
    hq: int
    hkv: int
    head_dim: int
    gamma: int
    ctx_lo: int
    ctx_hi: int
    heavy_pct: float          # share of prefix positions that are heavy hitters (percent)
    seed: int
    k_abs: int | None = None  # selected count, absolute
    k_pct: int | None = None  # selected count, percent of the prefix (rounded up)
    heavy_last: int = 0       # the last heavy_last prefix positions are also heavy
    shuffled: bool = True     # block table: seeded permutation of the page pool
    fp32_source: bool = False  # specified in fp32 (rounded to bf16 for the kernels)
    description: str = ""

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def rows(self) -> int:
        """Verify-window query rows per (sequence, KV head): (gamma + 1) * G."""
        return (self.gamma + 1) * self.group

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def ctx_lens(w: Workload) -> np.ndarray:
    """Committed prefix length L_b per sequence: fixed, or uniform in [lo, hi]."""
    if w.ctx_lo == w.ctx_hi:
        return np.full(w.batch, w.ctx_lo, dtype=np.int32)
    span = w.ctx_hi - w.ctx_lo + 1
    r = draws(stream_key(w.seed, TAG_LEN), np.arange(w.batch))
    return (w.ctx_lo + (r % np.uint64(span)).astype(np.int64)).astype(np.int32)


def k_per_seq(w: Workload, lens: np.ndarray) -> np.ndarray:
    """k_b = min(L_b, k_abs) or min(L_b, ceil(k_pct * L_b / 100))."""
    lens = np.asarray(lens, dtype=np.int64)
    if w.k_abs is not None:
        k = np.minimum(lens, w.k_abs)
    else:
        k = np.minimum(lens, (w.k_pct * lens + 99) // 100)
    return k.astype(np.int32)


def positions_needed(w: Workload, lens: np.ndarray) -> np.ndarray:
    """Cache positions one iteration touches: prefix, gamma+1 window, bonus, gamma-1 drafts."""
    return (np.asarray(lens, dtype=np.int64) + 2 * w.gamma + 1).astype(np.int64)


def tail_len(w: Workload, step: int) -> int:
    """Dense tail attended by draft step j: window (gamma+1), bonus, drafts 0..j-1."""
    return w.gamma + 2 + step


@dataclass
class PageMap:
    block_table: np.ndarray   # int32 [B][max_pages]; -1 past a sequence's pages
    num_pages: int
    owner: np.ndarray         # int32 [num_pages]: b * max_pages + logical page, -1 if unused
    max_pages: int
    pages: np.ndarray = field(default=None)  # int64 [B] pages per sequence


def page_map(w: Workload, lens: np.ndarray) -> PageMap:
    need = positions_needed(w, lens)
    pages = (need + PAGE_SIZE - 1) // PAGE_SIZE
    max_pages = int(pages.max())
    total = int(pages.sum())
    perm = np.arange(total, dtype=np.int64)
    if w.shuffled and total > 1:
        key = stream_key(w.seed, TAG_PERM)
        r = draws(key, np.arange(total))
        for i in range(total - 1, 0, -1):      # Fisher-Yates, high to low
            j = int(r[i] % np.uint64(i + 1))
            perm[i], perm[j] = perm[j], perm[i]
    bt = np.full((w.batch, max_pages), -1, dtype=np.int32)
    owner = np.full(total, -1, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        n = int(pages[b])
        phys = perm[off:off + n]
        bt[b, :n] = phys
        owner[phys] = b * max_pages + np.arange(n)
        off += n
    return PageMap(bt, total, owner, max_pages, pages)


def unit_direction(w: Workload) -> np.ndarray:
    z = normals(stream_key(w.seed, TAG_U), np.arange(w.head_dim)).astype(np.float64)
    return (z / np.sqrt(np.sum(z * z))).astype(np.float32)


def heavy_mask(w: Workload, layer: int, b: int, g: int, positions: np.ndarray,
               L_b: int) -> np.ndarray:
    pos = np.asarray(positions, dtype=np.int64)
    unit = b * w.hkv + g
    ctr = (np.uint64(unit) << np.uint64(UNIT_SHIFT)) + pos.astype(np.uint64)
    thresh = np.uint64(heavy_threshold(w))
    h = draws(stream_key(w.seed, TAG_HEAVY + LAYER_STRIDE * layer), ctr) < thresh
    if w.heavy_last:
        h |= (pos >= L_b - w.heavy_last) & (pos < L_b)
    return h & (pos < L_b)


def heavy_threshold(w: Workload) -> int:
    """A position is heavy when its uint64 draw is below this value."""
    return int(w.heavy_pct / 100.0 * 2.0 ** 64) & MASK64


def kv_rows_f32(w: Workload, layer: int, which: str, b: int, g: int,
                positions: np.ndarray, L_b: int) -> np.ndarray:
    """float32 K or V rows [n, d] of logical positions of sequence b, KV head g."""
    pos = np.asarray(positions, dtype=np.int64)
    d = w.head_dim
    tag = (TAG_K if which == "k" else TAG_V) + LAYER_STRIDE * layer
    unit = b * w.hkv + g
    base = ((np.uint64(unit) << np.uint64(UNIT_SHIFT)) + pos.astype(np.uint64)) * np.uint64(d)
    ctr = base[:, None] + np.arange(d, dtype=np.uint64)[None, :]
    z = normals(stream_key(w.seed, tag), ctr)
    if which == "k":
        hv = heavy_mask(w, layer, b, g, pos, L_b)
        if hv.any():
            u = unit_direction(w)
            planted = (F32_THREE * u)[None, :] + F32_POINT3 * z[hv]
            z[hv] = planted.astype(np.float32)
    return z


def kv_rows_bf16(w: Workload, layer: int, which: str, b: int, g: int,
                 positions: np.ndarray, L_b: int) -> np.ndarray:
    return f32_to_bf16_bits(kv_rows_f32(w, layer, which, b, g, positions, L_b))


def paged_cache_bf16(w: Workload, layer: int, which: str, lens: np.ndarray,
                     pm: PageMap) -> np.ndarray:
    """Whole paged cache [num_pages][Hkv][16][d] as bf16 bits; unused slots are 0."""
    d = w.head_dim
    out = np.zeros((pm.num_pages, w.hkv, PAGE_SIZE, d), dtype=np.uint16)
    need = positions_needed(w, lens)
    for b in range(w.batch):
        n = int(need[b])
        pos = np.arange(n, dtype=np.int64)
        phys = pm.block_table[b, pos // PAGE_SIZE]
        slot = pos % PAGE_SIZE
        for g in range(w.hkv):
            out[phys, g, slot, :] = kv_rows_bf16(w, layer, which, b, g, pos, int(lens[b]))
    return out


def verify_queries_f32(w: Workload, layer: int = 0) -> np.ndarray:
    """Verify-window queries [B][gamma+1][Hq][d]: z + 3u."""
    shape = (w.batch, w.gamma + 1, w.hq, w.head_dim)
    z = normals(stream_key(w.seed, TAG_QV + LAYER_STRIDE * layer),
                np.arange(int(np.prod(shape)))).reshape(shape)
    return (z + F32_THREE * unit_direction(w)).astype(np.float32)


def draft_queries_f32(w: Workload, layer: int = 0) -> np.ndarray:
    """Draft-step queries [gamma][B][Hq][d]: z + 3u, a fresh draw per step."""
    shape = (w.gamma, w.batch, w.hq, w.head_dim)
    z = normals(stream_key(w.seed, TAG_QD + LAYER_STRIDE * layer),
                np.arange(int(np.prod(shape)))).reshape(shape)
    return (z + F32_THREE * unit_direction(w)).astype(np.float32)
