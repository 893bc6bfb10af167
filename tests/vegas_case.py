"""Test helpers: build a seeded Vegas workload on the GPU and its fp64 oracle view.

The GPU side receives bf16 caches (drawn on the host, or by the device
generator for large shapes) and calls the kernels through the C-ABI binding.
The oracle side regenerates the same bf16 values on the host from the
counter-based generator and widens them to fp64.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import self_speculative_sparse_paged_gb300 as vg
from workload import gen

DEV = torch.device("cuda:0")


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


class Case:
    """One workload (one layer) resident on the GPU."""

    def __init__(self, w: gen.Workload, layer: int = 0, device_gen: bool = False,
                 lens: np.ndarray | None = None):
        self.w = w
        self.layer = layer
        self.lens = gen.ctx_lens(w) if lens is None else np.asarray(lens, dtype=np.int32)
        self.kps = gen.k_per_seq(w, self.lens)
        self.pm = gen.page_map(w, self.lens)
        self.scale = 1.0 / math.sqrt(w.head_dim)
        self.device_gen = device_gen
        shape = (self.pm.num_pages, w.hkv, 16, w.head_dim)
        if device_gen:
            self.k = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
            self.v = torch.empty(shape, dtype=torch.bfloat16, device=DEV)
            owner = to_dev(self.pm.owner)
            lens_t = to_dev(self.lens)
            need = to_dev(gen.positions_needed(w, self.lens).astype(np.int32))
            u = to_dev(gen.unit_direction(w))
            for which, t in ((0, self.k), (1, self.v)):
                vg.vegas_synth_paged_kv(t, which, w.seed, layer, owner, self.pm.num_pages, w.hkv,
                                        w.head_dim, self.pm.max_pages, lens_t, need,
                                        gen.heavy_threshold(w), w.heavy_last, u)
            self.k_bits = self.v_bits = None
        else:
            self.k_bits = gen.paged_cache_bf16(w, layer, "k", self.lens, self.pm)
            self.v_bits = gen.paged_cache_bf16(w, layer, "v", self.lens, self.pm)
            self.k = to_dev_bf16(self.k_bits)
            self.v = to_dev_bf16(self.v_bits)
        self.qv_bits = gen.f32_to_bf16_bits(gen.verify_queries_f32(w, layer))
        self.qd_bits = gen.f32_to_bf16_bits(gen.draft_queries_f32(w, layer))
        self.qv = to_dev_bf16(self.qv_bits)
        self.qd = to_dev_bf16(self.qd_bits)
        self.bt = to_dev(self.pm.block_table)
        self.lens_t = to_dev(self.lens)
        self.kps_t = to_dev(self.kps)
        self.kv = vg.paged_kv(self.k, self.v, self.bt, w.hq)
        self.stride = max(int(self.lens.max()), 1)
        self.k_max = max(int(self.kps.max()), 1)

    # ------------------------------------------------------------ GPU calls
    def verify(self, capture=True, rows=None, out=None, scores=None, mask=None):
        """Verify with capture rows (a, b), or with a row bit mask when mask is given."""
        w = self.w
        rows = rows if rows is not None else (0, w.gamma)
        out = torch.empty_like(self.qv) if out is None else out
        if capture and scores is None:
            scores = torch.full((w.batch, w.hkv, self.stride), float("nan"), device=DEV)
        nbytes = vg.vegas_verify_workspace_size(self.kv, w.batch, w.gamma)
        ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=DEV)
        if mask is not None:
            vg.vegas_verify_attn_capture_rows(self.kv, self.qv, out, scores if capture else None,
                                              self.stride, self.lens_t, w.batch, w.gamma, mask,
                                              self.scale, ws, ws.numel())
        else:
            vg.vegas_verify_attn_capture(self.kv, self.qv, out, scores if capture else None,
                                         self.stride, self.lens_t, w.batch, w.gamma, rows[0],
                                         rows[1], self.scale, ws, ws.numel())
        return out, scores

    def select(self, scores, k_per_seq=None, k_max=None):
        w = self.w
        kps_t = self.kps_t if k_per_seq is None else to_dev(np.asarray(k_per_seq, np.int32))
        k_max = self.k_max if k_max is None else k_max
        idx = torch.full((w.batch, w.hkv, k_max), -7, dtype=torch.int32, device=DEV)
        vg.vegas_select_topk(scores, scores.shape[-1], self.lens_t, kps_t, idx, w.batch, w.hkv,
                             k_max)
        return idx

    def sparse(self, step, idx, k_per_seq=None, tail_len=None, q=None):
        w = self.w
        k_max = idx.shape[-1]
        kps_t = self.kps_t if k_per_seq is None else to_dev(np.asarray(k_per_seq, np.int32))
        tl = gen.tail_len(w, step) if tail_len is None else tail_len
        tl_t = torch.full((w.batch,), tl, dtype=torch.int32, device=DEV)
        q = self.qd[step] if q is None else q
        out = torch.empty_like(q)
        vg.vegas_sparse_decode_attn(self.kv, q, out, idx, k_max, kps_t, self.lens_t, tl_t, tl,
                                    w.batch, self.scale)
        return out

    # ------------------------------------------------------------ oracle view
    def caches_f64(self):
        assert self.k_bits is not None, "full oracle caches need host-generated inputs"
        return gen.bf16_bits_to_f64(self.k_bits), gen.bf16_bits_to_f64(self.v_bits)

    def unit_rows(self, b: int, g: int, n: int):
        """fp64 K, V rows of logical positions [0, n) of unit (b, g), from the generator."""
        pos = np.arange(n)
        L = int(self.lens[b])
        K = gen.bf16_bits_to_f64(gen.kv_rows_bf16(self.w, self.layer, "k", b, g, pos, L))
        V = gen.bf16_bits_to_f64(gen.kv_rows_bf16(self.w, self.layer, "v", b, g, pos, L))
        return K, V

    def qv_f64(self):
        return gen.bf16_bits_to_f64(self.qv_bits)

    def qd_f64(self):
        return gen.bf16_bits_to_f64(self.qd_bits)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_attention_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    """Attention tolerance for bf16 inputs with fp32 accumulation:
    max-abs <= 2e-2 and relative Frobenius error <= 1e-2."""
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref).max()
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    assert err <= 2e-2, f"{what}: max-abs error {err}"
    assert rel <= 1e-2, f"{what}: relative Frobenius error {rel}"
    return err, rel


def score_bound(q_rows: np.ndarray, K: np.ndarray, scale: float) -> np.ndarray:
    """fp32-accumulation bound on a captured score: 2^-15 * sum_t sum_h sum_j |q_j k_j| * scale.
    q_rows: the captured query rows [r][d]; K: [n][d]."""
    return 2.0 ** -15 * (np.abs(K) @ np.abs(q_rows).sum(0)) * scale


def tie_band_ok(gpu_set, ref_set, s: np.ndarray, k: int) -> tuple[bool, str]:
    """Index sets may differ only at positions whose oracle score lies within
    1e-3 * max(|s_k|, RMS(s)) of the k-th largest oracle score s_k."""
    gpu_set, ref_set = set(int(i) for i in gpu_set), set(int(i) for i in ref_set)
    if len(gpu_set) != k:
        return False, f"gpu selected {len(gpu_set)} != {k}"
    diff = gpu_set ^ ref_set
    if not diff:
        return True, ""
    sk = np.sort(s)[::-1][k - 1]
    band = 1e-3 * max(abs(sk), float(np.sqrt(np.mean(s * s))))
    bad = [i for i in diff if abs(s[i] - sk) > band]
    return (not bad), f"{len(diff)} differ, {len(bad)} outside band {band:.3g}: {bad[:5]}"
