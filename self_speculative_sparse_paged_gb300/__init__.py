"""Python binding of libvegas.so, the GB300 (sm_103a) Vegas hot path.

Argument marshalling only: each function below forwards to the C entry point of
the same name declared in include/vegas.h.  Every step of the path runs in the
library's CUDA kernels; there is no Python or CPU fallback, and importing this
package fails loudly when the library has not been built
(``python -c "import __graft_entry__ as g; g.build()"``).

Pointer arguments accept a torch tensor (its data_ptr()), a plain integer
device address, or None (NULL).  ``stream`` accepts a torch.cuda.Stream, a raw
cudaStream_t integer, or None for torch's current stream on the current device.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

__all__ = [
    "VegasError", "PagedKV", "paged_kv", "lib", "library_path",
    "vegas_verify_workspace_size", "vegas_verify_attn_capture", "vegas_select_topk",
    "vegas_sparse_decode_attn", "vegas_synth_paged_kv", "vegas_verify_attn_capture_noalloc",
    "vegas_verify_noalloc_max_scratch_bytes", "vegas_check_bounded_wait", "Layer", "layer",
    "vegas_decode_iteration",
    "vegas_read_device_status", "vegas_status_string", "vegas_last_error_detail",
    "vegas_abi_version",
]

STATUS = {
    0: "VEGAS_OK", 1: "VEGAS_ERR_INVALID_ARG", 2: "VEGAS_ERR_UNSUPPORTED",
    3: "VEGAS_ERR_WORKSPACE_TOO_SMALL", 4: "VEGAS_ERR_CUDA", 5: "VEGAS_ERR_DEVICE_FAULT",
    6: "VEGAS_ERR_DEVICE_TIMEOUT",
}


class VegasError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{STATUS.get(status, status)}: {detail}")
        self.status = status
        self.detail = detail


class PagedKV(ctypes.Structure):
    """Mirror of vegas_paged_kv_t."""
    _fields_ = [
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("num_pages", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
    ]


def library_path() -> str:
    return _build.LIB


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(
            f"libvegas.so not found at {path}; build it first "
            "(python -c \"import __graft_entry__ as g; g.build()\")")
    return ctypes.CDLL(path)


lib = _load()

_c_void_p, _i32, _sz, _f32, _u64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t,
                                    ctypes.c_float, ctypes.c_uint64)
_P_KV = ctypes.POINTER(PagedKV)


def _sig(name, res, args):
    fn = getattr(lib, name)
    fn.restype = res
    fn.argtypes = args
    return fn


_verify_ws = _sig("vegas_verify_workspace_size", _sz, [_P_KV, _i32, _i32])
_verify = _sig("vegas_verify_attn_capture", _i32,
               [_P_KV, _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _i32, _i32, _i32, _i32,
                _f32, _c_void_p, _sz, _c_void_p])
_verify_rows = _sig("vegas_verify_attn_capture_rows", _i32,
                    [_P_KV, _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _i32, _i32,
                     ctypes.c_uint32, _f32, _c_void_p, _sz, _c_void_p])
_verify_raw = _sig("vegas_verify_attn_raw_logits", _i32,
                   [_P_KV, _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _i32, _i32,
                    ctypes.c_uint32, _f32, _c_void_p, _sz, _c_void_p])
_raw_agg = _sig("vegas_aggregate_raw_logits", _i32,
                [_c_void_p, _i32, _c_void_p, _i32, _i32, _i32, _i32, _i32, _c_void_p, _i32,
                 _c_void_p])
_verify_noalloc = _sig("vegas_verify_attn_capture_noalloc", _i32,
                       [_P_KV, _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _i32, _i32,
                        _i32, _i32, _f32, _c_void_p])
_noalloc_max = _sig("vegas_verify_noalloc_max_scratch_bytes", _sz, [])
_select = _sig("vegas_select_topk", _i32,
               [_c_void_p, _i32, _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32, _c_void_p])
_select_shared = _sig("vegas_select_topk_shared", _i32,
                      [_c_void_p, _i32, _c_void_p, _c_void_p, _c_void_p, _i32, _i32, _i32,
                       _c_void_p])
_window = _sig("vegas_select_window", _i32,
               [_c_void_p, _i32, _i32, _c_void_p, _c_void_p, _i32, _i32, _i32, _c_void_p])
_sparse = _sig("vegas_sparse_decode_attn", _i32,
               [_P_KV, _c_void_p, _c_void_p, _c_void_p, _i32, _c_void_p, _c_void_p, _c_void_p,
                _i32, _i32, _f32, _c_void_p])
_synth = _sig("vegas_synth_paged_kv", _i32,
              [_c_void_p, _i32, _u64, _i32, _c_void_p, _i32, _i32, _i32, _i32, _c_void_p,
               _c_void_p, _u64, _i32, _c_void_p, _c_void_p])
class Layer(ctypes.Structure):
    """Mirror of vegas_layer_t."""
    _fields_ = [
        ("kv", PagedKV),
        ("q_verify", ctypes.c_void_p),
        ("out_verify", ctypes.c_void_p),
        ("q_draft", ctypes.c_void_p),
        ("out_draft", ctypes.c_void_p),
        ("scores", ctypes.c_void_p),
        ("idx", ctypes.c_void_p),
    ]


_iteration = _sig("vegas_decode_iteration", _i32,
                  [ctypes.POINTER(Layer), _i32, _c_void_p, _c_void_p, _c_void_p, _i32, _i32,
                   _i32, _i32, _i32, _f32, _c_void_p, _sz, _c_void_p, _c_void_p])
_wait_check = _sig("vegas_check_bounded_wait", _i32, [_i32, _c_void_p, _c_void_p])
_read_status = _sig("vegas_read_device_status", _i32, [_c_void_p])
_status_string = _sig("vegas_status_string", ctypes.c_char_p, [_i32])
_detail = _sig("vegas_last_error_detail", ctypes.c_char_p, [])
_abi = _sig("vegas_abi_version", _i32, [])


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int):
    if status != 0:
        raise VegasError(status, vegas_last_error_detail())


def paged_kv(k_cache, v_cache, block_table, num_q_heads: int) -> PagedKV:
    """vegas_paged_kv_t for bf16 caches [pages][Hkv][16][d] and an int32 block table."""
    num_pages, hkv, page, d = k_cache.shape
    return PagedKV(_ptr(k_cache), _ptr(v_cache), _ptr(block_table), num_pages, page,
                   num_q_heads, hkv, d, block_table.shape[-1])


def vegas_verify_workspace_size(kv: PagedKV, batch: int, gamma: int) -> int:
    return _verify_ws(ctypes.byref(kv), batch, gamma)


def vegas_verify_attn_capture(kv: PagedKV, q, out, scores, score_stride: int, ctx_lens,
                              batch: int, gamma: int, capture_row_a: int, capture_row_b: int,
                              softmax_scale: float, workspace, workspace_bytes: int,
                              stream=None) -> None:
    _check(_verify(ctypes.byref(kv), _ptr(q), _ptr(out), _ptr(scores), score_stride,
                   _ptr(ctx_lens), batch, gamma, capture_row_a, capture_row_b, softmax_scale,
                   _ptr(workspace), workspace_bytes, _stream(stream)))


def vegas_verify_attn_capture_rows(kv: PagedKV, q, out, scores, score_stride: int, ctx_lens,
                                   batch: int, gamma: int, capture_row_mask: int,
                                   softmax_scale: float, workspace, workspace_bytes: int,
                                   stream=None) -> None:
    """vegas_verify_attn_capture with the captured rows as a bit mask (bit t: row t)."""
    _check(_verify_rows(ctypes.byref(kv), _ptr(q), _ptr(out), _ptr(scores), score_stride,
                        _ptr(ctx_lens), batch, gamma, capture_row_mask, softmax_scale,
                        _ptr(workspace), workspace_bytes, _stream(stream)))


def vegas_verify_attn_raw_logits(kv: PagedKV, q, out, raw, raw_stride: int, ctx_lens,
                                 batch: int, gamma: int, capture_row_mask: int,
                                 softmax_scale: float, workspace, workspace_bytes: int,
                                 stream=None) -> None:
    """Verify writing the raw logits of the captured rows of every query head."""
    _check(_verify_raw(ctypes.byref(kv), _ptr(q), _ptr(out), _ptr(raw), raw_stride,
                       _ptr(ctx_lens), batch, gamma, capture_row_mask, softmax_scale,
                       _ptr(workspace), workspace_bytes, _stream(stream)))


def vegas_aggregate_raw_logits(raw, raw_stride: int, ctx_lens, batch: int, num_rows: int,
                               num_q_heads: int, num_kv_heads: int, max_len: int, scores,
                               score_stride: int, stream=None) -> None:
    _check(_raw_agg(_ptr(raw), raw_stride, _ptr(ctx_lens), batch, num_rows, num_q_heads,
                    num_kv_heads, max_len, _ptr(scores), score_stride, _stream(stream)))


def vegas_verify_attn_capture_noalloc(kv: PagedKV, q, out, scores, score_stride: int, ctx_lens,
                                      batch: int, gamma: int, capture_row_a: int,
                                      capture_row_b: int, softmax_scale: float,
                                      stream=None) -> None:
    """vegas_verify_attn_capture without a workspace, for callers that cannot
    allocate device memory; the scratch is a fixed array inside the library."""
    _check(_verify_noalloc(ctypes.byref(kv), _ptr(q), _ptr(out), _ptr(scores), score_stride,
                           _ptr(ctx_lens), batch, gamma, capture_row_a, capture_row_b,
                           softmax_scale, _stream(stream)))


def vegas_verify_noalloc_max_scratch_bytes() -> int:
    return _noalloc_max()


def vegas_select_topk(scores, score_stride: int, ctx_lens, k_per_seq, out_idx, batch: int,
                      num_kv_heads: int, k_max: int, stream=None) -> None:
    _check(_select(_ptr(scores), score_stride, _ptr(ctx_lens), _ptr(k_per_seq), _ptr(out_idx),
                   batch, num_kv_heads, k_max, _stream(stream)))


def vegas_select_topk_shared(scores, score_stride: int, ctx_lens, k_per_seq, out_idx,
                             batch: int, num_kv_heads: int, k_max: int, stream=None) -> None:
    """One T per sequence from the scores summed over its KV heads, written to every head."""
    _check(_select_shared(_ptr(scores), score_stride, _ptr(ctx_lens), _ptr(k_per_seq),
                          _ptr(out_idx), batch, num_kv_heads, k_max, _stream(stream)))


def vegas_select_window(ctx_lens, num_sink: int, window: int, k_out, out_idx, batch: int,
                        num_kv_heads: int, k_max: int, stream=None) -> None:
    """The sink + sliding-window index set, in the layout of vegas_select_topk."""
    _check(_window(_ptr(ctx_lens), num_sink, window, _ptr(k_out), _ptr(out_idx), batch,
                   num_kv_heads, k_max, _stream(stream)))


def vegas_sparse_decode_attn(kv: PagedKV, q, out, idx, k_max: int, k_per_seq, tail_start,
                             tail_len, max_tail: int, batch: int, softmax_scale: float,
                             stream=None) -> None:
    _check(_sparse(ctypes.byref(kv), _ptr(q), _ptr(out), _ptr(idx), k_max, _ptr(k_per_seq),
                   _ptr(tail_start), _ptr(tail_len), max_tail, batch, softmax_scale,
                   _stream(stream)))


def vegas_synth_paged_kv(cache, which: int, seed: int, layer: int, owner, num_pages: int,
                         num_kv_heads: int, head_dim: int, max_pages_per_seq: int, ctx_lens,
                         positions, heavy_threshold: int, heavy_last: int, unit_dir,
                         stream=None) -> None:
    _check(_synth(_ptr(cache), which, seed, layer, _ptr(owner), num_pages, num_kv_heads,
                  head_dim, max_pages_per_seq, _ptr(ctx_lens), _ptr(positions), heavy_threshold,
                  heavy_last, _ptr(unit_dir), _stream(stream)))


def layer(kv: PagedKV, q_verify, out_verify, q_draft, out_draft, scores, idx) -> Layer:
    """vegas_layer_t of one layer's tensors."""
    return Layer(kv, _ptr(q_verify), _ptr(out_verify), _ptr(q_draft), _ptr(out_draft),
                 _ptr(scores), _ptr(idx))


def vegas_decode_iteration(layers, ctx_lens, k_per_seq, tail_lens, max_tail: int, batch: int,
                           gamma: int, score_stride: int, k_max: int, softmax_scale: float,
                           workspace, workspace_bytes: int, stream=None,
                           select_stream=None) -> None:
    """verify + select for every layer, then every draft step over every layer;
    select(l) overlaps verify(l + 1) when select_stream is given."""
    arr = (Layer * len(layers))(*layers)
    sel = None if select_stream is None else _stream(select_stream)
    _check(_iteration(arr, len(layers), _ptr(ctx_lens), _ptr(k_per_seq), _ptr(tail_lens),
                      max_tail, batch, gamma, score_stride, k_max, softmax_scale,
                      _ptr(workspace), workspace_bytes, _stream(stream), sel))


def vegas_check_bounded_wait(limit_us: int, outcome=None, stream=None) -> None:
    """Launches the failure-detection check: a wait that runs out after limit_us."""
    _check(_wait_check(limit_us, _ptr(outcome), _stream(stream)))


def vegas_read_device_status(stream=None) -> None:
    """Synchronises the stream; raises VegasError if a kernel recorded a fault."""
    _check(_read_status(_stream(stream)))


def vegas_status_string(status: int) -> str:
    return _status_string(status).decode()


def vegas_last_error_detail() -> str:
    return _detail().decode()


def vegas_abi_version() -> int:
    return _abi()
