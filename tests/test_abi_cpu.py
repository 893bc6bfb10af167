"""The C-ABI library loads and exports every declared entry point (no GPU needed).

Only host-side argument validation is exercised here: those calls return a
status before anything touches a device.  They pass made-up addresses, so
they run only where no GPU is visible: on a GPU machine a validation bug
would launch a kernel on them.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _gpu_visible() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except ImportError:
        return False


@pytest.fixture(scope="module")
def vg():
    if _gpu_visible():
        pytest.skip("made-up device addresses: host-validation tests run only without a GPU")
    import __graft_entry__
    try:
        __graft_entry__.build()
    except RuntimeError as e:          # no nvcc on this machine
        pytest.skip(str(e))
    import self_speculative_sparse_paged_gb300 as mod
    return mod


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(vegas_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(vg):
    decl = _declared_functions()
    assert "vegas_verify_attn_capture" in decl and "vegas_select_topk" in decl
    assert "vegas_sparse_decode_attn" in decl
    lib = ctypes.CDLL(vg.library_path())
    for name in decl:
        assert hasattr(lib, name), name


def test_binding_uses_the_same_names(vg):
    for name in _declared_functions():
        assert callable(getattr(vg, name)), name


def test_status_strings(vg):
    assert vg.vegas_abi_version() == 1
    for code, name in vg.STATUS.items():
        assert vg.vegas_status_string(code) == name


def test_host_validation_rejects_before_launch(vg):
    kv = vg.PagedKV(0, 0, 0, 1, 16, 8, 2, 64, 1)        # NULL caches
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_capture(kv, 16, 16, None, 0, 16, 1, 4, 0, 4, 0.125, None, 0,
                                     stream=0)
    assert ei.value.status == 1
    kv = vg.PagedKV(16, 16, 16, 1, 8, 8, 2, 64, 1)      # page size 8
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_capture(kv, 16, 16, None, 0, 16, 1, 4, 0, 4, 0.125, None, 0,
                                     stream=0)
    assert ei.value.status == 2
    kv = vg.PagedKV(16, 16, 16, 1, 16, 8, 2, 96, 1)     # head_dim 96
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_sparse_decode_attn(kv, 16, 16, 16, 4, 16, 16, 16, 1, 1, 0.1, stream=0)
    assert ei.value.status == 2
    kv = vg.PagedKV(16, 16, 16, 1, 16, 8, 2, 128, 1)    # 32769 draft entries
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_sparse_decode_attn(kv, 16, 16, 16, 32760, 16, 16, 16, 9, 1, 0.1, stream=0)
    assert ei.value.status == 2
    kv = vg.PagedKV(16, 16, 16, 1, 16, 64, 2, 128, 1)   # (gamma+1)*G = 5*32 rows
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_capture(kv, 16, 16, None, 0, 16, 1, 4, 0, 4, 0.125, None, 0,
                                     stream=0)
    assert ei.value.status == 2
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_select_topk(None, 16, 16, 16, 16, 1, 8, 10, stream=0)
    assert ei.value.status == 1
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_select_topk(16, 16 * 32768 + 1, 16, 16, 16, 1, 8, 10, stream=0)
    assert ei.value.status == 2


def test_host_validation_of_the_variant_entry_points(vg):
    kv = vg.PagedKV(16, 16, 16, 4, 16, 8, 2, 64, 4)
    # capture row masks must name rows inside [0, gamma]
    for mask in (0, 1 << 5):
        with pytest.raises(vg.VegasError) as ei:
            vg.vegas_verify_attn_capture_rows(kv, 16, 16, 16, 64, 16, 1, 4, mask, 0.125, None, 0,
                                              stream=0)
        assert ei.value.status == 1
    # raw-logit mode needs a buffer and a valid mask
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_raw_logits(kv, 16, 16, None, 64, 16, 1, 4, 0b10001, 0.125, None, 0,
                                        stream=0)
    assert ei.value.status == 1
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_raw_logits(kv, 16, 16, 16, 64, 16, 1, 4, 1 << 7, 0.125, None, 0,
                                        stream=0)
    assert ei.value.status == 1
    # q and out must be 16-byte aligned (the kernels store output rows in vectors)
    kv16 = vg.PagedKV(16, 16, 16, 4, 16, 8, 2, 64, 4)
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_capture(kv16, 16, 18, None, 0, 16, 1, 4, 0, 4, 0.125, None, 0,
                                     stream=0)
    assert ei.value.status == 1 and "aligned" in ei.value.detail
    # aggregate: query heads must be a multiple of the KV heads
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_aggregate_raw_logits(16, 64, 16, 1, 2, 6, 4, 64, 16, 64, stream=0)
    assert ei.value.status == 1
    # window selection needs k_max >= sinks + window
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_select_window(16, 4, 16, 16, 16, 1, 2, 10, stream=0)
    assert ei.value.status == 1
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_select_window(16, -1, 16, 16, 16, 1, 2, 20, stream=0)
    assert ei.value.status == 1
    # shared select: same argument checks as the per-head select
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_select_topk_shared(None, 64, 16, 16, 16, 1, 2, 8, stream=0)
    assert ei.value.status == 1
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_select_topk_shared(16, 9 * 32768, 16, 16, 16, 1, 2, 8, stream=0)
    assert ei.value.status == 2


def test_noalloc_checks_every_argument_before_its_scratch(vg):
    """The no-alloc verify rejects a bad call with the status of the workspace
    call, before it looks up or clears its scratch array (no device is needed
    to reach these answers)."""
    kv = vg.PagedKV(16, 16, 16, 4, 16, 8, 2, 64, 4)
    with pytest.raises(vg.VegasError) as ei:         # NULL queries
        vg.vegas_verify_attn_capture_noalloc(kv, None, 16, 16, 64, 16, 1, 4, 0, 4, 0.125,
                                             stream=0)
    assert ei.value.status == 1
    with pytest.raises(vg.VegasError) as ei:         # misaligned output
        vg.vegas_verify_attn_capture_noalloc(kv, 16, 24, 16, 64, 16, 1, 4, 0, 4, 0.125,
                                             stream=0)
    assert ei.value.status == 1
    with pytest.raises(vg.VegasError) as ei:         # gamma beyond 15: unsupported, not "too small"
        vg.vegas_verify_attn_capture_noalloc(kv, 16, 16, 16, 64, 16, 1, 16, 0, 16, 0.125,
                                             stream=0)
    assert ei.value.status == 2
    big = vg.PagedKV(16, 16, 16, 4, 16, 64, 2, 128, 4)   # (gamma+1)*G query rows too many
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_capture_noalloc(big, 16, 16, 16, 64, 16, 1, 4, 0, 4, 0.125,
                                             stream=0)
    assert ei.value.status == 2


def test_bounded_wait_check_limits_are_checked_on_the_host(vg):
    for bad in (0, -5, 1000001):
        with pytest.raises(vg.VegasError) as ei:
            vg.vegas_check_bounded_wait(bad, None, stream=0)
        assert ei.value.status == 1


def test_decode_iteration_checks_every_layer_before_launching(vg):
    kv = vg.PagedKV(16, 16, 16, 4, 16, 8, 2, 64, 4)
    good = vg.Layer(kv, 16, 16, 16, 16, 16, 16)
    bad_kv = vg.Layer(vg.PagedKV(16, 16, 16, 4, 16, 8, 2, 96, 4), 16, 16, 16, 16, 16, 16)
    other_heads = vg.Layer(vg.PagedKV(16, 16, 16, 4, 16, 4, 2, 64, 4), 16, 16, 16, 16, 16, 16)
    null_idx = vg.Layer(kv, 16, 16, 16, 16, 16, 0)
    args = (16, 16, 16, 8, 1, 4, 64, 8, 0.125, None, 0)
    for layers, status in (([good, bad_kv], 2), ([good, other_heads], 1), ([good, null_idx], 1),
                           ([], 1)):
        with pytest.raises(vg.VegasError) as ei:
            vg.vegas_decode_iteration(layers, *args, stream=0)
        assert ei.value.status == status
    with pytest.raises(vg.VegasError) as ei:           # gamma beyond 15
        vg.vegas_decode_iteration([good], 16, 16, 16, 8, 1, 16, 64, 8, 0.125, None, 0, stream=0)
    assert ei.value.status == 2
    with pytest.raises(vg.VegasError) as ei:           # the select stream must be another one
        vg.vegas_decode_iteration([good], *args, stream=5, select_stream=5)
    assert ei.value.status == 1
