"""Device-detected faults are reported through the error word, never by a trap."""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import self_speculative_sparse_paged_gb300 as vg  # noqa: E402
from vegas_case import Case, to_dev  # noqa: E402
from workload import configs  # noqa: E402

pytestmark = pytest.mark.gpu


def test_out_of_range_block_table_entry_sets_device_fault():
    c = Case(configs.TINY.with_(ctx_lo=200, ctx_hi=200))
    vg.vegas_read_device_status()
    bad = c.pm.block_table.copy()
    bad[0, 3] = c.pm.num_pages + 5          # the kernel clamps the access and records it
    c.bt.copy_(to_dev(bad))
    c.verify()
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_read_device_status()
    assert ei.value.status == 5
    vg.vegas_read_device_status()           # the word was cleared
    c.bt.copy_(to_dev(c.pm.block_table))
    c.verify()
    vg.vegas_read_device_status()


def test_selected_index_past_capacity_sets_device_fault():
    c = Case(configs.TINY.with_(ctx_lo=200, ctx_hi=200, k_abs=4))
    idx = np.array([[[0, 1, 2, 10 ** 6]] * c.w.hkv], dtype=np.int32)
    c.sparse(0, to_dev(idx))
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_read_device_status()
    assert ei.value.status == 5


def test_k_larger_than_prefix_sets_device_fault():
    c = Case(configs.TINY.with_(ctx_lo=50, ctx_hi=50, k_abs=10))
    _, s = c.verify()
    c.select(s, k_per_seq=[60], k_max=64)
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_read_device_status()
    assert ei.value.status == 5


def test_small_workspace_is_rejected_on_the_host():
    # 44 query rows at head_dim 128: the mma.sync kernel merges its splits
    # through the workspace
    c = Case(configs.QWEN3_8B_B1_32K.with_(gamma=10, ctx_lo=4000, ctx_hi=4000))
    need = vg.vegas_verify_workspace_size(c.kv, 1, c.w.gamma)
    assert need > 0
    ws = torch.zeros(need // 2, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(c.qv)
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_verify_attn_capture(c.kv, c.qv, out, None, 1, c.lens_t, 1, c.w.gamma, 0,
                                     c.w.gamma, c.scale, ws, ws.numel())
    assert ei.value.status == 3


def test_a_bounded_wait_that_runs_out_reports_a_timeout_and_the_gpu_stays_usable():
    """The failure-detection protocol end to end: a kernel's wait on a barrier
    nothing arrives on gives up after its limit (1 ms here), records
    VEGAS_ERR_DEVICE_TIMEOUT and returns; the host reads it once, the word
    clears, and the context keeps working."""
    vg.vegas_read_device_status()
    outcome = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    vg.vegas_check_bounded_wait(1000, outcome)
    with pytest.raises(vg.VegasError) as ei:
        vg.vegas_read_device_status()
    assert ei.value.status == 6
    assert int(outcome.item()) == 0             # the wait ran out
    vg.vegas_read_device_status()               # cleared
    c = Case(configs.TINY.with_(ctx_lo=100, ctx_hi=100))
    c.verify()
    vg.vegas_read_device_status()               # later kernels run normally
