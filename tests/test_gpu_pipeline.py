"""Layer-pipelined select: select(l) on a second stream overlapping verify(l + 1)
gives bit-for-bit the outputs of the serial schedule and of each layer run alone."""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bench  # noqa: E402
from vegas_case import Case  # noqa: E402
from workload import configs  # noqa: E402

pytestmark = pytest.mark.gpu


def _outputs(st):
    return ([o.clone() for o in st.out_v], [o.clone() for o in st.out_d],
            [i.clone() for i in st.idx])


@pytest.mark.parametrize("w,layers", [(configs.TINY, 3),
                                      (configs.QWEN3_8B_B1_32K.with_(ctx_lo=3000, ctx_hi=3000), 4)])
def test_pipelined_stack_equals_serial_and_single_layers(w, layers):
    st = bench.LayerStack(w, layers, torch.device("cuda"))
    st.step(pipelined=False)
    torch.cuda.synchronize()
    ser = _outputs(st)
    for buf in st.out_v + st.out_d:
        buf.fill_(float("nan"))
    for buf in st.idx:
        buf.fill_(-7)
    st.step(pipelined=True)
    torch.cuda.synchronize()
    pip = _outputs(st)
    for a, b in zip(ser[0] + ser[1], pip[0] + pip[1]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    for a, b in zip(ser[2], pip[2]):
        assert torch.equal(a, b)
    # the last layer equals that layer run alone through the single-layer calls
    c = Case(w, layer=layers - 1, device_gen=True)
    out_v, scores = c.verify()
    idx = c.select(scores)
    assert torch.equal(idx, pip[2][-1])
    assert torch.equal(out_v.view(torch.int16), pip[0][-1].view(torch.int16))
    for j in range(w.gamma):
        o = c.sparse(j, idx)
        assert torch.equal(o.view(torch.int16), pip[1][-1][j].view(torch.int16))


def test_stack_schedule_without_capture_runs_the_window_selector():
    """The overhead denominator: plain verify, window selection, the same drafts."""
    w = configs.TINY
    st = bench.LayerStack(w, 2, torch.device("cuda"))
    st.step_without_capture()
    torch.cuda.synchronize()
    sinks = min(64, st.k_max // 2)
    for layer in range(2):
        idx = st.idx[layer].cpu().numpy()
        L = int(st.lens[0])
        want = [i for i in range(L) if i < sinks or i >= L - (st.k_max - sinks)]
        assert list(idx[0, 0, :len(want)]) == want
        assert np.isfinite(st.out_d[layer].float().cpu().numpy()).all()
