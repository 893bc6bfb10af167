"""The device input generator reproduces the host generator bit for bit."""
import numpy as np
import pytest
import torch

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from vegas_case import Case  # noqa: E402
from workload import configs, gen  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("w", [
    configs.TINY,
    configs.GPTOSS_20B_B4_128K.with_(batch=2, ctx_lo=900, ctx_hi=1300),
    configs.QWEN3_8B_36L_B4_96K_120K.with_(batch=2, ctx_lo=500, ctx_hi=800),
])
@pytest.mark.parametrize("layer", [0, 3])
def test_device_generator_matches_host(w, layer):
    c = Case(w, layer=layer, device_gen=True)
    lens = c.lens
    for which, t in (("k", c.k), ("v", c.v)):
        host = gen.paged_cache_bf16(w, layer, which, lens, c.pm)
        dev = t.view(torch.int16).cpu().numpy().view(np.uint16)
        np.testing.assert_array_equal(dev, host)
