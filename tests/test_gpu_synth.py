"""The device input generator reproduces the host generator bit for bit."""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wname", ["tiny_fp32", "prefill_8k"])
def test_device_equals_host(cuda_ok, wname):
    w = synth.scaled(synth.WORKLOADS[wname], hot="first4")
    for name in ("q", "k", "v", "iq", "ik"):
        d = synth.device_tensor(w, name, "cuda:0")
        h = synth.host_tensor(w, name)
        assert np.array_equal(d.float().cpu().numpy(), h), name


def test_device_offset_fill(cuda_ok):
    w = synth.WORKLOADS["prefill_1m"]
    n, start = 1 << 20, (1 << 34) + 12345
    buf = torch.empty(n, dtype=torch.bfloat16, device="cuda:0")
    synth.fill_device(w, "k", buf, start=start)
    assert np.array_equal(buf.float().cpu().numpy(), synth.host_range(w, "k", start, n))
