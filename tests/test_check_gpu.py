"""vh_check on a GB300: the device status counters reach the caller.  Non-finite
values are made from the input (a NaN pixel); an expired wait is represented by
writing its counter, never by stalling the device."""
import numpy as np
import pytest

from visual_backbone_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(vhlib, wl, poison=False):
    import torch
    inp = synth.make_inputs(wl)
    x64 = inp.x_store.copy()
    if poison:
        x64.reshape(-1)[5] = np.nan if x64.dtype == np.float32 else np.uint16(0x7FC0)
    if wl.dtype == "bf16":
        x = torch.from_numpy(x64.view(np.int16)).view(torch.bfloat16).cuda()
    else:
        x = torch.from_numpy(x64).cuda()
    m = torch.from_numpy(inp.mem0).cuda()
    st = torch.zeros(8, dtype=torch.int64, device="cuda")
    vhlib.scan_forward(x, m, wl.d, stats=st,
                       params=vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init))
    return st


@pytest.mark.parametrize("name", ["tiny", "tc"])
def test_check_passes_a_clean_run(vhlib, name):
    wl = synth.WORKLOADS["tiny"] if name == "tiny" else synth.Workload("t", 1, 6, 6, 1, 32, 0, "bf16", seed=5)
    vhlib.check(_run(vhlib, wl))


@pytest.mark.parametrize("name", ["tiny", "tc"])
def test_check_reports_nonfinite_readout(vhlib, name):
    wl = synth.WORKLOADS["tiny"] if name == "tiny" else synth.Workload("t", 1, 6, 6, 1, 32, 0, "bf16", seed=5)
    st = _run(vhlib, wl, poison=True)
    with pytest.raises(vhlib.VhError, match="non-finite"):
        vhlib.check(st)
    assert int(st[3].item()) > 0


def test_check_reports_timeout_counter(vhlib):
    import torch
    st = torch.zeros(8, dtype=torch.int64, device="cuda")
    st[4] = 1
    st[3] = 7
    with pytest.raises(vhlib.VhError, match="timeout"):
        vhlib.check(st)
