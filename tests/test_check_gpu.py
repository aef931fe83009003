"""vh_check on a GB300: the device status counters reach the caller.  Non-finite
values are made from the input (a NaN pixel).  An expired wait is made without stalling
or faulting the device: a small wait limit with the test hook that never issues the
kernel's first input copy, so the first wait can only give up and the kernel then issues
no copy or MMA at all before it ends; the context stays usable afterwards."""
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


def test_expired_wait_reports_timeout_and_leaves_context_usable(vhlib, orc):
    import torch
    from tests._helpers import TOL, oracle_params_like, parity_err
    wl = synth.Workload("t", 1, 8, 8, 1, 32, 0, "bf16", seed=5, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    x = torch.from_numpy(inp.x_store.view(np.int16)).view(torch.bfloat16).cuda()
    m = torch.from_numpy(inp.mem0).cuda()
    for impl in ("tc_recur", "tc_wy", "tc_pipe"):
        st = torch.zeros(8, dtype=torch.int64, device="cuda")
        p = vhlib.ScanParams(alpha_init=wl.alpha_init, impl=impl, wait_limit=20000,
                             withhold_first_copy=True)
        vhlib.scan_forward(x, m, 32, stats=st, params=p)
        with pytest.raises(vhlib.VhError, match="timeout"):
            vhlib.check(st)
        assert int(st[4].item()) == 4   # every CTA (4 routes x 1 head) gave up once
        # the same context runs a normal call correctly afterwards
        st = torch.zeros(8, dtype=torch.int64, device="cuda")
        q = vhlib.ScanParams(alpha_init=wl.alpha_init, impl=impl)
        out = vhlib.scan_forward(x, m, 32, stats=st, params=q)
        vhlib.check(st)
        o = orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d, params=oracle_params_like(orc, q))
        assert parity_err(out.cpu().numpy(), o) < TOL


@pytest.mark.parametrize("d,impl", [(32, "tc_recur"), (32, "tc_wy"), (32, "tc_pipe"), (64, "tc_wy"),
                                    (64, "tc_recur")])
def test_wait_expiring_mid_scan_drains(vhlib, orc, d, impl):
    """A one-cycle wait limit makes the first wait that is not already complete give up
    while the CTA's own MMAs (and possibly a copy) are in flight.  The CTA lets them land
    before it frees TMEM and exits: the call reports VH_ERR_TIMEOUT, and the context then
    runs a normal call correctly."""
    import torch
    from tests._helpers import TOL, oracle_params_like, parity_err
    wl = synth.Workload("t", 2, 8, 12, 2, d, 0, "bf16", seed=6, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    x = torch.from_numpy(inp.x_store.view(np.int16)).view(torch.bfloat16).cuda()
    m = torch.from_numpy(inp.mem0).cuda()
    st = torch.zeros(8, dtype=torch.int64, device="cuda")
    p = vhlib.ScanParams(alpha_init=wl.alpha_init, impl=impl, wait_limit=1)
    vhlib.scan_forward(x, m, d, stats=st, params=p)
    with pytest.raises(vhlib.VhError, match="timeout"):
        vhlib.check(st)
    assert 1 <= int(st[4].item()) <= wl.B * 4 * wl.nh   # at most once per CTA
    st = torch.zeros(8, dtype=torch.int64, device="cuda")
    q = vhlib.ScanParams(alpha_init=wl.alpha_init, impl=impl)
    out = vhlib.scan_forward(x, m, d, stats=st, params=q)
    vhlib.check(st)
    o = orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d, params=oracle_params_like(orc, q))
    assert parity_err(out.cpu().numpy(), o) < TOL
