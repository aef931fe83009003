"""Parity of the tensor-core kernel's WY form of the shared gain with the fp64 oracle.

The WY form ("VisionHOPE", App. B.4 Prop. 2, Eqs. (46), (49) unrolled) forms the keys'
Gram matrix and assembles G = gamma_L I + W' K^T on the tensor core, and solves the
chunk's triangular system for W on CUDA cores.  It is selected with impl "tc_wy" for
the method as defined when every chunk fits one 64-token sub-tile; the default kernel
keeps the blocked recurrence (the faster form on this part).  These cases cover the
solve sizes built (28, 56 exactly; 32 and 64 with zero padding), both route
directions, the gate modes, small retentions whose products underflow, per-channel
lambda and the full-size workloads, plus the shapes the form rejects.
"""
import numpy as np
import pytest

from visual_backbone_gb300 import synth
from tests._helpers import TOL, oracle_params_like, parity_err, run_gpu, to_device_x

pytestmark = pytest.mark.gpu


def _compare(orc, vhlib, wl, impl="tc_wy", dirs=15, vhp=None, dir_scale=None):
    inp = synth.make_inputs(wl)
    if vhp is None:
        vhp = vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init)
    g = run_gpu(vhlib, inp, params=vhp, dirs=dirs, dir_scale=dir_scale, want_memories=True,
                want_stats=True, impl=impl)
    p = oracle_params_like(orc, vhp, dir_scale)
    o, om = orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d, dirs=dirs, params=p,
                        want_memories=True, nthreads=8)
    sel = [r for r in range(4) if dirs & (1 << r)]
    assert g["stats"][0] == inp.x64.shape[0] * len(sel) * wl.nh * wl.H * wl.W
    assert g["stats"][3] == 0 and g["stats"][4] == 0
    return parity_err(g["out"], o), parity_err(g["mem"][:, sel], om[:, sel])


@pytest.mark.parametrize("case", [
    # B, H, W, nh, alpha_init, eta_bias  (chunk = row / column)
    (1, 8, 8, 2, 0.999, 0.0),      # solve of 32, zero-padded
    (1, 28, 28, 2, 0.999, 0.0),    # solve of 28
    (1, 56, 56, 1, 0.999, 0.0),    # solve of 56 (the stage-1 chunk)
    (1, 56, 56, 1, 0.9, 0.0),      # the pages' retention: the state decays over the scan
    (2, 40, 13, 1, 0.999, 1.0),    # rows of 13 (32), columns of 40 (64), raised steps
    (1, 64, 64, 1, 0.999, 0.0),    # a full sub-tile
    (1, 33, 31, 2, 0.99, 1.0),     # one past 32 and one short of it
    (3, 1, 17, 1, 0.999, 0.0),     # one-row map
])
def test_wy_shapes(orc, vhlib, case):
    B, H, W, nh, ainit, eb = case
    wl = synth.Workload("wy", B, H, W, nh, 32, 0, "bf16", seed=H * 100 + W + 7, eta_bias=eb,
                        alpha_init=ainit)
    e_out, e_mem = _compare(orc, vhlib, wl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("dirs", [1, 2, 4, 8, 5, 10])
def test_wy_route_subsets(orc, vhlib, dirs):
    wl = synth.Workload("wyd", 1, 28, 20, 2, 32, 0, "bf16", seed=31, alpha_init=0.999)
    e_out, e_mem = _compare(orc, vhlib, wl, dirs=dirs)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("mode", ["unchanged", "forced_raw", "forced_exec", "tiny_alpha",
                                  "spec_heavy"])
def test_wy_gate_modes(orc, vhlib, mode):
    """Forced gates, including retentions whose products over a chunk underflow fp32
    (0.05^28 ~ 4e-37, 0.02^28 below the normal range): every factor of the WY form is a
    product of retentions, so it flushes to zero where the recurrence decays."""
    wl = synth.Workload("wyg", 1, 28, 28, 1, 32, 0, "bf16", seed=32, alpha_init=0.999)
    p = vhlib.ScanParams(alpha_init=wl.alpha_init)
    if mode == "unchanged":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.0, 1.0
    elif mode == "forced_raw":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.05, 0.8
    elif mode == "forced_exec":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_EXEC, 0.01, 0.95
    elif mode == "tiny_alpha":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.3, 0.02
    elif mode == "spec_heavy":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 50.0, 0.05
    e_out, e_mem = _compare(orc, vhlib, wl, vhp=p)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)
    if mode == "unchanged":
        inp = synth.make_inputs(wl)
        g = run_gpu(vhlib, inp, params=p, want_memories=True, impl="tc_wy")
        for r in range(4):
            np.testing.assert_array_equal(g["mem"][0, r], inp.mem0[r])


def test_wy_dir_scale(orc, vhlib):
    wl = synth.Workload("wyl", 2, 12, 20, 2, 32, 0, "bf16", seed=33, alpha_init=0.999)
    ds = synth.make_dir_scale(wl)
    e_out, e_mem = _compare(orc, vhlib, wl, dir_scale=ds)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


def test_wy_reversal_symmetry_bit_exact(vhlib):
    """scan(left, X) == rot180(scan(right, rot180 X)) bit for bit in the WY form too."""
    import torch
    wl = synth.Workload("wyr", 2, 28, 20, 2, 32, 0, "bf16", seed=34, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    inp.mem0[1] = inp.mem0[0]
    inp.mem0[3] = inp.mem0[2]
    x = to_device_x(inp)
    xr = torch.flip(x, dims=(1, 2)).contiguous()
    m = torch.from_numpy(inp.mem0).cuda()
    p = vhlib.ScanParams(alpha_init=wl.alpha_init, impl="tc_wy")
    for fwd, rev in ((1, 2), (4, 8)):
        a = vhlib.scan_forward(x, m, wl.d, dirs=rev, params=p)
        b = vhlib.scan_forward(xr, m, wl.d, dirs=fwd, params=p)
        torch.cuda.synchronize()
        assert torch.equal(a, torch.flip(b, dims=(1, 2)))


@pytest.mark.parametrize("name", ["stage1", "stage2"])
@pytest.mark.parametrize("variant", ["plain", "longmem"])
def test_wy_full_size_sampled(orc, vhlib, name, variant):
    """The whole batch through the WY form; the oracle on the first and last image."""
    wl = synth.WORKLOADS[name]
    if variant == "longmem":
        wl = wl.long_memory()
    inp = synth.make_inputs(wl)
    g = run_gpu(vhlib, inp, want_memories=True, want_stats=True, impl="tc_wy")
    assert g["stats"][0] == wl.B * 4 * wl.nh * wl.N and g["stats"][3] == 0 and g["stats"][4] == 0
    p = oracle_params_like(orc, vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init))
    for b in (0, wl.B - 1):
        o, om = orc.forward(inp.x64[b:b + 1], inp.mem0, wl.H, wl.W, wl.nh, wl.d, params=p,
                            want_memories=True, nthreads=8)
        e_out = parity_err(g["out"][b:b + 1], o)
        e_mem = parity_err(g["mem"][b:b + 1], om)
        assert e_out < TOL and e_mem < TOL, (b, e_out, e_mem)


def test_wy_rejects_other_shapes(vhlib):
    """The WY form needs the method as defined and chunks within one sub-tile."""
    import torch
    wl = synth.Workload("wyx", 1, 4, 70, 1, 32, 0, "bf16", seed=35)
    inp = synth.make_inputs(wl)
    x = to_device_x(inp)
    m = torch.from_numpy(inp.mem0).cuda()
    with pytest.raises(vhlib.VhError, match="unsupported"):
        vhlib.scan_forward(x, m, 32, params=vhlib.ScanParams(impl="tc_wy"))
    wl = synth.Workload("wyx", 1, 8, 8, 1, 32, 0, "bf16", seed=36)
    inp = synth.make_inputs(wl)
    x = to_device_x(inp)
    m = torch.from_numpy(inp.mem0).cuda()
    p = vhlib.ScanParams(impl="tc_wy", control_flags=vhlib.CTRL_HARD_INJ)
    with pytest.raises(vhlib.VhError, match="unsupported"):
        vhlib.scan_forward(x, m, 32, params=p)
