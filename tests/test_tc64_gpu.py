"""Parity of the head_dim 64 tensor-core kernel with the fp64 oracle.

The kernel takes bf16 maps with row/column chunks and the method as defined.  Where every
chunk fits one 32-token sub-tile it forms the shared gain in WY form ("VisionHOPE",
App. B.4 Prop. 2, Eqs. (46), (49) unrolled: Gram entries and the triangular system on
CUDA cores, G = gamma_L I + W' K^T on the tensor core); longer chunks run the blocked
recurrence across sub-tiles.  Both forms are covered here, with route subsets, per-channel
lambda, forced gates and the pages' retention, against the oracle on the same inputs.
"""
import numpy as np
import pytest

from visual_backbone_gb300 import synth
from tests._helpers import TOL, oracle_params_like, parity_err, run_gpu

pytestmark = pytest.mark.gpu


def _compare(orc, vhlib, wl, dirs=15, vhp=None, dir_scale=None, impl="tc"):
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
    unsel = [r for r in range(4) if not dirs & (1 << r)]
    if unsel:
        assert np.isnan(g["mem"][:, unsel]).all(), "disabled routes' memory slots were written"
    return parity_err(g["out"], o), parity_err(g["mem"][:, sel], om[:, sel])


@pytest.mark.parametrize("case", [
    # B, H, W, nh, alpha_init, eta_bias
    (1, 14, 14, 2, 0.999, 0.0),    # the stage-3 chunk (WY, system of 16)
    (2, 14, 14, 1, 0.9, 0.0),      # the pages' retention
    (2, 20, 31, 1, 0.99, 1.0),     # WY, system of 32, raised steps
    (1, 5, 9, 3, 0.9, 0.0),        # short chunks
    (1, 32, 32, 1, 0.999, 0.0),    # a full sub-tile
    (3, 1, 17, 1, 0.999, 0.0),     # one-row map
    (2, 3, 40, 1, 0.999, 0.0),     # rows of 40: the recurrence over two sub-tiles
    (1, 70, 5, 1, 0.99, 1.0),      # columns of 70: three sub-tiles, ragged tail
])
def test_tc64_shapes(orc, vhlib, case):
    B, H, W, nh, ainit, eb = case
    wl = synth.Workload("t64", B, H, W, nh, 64, 0, "bf16", seed=H * 100 + W + 11, eta_bias=eb,
                        alpha_init=ainit)
    e_out, e_mem = _compare(orc, vhlib, wl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("dirs", [1, 2, 4, 8, 5, 10])
def test_tc64_route_subsets(orc, vhlib, dirs):
    wl = synth.Workload("t64d", 1, 14, 10, 2, 64, 0, "bf16", seed=41, alpha_init=0.999)
    e_out, e_mem = _compare(orc, vhlib, wl, dirs=dirs)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("mode", ["unchanged", "forced_raw", "forced_exec", "tiny_alpha"])
def test_tc64_gate_modes(orc, vhlib, mode):
    wl = synth.Workload("t64g", 1, 14, 14, 1, 64, 0, "bf16", seed=42, alpha_init=0.999)
    p = vhlib.ScanParams(alpha_init=wl.alpha_init)
    if mode == "unchanged":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.0, 1.0
    elif mode == "forced_raw":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.05, 0.8
    elif mode == "forced_exec":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_EXEC, 0.01, 0.95
    elif mode == "tiny_alpha":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.3, 0.003
    e_out, e_mem = _compare(orc, vhlib, wl, vhp=p)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)
    if mode == "unchanged":
        inp = synth.make_inputs(wl)
        g = run_gpu(vhlib, inp, params=p, want_memories=True, impl="tc")
        for r in range(4):
            np.testing.assert_array_equal(g["mem"][0, r], inp.mem0[r])


def test_tc64_dir_scale(orc, vhlib):
    wl = synth.Workload("t64l", 2, 9, 14, 2, 64, 0, "bf16", seed=43, alpha_init=0.999)
    ds = synth.make_dir_scale(wl)
    e_out, e_mem = _compare(orc, vhlib, wl, dir_scale=ds)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("impl", ["tc_recur", "tc_wy"])
@pytest.mark.parametrize("case", [
    (2, 14, 14, 2, 0.999, 0.0),    # the stage-3 chunk
    (1, 9, 32, 1, 0.9, 1.0),       # rows of a full sub-tile, the pages' retention
])
def test_tc64_gain_forms(orc, vhlib, impl, case):
    """Either gain form forced on chunks that fit one sub-tile (where the default is WY)."""
    B, H, W, nh, ainit, eb = case
    wl = synth.Workload("t64f", B, H, W, nh, 64, 0, "bf16", seed=H * 7 + W, eta_bias=eb,
                        alpha_init=ainit)
    e_out, e_mem = _compare(orc, vhlib, wl, impl=impl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


def test_tc64_wy_rejects_long_chunks(vhlib):
    """WY at head_dim 64 needs every chunk within one 32-token sub-tile."""
    import torch
    from tests._helpers import to_device_x
    wl = synth.Workload("t64x", 1, 4, 40, 1, 64, 0, "bf16", seed=44)
    inp = synth.make_inputs(wl)
    x = to_device_x(inp)
    m = torch.from_numpy(inp.mem0).cuda()
    with pytest.raises(vhlib.VhError, match="unsupported"):
        vhlib.scan_forward(x, m, 64, params=vhlib.ScanParams(impl="tc_wy"))
