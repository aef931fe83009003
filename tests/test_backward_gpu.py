"""Outer gradients on the GPU (vh_scan_backward) against the gradient oracle
("VisionHOPE: Visual Backbones as Self-Modifying Learning Systems", Sec. 2.1.2: outer
gradients pass through the memory trajectory), element by element, on the same seeded
inputs: dx and dmemories0 of <dout, out> + <dmem_final, memories_final>."""
import copy

import numpy as np
import pytest

from visual_backbone_gb300 import synth
from tests._helpers import TOL, oracle_params_like, parity_err, to_device_x

pytestmark = pytest.mark.gpu

# The gradients pass through the whole trajectory (and the fp32 state accumulates its
# rounding over it like the forward), so they carry the forward's tolerance.
GTOL = TOL


def _run(vhlib, inp, vhp, dout, dirs=15, chunk=0, lam=None, dmf=None):
    import torch
    wl = inp.wl
    x = to_device_x(inp)
    mem0 = torch.from_numpy(inp.mem0).cuda()
    dx, dm = vhlib.scan_backward(
        x, mem0, wl.d, torch.from_numpy(dout.astype(np.float32)).cuda(), dirs=dirs, chunk=chunk,
        params=vhp, dir_scale=None if lam is None else torch.from_numpy(lam).cuda(),
        dmem_final=None if dmf is None else torch.from_numpy(dmf.astype(np.float32)).cuda())
    torch.cuda.synchronize()
    return dx.cpu().numpy(), dm.cpu().numpy()


def _oracle(orc, vhlib, inp, vhp, dout, dirs=15, chunk=0, lam=None, dmf=None):
    from oracle import vh_grad
    wl = inp.wl
    p = oracle_params_like(orc, vhp, lam)
    return vh_grad.backward(inp.x64, inp.mem0.astype(np.float64),
                            dout.astype(np.float32).astype(np.float64), wl.H, wl.W, wl.nh,
                            wl.d, dirs, chunk, p,
                            None if dmf is None else dmf.astype(np.float32).astype(np.float64))


def _dout(wl, B, seed):
    return np.random.default_rng(seed).standard_normal((B, wl.H, wl.W, wl.Cc))


CASES = [
    # name, workload, dirs, chunk, ScanParams overrides, dir_scale, dmem_final
    ("tiny", synth.WORKLOADS["tiny"], 15, 0, {}, False, False),
    ("6x6x2x32", synth.Workload("b1", 2, 6, 6, 2, 32, 0, "bf16", seed=51), 15, 0, {}, False, False),
    ("5x9_chunk7", synth.Workload("b2", 1, 5, 9, 2, 32, 0, "bf16", seed=52), 15, 7, {}, False, False),
    ("3x70x1x32", synth.Workload("b3", 1, 3, 70, 1, 32, 0, "bf16", seed=53), 15, 0, {}, False, False),
    ("7x7x1x64", synth.Workload("b4", 1, 7, 7, 1, 64, 0, "bf16", seed=54), 15, 0, {}, False, False),
    ("f32_d32", synth.Workload("b5", 1, 5, 6, 2, 32, 0, "f32", seed=55), 15, 0, {}, False, False),
    ("softcap", synth.Workload("b6", 1, 6, 6, 1, 32, 0, "bf16", seed=56, eta_bias=3.0), 15, 0,
     {}, False, False),
    ("spectral", synth.Workload("b7", 1, 5, 6, 1, 32, 0, "bf16", seed=57, alpha_init=0.05,
                                eta_bias=3.0), 15, 0, {}, False, False),
    ("forced_raw", synth.Workload("b8", 1, 5, 5, 1, 16, 0, "f32", seed=58), 15, 0,
     {"gate_mode": 1, "forced_eta": 0.3, "forced_alpha": 0.8}, False, False),
    ("forced_exec", synth.Workload("b9", 1, 5, 5, 1, 16, 0, "f32", seed=59), 15, 3,
     {"gate_mode": 2, "forced_eta": 0.2, "forced_alpha": 0.7}, False, False),
    ("lam_dirs5_dmf", synth.Workload("b10", 2, 4, 7, 2, 32, 0, "bf16", seed=60), 5, 0, {}, True,
     True),
    ("longmem", synth.Workload("b11", 1, 8, 8, 1, 32, 0, "bf16", seed=61, alpha_init=0.999),
     15, 0, {}, False, True),
    ("one_row", synth.Workload("b13", 2, 1, 17, 1, 32, 0, "bf16", seed=63), 15, 0, {}, False,
     False),
    ("one_column", synth.Workload("b14", 1, 17, 1, 2, 32, 0, "bf16", seed=64), 15, 0, {}, False,
     True),
    ("single_pixel", synth.Workload("b15", 1, 1, 1, 1, 16, 0, "f32", seed=65), 15, 0, {}, False,
     True),
]


@pytest.mark.parametrize("impl", ["simt", "auto"])
@pytest.mark.parametrize("name,wl,dirs,chunk,kw,use_lam,use_dmf", CASES, ids=[c[0] for c in CASES])
def test_backward_parity(orc, vhlib, name, wl, dirs, chunk, kw, use_lam, use_dmf, impl):
    """impl "simt" runs the whole backward in its own kernel; "auto" takes the chunk
    boundary states from the tensor-core forward where it applies (d = 32, bf16,
    aligned chunks)."""
    inp = synth.make_inputs(wl)
    vhp = vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init, impl=impl, **kw)
    B = inp.x64.shape[0]
    dout = _dout(wl, B, 100 + wl.seed)
    lam = synth.make_dir_scale(wl) if use_lam else None
    dmf = (np.random.default_rng(200 + wl.seed).standard_normal(
        (B, 4, wl.nh, 4 * wl.d * wl.d + 2 * wl.d)) * 0.3) if use_dmf else None
    gx, gm = _run(vhlib, inp, vhp, dout, dirs, chunk, lam, dmf)
    ox, om = _oracle(orc, vhlib, inp, vhp, dout, dirs, chunk, lam, dmf)
    e_x, e_m = parity_err(gx, ox), parity_err(gm, om)
    assert e_x < GTOL and e_m < GTOL, (e_x, e_m)
    unsel = [r for r in range(4) if not dirs & (1 << r)]
    assert not gm[unsel].any()


def test_backward_is_linear_in_dout(vhlib):
    """d(dout_1 + 2 dout_2) = d(dout_1) + 2 d(dout_2) (the adjoint is linear), to fp32."""
    wl = synth.Workload("b12", 1, 6, 6, 2, 32, 0, "bf16", seed=62)
    inp = synth.make_inputs(wl)
    vhp = vhlib.ScanParams()
    d1, d2 = _dout(wl, 1, 1), _dout(wl, 1, 2)
    a = _run(vhlib, inp, vhp, d1)
    b = _run(vhlib, inp, vhp, d2)
    c = _run(vhlib, inp, vhp, d1 + 2 * d2)
    for i in range(2):
        ref = a[i] + 2 * b[i]
        assert parity_err(c[i], ref) < 1e-4


SAMPLED = [("stage1", "plain"), ("stage1", "longmem"), ("stage2", "plain"),
           ("stage3", "plain"), ("highres", "plain")]


@pytest.mark.parametrize("config,variant", SAMPLED, ids=[f"{c}-{v}" for c, v in SAMPLED])
def test_backward_sampled(orc, vhlib, config, variant):
    """A whole batch of the configuration in the launch the backward bench times; dx of
    the first (and, for stage-1, the last) image against the oracle, and dmemories0 of a
    one-image call against the oracle on that image."""
    wl = synth.WORKLOADS[config]
    if variant == "longmem":
        wl = wl.long_memory()
    inp = synth.make_inputs(wl)
    vhp = vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init)
    dout = _dout(wl, wl.B, 300)
    gx, _ = _run(vhlib, inp, vhp, dout)
    images = (0, wl.B - 1) if (config, variant) == ("stage1", "plain") else (0,)
    for b in images:
        sub = copy.copy(inp)
        sub.x64 = inp.x64[b:b + 1]
        ox, om = _oracle(orc, vhlib, sub, vhp, dout[b:b + 1])
        assert parity_err(gx[b:b + 1], ox) < GTOL, b
        if b == 0:
            one = synth.make_inputs(wl, batch=1)
            _, gm1 = _run(vhlib, one, vhp, dout[:1])
            assert parity_err(gm1, om) < GTOL
