"""Parity of the VisionHOPE-exact readout on the GPU ("VisionHOPE: Visual Backbones as
Self-Modifying Learning Systems", Sec. 2.1.2 Eq. (14), App. B.5): outer query projection
shared by the routes, per-head normalisation, channel-wise skip; against the oracle."""
import numpy as np
import pytest

from visual_backbone_gb300 import synth
from tests._helpers import TOL, f32, oracle_params_like, parity_err, to_device_x

pytestmark = pytest.mark.gpu

IMPLS = ["simt", "auto"]


def _extras(Cc, seed):
    rng = np.random.default_rng(1000 + seed)
    wq = (rng.standard_normal((Cc, Cc)) / np.sqrt(Cc)).astype(np.float32)
    skip = rng.standard_normal((4, Cc)).astype(np.float32)
    lam = (0.5 + rng.random((4, Cc))).astype(np.float32)
    return wq, skip, lam


def _run(vhlib, inp, wq, skip, lam, impl, dirs=15, want_memories=True, accumulate_on=None,
         flags=0):
    import torch
    wl = inp.wl
    x = to_device_x(inp)
    mem0 = torch.from_numpy(inp.mem0).cuda()
    vhp = vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init, impl=impl,
                           control_flags=flags)
    mo = (torch.full((x.shape[0], 4, wl.nh, 4 * wl.d * wl.d + 2 * wl.d), float("nan"),
                     device="cuda") if want_memories else None)
    st = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = None if accumulate_on is None else torch.from_numpy(accumulate_on).cuda()
    out = vhlib.scan_forward(
        x, mem0, wl.d, dirs=dirs, params=vhp, out=out, accumulate=accumulate_on is not None,
        memories_out=mo, stats=st,
        w_query=None if wq is None else torch.from_numpy(wq).cuda(),
        skip=None if skip is None else torch.from_numpy(skip).cuda(),
        dir_scale=None if lam is None else torch.from_numpy(lam).cuda())
    torch.cuda.synchronize()
    vhlib.check(st)
    return out.cpu().numpy(), (mo.cpu().numpy() if mo is not None else None), st.cpu().numpy()


def _oracle(orc, vhlib, inp, wq, skip, lam, dirs=15, flags=0):
    wl = inp.wl
    p = oracle_params_like(orc, vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init,
                                                 control_flags=flags), lam)
    p.w_query = None if wq is None else wq.astype(np.float64)
    p.skip = None if skip is None else skip.astype(np.float64)
    return orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d, dirs=dirs, params=p,
                       want_memories=True, nthreads=8)


CASES = [
    ("tiny", synth.WORKLOADS["tiny"]),
    ("6x6x2x32", synth.Workload("e1", 2, 6, 6, 2, 32, 0, "bf16", seed=31, alpha_init=0.999)),
    ("5x70x2x32", synth.Workload("e2", 2, 5, 70, 2, 32, 0, "bf16", seed=32, alpha_init=0.999)),
    ("130x3x1x32", synth.Workload("e3", 1, 130, 3, 1, 32, 0, "bf16", seed=33, eta_bias=1.0)),
    ("7x7x2x64", synth.Workload("e4", 1, 7, 7, 2, 64, 0, "bf16", seed=34, alpha_init=0.999)),
]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_exact_small(orc, vhlib, impl, name, wl):
    inp = synth.make_inputs(wl)
    wq, skip, lam = _extras(wl.Cc, wl.seed)
    g, gm, st = _run(vhlib, inp, wq, skip, lam, impl)
    o, om = _oracle(orc, vhlib, inp, wq, skip, lam)
    e_out, e_mem = parity_err(g, o), parity_err(gm, om)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)
    assert st[0] == inp.x64.shape[0] * 4 * wl.nh * wl.H * wl.W


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name,wl", CASES[:3], ids=[c[0] for c in CASES[:3]])
def test_exact_intra_read(orc, vhlib, impl, name, wl):
    """The outer query read out from the working state M^m_b G_{t-1} (intra-chunk switch)."""
    inp = synth.make_inputs(wl)
    wq, skip, lam = _extras(wl.Cc, wl.seed)
    g, gm, _ = _run(vhlib, inp, wq, skip, lam, impl, flags=vhlib.CTRL_INTRA_READ)
    o, om = _oracle(orc, vhlib, inp, wq, skip, lam, flags=vhlib.CTRL_INTRA_READ)
    e_out, e_mem = parity_err(g, o), parity_err(gm, om)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("impl", IMPLS)
def test_memories_match_the_six_memory_form(vhlib, impl):
    """The outer query feeds only the readout: the same kernel leaves the same memories."""
    wl = synth.Workload("e5", 2, 6, 6, 2, 32, 0, "bf16", seed=35, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    wq, skip, lam = _extras(wl.Cc, wl.seed)
    _, m5, _ = _run(vhlib, inp, wq, skip, lam, impl)
    _, m6, _ = _run(vhlib, inp, None, None, lam, impl)
    np.testing.assert_array_equal(m5, m6)


@pytest.mark.parametrize("impl", IMPLS)
def test_skip_with_accumulate(orc, vhlib, impl):
    wl = synth.Workload("e6", 1, 6, 6, 2, 32, 0, "bf16", seed=36, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    wq, skip, lam = _extras(wl.Cc, wl.seed)
    base = np.random.default_rng(7).standard_normal((1, 6, 6, wl.Cc)).astype(np.float32)
    g, _, _ = _run(vhlib, inp, wq, skip, lam, impl, dirs=5, accumulate_on=base.copy())
    o, _ = _oracle(orc, vhlib, inp, wq, skip, lam, dirs=5)
    assert parity_err(g - base, o) < TOL


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("variant", ["plain", "longmem"])
def test_exact_stage1_sampled(orc, vhlib, impl, variant):
    """Whole stage-1 batch on the GPU; the oracle on the first and last image."""
    wl = synth.WORKLOADS["stage1"]
    if variant == "longmem":
        wl = wl.long_memory()
    inp = synth.make_inputs(wl)
    wq, skip, lam = _extras(wl.Cc, wl.seed)
    g, gm, st = _run(vhlib, inp, wq, skip, lam, impl)
    assert st[0] == wl.B * 4 * wl.nh * wl.N
    for b in (0, wl.B - 1):
        sub = synth.make_inputs(wl)
        sub.x64 = inp.x64[b:b + 1]
        o, om = _oracle(orc, vhlib, sub, wq, skip, lam)
        e_out, e_mem = parity_err(g[b:b + 1], o), parity_err(gm[b:b + 1], om)
        assert e_out < TOL and e_mem < TOL, (b, e_out, e_mem)
