"""The head_dim-32 tensor-core kernel with the sub-tiles of a line pipelined (impl
"tc_pipe").

A line longer than 64 tokens spans several sub-tiles of the chunk's gain recurrence
("VisionHOPE", App. B.4 Prop. 2, Eq. (46)).  In the pipelined form one warp pair reads
out sub-tile s - 1 and prepares sub-tile s (generation, per-token step, Gram entries)
while the other runs the gates and the gain over sub-tile s - 1.  The arithmetic and its
order are those of the sequential form ("tc_recur"), so the final memories agree bit for
bit; `out` sums the four routes' readouts with atomic adds in no fixed order, so it agrees
to the last bits only.  Parity with the fp64 oracle is checked as for every kernel: lines
of 2 to 4 sub-tiles with ragged last sub-tiles, both orientations, route subsets, gate
modes (including retentions small enough for the per-token gain path), per-channel
lambda, the full-size high-resolution workload, and the calls the form rejects.
"""
import numpy as np
import pytest

from visual_backbone_gb300 import synth
from tests._helpers import TOL, oracle_params_like, parity_err, run_gpu

pytestmark = pytest.mark.gpu

# `out` at a pixel is the sum of four routes' readouts, added in whatever order the atomic
# adds land: two orders differ by a few fp32 ulps of the largest term, and parity_err
# measures that against max(|out|, 1e-2 rms), so up to ~100 x 3 x 2^-24 x (term / rms)
OUT_ORDER_TOL = 1e-4


def _both(vhlib, wl, dirs=15, vhp=None, dir_scale=None):
    inp = synth.make_inputs(wl)
    res = {}
    for impl in ("tc_pipe", "tc_recur"):
        p = vhp or vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init)
        p.impl = impl
        res[impl] = run_gpu(vhlib, inp, params=p, dirs=dirs, dir_scale=dir_scale,
                            want_memories=True, want_stats=True, impl=impl)
    return inp, res


def _check(orc, vhlib, wl, dirs=15, vhp=None, dir_scale=None):
    inp, res = _both(vhlib, wl, dirs, vhp, dir_scale)
    g, s = res["tc_pipe"], res["tc_recur"]
    sel = [r for r in range(4) if dirs & (1 << r)]
    # the same arithmetic in the same order: identical memories, and the same statistics
    assert np.array_equal(g["mem"], s["mem"], equal_nan=True)
    assert np.array_equal(g["stats"], s["stats"])
    assert parity_err(g["out"], s["out"]) < OUT_ORDER_TOL
    assert g["stats"][0] == inp.x64.shape[0] * len(sel) * wl.nh * wl.H * wl.W
    assert g["stats"][3] == 0 and g["stats"][4] == 0
    p = oracle_params_like(orc, vhp or vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init),
                           dir_scale)
    o, om = orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d, dirs=dirs, params=p,
                        want_memories=True, nthreads=8)
    e_out, e_mem = parity_err(g["out"], o), parity_err(g["mem"][:, sel], om[:, sel])
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("case", [
    # B, H, W, nh, alpha_init, eta_bias  (chunk = row / column)
    (1, 8, 130, 1, 0.999, 0.0),    # rows of three sub-tiles, the last of two tokens
    (1, 130, 8, 1, 0.999, 0.0),    # the same along the columns
    (2, 65, 66, 2, 0.99, 1.0),     # two sub-tiles, one and two tokens past the first
    (1, 3, 256, 1, 0.9, 0.0),      # four full sub-tiles, the pages' retention
    (1, 200, 2, 2, 0.999, 0.0),    # four sub-tiles, the last of eight tokens
    (1, 128, 128, 1, 0.999, 0.0),  # two full sub-tiles both ways
    (3, 5, 64, 1, 0.999, 0.0),     # one sub-tile: the pipeline's shortest form
])
def test_pipe_shapes(orc, vhlib, case):
    B, H, W, nh, ainit, eb = case
    wl = synth.Workload("pipe", B, H, W, nh, 32, 0, "bf16", seed=H * 100 + W + 3, eta_bias=eb,
                        alpha_init=ainit)
    _check(orc, vhlib, wl)


@pytest.mark.parametrize("dirs", [1, 2, 4, 8, 5, 10, 6])
def test_pipe_route_subsets(orc, vhlib, dirs):
    wl = synth.Workload("piped", 1, 20, 150, 1, 32, 0, "bf16", seed=41, alpha_init=0.999)
    _check(orc, vhlib, wl, dirs=dirs)


@pytest.mark.parametrize("mode", ["unchanged", "forced_raw", "forced_exec", "tiny_alpha",
                                  "spec_heavy"])
def test_pipe_gate_modes(orc, vhlib, mode):
    """Forced gates; with retentions below 0.01 the gain pair takes its per-token path."""
    wl = synth.Workload("pipeg", 1, 10, 140, 1, 32, 0, "bf16", seed=42, alpha_init=0.999)
    p = vhlib.ScanParams(alpha_init=wl.alpha_init)
    if mode == "unchanged":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.0, 1.0
    elif mode == "forced_raw":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.05, 0.8
    elif mode == "forced_exec":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_EXEC, 0.01, 0.95
    elif mode == "tiny_alpha":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 0.3, 0.005
    elif mode == "spec_heavy":
        p.gate_mode, p.forced_eta, p.forced_alpha = vhlib.GATE_FORCED_RAW, 50.0, 0.05
    _check(orc, vhlib, wl, vhp=p)


def test_pipe_dir_scale(orc, vhlib):
    wl = synth.Workload("pipel", 2, 7, 100, 2, 32, 0, "bf16", seed=43, alpha_init=0.999)
    lam = np.random.default_rng(9).uniform(-1.5, 1.5, (4, wl.Cc)).astype(np.float32)
    _check(orc, vhlib, wl, dir_scale=lam)


@pytest.mark.parametrize("variant", ["plain", "longmem"])
def test_pipe_full_size_highres(orc, vhlib, variant):
    """The high-resolution workload (rows of 160 tokens, columns of 128) on the whole
    batch: memories identical to the sequential form on every image, oracle on the first
    and last image."""
    wl = synth.WORKLOADS["highres"]
    if variant == "longmem":
        wl = wl.long_memory()
    inp, res = _both(vhlib, wl)
    g, s = res["tc_pipe"], res["tc_recur"]
    assert np.array_equal(g["mem"], s["mem"])
    assert np.array_equal(g["stats"], s["stats"])
    assert g["stats"][0] == wl.B * 4 * wl.nh * wl.N and g["stats"][4] == 0
    assert parity_err(g["out"], s["out"]) < OUT_ORDER_TOL
    p = oracle_params_like(orc, vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init))
    for b in (0, wl.B - 1):
        o, om = orc.forward(inp.x64[b:b + 1], inp.mem0, wl.H, wl.W, wl.nh, wl.d, params=p,
                            want_memories=True, nthreads=8)
        e_out = parity_err(g["out"][b:b + 1], o)
        e_mem = parity_err(g["mem"][b:b + 1], om)
        assert e_out < TOL and e_mem < TOL, (b, e_out, e_mem)


def test_pipe_rejects_other_methods(vhlib):
    """The pipelined form runs the method as defined at head_dim 32 only."""
    import torch
    for d, kw in [(32, {"control_flags": vhlib.CTRL_HARD_INJ}), (64, {})]:
        wl = synth.Workload("pr", 1, 4, 70, 1, d, 0, "bf16", seed=44)
        inp = synth.make_inputs(wl)
        x = torch.from_numpy(inp.x_store.view(np.int16)).view(torch.bfloat16).cuda()
        m = torch.from_numpy(inp.mem0).cuda()
        with pytest.raises(vhlib.VhError, match="pipelined"):
            vhlib.scan_forward(x, m, d, params=vhlib.ScanParams(impl="tc_pipe", **kw))
    wl = synth.Workload("pr", 1, 4, 70, 1, 32, 0, "bf16", seed=44)
    inp = synth.make_inputs(wl)
    x = torch.from_numpy(inp.x_store.view(np.int16)).view(torch.bfloat16).cuda()
    m = torch.from_numpy(inp.mem0).cuda()
    wq = torch.randn(wl.Cc, wl.Cc).cuda()
    with pytest.raises(vhlib.VhError, match="pipelined"):
        vhlib.scan_forward(x, m, 32, w_query=wq, params=vhlib.ScanParams(impl="tc_pipe"))


def test_pipe_accumulates_onto_out(vhlib):
    """accumulate=True adds the readouts onto the caller's out, as the sequential form."""
    import torch
    from tests._helpers import to_device_x
    wl = synth.Workload("pacc", 1, 6, 100, 1, 32, 0, "bf16", seed=45, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    x = to_device_x(inp)
    m = torch.from_numpy(inp.mem0).cuda()
    base = torch.randn(1, wl.H, wl.W, wl.Cc, device="cuda")
    p = vhlib.ScanParams(alpha_init=wl.alpha_init, impl="tc_pipe")
    ref = vhlib.scan_forward(x, m, 32, dirs=3, params=p)
    out = base.clone()
    vhlib.scan_forward(x, m, 32, dirs=3, out=out, accumulate=True, params=p)
    torch.cuda.synchronize()
    torch.testing.assert_close(out, base + ref, rtol=1e-5, atol=1e-5)


def test_pipe_square_map_with_explicit_chunk(orc, vhlib):
    """A square map with chunk = H = W given explicitly (rows and columns of 96 tokens, two
    sub-tiles each) runs the aligned pipelined form."""
    wl = synth.Workload("psq", 1, 96, 96, 1, 32, 96, "bf16", seed=46, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    p = vhlib.ScanParams(alpha_init=wl.alpha_init, impl="tc_pipe")
    g = run_gpu(vhlib, inp, params=p, chunk=96, want_memories=True, want_stats=True, impl="tc_pipe")
    assert g["stats"][4] == 0
    o, om = orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d, chunk_len=96,
                        params=oracle_params_like(orc, p), want_memories=True, nthreads=8)
    assert parity_err(g["out"], o) < TOL and parity_err(g["mem"], om) < TOL
