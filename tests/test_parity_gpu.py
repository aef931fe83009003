"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Small cases run the whole operator on both sides; the workloads at full size
run the GPU on the whole batch (the launch configuration the benchmark
times) and the oracle on sampled images, whose outputs and final memories
it computes exactly.  Index maps are checked bit for bit.
"""
import numpy as np
import pytest

from visual_backbone_gb300 import synth
from tests._helpers import TOL, oracle_params_like, parity_err, run_gpu, to_device_x

pytestmark = pytest.mark.gpu

IMPLS = ["simt", "auto"]


def _oracle_params(orc, wl, vhp=None, dir_scale=None):
    import visual_backbone_gb300 as vh
    if vhp is None:
        vhp = vh.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init)
    return oracle_params_like(orc, vhp, dir_scale)


def _compare(orc, vhlib, wl, dirs=15, chunk=0, vhp=None, dir_scale=None, impl="auto",
             batch=None, nthreads=8):
    inp = synth.make_inputs(wl, batch)
    g = run_gpu(vhlib, inp, params=vhp, dirs=dirs, chunk=chunk, dir_scale=dir_scale,
                want_memories=True, want_stats=True, impl=impl)
    p = _oracle_params(orc, wl, vhp, dir_scale)
    o, om = orc.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d, dirs=dirs, chunk_len=chunk,
                        params=p, want_memories=True, nthreads=nthreads)
    e_out = parity_err(g["out"], o)
    sel = [r for r in range(4) if dirs & (1 << r)]
    e_mem = parity_err(g["mem"][:, sel], om[:, sel])
    unsel = [r for r in range(4) if not dirs & (1 << r)]
    if unsel:
        assert np.isnan(g["mem"][:, unsel]).all(), "disabled routes' memory slots were written"
    nd = len(sel)
    assert g["stats"][0] == inp.x64.shape[0] * nd * wl.nh * wl.H * wl.W
    assert g["stats"][3] == 0 and g["stats"][4] == 0
    return e_out, e_mem


# ------------------------------------------------------------ index maps

@pytest.mark.parametrize("H,W,dtype", [(3, 4, "f32"), (8, 8, "f32"), (5, 7, "bf16"),
                                       (56, 56, "bf16"), (128, 160, "bf16")])
def test_permute_bit_exact(orc, vhlib, H, W, dtype):
    wl = synth.Workload("perm", 2, H, W, 2, 16, dtype=dtype, seed=5)
    inp = synth.make_inputs(wl)
    x = to_device_x(inp)
    for r in range(4):
        seq = vhlib.debug_permute(x, r, 16)
        got = seq.view(seq.shape[0], -1).cpu()
        order = orc.route_order(r, H, W)
        want = inp.x_store.reshape(2, H * W, -1)[:, order, :]
        if dtype == "bf16":
            got = got.view(dtype=__import__("torch").int16).numpy().view(np.uint16)
        else:
            got = got.numpy()
        np.testing.assert_array_equal(got.reshape(want.shape), want)


# ----------------------------------------------------------- small cases

@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("variant", ["plain", "longmem"])
@pytest.mark.parametrize("chunk", [0, 1, 3, 5, 64])
def test_tiny_parity(orc, vhlib, impl, variant, chunk):
    wl = synth.WORKLOADS["tiny"]
    if variant == "longmem":
        wl = wl.long_memory()
    e_out, e_mem = _compare(orc, vhlib, wl, chunk=chunk, impl=impl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("dirs", [1, 2, 4, 8, 5, 10, 7])
def test_direction_subsets(orc, vhlib, impl, dirs):
    wl = synth.WORKLOADS["tiny"].long_memory()
    e_out, e_mem = _compare(orc, vhlib, wl, dirs=dirs, impl=impl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("case", [
    # B, H, W, nh, d, dtype, chunk, alpha_init, eta_bias
    (2, 5, 70, 2, 32, "bf16", 0, 0.999, 0.0),     # rows of 70: two tiles, ragged tail
    (1, 130, 3, 1, 32, "bf16", 0, 0.999, 1.0),    # columns of 130: three tiles
    (2, 4, 64, 2, 32, "bf16", 0, 0.9, 0.0),       # rows of exactly one tile
    (1, 2, 65, 3, 32, "bf16", 65, 0.999, 0.0),    # explicit chunk equal to the row length
    (2, 70, 5, 1, 32, "bf16", 0, 0.99, 1.0),      # columns of 70
    (1, 9, 11, 2, 32, "f32", 7, 0.999, 0.0),      # fixed chunk, partial last chunk
    (2, 3, 40, 1, 64, "bf16", 0, 0.999, 0.0),     # d = 64, rows of 40
    (1, 40, 3, 2, 64, "f32", 0, 0.9, 2.0),        # d = 64, columns of 40
    (1, 6, 6, 3, 16, "bf16", 4, 0.999, 0.0),      # d = 16, bf16
    (3, 1, 17, 1, 32, "bf16", 0, 0.999, 0.0),     # one-row map
    (2, 17, 1, 2, 32, "bf16", 0, 0.999, 0.0),     # one-column map
    (1, 1, 1, 1, 16, "f32", 0, 0.9, 0.0),         # single pixel
])
def test_small_shapes(orc, vhlib, impl, case):
    B, H, W, nh, d, dt, chunk, ainit, eb = case
    wl = synth.Workload("small", B, H, W, nh, d, chunk, dt, seed=H * 100 + W, eta_bias=eb,
                        alpha_init=ainit)
    e_out, e_mem = _compare(orc, vhlib, wl, chunk=chunk, impl=impl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("impl", IMPLS)
def test_dir_scale(orc, vhlib, impl):
    wl = synth.Workload("lam", 2, 6, 9, 2, 32, 0, "bf16", seed=21, alpha_init=0.999)
    ds = synth.make_dir_scale(wl)
    e_out, e_mem = _compare(orc, vhlib, wl, dir_scale=ds, impl=impl)
    assert e_out < TOL and e_mem < TOL


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("mode", ["unchanged", "forced_raw", "forced_exec", "no_controls",
                                  "spec_heavy"])
def test_gate_modes_and_switches(orc, vhlib, impl, mode):
    import visual_backbone_gb300 as vh
    wl = synth.Workload("gates", 1, 6, 8, 2, 16, 0, "f32", seed=22, alpha_init=0.999)
    p = vh.ScanParams(alpha_init=wl.alpha_init)
    if mode == "unchanged":
        p.gate_mode, p.forced_eta, p.forced_alpha = vh.GATE_FORCED_RAW, 0.0, 1.0
    elif mode == "forced_raw":
        p.gate_mode, p.forced_eta, p.forced_alpha = vh.GATE_FORCED_RAW, 0.05, 0.8
    elif mode == "forced_exec":
        p.gate_mode, p.forced_eta, p.forced_alpha = vh.GATE_FORCED_EXEC, 0.01, 0.95
    elif mode == "no_controls":
        p.control_flags = vh.CTRL_NO_SPEC_CLAMP
    elif mode == "spec_heavy":   # small alpha, large raw steps: the spectral clamp binds often
        p.gate_mode, p.forced_eta, p.forced_alpha = vh.GATE_FORCED_RAW, 50.0, 0.05
    e_out, e_mem = _compare(orc, vhlib, wl, vhp=p, impl=impl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)
    if mode == "unchanged":
        inp = synth.make_inputs(wl)
        g = run_gpu(vhlib, inp, params=p, want_memories=True, impl=impl)
        for r in range(4):
            np.testing.assert_array_equal(g["mem"][0, r], inp.mem0[r])


@pytest.mark.parametrize("impl", IMPLS)
def test_reversal_symmetry_bit_exact(vhlib, impl):
    """scan(left, X) == rot180(scan(right, rot180 X)) with equal initial states,
    bit for bit (one route per call, so no cross-route sum order enters)."""
    import torch
    wl = synth.Workload("rev", 2, 7, 9, 2, 32, 0, "bf16", seed=23, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    inp.mem0[1] = inp.mem0[0]
    inp.mem0[3] = inp.mem0[2]
    x = to_device_x(inp)
    xr = torch.flip(x, dims=(1, 2)).contiguous()
    m = torch.from_numpy(inp.mem0).cuda()
    import visual_backbone_gb300 as vh
    p = vh.ScanParams(alpha_init=wl.alpha_init, impl=impl)
    for fwd, rev in ((1, 2), (4, 8)):
        a = vh.scan_forward(x, m, wl.d, dirs=rev, params=p)
        b = vh.scan_forward(xr, m, wl.d, dirs=fwd, params=p)
        torch.cuda.synchronize()
        assert torch.equal(a, torch.flip(b, dims=(1, 2)))


def test_accumulate_adds(vhlib):
    import torch
    import visual_backbone_gb300 as vh
    wl = synth.Workload("acc", 1, 5, 6, 1, 32, 0, "bf16", seed=24, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    x = to_device_x(inp)
    m = torch.from_numpy(inp.mem0).cuda()
    base = torch.randn(1, 5, 6, 32, device="cuda")
    ref = vh.scan_forward(x, m, 32, dirs=1)
    out = base.clone()
    vh.scan_forward(x, m, 32, dirs=1, out=out, accumulate=True)
    torch.cuda.synchronize()
    torch.testing.assert_close(out, base + ref, rtol=1e-6, atol=1e-6)


# --------------------------------------------------- full-size workloads

FULL = ["stage1", "stage2", "stage3", "highres"]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("name", FULL)
@pytest.mark.parametrize("variant", ["plain", "longmem"])
def test_full_size_sampled(orc, vhlib, name, variant, impl):
    """GPU on the whole batch (as timed); oracle on the first and last image."""
    wl = synth.WORKLOADS[name]
    if variant == "longmem":
        wl = wl.long_memory()
    inp = synth.make_inputs(wl)
    g = run_gpu(vhlib, inp, want_memories=True, want_stats=True, impl=impl)
    assert g["stats"][0] == wl.B * 4 * wl.nh * wl.N and g["stats"][3] == 0
    assert g["stats"][4] == 0
    p = _oracle_params(orc, wl)
    for b in (0, wl.B - 1):
        o, om = orc.forward(inp.x64[b:b + 1], inp.mem0, wl.H, wl.W, wl.nh, wl.d, params=p,
                            want_memories=True, nthreads=8)
        e_out = parity_err(g["out"][b:b + 1], o)
        e_mem = parity_err(g["mem"][b:b + 1], om)
        assert e_out < TOL and e_mem < TOL, (b, e_out, e_mem)


@pytest.mark.parametrize("name", ["stage3"])
@pytest.mark.parametrize("variant", ["plain", "longmem"])
def test_full_size_sampled_d64_recurrence(orc, vhlib, name, variant):
    """Stage-3 with the head_dim-64 tensor-core kernel's blocked recurrence forced (the
    default there is the WY form): the whole batch, oracle on the first and last image."""
    test_full_size_sampled(orc, vhlib, name, variant, "tc_recur")


@pytest.mark.parametrize("name", FULL)
def test_full_size_kernels_agree_on_every_image(vhlib, name):
    """The tensor-core kernel (as benchmarked) and the CUDA-core kernel, two independent
    implementations, on the whole batch: every image, every element within the tolerance
    (the oracle checks the first and last image above)."""
    wl = synth.WORKLOADS[name].long_memory()
    inp = synth.make_inputs(wl)
    g = run_gpu(vhlib, inp, want_memories=True, impl="auto")
    s = run_gpu(vhlib, inp, want_memories=True, impl="simt")
    for b in range(wl.B):
        e_out = parity_err(g["out"][b:b + 1], s["out"][b:b + 1])
        e_mem = parity_err(g["mem"][b:b + 1], s["mem"][b:b + 1])
        assert e_out < TOL and e_mem < TOL, (b, e_out, e_mem)
