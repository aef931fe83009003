"""The ablation switches on the GPU ("VisionHOPE: Visual Backbones as Self-Modifying
Learning Systems", Sec. 3.5 and App. C.5) against the oracle, on both kernels."""
import numpy as np
import pytest

from visual_backbone_gb300 import synth
from tests._helpers import TOL
from tests.test_parity_gpu import _compare

pytestmark = pytest.mark.gpu

IMPLS = ["simt", "auto"]
FLAGS = {
    "hard_inj": 4, "soft_spec": 8, "no_dgd": 16, "freeze_kv": 32, "freeze_dyn": 64,
    "hard_inj+soft_spec": 12, "no_dgd+freeze_kv+freeze_dyn": 112,
    "intra_read": 128, "intra_read+no_dgd": 144,
}
SHAPES = [
    ("tiny", synth.WORKLOADS["tiny"]),
    ("6x6x2x32", synth.Workload("a1", 2, 6, 6, 2, 32, 0, "bf16", seed=41, alpha_init=0.999)),
    ("5x70x2x32", synth.Workload("a2", 1, 5, 70, 2, 32, 0, "bf16", seed=42, eta_bias=3.0)),
    # d = 64: the CUDA-core kernel's register-tiled update and its eta / alpha rows, three
    # 16-token tiles per row
    ("3x40x1x64", synth.Workload("a5", 1, 3, 40, 1, 64, 0, "bf16", seed=48, alpha_init=0.999)),
]


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("flag", list(FLAGS))
@pytest.mark.parametrize("name,wl", SHAPES, ids=[s[0] for s in SHAPES])
def test_ablation_parity(orc, vhlib, impl, flag, name, wl):
    vhp = vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init, impl=impl,
                           control_flags=FLAGS[flag])
    e_out, e_mem = _compare(orc, vhlib, wl, vhp=vhp, impl=impl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("H,W,nh,d", [(6, 6, 2, 32), (3, 40, 1, 64)])
def test_frozen_memories_unchanged_on_gpu(vhlib, impl, H, W, nh, d):
    from tests._helpers import run_gpu
    wl = synth.Workload("a3", 1, H, W, nh, d, 0, "bf16", seed=43, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    vhp = vhlib.ScanParams(alpha_init=wl.alpha_init, impl=impl, control_flags=32 | 64)
    g = run_gpu(vhlib, inp, params=vhp, want_memories=True)
    mo = g["mem"][0]
    m0 = inp.mem0
    for r in range(4):
        for h in range(wl.nh):
            np.testing.assert_array_equal(mo[r, h, :2 * d * d], m0[r, h, :2 * d * d])
            np.testing.assert_array_equal(mo[r, h, 4 * d * d:], m0[r, h, 4 * d * d:])
            assert not np.array_equal(mo[r, h, 3 * d * d:4 * d * d], m0[r, h, 3 * d * d:4 * d * d])


# the intra-chunk readout where the tensor-core kernel's gain takes its per-token path
# (some alpha < 0.01), over two sub-tiles; a short fixed chunk on the CUDA-core kernel
INTRA = [
    ("small_alpha", synth.Workload("i1", 1, 4, 70, 2, 32, 0, "bf16", seed=44, alpha_init=0.004),
     0, "auto"),
    ("chunk7", synth.Workload("i2", 1, 5, 9, 2, 32, 0, "bf16", seed=45), 7, "simt"),
    ("chunk7_d64", synth.Workload("i3", 1, 5, 9, 1, 64, 0, "bf16", seed=46), 7, "simt"),
]


@pytest.mark.parametrize("name,wl,chunk,impl", INTRA, ids=[c[0] for c in INTRA])
def test_intra_read_parity(orc, vhlib, name, wl, chunk, impl):
    vhp = vhlib.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init, impl=impl,
                           control_flags=128)
    e_out, e_mem = _compare(orc, vhlib, wl, chunk=chunk, vhp=vhp, impl=impl)
    assert e_out < TOL and e_mem < TOL, (e_out, e_mem)


@pytest.mark.parametrize("impl", IMPLS)
def test_intra_read_differs_from_boundary_readout(vhlib, impl):
    from tests._helpers import run_gpu
    wl = synth.Workload("i4", 1, 6, 6, 2, 32, 0, "bf16", seed=47)
    inp = synth.make_inputs(wl)
    a = run_gpu(vhlib, inp, params=vhlib.ScanParams(impl=impl), want_memories=True)
    b = run_gpu(vhlib, inp, params=vhlib.ScanParams(impl=impl, control_flags=128),
                want_memories=True)
    # the memories do not depend on the readout; the outputs do
    np.testing.assert_array_equal(a["mem"], b["mem"])
    assert np.abs(a["out"] - b["out"]).max() > 1e-3
