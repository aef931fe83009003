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
}
SHAPES = [
    ("tiny", synth.WORKLOADS["tiny"]),
    ("6x6x2x32", synth.Workload("a1", 2, 6, 6, 2, 32, 0, "bf16", seed=41, alpha_init=0.999)),
    ("5x70x2x32", synth.Workload("a2", 1, 5, 70, 2, 32, 0, "bf16", seed=42, eta_bias=3.0)),
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
def test_frozen_memories_unchanged_on_gpu(vhlib, impl):
    import torch
    from tests._helpers import run_gpu
    wl = synth.Workload("a3", 1, 6, 6, 2, 32, 0, "bf16", seed=43, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    vhp = vhlib.ScanParams(alpha_init=wl.alpha_init, impl=impl, control_flags=32 | 64)
    g = run_gpu(vhlib, inp, params=vhp, want_memories=True)
    d = wl.d
    mo = g["mem"][0]
    m0 = inp.mem0
    for r in range(4):
        for h in range(wl.nh):
            np.testing.assert_array_equal(mo[r, h, :2 * d * d], m0[r, h, :2 * d * d])
            np.testing.assert_array_equal(mo[r, h, 4 * d * d:], m0[r, h, 4 * d * d:])
            assert not np.array_equal(mo[r, h, 3 * d * d:4 * d * d], m0[r, h, 3 * d * d:4 * d * d])
