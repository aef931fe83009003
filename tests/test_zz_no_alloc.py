"""vh_scan_forward_static: the outer-query forward for callers that cannot allocate
device memory themselves (for instance a plug-in inside a host application that owns
every device allocation).  Its query scratch is a fixed array inside the library, so
the caller passes only inputs and outputs.

Checked through the C ABI against vh_scan_forward with a caller-allocated workspace, on
two calls in a row with different shapes (the second call reuses the array the first
one filled), on a call that fills the array almost to its limit, on a call that adds to
out (accumulate), and on the size limit.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest

from visual_backbone_gb300 import synth
from tests._helpers import TOL, parity_err, to_device_x

pytestmark = pytest.mark.gpu

STATIC_LIMIT = (16 << 20) // 6   # elements of x the 16 MiB array can serve


def _entry(vhlib):
    f = vhlib.lib().vh_scan_forward_static
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(vhlib.CParams), ctypes.c_int,
                  ctypes.c_int, ctypes.c_uint, ctypes.c_int, ctypes.c_void_p]
    return f


def _inputs(wl):
    import torch
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(500 + wl.seed)
    wq = torch.from_numpy((rng.standard_normal((wl.Cc, wl.Cc)) / np.sqrt(wl.Cc)).astype(np.float32))
    skip = torch.from_numpy(rng.standard_normal((4, wl.Cc)).astype(np.float32))
    lam = torch.from_numpy(rng.uniform(0.5, 1.5, (4, wl.Cc)).astype(np.float32))
    return (to_device_x(inp), torch.from_numpy(inp.mem0).cuda(), wq.cuda(), skip.cuda(), lam.cuda())


def test_static_scratch_matches_the_workspace_path(vhlib):
    import torch
    f = _entry(vhlib)
    cases = [synth.Workload("s1", 2, 12, 14, 3, 32, 0, "bf16", seed=71),   # tensor-core scan
             synth.Workload("s2", 1, 9, 7, 2, 16, 0, "f32", seed=72)]      # CUDA-core scan
    for wl in cases:
        x, mem0, wq, skip, lam = _inputs(wl)
        B, H, W, Cc = x.shape
        out = torch.full((B, H, W, Cc), float("nan"), device="cuda")
        cp = vhlib.make_cparams(B, Cc, wl.d, wl.dtype == "bf16", None,
                                dir_scale_ptr=lam.data_ptr(), stream_ptr=vhlib._stream_ptr(None),
                                w_query_ptr=wq.data_ptr(), skip_ptr=skip.data_ptr())
        st = f(x.data_ptr(), mem0.data_ptr(), ctypes.byref(cp), H, W, 15, 0, out.data_ptr())
        assert st == 0, vhlib.lib().vh_last_error().decode()
        ref = vhlib.scan_forward(x, mem0, wl.d, w_query=wq, skip=skip, dir_scale=lam)
        torch.cuda.synchronize()
        assert parity_err(out.cpu().numpy(), ref.cpu().numpy()) < TOL, wl.name


def test_static_scratch_rejects_what_does_not_fit(vhlib):
    f = _entry(vhlib)
    # a batch just large enough to pass the limit
    H, W, Cc = 64, 64, 384
    B = STATIC_LIMIT // (H * W * Cc) + 1
    cp = vhlib.make_cparams(B, Cc, 32, True, None, w_query_ptr=1 << 20)
    base = 1 << 36  # never dereferenced: the size check comes first
    assert f(base, base, ctypes.byref(cp), H, W, 15, 0, base) == -4
    assert b"static scratch" in vhlib.lib().vh_last_error()
    cp.w_query = None
    assert f(base, base, ctypes.byref(cp), H, W, 15, 0, base) == -1


def _call_both(vhlib, f, wl, accumulate=False):
    """The static entry and vh_scan_forward (caller workspace) on the same inputs; out
    starts from the same values on both sides (NaN unless accumulating)."""
    import torch
    x, mem0, wq, skip, lam = _inputs(wl)
    B, H, W, Cc = x.shape
    if accumulate:
        base = torch.randn(B, H, W, Cc, device="cuda")
        out, ref = base.clone(), base.clone()
    else:
        out = torch.full((B, H, W, Cc), float("nan"), device="cuda")
        ref = None
    cp = vhlib.make_cparams(B, Cc, wl.d, wl.dtype == "bf16", None, accumulate=accumulate,
                            dir_scale_ptr=lam.data_ptr(), stream_ptr=vhlib._stream_ptr(None),
                            w_query_ptr=wq.data_ptr(), skip_ptr=skip.data_ptr())
    st = f(x.data_ptr(), mem0.data_ptr(), ctypes.byref(cp), H, W, 15, 0, out.data_ptr())
    assert st == 0, vhlib.lib().vh_last_error().decode()
    ref = vhlib.scan_forward(x, mem0, wl.d, w_query=wq, skip=skip, dir_scale=lam, out=ref,
                             accumulate=accumulate)
    torch.cuda.synchronize()
    return out.cpu().numpy(), ref.cpu().numpy()


def test_static_scratch_near_its_limit(vhlib):
    """Nine stage-1 images, 97 % of the array: the whole scratch is usable."""
    f = _entry(vhlib)
    wl = synth.Workload("near", 9, 56, 56, 3, 32, 0, "bf16", seed=73, alpha_init=0.999)
    assert 0.95 * STATIC_LIMIT < wl.B * wl.N * wl.Cc <= STATIC_LIMIT
    got, ref = _call_both(vhlib, f, wl)
    assert parity_err(got, ref) < TOL


def test_static_scratch_accumulates(vhlib):
    f = _entry(vhlib)
    wl = synth.Workload("acc", 2, 10, 12, 2, 32, 0, "bf16", seed=74, alpha_init=0.999)
    got, ref = _call_both(vhlib, f, wl, accumulate=True)
    assert parity_err(got, ref) < TOL
