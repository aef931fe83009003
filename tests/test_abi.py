"""The C ABI on the host: the library loads, exports every declared
function, and rejects bad arguments before touching a device (no GPU needed)."""
import ctypes

import pytest


def test_exports_every_header_function(vhlib):
    names = vhlib.header_functions()
    assert {"vh_scan_forward", "vh_debug_permute", "vh_workspace_size", "vh_status_string",
            "vh_last_error", "vh_params_init", "vh_version", "vh_check"} <= set(names)
    L = vhlib.lib()
    for n in names:
        assert hasattr(L, n), n


def test_params_init_defaults(vhlib):
    p = vhlib.CParams()
    vhlib.lib().vh_params_init(ctypes.byref(p))
    assert abs(p.gamma_eta - 0.025) < 1e-9 and abs(p.alpha_init - 0.9) < 1e-7
    assert p.eps == pytest.approx(1e-6) and p.knorm_eps == pytest.approx(1e-6)
    assert p.inj_inward == pytest.approx(1e-3) and p.spec_inward == pytest.approx(1e-6)
    assert p.kk_floor == pytest.approx(1e-20)
    assert p.x_dtype == vhlib.DTYPE_BF16 and p.accumulate == 0 and p.stats is None


def test_status_strings_and_version(vhlib):
    L = vhlib.lib()
    assert L.vh_status_string(0) == b"ok"
    assert L.vh_status_string(-1) == b"invalid argument"
    assert L.vh_version() >= 100
    assert L.vh_workspace_size(None, 8, 8, 15, 0) == 0


FAKE = 0x10000  # a 16-byte aligned address that is never dereferenced


def _call(vhlib, B=1, Cc=32, d=32, H=4, W=4, dirs=15, chunk=0, x=FAKE, mem=FAKE,
          out=FAKE * 4096, **kw):
    p = vhlib.make_cparams(B, Cc, d, True)
    for k, v in kw.items():
        setattr(p, k, v)
    st = vhlib.lib().vh_scan_forward(x, mem, ctypes.byref(p), H, W, dirs, chunk, out)
    return st, vhlib.lib().vh_last_error().decode()


@pytest.mark.parametrize("kw,status", [
    (dict(dirs=0), -1), (dict(dirs=16), -1), (dict(chunk=-1), -1), (dict(H=0), -1),
    (dict(B=0), -1), (dict(d=48, Cc=96), -2), (dict(Cc=40), -1), (dict(x=FAKE + 8), -1),
    (dict(out=FAKE + 4), -1), (dict(x=0), -1), (dict(out=FAKE), -1),
    (dict(gate_mode=3), -1), (dict(alpha_init=1.0), -1), (dict(impl=7), -1),
    (dict(x_dtype=5), -2), (dict(wait_limit=-5), -1),
    # the withheld-copy hook belongs to the head_dim 32 tensor-core kernel only
    (dict(withhold_first_copy=1, d=16), -1), (dict(withhold_first_copy=1, impl=1), -1),
    (dict(withhold_first_copy=1, chunk=3), -1), (dict(withhold_first_copy=1, x_dtype=0), -1),
])
def test_bad_arguments_are_rejected_on_the_host(vhlib, kw, status):
    st, msg = _call(vhlib, **kw)
    assert st == status and msg


def test_debug_permute_rejects_bad_route(vhlib):
    p = vhlib.make_cparams(1, 16, 16, False)
    assert vhlib.lib().vh_debug_permute(FAKE, ctypes.byref(p), 3, 4, 4, FAKE * 64) == -1


def test_workspace_is_sized_and_required(vhlib):
    L = vhlib.lib()
    p = vhlib.make_cparams(2, 64, 32, True)
    assert L.vh_workspace_size(ctypes.byref(p), 5, 7, 15, 0) == 0
    p.w_query = FAKE
    assert L.vh_workspace_size(ctypes.byref(p), 5, 7, 15, 0) == 6 * 2 * 5 * 7 * 64
    st, msg = _call(vhlib, B=2, Cc=64, d=32, H=5, W=7, w_query=FAKE)
    assert st == -4 and "workspace" in msg
    st, _ = _call(vhlib, B=2, Cc=64, d=32, H=5, W=7, w_query=FAKE, workspace=FAKE * 16,
                  workspace_bytes=100)
    assert st == -4
    st, _ = _call(vhlib, B=2, Cc=64, d=32, H=5, W=7, w_query=FAKE, workspace=FAKE * 16 + 8,
                  workspace_bytes=1 << 20)
    assert st == -4
    st, msg = _call(vhlib, B=2, Cc=64, d=32, H=5, W=7, w_query=FAKE, workspace=FAKE,
                    workspace_bytes=1 << 20)
    assert st == -1 and "alias" in msg


def test_check_rejects_null_stats(vhlib):
    L = vhlib.lib()
    assert L.vh_check(None, None) == -1
    assert b"stats" in L.vh_last_error()


def test_binding_refuses_cpu_tensors(vhlib):
    import torch
    x = torch.zeros(1, 4, 4, 16)
    m = torch.zeros(4, 1, 4 * 256 + 32)
    with pytest.raises(ValueError, match="CUDA"):
        vhlib.scan_forward(x, m, 16)
    with pytest.raises(ValueError, match="CUDA"):
        vhlib.check(torch.zeros(8, dtype=torch.int64))


def _bwd_call(vhlib, B=1, Cc=32, d=32, H=4, W=4, dirs=15, chunk=0, ws=0, ws_bytes=0, **kw):
    p = vhlib.make_cparams(B, Cc, d, True, workspace_ptr=ws, workspace_bytes=ws_bytes)
    for k, v in kw.items():
        setattr(p, k, v)
    base = 1 << 36  # far-apart, 16-byte aligned fake device addresses, never dereferenced
    return vhlib.lib().vh_scan_backward(base, base + (1 << 30), ctypes.byref(p), H, W, dirs,
                                        chunk, base + (2 << 30), None, base + (3 << 30),
                                        base + (4 << 30))


def test_backward_workspace_size(vhlib):
    """Per scan: the boundary states of its chunks (4d^2 + 2d floats each) plus, for the
    longest chunk, a d^2 gain slice per four tokens and 4d + 24 floats per token (token
    record, gain record).  Where the tensor-core forward runs the pre-pass (d = 32, bf16 x,
    aligned chunks, impl not SIMT) it also writes a 3d + 8 float record for every token of
    every scan."""
    L = vhlib.lib()
    p = vhlib.make_cparams(2, 64, 32, True)

    def chunk_floats(lmax):
        return (lmax + 3) // 4 * 32 * 32 + lmax * (4 * 32 + 24)
    trec = 15 * (3 * 32 + 8)
    # 3 x 5 map, all routes, aligned chunks: rows of 5 (3 chunks), columns of 3 (5 chunks)
    per_scan = 5 * (4 * 32 * 32 + 64) + chunk_floats(5)
    assert L.vh_backward_workspace_size(ctypes.byref(p), 3, 5, 15, 0) == 2 * 4 * 2 * (per_scan + trec) * 4
    # rows only: 3 chunks of 5
    per_scan = 3 * (4 * 32 * 32 + 64) + chunk_floats(5)
    assert L.vh_backward_workspace_size(ctypes.byref(p), 3, 5, 3, 0) == 2 * 2 * 2 * (per_scan + trec) * 4
    # fixed chunk 4 over 15 tokens: 4 chunks, the longest 4 tokens; no token records
    per_scan = 4 * (4 * 32 * 32 + 64) + chunk_floats(4)
    assert L.vh_backward_workspace_size(ctypes.byref(p), 3, 5, 1, 4) == 2 * 1 * 2 * per_scan * 4
    # the CUDA-core implementation forced: no token records
    ps = vhlib.make_cparams(2, 64, 32, True, vhlib.ScanParams(impl="simt"))
    per_scan = 3 * (4 * 32 * 32 + 64) + chunk_floats(5)
    assert L.vh_backward_workspace_size(ctypes.byref(ps), 3, 5, 3, 0) == 2 * 2 * 2 * per_scan * 4
    assert L.vh_backward_workspace_size(None, 3, 5, 15, 0) == 0
    assert L.vh_backward_workspace_size(ctypes.byref(p), 3, 5, 0, 0) == 0


def test_backward_rejects_on_the_host(vhlib):
    big = 1 << 40
    assert _bwd_call(vhlib, control_flags=vhlib.CTRL_NO_DGD) == -2      # unsupported
    assert _bwd_call(vhlib, w_query=1 << 20) == -2
    assert _bwd_call(vhlib) == -4                                       # no workspace
    assert _bwd_call(vhlib, ws=big + 8, ws_bytes=1 << 30) == -4         # misaligned
    assert _bwd_call(vhlib, ws=big, ws_bytes=16) == -4                  # too small
    assert _bwd_call(vhlib, dirs=0, ws=big, ws_bytes=1 << 30) == -1
    assert _bwd_call(vhlib, d=24, Cc=48, ws=big, ws_bytes=1 << 30) == -2
    # workspace overlapping dx
    assert _bwd_call(vhlib, ws=(1 << 36) + (3 << 30), ws_bytes=1 << 30) == -1
    assert b"overlap" in vhlib.lib().vh_last_error()
    # dx overlapping dout
    p = vhlib.make_cparams(1, 32, 32, True, workspace_ptr=1 << 40, workspace_bytes=1 << 30)
    base = 1 << 36
    assert vhlib.lib().vh_scan_backward(base, base + (1 << 30), ctypes.byref(p), 4, 4, 15, 0,
                                        base + (2 << 30), None, base + (2 << 30),
                                        base + (4 << 30)) == -1
    assert b"alias" in vhlib.lib().vh_last_error()


def test_debug_gelu_rejects_bad_args(vhlib):
    L = vhlib.lib()
    assert L.vh_debug_gelu(FAKE, FAKE, -1, None) == -1
    assert L.vh_debug_gelu(None, FAKE, 8, None) == -1
    assert L.vh_debug_gelu(FAKE, None, 8, None) == -1
    assert L.vh_debug_gelu(None, None, 0, None) == 0   # nothing to do, nothing launched
