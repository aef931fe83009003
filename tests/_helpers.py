"""Shared helpers of the test suite: running the CUDA path on synthetic
inputs, and the parity metric.

Parity metric (the pages fix none; the tolerance is 2e-3): for a tensor
of oracle values o and GPU values g,
    err = max_i |g_i - o_i| / max(|o_i|, 1e-2 * rms(o), 1e-30).
The 1e-2 * rms term keeps elements near a zero crossing from dominating; the
1e-30 absolute floor reflects that fp32 state cannot carry relative precision
once values approach its normal range (the pages' random-init workloads drive
the memories towards 1e-100 and below, where fp32 underflows to zero while the
fp64 oracle does not).
"""
import numpy as np

TOL = 2e-3


def f32(v):
    """A method constant as the C ABI carries it (fp32), widened back to fp64,
    so that the oracle runs on exactly the parameter values the GPU receives
    (with alpha_init = 0.999 the fp32 rounding of 1 - alpha_init alone moves
    the outputs by ~2e-3)."""
    return float(np.float32(v))


def oracle_params_like(orc, vhp, dir_scale=None):
    """Oracle parameters equal to a ScanParams after the fp32 round trip."""
    p = orc.OracleParams(gamma_eta=f32(vhp.gamma_eta), alpha_init=f32(vhp.alpha_init),
                         eta_bias=f32(vhp.eta_bias), eps=f32(vhp.eps),
                         knorm_eps=f32(vhp.knorm_eps), inj_inward=f32(vhp.inj_inward),
                         spec_inward=f32(vhp.spec_inward), kk_floor=f32(vhp.kk_floor),
                         gate_mode=vhp.gate_mode, forced_eta=f32(vhp.forced_eta),
                         forced_alpha=f32(vhp.forced_alpha), control_flags=vhp.control_flags)
    if dir_scale is not None:
        p.dir_scale = np.asarray(dir_scale, dtype=np.float32).astype(np.float64)
    return p


def parity_err(g, o):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    if o.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(o * o)))
    den = np.maximum(np.abs(o), max(1e-2 * rms, 1e-30))
    return float(np.max(np.abs(g - o) / den))


def to_device_x(inp, device="cuda"):
    import torch
    if inp.wl.dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(inp.x_store).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(inp.x_store))
    return t.to(device)


def run_gpu(vh, inp, params=None, dirs=15, chunk=0, dir_scale=None, want_memories=False,
            want_stats=False, impl=None):
    import torch
    wl = inp.wl
    x = to_device_x(inp)
    mem0 = torch.from_numpy(inp.mem0).cuda()
    params = params or vh.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init)
    if impl is not None:
        params.impl = impl
    ds = torch.from_numpy(dir_scale).cuda() if dir_scale is not None else None
    mo = (torch.full((x.shape[0], 4, wl.nh, 4 * wl.d * wl.d + 2 * wl.d), float("nan"),
                     device="cuda") if want_memories else None)
    st = torch.zeros(8, dtype=torch.int64, device="cuda") if want_stats else None
    out = vh.scan_forward(x, mem0, wl.d, dirs=dirs, chunk=chunk, params=params, dir_scale=ds,
                          memories_out=mo, stats=st)
    torch.cuda.synchronize()
    res = {"out": out.cpu().numpy()}
    if want_memories:
        res["mem"] = mo.cpu().numpy()
    if want_stats:
        res["stats"] = st.cpu().numpy()
    return res
