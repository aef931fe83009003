"""Cases run through the checked-index library (libvh_dbg.so, VH_DEBUG_BOUNDS).

Run as a child process with VH_DEBUG_BOUNDS=1 in its environment (the binding then loads
libvh_dbg.so); prints one JSON line per case: the failed index checks it counted and its
parity error against the oracle."""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

# name, (B, H, W, nh, d, chunk, dtype), kwargs of the call
CASES = [
    ("tc32-8x8", (2, 8, 8, 1, 32, 0, "bf16"), {"impl": "tc"}),
    ("tc32-3x4", (1, 3, 4, 2, 32, 0, "bf16"), {"impl": "tc"}),
    ("tc32-70x5", (1, 70, 5, 1, 32, 0, "bf16"), {"impl": "tc"}),
    ("tc32-wy", (2, 9, 14, 2, 32, 0, "bf16"), {"impl": "tc_wy"}),
    ("tc32-pipe", (1, 6, 131, 1, 32, 0, "bf16"), {"impl": "tc_pipe"}),
    ("tc32-pipe-cols", (1, 70, 5, 1, 32, 0, "bf16"), {"impl": "tc_pipe"}),
    ("tc32-exact", (2, 7, 12, 2, 32, 0, "bf16"), {"impl": "tc", "exact": True}),
    ("tc64-14x14", (2, 14, 14, 1, 64, 0, "bf16"), {"impl": "tc"}),
    ("tc64-3x40", (1, 3, 40, 1, 64, 0, "bf16"), {"impl": "tc"}),
    ("simt-d16-chunk1", (1, 8, 8, 2, 16, 1, "f32"), {"impl": "simt"}),
    ("simt-d32-chunk7", (1, 5, 9, 1, 32, 7, "f32"), {"impl": "simt"}),
    ("simt-d64", (1, 6, 7, 1, 64, 0, "bf16"), {"impl": "simt"}),
    ("simt-exact", (1, 5, 6, 2, 16, 0, "f32"), {"impl": "simt", "exact": True}),
    ("backward-d16", (1, 6, 5, 2, 16, 0, "f32"), {"impl": "simt", "backward": True}),
    ("backward-tc32", (1, 8, 6, 1, 32, 0, "bf16"), {"impl": "auto", "backward": True}),
]


def run_case(vh, orc, name, shape, kw):
    import torch
    from visual_backbone_gb300 import synth
    from tests._helpers import oracle_params_like, parity_err, to_device_x
    B, H, W, nh, d, chunk, dtype = shape
    wl = synth.Workload(name, B, H, W, nh, d, chunk, dtype, seed=H * 31 + W, alpha_init=0.999)
    inp = synth.make_inputs(wl)
    x = to_device_x(inp)
    m = torch.from_numpy(inp.mem0).cuda()
    st = torch.zeros(8, dtype=torch.int64, device="cuda")
    p = vh.ScanParams(alpha_init=wl.alpha_init, impl=kw["impl"])
    extra, oextra = {}, {}
    if kw.get("exact"):
        g = torch.Generator().manual_seed(5)
        wq = torch.randn(wl.Cc, wl.Cc, generator=g) / wl.Cc ** 0.5
        extra = {"w_query": wq.cuda()}
        oextra = {"w_query": wq.double().numpy()}
    if kw.get("backward"):
        dout = torch.from_numpy(np.random.default_rng(3).standard_normal(
            (B, H, W, wl.Cc)).astype(np.float32)).cuda()
        dx, dm = vh.scan_backward(x, m, d, dout, chunk=chunk, params=p, stats=st)
        torch.cuda.synchronize()
        from oracle import vh_grad
        op = oracle_params_like(orc, p)
        rdx, rdm = vh_grad.backward(inp.x64, inp.mem0.astype(np.float64), dout.double().cpu().numpy(),
                                    H, W, nh, d, chunk_len=chunk, params=op)
        err = max(parity_err(dx.cpu().numpy(), rdx), parity_err(dm.cpu().numpy(), rdm))
    else:
        out = vh.scan_forward(x, m, d, chunk=chunk, params=p, stats=st, **extra)
        torch.cuda.synchronize()
        op = oracle_params_like(orc, p)
        for k, v in oextra.items():
            setattr(op, k, v)
        ref = orc.forward(inp.x64, inp.mem0, H, W, nh, d, chunk_len=chunk, params=op)
        err = parity_err(out.cpu().numpy(), ref)
    return {"name": name, "bounds": int(st[5].item()), "timeout": int(st[4].item()), "err": float(err)}


def main():
    import oracle as orc
    import visual_backbone_gb300 as vh
    orc.build()
    assert vh.lib().vh_debug_bounds_build() == 1, "not the checked-index library"
    for name, shape, kw in CASES:
        print(json.dumps(run_case(vh, orc, name, shape, kw)), flush=True)


if __name__ == "__main__":
    main()
