"""The VisionHOPE block on the GPU (vh_block_forward) against the block oracle
("VisionHOPE: Visual Backbones as Self-Modifying Learning Systems", Sec. 2.3 Eq. (27),
App. B.5), on the same seeded inputs and weights.

Tolerance.  Both sides round the same six intermediates to bf16 (LN1 and LN2 outputs,
Z, Y before Proj_out, FFN1's product before its bias, GELU output).  An intermediate within fp32 noise of a rounding
boundary lands one bf16 step (2^-8 of its value) apart; a step at LN2's output (|a| of
a few units) moves every channel of that pixel through the FFN by up to a few 1e-3 of the
output's rms.  Everywhere else the two agree to fp32 (about 1e-7 of the rms).  So the
test is two-sided, on e = |g - o| / rms(o):
  * the 90th percentile of e below P90_TOL = 1e-5: a wrong term, sign or index moves
    most elements and fails here;
  * the maximum of e below MAX_TOL = 2e-2, and fewer than 10 % of the pixels above 1e-4:
    the rounding-boundary steps stay isolated and bounded.
"""
import numpy as np
import pytest


P90_TOL, MAX_TOL = 1e-5, 2e-2


def block_err(g, o):
    """(90th percentile, maximum, share of pixels above 1e-4) of |g - o| / rms(o)."""
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    e = np.abs(g - o) / np.sqrt(np.mean(o * o))
    return float(np.percentile(e, 90)), float(e.max()), float(np.mean(e.reshape(-1, o.shape[-1]).max(1) > 1e-4))


def assert_block_close(g, o, what=""):
    p90, mx, frac = block_err(g, o)
    assert p90 < P90_TOL and mx < MAX_TOL and frac < 0.10, (what, p90, mx, frac)


pytestmark = pytest.mark.gpu


def _make(seed, B, H, W, D, Dm, d):
    import torch
    from oracle import vh_block as vb
    from visual_backbone_gb300 import synth
    inp = synth.make_block_inputs(B, H, W, D, Dm, d, seed)
    wt = vb.weights_from(inp["weights"])  # the oracle sees the values the GPU gets
    gpu = {}
    for f, a in inp["weights"].items():
        t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
        gpu[f] = t.to(torch.bfloat16) if f in synth.BLOCK_GEMM_WEIGHTS else t
    return (inp["x"], wt, gpu, inp["mem0"], inp["w_query"], inp["skip"], inp["dir_scale"],
            inp["nh"])


def _gpu(vhlib, x, gpu, mem0, wq, skip, lam, d, f32=False):
    import torch
    st = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = vhlib.block_forward(torch.from_numpy(x).cuda(), torch.from_numpy(mem0).cuda(), gpu, d,
                              w_query=torch.from_numpy(wq).cuda(),
                              skip=torch.from_numpy(skip).cuda(),
                              dir_scale=torch.from_numpy(lam).cuda(), stats=st,
                              f32_intermediates=f32)
    torch.cuda.synchronize()
    vhlib.check(st)
    return out.cpu().numpy()


def _oracle(orc, x, wt, mem0, wq, skip, lam, H, W, nh, d, round_bf16=True):
    from oracle import vh_block as vb
    p = orc.OracleParams(alpha_init=float(np.float32(0.9)), gamma_eta=float(np.float32(0.025)),
                         w_query=wq.astype(np.float64), skip=skip.astype(np.float64),
                         dir_scale=lam.astype(np.float64))
    return vb.block_forward(x.astype(np.float64), wt, mem0.astype(np.float64), H, W, nh, d, p,
                            round_bf16=round_bf16)


CASES = [
    # name, seed, B, H, W, D, D_m, d
    ("5x6_D64_Dm32_d32", 1, 1, 5, 6, 64, 32, 32),
    ("7x9_D64_Dm64_d32", 2, 2, 7, 9, 64, 64, 32),
    ("6x5_D32_Dm16_d16", 3, 1, 6, 5, 32, 16, 16),
    ("8x8_D128_Dm64_d16", 4, 1, 8, 8, 128, 64, 16),
    ("3x70_D64_Dm32_d32", 5, 1, 3, 70, 64, 32, 32),
    ("1x9_D32_Dm16_d16", 6, 2, 1, 9, 32, 16, 16),     # one-row map: the depthwise edges
    ("9x1_D64_Dm32_d32", 8, 1, 9, 1, 64, 32, 32),     # one-column map
    ("4x5_D256_Dm64_d32", 9, 1, 4, 5, 256, 64, 32),   # N tiles of 192 / 256 (hidden 1024)
    ("6x7_D192_Dm96_d32", 10, 2, 6, 7, 192, 96, 32),  # the stage-1 widths
]


@pytest.mark.parametrize("name,seed,B,H,W,D,Dm,d", CASES, ids=[c[0] for c in CASES])
def test_block_parity(orc, vhlib, name, seed, B, H, W, D, Dm, d):
    x, wt, gpu, mem0, wq, skip, lam, nh = _make(seed, B, H, W, D, Dm, d)
    g = _gpu(vhlib, x, gpu, mem0, wq, skip, lam, d)
    o = _oracle(orc, x, wt, mem0, wq, skip, lam, H, W, nh, d)
    assert_block_close(g, o, name)


def test_block_stage1_sampled(orc, vhlib):
    """The stage-1 block (B = 32, 56 x 56, D = 192, D_m = 96 as 3 heads of 32) in the
    launch the block bench times; the first and last image against the oracle."""
    B, H, W, D, Dm, d = 32, 56, 56, 192, 96, 32
    x, wt, gpu, mem0, wq, skip, lam, nh = _make(7, B, H, W, D, Dm, d)
    g = _gpu(vhlib, x, gpu, mem0, wq, skip, lam, d)
    for b in (0, B - 1):
        o = _oracle(orc, x[b:b + 1], wt, mem0, wq, skip, lam, H, W, nh, d)
        assert_block_close(g[b:b + 1], o, b)


def test_block_rejects_on_the_host(vhlib):
    import torch
    x = torch.zeros((1, 4, 4, 12), device="cuda")
    gpu = {k: torch.zeros(1, device="cuda") for k in
           ("cpe_w", "cpe_b", "ln1_g", "ln1_b", "b_in", "dw_w", "dw_b", "pos_w", "pos_b", "b_out",
            "ln2_g", "ln2_b", "b_ff1", "b_ff2")}
    for k in ("w_in", "w_out", "w_ff1", "w_ff2"):
        gpu[k] = torch.zeros((16, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(vhlib.VhError, match="dim 12"):
        vhlib.block_forward(x, torch.zeros(4 * 16 * 16 + 32, device="cuda"), gpu, 16)


# ---------------------------------------------------------- fp32-intermediate test mode
#
# With w->f32_intermediates the library rounds no intermediate to bf16: the GEMMs take each
# fp32 activation as three bf16 pieces against the weights tripled along K, GELU acts on
# the unrounded product, and the operator scans fp32 Z.  The oracle drops its rounding
# points as well, so no bf16 boundary can split the two, and every element is held to the
# scan's tolerance: max |g - o| / max(|o|, 1e-2 rms(o)) < 2e-3.

@pytest.mark.parametrize("name,seed,B,H,W,D,Dm,d", CASES, ids=[c[0] for c in CASES])
def test_block_f32_intermediates_elementwise(orc, vhlib, name, seed, B, H, W, D, Dm, d):
    from tests._helpers import TOL, parity_err
    x, wt, gpu, mem0, wq, skip, lam, nh = _make(seed, B, H, W, D, Dm, d)
    g = _gpu(vhlib, x, gpu, mem0, wq, skip, lam, d, f32=True)
    o = _oracle(orc, x, wt, mem0, wq, skip, lam, H, W, nh, d, round_bf16=False)
    err = parity_err(g, o)
    assert err < TOL, (name, err)


def test_block_f32_intermediates_stage1_sampled(orc, vhlib):
    """The stage-1 widths and map in the test mode; the first and last image."""
    from tests._helpers import TOL, parity_err
    B, H, W, D, Dm, d = 4, 56, 56, 192, 96, 32
    x, wt, gpu, mem0, wq, skip, lam, nh = _make(11, B, H, W, D, Dm, d)
    g = _gpu(vhlib, x, gpu, mem0, wq, skip, lam, d, f32=True)
    for b in (0, B - 1):
        o = _oracle(orc, x[b:b + 1], wt, mem0, wq, skip, lam, H, W, nh, d, round_bf16=False)
        err = parity_err(g[b:b + 1], o)
        assert err < TOL, (b, err)


def test_block_modes_differ_only_by_rounding(orc, vhlib):
    """The two modes on the same inputs: apart by bf16 rounding (about 2^-8 of a value at
    most), so a mode that dropped or misplaced a term would stand out."""
    x, wt, gpu, mem0, wq, skip, lam, nh = _make(12, 1, 6, 7, 64, 32, 32)
    g16 = _gpu(vhlib, x, gpu, mem0, wq, skip, lam, 32)
    g32 = _gpu(vhlib, x, gpu, mem0, wq, skip, lam, 32, f32=True)
    rel = np.abs(g16 - g32).max() / np.sqrt(np.mean(g32.astype(np.float64) ** 2))
    assert 0 < rel < 0.1, rel
