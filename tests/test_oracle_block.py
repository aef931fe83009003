"""Pins of the block oracle (oracle/vh_block.py), all on the CPU: each component against
a library routine or a closed form, and the block's wiring ("VisionHOPE: Visual
Backbones as Self-Modifying Learning Systems", Sec. 2.3 Eq. (27), App. B.5) by reducing
it to simpler forms with chosen weights."""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
scipy_signal = pytest.importorskip("scipy.signal")

from oracle import vh_block as vb  # noqa: E402
from visual_backbone_gb300 import synth  # noqa: E402


def test_bf16_rounding_matches_torch_and_ties_to_even():
    rng = np.random.default_rng(0)
    a = rng.standard_normal(10000) * np.exp(rng.uniform(-20, 20, 10000))
    want = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(vb.bf16(a), want)
    # halfway cases: 1 + 2^-8 -> 1 (even), 1 + 3 * 2^-8 -> 1 + 2^-6 (even)
    assert vb.bf16(1.0 + 2.0 ** -8) == 1.0
    assert vb.bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert vb.bf16(-(1.0 + 2.0 ** -8)) == -1.0


def test_depthwise_conv_matches_scipy_correlate():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 5, 7, 3))
    w = rng.standard_normal((3, 3, 3))
    b = rng.standard_normal(3)
    got = vb.dwconv3(x, w, b)
    for bi in range(2):
        for c in range(3):
            ref = scipy_signal.correlate2d(x[bi, :, :, c], w[c], mode="same", boundary="fill") + b[c]
            np.testing.assert_allclose(got[bi, :, :, c], ref, rtol=1e-13, atol=1e-13)


def test_layer_norm_matches_torch():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 4, 10)) * 3 + 1
    g, b = rng.standard_normal(10), rng.standard_normal(10)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (10,), torch.from_numpy(g),
                                         torch.from_numpy(b), eps=1e-5).numpy()
    np.testing.assert_allclose(vb.layer_norm(x, g, b, 1e-5), ref, rtol=1e-12, atol=1e-12)


def test_gelu_and_silu():
    assert vb.gelu(np.array(0.0)) == 0.0
    np.testing.assert_allclose(vb.gelu(np.array([1.0, -1.0])),
                               [0.8413447460685429, -0.15865525393145707], rtol=1e-15)
    a = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(vb.gelu(a), torch.nn.functional.gelu(torch.from_numpy(a)).numpy(),
                               rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(vb.silu(a), torch.nn.functional.silu(torch.from_numpy(a)).numpy(),
                               rtol=1e-14, atol=1e-15)
    # the lower tail in relative terms: Phi(-x) = phi(x) / x (1 - 1/x^2 + 3/x^4 - 15/x^6 +
    # 105/x^8 - ...), the asymptotic series of Mills' ratio (error below the first omitted term)
    for x in (10.0, 20.0):
        s = sum(c / x ** (2 * k) for k, c in enumerate([1, -1, 3, -15, 105, -945]))
        phi = math.exp(-x * x / 2) / math.sqrt(2 * math.pi) / x * s
        np.testing.assert_allclose(vb.gelu(np.array(-x)), -x * phi, rtol=1e-7)


def _setup(orc, D, Dm, d, seed, H=5, W=6, B=1):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, H, W, D))
    w = vb.weights_from(synth.make_block_weights(D, Dm, seed))
    nh = Dm // d
    mem0 = rng.standard_normal((4, nh, 4 * d * d + 2 * d)) / np.sqrt(d)
    p = orc.OracleParams(w_query=rng.standard_normal((Dm, Dm)) / np.sqrt(Dm),
                         skip=rng.standard_normal((4, Dm)),
                         dir_scale=rng.uniform(0.5, 1.5, (4, Dm)))
    return x, w, mem0, p, nh


def test_block_is_identity_without_branches(orc):
    x, w, mem0, p, nh = _setup(orc, 8, 8, 4, 3)
    w.cpe_w[:] = 0; w.cpe_b[:] = 0
    w.w_out[:] = 0; w.b_out[:] = 0
    w.w_ff2[:] = 0; w.b_ff2[:] = 0
    out = vb.block_forward(x, w, mem0, 5, 6, nh, 4, p)
    np.testing.assert_array_equal(out, x)


def test_block_ffn_branch_matches_torch_layers(orc):
    """Operator branch off: out = X0 + FFN(LN2(X0)) with X0 = X + CPE(X), the FFN built
    from torch.nn layers in fp64 (with the block's three bf16 rounding points there)."""
    x, w, mem0, p, nh = _setup(orc, 8, 8, 4, 4)
    w.w_out[:] = 0; w.b_out[:] = 0
    out = vb.block_forward(x, w, mem0, 5, 6, nh, 4, p)
    x0 = x + vb.dwconv3(x, w.cpe_w, w.cpe_b)
    t = torch.from_numpy(x0)
    ln = torch.nn.functional.layer_norm(t, (8,), torch.from_numpy(w.ln2_g),
                                        torch.from_numpy(w.ln2_b), eps=1e-5)
    a2 = torch.from_numpy(vb.bf16(ln.numpy()))
    pre = torch.nn.functional.linear(a2, torch.from_numpy(w.w_ff1))
    h = torch.nn.functional.gelu(torch.from_numpy(vb.bf16(pre.numpy())) + torch.from_numpy(w.b_ff1))
    h = torch.from_numpy(vb.bf16(h.numpy()))
    ref = t + torch.nn.functional.linear(h, torch.from_numpy(w.w_ff2), torch.from_numpy(w.b_ff2))
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_block_operator_branch_is_the_scan(orc):
    """D = D_m, Proj_in = Proj_out = I, no CPE, no depthwise branches, no FFN, plain LN1:
    out - X = bf16(F_VH(bf16(LN(X)))) with F_VH the oracle's four-route scan."""
    D = 8
    x, w, mem0, p, nh = _setup(orc, D, D, 4, 5)
    for a in (w.cpe_w, w.cpe_b, w.b_in, w.dw_w, w.dw_b, w.pos_w, w.pos_b, w.b_out, w.w_ff2,
              w.b_ff2, w.ln1_b):
        a[:] = 0
    w.ln1_g[:] = 1
    w.w_in = np.eye(D)
    w.w_out = np.eye(D)
    out = vb.block_forward(x, w, mem0, 5, 6, nh, 4, p)
    z = vb.bf16(vb.layer_norm(x, np.ones(D), np.zeros(D), 1e-5))
    y = orc.forward(z, mem0, 5, 6, nh, 4, params=p)
    np.testing.assert_allclose(out - x, vb.bf16(y), rtol=1e-12, atol=1e-12)


def test_gated_branch_and_positional_branch_enter_as_stated(orc):
    """Changing only the gated branch's bias moves Z by SiLU differences; changing only
    the positional bias adds the bias to Y before its bf16 rounding."""
    x, w, mem0, p, nh = _setup(orc, 8, 8, 4, 6)
    _, a = vb.block_forward(x, w, mem0, 5, 6, nh, 4, p, return_parts=True)
    u = a["u"]
    z_ref = vb.bf16(u + vb.silu(vb.dwconv3(u, w.dw_w, w.dw_b)))
    np.testing.assert_array_equal(a["z"], z_ref)
    np.testing.assert_array_equal(a["yb"], vb.bf16(a["y"] + vb.dwconv3(a["z"], w.pos_w, w.pos_b)))
    # the operator sees Z exactly
    y = orc.forward(a["z"], mem0, 5, 6, nh, 4, params=p)
    np.testing.assert_allclose(a["y"], y, rtol=0, atol=0)


def test_f32_mode_is_the_unrounded_block(orc):
    """round_bf16=False (the library's fp32-intermediate test mode) is the block with no
    rounding point: it differs from the rounded block, and its residual stream and FFN
    branch equal the layers written out in fp64 without rounding."""
    D, Dm, d = 32, 16, 16
    H, W = 5, 6
    x, w, mem0, p, nh = _setup(orc, D, Dm, d, seed=21)
    a = vb.block_forward(x, w, mem0, H, W, nh, d, p, round_bf16=False)
    b = vb.block_forward(x, w, mem0, H, W, nh, d, p, round_bf16=True)
    assert np.abs(a - b).max() > 0
    # the unrounded block against its parts written out without any rounding
    out, parts = vb.block_forward(x, w, mem0, H, W, nh, d, p, return_parts=True, round_bf16=False)
    x0 = x + vb.dwconv3(x, w.cpe_w, w.cpe_b)
    np.testing.assert_allclose(parts["x0"], x0, rtol=0, atol=0)
    u = vb.layer_norm(x0, w.ln1_g, w.ln1_b, w.ln_eps) @ w.w_in.T + w.b_in
    np.testing.assert_allclose(parts["u"], u, rtol=1e-13, atol=1e-13)
    x1 = parts["x1"]
    ref = x1 + vb.gelu(vb.layer_norm(x1, w.ln2_g, w.ln2_b, w.ln_eps) @ w.w_ff1.T + w.b_ff1) @ w.w_ff2.T + w.b_ff2
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
