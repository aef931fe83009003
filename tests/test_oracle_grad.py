"""Pins of the gradient oracle (oracle/vh_grad.py), all on the CPU.

The outer gradients of the VisionHOPE scan ("VisionHOPE: Visual Backbones as
Self-Modifying Learning Systems", Sec. 2.1.2: the recurrence is explicit and
differentiable) are checked against things other than the autograd they come from:
  * the PyTorch restatement of the forward equals the C oracle's forward;
  * directional derivatives equal central finite differences of the C oracle;
  * with alpha = 1 and a zero executed step no memory moves, and the gradient has the
    closed form of y_t = M^m_0 normalize(M^q_0 x_t), summed over the routes.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import vh_grad  # noqa: E402
from visual_backbone_gb300 import synth  # noqa: E402


def _case(seed, B, H, W, nh, d, scale_x=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, H, W, nh * d)) * scale_x
    mem0 = rng.standard_normal((4, nh, 4 * d * d + 2 * d)) / np.sqrt(d)
    return rng, x, mem0


CASES = [
    # name, seed, (B, H, W, nh, d), dirs, chunk, params
    ("aligned", 1, (2, 3, 4, 2, 4), 15, 0, {}),
    ("chunk5_ragged", 2, (1, 4, 3, 1, 6), 15, 5, {}),
    ("softcap", 3, (1, 3, 3, 1, 4), 5, 0, {"eta_bias": 4.0}),
    ("lowalpha", 4, (1, 3, 4, 1, 4), 10, 0, {"alpha_init": 0.3, "eta_bias": 2.0}),
    ("spectral", 7, (1, 3, 4, 1, 4), 15, 0, {"alpha_init": 0.05, "eta_bias": 3.0}),
    ("forced_raw", 5, (1, 3, 3, 1, 4), 15, 0, {"gate_mode": 1, "forced_eta": 0.3,
                                               "forced_alpha": 0.8}),
    ("forced_exec", 6, (1, 3, 3, 1, 4), 15, 2, {"gate_mode": 2, "forced_eta": 0.2,
                                                "forced_alpha": 0.7}),
]


def _params(orc, kw, nh, d, rng=None, lam=False):
    p = orc.OracleParams(**kw)
    if lam:
        p.dir_scale = rng.uniform(0.5, 1.5, size=(4, nh * d))
    return p


@pytest.mark.parametrize("name,seed,shape,dirs,chunk,kw", CASES, ids=[c[0] for c in CASES])
def test_torch_forward_equals_c_oracle(orc, name, seed, shape, dirs, chunk, kw):
    B, H, W, nh, d = shape
    rng, x, mem0 = _case(seed, *shape)
    p = _params(orc, kw, nh, d, rng, lam=True)
    o, om = orc.forward(x, mem0, H, W, nh, d, dirs=dirs, chunk_len=chunk, params=p,
                        want_memories=True)
    t, tm = vh_grad.forward_torch(torch.from_numpy(x), torch.from_numpy(mem0), H, W, nh, d,
                                  dirs, chunk, p)
    np.testing.assert_allclose(t.numpy(), o, rtol=1e-11, atol=1e-12)
    sel = [r for r in range(4) if dirs & (1 << r)]
    np.testing.assert_allclose(tm.numpy()[:, sel], om[:, sel], rtol=1e-11, atol=1e-12)


def test_spectral_case_hits_the_clamp(orc):
    """The "spectral" case above executes the spectral limit on some tokens (its
    gradient path through alpha is then covered by the finite differences)."""
    _, x, mem0 = _case(7, 1, 3, 4, 1, 4)
    p = orc.OracleParams(alpha_init=0.05, eta_bias=3.0)
    f = orc.diag_fields(4)
    _, _, diag = orc.chunk(mem0[0, 0], x[0, 0, :, :4], p)
    assert (diag[:, f["eta_spec"]] < diag[:, f["eta_bar"]]).any()
    assert (diag[:, f["eta_spec"]] > diag[:, f["eta_bar"]]).any()


def test_route_orders_match_c_oracle(orc):
    for H, W in [(3, 4), (5, 2), (1, 7)]:
        for r in range(4):
            np.testing.assert_array_equal(vh_grad._route_order(r, H, W), orc.route_order(r, H, W))


def _loss_c(orc, x, mem0, dout, dmf, H, W, nh, d, dirs, chunk, p):
    o, om = orc.forward(x, mem0, H, W, nh, d, dirs=dirs, chunk_len=chunk, params=p,
                        want_memories=True)
    sel = [r for r in range(4) if dirs & (1 << r)]
    return float((o * dout).sum() + (om[:, sel] * dmf[:, sel]).sum())


@pytest.mark.parametrize("name,seed,shape,dirs,chunk,kw", CASES, ids=[c[0] for c in CASES])
def test_gradient_matches_finite_differences(orc, name, seed, shape, dirs, chunk, kw):
    """<grad, v> against (L(theta + h v) - L(theta - h v)) / 2h of the C oracle."""
    B, H, W, nh, d = shape
    rng, x, mem0 = _case(seed, *shape)
    p = _params(orc, kw, nh, d, rng, lam=True)
    dout = rng.standard_normal((B, H, W, nh * d))
    dmf = rng.standard_normal((B, 4, nh, 4 * d * d + 2 * d)) * 0.5
    gx, gm = vh_grad.backward(x, mem0, dout, H, W, nh, d, dirs, chunk, p, dmem_final=dmf)
    h = 1e-6
    for trial in range(3):
        vx = rng.standard_normal(x.shape)
        vm = rng.standard_normal(mem0.shape)
        for which in ("x", "mem"):
            if which == "x":
                lp = _loss_c(orc, x + h * vx, mem0, dout, dmf, H, W, nh, d, dirs, chunk, p)
                lm = _loss_c(orc, x - h * vx, mem0, dout, dmf, H, W, nh, d, dirs, chunk, p)
                want = (gx * vx).sum()
            else:
                lp = _loss_c(orc, x, mem0 + h * vm, dout, dmf, H, W, nh, d, dirs, chunk, p)
                lm = _loss_c(orc, x, mem0 - h * vm, dout, dmf, H, W, nh, d, dirs, chunk, p)
                want = (gm * vm).sum()
            fd = (lp - lm) / (2 * h)
            assert abs(fd - want) <= 1e-6 * max(1.0, abs(want)), (which, trial, fd, want)


def test_gradient_closed_form_without_steps(orc):
    """alpha = 1, executed step 0 (forced): no memory moves, out = sum_r lambda_r M^m_r q_r(x)
    with q_r = n(M^q_r x), n(u) = u / sqrt(|u|^2 + 1e-6); so
    dx = sum_r M^q_r^T J_r^T M^m_r^T (lambda_r dout),  J = (I - q q^T) / |u|_eps,
    dM^m_r = sum_{b,p} (lambda_r dout) q^T,  dM^q_r = sum J^T M^m^T (lambda_r dout) x^T,
    and the k, v, eta, alpha memories get nothing from out."""
    rng, x, mem0 = _case(11, 2, 3, 4, 2, 5)
    B, H, W, nh, d = 2, 3, 4, 2, 5
    lam = rng.uniform(0.5, 1.5, size=(4, nh * d))
    p = orc.OracleParams(gate_mode=2, forced_eta=0.0, forced_alpha=1.0, dir_scale=lam)
    dout = rng.standard_normal((B, H, W, nh * d))
    gx, gm = vh_grad.backward(x, mem0, dout, H, W, nh, d, 15, 0, p)
    dd = d * d
    ex = np.zeros_like(x)
    em = np.zeros_like(mem0)
    for r in range(4):
        for h in range(nh):
            Mq = mem0[r, h, 2 * dd:3 * dd].reshape(d, d)
            Mm = mem0[r, h, 3 * dd:4 * dd].reshape(d, d)
            for b in range(B):
                for i in range(H):
                    for j in range(W):
                        xv = x[b, i, j, h * d:(h + 1) * d]
                        u = Mq @ xv
                        n = np.sqrt(u @ u + 1e-6)
                        q = u / n
                        gy = lam[r, h * d:(h + 1) * d] * dout[b, i, j, h * d:(h + 1) * d]
                        gq = Mm.T @ gy
                        gu = (gq - q * (q @ gq)) / n
                        ex[b, i, j, h * d:(h + 1) * d] += Mq.T @ gu
                        em[r, h, 3 * dd:4 * dd] += np.outer(gy, q).ravel()
                        em[r, h, 2 * dd:3 * dd] += np.outer(gu, xv).ravel()
    np.testing.assert_allclose(gx, ex, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gm, em, rtol=1e-10, atol=1e-12)


def test_disabled_routes_get_zero_gradient(orc):
    rng, x, mem0 = _case(12, 1, 3, 3, 1, 4)
    dout = rng.standard_normal(x.shape)
    _, gm = vh_grad.backward(x, mem0, dout, 3, 3, 1, 4, dirs=6)
    assert not gm[[0, 3]].any()
    assert np.abs(gm[[1, 2]]).max() > 0


def test_bf16_inputs_and_synthetic_recipe(orc):
    """The synthetic bf16 workload inputs go through unchanged (values already exact)."""
    wl = synth.Workload("g", 1, 4, 5, 1, 8, 0, "bf16", seed=13)
    inp = synth.make_inputs(wl)
    dout = np.random.default_rng(14).standard_normal(inp.x64.shape)
    gx, gm = vh_grad.backward(inp.x64, inp.mem0.astype(np.float64), dout, 4, 5, 1, 8)
    assert np.isfinite(gx).all() and np.isfinite(gm).all()
    assert gx.shape == inp.x64.shape and gm.shape == inp.mem0.shape
