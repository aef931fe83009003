"""Pins of the oracle's VisionHOPE-exact readout ("VisionHOPE: Visual Backbones as
Self-Modifying Learning Systems", Sec. 2.1.2 Eq. (14), App. B.5): an outer query
projection shared by the four routes, normalised within each head, and a channel-wise
skip from Z_r, fused by Eq. (26)."""
import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore")


def _inputs(B=2, H=3, W=4, nh=2, d=4, seed=0):
    rng = np.random.default_rng(seed)
    Cc = nh * d
    x = rng.standard_normal((B, H, W, Cc))
    mem0 = rng.standard_normal((4, nh, 4 * d * d + 2 * d)) / np.sqrt(d)
    wq = rng.standard_normal((Cc, Cc)) / np.sqrt(Cc)
    skip = rng.standard_normal((4, Cc))
    lam = 0.5 + rng.random((4, Cc))
    return x, mem0, wq, skip, lam


def _route_pixel(r, t, H, W):
    N = H * W
    if r == 0:
        return t
    if r == 1:
        return N - 1 - t
    s = t if r == 2 else N - 1 - t
    return (s % H) * W + s // H


def test_memories_evolve_as_in_the_six_memory_form(orc):
    x, mem0, wq, skip, lam = _inputs(seed=1)
    B, H, W, Cc = x.shape
    nh, d = 2, 4
    p6 = orc.OracleParams(dir_scale=lam)
    p5 = orc.OracleParams(dir_scale=lam, w_query=wq, skip=skip)
    o6, m6 = orc.forward(x, mem0, H, W, nh, d, params=p6, want_memories=True)
    o5, m5 = orc.forward(x, mem0, H, W, nh, d, params=p5, want_memories=True)
    assert np.array_equal(m5, m6)          # the query never feeds an update
    assert not np.allclose(o5, o6)         # but the readout differs


@pytest.mark.parametrize("zero_content", [False, True])
def test_frozen_memories_closed_form(orc, zero_content):
    """alpha = 1 and an executed step of 0 freeze every memory: then
    out = sum_r lam_r * (M^m_{0,r,h} normalize_h(W_q z) + skip_r * z), per pixel."""
    x, mem0, wq, skip, lam = _inputs(seed=2)
    B, H, W, Cc = x.shape
    nh, d = 2, 4
    if zero_content:
        mem0[:, :, 3 * d * d:4 * d * d] = 0.0
    p = orc.OracleParams(dir_scale=lam, w_query=wq, skip=skip, gate_mode=2, forced_eta=0.0,
                         forced_alpha=1.0)
    out, mo = orc.forward(x, mem0, H, W, nh, d, params=p, want_memories=True)
    for b in range(B):
        np.testing.assert_array_equal(mo[b], mem0)
    z = x.reshape(B, H * W, Cc)
    q = z @ wq.T
    exp = np.zeros_like(z)
    for h in range(nh):
        qh = q[:, :, h * d:(h + 1) * d]
        qh = qh / np.sqrt((qh * qh).sum(-1, keepdims=True) + 1e-6)
        for r in range(4):
            Mm = mem0[r, h, 3 * d * d:4 * d * d].reshape(d, d)
            sl = slice(h * d, (h + 1) * d)
            exp[:, :, sl] += lam[r, sl] * (qh @ Mm.T + skip[r, sl] * z[:, :, sl])
    np.testing.assert_allclose(out.reshape(B, H * W, Cc), exp, rtol=1e-12, atol=1e-12)
    if zero_content:   # only the skip term is left
        np.testing.assert_allclose(out.reshape(B, H * W, Cc),
                                   z * (lam * skip).sum(0), rtol=1e-12, atol=1e-12)


def test_block_diagonal_projection_matches_frozen_query_memory(orc):
    """With frozen memories and every route holding the same M^q per head, the
    six-memory readout q = normalize(M^q x_h) equals the outer projection with
    W_q = blockdiag(M^q_h)."""
    x, mem0, _, _, lam = _inputs(seed=3)
    B, H, W, Cc = x.shape
    nh, d = 2, 4
    dd = d * d
    wq = np.zeros((Cc, Cc))
    for h in range(nh):
        Mq = mem0[0, h, 2 * dd:3 * dd].reshape(d, d)
        mem0[:, h, 2 * dd:3 * dd] = Mq.reshape(-1)
        wq[h * d:(h + 1) * d, h * d:(h + 1) * d] = Mq
    frozen = dict(gate_mode=2, forced_eta=0.0, forced_alpha=1.0, dir_scale=lam)
    o6 = orc.forward(x, mem0, H, W, nh, d, params=orc.OracleParams(**frozen))
    o5 = orc.forward(x, mem0, H, W, nh, d, params=orc.OracleParams(w_query=wq, **frozen))
    np.testing.assert_allclose(o5, o6, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("fwd,rev", [(0, 1), (2, 3)])
def test_reversal_symmetry_with_live_memories(orc, fwd, rev):
    """The reverse route over X equals the forward route over X rotated by 180 degrees,
    rotated back, when both routes start from the same state: the outer query is a
    per-pixel map, so it must be taken in each route's own order (a mix-up of the
    step order and the pixel order breaks the identity)."""
    x, mem0, wq, skip, _ = _inputs(B=1, H=3, W=5, nh=2, d=4, seed=4)
    _, H, W, Cc = x.shape
    mem0[rev] = mem0[fwd]
    skip[rev] = skip[fwd]
    p = orc.OracleParams(w_query=wq, skip=skip, alpha_init=0.999)
    a = orc.forward(x, mem0, H, W, 2, 4, dirs=1 << rev, params=p)
    b = orc.forward(x[:, ::-1, ::-1].copy(), mem0, H, W, 2, 4, dirs=1 << fwd, params=p)
    np.testing.assert_array_equal(a, b[:, ::-1, ::-1])
    assert np.abs(a).max() > 1e-3


def test_token_indexed_mode_is_six_memory_only(orc):
    x, mem0, wq, _, _ = _inputs(B=1, seed=5)
    with pytest.raises(RuntimeError):
        orc.forward(x, mem0, 3, 4, 2, 4, params=orc.OracleParams(w_query=wq),
                    token_indexed_mode=True)
