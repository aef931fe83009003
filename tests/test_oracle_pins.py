"""Pins of the fp64 oracle against what the pages and the mathematics fix.

No test here compares the oracle with itself or with a retyped copy of its
own formula: each one checks it against a printed value, a closed form, an
independent formulation of the same step, or an invariant the pages prove.
"""
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_kv(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, v = line.split(None, 1) if ":" not in line else [s.strip() for s in line.split(":", 1)]
        out[k] = v
    return out


def _rand_state(rng, d, scale=None):
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    return rng.standard_normal(4 * d * d + 2 * d) * scale


# ---------------------------------------------------------------- routes

def test_route_orders_match_printed_3x4(orc):
    """VMamba explainer: printed row/column, forward/reverse orders of a 3x4 grid."""
    g = _golden_kv("cross_scan_3x4.txt")
    names = {0: "row_forward", 1: "row_reverse", 2: "column_forward", 3: "column_reverse"}
    for r, name in names.items():
        want = [int(v) for v in g[name].split()]
        assert orc.route_order(r, 3, 4).tolist() == want, name


@pytest.mark.parametrize("H,W", [(1, 1), (1, 7), (5, 1), (3, 4), (5, 7), (8, 8), (6, 9)])
def test_routes_are_transpose_flatten_and_flip(orc, H, W):
    """Column route = transpose then flatten; reverse routes flip the whole
    sequence; inverse of the column stream = reshape W x H, transpose back."""
    grid = np.arange(H * W).reshape(H, W)
    row = grid.flatten()
    col = grid.T.flatten()
    assert orc.route_order(0, H, W).tolist() == row.tolist()
    assert orc.route_order(1, H, W).tolist() == row[::-1].tolist()
    assert orc.route_order(2, H, W).tolist() == col.tolist()
    assert orc.route_order(3, H, W).tolist() == col[::-1].tolist()
    # rectangle inverse from the explainer's cross-merge section
    assert (orc.route_order(2, H, W).reshape(W, H).T == grid).all()


# ------------------------------------------------------ printed values

def test_worked_scalar_recurrence_as_d1_instance(orc):
    """0.5*2 + 0.2*3 = 1.6 (VMamba explainer) realised by one SR-DGD step with
    d = 1: k ~ 1 (M^k = 1000, x = 1), v = 2.5 so delta = -1.5, forced
    alpha = 0.7 and executed step 0.2 give A = 0.5 and M_b B = 0.2 * 3 on a
    content memory of 2."""
    g = _golden_kv("worked_recurrence.txt")
    h0, a, u, bcoef, want = (float(g[k]) for k in
                             ("previous_state", "retention", "input", "input_coefficient",
                              "next_state"))
    d = 1
    S = np.zeros(4 * d * d + 2 * d)
    S[0] = 1000.0   # M^k
    S[1] = 2.5      # M^v
    S[2] = 1000.0   # M^q (q ~ 1 after normalisation)
    S[3] = h0       # M^m (content)
    eta_t = bcoef
    alpha = a + eta_t * 1.0   # A = alpha - eta_t * k^2 with k ~ 1  ->  0.7
    p = orc.OracleParams(gate_mode=2, forced_eta=eta_t, forced_alpha=alpha)
    S1, y, diag = orc.chunk(S, np.array([[1.0]]), p)
    f = orc.diag_fields(d)
    assert abs(diag[0, f["k"]][0] - 1.0) < 1e-9
    assert abs(-diag[0, f["delta"]][0] * h0 - u) < 1e-9   # injected input M_b (-delta) = 3
    assert abs(S1[3] - want) < 1e-9
    assert abs(y[0, 0] - h0 * 1.0) < 1e-9                 # readout from the boundary state


def test_initial_raw_step_and_retention(orc):
    """App. C.1: with zero scalar memories eta = gamma_eta log 2, alpha = alpha_init."""
    g = _golden_kv("initial_gates.txt")
    gamma, ainit = float(g["gamma_eta"]), float(g["alpha_init"])
    rng = np.random.default_rng(0)
    d = 16
    S = _rand_state(rng, d)
    S[4 * d * d:] = 0.0
    p = orc.OracleParams(gamma_eta=gamma, alpha_init=ainit)
    _, _, diag = orc.chunk(S, rng.standard_normal((5, d)), p)
    f = orc.diag_fields(d)
    np.testing.assert_allclose(diag[:, f["eta"]], gamma * math.log(2.0), rtol=1e-14)
    np.testing.assert_allclose(diag[:, f["alpha"]], ainit, rtol=1e-14)


def test_gate_maps_shape(orc):
    """Eq. (53) maps: eta > 0 increasing in s^eta, asymptote gamma*s for large s;
    alpha in (0,1) increasing, alpha -> 1 for large logits."""
    d = 4
    rng = np.random.default_rng(1)
    S = _rand_state(rng, d)
    S[4 * d * d:] = 0.0
    S[4 * d * d] = 1.0          # m^eta = e_0
    S[4 * d * d + d] = 1.0      # m^alpha = e_0
    xs = np.zeros((5, d))
    xs[:, 0] = [-30.0, -1.0, 0.0, 2.0, 30.0]
    xs[:, 1] = 1.0
    _, _, diag = orc.chunk(S, xs, orc.OracleParams())
    f = orc.diag_fields(d)
    eta, alpha = diag[:, f["eta"]], diag[:, f["alpha"]]
    assert (eta > 0).all() and (np.diff(eta) > 0).all()
    assert abs(eta[-1] - 0.025 * 30.0) < 1e-12
    assert (alpha > 0).all() and (alpha < 1).all() and (np.diff(alpha) > 0).all()
    assert alpha[-1] > 1 - 1e-12


# --------------------------------------------------------- DGD (App. B.2)

@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dgd_closed_form_equals_proximal_minimiser(orc, seed):
    """Eqs. (4)-(6), (35)-(37): the retained DGD step with alpha = 1 and
    eta = lambda/(1+lambda||k||^2) is the minimiser of the proximal L2
    objective, found here by a direct linear solve of its normal equations."""
    rng = np.random.default_rng(seed)
    d = 7
    W0 = rng.standard_normal((d, d))
    k = rng.standard_normal(d)          # unnormalised key on purpose (App. B.2 keeps ||k||)
    u = rng.standard_normal(d)
    lam = 0.37
    eta = lam / (1.0 + lam * (k @ k))
    W_or = orc.retained_dgd(W0, k, -u, 1.0, eta)     # g = -u
    # brute force: W (I + lam k k^T) = W0 + lam u k^T  <=>  (I + lam k k^T) W^T = (...)^T
    Amat = np.eye(d) + lam * np.outer(k, k)
    rhs = W0 + lam * np.outer(u, k)
    W_bf = np.linalg.solve(Amat.T, rhs.T).T
    np.testing.assert_allclose(W_or, W_bf, rtol=1e-12, atol=1e-12)
    # first-order optimality of the objective at the oracle's answer
    grad = np.outer(W_or @ k - u, k) + (W_or - W0) / lam
    assert np.abs(grad).max() < 1e-10


def test_retention_scales_memory(orc):
    """Eq. (7) with eta = 0 is pure retention: W_t = alpha W_{t-1}."""
    rng = np.random.default_rng(3)
    M = rng.standard_normal((5, 5))
    out = orc.retained_dgd(M, rng.standard_normal(5), rng.standard_normal(5), 0.8, 0.0)
    np.testing.assert_allclose(out, 0.8 * M, rtol=1e-15)


# ----------------------------------------------- step control (Def. 1, B.3)

def _ctl(orc, kvec, delta, eta, alpha, **kw):
    return orc.step_control(kvec, delta, eta, alpha, orc.OracleParams(**kw))


def test_soft_cap_bounds_and_derivative(orc):
    """App. B.3 Eq. (38): 0 < eta_bar < eta_inj, d eta_bar / d eta = exp(-eta/eta_inj)."""
    rng = np.random.default_rng(4)
    k = rng.standard_normal(8)
    k /= np.linalg.norm(k) * 1.5
    delta = rng.standard_normal(8)
    for eta in [1e-4, 0.01, 0.3, 2.0]:
        for alpha in [0.5, 0.9, 0.99]:
            c = _ctl(orc, k, delta, eta, alpha, inj_inward=0.0)
            if eta / c["eta_inj"] < 30:   # beyond that 1 - exp(-u) rounds to 1 in fp64
                assert 0.0 < c["eta_bar"] < c["eta_inj"]
            else:
                assert 0.0 < c["eta_bar"] <= c["eta_inj"]
            h = eta * 1e-6
            c1 = _ctl(orc, k, delta, eta + h, alpha, inj_inward=0.0)
            c0 = _ctl(orc, k, delta, eta - h, alpha, inj_inward=0.0)
            deriv = (c1["eta_bar"] - c0["eta_bar"]) / (2 * h)
            assert abs(deriv - math.exp(-eta / c["eta_inj"])) < 1e-6


def test_soft_cap_first_order_expansion(orc):
    """Eq. (39): eta_bar = eta - eta^2/(2 eta_inj) + O(eta^3/eta_inj^2)."""
    k = np.array([0.6, 0.0, 0.0, 0.0])
    delta = np.array([0.0, 3.0, 0.0, 4.0])
    for eta in [1e-3, 1e-4, 1e-5]:
        c = _ctl(orc, k, delta, eta, 0.9, inj_inward=0.0)
        ei = c["eta_inj"]
        resid = c["eta_bar"] - (eta - eta ** 2 / (2 * ei))
        assert abs(resid) <= 0.5 * eta ** 3 / ei ** 2


def test_injection_limit_and_inward_factor(orc):
    """Eq. (19) with r = sqrt(||delta||^2 + eps^2) + eps and the 1 - 1e-3 inward
    factor of App. B.3 (the implemented limit is that much more conservative)."""
    k = np.array([1.0, 0.0, 0.0])
    delta = np.array([0.0, 3.0, 4.0])          # ||delta|| = 5
    pure = _ctl(orc, k, delta, 0.01, 0.9, inj_inward=0.0)
    impl = _ctl(orc, k, delta, 0.01, 0.9)
    assert abs(pure["r"] - (5.0 + 1e-6)) < 1e-12
    np.testing.assert_allclose(pure["eta_inj"], 0.1 / (5.0 + 1e-6), rtol=1e-12)
    np.testing.assert_allclose(impl["eta_inj"] / pure["eta_inj"], 1 - 1e-3, rtol=1e-14)


def test_spectral_clamp_branch(orc):
    """Eq. (20): a hand-built token whose capped candidate exceeds
    2 alpha / ||k||^2 executes the spectral limit, rounded toward zero after
    the 1 - 1e-6 inward factor, and then |alpha - eta_tilde ||k||^2| <= alpha
    (Eq. (41))."""
    k = np.array([1.0, 0.0])                    # ||k|| = 1
    delta = np.array([0.0, 0.01])               # tiny discrepancy -> large eta_inj
    alpha = 0.05
    c = _ctl(orc, k, delta, 100.0, alpha)
    assert c["eta_bar"] > 2 * alpha
    limit = (1 - 1e-6) * 2 * alpha
    assert c["eta_spec"] < limit and np.nextafter(c["eta_spec"], np.inf) >= limit
    assert c["eta_tilde"] == c["eta_spec"]
    kap = k @ k
    assert abs(alpha - c["eta_tilde"] * kap) <= alpha
    # a zero key: the floor keeps the limit finite and it never binds
    c0 = _ctl(orc, np.zeros(2), delta, 100.0, alpha)
    assert c0["eta_tilde"] == c0["eta_bar"]


def test_control_switches(orc):
    """Ablation switches: without the soft cap eta_bar = eta; without the
    spectral clamp eta_tilde = eta_bar."""
    k = np.array([1.0, 0.0])
    delta = np.array([0.0, 0.01])
    c = _ctl(orc, k, delta, 100.0, 0.05, control_flags=orc.NO_INJ_CAP | orc.NO_SPEC_CLAMP)
    assert c["eta_bar"] == 100.0 and c["eta_tilde"] == 100.0


def test_alpha_one_gives_zero_step(orc):
    """alpha = 1 leaves no injection margin: eta_inj = 0 and the executed step is 0."""
    c = _ctl(orc, np.array([0.3, 0.4]), np.array([1.0, 2.0]), 0.5, 1.0)
    assert c["eta_inj"] == 0.0 and c["eta_tilde"] == 0.0


# ------------------------------------------- operator bounds (B.3, B.4)

def _tiny_chunk_cases():
    # (seed, eta_bias, alpha_init, d, L, scale of the state)
    return [(0, 0.0, 0.9, 8, 12, None), (1, 3.0, 0.9, 8, 12, None), (2, 6.0, 0.5, 6, 10, 2.0),
            (3, 0.0, 0.999, 8, 16, None), (4, 8.0, 0.2, 5, 9, 0.05)]


@pytest.mark.parametrize("case", _tiny_chunk_cases())
def test_prop1_cor1_bounds_by_svd(orc, case):
    """Prop. 1: ||A_t|| <= alpha_t, ||B_t|| < 1 - alpha_t; Eq. (42): ||B_t|| =
    eta_tilde ||delta|| ||k||; Cor. 1: ||T_t|| < 1 -- every token, by SVD."""
    seed, bias, ainit, d, L, sc = case
    rng = np.random.default_rng(seed)
    S = _rand_state(rng, d, sc)
    p = orc.OracleParams(eta_bias=bias, alpha_init=ainit)
    _, _, diag = orc.chunk(S, rng.standard_normal((L, d)) * 2.0, p)
    f = orc.diag_fields(d)
    for t in range(L):
        k, dl = diag[t, f["k"]], diag[t, f["delta"]]
        al, et = diag[t, f["alpha"]], diag[t, f["eta_tilde"]]
        A = al * np.eye(d) - et * np.outer(k, k)
        Bm = -et * np.outer(dl, k)
        nA, nB = np.linalg.norm(A, 2), np.linalg.norm(Bm, 2)
        assert nA <= al * (1 + 1e-12)
        assert nB < 1 - al
        assert abs(nB - et * np.linalg.norm(dl) * np.linalg.norm(k)) <= 1e-12 * max(nB, 1e-300)
        assert np.linalg.norm(A + Bm, 2) < 1.0
        assert np.linalg.norm(k) <= 1.0


@pytest.mark.parametrize("case", _tiny_chunk_cases())
def test_prop2_literal_update_equals_shared_gain(orc, case):
    """Prop. 2 / Eq. (46): the oracle's literal per-memory update (each memory
    with its own v_hat and g) ends the chunk at M_b G with the gain recursion
    G_t = G_{t-1} A_t + B_t built here from the same tokens' (k, delta, alpha,
    eta_tilde); Thm. 1: ||G_t|| <= 1 and ||M_t||_F <= ||M_b||_F at every t."""
    seed, bias, ainit, d, L, sc = case
    rng = np.random.default_rng(seed)
    S = _rand_state(rng, d, sc)
    p = orc.OracleParams(eta_bias=bias, alpha_init=ainit)
    xs = rng.standard_normal((L, d)) * 2.0
    S_end, _, diag = orc.chunk(S, xs, p)
    f = orc.diag_fields(d)
    G = np.eye(d)
    mb = orc.split_memories(S, d)
    for t in range(L):
        k, dl = diag[t, f["k"]], diag[t, f["delta"]]
        al, et = diag[t, f["alpha"]], diag[t, f["eta_tilde"]]
        G = G @ (al * np.eye(d) - et * np.outer(k, k)) - et * np.outer(dl, k)
        assert np.linalg.norm(G, 2) <= 1.0 + 1e-12
        S_t, _, _ = orc.chunk(S, xs[: t + 1], p)
        mt = orc.split_memories(S_t, d)
        for name in mb:
            assert np.linalg.norm(mt[name]) <= np.linalg.norm(mb[name]) * (1 + 1e-12)
    me = orc.split_memories(S_end, d)
    for name in mb:
        want = mb[name] @ G
        np.testing.assert_allclose(me[name], want, rtol=1e-10,
                                   atol=1e-12 * max(np.abs(want).max(), 1e-300))


def test_readout_and_generation_use_boundary_state(orc):
    """Eqs. (15)-(16): within a chunk, y_t and the generated quantities of
    every token come from the boundary state, so running the chunk over a
    prefix gives the same per-token outputs as over the whole chunk."""
    rng = np.random.default_rng(7)
    d, L = 6, 9
    S = _rand_state(rng, d)
    xs = rng.standard_normal((L, d))
    _, y_all, diag_all = orc.chunk(S, xs)
    for t in range(1, L):
        _, y_pre, diag_pre = orc.chunk(S, xs[:t])
        np.testing.assert_array_equal(y_pre, y_all[:t])
        np.testing.assert_array_equal(diag_pre, diag_all[:t])


# ---------------------------------------------- whole operator (Sec. 2.3)

def _tiny_inputs(rng, B, H, W, nh, d, scale=None):
    x = rng.standard_normal((B, H, W, nh * d))
    mem0 = np.stack([np.stack([_rand_state(rng, d, scale) for _ in range(nh)]) for _ in range(4)])
    return x, mem0


@pytest.mark.parametrize("H,W,chunk_len", [(3, 4, 0), (4, 6, 0), (5, 3, 4), (4, 4, 3)])
def test_chunk_one_equals_token_indexed(orc, H, W, chunk_len):
    """Sec. 2.1.3: with C = 1 the chunk form is the token-indexed recurrence;
    the token-indexed routine builds T_t of Eq. (21) and multiplies it out."""
    rng = np.random.default_rng(H * 10 + W)
    nh, d = 2, 6
    x, mem0 = _tiny_inputs(rng, 2, H, W, nh, d)
    p = orc.OracleParams(eta_bias=1.0)
    o1, m1 = orc.forward(x, mem0, H, W, nh, d, chunk_len=1, params=p, want_memories=True)
    o2, m2 = orc.forward(x, mem0, H, W, nh, d, params=p, want_memories=True,
                         token_indexed_mode=True)
    np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(m1, m2, rtol=1e-11, atol=1e-13)
    if chunk_len:  # a longer chunk differs from the token-indexed form
        o3 = orc.forward(x, mem0, H, W, nh, d, chunk_len=chunk_len, params=p)
        assert np.abs(o3 - o2).max() > 1e-8


def test_alpha_one_eta_zero_closed_form(orc):
    """alpha = 1, eta = 0 => A = I, B = 0: every memory is unchanged and the
    output is the closed form sum_r lambda_r M^m_{0,r} normalize(M^q_{0,r} x_p)."""
    rng = np.random.default_rng(11)
    B, H, W, nh, d = 2, 5, 7, 2, 8
    x, mem0 = _tiny_inputs(rng, B, H, W, nh, d)
    lam = rng.uniform(0.5, 1.5, size=(4, nh * d))
    p = orc.OracleParams(gate_mode=1, forced_eta=0.0, forced_alpha=1.0, dir_scale=lam)
    out, mo = orc.forward(x, mem0, H, W, nh, d, params=p, want_memories=True)
    for b in range(B):
        for r in range(4):
            np.testing.assert_array_equal(mo[b, r], mem0[r])
    want = np.zeros_like(out)
    for r in range(4):
        for h in range(nh):
            mm = orc.split_memories(mem0[r, h], d)
            xh = x[..., h * d:(h + 1) * d]
            qr = xh @ mm["q"].T
            q = qr / np.sqrt((qr ** 2).sum(-1, keepdims=True) + 1e-6)
            want[..., h * d:(h + 1) * d] += lam[r, h * d:(h + 1) * d] * (q @ mm["m"].T)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-14)


def test_identity_routes_merge_to_four_times(orc):
    """Cross-merge sums (not averages) the restored routes: four routes that
    each return the same per-pixel value give four times that value."""
    rng = np.random.default_rng(12)
    B, H, W, nh, d = 1, 3, 4, 1, 4
    x, _ = _tiny_inputs(rng, B, H, W, nh, d)
    S = np.zeros(4 * d * d + 2 * d)
    S[2 * d * d:3 * d * d] = np.eye(d).ravel()   # M^q = I
    S[3 * d * d:4 * d * d] = np.eye(d).ravel()   # M^m = I
    mem0 = np.tile(S, (4, nh, 1))
    p = orc.OracleParams(gate_mode=1, forced_eta=0.0, forced_alpha=1.0)
    out4 = orc.forward(x, mem0, H, W, nh, d, params=p)
    out1 = orc.forward(x, mem0, H, W, nh, d, dirs=1, params=p)
    np.testing.assert_allclose(out4, 4 * out1, rtol=1e-15)
    for r in (2, 4, 8):
        np.testing.assert_array_equal(orc.forward(x, mem0, H, W, nh, d, dirs=r, params=p), out1)


@pytest.mark.parametrize("H,W,chunk_len", [(4, 6, 0), (5, 3, 0), (4, 5, 3)])
def test_reversal_symmetry(orc, H, W, chunk_len):
    """Eq. (24) reverse routes: scan(left, X) = rot180(scan(right, rot180 X)) and
    scan(up, X) = rot180(scan(down, rot180 X)) with the same initial state, bit for bit."""
    rng = np.random.default_rng(13)
    nh, d = 2, 5
    x, mem0 = _tiny_inputs(rng, 2, H, W, nh, d)
    mem0[1] = mem0[0]
    mem0[3] = mem0[2]
    p = orc.OracleParams(eta_bias=0.5)
    xr = x[:, ::-1, ::-1, :].copy()
    for fwd, rev in ((1, 2), (4, 8)):
        a = orc.forward(x, mem0, H, W, nh, d, dirs=rev, chunk_len=chunk_len, params=p)
        b = orc.forward(xr, mem0, H, W, nh, d, dirs=fwd, chunk_len=chunk_len, params=p)
        np.testing.assert_array_equal(a, b[:, ::-1, ::-1, :])


def test_whole_scan_is_non_expansive(orc):
    """Thm. 1 applied chunk after chunk: every memory's Frobenius norm at the
    end of every route is at most its initial norm."""
    rng = np.random.default_rng(14)
    B, H, W, nh, d = 2, 6, 5, 2, 6
    x, mem0 = _tiny_inputs(rng, B, H, W, nh, d, scale=1.0)
    for ainit in (0.9, 0.999):
        _, mo = orc.forward(x, mem0, H, W, nh, d, params=orc.OracleParams(alpha_init=ainit),
                            want_memories=True)
        for b in range(B):
            for r in range(4):
                for h in range(nh):
                    m0 = orc.split_memories(mem0[r, h], d)
                    m1 = orc.split_memories(mo[b, r, h], d)
                    for name in m0:
                        assert np.linalg.norm(m1[name]) <= np.linalg.norm(m0[name]) * (1 + 1e-12)


def test_threads_do_not_change_results(orc):
    rng = np.random.default_rng(15)
    x, mem0 = _tiny_inputs(rng, 3, 4, 5, 2, 8)
    a = orc.forward(x, mem0, 4, 5, 2, 8, nthreads=1)
    b = orc.forward(x, mem0, 4, 5, 2, 8, nthreads=4)
    np.testing.assert_array_equal(a, b)


def test_mutated_oracle_fails_a_pin(orc):
    """The pins bite: a copy of the oracle with the DGD correction term dropped
    (built from the same source with one term removed, on the CPU) violates
    Prop. 2 against the gain built from Eq. (21)."""
    import ctypes
    import subprocess
    import tempfile
    src = open(os.path.join(os.path.dirname(orc.__file__), "vh_oracle.c")).read()
    needle = "row[j] = alpha * row[j] - eta * mk * k[j] - eta * g[i] * k[j];"
    assert needle in src
    bad = src.replace(needle, "row[j] = alpha * row[j] - eta * g[i] * k[j];")
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "bad.c")
        so = os.path.join(td, "bad.so")
        open(c, "w").write(bad)
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", so, c, "-lm"])
        badlib = ctypes.CDLL(so)
        badlib.vho_chunk.restype = ctypes.c_int
        badlib.vho_chunk.argtypes = orc.lib().vho_chunk.argtypes
        rng = np.random.default_rng(16)
        d, L = 6, 8
        S = _rand_state(rng, d)
        xs = rng.standard_normal((L, d))
        pp, keep = orc.OracleParams()._c()
        S_bad = S.copy()
        y = np.zeros((L, d))
        diag = np.zeros((L, 4 * d + 7))
        vp = ctypes.c_void_p
        assert badlib.vho_chunk(S_bad.ctypes.data_as(vp), d, xs.ctypes.data_as(vp), L,
                                ctypes.byref(pp), y.ctypes.data_as(vp), diag.ctypes.data_as(vp)) == 0
        f = orc.diag_fields(d)
        G = np.eye(d)
        for t in range(L):
            k, dl = diag[t, f["k"]], diag[t, f["delta"]]
            al, et = diag[t, f["alpha"]], diag[t, f["eta_tilde"]]
            G = G @ (al * np.eye(d) - et * np.outer(k, k)) - et * np.outer(dl, k)
        mb = orc.split_memories(S, d)
        me = orc.split_memories(S_bad, d)
        assert np.abs(me["m"] - mb["m"] @ G).max() > 1e-6
