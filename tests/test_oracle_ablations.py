"""Pins of the oracle's ablation switches ("VisionHOPE: Visual Backbones as Self-Modifying
Learning Systems", Sec. 3.5 and App. C.5 "Step-size control behavior"): injection clamp,
soft spectral cap, no DGD correction, frozen K/V memories, frozen dynamics memories."""
import numpy as np
import pytest

from tests.test_oracle_pins import _rand_state, _tiny_inputs


def _ctl(orc, k, delta, eta, alpha, **kw):
    return orc.step_control(k, delta, eta, alpha, orc.OracleParams(**kw))


@pytest.mark.parametrize("eta", [1e-4, 0.02, 0.3, 5.0])
def test_hard_injection_clamp_is_min(orc, eta):
    rng = np.random.default_rng(int(eta * 1000))
    k = rng.standard_normal(8)
    k /= np.linalg.norm(k)
    delta = rng.standard_normal(8) * 0.3
    soft = _ctl(orc, k, delta, eta, 0.8)
    hard = _ctl(orc, k, delta, eta, 0.8, control_flags=orc.HARD_INJ)
    assert hard["eta_inj"] == soft["eta_inj"]
    assert hard["eta_bar"] == min(eta, soft["eta_inj"])
    assert hard["eta_bar"] >= soft["eta_bar"]  # 1 - e^-u < min(u, 1) for the soft cap


@pytest.mark.parametrize("alpha,kscale", [(0.9, 1.0), (0.05, 1.0), (0.6, 30.0), (0.999, 0.2)])
def test_soft_spectral_cap_properties(orc, alpha, kscale):
    """eta_spec (1 - exp(-eta_bar / eta_spec)): never above the spectral limit, strictly
    below a positive candidate, and equal to it to first order for small candidates."""
    rng = np.random.default_rng(int(alpha * 100))
    k = rng.standard_normal(6) * kscale
    for eta in [1e-6, 1e-3, 0.1, 2.0, 50.0]:
        c = _ctl(orc, k, rng.standard_normal(6) * 1e-3, eta, alpha,
                 control_flags=orc.SOFT_SPEC | orc.NO_INJ_CAP)
        eb, sp, et = c["eta_bar"], c["eta_spec"], c["eta_tilde"]
        assert eb == eta
        assert et <= sp and et < eb
        assert np.isclose(et, sp * -np.expm1(-eb / sp), rtol=1e-15)
        if eb < 1e-3 * sp:
            assert abs(et / eb - 1.0) <= eb / sp
    # with the clamp switched off as well, the clamp switch wins
    c = _ctl(orc, k, np.zeros(6), 3.0, alpha, control_flags=orc.SOFT_SPEC | orc.NO_SPEC_CLAMP)
    assert c["eta_tilde"] == c["eta_bar"]


def test_flag_precedence(orc):
    rng = np.random.default_rng(9)
    k, dl = rng.standard_normal(8), rng.standard_normal(8)
    a = _ctl(orc, k, dl, 0.7, 0.4, control_flags=orc.NO_INJ_CAP)
    b = _ctl(orc, k, dl, 0.7, 0.4, control_flags=orc.NO_INJ_CAP | orc.HARD_INJ)
    assert a == b


@pytest.mark.parametrize("flags", ["HARD_INJ", "SOFT_SPEC"])
def test_prop1_bounds_hold_for_the_alternative_maps(orc, flags):
    """The injection clamp keeps eta_bar <= eta_inj, so ||B|| < 1 - alpha; the soft
    spectral cap keeps eta_tilde <= eta_spec, so ||A|| <= alpha (App. C.5)."""
    rng = np.random.default_rng(11)
    d, L = 8, 14
    S = _rand_state(rng, d)
    p = orc.OracleParams(eta_bias=4.0, control_flags=getattr(orc, flags))
    _, _, diag = orc.chunk(S, rng.standard_normal((L, d)) * 2.0, p)
    f = orc.diag_fields(d)
    for t in range(L):
        k, dl = diag[t, f["k"]], diag[t, f["delta"]]
        al, et = diag[t, f["alpha"]], diag[t, f["eta_tilde"]]
        assert np.linalg.norm(al * np.eye(d) - et * np.outer(k, k), 2) <= al * (1 + 1e-12)
        assert np.linalg.norm(et * np.outer(dl, k), 2) < 1 - al


def test_no_dgd_step_closed_form(orc):
    rng = np.random.default_rng(12)
    d = 5
    M = rng.standard_normal((d, d))
    k, g = rng.standard_normal(d), rng.standard_normal(d)
    M_full = orc.retained_dgd(M, k, g, 0.8, 0.3)
    np.testing.assert_allclose(M_full, M @ (0.8 * np.eye(d) - 0.3 * np.outer(k, k)) - 0.3 * np.outer(g, k),
                               rtol=1e-13)
    S = _rand_state(rng, d)
    xs = rng.standard_normal((1, d))
    p = orc.OracleParams(control_flags=orc.NO_DGD)
    S1, _, diag = orc.chunk(S, xs, p)
    f = orc.diag_fields(d)
    k, dl = diag[0, f["k"]], diag[0, f["delta"]]
    al, et = diag[0, f["alpha"]], diag[0, f["eta_tilde"]]
    for name, Mb in orc.split_memories(S, d).items():  # M <- alpha M - eta M_b delta k^T
        np.testing.assert_allclose(orc.split_memories(S1, d)[name],
                                   al * Mb - et * np.outer(Mb @ dl, k), rtol=1e-12, atol=1e-15)


def test_no_dgd_shared_gain(orc):
    """Without the correction the gain recursion is G_t = alpha_t G_{t-1} - eta_t delta_t k_t^T
    and the literal per-memory update still ends the chunk at M_b G."""
    rng = np.random.default_rng(13)
    d, L = 7, 11
    S = _rand_state(rng, d)
    p = orc.OracleParams(eta_bias=2.0, control_flags=orc.NO_DGD)
    S_end, _, diag = orc.chunk(S, rng.standard_normal((L, d)) * 2.0, p)
    f = orc.diag_fields(d)
    G = np.eye(d)
    for t in range(L):
        k, dl = diag[t, f["k"]], diag[t, f["delta"]]
        G = diag[t, f["alpha"]] * G - diag[t, f["eta_tilde"]] * np.outer(dl, k)
    for name, Mb in orc.split_memories(S, d).items():
        np.testing.assert_allclose(orc.split_memories(S_end, d)[name], Mb @ G, rtol=1e-10,
                                   atol=1e-13)


@pytest.mark.parametrize("flags", [("FREEZE_KV",), ("FREEZE_DYN",), ("FREEZE_KV", "FREEZE_DYN")])
def test_frozen_memories_stay_fixed(orc, flags):
    rng = np.random.default_rng(14)
    x, mem0 = _tiny_inputs(rng, 1, 4, 5, 2, 6)
    cf = sum(getattr(orc, f) for f in flags)
    _, mo = orc.forward(x, mem0, 4, 5, 2, 6, params=orc.OracleParams(control_flags=cf),
                        want_memories=True)
    d = 6
    for r in range(4):
        for h in range(2):
            m0 = orc.split_memories(mem0[r, h], d)
            m1 = orc.split_memories(mo[0, r, h], d)
            fixed = set()
            if "FREEZE_KV" in flags:
                fixed |= {"k", "v"}
            if "FREEZE_DYN" in flags:
                fixed |= {"eta", "alpha"}
            for name in m0:
                if name in fixed:
                    np.testing.assert_array_equal(m1[name], m0[name])
                else:
                    assert not np.array_equal(m1[name], m0[name]), name


@pytest.mark.parametrize("flags", ["HARD_INJ", "SOFT_SPEC", "NO_DGD", "FREEZE_KV", "FREEZE_DYN"])
def test_chunk_one_equals_token_indexed_with_switches(orc, flags):
    rng = np.random.default_rng(15)
    x, mem0 = _tiny_inputs(rng, 1, 3, 4, 2, 5)
    p = orc.OracleParams(eta_bias=1.0, control_flags=getattr(orc, flags))
    a, ma = orc.forward(x, mem0, 3, 4, 2, 5, chunk_len=1, params=p, want_memories=True)
    b, mb = orc.forward(x, mem0, 3, 4, 2, 5, params=p, want_memories=True, token_indexed_mode=True)
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(ma, mb, rtol=1e-11, atol=1e-14)


def test_intra_chunk_readout_equals_boundary_readout_at_chunk_one(orc):
    rng = np.random.default_rng(16)
    x, mem0 = _tiny_inputs(rng, 1, 3, 4, 2, 5)
    p0 = orc.OracleParams(eta_bias=1.0)
    p1 = orc.OracleParams(eta_bias=1.0, control_flags=orc.INTRA_READ)
    a = orc.forward(x, mem0, 3, 4, 2, 5, chunk_len=1, params=p0)
    b = orc.forward(x, mem0, 3, 4, 2, 5, chunk_len=1, params=p1)
    np.testing.assert_array_equal(a, b)
    c = orc.forward(x, mem0, 3, 4, 2, 5, params=p0)
    e = orc.forward(x, mem0, 3, 4, 2, 5, params=p1)
    assert not np.allclose(c, e)   # differs once a chunk holds several tokens


def test_intra_chunk_readout_is_boundary_state_times_gain(orc):
    """y_t = M^m_b G_{t-1} q_t with the gain recursion built here from the tokens' own
    (k, delta, alpha, eta_tilde) -- the shared-gain form of the working state (Prop. 2)."""
    rng = np.random.default_rng(17)
    d, L = 6, 10
    S = _rand_state(rng, d)
    xs = rng.standard_normal((L, d)) * 2.0
    p = orc.OracleParams(eta_bias=2.0, control_flags=orc.INTRA_READ)
    _, y, diag = orc.chunk(S, xs, p)
    f = orc.diag_fields(d)
    Mm = orc.split_memories(S, d)["m"]
    G = np.eye(d)
    for t in range(L):
        q = diag[t, f["q"]]
        np.testing.assert_allclose(y[t], Mm @ G @ q, rtol=1e-10, atol=1e-13)
        k, dl = diag[t, f["k"]], diag[t, f["delta"]]
        al, et = diag[t, f["alpha"]], diag[t, f["eta_tilde"]]
        G = G @ (al * np.eye(d) - et * np.outer(k, k)) - et * np.outer(dl, k)
