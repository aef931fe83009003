"""The block's GELU (FFN1 epilogue) element by element against the exact definition.

GELU(a) = a Phi(a) = a (1 + erf(a / sqrt 2)) / 2 ("VisionHOPE", Sec. 2.3 Eq. (27), the
block's FFN; the exact erf form), evaluated by the oracle's fp64 formula (its erfc form,
exact in relative terms on both tails) and rounded to bf16, against the device function through `vh_debug_gelu`.  The device result may differ
by one bf16 step only where the exact value lies within the fp32 evaluation's error of a
rounding boundary (half-way between two bf16 values)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

REL = 2e-6   # bound on the fp32 evaluation's relative error, with margin


def _bf16_round(y):
    import torch
    return torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16).float().numpy().astype(np.float64)


def _exact(a64):
    from oracle import vh_block
    return vh_block.gelu(a64)


def _near_boundary(y):
    """True where y lies within REL of a midpoint between two adjacent bf16 values."""
    import torch
    rb = torch.from_numpy(y.astype(np.float32)).to(torch.bfloat16)
    bits = rb.view(torch.int16)
    up = (bits + 1).view(torch.bfloat16).double().numpy()      # the two neighbours in the
    dn = (bits - 1).view(torch.bfloat16).double().numpy()      # bit order of the magnitude
    r = rb.double().numpy()
    dist = np.minimum(np.abs(y - (r + up) / 2), np.abs(y - (r + dn) / 2))
    return dist <= REL * np.abs(y) + 1e-45


def _check(vhlib, a32):
    import torch
    g = vhlib.debug_gelu(torch.from_numpy(a32).cuda()).float().cpu().numpy().astype(np.float64)
    y = _exact(a32.astype(np.float64))
    r = _bf16_round(y)
    bad = (g != r) & ~_near_boundary(y)
    assert not bad.any(), (a32[bad][:8], g[bad][:8], r[bad][:8])
    return np.mean(g != r)


def test_gelu_dense_grid(vhlib):
    a = np.linspace(-13.0, 13.0, 1_000_001).astype(np.float32)
    _check(vhlib, a)


def test_gelu_far_tails(vhlib):
    """Beyond |a| = 13 the lower tail is below 1e-37 and may flush to zero; the upper is a."""
    import torch
    a = np.linspace(13.0, 40.0, 10001).astype(np.float32)
    g = vhlib.debug_gelu(torch.from_numpy(np.concatenate([-a, a])).cuda()).float().cpu().numpy()
    lo, hi = g[:a.size], g[a.size:]
    assert (np.abs(lo) <= 1e-37).all() and (lo <= 0).all()
    np.testing.assert_array_equal(hi, _bf16_round(a.astype(np.float64)).astype(np.float32))


@pytest.mark.parametrize("sigma", [0.5, 1.0, 3.0])
def test_gelu_normal_samples(vhlib, sigma):
    a = (np.random.default_rng(7).standard_normal(2_000_000) * sigma).astype(np.float32)
    flips = _check(vhlib, a[np.abs(a) <= 13.0])   # (beyond 13: test_gelu_far_tails)
    assert flips < 1e-4, flips


def test_gelu_special_values(vhlib):
    import torch
    a = np.array([0.0, -0.0, 1e-30, -1e-30, 20.0, -20.0, np.inf, np.nan, 3e38], dtype=np.float32)
    g = vhlib.debug_gelu(torch.from_numpy(a).cuda()).float().cpu().numpy()
    assert g[0] == 0 and g[1] == 0
    assert g[4] == 20.0 and g[5] == 0 and g[6] == np.inf and np.isnan(g[7]) and g[8] == np.float32(
        torch.tensor(3e38).to(torch.bfloat16).float().item())
    assert abs(g[2] - 5e-31) <= 5e-31 * 2 ** -7 and abs(g[3] + 5e-31) <= 5e-31 * 2 ** -7
