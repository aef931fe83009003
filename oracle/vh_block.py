"""The VisionHOPE block around the operator, fp64 on the CPU (oracle).

TEST INFRASTRUCTURE ONLY: the tests and ``bench.py``'s CPU baseline leg may use this
module; the product path never does.

[VH] "VisionHOPE: Visual Backbones as Self-Modifying Learning Systems", Sec. 2.3
Eq. (27) and App. B.5, for a block input X (here NHWC, B x H x W x D):

    X0  = X + CPE(X)                              conditional positional encoding
    U   = Proj_in(LN1(X0))                         D -> D_m, pointwise
    Z   = U + DWg(U)                               gated depthwise residual branch
    Y   = F_VH(Z) + DWp(Z)                         operator + depthwise positional skip
    X1  = X0 + Proj_out(Y)                         D_m -> D, pointwise
    out = X1 + FFN(LN2(X1)),  FFN = W2 GELU(W1 . + b1) + b2, width 4 D

with F_VH the VisionHOPE-exact operator (outer query projection shared by the routes,
channel-wise skip from Z_r, direction scales lambda_r), computed by the C oracle.

Readings where the pages leave a step open (kept in one place, see the module's pins):
  * CPE is a 3 x 3 depthwise convolution with zero padding added to its input;
  * the gated depthwise branch is DWg(U) = SiLU(DW3x3(U)), SiLU(a) = a sigmoid(a);
  * the positional branch is a 3 x 3 depthwise convolution of Z;
  * every depthwise convolution has a per-channel bias; LN normalises the D channels of
    each pixel with eps 1e-5 and has a per-channel scale and shift;
  * the projections and both FFN layers have biases; GELU is the exact (erf) form.

Precision points (the GPU path's, replicated here so the two compute the same function):
the GEMM weights are bf16 values; LN1's output, Z, Y (before Proj_out), LN2's output,
FFN1's product (before its bias) and GELU's output are rounded to bf16 (round to nearest
even); everything else is fp64 here.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import OracleParams, forward as scan_forward


def bf16(a) -> np.ndarray:
    """Round to the nearest bfloat16 value (ties to even), returned as fp64."""
    f = np.asarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


@dataclass
class BlockWeights:
    """Parameters of one block (fp64 arrays; the GEMM weights hold bf16 values)."""
    cpe_w: np.ndarray    # [D][3][3]
    cpe_b: np.ndarray    # [D]
    ln1_g: np.ndarray    # [D]
    ln1_b: np.ndarray
    w_in: np.ndarray     # [D_m][D]
    b_in: np.ndarray     # [D_m]
    dw_w: np.ndarray     # [D_m][3][3]  gated depthwise branch
    dw_b: np.ndarray
    pos_w: np.ndarray    # [D_m][3][3]  positional branch
    pos_b: np.ndarray
    w_out: np.ndarray    # [D][D_m]
    b_out: np.ndarray    # [D]
    ln2_g: np.ndarray
    ln2_b: np.ndarray
    w_ff1: np.ndarray    # [4D][D]
    b_ff1: np.ndarray
    w_ff2: np.ndarray    # [D][4D]
    b_ff2: np.ndarray
    ln_eps: float = 1e-5


def dwconv3(x, w, b):
    """Depthwise 3 x 3 cross-correlation with zero padding, NHWC: out[b, i, j, c] =
    b[c] + sum_{di, dj in -1..1} w[c, di + 1, dj + 1] x[b, i + di, j + dj, c]."""
    B, H, W, C = x.shape
    p = np.zeros((B, H + 2, W + 2, C))
    p[:, 1:-1, 1:-1, :] = x
    out = np.broadcast_to(b, x.shape).copy()
    for di in range(3):
        for dj in range(3):
            out += w[:, di, dj] * p[:, di:di + H, dj:dj + W, :]
    return out


def layer_norm(x, g, b, eps):
    """Normalise the last axis to zero mean and unit variance (biased), then scale/shift."""
    mu = x.mean(-1, keepdims=True)
    var = ((x - mu) ** 2).mean(-1, keepdims=True)
    return (x - mu) / np.sqrt(var + eps) * g + b


def silu(a):
    return a / (1.0 + np.exp(-a))


_erfc = np.vectorize(math.erfc, otypes=[np.float64])


def gelu(a):
    """Exact GELU, a Phi(a) = a (1 + erf(a / sqrt 2)) / 2, written as a erfc(-a / sqrt 2) / 2
    (the same function; the erfc form keeps full precision in the lower tail, where
    1 + erf cancels)."""
    return 0.5 * a * _erfc(-a / math.sqrt(2.0))


def block_forward(x, w: BlockWeights, memories0, H: int, W: int, nh: int, d: int,
                  params: OracleParams, dirs: int = 15, return_parts: bool = False,
                  nthreads: int = 8, round_bf16: bool = True):
    """x [B][H][W][D] fp64 -> block output [B][H][W][D] (Eq. (27) with App. B.5).

    ``params`` carries the operator's constants, w_query [D_m][D_m], skip [4][D_m] and
    dir_scale [4][D_m]; the operator runs row/column-aligned chunks.  round_bf16=False
    drops every bf16 rounding point (the library's fp32-intermediate test mode)."""
    rnd = bf16 if round_bf16 else (lambda v: v)
    x = np.asarray(x, dtype=np.float64)
    x0 = x + dwconv3(x, w.cpe_w, w.cpe_b)
    a1 = rnd(layer_norm(x0, w.ln1_g, w.ln1_b, w.ln_eps))
    u = a1 @ w.w_in.T + w.b_in
    z = rnd(u + silu(dwconv3(u, w.dw_w, w.dw_b)))
    y = scan_forward(z, memories0, H, W, nh, d, dirs=dirs, params=params, nthreads=nthreads)
    yb = rnd(y + dwconv3(z, w.pos_w, w.pos_b))
    x1 = x0 + yb @ w.w_out.T + w.b_out
    a2 = rnd(layer_norm(x1, w.ln2_g, w.ln2_b, w.ln_eps))
    h = rnd(gelu(rnd(a2 @ w.w_ff1.T) + w.b_ff1))
    out = x1 + h @ w.w_ff2.T + w.b_ff2
    if return_parts:
        return out, dict(x0=x0, u=u, z=z, y=y, yb=yb, x1=x1, h=h)
    return out


def weights_from(arrays: dict, ln_eps: float = 1e-5) -> BlockWeights:
    """BlockWeights (fp64) holding exactly the given arrays' values."""
    return BlockWeights(**{k: np.asarray(v, dtype=np.float64) for k, v in arrays.items()},
                        ln_eps=ln_eps)
