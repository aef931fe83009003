"""Outer gradients of the VisionHOPE scan through the memory trajectory (fp64 CPU oracle).

TEST INFRASTRUCTURE ONLY: the tests and ``bench.py``'s CPU baseline leg may use this
module; the product path never does.

[VH] "VisionHOPE: Visual Backbones as Self-Modifying Learning Systems", Sec. 2.1.2:
the recurrence is explicit and differentiable, so outer gradients pass through the
memory trajectory without an inner solver.  This module restates the chunk-wise
forward of the C oracle in plain PyTorch fp64 ops, step for step:

  * routes and chunks, Eqs. (24)-(25): token t of route r visits pixel P_r(t); chunks
    of C_r tokens (row length for the row routes, column length for the column routes,
    or a fixed length), the last one partial;
  * generation from the chunk's boundary state, Eq. (15): k, v, q from M^k_b, M^v_b,
    M^q_b, the scalar outputs s^eta = m^eta_b x + b_eta and s^alpha = m^alpha_b x; k and q
    L2-normalised with the stabilised norm sqrt(||.||^2 + 1e-6) (App. C.1, App. B.5);
    eta = gamma_eta softplus(s^eta), alpha = sigmoid(s^alpha + logit alpha_init) (Eq. (53));
  * the executed step of Def. 1 (Eqs. (19)-(20)) with the App. B.3 safeguards: injection
    limit (1 - 1e-3)(1 - alpha)/r with r = sqrt(||delta||^2 + eps^2) + eps, soft cap
    eta_inj (1 - exp(-eta/eta_inj)), spectral limit (1 - 1e-6) 2 alpha / max(||k||^2, 1e-20)
    rounded one step toward zero, executed step the smaller of the two;
  * the readout from the boundary content memory y_t = M^m_b q_t (Eq. (16)), restored to
    its pixel and summed over routes with the scales lambda_r (Eq. (26));
  * the retained DGD step of every memory (Eq. (13) with Eq. (16)'s signal):
    M <- alpha M - eta_t (M k) k^T - eta_t (M_b delta) k^T, delta = k - v.

Every step is an elementwise op, a small matmul or a reduction over one vector; the
whole batch and all heads advance together (they are independent).  The gradient is
``torch.autograd.grad`` of the scalar <dout, out> + <dmem_final, memories_final>.  The
branch of every min/where follows the forward's choice; the one-ulp rounding of the
spectral limit passes the gradient of the unrounded value.

Pins (tests/test_oracle_grad.py): the forward equals the C oracle's; directional
derivatives equal central finite differences of the C oracle's forward; at alpha = 1 and a
zero executed step the gradient equals the closed form of y = M^m_0 normalize(M^q_0 x).

Supported: the method as defined (no ablation switch), the three gate modes, dir_scale,
any route subset, aligned or fixed chunks.  Not supported: the VisionHOPE-exact readout.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import OracleParams


def _route_order(r: int, H: int, W: int) -> np.ndarray:
    """Pixel visited at step t of route r: row-major, its reversal, the transpose
    flattened, its reversal (Eq. (24); the VMamba explainer's four orders)."""
    N = H * W
    t = np.arange(N)
    s = N - 1 - t if r & 1 else t
    return s if r < 2 else (s % H) * W + s // H


def _softplus(s):
    return torch.clamp(s, min=0.0) + torch.log1p(torch.exp(-torch.abs(s)))


def _step(k, delta, eta, alpha, p: OracleParams):
    """Executed step eta_tilde of Def. 1 (Eqs. (19)-(20), App. B.3); shapes [...]."""
    dd = (delta * delta).sum(-1)
    r = torch.sqrt(dd + p.eps * p.eps) + p.eps
    eta_inj = (1.0 - p.inj_inward) * (1.0 - alpha) / r
    pos = eta_inj > 0
    safe = torch.where(pos, eta_inj, torch.ones_like(eta_inj))
    eta_bar = torch.where(pos, safe * (-torch.expm1(-eta / safe)), torch.zeros_like(eta_inj))
    kk = (k * k).sum(-1)
    spec = (1.0 - p.spec_inward) * 2.0 * alpha / torch.clamp(kk, min=p.kk_floor)
    rounded = torch.nextafter(spec.detach(), torch.zeros_like(spec))
    spec = spec + (rounded - spec.detach())
    return torch.where(eta_bar < spec, eta_bar, spec)


def forward_torch(x, mem0, H: int, W: int, nh: int, d: int, dirs: int = 15, chunk_len: int = 0,
                  params: OracleParams | None = None):
    """x [B][H][W][nh d], mem0 [4][nh][4d^2+2d] (torch fp64) -> (out, memories [B][4][nh][..])."""
    p = params or OracleParams()
    if p.control_flags or p.w_query is not None or p.skip is not None:
        raise ValueError("the gradient oracle covers the method as defined only")
    B = x.shape[0]
    N = H * W
    Cc = nh * d
    dd = d * d
    R = 4 * d + 2
    xt = x.reshape(B, N, nh, d).permute(0, 2, 1, 3)            # [B][nh][N][d]
    out = torch.zeros(B, nh, N, d, dtype=torch.float64)
    mems = []
    logit = math.log(p.alpha_init / (1.0 - p.alpha_init))
    for r in range(4):
        if not dirs & (1 << r):
            mems.append(torch.zeros(B, nh, 4 * dd + 2 * d, dtype=torch.float64))
            continue
        order = torch.from_numpy(_route_order(r, H, W))
        xs = xt[:, :, order, :]                                  # route order
        m0 = mem0[r]                                             # [nh][4d^2+2d]
        S = torch.cat([m0[:, :4 * dd].reshape(nh, 4 * d, d), m0[:, 4 * dd:].reshape(nh, 2, d)], 1)
        S = S.unsqueeze(0).expand(B, nh, R, d)
        lam = (torch.from_numpy(np.asarray(p.dir_scale, dtype=np.float64)[r]).reshape(nh, 1, d)
               if p.dir_scale is not None else None)
        Cr = chunk_len if chunk_len > 0 else (W if r < 2 else H)
        ys = []
        for c0 in range(0, N, Cr):
            L = min(Cr, N - c0)
            X = xs[:, :, c0:c0 + L, :]                           # [B][nh][L][d]
            Sb = S
            # generation from the boundary state, Eq. (15)
            G = torch.einsum("bhod,bhld->bhlo", Sb, X)            # [B][nh][L][4d+2]
            kr, v, qr = G[..., :d], G[..., d:2 * d], G[..., 2 * d:3 * d]
            se, sa = G[..., 4 * d] + p.eta_bias, G[..., 4 * d + 1]
            k = kr / torch.sqrt((kr * kr).sum(-1, keepdim=True) + p.knorm_eps)
            q = qr / torch.sqrt((qr * qr).sum(-1, keepdim=True) + p.knorm_eps)
            if p.gate_mode == 0:
                eta = p.gamma_eta * _softplus(se)
                alpha = torch.sigmoid(sa + logit)
            else:
                eta = torch.full_like(se, p.forced_eta)
                alpha = torch.full_like(sa, p.forced_alpha)
            delta = k - v
            eta_t = eta if p.gate_mode == 2 else _step(k, delta, eta, alpha, p)
            # readout from the boundary content memory, Eq. (16)
            ys.append(torch.einsum("bhij,bhlj->bhli", Sb[:, :, 3 * d:4 * d, :], q))
            # retained DGD step of all six memories, token by token (Eq. (13))
            g = torch.einsum("bhod,bhld->bhlo", Sb, delta)        # M_b delta, every row
            for t in range(L):
                kt = k[:, :, t, :]
                Sk = torch.einsum("bhod,bhd->bho", S, kt)
                a = alpha[:, :, t].reshape(B, nh, 1, 1)
                e = eta_t[:, :, t].reshape(B, nh, 1, 1)
                S = a * S - e * (Sk + g[:, :, t, :]).unsqueeze(-1) * kt.unsqueeze(-2)
        Y = torch.cat(ys, 2)                                     # [B][nh][N][d], route order
        if lam is not None:
            Y = Y * lam
        inv = torch.empty(N, dtype=torch.int64)
        inv[order] = torch.arange(N)
        out = out + Y[:, :, inv, :]                              # restore positions, Eq. (26)
        mems.append(torch.cat([S[:, :, :4 * d, :].reshape(B, nh, 4 * dd),
                               S[:, :, 4 * d:, :].reshape(B, nh, 2 * d)], -1))
    out = out.permute(0, 2, 1, 3).reshape(B, H, W, Cc)
    return out, torch.stack(mems, 1)


def backward(x, mem0, dout, H: int, W: int, nh: int, d: int, dirs: int = 15, chunk_len: int = 0,
             params: OracleParams | None = None, dmem_final=None):
    """Gradients (dx [B][H][W][nh d], dmem0 [4][nh][4d^2+2d]) of <dout, out> +
    <dmem_final, memories_final> (numpy in, numpy out, fp64)."""
    xt = torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True)
    mt = torch.tensor(np.asarray(mem0, dtype=np.float64), requires_grad=True)
    out, mems = forward_torch(xt, mt, H, W, nh, d, dirs, chunk_len, params)
    loss = (out * torch.from_numpy(np.asarray(dout, dtype=np.float64))).sum()
    if dmem_final is not None:
        loss = loss + (mems * torch.from_numpy(np.asarray(dmem_final, dtype=np.float64))).sum()
    gx, gm = torch.autograd.grad(loss, (xt, mt))
    gm = gm.numpy().copy()
    for r in range(4):
        if not dirs & (1 << r):
            gm[r] = 0.0
    return gx.numpy(), gm
