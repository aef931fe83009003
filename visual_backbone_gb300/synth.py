"""Seeded synthetic inputs for the scan: the one module both the CUDA path's
callers (tests, benchmark) and the oracle's tests draw their inputs from.

It holds none of the method's arithmetic: it only draws random numbers and
rounds them to the storage types.

Recipe (workloads shaped like the backbone stages of "VisionHOPE: Visual
Backbones as Self-Modifying Learning Systems", App. C.1 chunk lengths
(56, 28, 14), and a dense-prediction map; synthetic stand-ins for
ImageNet-1K / COCO / ADE20K feature maps, which are not used):
  x         ~ N(0, 1) drawn in fp64 with numpy default_rng(seed), rounded to
              fp32 (round-to-nearest-even), then to bf16 (RNE) for bf16 maps.
  memories0 ~ N(0, 1/d) for all six memories of every (route, head), fp32.
              With x ~ N(0,1) this makes the eta/alpha logits m.x ~ N(0, 1).
  eta_bias  +1 on the high-resolution map (eta logits ~ N(1, 1)).
The "long-memory" variant of a workload only changes alpha_init to 0.999 so
that the state survives all chunks of a route (with 0.9 and chunks of 56
tokens the memories shrink by about 0.9^56 per chunk once the keys fall
below the normalisation stabiliser).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    W: int
    nh: int
    d: int
    chunk: int = 0          # 0 = row/column aligned (Eq. (25))
    dtype: str = "bf16"     # storage type of x
    seed: int = 0
    eta_bias: float = 0.0
    alpha_init: float = 0.9
    dirs: int = 15

    @property
    def Cc(self) -> int:
        return self.nh * self.d

    @property
    def N(self) -> int:
        return self.H * self.W

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.W

    def long_memory(self) -> "Workload":
        return replace(self, name=self.name + "-longmem", alpha_init=0.999)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 8, 8, 1, 16, 0, "f32", 0),
    "stage1": Workload("stage1", 32, 56, 56, 3, 32, 0, "bf16", 1),
    "stage2": Workload("stage2", 32, 28, 28, 6, 32, 0, "bf16", 2),
    "stage3": Workload("stage3", 128, 14, 14, 6, 64, 0, "bf16", 3),
    "highres": Workload("highres", 4, 128, 160, 3, 32, 0, "bf16", 4, eta_bias=1.0),
}


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


@dataclass
class Inputs:
    """x_store: the exact stored values (float32 array, or uint16 bf16 bits);
    x64: the same values widened to fp64; mem0: fp32 [4][nh][4d^2+2d]."""
    wl: Workload
    x_store: np.ndarray
    x64: np.ndarray
    mem0: np.ndarray


def make_inputs(wl: Workload, batch: int | None = None, first_image: int = 0) -> Inputs:
    """Draw the workload's inputs.  Images are drawn in order from one stream after
    memories0, so ``batch`` images starting at ``first_image`` are exactly those images of
    any longer draw: a rank holding images [s, s + n) of a batch sharded across ranks draws
    them with first_image = s, batch = n (the images before s are drawn and discarded)."""
    rng = np.random.default_rng(wl.seed)
    d = wl.d
    mem0 = (rng.standard_normal((4, wl.nh, 4 * d * d + 2 * d)) / np.sqrt(d)).astype(np.float32)
    B = wl.B if batch is None else batch
    for _ in range(first_image):
        rng.standard_normal((wl.H, wl.W, wl.Cc))
    x = rng.standard_normal((B, wl.H, wl.W, wl.Cc)).astype(np.float32)
    if wl.dtype == "bf16":
        bits = f32_to_bf16_bits(x)
        return Inputs(wl, bits, bf16_bits_to_f64(bits), mem0)
    return Inputs(wl, x, x.astype(np.float64), mem0)


def make_dir_scale(wl: Workload, seed: int = 1234) -> np.ndarray:
    """Channel-wise route scales lambda_r ~ U(0.5, 1.5), fp32 [4][Cc]."""
    rng = np.random.default_rng(seed)
    return rng.uniform(0.5, 1.5, size=(4, wl.Cc)).astype(np.float32)


BLOCK_GEMM_WEIGHTS = ("w_in", "w_out", "w_ff1", "w_ff2")


def make_block_weights(D: int, Dm: int, seed: int, hidden: int | None = None) -> dict:
    """Synthetic parameters of one VisionHOPE block (fp32 numpy arrays; the four GEMM
    weights hold bf16 values): GEMM weights ~ N(0, 1/fan_in), depthwise kernels
    ~ N(0, 1/9) for CPE and N(0, 1/36) for the two branches, LN scales ~ 1 + N(0, 0.1^2),
    biases ~ N(0, 0.02^2).  Shapes as in vh_block_weights, hidden = 4 D by default."""
    rng = np.random.default_rng(seed)
    hidden = hidden or 4 * D

    def lin(o, i):
        a = (rng.standard_normal((o, i)) / np.sqrt(i)).astype(np.float32)
        return bf16_bits_to_f64(f32_to_bf16_bits(a)).astype(np.float32)

    def vec(n, s=0.02):
        return (rng.standard_normal(n) * s).astype(np.float32)

    return dict(
        cpe_w=(rng.standard_normal((D, 3, 3)) / 3.0).astype(np.float32), cpe_b=vec(D),
        ln1_g=1.0 + vec(D, 0.1), ln1_b=vec(D),
        w_in=lin(Dm, D), b_in=vec(Dm),
        dw_w=(rng.standard_normal((Dm, 3, 3)) / 6.0).astype(np.float32), dw_b=vec(Dm),
        pos_w=(rng.standard_normal((Dm, 3, 3)) / 6.0).astype(np.float32), pos_b=vec(Dm),
        w_out=lin(D, Dm), b_out=vec(D),
        ln2_g=1.0 + vec(D, 0.1), ln2_b=vec(D),
        w_ff1=lin(hidden, D), b_ff1=vec(hidden),
        w_ff2=lin(D, hidden), b_ff2=vec(D))


def make_block_inputs(B: int, H: int, W: int, D: int, Dm: int, d: int, seed: int,
                      first_image: int = 0) -> dict:
    """x [B][H][W][D] ~ N(0, 1) fp32, the block weights, and the operator's inputs:
    memories0 ~ N(0, 1/d), the outer query W_q ~ N(0, 1/D_m), the skip ~ N(0, 1) and the
    route scales lambda ~ U(0.5, 1.5) (all fp32).  The parameters are drawn first and the
    images after them in order, so ``first_image`` selects a rank's images of a sharded
    batch while every rank draws the same parameters."""
    rng = np.random.default_rng(seed)
    nh = Dm // d
    mem0 = (rng.standard_normal((4, nh, 4 * d * d + 2 * d)) / np.sqrt(d)).astype(np.float32)
    w_query = (rng.standard_normal((Dm, Dm)) / np.sqrt(Dm)).astype(np.float32)
    skip = rng.standard_normal((4, Dm)).astype(np.float32)
    dir_scale = rng.uniform(0.5, 1.5, (4, Dm)).astype(np.float32)
    for _ in range(first_image):
        rng.standard_normal((H, W, D))
    x = rng.standard_normal((B, H, W, D)).astype(np.float32)
    return dict(x=x, weights=make_block_weights(D, Dm, seed), mem0=mem0, w_query=w_query,
                skip=skip, dir_scale=dir_scale, nh=nh)
