"""fp64 CPU oracle of the VisionHOPE four-direction memory scan (ctypes binding).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package; the product path never
does.  The arithmetic lives in ``vh_oracle.c`` (plain C, fp64); this module
only marshals numpy arrays.  See the header of ``vh_oracle.c`` for the
passages each routine follows and the pins that check it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vh_oracle.c")
_LIB = os.path.join(_HERE, "libvh_oracle.so")

NO_INJ_CAP = 1
NO_SPEC_CLAMP = 2
HARD_INJ = 4
SOFT_SPEC = 8
NO_DGD = 16
FREEZE_KV = 32
FREEZE_DYN = 64
INTRA_READ = 128


def build(force: bool = False) -> str:
    """Compile ``vh_oracle.c`` with gcc into ``libvh_oracle.so`` (IEEE fp64, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC,
                               "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


class _Params(ctypes.Structure):
    _fields_ = [
        ("gamma_eta", ctypes.c_double), ("alpha_init", ctypes.c_double),
        ("eta_bias", ctypes.c_double), ("eps", ctypes.c_double),
        ("knorm_eps", ctypes.c_double), ("inj_inward", ctypes.c_double),
        ("spec_inward", ctypes.c_double), ("kk_floor", ctypes.c_double),
        ("dir_scale", ctypes.POINTER(ctypes.c_double)),
        ("gate_mode", ctypes.c_int), ("forced_eta", ctypes.c_double),
        ("forced_alpha", ctypes.c_double), ("control_flags", ctypes.c_uint),
        ("w_query", ctypes.POINTER(ctypes.c_double)),
        ("skip", ctypes.POINTER(ctypes.c_double)),
    ]


@dataclass
class OracleParams:
    """Constants of the method (App. C.1 and App. B.3 of the VisionHOPE page)."""
    gamma_eta: float = 0.025
    alpha_init: float = 0.9
    eta_bias: float = 0.0
    eps: float = 1e-6
    knorm_eps: float = 1e-6
    inj_inward: float = 1e-3
    spec_inward: float = 1e-6
    kk_floor: float = 1e-20
    dir_scale: Optional[np.ndarray] = None   # [4][Cc]
    gate_mode: int = 0
    forced_eta: float = 0.0
    forced_alpha: float = 0.0
    control_flags: int = 0
    w_query: Optional[np.ndarray] = None     # [Cc][Cc]: VisionHOPE-exact readout query
    skip: Optional[np.ndarray] = None        # [4][Cc]: channel-wise skip of each route

    def _c(self):
        keep = []

        def arr(a):
            if a is None:
                return None
            a = np.ascontiguousarray(a, dtype=np.float64)
            keep.append(a)
            return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))
        p = _Params(self.gamma_eta, self.alpha_init, self.eta_bias, self.eps, self.knorm_eps,
                    self.inj_inward, self.spec_inward, self.kk_floor, arr(self.dir_scale),
                    self.gate_mode, self.forced_eta, self.forced_alpha, self.control_flags,
                    arr(self.w_query), arr(self.skip))
        return p, keep


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        D = ctypes.c_double
        P = ctypes.c_void_p
        _lib.vho_route_pixel.restype = ctypes.c_long
        _lib.vho_route_pixel.argtypes = [ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.c_int]
        _lib.vho_step_control.restype = D
        _lib.vho_step_control.argtypes = [P, P, ctypes.c_int, D, D, ctypes.POINTER(_Params), P]
        _lib.vho_retained_dgd.restype = None
        _lib.vho_retained_dgd.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, D, D]
        _lib.vho_chunk.restype = ctypes.c_int
        _lib.vho_chunk.argtypes = [P, ctypes.c_int, P, ctypes.c_int, ctypes.POINTER(_Params), P, P]
        _lib.vho_token_indexed.restype = ctypes.c_int
        _lib.vho_token_indexed.argtypes = [P, ctypes.c_int, P, ctypes.c_int,
                                           ctypes.POINTER(_Params), P]
        _lib.vho_forward.restype = ctypes.c_int
        _lib.vho_forward.argtypes = [P, P] + [ctypes.c_int] * 5 + [ctypes.c_uint, ctypes.c_int,
                                     ctypes.c_int, ctypes.POINTER(_Params), P, P, ctypes.c_int]
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def route_pixel(r: int, t: int, H: int, W: int) -> int:
    """Pixel index visited at step t of route r (0 right, 1 left, 2 down, 3 up)."""
    return int(lib().vho_route_pixel(r, t, H, W))


def route_order(r: int, H: int, W: int) -> np.ndarray:
    return np.array([route_pixel(r, t, H, W) for t in range(H * W)], dtype=np.int64)


def step_control(k, delta, eta: float, alpha: float, params: OracleParams | None = None) -> dict:
    """Def. 1 with the finite-precision safeguards; returns every intermediate limit."""
    params = params or OracleParams()
    k = _f64(k)
    delta = _f64(delta)
    out = np.zeros(5)
    p, keep = params._c()
    et = lib().vho_step_control(_ptr(k), _ptr(delta), k.size, eta, alpha, ctypes.byref(p), _ptr(out))
    return dict(eta_inj=out[0], eta_bar=out[1], eta_spec=out[2], eta_tilde=out[3], r=out[4],
                ret=et)


def retained_dgd(M, k, g, alpha: float, eta: float) -> np.ndarray:
    """One retained DGD step M(alpha I - eta k k^T) - eta g k^T on an R x d memory."""
    M = _f64(M).copy()
    R, d = M.shape
    lib().vho_retained_dgd(_ptr(M), R, d, _ptr(_f64(k)), _ptr(_f64(g)), alpha, eta)
    return M


def diag_fields(d: int) -> dict:
    return dict(k=slice(0, d), v=slice(d, 2 * d), q=slice(2 * d, 3 * d),
                delta=slice(3 * d, 4 * d), eta=4 * d, alpha=4 * d + 1, eta_inj=4 * d + 2,
                eta_bar=4 * d + 3, eta_spec=4 * d + 4, eta_tilde=4 * d + 5, r=4 * d + 6)


def chunk(S, xs, params: OracleParams | None = None):
    """One chunk of the chunk-wise recurrence from boundary state S over tokens xs [L][d].

    Returns (S_end, y [L][d], diag [L][4d+7])."""
    params = params or OracleParams()
    S = _f64(S).copy()
    xs = _f64(xs)
    L, d = xs.shape
    assert S.size == 4 * d * d + 2 * d
    y = np.zeros((L, d))
    diag = np.zeros((L, 4 * d + 7))
    p, keep = params._c()
    rc = lib().vho_chunk(_ptr(S), d, _ptr(xs), L, ctypes.byref(p), _ptr(y), _ptr(diag))
    assert rc == 0, rc
    return S, y, diag


def token_indexed(S, xs, params: OracleParams | None = None):
    """Fully token-indexed recurrence (transition T_t built explicitly) over xs [L][d]."""
    params = params or OracleParams()
    S = _f64(S).copy()
    xs = _f64(xs)
    L, d = xs.shape
    y = np.zeros((L, d))
    p, keep = params._c()
    rc = lib().vho_token_indexed(_ptr(S), d, _ptr(xs), L, ctypes.byref(p), _ptr(y))
    assert rc == 0, rc
    return S, y


def forward(x, mem0, H: int, W: int, nh: int, d: int, dirs: int = 15, chunk_len: int = 0,
            params: OracleParams | None = None, want_memories: bool = False,
            token_indexed_mode: bool = False, nthreads: int = 1):
    """The whole operator: x [B][H][W][nh*d], mem0 [4][nh][4d^2+2d] -> out (, memories)."""
    params = params or OracleParams()
    x = _f64(x)
    mem0 = _f64(mem0)
    B = x.shape[0]
    out = np.zeros((B, H, W, nh * d))
    mo = np.zeros((B, 4, nh, 4 * d * d + 2 * d)) if want_memories else None
    p, keep = params._c()
    rc = lib().vho_forward(_ptr(x), _ptr(mem0), B, H, W, nh, d, dirs, chunk_len,
                           1 if token_indexed_mode else 0, ctypes.byref(p), _ptr(out),
                           _ptr(mo) if mo is not None else None, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle vho_forward failed: {rc}")
    return (out, mo) if want_memories else out


def split_memories(S, d: int) -> dict:
    """Views of the six memories in one state block."""
    S = np.asarray(S)
    dd = d * d
    return dict(k=S[0:dd].reshape(d, d), v=S[dd:2 * dd].reshape(d, d),
                q=S[2 * dd:3 * dd].reshape(d, d), m=S[3 * dd:4 * dd].reshape(d, d),
                eta=S[4 * dd:4 * dd + d].reshape(1, d), alpha=S[4 * dd + d:].reshape(1, d))
