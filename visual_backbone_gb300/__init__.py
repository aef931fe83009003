"""GB300-native VisionHOPE four-direction self-referential memory scan.

Python binding of ``libvh.so`` (C ABI in ``include/vh.h``).  This module only
marshals arguments: every step of the scan runs in the library's CUDA
kernels.  There is no CPU fallback; if the library is missing or the tensors
are not on a CUDA device, the call raises.

Method: "VisionHOPE: Visual Backbones as Self-Modifying Learning Systems",
Sec. 2.1-2.3 (the VisionHOPE operator, Eqs. (24)-(26)), with the six-memory
set of "Nested Learning: The Illusion of Deep Learning Architectures",
part 12, Eqs. (94)-(96).
"""
from __future__ import annotations

import ctypes
import os
import re
from dataclasses import dataclass
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvh.so")
# VH_DEBUG_BOUNDS=1 in the environment loads the checked-index build instead
# (``_build.build(debug=True)``); its failed checks show up as VH_ERR_BOUNDS in check()
if os.environ.get("VH_DEBUG_BOUNDS") == "1":
    LIB_PATH = os.path.join(_HERE, "libvh_dbg.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "vh.h")

DIR_RIGHT, DIR_LEFT, DIR_DOWN, DIR_UP, DIR_ALL = 1, 2, 4, 8, 15
DTYPE_F32, DTYPE_BF16 = 0, 1
GATE_GENERATED, GATE_FORCED_RAW, GATE_FORCED_EXEC = 0, 1, 2
CTRL_NO_INJ_CAP, CTRL_NO_SPEC_CLAMP, CTRL_HARD_INJ, CTRL_SOFT_SPEC = 1, 2, 4, 8
CTRL_NO_DGD, CTRL_FREEZE_KV, CTRL_FREEZE_DYN, CTRL_INTRA_READ = 16, 32, 64, 128
IMPL = {"auto": 0, "simt": 1, "tc": 2, "tc_wy": 3, "tc_recur": 4, "tc_pipe": 5}
STAT_TOKENS, STAT_SPEC_ACTIVE, STAT_INJ_RATIO_GT1, STAT_NONFINITE = 0, 1, 2, 3
STAT_TIMEOUT, STAT_BOUNDS, STAT_COUNT = 4, 5, 8


class VhError(RuntimeError):
    """A libvh call returned a non-OK status."""


class CParams(ctypes.Structure):
    """Mirror of ``vh_params`` (include/vh.h)."""
    _fields_ = [
        ("batch", ctypes.c_int), ("channels", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("x_dtype", ctypes.c_int),
        ("gamma_eta", ctypes.c_float), ("alpha_init", ctypes.c_float),
        ("eta_bias", ctypes.c_float), ("eps", ctypes.c_float), ("knorm_eps", ctypes.c_float),
        ("inj_inward", ctypes.c_float), ("spec_inward", ctypes.c_float),
        ("kk_floor", ctypes.c_float),
        ("dir_scale", ctypes.c_void_p), ("memories_out", ctypes.c_void_p),
        ("gate_mode", ctypes.c_int), ("forced_eta", ctypes.c_float),
        ("forced_alpha", ctypes.c_float), ("control_flags", ctypes.c_uint),
        ("stats", ctypes.c_void_p), ("impl", ctypes.c_int), ("accumulate", ctypes.c_int),
        ("stream", ctypes.c_void_p),
        ("w_query", ctypes.c_void_p), ("skip", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("wait_limit", ctypes.c_longlong), ("withhold_first_copy", ctypes.c_int),
    ]


BLOCK_WEIGHT_NAMES = ("cpe_w", "cpe_b", "ln1_g", "ln1_b", "w_in", "b_in", "dw_w", "dw_b", "pos_w",
                      "pos_b", "w_out", "b_out", "ln2_g", "ln2_b", "w_ff1", "b_ff1", "w_ff2", "b_ff2")


class CBlockWeights(ctypes.Structure):
    """Mirror of ``vh_block_weights`` (include/vh.h)."""
    _fields_ = ([("dim", ctypes.c_int), ("hidden", ctypes.c_int), ("ln_eps", ctypes.c_float)] +
                [(n, ctypes.c_void_p) for n in BLOCK_WEIGHT_NAMES] +
                [("f32_intermediates", ctypes.c_int)])


BLOCK_GEMM_WEIGHTS = ("w_in", "w_out", "w_ff1", "w_ff2")   # bf16; the rest fp32


@dataclass
class ScanParams:
    """Method constants and switches of one call (defaults: the pages' values)."""
    gamma_eta: float = 0.025
    alpha_init: float = 0.9
    eta_bias: float = 0.0
    eps: float = 1e-6
    knorm_eps: float = 1e-6
    inj_inward: float = 1e-3
    spec_inward: float = 1e-6
    kk_floor: float = 1e-20
    gate_mode: int = GATE_GENERATED
    forced_eta: float = 0.0
    forced_alpha: float = 0.0
    control_flags: int = 0
    impl: str = "auto"
    wait_limit: int = 0               # cycles before a bounded wait gives up; 0 = 2^32
    withhold_first_copy: bool = False  # test hook: the first input copy is never issued


_lib = None


def lib() -> ctypes.CDLL:
    """Load libvh.so (built by ``__graft_entry__.build()``); raise if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); run "
                               "__graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, ci, cu = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint
        L.vh_scan_forward.restype = ci
        L.vh_scan_forward.argtypes = [vp, vp, ctypes.POINTER(CParams), ci, ci, cu, ci, vp]
        L.vh_debug_permute.restype = ci
        L.vh_debug_permute.argtypes = [vp, ctypes.POINTER(CParams), ci, ci, ci, vp]
        L.vh_debug_gelu.restype = ci
        L.vh_debug_gelu.argtypes = [vp, vp, ctypes.c_longlong, vp]
        L.vh_workspace_size.restype = ctypes.c_size_t
        L.vh_workspace_size.argtypes = [ctypes.POINTER(CParams), ci, ci, cu, ci]
        L.vh_scan_backward.restype = ci
        L.vh_scan_backward.argtypes = [vp, vp, ctypes.POINTER(CParams), ci, ci, cu, ci, vp, vp,
                                       vp, vp]
        L.vh_backward_workspace_size.restype = ctypes.c_size_t
        L.vh_backward_workspace_size.argtypes = [ctypes.POINTER(CParams), ci, ci, cu, ci]
        L.vh_block_forward.restype = ci
        L.vh_block_forward.argtypes = [vp, vp, ctypes.POINTER(CParams),
                                       ctypes.POINTER(CBlockWeights), ci, ci, vp]
        L.vh_block_workspace_size.restype = ctypes.c_size_t
        L.vh_block_workspace_size.argtypes = [ctypes.POINTER(CParams),
                                              ctypes.POINTER(CBlockWeights), ci, ci]
        L.vh_status_string.restype = ctypes.c_char_p
        L.vh_status_string.argtypes = [ci]
        L.vh_last_error.restype = ctypes.c_char_p
        L.vh_last_error.argtypes = []
        L.vh_version.restype = ci
        L.vh_check.restype = ci
        L.vh_check.argtypes = [vp, vp]
        L.vh_params_init.restype = None
        L.vh_params_init.argtypes = [ctypes.POINTER(CParams)]
        _lib = L
    return _lib


def header_functions() -> list[str]:
    """Names of the functions ``include/vh.h`` declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vh_[a-z_]+)\s*\(", text)))


def shard_images(global_batch: int, world: int, rank: int) -> range:
    """Images of a batch held by one rank when the batch is sharded across ``world``
    ranks: contiguous blocks, the first ``global_batch % world`` ranks one image larger.
    Images are independent (every route of every image starts from memories0), so the
    shards need no exchange; the union over ranks is the batch, each image once."""
    if world < 1 or not 0 <= rank < world or global_batch < 0:
        raise ValueError(f"shard_images({global_batch}, {world}, {rank})")
    base, extra = divmod(global_batch, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def _check(status: int):
    if status != 0:
        L = lib()
        raise VhError(f"{L.vh_status_string(status).decode()} ({status}): "
                      f"{L.vh_last_error().decode()}")


def make_cparams(batch: int, channels: int, head_dim: int, x_is_bf16: bool,
                 params: Optional[ScanParams] = None, *, dir_scale_ptr: int = 0,
                 memories_out_ptr: int = 0, stats_ptr: int = 0, stream_ptr: int = 0,
                 accumulate: bool = False, w_query_ptr: int = 0, skip_ptr: int = 0,
                 workspace_ptr: int = 0, workspace_bytes: int = 0) -> CParams:
    p = params or ScanParams()
    if p.impl not in IMPL:
        raise ValueError(f"impl must be one of {sorted(IMPL)}")
    return CParams(batch, channels, head_dim, DTYPE_BF16 if x_is_bf16 else DTYPE_F32,
                   p.gamma_eta, p.alpha_init, p.eta_bias, p.eps, p.knorm_eps, p.inj_inward,
                   p.spec_inward, p.kk_floor, dir_scale_ptr or None, memories_out_ptr or None,
                   p.gate_mode, p.forced_eta, p.forced_alpha, p.control_flags,
                   stats_ptr or None, IMPL[p.impl], 1 if accumulate else 0,
                   stream_ptr or None, w_query_ptr or None, skip_ptr or None,
                   workspace_ptr or None, workspace_bytes, int(p.wait_limit),
                   1 if p.withhold_first_copy else 0)


def _stream_ptr(stream) -> int:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _require_cuda(name, t, dtypes):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype not in dtypes:
        raise ValueError(f"{name} dtype {t.dtype} not in {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def scan_forward(x, memories0, head_dim: int, dirs: int = DIR_ALL, chunk: int = 0, out=None,
                 params: Optional[ScanParams] = None, dir_scale=None, memories_out=None,
                 stats=None, stream=None, accumulate: bool = False, w_query=None, skip=None,
                 workspace=None):
    """VisionHOPE operator: x [B][H][W][Cc] (bf16/fp32, CUDA) -> out [B][H][W][Cc] fp32.

    memories0: fp32 [4][Cc/head_dim][4d^2+2d] initial state per (route, head).
    Optional: dir_scale fp32 [4][Cc]; memories_out fp32 [B][4][nh][4d^2+2d];
    stats uint64/int64 [8] (accumulated).  accumulate=True adds to ``out``
    instead of overwriting it.  w_query fp32 [Cc][Cc] selects the VisionHOPE-exact
    readout (outer query projection shared by the routes) and skip fp32 [4][Cc] adds
    the channel-wise skip; the query planes live in ``workspace`` (uint8, at least
    vh_workspace_size bytes; allocated here when not given).  Runs on ``stream``
    (default: torch's current stream) asynchronously."""
    import torch
    _require_cuda("x", x, (torch.bfloat16, torch.float32))
    _require_cuda("memories0", memories0, (torch.float32,))
    B, H, W, Cc = x.shape
    nh = Cc // head_dim
    if memories0.numel() != 4 * nh * (4 * head_dim * head_dim + 2 * head_dim):
        raise ValueError("memories0 must hold [4][nh][4d^2+2d] floats")
    if out is None:
        if accumulate:
            raise ValueError("accumulate=True needs an out tensor")
        out = torch.empty((B, H, W, Cc), dtype=torch.float32, device=x.device)
    _require_cuda("out", out, (torch.float32,))
    if dir_scale is not None:
        _require_cuda("dir_scale", dir_scale, (torch.float32,))
    if memories_out is not None:
        _require_cuda("memories_out", memories_out, (torch.float32,))
    if stats is not None:
        _require_cuda("stats", stats, (torch.int64, torch.uint64) if hasattr(torch, "uint64") else (torch.int64,))
    if w_query is not None:
        _require_cuda("w_query", w_query, (torch.float32,))
    if skip is not None:
        _require_cuda("skip", skip, (torch.float32,))
    cp = make_cparams(B, Cc, head_dim, x.dtype == torch.bfloat16, params,
                      dir_scale_ptr=dir_scale.data_ptr() if dir_scale is not None else 0,
                      memories_out_ptr=memories_out.data_ptr() if memories_out is not None else 0,
                      stats_ptr=stats.data_ptr() if stats is not None else 0,
                      stream_ptr=_stream_ptr(stream), accumulate=accumulate,
                      w_query_ptr=w_query.data_ptr() if w_query is not None else 0,
                      skip_ptr=skip.data_ptr() if skip is not None else 0)
    need = lib().vh_workspace_size(ctypes.byref(cp), H, W, dirs, chunk)
    if need:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
        _require_cuda("workspace", workspace, (torch.uint8,))
        cp.workspace = workspace.data_ptr()
        cp.workspace_bytes = workspace.numel()
    _check(lib().vh_scan_forward(x.data_ptr(), memories0.data_ptr(), ctypes.byref(cp), H, W,
                                 dirs, chunk, out.data_ptr()))
    return out


def backward_workspace_size(x, head_dim: int, dirs: int = DIR_ALL, chunk: int = 0) -> int:
    """Bytes of workspace scan_backward needs for x's shape."""
    import torch
    B, H, W, Cc = x.shape
    cp = make_cparams(B, Cc, head_dim, x.dtype == torch.bfloat16, None)
    return int(lib().vh_backward_workspace_size(ctypes.byref(cp), H, W, dirs, chunk))


def scan_backward(x, memories0, head_dim: int, dout, dirs: int = DIR_ALL, chunk: int = 0,
                  params: Optional[ScanParams] = None, dir_scale=None, dmem_final=None,
                  dx=None, dmem0=None, workspace=None, stream=None, stats=None):
    """Outer gradients of scan_forward: (dx fp32 [B][H][W][Cc], dmem0 fp32 [4][nh][4d^2+2d])
    of <dout, out> + <dmem_final, memories_out> for the same x, memories0, params, dirs,
    chunk and dir_scale.  dmem_final (fp32 [B][4][nh][4d^2+2d]) may be None.  The
    workspace (uint8, at least backward_workspace_size bytes) is allocated here when not
    given.  Runs on ``stream`` asynchronously."""
    import torch
    _require_cuda("x", x, (torch.bfloat16, torch.float32))
    _require_cuda("memories0", memories0, (torch.float32,))
    _require_cuda("dout", dout, (torch.float32,))
    B, H, W, Cc = x.shape
    nh = Cc // head_dim
    if memories0.numel() != 4 * nh * (4 * head_dim * head_dim + 2 * head_dim):
        raise ValueError("memories0 must hold [4][nh][4d^2+2d] floats")
    if tuple(dout.shape) != (B, H, W, Cc):
        raise ValueError("dout must have x's shape")
    if dmem_final is not None:
        _require_cuda("dmem_final", dmem_final, (torch.float32,))
    if dir_scale is not None:
        _require_cuda("dir_scale", dir_scale, (torch.float32,))
    if dx is None:
        dx = torch.empty((B, H, W, Cc), dtype=torch.float32, device=x.device)
    if dmem0 is None:
        dmem0 = torch.empty_like(memories0)
    _require_cuda("dx", dx, (torch.float32,))
    _require_cuda("dmem0", dmem0, (torch.float32,))
    if stats is not None:
        _require_cuda("stats", stats, (torch.int64,))
    cp = make_cparams(B, Cc, head_dim, x.dtype == torch.bfloat16, params,
                      dir_scale_ptr=dir_scale.data_ptr() if dir_scale is not None else 0,
                      stats_ptr=stats.data_ptr() if stats is not None else 0,
                      stream_ptr=_stream_ptr(stream))
    need = lib().vh_backward_workspace_size(ctypes.byref(cp), H, W, dirs, chunk)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _require_cuda("workspace", workspace, (torch.uint8,))
    cp.workspace = workspace.data_ptr()
    cp.workspace_bytes = workspace.numel()
    _check(lib().vh_scan_backward(x.data_ptr(), memories0.data_ptr(), ctypes.byref(cp), H, W,
                                  dirs, chunk, dout.data_ptr(),
                                  dmem_final.data_ptr() if dmem_final is not None else None,
                                  dx.data_ptr(), dmem0.data_ptr()))
    return dx, dmem0


def block_forward(x, memories0, weights: dict, head_dim: int, params: Optional[ScanParams] = None,
                  w_query=None, skip=None, dir_scale=None, out=None, workspace=None,
                  stats=None, stream=None, ln_eps: float = 1e-5, f32_intermediates: bool = False):
    """One VisionHOPE block (Eq. (27), App. B.5): x fp32 [B][H][W][D] (CUDA) -> out.

    ``weights`` maps the fields of ``vh_block_weights`` to contiguous CUDA tensors: the
    four GEMM weights (w_in [D_m][D], w_out [D][D_m], w_ff1 [hidden][D], w_ff2
    [D][hidden]) bf16, the rest fp32.  The operator runs on D_m = w_in.shape[0] channels
    as heads of ``head_dim`` with memories0, the outer query w_query [D_m][D_m], the skip
    [4][D_m] and dir_scale [4][D_m] as in scan_forward.  The workspace (uint8, at least
    vh_block_workspace_size bytes) is allocated here when not given.  f32_intermediates
    selects the test mode that rounds no intermediate to bf16."""
    import torch
    _require_cuda("x", x, (torch.float32,))
    _require_cuda("memories0", memories0, (torch.float32,))
    B, H, W, D = x.shape
    for name in BLOCK_WEIGHT_NAMES:
        _require_cuda(name, weights[name],
                      (torch.bfloat16,) if name in BLOCK_GEMM_WEIGHTS else (torch.float32,))
    Dm = weights["w_in"].shape[0]
    hidden = weights["w_ff1"].shape[0]
    for t, name in ((w_query, "w_query"), (skip, "skip"), (dir_scale, "dir_scale")):
        if t is not None:
            _require_cuda(name, t, (torch.float32,))
    if out is None:
        out = torch.empty_like(x)
    _require_cuda("out", out, (torch.float32,))
    cw = CBlockWeights(D, hidden, ln_eps, *[weights[n].data_ptr() for n in BLOCK_WEIGHT_NAMES],
                       1 if f32_intermediates else 0)
    cp = make_cparams(B, Dm, head_dim, True, params,
                      dir_scale_ptr=dir_scale.data_ptr() if dir_scale is not None else 0,
                      stats_ptr=stats.data_ptr() if stats is not None else 0,
                      stream_ptr=_stream_ptr(stream),
                      w_query_ptr=w_query.data_ptr() if w_query is not None else 0,
                      skip_ptr=skip.data_ptr() if skip is not None else 0)
    need = lib().vh_block_workspace_size(ctypes.byref(cp), ctypes.byref(cw), H, W)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _require_cuda("workspace", workspace, (torch.uint8,))
    cp.workspace = workspace.data_ptr()
    cp.workspace_bytes = workspace.numel()
    _check(lib().vh_block_forward(x.data_ptr(), memories0.data_ptr(), ctypes.byref(cp),
                                  ctypes.byref(cw), H, W, out.data_ptr()))
    return out


def block_workspace_size(x, weights: dict, head_dim: int, with_query: bool = True,
                         f32_intermediates: bool = False) -> int:
    """Bytes of workspace block_forward needs for x's shape and these weights."""
    B, H, W, D = x.shape
    cp = make_cparams(B, weights["w_in"].shape[0], head_dim, True, None,
                      w_query_ptr=1 if with_query else 0)
    cw = CBlockWeights(D, weights["w_ff1"].shape[0], 1e-5, *([None] * len(BLOCK_WEIGHT_NAMES)),
                       1 if f32_intermediates else 0)
    return int(lib().vh_block_workspace_size(ctypes.byref(cp), ctypes.byref(cw), H, W))


def check(stats, stream=None):
    """Wait for `stream` and raise VhError if the counters in `stats` (the tensor passed
    to scan_forward) report an expired wait or a non-finite readout value."""
    import torch
    _require_cuda("stats", stats, (torch.int64,))
    _check(lib().vh_check(stats.data_ptr(), _stream_ptr(stream)))


def debug_gelu(a, stream=None):
    """bf16(GELU(a)) elementwise with the exact GELU the block's FFN1 epilogue applies."""
    import torch
    _require_cuda("a", a, (torch.float32,))
    a = a.contiguous()
    out = torch.empty(a.shape, dtype=torch.bfloat16, device=a.device)
    _check(lib().vh_debug_gelu(a.data_ptr(), out.data_ptr(), a.numel(), _stream_ptr(stream)))
    return out


def debug_permute(x, route: int, head_dim: int, stream=None):
    """Z_r = P_r(Z) for one route, gathered by the library's device index code."""
    import torch
    _require_cuda("x", x, (torch.bfloat16, torch.float32))
    B, H, W, Cc = x.shape
    seq = torch.empty((B, H * W, Cc), dtype=x.dtype, device=x.device)
    cp = make_cparams(B, Cc, head_dim, x.dtype == torch.bfloat16, None,
                      stream_ptr=_stream_ptr(stream))
    _check(lib().vh_debug_permute(x.data_ptr(), ctypes.byref(cp), H, W, route, seq.data_ptr()))
    return seq
