"""ctypes binding of libmuon_gb300.so (the C ABI declared in include/muon.h).

Argument marshalling only: torch tensors become device pointers and shapes, the
current torch CUDA stream becomes the cudaStream_t.  Every computation runs in the
library's CUDA kernels; there is no fallback.  Loading fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
# The in-tree build; MUON_GB300_LIB names another build of the same sources (for
# example one compiled with tuning defines through build.build(defines=..., out=...)).
LIB_PATH = os.environ.get("MUON_GB300_LIB") or os.path.join(HERE, "libmuon_gb300.so")

MUON_OK = 0
MUON_ERR_INVALID = -1
MUON_ERR_UNSUPPORTED = -2
MUON_ERR_WORKSPACE = -3
MUON_ERR_CUDA = -4
MUON_ERR_TIMEOUT = -5
MUON_ERR_NO_DEVICE = -6
MUON_ERR_NONFINITE = -7
MUON_DTYPE_F32 = 0
MUON_DTYPE_BF16 = 1
MUON_NS5_BF16 = 0
MUON_NS5_F32 = 1
MUON_BRANCH_ROWNORM = 0
MUON_BRANCH_NS5 = 1
MUON_DEBUG_STALL_PRODUCER = 1
MUON_DEBUG_NO_CLUSTER = 2
MUON_DEBUG_NO_OVERLAP = 4
MUON_DEBUG_TALL_CLUSTER = 8
MUON_DEBUG_NO_PAIR = 16

_NS5_MODES = {"bf16": MUON_NS5_BF16, "f32": MUON_NS5_F32}


class MuonError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({status_str(status)})")


MUON_SCALE_ADJUSTED_LR = 0
MUON_SCALE_UPDATE_NORM = 1
_SCALE_MODES = {"adjusted_lr": MUON_SCALE_ADJUSTED_LR, "update_norm": MUON_SCALE_UPDATE_NORM}


class MuonStepOptions(ctypes.Structure):
    _fields_ = [("scale_mode", ctypes.c_int), ("update_rms", ctypes.c_void_p), ("check_finite", ctypes.c_int)]


class MuonAdamwParam(ctypes.Structure):
    _fields_ = [("P", ctypes.c_void_p), ("G", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("numel", ctypes.c_int64), ("p_dtype", ctypes.c_int32), ("g_dtype", ctypes.c_int32)]


class MuonMatrix(ctypes.Structure):
    _fields_ = [("W", ctypes.c_void_p), ("G", ctypes.c_void_p), ("M", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("w_dtype", ctypes.c_int32), ("g_dtype", ctypes.c_int32)]


_lib = None


def load_library(path: Optional[str] = None):
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing (run __graft_entry__.build())")
    lib = ctypes.CDLL(p)
    vp, sz, i32, i64, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    mp = ctypes.POINTER(MuonMatrix)
    ptrs = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "muon_workspace_size": (sz, [mp, i32, i32]),
        "muon_momentum": (i32, [mp, i32, f32, vp, vp, sz, vp]),
        "muon_fro_norm": (i32, [mp, i32, vp, vp, sz, vp]),
        "muon_fro_norm_noalloc": (i32, [mp, i32, vp, vp]),
        "muon_ns5_batched": (i32, [mp, i32, i32, ptrs, i32, vp, sz, vp]),
        "muon_rownorm": (i32, [mp, i32, ptrs, vp, sz, vp]),
        "muon_apply": (i32, [mp, i32, ptrs, i32, f32, f32, f32, vp]),
        "muon_periodic_step": (i32, [mp, i32, i64, i32, f32, f32, f32, f32, i32, vp, sz, vp,
                                     ctypes.POINTER(ctypes.c_int)]),
        "muon_periodic_step_ex": (i32, [mp, i32, i64, i32, f32, f32, f32, f32, i32,
                                        ctypes.POINTER(MuonStepOptions), vp, sz, vp,
                                        ctypes.POINTER(ctypes.c_int)]),
        "muon_workspace_init": (i32, [vp, sz, vp]),
        "muon_check_status": (i32, [vp, sz, vp]),
        "muon_status_str": (ctypes.c_char_p, [i32]),
        "muon_abi_version": (i32, []),
        "muon_init": (i32, []),
        "muon_debug_set": (i32, [i32, i32]),
        "muon_profile_events": (i32, [ptrs, i32]),
        "muon_adamw_step": (i32, [ctypes.POINTER(MuonAdamwParam), i32, i64, f32, ctypes.c_double, ctypes.c_double,
                                  f32, f32, vp]),
        "muon_launch_count": (i32, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_str(status: int) -> str:
    return load_library().muon_status_str(status).decode()


def _check(fn: str, st: int):
    if st != MUON_OK:
        raise MuonError(fn, st)


def _dt(t: Optional[torch.Tensor]) -> int:
    if t is None:
        return MUON_DTYPE_BF16
    if t.dtype == torch.bfloat16:
        return MUON_DTYPE_BF16
    if t.dtype == torch.float32:
        return MUON_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def make_matrices(M: Sequence[torch.Tensor], W: Optional[Sequence[torch.Tensor]] = None,
                  G: Optional[Sequence[torch.Tensor]] = None):
    n = len(M)
    arr = (MuonMatrix * max(n, 1))()
    for i in range(n):
        m = M[i]
        if m.dim() != 2 or m.dtype != torch.float32:
            raise ValueError("M must be 2-D fp32")
        w = W[i] if W is not None else None
        g = G[i] if G is not None else None
        for t in (w, g):
            if t is not None and tuple(t.shape) != tuple(m.shape):
                raise ValueError("W, G and M must have the same shape")
        arr[i] = MuonMatrix(_ptr(w), _ptr(g), _ptr(m), int(m.shape[0]), int(m.shape[1]),
                            _dt(w if w is not None else (g if g is not None else None)), _dt(g if g is not None else w))
    return arr, n


def make_matrices_w(W: Sequence[torch.Tensor]):
    n = len(W)
    arr = (MuonMatrix * max(n, 1))()
    for i, w in enumerate(W):
        if w.dim() != 2:
            raise ValueError("W must be 2-D")
        arr[i] = MuonMatrix(_ptr(w), None, None, int(w.shape[0]), int(w.shape[1]), _dt(w), _dt(w))
    return arr, n


def _shape_matrices(shapes: Sequence[Sequence[int]]):
    n = len(shapes)
    arr = (MuonMatrix * max(n, 1))()
    for i, (r, c) in enumerate(shapes):
        arr[i] = MuonMatrix(None, None, None, int(r), int(c), MUON_DTYPE_BF16, MUON_DTYPE_BF16)
    return arr, n


def _ptr_array(ts: Sequence[torch.Tensor]):
    a = (ctypes.c_void_p * max(len(ts), 1))()
    for i, t in enumerate(ts):
        a[i] = _ptr(t)
    return a


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------

def muon_workspace_size(shapes: Sequence[Sequence[int]], ns5_mode: str = "bf16") -> int:
    arr, n = _shape_matrices(shapes)
    v = load_library().muon_workspace_size(arr, n, _NS5_MODES[ns5_mode])
    if v == ctypes.c_size_t(-1).value:
        raise MuonError("muon_workspace_size", MUON_ERR_INVALID)
    return int(v)


def muon_workspace_init(ws: torch.Tensor, stream=None):
    _check("muon_workspace_init", load_library().muon_workspace_init(_ptr(ws), ws.numel(), _stream(stream)))


def alloc_workspace(shapes: Sequence[Sequence[int]], ns5_mode: str = "bf16", device=None) -> torch.Tensor:
    nbytes = max(muon_workspace_size(shapes, ns5_mode), 256)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
    muon_workspace_init(ws)
    return ws


def muon_check_status(ws: torch.Tensor, stream=None) -> int:
    return int(load_library().muon_check_status(_ptr(ws), ws.numel(), _stream(stream)))


def muon_momentum(G: Sequence[torch.Tensor], M: Sequence[torch.Tensor], mu: float,
                  fro_sq_out: Optional[torch.Tensor] = None, ws: Optional[torch.Tensor] = None, stream=None):
    arr, n = make_matrices(M, None, G)
    _check("muon_momentum", load_library().muon_momentum(
        arr, n, mu, _ptr(fro_sq_out), _ptr(ws), ws.numel() if ws is not None else 0, _stream(stream)))


def muon_fro_norm(M: Sequence[torch.Tensor], fro_out: torch.Tensor, ws: torch.Tensor, stream=None):
    arr, n = make_matrices(M)
    _check("muon_fro_norm", load_library().muon_fro_norm(arr, n, _ptr(fro_out), _ptr(ws), ws.numel(),
                                                         _stream(stream)))


def muon_fro_norm_noalloc(M: Sequence[torch.Tensor], fro_out: torch.Tensor, stream=None):
    """||M_i||_F without a workspace (scratch fixed inside the library)."""
    arr, n = make_matrices(M)
    _check("muon_fro_norm_noalloc", load_library().muon_fro_norm_noalloc(arr, n, _ptr(fro_out), _stream(stream)))


def muon_ns5_batched(M: Sequence[torch.Tensor], O: Sequence[torch.Tensor], ws: torch.Tensor,
                     ns5_mode: str = "bf16", stream=None):
    arr, n = make_matrices(M)
    o_dt = _dt(O[0]) if O else MUON_DTYPE_BF16
    _check("muon_ns5_batched", load_library().muon_ns5_batched(
        arr, n, _NS5_MODES[ns5_mode], _ptr_array(O), o_dt, _ptr(ws), ws.numel(), _stream(stream)))


def muon_rownorm(M: Sequence[torch.Tensor], R: Sequence[torch.Tensor], ws: torch.Tensor, stream=None):
    arr, n = make_matrices(M)
    _check("muon_rownorm", load_library().muon_rownorm(arr, n, _ptr_array(R), _ptr(ws), ws.numel(),
                                                       _stream(stream)))


def muon_apply(W: Sequence[torch.Tensor], U: Sequence[torch.Tensor], scale_mul: float, eta: float, lam: float,
               stream=None):
    arr, n = make_matrices_w(W)
    u_dt = _dt(U[0]) if U else MUON_DTYPE_BF16
    _check("muon_apply", load_library().muon_apply(arr, n, _ptr_array(U), u_dt, scale_mul, eta, lam,
                                                   _stream(stream)))


def muon_periodic_step(W: Sequence[torch.Tensor], G: Sequence[torch.Tensor], M: Sequence[torch.Tensor],
                       step: int, ws: torch.Tensor, K: int = 3, gamma: float = 0.15, mu: float = 0.95,
                       eta: float = 0.02, lam: float = 0.01, ns5_mode: str = "bf16", stream=None,
                       scale_mode: str = "adjusted_lr", update_rms: Optional[torch.Tensor] = None,
                       check_finite: bool = False) -> int:
    """One Periodic Row-wise Muon step; returns MUON_BRANCH_NS5 or MUON_BRANCH_ROWNORM.
    scale_mode "update_norm" selects Eq. (6); update_rms (n fp32 on the device) receives
    the RMS of each matrix's direction; check_finite makes muon_check_status report
    MUON_ERR_NONFINITE when a momentum norm of this step was NaN or Inf."""
    arr, n = make_matrices(M, W, G)
    br = ctypes.c_int(-1)
    lib = load_library()
    if scale_mode == "adjusted_lr" and update_rms is None and not check_finite:
        st = lib.muon_periodic_step(arr, n, int(step), int(K), gamma, mu, eta, lam, _NS5_MODES[ns5_mode],
                                    _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(br))
    else:
        opts = MuonStepOptions(_SCALE_MODES[scale_mode], _ptr(update_rms), 1 if check_finite else 0)
        st = lib.muon_periodic_step_ex(arr, n, int(step), int(K), gamma, mu, eta, lam, _NS5_MODES[ns5_mode],
                                       ctypes.byref(opts), _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(br))
    _check("muon_periodic_step", st)
    return br.value


def periodic_step_prepared(arr, n: int, step: int, ws: torch.Tensor, K: int, gamma: float, mu: float, eta: float,
                           lam: float, ns5_mode: str, stream=None) -> int:
    """muon_periodic_step on a matrix array built once by make_matrices and kept by the
    caller (the stateful wrapper updates only the gradient pointers between steps)."""
    br = ctypes.c_int(-1)
    st = load_library().muon_periodic_step(arr, n, int(step), int(K), gamma, mu, eta, lam, _NS5_MODES[ns5_mode],
                                           _ptr(ws), ws.numel(), _stream(stream), ctypes.byref(br))
    _check("muon_periodic_step", st)
    return br.value


def muon_init():
    """One-time set-up of the current device and calling thread (makes the first step capturable)."""
    _check("muon_init", load_library().muon_init())


def muon_debug_set(flags: int = 0, timeout_ms: int = 0):
    _check("muon_debug_set", load_library().muon_debug_set(int(flags), int(timeout_ms)))


def muon_profile_events(events: Sequence) -> None:
    """events: up to 5 torch.cuda.Event (or None) recorded at the step's phase boundaries."""
    arr = (ctypes.c_void_p * 5)()
    for i, e in enumerate(events):
        arr[i] = None if e is None else int(e.cuda_event)
    _check("muon_profile_events", load_library().muon_profile_events(arr, len(events)))


def muon_launch_count() -> int:
    return int(load_library().muon_launch_count())


def muon_adamw_step(P: Sequence[torch.Tensor], G: Sequence[torch.Tensor], m: Sequence[torch.Tensor],
                    v: Sequence[torch.Tensor], t: int, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                    eps: float = 1e-8, weight_decay: float = 0.0, stream=None):
    """AdamW on parameters Muon does not take (any shape; m, v fp32 of the same size)."""
    n = len(P)
    arr = (MuonAdamwParam * max(n, 1))()
    for i in range(n):
        if not (P[i].numel() == G[i].numel() == m[i].numel() == v[i].numel()):
            raise ValueError("P, G, m, v must have the same number of elements")
        if m[i].dtype != torch.float32 or v[i].dtype != torch.float32:
            raise ValueError("AdamW moments are fp32")
        arr[i] = MuonAdamwParam(_ptr(P[i]), _ptr(G[i]), _ptr(m[i]), _ptr(v[i]), int(P[i].numel()),
                                _dt(P[i]), _dt(G[i]))
    _check("muon_adamw_step", load_library().muon_adamw_step(arr, n, int(t), lr, beta1, beta2, eps,
                                                             weight_decay, _stream(stream)))
