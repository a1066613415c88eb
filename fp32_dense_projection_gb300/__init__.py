"""GB300 (sm_103a) dense projection GEMMs -- Python binding of ``libdp_gb300.so``.

The functions here marshal torch tensors into the C ABI of ``include/dp_gemm.h``
(pointers, sizes, leading dimensions, the current CUDA stream) and return the
output tensor.  Every step of the computation runs in the library's CUDA
kernels; there is no Python or CPU fallback.  If the library is not built, the
first call raises.

  dp_gemm_fwd(X, W)        Y  = X W^T       X[T,K], W[N,K]  (bf16)  -> Y[T,N]
  dp_gemm_dgrad(dY, W)     dX = dY W        dY[T,N], W[N,K] (bf16)  -> dX[T,K]
  dp_gemm_wgrad(dY, X)     dW = dY^T X      dY[T,N], X[T,K] (bf16)  -> dW[N,K]
  dp_gemm_bwd(dY, X, W)    (dX, dW) of one layer: two single-op calls, or one
                           co-scheduled launch over both problems' tiles
  router_fwd / router_dgrad / router_wgrad: the same on FP32 operands through
  BF16x3 emulation, FP32 output.

Outputs are bf16 (``out_dtype=torch.bfloat16``) or fp32 for the BF16 ops.  An
``out=`` tensor may be a column slice of a wider buffer (padded row stride).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdp_gb300.so")

DP_OUT_BF16, DP_OUT_F32 = 0, 1
OP_FWD, OP_DGRAD, OP_WGRAD, OP_ROUTER_FWD, OP_ROUTER_DGRAD, OP_ROUTER_WGRAD = range(6)
OP_NAMES = {"fwd": OP_FWD, "dgrad": OP_DGRAD, "wgrad": OP_WGRAD,
            "router_fwd": OP_ROUTER_FWD, "router_dgrad": OP_ROUTER_DGRAD, "router_wgrad": OP_ROUTER_WGRAD}

_lib = None
_lock = threading.Lock()


class DPError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "block_m", "block_n", "block_k", "stages", "splits", "raster_group", "grid",
        "a_mn_major", "b_mn_major", "swap_ab", "cta_pair", "raster_rows", "stream_k")] + [(n, ctypes.c_int64) for n in (
        "gemm_m", "gemm_n", "gemm_k", "tiles_m", "tiles_n", "k_blocks", "units", "full_units")] + [
        ("workspace_bytes", ctypes.c_uint64), ("model_us", ctypes.c_double),
        ("batch", ctypes.c_int64), ("tiles", ctypes.c_int64), ("weight_kn", ctypes.c_int32),
        ("program", ctypes.c_int32), ("atomic", ctypes.c_int32), ("blocks_per_stage", ctypes.c_int32),
        ("cluster_sum", ctypes.c_int32)]


class BwdPlanInfo(ctypes.Structure):
    _fields_ = [("fused", ctypes.c_int32), ("wgrad_first", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("blocks_per_stage", ctypes.c_int32), ("model_us", ctypes.c_double), ("separate_us", ctypes.c_double),
                ("workspace_bytes", ctypes.c_uint64), ("dgrad", PlanInfo), ("wgrad", PlanInfo)]


def lib():
    """Load libdp_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m fp32_dense_projection_gb300.build` (or __graft_entry__.build())")
        L = ctypes.CDLL(LIB_PATH)
        P, I, Z, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int
        tail = [I, I, I, S, S, P, Z, P]          # T N K out deterministic ws ws_bytes stream
        rtail = [I, I, I, S, P, Z, P]            # T N K deterministic ws ws_bytes stream
        for name in ("dp_gemm_fwd", "dp_gemm_dgrad", "dp_gemm_wgrad"):
            getattr(L, name).argtypes = [P, P, P] + tail
            getattr(L, name + "_ex").argtypes = [P, I, P, I, P, I] + tail
        for name in ("router_fwd", "router_dgrad", "router_wgrad"):
            getattr(L, name).argtypes = [P, P, P] + rtail
            getattr(L, name + "_ex").argtypes = [P, I, P, I, P, I] + rtail
        L.dp_plan_query.argtypes = [S, I, I, I, S, S, ctypes.POINTER(PlanInfo)]
        L.dp_plan_query_ex.argtypes = [S, I, I, I, S, S, S, ctypes.POINTER(PlanInfo)]
        L.dp_plan_query_batched.argtypes = [S, I, I, I, I, S, S, S, ctypes.POINTER(PlanInfo)]
        L.dp_workspace_size_batched.argtypes = [S, I, I, I, I, S, S, S, ctypes.POINTER(ctypes.c_size_t)]
        btail = [I, I, I, I, S, S, P, Z, P]      # B T N K out deterministic ws ws_bytes stream
        L.dp_gemm_fwd_batched.argtypes = [P, I, I, P, I, I, S, P, I, I] + btail
        L.dp_gemm_dgrad_batched.argtypes = [P, I, I, P, I, I, S, P, I, I] + btail
        L.dp_gemm_wgrad_batched.argtypes = [P, I, I, P, I, I, P, I, I, S] + btail
        L.dp_workspace_size.argtypes = [S, I, I, I, S, S, ctypes.POINTER(ctypes.c_size_t)]
        L.dp_gemm_bwd.argtypes = [P, I, P, I, P, I, P, I, S, P, I, S, I, I, I, S, P, Z, P]
        L.dp_plan_query_bwd.argtypes = [I, I, I, S, S, S, ctypes.POINTER(BwdPlanInfo)]
        L.dp_workspace_size_bwd.argtypes = [I, I, I, S, S, S, ctypes.POINTER(ctypes.c_size_t)]
        L.dp_init.argtypes = [S]
        L.dp_device_error.argtypes = [S]
        L.dp_status_string.argtypes = [S]
        L.dp_status_string.restype = ctypes.c_char_p
        L.dp_version.argtypes = []
        L.dp_wait_probe.argtypes = [ctypes.c_uint64, S, P]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().dp_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - library missing
        return f"status {status}"


def _check(status: int, what: str):
    if status != 0:
        raise DPError(status, what)


def plan(op, T: int, N: int, K: int, out_f32: bool = False, sm_count: int = 0, deterministic: bool = True) -> dict:
    """The library's plan for a call (pure function of the shape, SM count and the
    deterministic flag)."""
    op = OP_NAMES.get(op, op)
    info = PlanInfo()
    _check(lib().dp_plan_query_ex(int(op), T, N, K, int(bool(out_f32)), int(bool(deterministic)), int(sm_count),
                                  ctypes.byref(info)), "dp_plan_query_ex")
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_ if not name.startswith("reserved")}


def plan_batched(op, B: int, T: int, N: int, K: int, out_f32: bool = False, weight_kn: bool = False,
                 sm_count: int = 0) -> dict:
    """The plan of a batched BF16 call (op "fwd" / "dgrad" / "wgrad")."""
    op = OP_NAMES.get(op, op)
    info = PlanInfo()
    _check(lib().dp_plan_query_batched(int(op), B, T, N, K, int(bool(out_f32)), int(bool(weight_kn)),
                                       int(sm_count), ctypes.byref(info)), "dp_plan_query_batched")
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_ if not name.startswith("reserved")}


def workspace_size_batched(op, B: int, T: int, N: int, K: int, out_f32: bool = False, weight_kn: bool = False,
                           sm_count: int = 0) -> int:
    op = OP_NAMES.get(op, op)
    n = ctypes.c_size_t(0)
    _check(lib().dp_workspace_size_batched(int(op), B, T, N, K, int(bool(out_f32)), int(bool(weight_kn)),
                                           int(sm_count), ctypes.byref(n)), "dp_workspace_size_batched")
    return int(n.value)


def workspace_size(op, T: int, N: int, K: int, out_f32: bool = False, sm_count: int = 0) -> int:
    op = OP_NAMES.get(op, op)
    n = ctypes.c_size_t(0)
    _check(lib().dp_workspace_size(int(op), T, N, K, int(bool(out_f32)), int(sm_count), ctypes.byref(n)),
           "dp_workspace_size")
    return int(n.value)


def _info_dict(info: PlanInfo) -> dict:
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_ if not name.startswith("reserved")}


def plan_bwd(T: int, N: int, K: int, dx_f32: bool = False, dw_f32: bool = False, sm_count: int = 0) -> dict:
    """The backward pass's plan: {"fused", "wgrad_first", "grid", "blocks_per_stage", "model_us",
    "separate_us", "workspace_bytes", "dgrad": {...}, "wgrad": {...}}."""
    info = BwdPlanInfo()
    _check(lib().dp_plan_query_bwd(T, N, K, int(bool(dx_f32)), int(bool(dw_f32)), int(sm_count),
                                   ctypes.byref(info)), "dp_plan_query_bwd")
    out = {name: getattr(info, name) for name, _ in BwdPlanInfo._fields_[:7] if name != "reserved"}
    out["dgrad"], out["wgrad"] = _info_dict(info.dgrad), _info_dict(info.wgrad)
    return out


def workspace_size_bwd(T: int, N: int, K: int, dx_f32: bool = False, dw_f32: bool = False,
                       sm_count: int = 0) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().dp_workspace_size_bwd(T, N, K, int(bool(dx_f32)), int(bool(dw_f32)), int(sm_count),
                                       ctypes.byref(n)), "dp_workspace_size_bwd")
    return int(n.value)


def init(device: int = -1):
    _check(lib().dp_init(int(device)), "dp_init")


def device_error(clear: bool = True) -> int:
    """Synchronise and return the library's device fault status (0 = none)."""
    return int(lib().dp_device_error(int(bool(clear))))


def wait_probe(limit_ns: int, arrive: bool = False, stream=None):
    """Enqueue the library's bounded-wait probe (one CTA waiting on a barrier that
    nothing arrives on, or that it arrived on itself): a wait that runs out after
    ``limit_ns`` shows up as ``device_error() == 7`` (DP_ERR_TIMEOUT)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _check(lib().dp_wait_probe(int(limit_ns), int(bool(arrive)), _stream(dev, stream)), "dp_wait_probe")


# ------------------------------------------------------------------ workspace

class Workspace:
    """A caller-owned device workspace that grows on demand.

    The library uses it as scratch (split partials, the router's bf16 operand
    copies) and needs no initial value in it.
    """

    def __init__(self, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else device)
        self.buf = None

    def get(self, nbytes: int):
        if nbytes == 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        return self.buf


_workspaces: dict = {}


def _default_workspace(device: torch.device) -> Workspace:
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    ws = _workspaces.get(key)
    if ws is None:
        ws = _workspaces[key] = Workspace(device.index)
    return ws


# --------------------------------------------------------------- marshalling

def _ld(t: torch.Tensor) -> int:
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise ValueError("operands must be 2-D with unit column stride")
    if t.size(0) <= 1:
        return max(t.stride(0), t.size(1))
    return t.stride(0)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device: torch.device, stream):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ws(op, T, N, K, out_f32, device, workspace):
    # a caller's workspace goes straight through (the library checks its size)
    buf = _default_workspace(device).get(workspace_size(op, T, N, K, out_f32)) if workspace is None else workspace
    nbytes = 0 if buf is None else buf.numel() * buf.element_size()
    return buf, nbytes


def _gemm(op: int, name: str, a: torch.Tensor, b: torch.Tensor, out_shape, out, out_dtype, deterministic,
          workspace, stream, T, N, K):
    router = op >= OP_ROUTER_FWD
    in_dtype = torch.float32 if router else torch.bfloat16
    if a.dtype != in_dtype or b.dtype != in_dtype:
        raise TypeError(f"{name}: operands must be {in_dtype}")
    if not (a.is_cuda and b.is_cuda):
        raise ValueError(f"{name}: operands must be CUDA tensors")
    device = a.device
    if router:
        out_dtype = torch.float32
    if out is None:
        out = torch.empty(out_shape, dtype=out_dtype, device=device)
    elif tuple(out.shape) != tuple(out_shape) or out.dtype != out_dtype:
        raise ValueError(f"{name}: out must be {tuple(out_shape)} {out_dtype}")
    out_f32 = out.dtype == torch.float32
    buf, nbytes = _ws(op, T, N, K, out_f32, device, workspace)
    fn = getattr(lib(), name + "_ex")

    def call():
        st = _stream(device, stream)
        if router:
            return fn(_ptr(a), _ld(a), _ptr(b), _ld(b), _ptr(out), _ld(out), T, N, K, int(bool(deterministic)),
                      _ptr(buf), nbytes, st)
        return fn(_ptr(a), _ld(a), _ptr(b), _ld(b), _ptr(out), _ld(out), T, N, K,
                  DP_OUT_F32 if out_f32 else DP_OUT_BF16, int(bool(deterministic)), _ptr(buf), nbytes, st)

    if device.index == torch.cuda.current_device():
        status = call()
    else:
        with torch.cuda.device(device):
            status = call()
    _check(status, name)
    return out


def dp_gemm_fwd(X, W, out=None, out_dtype=torch.bfloat16, deterministic=True, workspace=None, stream=None):
    """Y[T,N] = X[T,K] W[N,K]^T (bf16 in, FP32 accumulate, bf16 or fp32 out)."""
    T, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("dp_gemm_fwd: W must be N x K")
    return _gemm(OP_FWD, "dp_gemm_fwd", X, W, (T, N), out, out_dtype, deterministic, workspace, stream, T, N, K)


def dp_gemm_dgrad(dY, W, out=None, out_dtype=torch.bfloat16, deterministic=True, workspace=None, stream=None):
    """dX[T,K] = dY[T,N] W[N,K]."""
    T, N = dY.shape
    K = W.shape[1]
    if W.shape[0] != N:
        raise ValueError("dp_gemm_dgrad: W must be N x K")
    return _gemm(OP_DGRAD, "dp_gemm_dgrad", dY, W, (T, K), out, out_dtype, deterministic, workspace, stream,
                 T, N, K)


def dp_gemm_wgrad(dY, X, out=None, out_dtype=torch.bfloat16, deterministic=True, workspace=None, stream=None):
    """dW[N,K] = dY[T,N]^T X[T,K] (contraction over the T tokens)."""
    T, N = dY.shape
    K = X.shape[1]
    if X.shape[0] != T:
        raise ValueError("dp_gemm_wgrad: X must be T x K")
    return _gemm(OP_WGRAD, "dp_gemm_wgrad", dY, X, (N, K), out, out_dtype, deterministic, workspace, stream,
                 T, N, K)


def dp_gemm_bwd(dY, X, W, dX=None, dW=None, dx_dtype=torch.bfloat16, dw_dtype=torch.bfloat16,
                deterministic=True, workspace=None, stream=None):
    """(dX[T,K] = dY W, dW[N,K] = dY^T X) of one layer in one call: the two single-op
    calls, or one co-scheduled launch over both problems' whole-K tiles."""
    T, N = dY.shape
    K = X.shape[1]
    if X.shape[0] != T or tuple(W.shape) != (N, K):
        raise ValueError("dp_gemm_bwd: dY must be T x N, X T x K and W N x K")
    for t, nm in ((dY, "dY"), (X, "X"), (W, "W")):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"dp_gemm_bwd: {nm} must be a CUDA bfloat16 tensor")
    device = dY.device
    if dX is None:
        dX = torch.empty((T, K), dtype=dx_dtype, device=device)
    elif tuple(dX.shape) != (T, K) or dX.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("dp_gemm_bwd: dX must be T x K, bf16 or fp32")
    if dW is None:
        dW = torch.empty((N, K), dtype=dw_dtype, device=device)
    elif tuple(dW.shape) != (N, K) or dW.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("dp_gemm_bwd: dW must be N x K, bf16 or fp32")
    dx32, dw32 = dX.dtype == torch.float32, dW.dtype == torch.float32
    if workspace is None:
        workspace = _default_workspace(device).get(workspace_size_bwd(T, N, K, dx32, dw32))
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()

    def call():
        return lib().dp_gemm_bwd(_ptr(dY), _ld(dY), _ptr(X), _ld(X), _ptr(W), _ld(W), _ptr(dX), _ld(dX),
                                 DP_OUT_F32 if dx32 else DP_OUT_BF16, _ptr(dW), _ld(dW),
                                 DP_OUT_F32 if dw32 else DP_OUT_BF16, T, N, K, int(bool(deterministic)),
                                 _ptr(workspace), nbytes, _stream(device, stream))

    if device.index == torch.cuda.current_device():
        status = call()
    else:
        with torch.cuda.device(device):
            status = call()
    _check(status, "dp_gemm_bwd")
    return dX, dW


def router_fwd(X, W, out=None, deterministic=True, workspace=None, stream=None):
    """FP32 router forward through BF16x3: Y[T,E] = X[T,H] W[E,H]^T."""
    T, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("router_fwd: W must be E x H")
    return _gemm(OP_ROUTER_FWD, "router_fwd", X, W, (T, N), out, torch.float32, deterministic, workspace,
                 stream, T, N, K)


def router_dgrad(dY, W, out=None, deterministic=True, workspace=None, stream=None):
    """FP32 router input gradient through BF16x3: dX[T,H] = dY[T,E] W[E,H]."""
    T, N = dY.shape
    K = W.shape[1]
    if W.shape[0] != N:
        raise ValueError("router_dgrad: W must be E x H")
    return _gemm(OP_ROUTER_DGRAD, "router_dgrad", dY, W, (T, K), out, torch.float32, deterministic, workspace,
                 stream, T, N, K)


def router_wgrad(dY, X, out=None, deterministic=True, workspace=None, stream=None):
    """FP32 router weight gradient through BF16x3: dW[E,H] = dY[T,E]^T X[T,H]."""
    T, N = dY.shape
    K = X.shape[1]
    if X.shape[0] != T:
        raise ValueError("router_wgrad: X must be T x H")
    return _gemm(OP_ROUTER_WGRAD, "router_wgrad", dY, X, (N, K), out, torch.float32, deterministic, workspace,
                 stream, T, N, K)


def _bview(t: torch.Tensor, name: str):
    """(leading dimension, batch stride) of a [B, rows, cols] view with unit column stride."""
    if t.dim() != 3 or (t.size(2) > 1 and t.stride(2) != 1):
        raise ValueError(f"{name}: operands must be [B, rows, cols] views with unit column stride")
    ld = t.stride(1) if t.size(1) > 1 else t.size(2)
    bs = t.stride(0) if t.size(0) > 1 else t.size(1) * ld
    return ld, bs


def _batched(op: int, name: str, a, b, out, out_shape, out_dtype, weight_kn, deterministic, workspace, stream,
             B, T, N, K):
    for t, nm in ((a, "first operand"), (b, "second operand")):
        if t.dtype != torch.bfloat16 or not t.is_cuda:
            raise TypeError(f"{name}: {nm} must be a CUDA bfloat16 tensor")
    device = a.device
    if out is None:
        out = torch.empty(out_shape, dtype=out_dtype, device=device)
    elif tuple(out.shape) != tuple(out_shape) or out.dtype != out_dtype:
        raise ValueError(f"{name}: out must be {tuple(out_shape)} {out_dtype}")
    out_f32 = out.dtype == torch.float32
    if workspace is None:
        workspace = _default_workspace(device).get(workspace_size_batched(op, B, T, N, K, out_f32, weight_kn))
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    (lda, bsa), (ldb, bsb), (ldo, bso) = _bview(a, name), _bview(b, name), _bview(out, name)
    fn = getattr(lib(), name)
    code = DP_OUT_F32 if out_f32 else DP_OUT_BF16

    def call():
        st = _stream(device, stream)
        if op == OP_WGRAD:
            return fn(_ptr(a), lda, bsa, _ptr(b), ldb, bsb, _ptr(out), ldo, bso, int(bool(weight_kn)), B, T, N, K,
                      code, int(bool(deterministic)), _ptr(workspace), nbytes, st)
        return fn(_ptr(a), lda, bsa, _ptr(b), ldb, bsb, int(bool(weight_kn)), _ptr(out), ldo, bso, B, T, N, K,
                  code, int(bool(deterministic)), _ptr(workspace), nbytes, st)

    if device.index == torch.cuda.current_device():
        status = call()
    else:
        with torch.cuda.device(device):
            status = call()
    _check(status, name)
    return out


def dp_gemm_fwd_batched(X, W, out=None, out_dtype=torch.bfloat16, weight_layout="nk", deterministic=True,
                        workspace=None, stream=None):
    """Y[b] = X[b] W[b]^T for each b: X [B,T,K]; W [B,N,K] ("nk") or [B,K,N] ("kn"); Y [B,T,N]."""
    kn = _layout(weight_layout)
    B, T, K = X.shape
    N = W.shape[2] if kn else W.shape[1]
    if W.shape[0] != B or (W.shape[1] if kn else W.shape[2]) != K:
        raise ValueError("dp_gemm_fwd_batched: W does not match X")
    return _batched(OP_FWD, "dp_gemm_fwd_batched", X, W, out, (B, T, N), out_dtype, kn, deterministic,
                    workspace, stream, B, T, N, K)


def dp_gemm_dgrad_batched(dY, W, out=None, out_dtype=torch.bfloat16, weight_layout="nk", deterministic=True,
                          workspace=None, stream=None):
    """dX[b] = dY[b] W[b]: dY [B,T,N]; W [B,N,K] ("nk") or [B,K,N] ("kn"); dX [B,T,K]."""
    kn = _layout(weight_layout)
    B, T, N = dY.shape
    K = W.shape[1] if kn else W.shape[2]
    if W.shape[0] != B or (W.shape[2] if kn else W.shape[1]) != N:
        raise ValueError("dp_gemm_dgrad_batched: W does not match dY")
    return _batched(OP_DGRAD, "dp_gemm_dgrad_batched", dY, W, out, (B, T, K), out_dtype, kn, deterministic,
                    workspace, stream, B, T, N, K)


def dp_gemm_wgrad_batched(dY, X, out=None, out_dtype=torch.bfloat16, weight_layout="nk", deterministic=True,
                          workspace=None, stream=None):
    """dW[b] = dY[b]^T X[b]: dY [B,T,N]; X [B,T,K]; dW [B,N,K] ("nk") or [B,K,N] ("kn")."""
    kn = _layout(weight_layout)
    B, T, N = dY.shape
    K = X.shape[2]
    if X.shape[0] != B or X.shape[1] != T:
        raise ValueError("dp_gemm_wgrad_batched: X does not match dY")
    return _batched(OP_WGRAD, "dp_gemm_wgrad_batched", dY, X, out, (B, K, N) if kn else (B, N, K), out_dtype, kn,
                    deterministic, workspace, stream, B, T, N, K)


def _layout(weight_layout) -> bool:
    if weight_layout not in ("nk", "kn"):
        raise ValueError('weight_layout must be "nk" ([N, K] weights) or "kn" ([K, N])')
    return weight_layout == "kn"


OPS = {"fwd": dp_gemm_fwd, "dgrad": dp_gemm_dgrad, "wgrad": dp_gemm_wgrad,
       "router_fwd": router_fwd, "router_dgrad": router_dgrad, "router_wgrad": router_wgrad}


def dp_gemm_wgrad_noalloc(dY, X, out, out_dtype=None, deterministic=True, stream=None):
    """Weight gradient through the entry point that allocates nothing.

    For callers that cannot allocate device memory (a runtime that pre-reserves all
    memory, a host that forbids cudaMalloc on its hot path): the split scratch lives
    in a 64 MiB array inside the library.
    ``out`` must be given (the caller owns every buffer).  Calls on different streams
    must not overlap: they share the one scratch array.
    """
    T, N = dY.shape
    K = X.shape[1]
    if X.shape[0] != T or tuple(out.shape) != (N, K):
        raise ValueError("dp_gemm_wgrad_noalloc: dY[T,N], X[T,K], out[N,K]")
    if dY.dtype != torch.bfloat16 or X.dtype != torch.bfloat16:
        raise TypeError("dp_gemm_wgrad_noalloc: operands must be bf16")
    if out.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("dp_gemm_wgrad_noalloc: out must be float32 or bfloat16")
    if out_dtype is not None and out.dtype != out_dtype:
        raise TypeError(f"dp_gemm_wgrad_noalloc: out is {out.dtype}, out_dtype says {out_dtype}")
    if not (dY.is_cuda and X.is_cuda and out.is_cuda) or not (dY.device == X.device == out.device):
        raise ValueError("dp_gemm_wgrad_noalloc: dY, X and out must be CUDA tensors on one device")
    L = lib()
    fn = L.dp_gemm_wgrad_noalloc
    P, I, S = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [P, I, P, I, P, I, I, I, I, S, S, P]
    out_f32 = out.dtype == torch.float32
    with torch.cuda.device(dY.device):
        status = fn(_ptr(dY), _ld(dY), _ptr(X), _ld(X), _ptr(out), _ld(out), T, N, K,
                    DP_OUT_F32 if out_f32 else DP_OUT_BF16, int(bool(deterministic)), _stream(dY.device, stream))
    _check(status, "dp_gemm_wgrad_noalloc")
    return out
