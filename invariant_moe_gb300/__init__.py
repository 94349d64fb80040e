"""Python binding of libbimoe.so, the batch-invariant MoE hot path for GB300.

Argument marshalling only: every function checks tensor dtypes / devices /
contiguity, passes raw device pointers and the current CUDA stream to the C
ABI declared in ``include/bimoe.h``, and raises on a non-zero status.  All
arithmetic runs in the library's CUDA kernels; there is no CPU fallback.  If
the library is missing the first call raises ``RuntimeError`` -- build it with
``python -m invariant_moe_gb300._build`` (or ``__graft_entry__.build()``).

Names follow the C entry points: ``bi_router_gemm``, ``bi_topk``,
``bi_moe_forward`` and the per-stage calls.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbimoe.so")

BI_OK = 0
STATUS = {0: "BI_OK", 1: "BI_ERR_INVALID_ARG", 2: "BI_ERR_UNSUPPORTED", 3: "BI_ERR_WORKSPACE",
          4: "BI_ERR_CUDA", 5: "BI_ERR_DEVICE"}
DEVERR = {0: "none", 1: "expert id out of range", 2: "repeated expert in a row",
          3: "bounded wait timed out", 4: "offsets / perm are not a grouping of the pairs"}

# every symbol include/bimoe.h declares (checked by the CPU test-suite)
EXPORTS = [
    "bi_status_str", "bi_last_error_message", "bi_version", "bi_device_error",
    "bi_cast_bf16_to_f32", "bi_router_gemm", "bi_router_gemm_schedule",
    "bi_router_gemm_splitk_negctl", "bi_topk", "bi_moe_workspace_bytes", "bi_moe_forward",
    "bi_moe_permute_workspace_bytes", "bi_moe_permute", "bi_moe_gather",
    "bi_moe_gate_up", "bi_moe_down", "bi_moe_combine", "bi_moe_combine_consume", "bi_moe_forward_noalloc",
    "bi_fp32_fma_probe", "bi_wait_timeout_probe", "bi_moe_gemm_variant", "bi_router_topk", "bi_router_topk_schedule",
    "bi_topk_window", "bi_router_gemm_bf16", "bi_router_gemm_bf16_schedule", "bi_router_topk_bf16",
    "bi_moe_gather_routing", "bi_moe_scatter_contrib", "bi_router_topk_bf16_schedule",
    "bi_moe_gate_up_tokens", "bi_moe_gate_up_feed", "bi_moe_layer", "bi_moe_decode_fused",
]


class BimoeError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {STATUS.get(status, status)}: {msg}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """dlopen libbimoe.so and declare its signatures (no GPU needed)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"CUDA library {path} is missing; build it with "
                "`python -m invariant_moe_gb300._build`")
        lib = ctypes.CDLL(path)
        P, I64, I32, SZ, ST = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                               ctypes.c_size_t, ctypes.c_int)
        sig = {
            "bi_status_str": ([ctypes.c_int], ctypes.c_char_p),
            "bi_last_error_message": ([], ctypes.c_char_p),
            "bi_version": ([], ctypes.c_char_p),
            "bi_device_error": ([P], ST),
            "bi_cast_bf16_to_f32": ([P, P, I64, P], ST),
            "bi_router_gemm": ([P, P, P, P, I64, I64, I64, P], ST),
            "bi_router_gemm_schedule": ([P, P, P, P, I64, I64, I64, I32, P], ST),
            "bi_router_gemm_splitk_negctl": ([P, P, P, P, I64, I64, I64, P], ST),
            "bi_topk": ([P, P, P, P, I64, I64, I32, P], ST),
            "bi_moe_workspace_bytes": ([I64, I64, I64, I32, I64], SZ),
            "bi_moe_forward": ([P, P, P, P, P, P, I64, I64, I64, I32, I64, P, SZ, P], ST),
            "bi_moe_permute_workspace_bytes": ([I64, I64], SZ),
            "bi_moe_permute": ([P, P, P, I64, I64, I32, P, SZ, P], ST),
            "bi_moe_gather": ([P, P, P, P, I64, I64, I64, I32, P], ST),
            "bi_moe_gate_up": ([P, P, P, P, P, P, I64, I64, I64, I32, I64, P], ST),
            "bi_moe_down": ([P, P, P, P, P, I64, I64, I64, I32, I64, P], ST),
            "bi_moe_combine": ([P, P, I64, I64, I32, P], ST),
            "bi_moe_combine_consume": ([P, P, I64, I64, I32, P], ST),
            "bi_moe_gemm_variant": ([I32, P], ST),
            "bi_moe_gate_up_feed": ([I32, P], ST),
            "bi_moe_decode_fused": ([I32, P], ST),
            "bi_moe_layer": ([P, P, P, P, P, P, P, P, P, I64, I64, I64, I32, I64, P, SZ, P], ST),
            "bi_moe_gate_up_tokens": ([P, P, P, P, P, P, I64, I64, I64, I32, I64, P], ST),
            "bi_router_topk": ([P, P, P, P, P, P, P, I64, I64, I64, I32, P], ST),
            "bi_router_topk_schedule": ([P, P, P, P, P, P, P, I64, I64, I64, I32, I32, P], ST),
            "bi_topk_window": ([P, I64, P, P, I64, I64, I32, P, P], ST),
            "bi_router_gemm_bf16": ([P, P, P, P, I64, I64, I64, P], ST),
            "bi_router_gemm_bf16_schedule": ([P, P, P, P, I64, I64, I64, I32, P], ST),
            "bi_router_topk_bf16": ([P, P, P, P, P, P, P, I64, I64, I64, I32, P], ST),
            "bi_router_topk_bf16_schedule": ([P, P, P, P, P, P, P, I64, I64, I64, I32, I32, P], ST),
            "bi_moe_forward_noalloc": ([P, P, P, P, P, P, I64, I64, I64, I32, I64, P], ST),
            "bi_fp32_fma_probe": ([P, I64, I32, P], ST),
            "bi_wait_timeout_probe": ([I32, P], ST),
            "bi_moe_gather_routing": ([P, P, P, P, P, P, I64, I64, I32, I64, P], ST),
            "bi_moe_scatter_contrib": ([P, P, P, P, I64, I64, I64, I32, P], ST),
        }
        for name, (args, res) in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
        return lib


def _call(name, *args):
    lib = load_library()
    st = getattr(lib, name)(*args)
    if st != BI_OK:
        raise BimoeError(name, st, lib.bi_last_error_message().decode())


def _ptr(t, dtype, name, device=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must live on a CUDA device")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def device_error() -> int:
    """Read and clear the device error word (synchronises the device)."""
    lib = load_library()
    v = ctypes.c_int32(0)
    st = lib.bi_device_error(ctypes.byref(v))
    if st != BI_OK:
        raise BimoeError("bi_device_error", st, lib.bi_last_error_message().decode())
    return v.value


# ----------------------------------------------------------------- router --
def bi_cast_bf16_to_f32(x, out=None, stream=None):
    out = out if out is not None else torch.empty(x.shape, dtype=torch.float32, device=x.device)
    _call("bi_cast_bf16_to_f32", _ptr(x, torch.bfloat16, "x"), _ptr(out, torch.float32, "out", x.device),
          x.numel(), _stream(stream))
    return out


def bi_router_gemm(x, w, bias=None, out=None, schedule=0, stream=None):
    """y[M,N] = x[M,K] @ w[N,K]^T (+ bias), fp32, batch-invariant recipe.  x is
    fp32 or bf16 (bf16 values are read as their exact fp32 values)."""
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K:
        raise ValueError("w must be [N, K]")
    out = out if out is not None else torch.empty(M, N, dtype=torch.float32, device=x.device)
    if out.shape != (M, N):
        raise ValueError("out must be [M, N]")
    bf16 = x.dtype == torch.bfloat16
    args = (_ptr(x, torch.bfloat16 if bf16 else torch.float32, "x"), _ptr(w, torch.float32, "w", x.device),
            _ptr(bias, torch.float32, "bias", x.device), _ptr(out, torch.float32, "out", x.device),
            M, K, N)
    name = "bi_router_gemm_bf16" if bf16 else "bi_router_gemm"
    if schedule:
        _call(name + "_schedule", *args, schedule, _stream(stream))
    else:
        _call(name, *args, _stream(stream))
    return out


def bi_router_gemm_splitk_negctl(x, w, bias=None, out=None, stream=None):
    """Negative control (tests only): K split depends on M."""
    M, K = x.shape
    N = w.shape[0]
    out = out if out is not None else torch.empty(M, N, dtype=torch.float32, device=x.device)
    _call("bi_router_gemm_splitk_negctl", _ptr(x, torch.float32, "x"),
          _ptr(w, torch.float32, "w", x.device), _ptr(bias, torch.float32, "bias", x.device),
          _ptr(out, torch.float32, "out", x.device), M, K, N, _stream(stream))
    return out


# ------------------------------------------------------------------ top-k --
def bi_topk(scores, top_k, ids=None, wts=None, probs=None, want_probs=False, stream=None):
    """(ids int32 [M,k], wts fp32 [M,k], probs fp32 [M,E] or None)."""
    M, E = scores.shape
    dev = scores.device
    ids = ids if ids is not None else torch.empty(M, top_k, dtype=torch.int32, device=dev)
    wts = wts if wts is not None else torch.empty(M, top_k, dtype=torch.float32, device=dev)
    if want_probs and probs is None:
        probs = torch.empty(M, E, dtype=torch.float32, device=dev)
    _call("bi_topk", _ptr(scores, torch.float32, "scores"), _ptr(probs, torch.float32, "probs", dev),
          _ptr(ids, torch.int32, "ids", dev), _ptr(wts, torch.float32, "wts", dev),
          M, E, top_k, _stream(stream))
    return ids, wts, probs


# -------------------------------------------------------------------- MoE --
def bi_moe_workspace_bytes(M, H, E, top_k, I) -> int:
    return int(load_library().bi_moe_workspace_bytes(M, H, E, top_k, I))


def moe_workspace(M, H, E, top_k, I, device):
    n = bi_moe_workspace_bytes(M, H, E, top_k, I)
    if n == 0 and M > 0:
        raise ValueError("unsupported MoE sizes")
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def bi_moe_forward(x, ids, wts, w13, w2, out=None, workspace=None, stream=None):
    """out[M,H] bf16 = batch-invariant SwiGLU MoE of x [M,H] bf16."""
    M, H, E, I, top_k = _check_moe_shapes(x, ids, wts, w13, w2, out)
    dev = x.device
    out = out if out is not None else torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = moe_workspace(M, H, E, top_k, I, dev)
    _call("bi_moe_forward", _ptr(x, torch.bfloat16, "x"), _ptr(ids, torch.int32, "ids", dev),
          _ptr(wts, torch.float32, "wts", dev), _ptr(w13, torch.bfloat16, "w13", dev),
          _ptr(w2, torch.bfloat16, "w2", dev), _ptr(out, torch.bfloat16, "out", dev),
          M, H, E, top_k, I, _ptr(workspace, torch.uint8, "workspace", dev),
          workspace.numel(), _stream(stream))
    return out


def _check_moe_shapes(x, ids, wts, w13, w2, out):
    M, H = x.shape
    E, twoI, H2 = w13.shape
    I = twoI // 2
    if H2 != H or twoI % 2 or tuple(w2.shape) != (E, H, I):
        raise ValueError("w13 must be [E, 2I, H] and w2 [E, H, I]")
    if ids.dim() != 2 or ids.shape[0] != M or tuple(wts.shape) != tuple(ids.shape):
        raise ValueError("ids and wts must be [M, top_k]")
    if out is not None and tuple(out.shape) != (M, H):
        raise ValueError("out must be [M, H]")
    return M, H, E, I, ids.shape[1]


def bi_moe_forward_noalloc(x, ids, wts, w13, w2, out=None, stream=None):
    """bi_moe_forward with the library's built-in scratch array instead of a
    caller workspace (for callers that cannot allocate device memory; the
    output tensor, if not given, is still allocated here by torch).  The call
    runs with x's device current, whose scratch array the library uses."""
    M, H, E, I, top_k = _check_moe_shapes(x, ids, wts, w13, w2, out)
    dev = x.device
    if not x.is_cuda:
        raise ValueError("x must live on a CUDA device")
    with torch.cuda.device(dev):
        out = out if out is not None else torch.empty(M, H, dtype=torch.bfloat16, device=dev)
        if stream is not None and stream.device != dev:
            raise ValueError(f"stream is on {stream.device}, expected {dev}")
        _call("bi_moe_forward_noalloc", _ptr(x, torch.bfloat16, "x"), _ptr(ids, torch.int32, "ids", dev),
              _ptr(wts, torch.float32, "wts", dev), _ptr(w13, torch.bfloat16, "w13", dev),
              _ptr(w2, torch.bfloat16, "w2", dev), _ptr(out, torch.bfloat16, "out", dev),
              M, H, E, top_k, I, _stream(stream))
    return out


def bi_moe_permute(ids, E, offsets=None, perm=None, workspace=None, stream=None):
    M, top_k = ids.shape
    dev = ids.device
    lib = load_library()
    offsets = offsets if offsets is not None else torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = perm if perm is not None else torch.empty(max(M * top_k, 1), dtype=torch.int32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(int(lib.bi_moe_permute_workspace_bytes(M, E)), 256),
                                dtype=torch.uint8, device=dev)
    _call("bi_moe_permute", _ptr(ids, torch.int32, "ids"), _ptr(offsets, torch.int32, "offsets", dev),
          _ptr(perm, torch.int32, "perm", dev), M, E, top_k,
          _ptr(workspace, torch.uint8, "workspace", dev), workspace.numel(), _stream(stream))
    return offsets, perm


def bi_moe_gather(x, offsets, perm, top_k, x_perm=None, stream=None):
    """x_perm [M*top_k, H] bf16: token rows in expert order."""
    M, H = x.shape
    E = offsets.numel() - 1
    dev = x.device
    x_perm = x_perm if x_perm is not None else torch.empty(M * top_k, H, dtype=torch.bfloat16, device=dev)
    _call("bi_moe_gather", _ptr(x, torch.bfloat16, "x"), _ptr(offsets, torch.int32, "offsets", dev),
          _ptr(perm, torch.int32, "perm", dev), _ptr(x_perm, torch.bfloat16, "x_perm", dev),
          M, H, E, top_k, _stream(stream))
    return x_perm


def bi_moe_gate_up(x_perm, offsets, perm, wts, w13, top_k, act=None, stream=None):
    """act [M*top_k, I] bf16 from gathered rows x_perm [M*top_k, H]."""
    P, H = x_perm.shape
    M = P // top_k
    E, twoI, _ = w13.shape
    I = twoI // 2
    dev = x_perm.device
    act = act if act is not None else torch.empty(P, I, dtype=torch.bfloat16, device=dev)
    _call("bi_moe_gate_up", _ptr(x_perm, torch.bfloat16, "x_perm"),
          _ptr(offsets, torch.int32, "offsets", dev), _ptr(perm, torch.int32, "perm", dev),
          _ptr(wts, torch.float32, "wts", dev), _ptr(w13, torch.bfloat16, "w13", dev),
          _ptr(act, torch.bfloat16, "act", dev), M, H, E, top_k, I, _stream(stream))
    return act


def bi_moe_gate_up_tokens(x, offsets, perm, wts, w13, top_k, act=None, stream=None):
    """act [M*top_k, I] bf16, the gate/up GEMM gathering the token rows of
    x [M, H] itself (no gathered copy)."""
    M, H = x.shape
    E, twoI, _ = w13.shape
    I = twoI // 2
    dev = x.device
    act = act if act is not None else torch.empty(M * top_k, I, dtype=torch.bfloat16, device=dev)
    _call("bi_moe_gate_up_tokens", _ptr(x, torch.bfloat16, "x"),
          _ptr(offsets, torch.int32, "offsets", dev), _ptr(perm, torch.int32, "perm", dev),
          _ptr(wts, torch.float32, "wts", dev), _ptr(w13, torch.bfloat16, "w13", dev),
          _ptr(act, torch.bfloat16, "act", dev), M, H, E, top_k, I, _stream(stream))
    return act


def bi_moe_gate_up_feed(mode):
    """How bi_moe_forward feeds the gate/up GEMM (0 automatic = the gathered
    copy, 1 gathered copy, 2 gathered by the GEMM); returns the previous
    setting."""
    prev = ctypes.c_int32(0)
    _call("bi_moe_gate_up_feed", int(mode), ctypes.byref(prev))
    return prev.value


def bi_moe_decode_fused(mode):
    """How bi_moe_layer runs a decode-sized batch's expert GEMMs (0 automatic
    = one launch where it applies, 1 = a gate/up and a down launch); returns
    the previous setting."""
    prev = ctypes.c_int32(0)
    _call("bi_moe_decode_fused", int(mode), ctypes.byref(prev))
    return prev.value


def bi_moe_down(act, offsets, perm, w2, M, top_k, contrib=None, stream=None):
    E, H, I = w2.shape
    dev = act.device
    contrib = contrib if contrib is not None else torch.empty(M * top_k, H, dtype=torch.float32, device=dev)
    _call("bi_moe_down", _ptr(act, torch.bfloat16, "act"), _ptr(offsets, torch.int32, "offsets", dev),
          _ptr(perm, torch.int32, "perm", dev), _ptr(w2, torch.bfloat16, "w2", dev),
          _ptr(contrib, torch.float32, "contrib", dev), M, H, E, top_k, I, _stream(stream))
    return contrib


def bi_moe_gather_routing(ids, wts, offsets, perm, experts_per_rank, lid=None, pw=None, stream=None):
    """(lid int32 [M*top_k], pw fp32 [M*top_k]): for each permuted position,
    the expert's index on the rank that owns it and the routing probability."""
    M, top_k = ids.shape
    E = offsets.numel() - 1
    dev = ids.device
    P = M * top_k
    lid = lid if lid is not None else torch.empty(max(P, 1), dtype=torch.int32, device=dev)
    pw = pw if pw is not None else torch.empty(max(P, 1), dtype=torch.float32, device=dev)
    _call("bi_moe_gather_routing", _ptr(ids, torch.int32, "ids"), _ptr(wts, torch.float32, "wts", dev),
          _ptr(offsets, torch.int32, "offsets", dev), _ptr(perm, torch.int32, "perm", dev),
          _ptr(lid, torch.int32, "lid", dev), _ptr(pw, torch.float32, "pw", dev), M, E, top_k,
          experts_per_rank, _stream(stream))
    return lid, pw


def bi_moe_scatter_contrib(rows, offsets, perm, M, top_k, contrib=None, stream=None):
    """contrib [M*top_k, H] fp32 with contrib[perm[p]] = rows[p] for p < offsets[E]."""
    H = rows.shape[-1]
    E = offsets.numel() - 1
    dev = rows.device
    contrib = contrib if contrib is not None else torch.empty(M * top_k, H, dtype=torch.float32, device=dev)
    _call("bi_moe_scatter_contrib", _ptr(rows, torch.float32, "rows"), _ptr(offsets, torch.int32, "offsets", dev),
          _ptr(perm, torch.int32, "perm", dev), _ptr(contrib, torch.float32, "contrib", dev), M, H, E, top_k,
          _stream(stream))
    return contrib


def bi_moe_combine(contrib, M, top_k, out=None, stream=None):
    H = contrib.shape[-1]
    dev = contrib.device
    out = out if out is not None else torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    _call("bi_moe_combine", _ptr(contrib, torch.float32, "contrib"), _ptr(out, torch.bfloat16, "out", dev),
          M, H, top_k, _stream(stream))
    return out


def bi_moe_combine_consume(contrib, M, top_k, out=None, stream=None):
    """bi_moe_combine for a caller that never reads ``contrib`` again: its
    lines are dropped from L2 once summed, and its contents are indeterminate
    afterwards."""
    H = contrib.shape[-1]
    dev = contrib.device
    out = out if out is not None else torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    _call("bi_moe_combine_consume", _ptr(contrib, torch.float32, "contrib"),
          _ptr(out, torch.bfloat16, "out", dev), M, H, top_k, _stream(stream))
    return out


def bi_router_topk(x, w, top_k, bias=None, out=None, want_probs=False, schedule=0, stream=None,
                   ids=None, wts=None):
    """Router scores and top-k selection in one call (the selection grid as a
    programmatic dependent of the router grid; schedule 10 forces the
    one-kernel cluster path for up to 4 rows, 1..9 a router schedule).  Returns
    (scores [M,N] fp32, ids [M,top_k] int32, wts [M,top_k] fp32, probs or None)."""
    M, K = x.shape
    N = w.shape[0]
    dev = x.device
    y = out if out is not None else torch.empty(M, N, dtype=torch.float32, device=dev)
    ids = ids if ids is not None else torch.empty(M, top_k, dtype=torch.int32, device=dev)
    wts = wts if wts is not None else torch.empty(M, top_k, dtype=torch.float32, device=dev)
    if ids.shape != (M, top_k) or wts.shape != (M, top_k):
        raise ValueError("ids and wts must be [M, top_k]")
    probs = torch.empty(M, N, dtype=torch.float32, device=dev) if want_probs else None
    ptrs = (_ptr(w, torch.float32, "w", dev), _ptr(bias, torch.float32, "bias", dev),
            _ptr(y, torch.float32, "out", dev), _ptr(probs, torch.float32, "probs", dev),
            _ptr(ids, torch.int32, "ids", dev), _ptr(wts, torch.float32, "wts", dev))
    if x.dtype == torch.bfloat16:
        _call("bi_router_topk_bf16_schedule", _ptr(x, torch.bfloat16, "x"), *ptrs, M, K, N, top_k, schedule,
              _stream(stream))
    else:
        _call("bi_router_topk_schedule", _ptr(x, torch.float32, "x"), *ptrs, M, K, N, top_k, schedule,
              _stream(stream))
    return y, ids, wts, probs


def bi_topk_window(scores, k, row_start=None, row_end=None, num_cols=None, out=None, stream=None):
    """Windowed per-row top-k: int32 [n_rows, k] window-relative columns of
    the k best in-window scores, ascending, -1 tail.  scores is fp32
    [n_rows, ld] with unit column stride (row stride ld >= num_cols)."""
    if scores.dim() != 2 or scores.stride(1) != 1:
        raise ValueError("scores must be 2-D with unit column stride")
    n_rows = scores.shape[0]
    ld = scores.stride(0) if n_rows > 1 else scores.shape[1]
    num_cols = scores.shape[1] if num_cols is None else num_cols
    dev = scores.device
    if scores.dtype != torch.float32 or not scores.is_cuda:
        raise TypeError("scores must be a CUDA float32 tensor")
    out = out if out is not None else torch.empty(n_rows, k, dtype=torch.int32, device=dev)
    _call("bi_topk_window", ctypes.c_void_p(scores.data_ptr()), ld,
          _ptr(row_start, torch.int64, "row_start", dev), _ptr(row_end, torch.int64, "row_end", dev),
          n_rows, num_cols, k, _ptr(out, torch.int32, "out", dev), _stream(stream))
    return out


def bi_moe_gemm_variant(variant):
    """Select the expert-GEMM schedule for the process (0 automatic, 1 one CTA
    per tile, 2 CTA pairs, 3 CTA pairs with interleaved gate/up rows for the
    gate/up GEMM, 4 one CTA per tile with interleaved gate/up rows); returns
    the previous setting."""
    prev = ctypes.c_int32(0)
    _call("bi_moe_gemm_variant", int(variant), ctypes.byref(prev))
    return prev.value


def bi_fp32_fma_probe(blocks, iters, stream=None, out=None):
    """Run the FP32 FMA throughput probe; returns its output tensor."""
    if out is None:
        out = torch.empty(blocks * 256, dtype=torch.float32, device="cuda")
    elif out.numel() < blocks * 256:
        raise ValueError("out holds fewer than blocks * 256 floats")
    _call("bi_fp32_fma_probe", _ptr(out, torch.float32, "out"), blocks, iters, _stream(stream))
    return out


def bi_wait_timeout_probe(which=0, stream=None):
    """Test use only: a kernel whose bounded wait runs out (about one second):
    which = 0 the mbarrier wait, 1 the arrival-count wait; read the recorded
    BI_DEVERR_WAIT_TIMEOUT with device_error()."""
    _call("bi_wait_timeout_probe", int(which), _stream(stream))


def bi_moe_layer(x, w_router, w13, w2, top_k, bias=None, out=None, scores=None, ids=None, wts=None,
                 workspace=None, stream=None):
    """Whole hot path of one MoE layer in one library call: router (on the
    bf16 tokens, read as their exact fp32 values) -> top-k -> experts.
    Returns (out, scores, ids, wts)."""
    M, H = x.shape
    E, H2 = w_router.shape
    if H2 != H:
        raise ValueError("w_router must be [E, H]")
    dev = x.device
    ids = ids if ids is not None else torch.empty(M, top_k, dtype=torch.int32, device=dev)
    wts = wts if wts is not None else torch.empty(M, top_k, dtype=torch.float32, device=dev)
    _, _, _, I, _ = _check_moe_shapes(x, ids, wts, w13, w2, out)
    if w13.shape[0] != E:
        raise ValueError("w_router, w13 and w2 must have the same number of experts")
    out = out if out is not None else torch.empty(M, H, dtype=torch.bfloat16, device=dev)
    scores = scores if scores is not None else torch.empty(M, E, dtype=torch.float32, device=dev)
    if tuple(scores.shape) != (M, E):
        raise ValueError("scores must be [M, E]")
    if workspace is None:
        workspace = moe_workspace(M, H, E, top_k, I, dev)
    _call("bi_moe_layer", _ptr(x, torch.bfloat16, "x"), _ptr(w_router, torch.float32, "w_router", dev),
          _ptr(bias, torch.float32, "bias", dev), _ptr(w13, torch.bfloat16, "w13", dev),
          _ptr(w2, torch.bfloat16, "w2", dev), _ptr(out, torch.bfloat16, "out", dev),
          _ptr(scores, torch.float32, "scores", dev), _ptr(ids, torch.int32, "ids", dev),
          _ptr(wts, torch.float32, "wts", dev), M, H, E, top_k, I,
          _ptr(workspace, torch.uint8, "workspace", dev), workspace.numel(), _stream(stream))
    return out, scores, ids, wts


def moe_layer(x_bf16, w_router, w13, w2, top_k, bias=None, stream=None):
    """Whole hot path of one MoE layer (bi_moe_layer).  Returns (out, scores,
    ids, wts)."""
    return bi_moe_layer(x_bf16, w_router, w13, w2, top_k, bias=bias, stream=stream)
