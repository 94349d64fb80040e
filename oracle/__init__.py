"""fp64 CPU oracle for the batch-invariant MoE hot path (ctypes binding).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py``.  The product package
never imports it, and it imports nothing from the product package.

The arithmetic lives in ``bimoe_oracle.c`` (plain loops, fp64); this module
only compiles it with gcc and marshals numpy arrays.  bf16 tensors are passed
as their raw uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bimoe_oracle.c")
_LIB = os.path.join(_HERE, "libbimoe_oracle.so")
# -ffp-contract=off: no fused multiply-add contraction, so the same doubles
# come out on x86-64 and aarch64 hosts.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-fvisibility=hidden"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library next to its source (idempotent)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I32 = ctypes.c_int32
            lib.oracle_router.argtypes = [P, P, P, I64, I64, I64, P]
            lib.oracle_sigmoid.argtypes = [ctypes.c_double]
            lib.oracle_sigmoid.restype = ctypes.c_double
            lib.oracle_sigmoid_vec.argtypes = [P, I64, P]
            lib.oracle_score_key.argtypes = [ctypes.c_float]
            lib.oracle_score_key.restype = I32
            lib.oracle_topk.argtypes = [P, I64, I64, I32, P, P]
            lib.oracle_topk_window.argtypes = [P, I64, P, P, I64, I64, I32, P]
            lib.oracle_permute.argtypes = [P, I64, I64, I32, P, P]
            lib.oracle_permute.restype = ctypes.c_int
            lib.oracle_moe.argtypes = [P, P, P, P, P, I64, I64, I64, I32, I64, P]
            lib.oracle_gate_up.argtypes = [P, P, P, P, P, I64, I64, I32, I64, P]
            lib.oracle_down.argtypes = [P, P, P, P, I64, I64, I64, P]
            lib.oracle_combine.argtypes = [P, I64, I64, I32, P]
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def router(x, w, b=None):
    """r = x @ w.T (+ b) in fp64.  x [M,K] f32, w [N,K] f32, b [N] f32 or None."""
    lib = _load()
    x, px = _c(x, np.float32)
    w, pw = _c(w, np.float32)
    M, K = x.shape
    N = w.shape[0]
    assert w.shape[1] == K
    pb = None
    if b is not None:
        b, pb = _c(b, np.float32)
        assert b.shape == (N,)
    r = np.empty((M, N), np.float64)
    lib.oracle_router(px, pw, pb, M, K, N, r.ctypes.data_as(ctypes.c_void_p))
    return r


def sigmoid(v):
    """Elementwise fp64 sigmoid of fp32 values."""
    lib = _load()
    v, pv = _c(v, np.float32)
    out = np.empty(v.shape, np.float64)
    lib.oracle_sigmoid_vec(pv, v.size, out.ctypes.data_as(ctypes.c_void_p))
    return out


def score_key(v: float) -> int:
    return int(_load().oracle_score_key(ctypes.c_float(v)))


def topk(scores, top_k):
    """(ids int32 [M,k], wts fp64 [M,k]) selected on fp32 scores [M,E]."""
    lib = _load()
    s, ps = _c(scores, np.float32)
    M, E = s.shape
    assert 0 < top_k <= E
    ids = np.empty((M, top_k), np.int32)
    wts = np.empty((M, top_k), np.float64)
    lib.oracle_topk(ps, M, E, top_k, ids.ctypes.data_as(ctypes.c_void_p),
                    wts.ctypes.data_as(ctypes.c_void_p))
    return ids, wts


def topk_window(scores, k, row_start=None, row_end=None, num_cols=None):
    """Windowed per-row top-k (int32 [n_rows, k]): window-relative columns of
    the k best in-window scores, ascending, -1 tail.  scores is fp32
    [n_rows, width] (width = the row stride); num_cols <= width columns exist
    (default width); row_start / row_end are int64 [n_rows] or None."""
    lib = _load()
    s = np.ascontiguousarray(scores, dtype=np.float32)
    n_rows, width = s.shape
    num_cols = width if num_cols is None else num_cols
    assert 0 <= num_cols <= width and k > 0
    rs = None if row_start is None else np.ascontiguousarray(row_start, dtype=np.int64)
    re = None if row_end is None else np.ascontiguousarray(row_end, dtype=np.int64)
    out = np.empty((n_rows, k), np.int32)
    lib.oracle_topk_window(s.ctypes.data_as(ctypes.c_void_p), width,
                           None if rs is None else rs.ctypes.data_as(ctypes.c_void_p),
                           None if re is None else re.ctypes.data_as(ctypes.c_void_p),
                           n_rows, num_cols, k, out.ctypes.data_as(ctypes.c_void_p))
    return out


def permute(ids, E):
    """(offsets int32 [E+1], perm int32 [M*k]) for expert ids [M,k]."""
    lib = _load()
    ids, pi = _c(ids, np.int32)
    M, k = ids.shape
    offsets = np.empty(E + 1, np.int32)
    perm = np.empty(M * k, np.int32)
    rc = lib.oracle_permute(pi, M, E, k, offsets.ctypes.data_as(ctypes.c_void_p),
                            perm.ctypes.data_as(ctypes.c_void_p))
    if rc != 0:
        raise ValueError("expert id out of range")
    return offsets, perm


def moe(x_bits, ids, wts, w13_bits, w2_bits, E, I):
    """Full MoE expert path in fp64.  bf16 arrays are uint16 bit patterns:
    x [M,H], w13 [E,2I,H], w2 [E,H,I]; ids [M,k] int32; wts [M,k] f32."""
    lib = _load()
    x, px = _c(x_bits, np.uint16)
    ids, pi = _c(ids, np.int32)
    wts, pwt = _c(wts, np.float32)
    w13, p13 = _c(w13_bits, np.uint16)
    w2, p2 = _c(w2_bits, np.uint16)
    M, H = x.shape
    k = ids.shape[1]
    assert w13.size == E * 2 * I * H and w2.size == E * H * I
    out = np.empty((M, H), np.float64)
    lib.oracle_moe(px, pi, pwt, p13, p2, M, H, E, k, I, out.ctypes.data_as(ctypes.c_void_p))
    return out


def gate_up(x_bits, offsets, perm, wts, w13_bits, E, top_k, I):
    """act [P, I] fp64 for the permuted pairs."""
    lib = _load()
    x, px = _c(x_bits, np.uint16)
    off, po = _c(offsets, np.int32)
    perm, pp = _c(perm, np.int32)
    wts, pw = _c(wts, np.float32)
    w13, p13 = _c(w13_bits, np.uint16)
    H = x.shape[1]
    P = int(off[E])
    act = np.empty((P, I), np.float64)
    lib.oracle_gate_up(px, po, pp, pw, p13, H, E, top_k, I, act.ctypes.data_as(ctypes.c_void_p))
    return act


def down(act_bits, offsets, perm, w2_bits, M, H, E, top_k, I):
    """contrib [M*top_k, H] fp64 from permuted bf16 activations [P, I]."""
    lib = _load()
    a, pa = _c(act_bits, np.uint16)
    off, po = _c(offsets, np.int32)
    perm, pp = _c(perm, np.int32)
    w2, p2 = _c(w2_bits, np.uint16)
    contrib = np.zeros((M * top_k, H), np.float64)
    lib.oracle_down(pa, po, pp, p2, H, E, I, contrib.ctypes.data_as(ctypes.c_void_p))
    return contrib


def combine(contrib, top_k):
    """out [M, H] fp64 = slot-order sum of fp32 contrib [M*top_k, H]."""
    lib = _load()
    c, pc = _c(contrib, np.float32)
    H = c.shape[-1]
    M = c.size // (H * top_k)
    out = np.empty((M, H), np.float64)
    lib.oracle_combine(pc, M, H, top_k, out.ctypes.data_as(ctypes.c_void_p))
    return out
