"""CPU oracle for the shard-reduction GEMM -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It shares no code with the CUDA library and never
imports it. The arithmetic lives in ``gsr_oracle.c`` (plain C, fp64); this
module only builds it and marshals numpy arrays of bf16 bit patterns.

Functions (pages: PR #53053 summary "Extend GEMM-RS to GEMM-AR", test section,
``_reference``; PR #54151 "[Kimi-K3] AG-GEMM for Sequence Parallelism",
Purpose):

* ``ar(X_r, W_r, N)``        Y = sum_r X_r . W_r^T, fp64, M x N
* ``ar_at(X_r, W_r, rows, cols)``   the same at listed points
* ``rs(X_r, W_r)``           per-shard row slices of the AR result
* ``rs_rows(M, R, s)``       (first row, row count) owned by shard s
* ``ag(A_r, W)``             Y = concat_r(A_r) . W^T, fp64
* ``ag_at(A_r, W, rows, cols)``     the same at listed points
* ``pack_gather(S, rows_out)``  the packed gather of per-rank states (PR #51070
  summary "Kimi K3 SP: pack the per-layer all-gathers into one"): rows_out x T*H
* ``bf16_to_f64(bits)``      exact widening of one bf16 bit pattern

Every function's pin (brute force, invariants, special cases) is in
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import fcntl
import os
import subprocess
from typing import List, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gsr_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "libgsr_oracle.so")

_lib = None


def _fresh() -> bool:
    return os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP when available). Returns the .so path.
    Processes that build at the same time take turns (a lock file), and the
    library is replaced atomically."""
    if not force and _fresh():
        return _LIB
    os.makedirs(_OUT_DIR, exist_ok=True)
    with open(os.path.join(_OUT_DIR, ".build.lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and _fresh():
                return _LIB
            tmp = f"{_LIB}.{os.getpid()}.tmp"
            base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    _SRC, "-o", tmp]
            try:
                subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                               capture_output=True, text=True)
            except subprocess.CalledProcessError:
                subprocess.run(base, check=True, capture_output=True, text=True)
            os.replace(tmp, _LIB)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i64, i32, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.gsr_oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.gsr_oracle_bf16_to_f64.restype = ctypes.c_double
    lib.gsr_oracle_threads.restype = i32
    lib.gsr_oracle_ar.argtypes = [i64, i64, i32, dp, dp, dp, dp]
    lib.gsr_oracle_ar_at.argtypes = [i64, i64, i32, dp, dp, dp, i64, dp, dp, dp]
    lib.gsr_oracle_rs_rows.argtypes = [i64, i32, i32, dp, dp]
    lib.gsr_oracle_rs.argtypes = [i64, i64, i32, dp, dp, dp, dp]
    lib.gsr_oracle_ag.argtypes = [i64, i64, i32, dp, dp, dp, dp]
    lib.gsr_oracle_ag_at.argtypes = [i64, i64, i32, dp, dp, dp, i64, dp, dp, dp]
    lib.gsr_oracle_pack_gather.argtypes = [i32, dp, i32, i64, dp, i64, dp]
    for f in ("gsr_oracle_ar", "gsr_oracle_ar_at", "gsr_oracle_rs_rows",
              "gsr_oracle_rs", "gsr_oracle_ag", "gsr_oracle_ag_at", "gsr_oracle_pack_gather"):
        getattr(lib, f).restype = None
    _lib = lib
    return lib


def _bits(a) -> np.ndarray:
    """Accept a numpy uint16 array or a torch bf16 tensor; return C-contiguous uint16."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns (uint16), got {a.dtype}")
    return a


def _ptrs(arrs: Sequence[np.ndarray]):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def _i64(vals) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(vals, dtype=np.int64))


def threads() -> int:
    return int(_load().gsr_oracle_threads())


def bf16_to_f64(bits: int) -> float:
    return float(_load().gsr_oracle_bf16_to_f64(int(bits) & 0xFFFF))


def _ar_args(X_r, W_r):
    X = [_bits(x) for x in X_r]
    W = [_bits(w) for w in W_r]
    if len(X) != len(W) or not X:
        raise ValueError("X_r and W_r need the same, non-zero number of shards")
    M = X[0].shape[0]
    N = W[0].shape[0]
    K_r = [x.shape[1] for x in X]
    for x, w, k in zip(X, W, K_r):
        if x.shape != (M, k) or w.shape != (N, k):
            raise ValueError("shard shapes disagree")
    return X, W, M, N, K_r


def ar(X_r, W_r) -> np.ndarray:
    """Y = sum_r X_r . W_r^T in fp64 (M x N)."""
    X, W, M, N, K_r = _ar_args(X_r, W_r)
    Y = np.empty((M, N), dtype=np.float64)
    k = _i64(K_r)
    _load().gsr_oracle_ar(M, N, len(X), k.ctypes.data, _ptrs(X), _ptrs(W),
                          Y.ctypes.data)
    return Y


def ar_at(X_r, W_r, rows, cols) -> np.ndarray:
    X, W, M, N, K_r = _ar_args(X_r, W_r)
    rows, cols = _i64(rows), _i64(cols)
    if rows.shape != cols.shape:
        raise ValueError("rows/cols length mismatch")
    if rows.size and (rows.min() < 0 or rows.max() >= M or cols.min() < 0
                      or cols.max() >= N):
        raise IndexError("sample point out of range")
    out = np.empty(rows.shape, dtype=np.float64)
    k = _i64(K_r)
    _load().gsr_oracle_ar_at(M, N, len(X), k.ctypes.data, _ptrs(X), _ptrs(W),
                             rows.size, rows.ctypes.data, cols.ctypes.data,
                             out.ctypes.data)
    return out


def rs_rows(M: int, R: int, s: int) -> Tuple[int, int]:
    first, count = ctypes.c_int64(), ctypes.c_int64()
    _load().gsr_oracle_rs_rows(M, R, s, ctypes.byref(first), ctypes.byref(count))
    return first.value, count.value


def rs(X_r, W_r) -> List[np.ndarray]:
    """Per-shard outputs: entry s has ceil(M/R) rows; rows past the shard's
    valid count are NaN (the oracle writes no value there)."""
    X, W, M, N, K_r = _ar_args(X_r, W_r)
    R = len(X)
    rps = -(-M // R)
    outs = [np.full((rps, N), np.nan, dtype=np.float64) for _ in range(R)]
    k = _i64(K_r)
    _load().gsr_oracle_rs(M, N, R, k.ctypes.data, _ptrs(X), _ptrs(W), _ptrs(outs))
    return outs


def _ag_args(A_r, W):
    A = [_bits(a) for a in A_r]
    Wb = _bits(W)
    if not A:
        raise ValueError("need at least one shard")
    N, K = Wb.shape
    M_r = [a.shape[0] for a in A]
    for a in A:
        if a.ndim != 2 or a.shape[1] != K:
            raise ValueError("shard shapes disagree")
    return A, Wb, N, K, M_r


def ag(A_r, W) -> np.ndarray:
    """Y = concat_r(A_r) . W^T in fp64 ((sum M_r) x N)."""
    A, Wb, N, K, M_r = _ag_args(A_r, W)
    Y = np.empty((sum(M_r), N), dtype=np.float64)
    m = _i64(M_r)
    _load().gsr_oracle_ag(N, K, len(A), m.ctypes.data, _ptrs(A), Wb.ctypes.data,
                          Y.ctypes.data)
    return Y


def ag_at(A_r, W, rows, cols) -> np.ndarray:
    A, Wb, N, K, M_r = _ag_args(A_r, W)
    rows, cols = _i64(rows), _i64(cols)
    if rows.shape != cols.shape:
        raise ValueError("rows/cols length mismatch")
    if rows.size and (rows.min() < 0 or rows.max() >= sum(M_r) or cols.min() < 0
                      or cols.max() >= N):
        raise IndexError("sample point out of range")
    out = np.empty(rows.shape, dtype=np.float64)
    m = _i64(M_r)
    _load().gsr_oracle_ag_at(N, K, len(A), m.ctypes.data, _ptrs(A), Wb.ctypes.data,
                             rows.size, rows.ctypes.data, cols.ctypes.data,
                             out.ctypes.data)
    return out


def pack_gather(S, rows_out: int) -> np.ndarray:
    """S[r][t]: rank r's state t (M_r x H bf16 bits). Returns P (rows_out x T*H,
    uint16): the ranks' states concatenated along the last dimension, stacked in
    rank order and cut to rows_out rows."""
    R = len(S)
    if R == 0 or any(len(s) != len(S[0]) for s in S) or not S[0]:
        raise ValueError("need R >= 1 ranks with the same T >= 1 states each")
    T = len(S[0])
    flat = [_bits(a) for s in S for a in s]
    H = flat[0].shape[1]
    M_r = []
    for r in range(R):
        shapes = {flat[r * T + t].shape for t in range(T)}
        if len(shapes) != 1 or flat[r * T].ndim != 2 or flat[r * T].shape[1] != H:
            raise ValueError("state shapes disagree")
        M_r.append(flat[r * T].shape[0])
    if not 0 <= rows_out <= sum(M_r):
        raise ValueError("rows_out outside 0 .. sum of M_r")
    P = np.empty((rows_out, T * H), dtype=np.uint16)
    m = _i64(M_r)
    _load().gsr_oracle_pack_gather(R, m.ctypes.data, T, H, _ptrs(flat), rows_out,
                                   P.ctypes.data)
    return P
