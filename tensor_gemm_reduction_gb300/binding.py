"""Python binding of the C ABI in ``include/gsr.h``: argument marshalling only.

Every function here has the name of the C entry point it calls. Tensors are
checked for dtype, device, contiguity and shape, turned into raw pointers and
passed to the library with the current CUDA stream; all arithmetic runs in the
library's kernels. There is no fallback: if the library has not been built, the
first call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libgsr.so")
_lib = None

GSR_OK = 0
GSR_ERR_INVALID_VALUE = 1
GSR_ERR_UNSUPPORTED = 2
GSR_ERR_WORKSPACE = 3
GSR_ERR_CUDA = 4
GSR_ERR_TIMEOUT = 5
GSR_MAX_SHARDS = 16

GSR_OPT_SPLIT_K = 1
GSR_OPT_BLOCK_N = 2
GSR_OPT_TIMEOUT_NS = 3
GSR_OPT_MAX_CTAS = 4
GSR_OPT_RASTER_M = 5
GSR_OPT_L2_HINTS = 6
GSR_OPT_CTA_GROUP = 7
GSR_OPT_SCHEDULE = 8
GSR_OPT_SMALL_M = 9
GSR_OPT_SMALL_TILE_ROWS = 10
GSR_OPT_RASTER_N = 11
GSR_OPT_SMALL_KBLOCKS = 12

MODE_AR, MODE_RS, MODE_AG = 0, 1, 2

_STATUS_NAMES = {
    GSR_OK: "GSR_OK",
    GSR_ERR_INVALID_VALUE: "GSR_ERR_INVALID_VALUE",
    GSR_ERR_UNSUPPORTED: "GSR_ERR_UNSUPPORTED",
    GSR_ERR_WORKSPACE: "GSR_ERR_WORKSPACE",
    GSR_ERR_CUDA: "GSR_ERR_CUDA",
    GSR_ERR_TIMEOUT: "GSR_ERR_TIMEOUT",
}

EXPORTED = (
    "gemm_shard_plan_create", "gemm_shard_plan_create_host", "gemm_shard_plan_destroy", "gemm_shard_plan_set_option",
    "gemm_shard_workspace_size", "gemm_shard_workspace_init", "gemm_ar", "gemm_rs",
    "gemm_ag", "gemm_shard_check_status", "gsr_last_error_string", "gemm_shard_describe",
    "gemm_ar_noalloc", "gemm_ag_flagged", "gemm_shard_signal", "gemm_ar_replicated",
    "gemm_shard_pack_gather", "gemm_ar_noalloc_check_status",
)


class GsrConfig(ctypes.Structure):
    """Mirror of gsr_config (include/gsr.h)."""
    _fields_ = [("block_n", ctypes.c_int), ("cta_group", ctypes.c_int),
                ("schedule", ctypes.c_int), ("split", ctypes.c_int),
                ("tiles", ctypes.c_int64), ("dp_tiles", ctypes.c_int64),
                ("sk_iters", ctypes.c_int64), ("ctas", ctypes.c_int),
                ("workspace_bytes", ctypes.c_size_t), ("kblocks", ctypes.c_int),
                ("l2_hints", ctypes.c_int)]


class GsrError(RuntimeError):
    """A non-zero gsr_status, with the library's message."""

    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load the built library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"the CUDA library {_LIB_PATH} is not built; run "
            "`python -m tensor_gemm_reduction_gb300.build` (or __graft_entry__.build())")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    ptr_arr = ctypes.POINTER(ctypes.c_void_p)
    i64_arr = ctypes.POINTER(ctypes.c_int64)
    lib.gemm_shard_plan_create.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i64, i32]
    lib.gemm_shard_plan_create_host.argtypes = [ctypes.POINTER(vp), i32, i64, i64, i64, i32]
    lib.gemm_shard_plan_destroy.argtypes = [vp]
    lib.gemm_shard_plan_set_option.argtypes = [vp, i32, i64]
    lib.gemm_shard_workspace_size.argtypes = [vp]
    lib.gemm_shard_workspace_size.restype = sz
    lib.gemm_shard_workspace_init.argtypes = [vp, vp, sz, vp]
    lib.gemm_ar.argtypes = [vp, i64, i64, i32, i64_arr, ptr_arr, ptr_arr, vp, vp, sz, vp]
    lib.gemm_rs.argtypes = [vp, i64, i64, i32, i64_arr, ptr_arr, ptr_arr, ptr_arr, vp, sz, vp]
    lib.gemm_ar_replicated.argtypes = [vp, i64, i64, i32, i64_arr, ptr_arr, ptr_arr, ptr_arr, vp,
                                       sz, vp]
    lib.gemm_ag.argtypes = [vp, i64, i64, i32, i64_arr, ptr_arr, vp, vp, vp, sz, vp]
    lib.gemm_ar_noalloc.argtypes = [vp, i64, i64, i32, i64_arr, ptr_arr, ptr_arr, vp, vp]
    lib.gemm_ag_flagged.argtypes = [vp, i64, i64, i32, i64_arr, ptr_arr, vp, vp, vp,
                                    ctypes.c_uint32, vp, sz, vp]
    lib.gemm_shard_signal.argtypes = [vp, vp, ctypes.c_uint32, vp]
    lib.gemm_shard_pack_gather.argtypes = [vp, i32, i64_arr, i32, i64, ptr_arr, i64, vp, vp, sz, vp]
    lib.gemm_shard_check_status.argtypes = [vp, vp, vp]
    lib.gemm_ar_noalloc_check_status.argtypes = [vp, vp]
    lib.gsr_last_error_string.restype = ctypes.c_char_p
    lib.gemm_shard_describe.argtypes = [vp, i32, i64, i64, i64, i32, i64_arr,
                                        ctypes.POINTER(GsrConfig)]
    for name in EXPORTED:
        if name not in ("gemm_shard_workspace_size", "gsr_last_error_string"):
            getattr(lib, name).restype = i32
    _lib = lib
    return lib


def gsr_last_error_string() -> str:
    return load_library().gsr_last_error_string().decode()


def _check(status: int) -> None:
    if status != GSR_OK:
        raise GsrError(status, gsr_last_error_string())


class Plan:
    """Owns a gemm_shard_plan handle; destroyed with the object."""

    def __init__(self, handle: int, device: int, max_M: int, max_N: int, max_K: int, max_R: int):
        self.handle = ctypes.c_void_p(handle)
        self.device, self.max_M, self.max_N, self.max_K, self.max_R = device, max_M, max_N, max_K, max_R

    def __del__(self):
        if getattr(self, "handle", None) and self.handle.value and _lib is not None:
            _lib.gemm_shard_plan_destroy(self.handle)
            self.handle = ctypes.c_void_p(0)


def gemm_shard_plan_create(device: int, max_M: int, max_N: int, max_K: int, max_R: int) -> Plan:
    lib = load_library()
    h = ctypes.c_void_p()
    _check(lib.gemm_shard_plan_create(ctypes.byref(h), int(device), int(max_M), int(max_N),
                                      int(max_K), int(max_R)))
    return Plan(h.value, device, max_M, max_N, max_K, max_R)


def gemm_shard_plan_create_host(sm_count: int, max_M: int, max_N: int, max_K: int,
                                max_R: int) -> Plan:
    """A plan bound to no device (argument checks, configuration, workspace size)."""
    lib = load_library()
    h = ctypes.c_void_p()
    _check(lib.gemm_shard_plan_create_host(ctypes.byref(h), int(sm_count), int(max_M),
                                           int(max_N), int(max_K), int(max_R)))
    return Plan(h.value, -1, max_M, max_N, max_K, max_R)


def gemm_shard_plan_destroy(plan: Plan) -> None:
    if plan.handle.value:
        _check(load_library().gemm_shard_plan_destroy(plan.handle))
        plan.handle = ctypes.c_void_p(0)


def gemm_shard_plan_set_option(plan: Plan, option: int, value: int) -> None:
    _check(load_library().gemm_shard_plan_set_option(plan.handle, int(option), int(value)))


def gemm_shard_workspace_size(plan: Plan) -> int:
    return int(load_library().gemm_shard_workspace_size(plan.handle))


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _ws(ws: torch.Tensor):
    if not (ws.is_cuda and ws.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return ctypes.c_void_p(ws.data_ptr()), ws.numel() * ws.element_size()


def gemm_shard_workspace_alloc(plan: Plan) -> torch.Tensor:
    """A workspace tensor of gemm_shard_workspace_size bytes (torch allocates it)."""
    n = gemm_shard_workspace_size(plan)
    return torch.empty(n, dtype=torch.uint8, device=f"cuda:{plan.device}")


def gemm_shard_workspace_init(plan: Plan, ws: torch.Tensor, stream=None) -> None:
    p, n = _ws(ws)
    _check(load_library().gemm_shard_workspace_init(plan.handle, p, n, _stream(stream)))


_BF16 = torch.bfloat16


def _bf16_2d(t: torch.Tensor, name: str) -> None:
    if t.dtype is not _BF16 or not t.is_cuda or t.dim() != 2 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D bf16 CUDA tensor")


class PreparedCall:
    """A validated, marshalled call of one entry point on fixed buffers.

    Serving loops reuse the same shard, output and workspace buffers every
    step; preparing the call once moves the per-call Python cost to a single
    ctypes call. The buffers must stay alive and keep their shapes; their
    contents may change. The stream is read at each call unless fixed."""

    def __init__(self, fn, args, keep, stream=None):
        self._fn, self._args, self._keep = fn, args, keep
        self._stream = None if stream is None else _stream(stream)

    def __call__(self, stream=None):
        st = self._stream if stream is None and self._stream is not None else _stream(stream)
        _check(self._fn(*self._args, st))


def _ptrs(ts: Sequence[Optional[torch.Tensor]]):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() if t is not None else 0 for t in ts])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _i64s(vals: Sequence[int]):
    arr = (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_int64)), arr


def _ar_args(plan, X_r, W_r, Y, ws):
    R = len(X_r)
    if R != len(W_r) or R == 0:
        raise ValueError("X_r and W_r need the same, non-zero number of shards")
    _bf16_2d(Y, "Y")
    M, N = Y.shape
    K_r = []
    for r in range(R):
        x, w = X_r[r], W_r[r]
        _bf16_2d(x, f"X_r[{r}]")
        _bf16_2d(w, f"W_r[{r}]")
        k = x.shape[1]
        if x.shape[0] != M or w.shape[0] != N or w.shape[1] != k:
            raise ValueError(f"shard {r}: X_r must be {M} x K_r and W_r {N} x K_r")
        K_r.append(k)
    k, ka = _i64s(K_r)
    xp, xa = _ptrs(X_r)
    wp, wa = _ptrs(W_r)
    wsp, wsn = _ws(ws)
    args = (plan.handle, M, N, R, k, xp, wp, ctypes.c_void_p(Y.data_ptr()), wsp, wsn)
    return args, (ka, xa, wa, X_r, W_r, Y, ws)


def gemm_ar(plan: Plan, X_r: Sequence[torch.Tensor], W_r: Sequence[torch.Tensor],
            Y: torch.Tensor, ws: torch.Tensor, stream=None) -> torch.Tensor:
    """Y = sum_r X_r @ W_r.T (X_r: M x K_r, W_r: N x K_r, Y: M x N, all bf16)."""
    args, keep = _ar_args(plan, X_r, W_r, Y, ws)
    _check(load_library().gemm_ar(*args, _stream(stream)))
    return Y


def prepare_ar(plan: Plan, X_r, W_r, Y, ws, stream=None) -> PreparedCall:
    """gemm_ar on fixed buffers, validated and marshalled once."""
    args, keep = _ar_args(plan, X_r, W_r, Y, ws)
    return PreparedCall(load_library().gemm_ar, args, keep, stream)


def gemm_ar_replicated(plan: Plan, X_r: Sequence[torch.Tensor], W_r: Sequence[torch.Tensor],
                       Y_r: Sequence[torch.Tensor], ws: torch.Tensor, stream=None):
    """Y_r[r] = sum_q X_q @ W_q.T for every r (R outputs of M x N, all bf16)."""
    R = len(X_r)
    if len(Y_r) != R:
        raise ValueError("need one output per shard")
    for r in range(R):
        _bf16_2d(Y_r[r], f"Y_r[{r}]")
        if Y_r[r].shape != Y_r[0].shape:
            raise ValueError("all outputs must have the same shape")
    args, keep = _ar_args(plan, X_r, W_r, Y_r[0], ws)
    yp, ya = _ptrs(Y_r)
    # same marshalling as gemm_ar, with the output pointer array in place of Y
    args = args[:7] + (yp,) + args[8:]
    _check(load_library().gemm_ar_replicated(*args, _stream(stream)))
    return Y_r


def gemm_ar_noalloc(plan: Plan, X_r: Sequence[torch.Tensor], W_r: Sequence[torch.Tensor],
                    Y: torch.Tensor, stream=None) -> torch.Tensor:
    """gemm_ar for callers that cannot allocate device memory: no workspace; the
    library's built-in 24 MiB device scratch is used (shared by every call on a
    device, so calls must not overlap on the GPU)."""
    R = len(X_r)
    if R != len(W_r) or R == 0:
        raise ValueError("X_r and W_r need the same, non-zero number of shards")
    for r in range(R):
        _bf16_2d(X_r[r], f"X_r[{r}]")
        _bf16_2d(W_r[r], f"W_r[{r}]")
    _bf16_2d(Y, "Y")
    M, N = Y.shape
    K_r = [x.shape[1] for x in X_r]
    for r in range(R):
        if X_r[r].shape[0] != M or W_r[r].shape != (N, K_r[r]):
            raise ValueError(f"shard {r}: X_r must be {M} x K_r and W_r {N} x K_r")
    k, ka = _i64s(K_r)
    xp, xa = _ptrs(X_r)
    wp, wa = _ptrs(W_r)
    _check(load_library().gemm_ar_noalloc(plan.handle, M, N, R, k, xp, wp,
                                          ctypes.c_void_p(Y.data_ptr()), _stream(stream)))
    return Y


def gemm_ar_noalloc_check_status(plan: Plan, stream=None) -> None:
    """Synchronise, then raise GsrError(GSR_ERR_TIMEOUT) if the last
    gemm_ar_noalloc call on the plan's device had an in-kernel wait run out."""
    _check(load_library().gemm_ar_noalloc_check_status(plan.handle, _stream(stream)))


def _rs_args(plan, X_r, W_r, Y_r, ws, M=None):
    R = len(X_r)
    if R != len(W_r) or R != len(Y_r) or R == 0:
        raise ValueError("X_r, W_r and Y_r need the same, non-zero number of shards")
    M = X_r[0].shape[0] if M is None else int(M)
    N = W_r[0].shape[0]
    rps = -(-M // R)
    K_r = []
    for r in range(R):
        _bf16_2d(X_r[r], f"X_r[{r}]")
        _bf16_2d(W_r[r], f"W_r[{r}]")
        _bf16_2d(Y_r[r], f"Y_r[{r}]")
        k = X_r[r].shape[1]
        if X_r[r].shape[0] != M or W_r[r].shape != (N, k):
            raise ValueError(f"shard {r}: X_r must be {M} x K_r and W_r {N} x K_r")
        if Y_r[r].shape[0] < rps or Y_r[r].shape[1] != N:
            raise ValueError(f"Y_r[{r}] must hold at least {rps} rows of {N}")
        K_r.append(k)
    k, ka = _i64s(K_r)
    xp, xa = _ptrs(X_r)
    wp, wa = _ptrs(W_r)
    yp, ya = _ptrs(Y_r)
    wsp, wsn = _ws(ws)
    args = (plan.handle, M, N, R, k, xp, wp, yp, wsp, wsn)
    return args, (ka, xa, wa, ya, X_r, W_r, Y_r, ws)


def gemm_rs(plan: Plan, X_r: Sequence[torch.Tensor], W_r: Sequence[torch.Tensor],
            Y_r: Sequence[torch.Tensor], ws: torch.Tensor, M: Optional[int] = None,
            stream=None) -> Sequence[torch.Tensor]:
    """Y_r[s] = rows [s*rps, min(M,(s+1)*rps)) of sum_r X_r @ W_r.T, rps = ceil(M/R)."""
    args, keep = _rs_args(plan, X_r, W_r, Y_r, ws, M)
    _check(load_library().gemm_rs(*args, _stream(stream)))
    return Y_r


def prepare_rs(plan: Plan, X_r, W_r, Y_r, ws, M=None, stream=None) -> PreparedCall:
    """gemm_rs on fixed buffers, validated and marshalled once."""
    args, keep = _rs_args(plan, X_r, W_r, Y_r, ws, M)
    return PreparedCall(load_library().gemm_rs, args, keep, stream)


def _ag_call_args(plan, A_r, W, Y, ws):
    N, K, M_r = _ag_args(A_r, W, Y)
    m, ma = _i64s(M_r)
    ap, aa = _ptrs([a if a.numel() else None for a in A_r])
    wsp, wsn = _ws(ws)
    args = (plan.handle, N, K, len(A_r), m, ap, ctypes.c_void_p(W.data_ptr()),
            ctypes.c_void_p(Y.data_ptr()), wsp, wsn)
    return args, (ma, aa, A_r, W, Y, ws)


def gemm_ag(plan: Plan, A_r: Sequence[torch.Tensor], W: torch.Tensor, Y: torch.Tensor,
            ws: torch.Tensor, stream=None) -> torch.Tensor:
    """Y = cat(A_r) @ W.T (A_r: M_r x K, W: N x K, Y: sum(M_r) x N, all bf16)."""
    args, keep = _ag_call_args(plan, A_r, W, Y, ws)
    _check(load_library().gemm_ag(*args, _stream(stream)))
    return Y


def prepare_ag(plan: Plan, A_r, W, Y, ws, stream=None) -> PreparedCall:
    """gemm_ag on fixed buffers, validated and marshalled once."""
    args, keep = _ag_call_args(plan, A_r, W, Y, ws)
    return PreparedCall(load_library().gemm_ag, args, keep, stream)


def _ag_args(A_r, W, Y):
    R = len(A_r)
    if R == 0:
        raise ValueError("need at least one shard")
    _bf16_2d(W, "W")
    _bf16_2d(Y, "Y")
    N, K = W.shape
    M_r = []
    for r, a in enumerate(A_r):
        if a.numel() == 0:
            M_r.append(0)
            continue
        _bf16_2d(a, f"A_r[{r}]")
        if a.shape[1] != K:
            raise ValueError(f"A_r[{r}] must have K={K} columns")
        M_r.append(a.shape[0])
    if Y.shape != (sum(M_r), N):
        raise ValueError(f"Y must be {sum(M_r)} x {N}")
    return N, K, M_r


def gemm_ag_flagged(plan: Plan, A_r: Sequence[torch.Tensor], W: torch.Tensor, Y: torch.Tensor,
                    ready: torch.Tensor, epoch: int, ws: torch.Tensor, stream=None) -> torch.Tensor:
    """gemm_ag that waits in the kernel until ready[r] reaches epoch before reading A_r.
    `ready` is a CUDA int32/uint32 tensor of R words."""
    N, K, M_r = _ag_args(A_r, W, Y)
    if not ready.is_cuda or ready.numel() < len(A_r) or ready.element_size() != 4:
        raise ValueError("ready must be a CUDA tensor of R 32-bit words")
    m, ma = _i64s(M_r)
    ap, aa = _ptrs([a if a.numel() else None for a in A_r])
    wsp, wsn = _ws(ws)
    _check(load_library().gemm_ag_flagged(plan.handle, N, K, len(A_r), m, ap,
                                          ctypes.c_void_p(W.data_ptr()),
                                          ctypes.c_void_p(Y.data_ptr()),
                                          ctypes.c_void_p(ready.data_ptr()),
                                          ctypes.c_uint32(epoch & 0xFFFFFFFF), wsp, wsn,
                                          _stream(stream)))
    return Y


def gemm_shard_signal(plan: Plan, flag_ptr: int, value: int, stream=None) -> None:
    """Enqueue a write of `value` to the device word at `flag_ptr` on `stream`."""
    _check(load_library().gemm_shard_signal(plan.handle, ctypes.c_void_p(int(flag_ptr)),
                                            ctypes.c_uint32(value & 0xFFFFFFFF), _stream(stream)))


def gemm_shard_check_status(plan: Plan, ws: torch.Tensor, stream=None) -> None:
    p, _ = _ws(ws)
    _check(load_library().gemm_shard_check_status(plan.handle, p, _stream(stream)))


def gemm_shard_describe(plan: Plan, mode: int, M: int, N: int, K: int,
                        sizes: Sequence[int]) -> dict:
    lib = load_library()
    s, sa = _i64s(sizes)
    cfg = GsrConfig()
    _check(lib.gemm_shard_describe(plan.handle, int(mode), int(M), int(N), int(K), len(sizes), s,
                                   ctypes.byref(cfg)))
    return {name: getattr(cfg, name) for name, _ in GsrConfig._fields_}


def _pack_args(plan, S, rows_out, P, ws):
    R = len(S)
    if R == 0 or any(len(s) != len(S[0]) for s in S) or not S[0]:
        raise ValueError("S must hold R >= 1 shards with the same T >= 1 states each")
    T = len(S[0])
    _bf16_2d(P, "P")
    H = P.shape[1] // T
    if P.shape != (rows_out, T * H) or H * T != P.shape[1]:
        raise ValueError(f"P must be rows_out x (T*H) = {rows_out} x {T}*H")
    M_r, flat = [], []
    for r, states in enumerate(S):
        m = states[0].shape[0]
        for t, st in enumerate(states):
            if st.numel() == 0 and m == 0:
                flat.append(None)
                continue
            _bf16_2d(st, f"S[{r}][{t}]")
            if st.shape != (m, H):
                raise ValueError(f"S[{r}][{t}] must be {m} x {H}")
            flat.append(st)
        M_r.append(m)
    m, ma = _i64s(M_r)
    sp, sa = _ptrs(flat)
    wsp, wsn = _ws(ws)
    args = (plan.handle, R, m, T, H, sp, rows_out, ctypes.c_void_p(P.data_ptr()), wsp, wsn)
    return args, (ma, sa, S, P, ws)


def gemm_shard_pack_gather(plan: Plan, S: Sequence[Sequence[torch.Tensor]], rows_out: int,
                           P: torch.Tensor, ws: torch.Tensor, stream=None) -> torch.Tensor:
    """P[g, t*H:(t+1)*H] = cat_r(S[r][t])[g] for g < rows_out (S[r][t]: M_r x H, bf16;
    P: rows_out x T*H). Returns P; the state-t view is P[:, t*H:(t+1)*H]."""
    args, keep = _pack_args(plan, S, rows_out, P, ws)
    _check(load_library().gemm_shard_pack_gather(*args, _stream(stream)))
    return P


def prepare_pack_gather(plan: Plan, S, rows_out, P, ws, stream=None) -> PreparedCall:
    """gemm_shard_pack_gather on fixed buffers, validated and marshalled once."""
    args, keep = _pack_args(plan, S, rows_out, P, ws)
    return PreparedCall(load_library().gemm_shard_pack_gather, args, keep, stream)
