"""Helpers shared by the GPU tests: plans, guarded output buffers and the
element-wise parity check against the oracle."""
from __future__ import annotations

import numpy as np
import torch

from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import build as gbuild

# Per-element bound of the parity check: |y - ref| <= RTOL * |ref| + ATOL.
RTOL = 1e-2
ATOL = 1e-2
SENTINEL = 0x7FC1          # a bf16 NaN pattern no computation produces here
GUARD_ROWS = 2


def device() -> torch.device:
    return torch.device("cuda:0")


_PLANS = {}


def plan(max_M=34816, max_N=8192, max_K=8192, max_R=16, **options):
    """Options are GSR_OPT_* names in lower case (split_k, block_n, cta_group, ...)."""
    """A cached plan + initialised workspace for the given maxima and options."""
    key = (max_M, max_N, max_K, max_R, tuple(sorted(options.items())))
    if key not in _PLANS:
        gbuild.build()
        p = B.gemm_shard_plan_create(0, max_M, max_N, max_K, max_R)
        for name, value in options.items():
            B.gemm_shard_plan_set_option(p, getattr(B, f"GSR_OPT_{name.upper()}"), value)
        ws = B.gemm_shard_workspace_alloc(p)
        B.gemm_shard_workspace_init(p, ws)
        _PLANS[key] = (p, ws)
    return _PLANS[key]


class Guarded:
    """A rows x N bf16 output with GUARD_ROWS sentinel rows before and after."""

    def __init__(self, rows: int, N: int, dev=None):
        dev = dev or device()
        self.rows, self.N = rows, N
        self.full = torch.full((rows + 2 * GUARD_ROWS, N), 0, dtype=torch.int16, device=dev)
        self.full.fill_(SENTINEL)
        self.full = self.full.view(torch.bfloat16)
        self.out = self.full[GUARD_ROWS:GUARD_ROWS + rows]

    def bits(self) -> np.ndarray:
        return self.full.view(torch.int16).cpu().numpy().view(np.uint16)

    def guards_intact(self, valid_rows: int | None = None) -> bool:
        b = self.bits()
        v = self.rows if valid_rows is None else valid_rows
        pre = b[:GUARD_ROWS]
        post = b[GUARD_ROWS + v:]
        return bool((pre == SENTINEL).all() and (post == SENTINEL).all())


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(torch.float64).cpu().numpy()


def assert_close(y: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.isfinite(y).all(), f"{what}: non-finite output"
    err = np.abs(y - ref)
    bound = RTOL * np.abs(ref) + ATOL
    bad = err > bound
    assert not bad.any(), (
        f"{what}: {int(bad.sum())} of {bad.size} elements out of bound; "
        f"max abs err {err.max():.4g}, max rel err {(err / (np.abs(ref) + 1e-30)).max():.4g}")


def shards_to(dev, tensors, reverse_order=False):
    """Copy shards to the device, each in its own allocation (optionally in reverse
    allocation order, with spacer allocations in between)."""
    out = [None] * len(tensors)
    spacers = []
    order = range(len(tensors) - 1, -1, -1) if reverse_order else range(len(tensors))
    for i in order:
        out[i] = tensors[i].to(dev).contiguous()
        if reverse_order:
            spacers.append(torch.empty(4096 + 512 * i, dtype=torch.uint8, device=dev))
    return out, spacers


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# One line per element-wise comparison at full size, printed in the run's
# terminal summary (conftest.py).
PARITY_LOG: list = []


class ParityStats:
    """Running element-wise comparison of a GPU output with the oracle, block by
    block: the count of elements over |y - ref| <= RTOL*|ref| + ATOL, the max
    abs error, the max relative error over |ref| >= ATOL, and how much of the
    bound the worst element used."""

    def __init__(self, what: str):
        self.what = what
        self.n = 0
        self.bad = 0
        self.nonfinite = 0
        self.max_abs = 0.0
        self.max_rel = 0.0
        self.max_bound_use = 0.0

    def add(self, y: np.ndarray, ref: np.ndarray) -> None:
        assert y.shape == ref.shape, (y.shape, ref.shape)
        self.n += y.size
        fin = np.isfinite(y)
        self.nonfinite += int(y.size - np.count_nonzero(fin))
        err = np.abs(y - ref)
        aref = np.abs(ref)
        bound = RTOL * aref + ATOL
        self.bad += int(np.count_nonzero(~(err <= bound)))
        if y.size:
            self.max_abs = max(self.max_abs, float(np.nanmax(np.where(fin, err, 0.0))))
            self.max_bound_use = max(self.max_bound_use,
                                     float(np.nanmax(np.where(fin, err / bound, np.inf))))
            big = aref >= ATOL
            if big.any():
                self.max_rel = max(self.max_rel,
                                   float(np.nanmax(np.where(fin & big, err, 0.0)[big] / aref[big])))

    def line(self) -> str:
        return (f"{self.what}: {self.n} elements, {self.bad} over the bound, "
                f"{self.nonfinite} non-finite; max abs err {self.max_abs:.3g}, "
                f"max rel err {self.max_rel:.3g} (|ref| >= {ATOL:g}), "
                f"worst element at {self.max_bound_use:.3f} of its bound")

    def finish(self, expect_elements: int | None = None) -> None:
        PARITY_LOG.append(self.line())
        if expect_elements is not None:
            assert self.n == expect_elements, f"{self.what}: compared {self.n} of {expect_elements}"
        assert self.nonfinite == 0 and self.bad == 0, self.line()
