"""Seeded synthetic inputs for the shard-reduction GEMM, shared by the tests,
the benchmark and the smoke check.

This module draws random numbers and slices them into shard buffers. It holds
none of the method's arithmetic: no product, no sum over shards, no rounding of
results. Every bf16 tensor it returns is the round-to-nearest-even cast of an
fp32 draw (``Tensor.to(torch.bfloat16)``).

Recipe (the projections of the Kimi-K3 serving pages: the GEMM-RS/AR kernel
page, test section, and the AG-GEMM page, microbenchmark tables):

* AR/RS: draw the full activation ``X`` (``M x K``, fp32 ``randn``) and then the
  full weight ``W`` (``N x K``, ``randn / sqrt(K)``) from one CPU generator
  seeded with ``seed``; cast both to bf16; copy K-column slices of widths
  ``K_r`` into R separate contiguous buffers ``X_r`` (``M x K_r``) and
  ``W_r`` (``N x K_r``).
* AG: draw ``A`` (``sum(M_r) x K``) then ``W`` (``N x K``, ``randn/sqrt(K)``);
  cast; copy M-row slices into R separate buffers ``A_r`` (``M_r x K``).
* Integer-valued variants draw uniform integers in ``[-amp, amp]``; every such
  value is exact in bf16, so products and sums of them are exact in fp64.

The default seed of a workload is ``2000 + M + K``, after the seeding rule of
the GEMM-RS/AR page's test (``manual_seed(2000 + M + K)``); the tiny AR case
uses seed 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Sequence

import torch


def _gen(seed: int, device: str | torch.device = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def default_seed(M: int, K: int) -> int:
    return 2000 + int(M) + int(K)


@dataclass
class ARInputs:
    """K-sharded operands: ``X_r`` is ``M x K_r``, ``W_r`` is ``N x K_r``."""
    M: int
    N: int
    K_r: List[int]
    X_r: List[torch.Tensor]
    W_r: List[torch.Tensor]

    @property
    def R(self) -> int:
        return len(self.K_r)

    @property
    def K(self) -> int:
        return sum(self.K_r)


@dataclass
class AGInputs:
    """M-sharded operands: ``A_r`` is ``M_r x K``, ``W`` is ``N x K``."""
    N: int
    K: int
    M_r: List[int]
    A_r: List[torch.Tensor]
    W: torch.Tensor

    @property
    def R(self) -> int:
        return len(self.M_r)

    @property
    def M(self) -> int:
        return sum(self.M_r)


def _split_cols(t: torch.Tensor, widths: Sequence[int]) -> List[torch.Tensor]:
    out, c = [], 0
    for w in widths:
        out.append(t[:, c:c + w].contiguous().clone())
        c += w
    return out


def _split_rows(t: torch.Tensor, heights: Sequence[int]) -> List[torch.Tensor]:
    out, r = [], 0
    for h in heights:
        out.append(t[r:r + h, :].contiguous().clone())
        r += h
    return out


def gaussian_ar(M: int, N: int, K_r: Sequence[int], seed: int | None = None,
                device: str | torch.device = "cpu") -> ARInputs:
    """X ~ N(0,1), W ~ N(0,1/K) in bf16, sliced into K-shards."""
    K_r = [int(k) for k in K_r]
    K = sum(K_r)
    if seed is None:
        seed = default_seed(M, K)
    g = _gen(seed, device)
    X = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    W = torch.randn(N, K, generator=g, device=device, dtype=torch.float32)
    W.div_(math.sqrt(K))
    Xb = X.to(torch.bfloat16)
    del X
    Wb = W.to(torch.bfloat16)
    del W
    return ARInputs(M, N, K_r, _split_cols(Xb, K_r), _split_cols(Wb, K_r))


def gaussian_ag(M_r: Sequence[int], N: int, K: int, seed: int | None = None,
                device: str | torch.device = "cpu") -> AGInputs:
    """A ~ N(0,1), W ~ N(0,1/K) in bf16, A sliced into M-row shards."""
    M_r = [int(m) for m in M_r]
    M = sum(M_r)
    if seed is None:
        seed = default_seed(M, K)
    g = _gen(seed, device)
    A = torch.randn(M, K, generator=g, device=device, dtype=torch.float32)
    W = torch.randn(N, K, generator=g, device=device, dtype=torch.float32)
    W.div_(math.sqrt(K))
    Ab = A.to(torch.bfloat16)
    del A
    Wb = W.to(torch.bfloat16).contiguous()
    del W
    return AGInputs(N, K, M_r, _split_rows(Ab, M_r), Wb)


def _randint(shape, amp: int, g: torch.Generator, device) -> torch.Tensor:
    return torch.randint(-amp, amp + 1, shape, generator=g, device=device,
                         dtype=torch.int64).to(torch.bfloat16)


def integer_ar(M: int, N: int, K_r: Sequence[int], amp: int = 3, seed: int = 1,
               device: str | torch.device = "cpu") -> ARInputs:
    """Uniform integers in [-amp, amp] (exact in bf16), sliced into K-shards."""
    K_r = [int(k) for k in K_r]
    g = _gen(seed, device)
    X = _randint((M, sum(K_r)), amp, g, device)
    W = _randint((N, sum(K_r)), amp, g, device)
    return ARInputs(M, N, K_r, _split_cols(X, K_r), _split_cols(W, K_r))


def integer_ag(M_r: Sequence[int], N: int, K: int, amp: int = 3, seed: int = 1,
               device: str | torch.device = "cpu") -> AGInputs:
    """Uniform integers in [-amp, amp] (exact in bf16), sliced into M-shards."""
    M_r = [int(m) for m in M_r]
    g = _gen(seed, device)
    A = _randint((sum(M_r), K), amp, g, device)
    W = _randint((N, K), amp, g, device).contiguous()
    return AGInputs(N, K, M_r, _split_rows(A, M_r), W)


def gaussian_states(M_r: Sequence[int], T: int, H: int, seed: int = 1,
                    device: str | torch.device = "cpu") -> List[List[torch.Tensor]]:
    """T states per shard (the hidden state and T-1 auxiliary states of the
    packed gather), N(0,1) in bf16: S[r][t] is M_r x H, each its own allocation."""
    g = _gen(seed, device)
    return [[torch.randn(int(m), H, generator=g, device=device).to(torch.bfloat16)
             for _ in range(T)] for m in M_r]


@dataclass(frozen=True)
class PackWorkload:
    """A packed gather: R shards of M_r rows, T states of H columns, the first
    rows_out rows kept (the token count before sequence-parallel padding)."""
    name: str
    R: int
    M_r: int
    T: int
    H: int
    rows_out: int
    seed: int = 7

    @property
    def bytes(self) -> int:
        """Algorithmic bytes: every kept state row read once, P written once."""
        return 2 * (2 * self.rows_out * self.T * self.H)


# Kimi-K3-like: hidden size 7168, the hidden state and three auxiliary states,
# 8 sequence-parallel shards of 4096 rows, 5 padding rows dropped.
PACK_SP = PackWorkload("pack_sp_t4", R=8, M_r=4096, T=4, H=7168, rows_out=8 * 4096 - 5)


def bf16_bits(t: torch.Tensor):
    """The raw bf16 bit patterns of a CPU tensor as a numpy uint16 array."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


# Workloads: the projection shapes of the pages (AG-GEMM page, microbenchmark
# and component-breakdown tables; GEMM-RS/AR page, o_proj call sites).

@dataclass(frozen=True)
class Workload:
    name: str
    mode: str                 # "ar", "rs" or "ag"
    N: int
    K: int                    # total reduction length
    R: int
    M: int                    # AR/RS rows, or global AG rows
    seed: int | None = None
    sizes: tuple = field(default=())   # K_r (AR/RS) or M_r (AG)

    def shard_sizes(self) -> List[int]:
        if self.sizes:
            return list(self.sizes)
        if self.mode == "ag":
            return [self.M // self.R] * self.R
        return [self.K // self.R] * self.R

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def bytes(self) -> int:
        """Algorithmic bytes: each input read once, the output written once."""
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


AR_TINY = Workload("ar_tiny", "ar", N=256, K=256, R=2, M=128, seed=0)
AG_LOCAL_M = (256, 384, 448, 512, 1024, 2048, 4096)
AG_KDA = [Workload(f"ag_kda_m{8 * m}", "ag", N=6288, K=7168, R=8, M=8 * m)
          for m in AG_LOCAL_M]
AG_MLA = [Workload(f"ag_mla_m{8 * m}", "ag", N=3648, K=7168, R=8, M=8 * m)
          for m in AG_LOCAL_M]
AR_OPROJ = [Workload(f"ar_oproj_m{m}", "ar", N=7168, K=7168, R=8, M=m)
            for m in (128, 129, 1000, 4096, 32768)]
# Decode batches below 128 rows, where the pages' fused AR was slower than the
# unfused path (GEMM-RS/AR page, risks and impact): the same projection.
AR_DECODE = [Workload(f"ar_oproj_m{m}", "ar", N=7168, K=7168, R=8, M=m) for m in (1, 16, 64)]
# The largest batch the small-M kernel serves (its 256-row MMA form).
AR_SMALL_TOP = [Workload("ar_oproj_m256", "ar", N=7168, K=7168, R=8, M=256)]
# RS shares its seed with AR o_proj M=32768, so one set of inputs serves both.
RS_ALL = [Workload(f"rs_r{r}", "rs", N=7168, K=7168, R=r, M=32768,
                   seed=default_seed(32768, 7168)) for r in (2, 4, 8, 16)]
ALL_WORKLOADS = [AR_TINY] + AG_KDA + AG_MLA + AR_DECODE + AR_OPROJ[:2] + AR_SMALL_TOP + AR_OPROJ[2:] + RS_ALL


def make_inputs(w: Workload, device: str | torch.device = "cpu"):
    if w.mode == "ag":
        return gaussian_ag(w.shard_sizes(), w.N, w.K, seed=w.seed, device=device)
    return gaussian_ar(w.M, w.N, w.shard_sizes(), seed=w.seed, device=device)
