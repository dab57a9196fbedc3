"""gemm_ar_noalloc: the AR entry point for callers that cannot allocate device
memory (for example an inference engine that has claimed all free HBM for its
KV cache, or a caller that cannot afford cudaMalloc's implicit device
synchronisation). It runs with the library's built-in device scratch instead of
a caller workspace. This file is collected last, so that a run stopping at the
first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import build as gbuild
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import assert_close, bits_of, to_f64

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 24 << 20


@pytest.fixture(scope="module")
def setup():
    gbuild.build()
    plan = B.gemm_shard_plan_create(0, 4096, 8192, 8192, 16)
    ws = B.gemm_shard_workspace_alloc(plan)
    B.gemm_shard_workspace_init(plan, ws)
    return plan, ws


def _inputs(M, N, K_r, seed):
    inp = gi.gaussian_ar(M, N, K_r, seed=seed)
    dev = torch.device("cuda:0")
    return inp, [x.to(dev) for x in inp.X_r], [w.to(dev) for w in inp.W_r]


def test_noalloc_equals_workspace_entry_point_bit_for_bit_on_calls_in_a_row(setup):
    """Where the plan's own configuration fits the built-in scratch, the call
    runs exactly gemm_ar's kernel configuration and summation order, so the
    outputs must be bit-identical. The three calls in a row reuse the one
    array: M=1000 cuts tail tiles into pieces (fp32 partial slots and arrival
    counters in the scratch), M=700 cuts every tile into three uniform
    pieces, M=128 runs the small-M kernel (only the status word)."""
    plan, ws = setup
    cases = [(1000, 7168, [896] * 8, 11, 4), (700, 2048, [512, 512], 12, 1),
             (128, 7168, [896] * 8, 13, 3)]
    for M, N, K_r, seed, schedule in cases:
        d = B.gemm_shard_describe(plan, B.MODE_AR, M, N, 0, K_r)
        assert d["schedule"] == schedule and d["workspace_bytes"] <= SCRATCH_BYTES, d
        if schedule != 3:
            assert d["split"] > 1
        inp, X, W = _inputs(M, N, K_r, seed)
        y_ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda:0")
        y_new = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda:0")
        B.gemm_ar(plan, X, W, y_ref, ws)
        B.gemm_ar_noalloc(plan, X, W, y_new)
        B.gemm_ar_noalloc_check_status(plan)
        assert np.array_equal(bits_of(y_new), bits_of(y_ref)), f"noalloc vs gemm_ar, M={M}"
        if M == 1000:
            assert_close(to_f64(y_new), oracle.ar(inp.X_r, inp.W_r), "noalloc vs the oracle")


def test_noalloc_rejects_oversized_scratch(setup):
    plan = B.gemm_shard_plan_create(0, 4096, 8192, 8192, 16)
    B.gemm_shard_plan_set_option(plan, B.GSR_OPT_SPLIT_K, 16)
    _, X, W = _inputs(1024, 4096, [512, 512], 13)
    Y = torch.empty(1024, 4096, dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(B.GsrError) as e:
        B.gemm_ar_noalloc(plan, X, W, Y)
    assert e.value.status == B.GSR_ERR_WORKSPACE
    assert "built-in scratch" in str(e.value)


def test_noalloc_falls_back_when_the_heuristic_needs_more_scratch(setup):
    """M=2560, N=7168: the plan's stream-K configuration (280 pair tiles on 76
    pairs, a 52-tile partial wave) needs more scratch than the built-in array
    holds, so the call runs the uniform schedule: another summation order, so
    the results agree with gemm_ar within the test tolerance, not bit for bit,
    on two calls in a row."""
    plan, ws = setup
    d = B.gemm_shard_describe(plan, B.MODE_AR, 2560, 7168, 0, [896] * 8)
    assert d["schedule"] == 2 and d["workspace_bytes"] > SCRATCH_BYTES
    for seed in (31, 32):
        _, X, W = _inputs(2560, 7168, [896] * 8, seed)
        y_ref = torch.empty(2560, 7168, dtype=torch.bfloat16, device="cuda:0")
        y_new = torch.full((2560, 7168), float("nan"), dtype=torch.bfloat16, device="cuda:0")
        B.gemm_ar(plan, X, W, y_ref, ws)
        B.gemm_ar_noalloc(plan, X, W, y_new)
        B.gemm_ar_noalloc_check_status(plan)
        assert_close(to_f64(y_new), to_f64(y_ref), f"noalloc fallback, seed {seed}")
