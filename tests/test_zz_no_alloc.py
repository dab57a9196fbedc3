"""gemm_ar_noalloc: the AR entry point for callers that cannot allocate device
memory (for example an inference engine that has claimed all free HBM for its
KV cache, or a caller that cannot afford cudaMalloc's implicit device
synchronisation). It runs with the library's built-in device scratch instead of
a caller workspace. This file is collected last, so that a run stopping at the
first failure has already run every other test."""
import pytest
import torch

from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import build as gbuild
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import assert_close, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def setup():
    gbuild.build()
    plan = B.gemm_shard_plan_create(0, 4096, 8192, 8192, 16)
    ws = B.gemm_shard_workspace_alloc(plan)
    B.gemm_shard_workspace_init(plan, ws)
    return plan, ws


def _device_inputs(M, N, K_r, seed):
    inp = gi.gaussian_ar(M, N, K_r, seed=seed)
    dev = torch.device("cuda:0")
    return [x.to(dev) for x in inp.X_r], [w.to(dev) for w in inp.W_r]


def test_noalloc_matches_workspace_entry_point_on_two_calls(setup):
    plan, ws = setup
    # M=128 cuts every tile's k range into pieces (the scratch holds the fp32
    # partials and the arrival counters); the second call uses other inputs and
    # another shape.
    cases = [(128, 7168, [896] * 8, 11), (300, 1032, [72, 200, 64], 12)]
    d = B.gemm_shard_describe(plan, B.MODE_AR, 128, 7168, 0, [896] * 8)
    assert d["split"] > 1 or d["sk_iters"] > 0
    for M, N, K_r, seed in cases:
        X, W = _device_inputs(M, N, K_r, seed)
        y_ref = torch.empty(M, N, dtype=torch.bfloat16, device="cuda:0")
        y_new = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda:0")
        B.gemm_ar(plan, X, W, y_ref, ws)
        B.gemm_ar_noalloc(plan, X, W, y_new)
        torch.cuda.synchronize()
        assert_close(to_f64(y_new), to_f64(y_ref), f"noalloc vs gemm_ar, M={M}")


def test_noalloc_rejects_oversized_scratch(setup):
    plan = B.gemm_shard_plan_create(0, 4096, 8192, 8192, 16)
    B.gemm_shard_plan_set_option(plan, B.GSR_OPT_SPLIT_K, 16)
    X, W = _device_inputs(1024, 4096, [512, 512], 13)
    Y = torch.empty(1024, 4096, dtype=torch.bfloat16, device="cuda:0")
    with pytest.raises(B.GsrError) as e:
        B.gemm_ar_noalloc(plan, X, W, Y)
    assert e.value.status == B.GSR_ERR_WORKSPACE
    assert "built-in scratch" in str(e.value)


def test_noalloc_falls_back_when_the_heuristic_needs_more_scratch(setup):
    """M=2560, N=7168: the plan's stream-K configuration (280 pair tiles on 76
    pairs, a 52-tile partial wave) needs more scratch than the built-in array
    holds, so the call runs the uniform schedule; results agree with gemm_ar
    within the test tolerance, on two calls in a row."""
    plan, ws = setup
    d = B.gemm_shard_describe(plan, B.MODE_AR, 2560, 7168, 0, [896] * 8)
    assert d["schedule"] == 2 and d["workspace_bytes"] > 24 << 20
    for seed in (31, 32):
        X, W = _device_inputs(2560, 7168, [896] * 8, seed)
        y_ref = torch.empty(2560, 7168, dtype=torch.bfloat16, device="cuda:0")
        y_new = torch.full((2560, 7168), float("nan"), dtype=torch.bfloat16, device="cuda:0")
        B.gemm_ar(plan, X, W, y_ref, ws)
        B.gemm_ar_noalloc(plan, X, W, y_new)
        torch.cuda.synchronize()
        assert_close(to_f64(y_new), to_f64(y_ref), f"noalloc fallback, seed {seed}")
