"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times (same plan maxima, heuristic configuration).

The projections: AG KDA-like (N=6288) and MLA-like (N=3648) with R=8 shards of
256..4096 rows and K=7168 (AG-GEMM page, microbenchmark tables); AR o_proj-like
(R=8 K-shards of 896, N=7168, M in {128, 129, 1000, 4096, 32768}); RS with
R in {2,4,8,16} at M=32768. Inputs are seeded on the device (torch's CUDA
generator, same recipe as the CPU one) and copied to the host for the oracle,
which checks whole rows at every tile and shard boundary plus random rows and
random points. RS must equal the matching rows of AR bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import assert_close, bits_of, device, plan

pytestmark = pytest.mark.gpu


def sample_rows(M: int, boundaries, n_random: int = 12, seed: int = 0):
    rows = {0, 1, M - 1, M - 2}
    for b in boundaries:
        for d in (-1, 0, 1):
            if 0 <= b + d < M:
                rows.add(b + d)
    for t in range(128, M, 128 * max(1, M // (128 * 16))):
        rows.update({t - 1, t})
    rng = np.random.default_rng(seed)
    rows.update(int(r) for r in rng.integers(0, M, n_random))
    return np.array(sorted(r for r in rows if 0 <= r < M))


def check_rows(Y_dev: torch.Tensor, rows, ref_fn, N, what):
    y = Y_dev[torch.as_tensor(rows, device=Y_dev.device)].to(torch.float64).cpu().numpy()
    r = np.repeat(rows, N)
    c = np.tile(np.arange(N), len(rows))
    ref = ref_fn(r, c).reshape(len(rows), N)
    assert_close(y, ref, what + " (rows)")


def check_points(Y_dev, M, N, ref_fn, what, n=4000, seed=1):
    rng = np.random.default_rng(seed)
    r, c = rng.integers(0, M, n), rng.integers(0, N, n)
    y = Y_dev[torch.as_tensor(r, device=Y_dev.device), torch.as_tensor(c, device=Y_dev.device)]
    assert_close(y.to(torch.float64).cpu().numpy(), ref_fn(r, c), what + " (points)")


@pytest.mark.parametrize("w", gi.AG_KDA + gi.AG_MLA, ids=lambda w: w.name)
def test_ag_full_size(w):
    p, ws = plan()
    dev = device()
    inp = gi.make_inputs(w, device=dev)
    Y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    B.gemm_ag(p, inp.A_r, inp.W, Y, ws)
    B.gemm_shard_check_status(p, ws)
    A_h = [a.cpu() for a in inp.A_r]
    W_h = inp.W.cpu()
    bounds = list(np.cumsum([0] + inp.M_r))
    ref = lambda r, c: oracle.ag_at(A_h, W_h, r, c)
    check_rows(Y, sample_rows(w.M, bounds), ref, w.N, w.name)
    check_points(Y, w.M, w.N, ref, w.name)
    assert torch.isfinite(Y.float()).all()


@pytest.mark.parametrize("w", gi.AR_OPROJ, ids=lambda w: w.name)
def test_ar_full_size(w):
    p, ws = plan()
    dev = device()
    inp = gi.make_inputs(w, device=dev)
    Y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    B.gemm_ar(p, inp.X_r, inp.W_r, Y, ws)
    B.gemm_shard_check_status(p, ws)
    X_h = [x.cpu() for x in inp.X_r]
    W_h = [x.cpu() for x in inp.W_r]
    ref = lambda r, c: oracle.ar_at(X_h, W_h, r, c)
    check_rows(Y, sample_rows(w.M, []), ref, w.N, w.name)
    check_points(Y, w.M, w.N, ref, w.name)
    assert torch.isfinite(Y.float()).all()


@pytest.fixture(scope="module")
def rs_inputs():
    """The M=32768, K=7168, N=7168 inputs in 16 K-shards; coarser shardings are
    concatenations of neighbours, identical to slicing the full matrices."""
    w = gi.RS_ALL[-1]
    return gi.gaussian_ar(w.M, w.N, [w.K // 16] * 16, seed=w.seed, device=device())


@pytest.mark.parametrize("w", gi.RS_ALL, ids=lambda w: w.name)
def test_rs_full_size(w, rs_inputs):
    p, ws = plan()
    dev = device()
    g = 16 // w.R
    X = [torch.cat(rs_inputs.X_r[i * g:(i + 1) * g], dim=1).contiguous() for i in range(w.R)]
    W = [torch.cat(rs_inputs.W_r[i * g:(i + 1) * g], dim=1).contiguous() for i in range(w.R)]
    rps = w.M // w.R
    Y_r = [torch.empty(rps, w.N, dtype=torch.bfloat16, device=dev) for _ in range(w.R)]
    B.gemm_rs(p, X, W, Y_r, ws)
    Y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    B.gemm_ar(p, X, W, Y, ws)
    B.gemm_shard_check_status(p, ws)
    # bit-identical to the matching AR rows
    assert torch.equal(torch.cat(Y_r).view(torch.int16), Y.view(torch.int16))
    X_h = [x.cpu() for x in X]
    W_h = [x.cpu() for x in W]
    ref = lambda r, c: oracle.ar_at(X_h, W_h, r, c)
    bounds = [s * rps for s in range(w.R)]
    check_rows(Y, sample_rows(w.M, bounds, n_random=6), ref, w.N, w.name)
    check_points(Y, w.M, w.N, ref, w.name, n=2000)
