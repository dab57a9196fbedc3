"""GPU tests of the AG-GEMM with in-kernel waiting (gemm_ag_flagged): the kernel
waits, bounded, for each shard's arrival flag before reading it, so the copies
that bring the shards in overlap the GEMM. The single kernel with in-kernel
waiting is the future work the AG-GEMM page names ("[Kimi-K3] AG-GEMM for
Sequence Parallelism", Component breakdown, closing remark).

The timeout test makes a wait run out the way the environment asks for: a flag
that nothing sets, a short limit, and a status word the host reads afterwards;
the same context then runs a normal call."""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import assert_close, bits_of, device, plan, to_f64

pytestmark = pytest.mark.gpu

CONFIGS = {
    "auto": {},
    "cta1": dict(cta_group=1),
    "pairs": dict(cta_group=2, schedule=1),
    "sk8": dict(schedule=2, max_ctas=8),
}


def _ready(R, value=0):
    return torch.full((R,), value, dtype=torch.int32, device=device())


@pytest.mark.parametrize("cfg", list(CONFIGS))
def test_flags_already_set_match_plain_ag(cfg):
    p, ws = plan(**CONFIGS[cfg])
    inp = gi.gaussian_ag([300, 5, 700, 128], 520, 256, seed=21)
    dev = device()
    A = [a.to(dev) for a in inp.A_r]
    W = inp.W.to(dev)
    Y0 = torch.empty(inp.M, inp.N, dtype=torch.bfloat16, device=dev)
    Y1 = torch.empty_like(Y0)
    B.gemm_ag(p, A, W, Y0, ws)
    B.gemm_ag_flagged(p, A, W, Y1, _ready(4, 3), 3, ws)
    B.gemm_shard_check_status(p, ws)
    assert np.array_equal(bits_of(Y1), bits_of(Y0))


@pytest.mark.parametrize("M_r", [[2048, 2048, 1024, 2048], [448, 448, 1088, 448]],
                         ids=["128-row granules", "64-row granules"])
@pytest.mark.parametrize("cfg", ["auto", "cta1"])
def test_kernel_waits_for_shards_copied_while_it_runs(cfg, M_r):
    """The GEMM is launched before its shards exist on the device; a second
    stream copies them in from pinned host memory, one shard at a time, and
    signals each one. The result must equal the plain AG on resident shards.
    With 64-row granules a CTA's rows may come from two shards, and it waits
    for both."""
    p, ws = plan(**CONFIGS[cfg])
    inp = gi.gaussian_ag(M_r, 3648, 2048, seed=22)
    dev = device()
    host = [a.pin_memory() for a in inp.A_r]
    A = [torch.empty_like(a, device=dev) for a in inp.A_r]
    W = inp.W.to(dev)
    ready = _ready(4, 0)
    Y = torch.empty(inp.M, inp.N, dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    gemm_stream = torch.cuda.Stream()     # torch's pool streams do not block on each other
    copy_stream = torch.cuda.Stream()
    epoch = 5
    with torch.cuda.stream(gemm_stream):
        B.gemm_ag_flagged(p, A, W, Y, ready, epoch, ws)       # waits in the kernel
    with torch.cuda.stream(copy_stream):
        for r in range(4):
            A[r].copy_(host[r], non_blocking=True)
            B.gemm_shard_signal(p, ready.data_ptr() + 4 * r, epoch, stream=copy_stream)
    torch.cuda.synchronize()
    B.gemm_shard_check_status(p, ws)
    Y_ref = torch.empty_like(Y)
    B.gemm_ag(p, A, W, Y_ref, ws)
    B.gemm_shard_check_status(p, ws)
    assert np.array_equal(bits_of(Y), bits_of(Y_ref))
    bounds = np.cumsum(M_r)[:-1]
    rows = np.unique(np.concatenate([[0, 1, inp.M - 1], bounds - 1, bounds]))
    r = np.repeat(rows, inp.N)
    c = np.tile(np.arange(inp.N), len(rows))
    ref = oracle.ag_at(inp.A_r, inp.W, r, c).reshape(len(rows), inp.N)
    assert_close(to_f64(Y[torch.as_tensor(rows, device=dev)]), ref, "flagged ag rows")


@pytest.mark.parametrize("cfg", list(CONFIGS))
def test_missing_flag_times_out_and_context_stays_usable(cfg):
    opts = dict(CONFIGS[cfg], timeout_ns=50_000_000)          # 50 ms
    p, ws = plan(max_M=8192, max_N=4096, max_K=4096, max_R=4, **opts)
    inp = gi.gaussian_ag([300, 200], 520, 256, seed=23)
    dev = device()
    A = [a.to(dev) for a in inp.A_r]
    W = inp.W.to(dev)
    ready = _ready(2, 0)
    ready[0] = 9                                               # shard 1 never arrives
    Y = torch.zeros(inp.M, inp.N, dtype=torch.bfloat16, device=dev)
    B.gemm_ag_flagged(p, A, W, Y, ready, 9, ws)
    with pytest.raises(B.GsrError) as e:
        B.gemm_shard_check_status(p, ws)
    assert e.value.status == B.GSR_ERR_TIMEOUT
    assert "role 1, site 3" in str(e.value)                   # the producer's flag wait
    # the context and the library still work after a workspace re-init
    B.gemm_shard_workspace_init(p, ws)
    Y2 = torch.empty_like(Y)
    B.gemm_ag(p, A, W, Y2, ws)
    B.gemm_shard_check_status(p, ws)
    assert_close(to_f64(Y2), oracle.ag(inp.A_r, inp.W), "after timeout")
