"""CUDA graph capture of the library's calls. A call's launches are recorded in
a stream capture like any kernel's: its tensor maps and kernel parameters are
built on the host when the call is made (so the graph holds that call's
pointers and shapes), the split-K arrival counters reset themselves inside
the kernel, and no call synchronises or allocates. A replay must therefore give
the bits of an eager call on the buffers' current values, replay after replay.
Decode-size calls are launch-bound (a few microseconds of kernel after several
of host work), which is what a graph of many calls removes."""
import pytest
import torch

from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import bits_of, device, plan, shards_to

pytestmark = pytest.mark.gpu

REPLAYS = 3


def capture(call):
    """Warm the call up on a side stream, then record it into a graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    return g


def refill(dst, src):
    for d, s in zip(dst, src):
        d.copy_(s)


# (M, N, K_r): the small-M kernel (one and a hundred rows, ragged tiles), and
# the main kernel with a split last wave (its pieces meet through the
# workspace counters, which must be back at zero for the next replay).
AR_CASES = [(1, 1024, [256] * 4), (100, 1000, [448, 64]), (1000, 1024, [256] * 4)]


@pytest.mark.parametrize("M,N,K_r", AR_CASES, ids=lambda v: str(v).replace(" ", ""))
def test_ar_graph_replays_match_eager_calls(M, N, K_r):
    p, ws = plan()
    dev = device()
    first = gi.gaussian_ar(M, N, K_r, seed=21)
    (X_r, _), (W_r, _) = shards_to(dev, first.X_r), shards_to(dev, first.W_r)
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    g = capture(B.prepare_ar(p, X_r, W_r, Y, ws))
    Y_eager = torch.empty_like(Y)
    for step in range(REPLAYS):
        # New values in the captured buffers, then an eager call and a replay.
        nxt = gi.gaussian_ar(M, N, K_r, seed=22 + step)
        refill(X_r + W_r, nxt.X_r + nxt.W_r)
        B.gemm_ar(p, X_r, W_r, Y_eager, ws)
        Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        B.gemm_shard_check_status(p, ws)
        assert (bits_of(Y) == bits_of(Y_eager)).all(), f"replay {step}"


def test_rs_graph_replays_match_eager_calls():
    M, N, K_r = 1000, 1024, [256] * 4
    p, ws = plan()
    dev = device()
    R = len(K_r)
    rps = -(-M // R)
    first = gi.gaussian_ar(M, N, K_r, seed=31)
    (X_r, _), (W_r, _) = shards_to(dev, first.X_r), shards_to(dev, first.W_r)
    Y_r = [torch.empty(rps, N, dtype=torch.bfloat16, device=dev) for _ in range(R)]
    g = capture(B.prepare_rs(p, X_r, W_r, Y_r, ws, M=M))
    Y_eager = [torch.empty_like(y) for y in Y_r]
    for step in range(REPLAYS):
        nxt = gi.gaussian_ar(M, N, K_r, seed=32 + step)
        refill(X_r + W_r, nxt.X_r + nxt.W_r)
        B.gemm_rs(p, X_r, W_r, Y_eager, ws, M=M)
        for y in Y_r:
            y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        B.gemm_shard_check_status(p, ws)
        for s in range(R):
            assert (bits_of(Y_r[s]) == bits_of(Y_eager[s])).all(), f"replay {step}, shard {s}"


@pytest.mark.parametrize("M_r,N", [([256] * 8, 3648), ([384, 0, 200, 512], 1000)],
                         ids=["mla_m2048", "ragged"])
def test_ag_graph_replays_match_eager_calls(M_r, N):
    K = 1024
    p, ws = plan()
    dev = device()
    first = gi.gaussian_ag(M_r, N, K, seed=41)
    A_r, _ = shards_to(dev, first.A_r)
    W = first.W.to(dev)
    Y = torch.empty(sum(M_r), N, dtype=torch.bfloat16, device=dev)
    g = capture(B.prepare_ag(p, A_r, W, Y, ws))
    Y_eager = torch.empty_like(Y)
    for step in range(REPLAYS):
        nxt = gi.gaussian_ag(M_r, N, K, seed=42 + step)
        refill(A_r + [W], nxt.A_r + [nxt.W])
        B.gemm_ag(p, A_r, W, Y_eager, ws)
        Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        B.gemm_shard_check_status(p, ws)
        assert (bits_of(Y) == bits_of(Y_eager)).all(), f"replay {step}"


def test_graph_of_many_decode_calls():
    """Sixteen decode-size AR calls (two alternating output buffers) in one
    graph: each output equals its eager call's."""
    M, N, K_r = 8, 2048, [512] * 4
    p, ws = plan()
    dev = device()
    first = gi.gaussian_ar(M, N, K_r, seed=51)
    (X_r, _), (W_r, _) = shards_to(dev, first.X_r), shards_to(dev, first.W_r)
    Ys = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    calls = [B.prepare_ar(p, X_r, W_r, Ys[i % 2], ws) for i in range(16)]

    def all_calls():
        for c in calls:
            c()

    g = capture(all_calls)
    nxt = gi.gaussian_ar(M, N, K_r, seed=52)
    refill(X_r + W_r, nxt.X_r + nxt.W_r)
    Y_eager = torch.empty_like(Ys[0])
    B.gemm_ar(p, X_r, W_r, Y_eager, ws)
    for y in Ys:
        y.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    B.gemm_shard_check_status(p, ws)
    for y in Ys:
        assert (bits_of(y) == bits_of(Y_eager)).all()
