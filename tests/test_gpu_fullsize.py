"""GPU parity at the full workload sizes: EVERY element of every benchmarked
output is compared with the fp64 oracle, in the launch configuration the
benchmark times (same plan maxima, heuristic configuration).

The workloads are the pages' projections: AG KDA-like (N=6288) and MLA-like
(N=3648) with R=8 shards of 256..4096 rows and K=7168 (AG-GEMM page,
microbenchmark tables); AR o_proj-like (R=8 K-shards of 896, N=7168, M in
{1, 16, 64, 128, 129, 1000, 4096, 32768}); RS with R in {2, 4, 8, 16} at M=32768 (the
GEMM-RS/AR page, test `_reference`: rank s keeps rows [s*M/R, (s+1)*M/R) of
the all-reduced product).

Inputs are seeded on the device (torch's CUDA generator, the same recipe as the
CPU one) and their bits copied to the host for the oracle, which computes the
reference in row blocks from the same separate shard arrays the GPU reads.

RS shares its seed, and so its full X and W, with AR o_proj M=32768 (checked
here bit for bit). One oracle run therefore serves all five: each RS output is
first checked to equal, bit for bit, the AR output at its own R (the pages'
RS and AR take the same sums), and every one of those AR outputs is then
compared element by element with the oracle.

Each comparison's max abs error, max relative error and count over the bound
are printed in the run's terminal summary."""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import ParityStats, device, plan

pytestmark = pytest.mark.gpu

# Rows per oracle call: about 2e11 multiply-adds at N = K = 7168, a few
# seconds on the host cores; the fp64 block stays near 100 MB.
ORACLE_ROWS = 2048


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 patterns exactly (they are the upper halves of binary32s)."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def check_ar_rows(stats_list, Y_bits_list, X_h, W_h, M):
    """Compare each output (bf16 bits, M x N) with the oracle, block by block."""
    for m0 in range(0, M, ORACLE_ROWS):
        m1 = min(M, m0 + ORACLE_ROWS)
        ref = oracle.ar([x[m0:m1] for x in X_h], W_h)
        for st, yb in zip(stats_list, Y_bits_list):
            st.add(bf16_bits_to_f64(yb[m0:m1]), ref)


@pytest.mark.parametrize("w", gi.AG_KDA + gi.AG_MLA, ids=lambda w: w.name)
def test_ag_full_size_every_element(w):
    p, ws = plan()
    dev = device()
    inp = gi.make_inputs(w, device=dev)
    Y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    B.gemm_ag(p, inp.A_r, inp.W, Y, ws)
    B.gemm_shard_check_status(p, ws)
    y_bits = host_bits(Y)
    A_h = [host_bits(a) for a in inp.A_r]
    W_h = host_bits(inp.W)
    del inp, Y
    st = ParityStats(w.name)
    row0 = 0
    for a in A_h:                          # shard by shard, in row blocks
        for m0 in range(0, a.shape[0], ORACLE_ROWS):
            m1 = min(a.shape[0], m0 + ORACLE_ROWS)
            ref = oracle.ag([a[m0:m1]], W_h)
            st.add(bf16_bits_to_f64(y_bits[row0 + m0:row0 + m1]), ref)
        row0 += a.shape[0]
    assert row0 == w.M
    st.finish(expect_elements=w.M * w.N)


@pytest.mark.parametrize("w", [x for x in gi.AR_DECODE + gi.AR_SMALL_TOP + gi.AR_OPROJ if x.M != 32768],
                         ids=lambda w: w.name)
def test_ar_full_size_every_element(w):
    p, ws = plan()
    dev = device()
    inp = gi.make_inputs(w, device=dev)
    Y = torch.empty(w.M, w.N, dtype=torch.bfloat16, device=dev)
    B.gemm_ar(p, inp.X_r, inp.W_r, Y, ws)
    B.gemm_shard_check_status(p, ws)
    y_bits = host_bits(Y)
    X_h = [host_bits(x) for x in inp.X_r]
    W_h = [host_bits(x) for x in inp.W_r]
    del inp, Y
    st = ParityStats(w.name)
    check_ar_rows([st], [y_bits], X_h, W_h, w.M)
    st.finish(expect_elements=w.M * w.N)


def test_ar_m32768_and_rs_every_element():
    """ar_oproj_m32768 and rs_r2/4/8/16 on one set of inputs and one oracle run."""
    ar_w = next(x for x in gi.AR_OPROJ if x.M == 32768)
    p, ws = plan()
    dev = device()
    M, N = ar_w.M, ar_w.N
    # the finest sharding; coarser ones are concatenations of neighbours
    fine = gi.gaussian_ar(M, N, [ar_w.K // 16] * 16, seed=gi.RS_ALL[0].seed, device=dev)
    ref_inp = gi.make_inputs(ar_w, device=dev)
    assert torch.equal(torch.cat(fine.X_r, 1).view(torch.int16),
                       torch.cat(ref_inp.X_r, 1).view(torch.int16))
    assert torch.equal(torch.cat(fine.W_r, 1).view(torch.int16),
                       torch.cat(ref_inp.W_r, 1).view(torch.int16))

    names, outs = [], []
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    B.gemm_ar(p, ref_inp.X_r, ref_inp.W_r, Y, ws)
    B.gemm_shard_check_status(p, ws)
    names.append(ar_w.name)
    outs.append(host_bits(Y))
    for w in gi.RS_ALL:
        g = 16 // w.R
        X = [torch.cat(fine.X_r[i * g:(i + 1) * g], dim=1).contiguous() for i in range(w.R)]
        W = [torch.cat(fine.W_r[i * g:(i + 1) * g], dim=1).contiguous() for i in range(w.R)]
        rps = M // w.R
        Y_r = [torch.empty(rps, N, dtype=torch.bfloat16, device=dev) for _ in range(w.R)]
        B.gemm_rs(p, X, W, Y_r, ws)
        B.gemm_ar(p, X, W, Y, ws)
        B.gemm_shard_check_status(p, ws)
        assert torch.equal(torch.cat(Y_r).view(torch.int16), Y.view(torch.int16)), \
            f"{w.name}: RS rows differ from the AR rows at R={w.R}"
        names.append(w.name)
        outs.append(host_bits(torch.cat(Y_r)))
        del X, W, Y_r
    X_h = [host_bits(x) for x in ref_inp.X_r]
    W_h = [host_bits(x) for x in ref_inp.W_r]
    del fine, ref_inp, Y
    torch.cuda.empty_cache()
    stats = [ParityStats(n) for n in names]
    check_ar_rows(stats, outs, X_h, W_h, M)
    for st in stats:
        st.finish(expect_elements=M * N)
