"""GPU parity of the packed gather (gemm_shard_pack_gather): every output element
bit-identical to the CPU oracle on the same seeded states, rows past rows_out
and guard rows untouched, inputs unchanged, NULL states allowed for shards with
no kept row, and the full Kimi-K3-like size (8 shards x 4096 rows, the hidden
state and three auxiliary states of 7168 columns, 5 padding rows dropped)."""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import Guarded, bits_of, device, plan, shards_to

pytestmark = pytest.mark.gpu

# (M_r, T, H, rows_out): ragged and empty shards, truncation inside and at the
# end of a shard, one to sixteen states, state rows of 16 B .. 32 KB (one or two
# bulk-copy pieces), more pieces than CTAs and fewer.
SHAPES = [
    ([1], 1, 8, 1),
    ([3, 0, 5, 2], 2, 8, 10),
    ([3, 0, 5, 2], 2, 8, 6),
    ([0, 0, 7], 4, 24, 7),
    ([100, 37, 128], 3, 136, 250),
    ([50, 60], 2, 16384, 110),
    ([50, 60], 3, 12288, 57),
    ([10, 10, 10], 16, 64, 25),
    ([513, 300], 4, 7168, 800),
]


def run_pack(S_dev, rows_out, T, H, p=None):
    p, ws = p or plan()
    P = Guarded(rows_out, T * H)
    B.gemm_shard_pack_gather(p, S_dev, rows_out, P.out, ws)
    B.gemm_shard_check_status(p, ws)
    return P


@pytest.mark.parametrize("M_r,T,H,rows_out", SHAPES)
def test_pack_gather_matches_oracle_bitwise(M_r, T, H, rows_out):
    S = gi.gaussian_states(M_r, T, H, seed=sum(M_r) + T)
    dev = device()
    S_dev = [shards_to(dev, states)[0] for states in S]
    P = run_pack(S_dev, rows_out, T, H)
    ref = oracle.pack_gather(S, rows_out)
    assert np.array_equal(bits_of(P.out), ref)
    assert P.guards_intact()
    # inputs are read, never written
    for states, states_dev in zip(S, S_dev):
        for a, b in zip(states, states_dev):
            assert np.array_equal(bits_of(a), bits_of(b))


def test_pack_gather_split_views_are_the_gathered_states():
    M_r, T, H, rows_out = [64, 64, 64], 3, 264, 190
    S = gi.gaussian_states(M_r, T, H, seed=3, device=device())
    P = run_pack(S, rows_out, T, H)
    for t in range(T):
        view = P.out[:, t * H:(t + 1) * H]
        gathered = torch.cat([S[r][t] for r in range(len(M_r))])[:rows_out]
        assert torch.equal(view.view(torch.int16), gathered.view(torch.int16))


def test_pack_gather_skips_shards_past_rows_out():
    """Through the C ABI: a shard whose rows all lie at or past rows_out is not
    read (its state pointers are NULL here), and an empty shard is skipped."""
    import ctypes
    dev = device()
    p, ws = plan()
    S = gi.gaussian_states([20, 0, 20, 20], 2, 16, seed=4, device=dev)
    ptrs = [S[0][0].data_ptr(), S[0][1].data_ptr(), 0, 0,
            S[2][0].data_ptr(), S[2][1].data_ptr(), 0, 0]
    P = Guarded(33, 32)
    lib = B.load_library()
    wsp, wsn = B._ws(ws)
    st = lib.gemm_shard_pack_gather(
        p.handle, 4, (ctypes.c_int64 * 4)(20, 0, 20, 20), 2, 16,
        ctypes.cast((ctypes.c_void_p * 8)(*ptrs), ctypes.POINTER(ctypes.c_void_p)), 33,
        ctypes.c_void_p(P.out.data_ptr()), wsp, wsn, B._stream(None))
    assert st == B.GSR_OK, B.gsr_last_error_string()
    B.gemm_shard_check_status(p, ws)
    ref = oracle.pack_gather([[x.cpu() for x in st_] for st_ in S[:3]], 33)
    assert np.array_equal(bits_of(P.out), ref)
    assert P.guards_intact()


def test_pack_gather_repeat_and_prepared_calls_agree():
    p, ws = plan()
    M_r, T, H, rows_out = [300, 5, 700], 4, 520, 1000
    S = gi.gaussian_states(M_r, T, H, seed=5, device=device())
    P1 = torch.empty(rows_out, T * H, dtype=torch.bfloat16, device=device())
    P2 = torch.empty_like(P1)
    B.gemm_shard_pack_gather(p, S, rows_out, P1, ws)
    call = B.prepare_pack_gather(p, S, rows_out, P2, ws)
    call()
    call()
    B.gemm_shard_check_status(p, ws)
    assert torch.equal(P1.view(torch.int16), P2.view(torch.int16))


def test_pack_gather_full_size():
    w = gi.PACK_SP
    dev = device()
    S = gi.gaussian_states([w.M_r] * w.R, w.T, w.H, seed=w.seed, device=dev)
    P = run_pack(S, w.rows_out, w.T, w.H)
    ref = oracle.pack_gather([[x.cpu() for x in st] for st in S], w.rows_out)
    assert np.array_equal(bits_of(P.out), ref)
    assert P.guards_intact()


def test_packed_states_feed_the_ag_projection():
    """The packed gather feeding AG: the gathered rows P (rows_out x T*H: each
    rank's hidden and auxiliary states side by side, the ranks stacked) are the
    activation of a projection over the concatenated states, W: N x T*H (the
    fused input of an EAGLE-style drafter's first layer). AG reads P in place,
    either as one shard or as the ranks' row ranges of P (contiguous sub-buffers,
    no copy); both match the oracle's AG over the oracle's pack within the
    test tolerance."""
    from gpu_util import assert_close, to_f64
    M_r, T, H, rows_out, N = [96, 64, 130], 3, 256, 285, 264
    S = gi.gaussian_states(M_r, T, H, seed=11)
    dev = device()
    S_dev = [shards_to(dev, states)[0] for states in S]
    P = run_pack(S_dev, rows_out, T, H).out
    W = (torch.randn(N, T * H, generator=torch.Generator().manual_seed(12)) / (T * H) ** 0.5
         ).to(torch.bfloat16)
    ref = oracle.ag([oracle.pack_gather(S, rows_out)], gi.bf16_bits(W))
    p, ws = plan()
    W_dev = W.to(dev)
    Y1 = Guarded(rows_out, N)
    B.gemm_ag(p, [P], W_dev, Y1.out, ws)
    # the ranks' kept rows as separate shards pointing into P
    bounds = np.minimum(np.cumsum([0] + M_r), rows_out)
    views = [P[a:b] for a, b in zip(bounds[:-1], bounds[1:])]
    Y2 = Guarded(rows_out, N)
    B.gemm_ag(p, views, W_dev, Y2.out, ws)
    B.gemm_shard_check_status(p, ws)
    assert_close(to_f64(Y1.out), ref, "pack -> AG (one shard)")
    assert Y1.guards_intact() and Y2.guards_intact()
    assert_close(to_f64(Y2.out), ref, "pack -> AG (rank row ranges)")
