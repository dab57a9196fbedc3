"""GPU parity of the small-M kernel (AR/RS with at most 256 activation rows):
operands swapped (128-row tiles of W against all M rows), each tile split over
K between the two CTAs of a cluster and summed in distributed shared memory.
Checked element by element against the fp64 oracle (|y - ref| <= 1e-2 |ref| +
1e-2), RS and replicated AR bit-identical to AR, guard rows untouched."""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import Guarded, assert_close, bits_of, device, plan, shards_to, to_f64

pytestmark = pytest.mark.gpu

# (M, N, K_r): M from 1 to 256 (m_pad 16 .. 256, every ring depth), N with a
# ragged last tile, shards with ragged last k-blocks, one to sixteen shards.
SHAPES = [
    (1, 8, [8, 8]),
    (16, 136, [64, 64]),
    (17, 264, [136]),
    (48, 1000, [72, 8, 200]),
    (100, 2056, [448] * 4),
    (128, 384, [128] * 3),
    (129, 520, [64, 200, 72]),
    (144, 264, [8] * 16),
    (200, 1032, [520]),
    (255, 520, [128, 256]),
    (256, 392, [64, 64, 64]),
]


def small_plan(**opts):
    return plan(small_m=2, **opts)


def run(inp, p, mode="ar"):
    p, ws = p
    dev = device()
    X, _ = shards_to(dev, inp.X_r)
    W, _ = shards_to(dev, inp.W_r)
    if mode == "ar":
        Y = Guarded(inp.M, inp.N)
        B.gemm_ar(p, X, W, Y.out, ws)
        out = Y
    elif mode == "rs":
        rps = -(-inp.M // inp.R)
        out = [Guarded(rps, inp.N) for _ in range(inp.R)]
        B.gemm_rs(p, X, W, [y.out for y in out], ws, M=inp.M)
    else:
        out = [Guarded(inp.M, inp.N) for _ in range(inp.R)]
        B.gemm_ar_replicated(p, X, W, [y.out for y in out], ws)
    B.gemm_shard_check_status(p, ws)
    return out


@pytest.mark.parametrize("M,N,K_r", SHAPES)
def test_small_ar_rs_replicated(M, N, K_r):
    p = small_plan()
    d = B.gemm_shard_describe(p[0], B.MODE_AR, M, N, 0, K_r)
    assert d["schedule"] == 3
    inp = gi.gaussian_ar(M, N, K_r)
    Y = run(inp, p)
    assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), f"small ar {M}x{N} K_r={K_r}")
    assert Y.guards_intact()
    ar_bits = bits_of(Y.out)
    Ys = run(inp, p, "rs")
    for s, y in enumerate(Ys):
        first, count = oracle.rs_rows(M, inp.R, s)
        assert y.guards_intact(valid_rows=count), f"shard {s}: row past its valid count written"
        assert np.array_equal(bits_of(y.out[:count]), ar_bits[first:first + count]), s
    for y in run(inp, p, "rep"):
        assert np.array_equal(bits_of(y.out), ar_bits)
        assert y.guards_intact()


@pytest.mark.parametrize("ctas", [2, 6])
def test_small_many_tiles_per_cluster(ctas):
    """One or three clusters walk 17 tiles each in turn: both TMEM accumulators
    and every phase of the staging handshake are reused."""
    p = small_plan(max_ctas=ctas)
    inp = gi.gaussian_ar(129, 2120, [200, 64, 256], seed=21)
    Y = run(inp, p)
    assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), f"small, {ctas} CTAs")
    assert Y.guards_intact()
    Ys = run(inp, p, "rs")
    ar_bits = bits_of(Y.out)
    for s, y in enumerate(Ys):
        first, count = oracle.rs_rows(129, 3, s)
        assert np.array_equal(bits_of(y.out[:count]), ar_bits[first:first + count])
    # the same bits as the full grid (the sums do not depend on the grid)
    Yf = run(inp, small_plan())
    assert np.array_equal(bits_of(Yf.out), ar_bits)


def test_small_integer_inputs_exact():
    """Values in {-1, 0, 1} with K = 320: both halves and their sum are exact,
    so the result equals the exact oracle bit for bit."""
    inp = gi.integer_ar(100, 264, [128, 64, 128], amp=1, seed=5)
    Y = run(inp, small_plan())
    assert np.array_equal(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r))


def test_small_repeat_calls_and_main_kernel_agree():
    inp = gi.gaussian_ar(77, 1000, [448, 448], seed=8)
    ref = oracle.ar(inp.X_r, inp.W_r)
    a = run(inp, small_plan())
    b = run(inp, small_plan())
    assert np.array_equal(bits_of(a.out), bits_of(b.out))
    main = run(inp, plan(small_m=1))
    assert B.gemm_shard_describe(plan(small_m=1)[0], B.MODE_AR, 77, 1000, 0, [448, 448])["schedule"] != 3
    assert_close(to_f64(a.out), ref, "small")
    assert_close(to_f64(main.out), ref, "main")


def test_small_full_o_proj_matches_oracle_every_element():
    """The o_proj-like shape (R = 8 K-shards of 896, N = 7168) at decode sizes
    M = 1, 16 and 64 and at M = 128 and 129: every element against the oracle."""
    for M in (1, 16, 64, 128, 129):
        inp = gi.gaussian_ar(M, 7168, [896] * 8, seed=2000 + M + 7168)
        Y = run(inp, plan())
        assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), f"o_proj m{M}")
        assert Y.guards_intact()


@pytest.mark.parametrize("rows", [8, 40, 96, 120])
def test_small_tile_rows_agree_bitwise(rows):
    """Every tile height sums each output in the same order (the two halves of
    K added once), so the outputs are bit-identical to 128-row tiles. The MMA
    is always 128 rows tall: with shorter tiles its rows past the tile read
    stale shared memory into TMEM lanes that must never be stored (guards,
    ragged last tile of N = 1000, several tiles per cluster at 8 rows)."""
    inp = gi.gaussian_ar(100, 1000, [448, 200, 72], seed=31)
    ref_bits = bits_of(run(inp, small_plan(small_tile_rows=128)).out)
    Y = run(inp, small_plan(small_tile_rows=rows))
    assert Y.guards_intact()
    assert np.array_equal(bits_of(Y.out), ref_bits)
    assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), f"small, {rows}-row tiles")
    for s, y in enumerate(run(inp, small_plan(small_tile_rows=rows), "rs")):
        first, count = oracle.rs_rows(100, 3, s)
        assert y.guards_intact(valid_rows=count)
        assert np.array_equal(bits_of(y.out[:count]), ref_bits[first:first + count])
