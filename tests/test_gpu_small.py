"""GPU parity of the small-M kernel (AR/RS with at most 256 activation rows):
one CTA pair per tile of W rows over the whole K range, the activation rows as
the pair MMA's M (128 up to 128 rows, else 256) and the tile's W rows as its N.
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

# (M, N, K_r): M from 1 to 256 (both MMA heights; up to 64 rows the second
# CTA of a pair loads no activations), N with a ragged last tile, shards with
# ragged last k-blocks, one to sixteen shards, a single k-block.
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
    (65, 72, [40]),
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
    """One or three pairs walk 9 or 3 tiles each in turn: both TMEM
    accumulators are reused, each handed back to the MMA issuer before the
    tile two further on."""
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
    """Values in {-1, 0, 1} with K = 320: every partial sum is exact, so the
    result equals the exact oracle bit for bit."""
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


@pytest.mark.parametrize("M,K_r", [(1, [512, 256, 1024]), (64, [896, 192]), (100, [512, 256, 1024]),
                                   (200, [896, 192, 64])])
def test_small_kblocks_per_copy_agree_bitwise(M, K_r):
    """Copies of 1 to 4 k-blocks (a 2-D box, or a 3-D box over a strided
    {64, rows, K_r / 64} view of each shard) feed the same MMAs in the same
    order, so the outputs are bit-identical. Shards of 14, 3 and 1 k-blocks
    end in a copy that runs past the shard: its zero-filled k-blocks add
    nothing."""
    inp = gi.gaussian_ar(M, 1000, K_r, seed=41)
    ref = oracle.ar(inp.X_r, inp.W_r)
    seen, bits = set(), None
    for kz in (1, 2, 3, 4):
        p = small_plan(small_kblocks=kz)
        seen.add(B.gemm_shard_describe(p[0], B.MODE_AR, M, 1000, 0, K_r)["kblocks"])
        Y = run(inp, p)
        assert Y.guards_intact()
        assert_close(to_f64(Y.out), ref, f"small m{M}, {kz} k-blocks per copy")
        if bits is None:
            bits = bits_of(Y.out)
        assert np.array_equal(bits_of(Y.out), bits), kz
        for s, y in enumerate(run(inp, p, "rs")):
            first, count = oracle.rs_rows(M, len(K_r), s)
            assert np.array_equal(bits_of(y.out[:count]), bits[first:first + count])
    assert 1 in seen and 2 in seen


def test_small_full_o_proj_matches_oracle_every_element():
    """The o_proj-like shape (R = 8 K-shards of 896, N = 7168) at decode sizes
    M = 1, 16 and 64 and at M = 128 and 129: every element against the oracle."""
    for M in (1, 16, 64, 128, 129):
        inp = gi.gaussian_ar(M, 7168, [896] * 8, seed=2000 + M + 7168)
        Y = run(inp, plan())
        assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), f"o_proj m{M}")
        assert Y.guards_intact()


@pytest.mark.parametrize("rows", [16, 48, 96, 112, 256])
def test_small_tile_rows_agree_bitwise(rows):
    """Every tile height sums each output in the same order (every k-block in
    turn, through an MMA of the same height), so the outputs are bit-identical
    to 128-row tiles (guards, ragged last tile of N = 1000; 16-row tiles put
    8 rows in each CTA's half, and a ragged 8-column last chunk in TMEM)."""
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
