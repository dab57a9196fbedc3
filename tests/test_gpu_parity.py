"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle, element
by element on the same seeded inputs, at sizes the oracle finishes in seconds
that still span several tiles and ragged tails. Bound per element:
|y - ref| <= 1e-2 |ref| + 1e-2 (fp32 accumulation, one bf16 rounding)."""
import numpy as np
import pytest
import torch

import oracle
from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import inputs as gi

from gpu_util import (Guarded, assert_close, bits_of, device, plan, shards_to, to_f64,
                      SENTINEL)

pytestmark = pytest.mark.gpu

# Kernel configurations every ragged shape runs under (they must all agree with
# the oracle): the heuristic; the uniform schedule; stream-K on only 8 CTAs (so
# that even small shapes cut tiles into several pieces); CTA pairs with 128-
# and 256-column whole tiles; CTA pairs with stream-K; CTA pairs with a
# uniform 3-way split; CTA pairs with 192-column tiles; clusters of two CTA
# pairs that share each copy of B.
VARIANTS = {
    "auto": {},
    "uniform": dict(schedule=1),
    "sk8": dict(schedule=2, max_ctas=8),
    "pair128": dict(cta_group=2, block_n=128, schedule=1),
    "pair256": dict(cta_group=2, block_n=256, schedule=1),
    "pair192": dict(cta_group=2, block_n=192),
    "pairsk8": dict(cta_group=2, schedule=2, max_ctas=8),
    "pairsk8last": dict(cta_group=2, schedule=4, max_ctas=8),
    "pairsplit": dict(max_M=4096, max_N=8192, max_K=8192, max_R=16, cta_group=2, split_k=3),
    "rastern": dict(raster_n=3),
    "splittail": dict(cta_group=2, schedule=5, max_ctas=16),
    # two CTA pairs per cluster sharing each copy of B (whole tiles, stream-K
    # on four clusters, 192-column tiles)
    "quad": dict(cta_group=4),
    "quadsk": dict(cta_group=4, schedule=2, max_ctas=16),
    "quad192": dict(cta_group=4, block_n=192),
}


def vplan(variant):
    return plan(**VARIANTS[variant])


def run_ar(inp, p=None, reverse=False):
    p, ws = p or plan()
    dev = device()
    X, s1 = shards_to(dev, inp.X_r, reverse)
    W, s2 = shards_to(dev, inp.W_r, reverse)
    Y = Guarded(inp.M, inp.N)
    B.gemm_ar(p, X, W, Y.out, ws)
    B.gemm_shard_check_status(p, ws)
    return Y, X, W


def run_rs(inp, p=None):
    p, ws = p or plan()
    dev = device()
    X, _ = shards_to(dev, inp.X_r)
    W, _ = shards_to(dev, inp.W_r)
    R = inp.R
    rps = -(-inp.M // R)
    Ys = [Guarded(rps, inp.N) for _ in range(R)]
    B.gemm_rs(p, X, W, [y.out for y in Ys], ws, M=inp.M)
    B.gemm_shard_check_status(p, ws)
    return Ys


def run_ag(inp, p=None, reverse=False):
    p, ws = p or plan()
    dev = device()
    A, s1 = shards_to(dev, inp.A_r, reverse)
    W = inp.W.to(dev)
    Y = Guarded(inp.M, inp.N)
    B.gemm_ag(p, A, W, Y.out, ws)
    B.gemm_shard_check_status(p, ws)
    return Y


# ------------------------------------------------------------------ AR

def test_ar_tiny_config():
    """AR, R=2 shards of K=128, M=128, N=256, seed 0."""
    w = gi.AR_TINY
    inp = gi.make_inputs(w)
    Y, _, _ = run_ar(inp)
    assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), "ar tiny")
    assert Y.guards_intact()


AR_SHAPES = [
    (1, 8, [8]),
    (7, 136, [72, 8]),
    (127, 264, [136]),
    (128, 256, [64, 64]),
    (129, 520, [64, 200, 72]),
    (257, 1032, [128, 128, 128]),
    (300, 256, [8] * 16),
    (513, 640, [520]),
    (200, 7168, [896, 896]),
    (131, 520, [128, 256]),
]


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("M,N,K_r", AR_SHAPES)
def test_ar_ragged(M, N, K_r, variant):
    inp = gi.gaussian_ar(M, N, K_r)
    Y, _, _ = run_ar(inp, p=vplan(variant))
    assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), f"ar {M}x{N} K_r={K_r}")
    assert Y.guards_intact()


def test_ar_shards_in_reverse_allocation_order():
    inp = gi.gaussian_ar(190, 392, [40, 96, 16, 64])
    Y, _, _ = run_ar(inp, reverse=True)
    assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), "ar reversed allocations")


def test_ar_integer_inputs_exact():
    """Values in {-1,0,1}, K=256: every partial and the result are exact in fp32
    and bf16, so the GPU must equal the exact oracle bit for bit."""
    inp = gi.integer_ar(128, 256, [128, 128], amp=1, seed=3)
    Y, _, _ = run_ar(inp)
    ref = oracle.ar(inp.X_r, inp.W_r)
    assert np.array_equal(to_f64(Y.out), ref)


def test_ar_identity_weight_returns_x_bitwise():
    K_r = [64, 128, 64]
    K = sum(K_r)
    inp = gi.gaussian_ar(200, K, K_r, seed=12)
    eye = torch.eye(K, dtype=torch.bfloat16)
    W_r, c = [], 0
    for k in K_r:
        W_r.append(eye[:, c:c + k].contiguous())
        c += k
    inp.W_r = W_r
    Y, _, _ = run_ar(inp)
    assert np.array_equal(bits_of(Y.out), bits_of(torch.cat(inp.X_r, dim=1)))


def _one_hot(M: int, K: int, seed: int):
    g = torch.Generator().manual_seed(seed)
    cols = torch.randint(0, K, (M,), generator=g)
    X = torch.zeros(M, K, dtype=torch.bfloat16)
    X[torch.arange(M), cols] = 1.0
    return X, cols


@pytest.mark.parametrize("variant", ["auto", "sk8", "pairsk8", "splittail", "pairsplit"])
@pytest.mark.parametrize("M", [100, 300])
def test_ar_one_hot_rows_select_weight_columns_bitwise(M, variant):
    """Row m of X is one-hot at column k_m (anywhere in any shard): every
    product but one is zero, so Y[m, n] = W[n, k_m] exactly, whatever the
    split, the schedule or the kernel (M = 100 runs the small-M kernel)."""
    K_r = [128, 64, 192]
    inp = gi.gaussian_ar(M, 264, K_r, seed=21)
    X, cols = _one_hot(M, sum(K_r), seed=M)
    inp.X_r = [X[:, a:a + k].contiguous() for a, k in zip((0, 128, 192), K_r)]
    Y, _, _ = run_ar(inp, p=vplan(variant))
    W = torch.cat(inp.W_r, dim=1)
    assert np.array_equal(bits_of(Y.out), bits_of(W[:, cols].t().contiguous()))


@pytest.mark.parametrize("variant", ["auto", "sk8", "pairsk8"])
def test_ag_one_hot_rows_select_weight_columns_bitwise(variant):
    M_r = [100, 0, 257, 64]
    inp = gi.gaussian_ag(M_r, 200, 320, seed=22)
    X, cols = _one_hot(sum(M_r), 320, seed=5)
    inp.A_r, r0 = [], 0
    for m in M_r:
        inp.A_r.append(X[r0:r0 + m].contiguous())
        r0 += m
    Y = run_ag(inp, p=vplan(variant))
    assert np.array_equal(bits_of(Y.out), bits_of(inp.W[:, cols].t().contiguous()))
    assert Y.guards_intact()


@pytest.mark.parametrize("M", [64, 1000])
def test_zero_activations_give_zero_output(M):
    inp = gi.gaussian_ar(M, 520, [256, 256], seed=23)
    inp.X_r = [torch.zeros_like(x) for x in inp.X_r]
    Y, _, _ = run_ar(inp)
    assert not to_f64(Y.out).any()
    assert Y.guards_intact()


def test_ar_negated_input_negates_output_and_keeps_first_result():
    """After the page's lifetime test (M=257, K=768, seed 2500): a second call with
    -X gives exactly -Y, and the first result, in its own buffer, is untouched."""
    inp = gi.gaussian_ar(257, 512, [256, 512], seed=2500)
    p, ws = plan()
    dev = device()
    X = [x.to(dev) for x in inp.X_r]
    W = [w.to(dev) for w in inp.W_r]
    Y1 = torch.empty(257, 512, dtype=torch.bfloat16, device=dev)
    Y2 = torch.empty_like(Y1)
    B.gemm_ar(p, X, W, Y1, ws)
    snap = Y1.clone()
    B.gemm_ar(p, [-x for x in X], W, Y2, ws)
    B.gemm_shard_check_status(p, ws)
    assert torch.equal(Y1.view(torch.int16), snap.view(torch.int16))
    assert torch.equal(Y2.view(torch.int16), (-Y1).view(torch.int16))
    assert_close(to_f64(Y1), oracle.ar(inp.X_r, inp.W_r), "first call")


def test_inputs_unchanged():
    inp = gi.gaussian_ar(150, 264, [64, 72])
    before = [bits_of(t) for t in inp.X_r + inp.W_r]
    _, X, W = run_ar(inp)
    after = [bits_of(t) for t in X + W]
    assert all(np.array_equal(a, b) for a, b in zip(before, after))


def test_m_zero_writes_nothing():
    p, ws = plan()
    dev = device()
    X = [torch.empty(0, 64, dtype=torch.bfloat16, device=dev)]
    W = [torch.randn(64, 64, device=dev).to(torch.bfloat16)]
    Y = torch.empty(0, 64, dtype=torch.bfloat16, device=dev)
    B.gemm_ar(p, X, W, Y, ws)
    B.gemm_shard_check_status(p, ws)


# ------------------------------------------------------------------ RS

RS_SHAPES = [
    (129, 520, [64, 64]),          # M % R != 0: shard 1 has one unwritten row
    (257, 264, [72, 8, 136]),
    (5, 256, [64, 64, 64]),
    (64, 136, [8] * 16),           # 16 shards of 4 rows
    (300, 7168, [448] * 16),
    (257, 264, [128, 256, 128]),   # M % R != 0
]


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("M,N,K_r", RS_SHAPES)
def test_rs_matches_oracle_and_ar_bitwise(M, N, K_r, variant):
    inp = gi.gaussian_ar(M, N, K_r)
    Ys = run_rs(inp, p=vplan(variant))
    Yar, _, _ = run_ar(inp, p=vplan(variant))
    ar_bits = bits_of(Yar.out)
    ref = oracle.rs(inp.X_r, inp.W_r)
    for s, y in enumerate(Ys):
        first, count = oracle.rs_rows(M, inp.R, s)
        assert y.guards_intact(valid_rows=count), f"shard {s}: row past its valid count written"
        if count == 0:
            continue
        assert_close(to_f64(y.out[:count]), ref[s][:count], f"rs shard {s}")
        assert np.array_equal(bits_of(y.out[:count]), ar_bits[first:first + count]), \
            f"shard {s} differs from AR rows bitwise"


# ------------------------------------------------------------------ AG

AG_SHAPES = [
    ([1], 8, 8),
    ([130, 1, 257], 520, 200),
    ([0, 64, 0, 128], 264, 128),
    ([256] * 8, 6288, 1024),
    ([448, 384], 3648, 512),
    ([300, 5, 700], 520, 256),
    ([384, 384, 384], 264, 128),        # pair tiles across shard boundaries
    ([384, 0, 200, 0], 520, 136),       # odd half-tile count, empty shards
    ([0, 0, 130], 136, 64),             # leading empty shards, idle last half
    # 64-row granules (shards multiples of 64 but not 128): a CTA's 128 rows
    # may come from two shards
    ([448] * 4, 520, 256),
    ([64, 448, 192, 0, 320], 264, 128),   # empty shard in between
    ([448, 448, 64], 3648, 256),          # odd granule count: last tile half empty
]


@pytest.mark.parametrize("variant", list(VARIANTS))
@pytest.mark.parametrize("M_r,N,K", AG_SHAPES)
def test_ag_ragged(M_r, N, K, variant):
    inp = gi.gaussian_ag(M_r, N, K)
    Y = run_ag(inp, p=vplan(variant))
    assert_close(to_f64(Y.out), oracle.ag(inp.A_r, inp.W), f"ag M_r={M_r} N={N} K={K}")
    assert Y.guards_intact()


def test_ag_reverse_allocation_order_and_integers_exact():
    inp = gi.integer_ag([100, 37, 128], 256, 256, amp=1, seed=4)
    Y = run_ag(inp, reverse=True)
    assert np.array_equal(to_f64(Y.out), oracle.ag(inp.A_r, inp.W))


# ------------------------------------------------------------------ split-K

@pytest.mark.parametrize("split", [2, 3, 7])
def test_forced_split_k(split):
    ps = plan(max_M=4096, max_N=2048, max_K=4096, max_R=16, split_k=split)
    inp = gi.gaussian_ar(129, 520, [256, 512, 64])
    Y, _, _ = run_ar(inp, p=ps)
    assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), f"split {split}")
    assert Y.guards_intact()
    # RS under the same split writes the same bits as AR
    Ys = run_rs(inp, p=ps)
    ar_bits = bits_of(Y.out)
    for s, y in enumerate(Ys):
        first, count = oracle.rs_rows(129, 3, s)
        assert np.array_equal(bits_of(y.out[:count]), ar_bits[first:first + count])
        assert y.guards_intact(valid_rows=count)
    # repeated calls reuse the self-resetting counters
    Y2, _, _ = run_ar(inp, p=ps)
    assert np.array_equal(bits_of(Y2.out), ar_bits)


def test_split_k_ag_and_block_n_128():
    ps = plan(max_M=4096, max_N=2048, max_K=4096, max_R=16, split_k=4, block_n=128)
    inp = gi.gaussian_ag([300, 5], 392, 1024)
    Y = run_ag(inp, p=ps)
    assert_close(to_f64(Y.out), oracle.ag(inp.A_r, inp.W), "ag split 4 bn 128")
    assert Y.guards_intact()


def test_heuristic_split_small_m_matches_oracle():
    """M=128, N=7168, 8 shards of 896 on the main kernel (the small-M kernel
    off): the plan cuts every tile's k range into pieces summed in k order."""
    p, ws = plan(small_m=1)
    d = B.gemm_shard_describe(p, B.MODE_AR, 128, 7168, 0, [896] * 8)
    assert d["split"] > 1 or d["sk_iters"] > 0
    inp = gi.gaussian_ar(128, 7168, [896] * 8, seed=99)
    Y, _, _ = run_ar(inp, (p, ws))
    assert_close(to_f64(Y.out), oracle.ar(inp.X_r, inp.W_r), "ar m128 split")


def test_prepared_calls_match_plain_calls():
    """prepare_ar/rs/ag validate and marshal once; each call gives the same bits."""
    p, ws = plan()
    dev = device()
    inp = gi.gaussian_ar(257, 520, [128, 72])
    X = [x.to(dev) for x in inp.X_r]
    W = [w.to(dev) for w in inp.W_r]
    Y0 = torch.empty(257, 520, dtype=torch.bfloat16, device=dev)
    Y1 = torch.empty_like(Y0)
    B.gemm_ar(p, X, W, Y0, ws)
    call = B.prepare_ar(p, X, W, Y1, ws)
    call()
    call()
    rps = 129
    R0 = [torch.empty(rps, 520, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    B.prepare_rs(p, X, W, R0, ws)()
    ag = gi.gaussian_ag([100, 200], 264, 128)
    A = [a.to(dev) for a in ag.A_r]
    Wa = ag.W.to(dev)
    Ya0 = torch.empty(300, 264, dtype=torch.bfloat16, device=dev)
    Ya1 = torch.empty_like(Ya0)
    B.gemm_ag(p, A, Wa, Ya0, ws)
    B.prepare_ag(p, A, Wa, Ya1, ws)()
    B.gemm_shard_check_status(p, ws)
    assert np.array_equal(bits_of(Y1), bits_of(Y0))
    assert np.array_equal(bits_of(torch.cat(R0)[:257]), bits_of(Y0))
    assert np.array_equal(bits_of(Ya1), bits_of(Ya0))


@pytest.mark.parametrize("variant", ["auto", "uniform", "sk8", "pair256", "pairsk8"])
@pytest.mark.parametrize("M,N,K_r", [(129, 520, [64, 200, 72]), (300, 7168, [448] * 4), (5, 136, [8, 8])])
def test_ar_replicated_outputs_equal_ar_bitwise(M, N, K_r, variant):
    """Every one of the R outputs holds the whole AR result, bit for bit."""
    p, ws = vplan(variant)
    inp = gi.gaussian_ar(M, N, K_r)
    dev = device()
    X = [x.to(dev) for x in inp.X_r]
    W = [w.to(dev) for w in inp.W_r]
    Y = Guarded(M, N)
    B.gemm_ar(p, X, W, Y.out, ws)
    reps = [Guarded(M, N) for _ in K_r]
    B.gemm_ar_replicated(p, X, W, [g.out for g in reps], ws)
    B.gemm_shard_check_status(p, ws)
    ref = bits_of(Y.out)
    for g in reps:
        assert np.array_equal(bits_of(g.out), ref)
        assert g.guards_intact()
    assert_close(to_f64(reps[-1].out), oracle.ar(inp.X_r, inp.W_r), "replicated")


@pytest.mark.parametrize("mode", ["ar", "ag"])
def test_l2_hints_change_no_bit(mode):
    """The TMA L2 eviction hints (none, A evict-last / B evict-first, the
    reverse) change only what the L2 keeps: the configuration and the
    summation order are the same, so the outputs are bit-identical. The shapes
    fit in L2, where the heuristic takes the hints."""
    if mode == "ar":
        inp = gi.gaussian_ar(700, 1032, [512, 384], seed=61)
        outs = [run_ar(inp, p=plan(l2_hints=h))[0] for h in (1, 2, 3)]
        ref = oracle.ar(inp.X_r, inp.W_r)
    else:
        inp = gi.gaussian_ag([300, 0, 448, 129], 1032, 512, seed=62)
        outs = [run_ag(inp, p=plan(l2_hints=h)) for h in (1, 2, 3)]
        ref = oracle.ag(inp.A_r, inp.W)
    assert B.gemm_shard_describe(plan()[0], B.MODE_AR if mode == "ar" else B.MODE_AG,
                                 700 if mode == "ar" else 0, 1032, 0 if mode == "ar" else 512,
                                 [512, 384] if mode == "ar" else [300, 0, 448, 129])["l2_hints"] == 2
    for y in outs:
        assert y.guards_intact()
        assert np.array_equal(bits_of(y.out), bits_of(outs[0].out))
    assert_close(to_f64(outs[0].out), ref, f"{mode} with L2 hints")
