"""Pins for the CPU oracle (no GPU).

The oracle is the fp64 statement of the shard-reduction GEMM; here it is checked
against things other than itself: values worked by hand from the pages'
definitions (tests/golden/), exact brute force in Python integers, the bf16
format and torch's own bf16 widening, invariants (sum of per-shard partials =
full-K product; AG over shards = GEMM on the concatenation), special cases
(R = 1 is a textbook GEMM, identity and one-hot weights, zero and negated
inputs), and mutants of the oracle source that each pin must catch. The packed
gather (a copy) is pinned by a hand-worked example, brute force in Python lists,
the page's split-back symmetry checked with numpy.concatenate, and its special
cases (T = 1 is a plain gather, R = 1 a plain concatenation).
"""
import json
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from tensor_gemm_reduction_gb300 import inputs as gi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(vals) -> torch.Tensor:
    t = torch.tensor(vals, dtype=torch.float64).to(torch.bfloat16)
    assert torch.equal(t.to(torch.float64), torch.tensor(vals, dtype=torch.float64)), \
        "golden input not exact in bf16"
    return t


def _ints(t: torch.Tensor):
    """Integer-valued bf16 tensor -> nested Python ints (no oracle code)."""
    f = t.to(torch.float64)
    assert torch.equal(f, torch.round(f))
    return [[int(v) for v in row] for row in f.tolist()]


def py_ar(X_r, W_r):
    """Exact brute force in Python integers: sum over shards of X_r . W_r^T."""
    Xs, Ws = [_ints(x) for x in X_r], [_ints(w) for w in W_r]
    M, N = len(Xs[0]), len(Ws[0])
    Y = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc = 0
            for X, W in zip(Xs, Ws):
                for a, b in zip(X[m], W[n]):
                    acc += a * b
            Y[m][n] = acc
    return np.array(Y, dtype=np.float64).reshape(M, N)


def py_ag(A_r, W):
    rows = [row for a in A_r for row in _ints(a)]
    Wi = _ints(W)
    Y = [[sum(a * b for a, b in zip(r, w)) for w in Wi] for r in rows]
    return np.array(Y, dtype=np.float64).reshape(len(rows), len(Wi))


# ---------------------------------------------------------------- bf16 decode

def test_bf16_decode_golden(oracle_mod):
    with open(os.path.join(GOLDEN, "bf16_patterns.json")) as f:
        pats = json.load(f)["patterns"]
    for hexbits, value, _why in pats:
        got = oracle_mod.bf16_to_f64(int(hexbits, 16))
        want = float(value)
        assert got == want, (hexbits, got, want)
        assert math.copysign(1.0, got) == math.copysign(1.0, want), hexbits


def test_bf16_decode_all_patterns_match_torch(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.bf16_to_f64(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


# ---------------------------------------------------------------- hand-worked

def _golden():
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        return json.load(f)


def test_ar_hand_worked(oracle_mod):
    g = _golden()["ar"]
    X = [_bf16(x) for x in g["X_r"]]
    W = [_bf16(w) for w in g["W_r"]]
    assert np.array_equal(oracle_mod.ar(X, W), np.array(g["Y"], dtype=np.float64))


def test_rs_hand_worked(oracle_mod):
    g = _golden()
    X = [_bf16(x) for x in g["ar"]["X_r"]]
    W = [_bf16(w) for w in g["ar"]["W_r"]]
    outs = oracle_mod.rs(X, W)
    rs = g["rs"]
    assert len(outs) == 2
    for s, (o, nvalid, want) in enumerate(zip(outs, rs["valid_rows"], rs["Y_s"])):
        assert o.shape[0] == rs["rows_per_shard"]
        assert oracle_mod.rs_rows(3, 2, s)[1] == nvalid
        assert np.array_equal(o[:nvalid], np.array(want, dtype=np.float64))
        assert np.isnan(o[nvalid:]).all()


def test_ag_hand_worked(oracle_mod):
    g = _golden()["ag"]
    A = [_bf16(a) for a in g["A_r"]]
    W = _bf16(g["W"])
    assert np.array_equal(oracle_mod.ag(A, W), np.array(g["Y"], dtype=np.float64))


# ---------------------------------------------------------------- brute force

AR_SHAPES = [
    (1, 1, [1]),
    (5, 7, [8]),
    (9, 4, [8, 16, 3]),
    (33, 40, [16, 8, 24]),
    (4, 9, [2, 5]),
]


@pytest.mark.parametrize("M,N,K_r", AR_SHAPES)
def test_ar_bruteforce_integers(oracle_mod, M, N, K_r):
    inp = gi.integer_ar(M, N, K_r, amp=3, seed=7 + M)
    assert np.array_equal(oracle_mod.ar(inp.X_r, inp.W_r), py_ar(inp.X_r, inp.W_r))


@pytest.mark.parametrize("M,R", [(129, 2), (5, 3), (4, 3), (7, 16), (32, 4), (1, 2)])
def test_rs_rows_and_values(oracle_mod, M, R):
    rps = -(-M // R)
    covered = []
    for s in range(R):
        first, count = oracle_mod.rs_rows(M, R, s)
        assert first == min(M, s * rps)
        assert count == max(0, min(M, (s + 1) * rps) - s * rps)
        covered += list(range(first, first + count))
    assert covered == list(range(M))
    K_r = [8] * R if R <= 3 else [4] * R
    inp = gi.integer_ar(M, 6, K_r, amp=2, seed=M + R)
    Y = py_ar(inp.X_r, inp.W_r)
    outs = oracle_mod.rs(inp.X_r, inp.W_r)
    for s, o in enumerate(outs):
        first, count = oracle_mod.rs_rows(M, R, s)
        assert o.shape == (rps, 6)
        assert np.array_equal(o[:count], Y[first:first + count])
        assert np.isnan(o[count:]).all()


@pytest.mark.parametrize("M_r,N,K", [([3, 0, 4], 5, 9), ([1], 3, 8), ([2, 7, 1, 5], 11, 16)])
def test_ag_bruteforce_integers(oracle_mod, M_r, N, K):
    inp = gi.integer_ag(M_r, N, K, amp=3, seed=sum(M_r))
    assert np.array_equal(oracle_mod.ag(inp.A_r, inp.W), py_ag(inp.A_r, inp.W))


# ---------------------------------------------------------------- invariants

def test_partial_sum_invariant_integers(oracle_mod):
    inp = gi.integer_ar(17, 23, [8, 24, 16, 8], amp=3, seed=3)
    full_X = torch.cat(inp.X_r, dim=1)
    full_W = torch.cat(inp.W_r, dim=1)
    assert np.array_equal(oracle_mod.ar(inp.X_r, inp.W_r), oracle_mod.ar([full_X], [full_W]))


def test_partial_sum_invariant_gaussian(oracle_mod):
    inp = gi.gaussian_ar(40, 48, [64, 32, 96], seed=11)
    full_X = torch.cat(inp.X_r, dim=1)
    full_W = torch.cat(inp.W_r, dim=1)
    a = oracle_mod.ar(inp.X_r, inp.W_r)
    b = oracle_mod.ar([full_X], [full_W])
    assert np.max(np.abs(a - b) / (np.abs(b) + 1e-300)) <= 1e-12 or np.allclose(a, b, rtol=1e-12, atol=1e-14)


def test_ag_identity_equals_gemm_on_concatenation(oracle_mod):
    inp = gi.gaussian_ag([13, 1, 30, 7], 21, 40, seed=5)
    cat = torch.cat(inp.A_r, dim=0)
    assert np.array_equal(oracle_mod.ag(inp.A_r, inp.W), oracle_mod.ar([cat], [inp.W]))


# ---------------------------------------------------------------- special cases

def test_r1_is_textbook_gemm(oracle_mod):
    inp = gi.gaussian_ar(19, 27, [72], seed=2)
    X = inp.X_r[0].to(torch.float64).numpy()
    W = inp.W_r[0].to(torch.float64).numpy()
    ref = X @ W.T
    got = oracle_mod.ar(inp.X_r, inp.W_r)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_identity_weight_returns_x(oracle_mod):
    K_r = [8, 16, 8]
    K = sum(K_r)
    inp = gi.gaussian_ar(11, K, K_r, seed=4)
    eye = torch.eye(K, dtype=torch.bfloat16)
    W_r, c = [], 0
    for k in K_r:
        W_r.append(eye[:, c:c + k].contiguous())
        c += k
    X = torch.cat(inp.X_r, dim=1).to(torch.float64).numpy()
    assert np.array_equal(oracle_mod.ar(inp.X_r, W_r), X)


def test_one_hot_rows_select_weight_columns(oracle_mod):
    K_r = [8, 8]
    K, M, N = 16, 16, 9
    X = torch.zeros(M, K, dtype=torch.bfloat16)
    for m in range(M):
        X[m, (5 * m + 3) % K] = 1.0
    inp = gi.gaussian_ar(M, N, K_r, seed=6)
    X_r = [X[:, :8].contiguous(), X[:, 8:].contiguous()]
    W = torch.cat(inp.W_r, dim=1).to(torch.float64).numpy()
    Y = oracle_mod.ar(X_r, inp.W_r)
    for m in range(M):
        assert np.array_equal(Y[m], W[:, (5 * m + 3) % K])


def test_zero_and_negated_inputs(oracle_mod):
    inp = gi.gaussian_ar(9, 10, [16, 8], seed=8)
    Z = [torch.zeros_like(x) for x in inp.X_r]
    assert np.array_equal(oracle_mod.ar(Z, inp.W_r), np.zeros((9, 10)))
    Y = oracle_mod.ar(inp.X_r, inp.W_r)
    Yn = oracle_mod.ar([-x for x in inp.X_r], inp.W_r)
    assert np.array_equal(Yn, -Y)


def test_point_queries_match_full(oracle_mod):
    inp = gi.gaussian_ar(37, 29, [24, 8], seed=9)
    Y = oracle_mod.ar(inp.X_r, inp.W_r)
    rng = np.random.default_rng(0)
    rows, cols = rng.integers(0, 37, 200), rng.integers(0, 29, 200)
    assert np.array_equal(oracle_mod.ar_at(inp.X_r, inp.W_r, rows, cols), Y[rows, cols])
    ag = gi.gaussian_ag([5, 11, 3], 17, 24, seed=10)
    Ya = oracle_mod.ag(ag.A_r, ag.W)
    rows, cols = rng.integers(0, 19, 200), rng.integers(0, 17, 200)
    assert np.array_equal(oracle_mod.ag_at(ag.A_r, ag.W, rows, cols), Ya[rows, cols])


# ---------------------------------------------------------------- packed gather

def _bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def py_pack(S, rows_out):
    """The packed gather in plain Python lists (no oracle code): every rank's rows
    in rank order, each row the concatenation of the rank's T states."""
    rows = []
    for states in S:
        for i in range(len(states[0])):
            rows.append([v for st in states for v in st[i]])
    return rows[:rows_out]


def _random_states(M_r, T, H, seed):
    g = torch.Generator().manual_seed(seed)
    return [[_bits_of(torch.randn(m, H, generator=g).to(torch.bfloat16)) for _ in range(T)]
            for m in M_r]


def test_pack_gather_hand_worked(oracle_mod):
    gold = json.load(open(os.path.join(GOLDEN, "pack_gather.json")))
    S = [[_bits_of(_bf16(st)) for st in rank] for rank in gold["S"]]
    P = oracle_mod.pack_gather(S, gold["rows_out"])
    assert np.array_equal(P, _bits_of(_bf16(gold["P"])))


PACK_SHAPES = [([3, 0, 5, 2], 2, 8, 10), ([4, 4], 1, 16, 7), ([1], 4, 8, 1),
               ([0, 6], 3, 8, 6), ([5, 5, 5], 2, 24, 11), ([2, 3], 5, 8, 5)]


@pytest.mark.parametrize("M_r,T,H,rows_out", PACK_SHAPES)
def test_pack_gather_bruteforce(oracle_mod, M_r, T, H, rows_out):
    S = _random_states(M_r, T, H, seed=sum(M_r) + T + H)
    P = oracle_mod.pack_gather(S, rows_out)
    assert P.tolist() == py_pack([[s.tolist() for s in st] for st in S], rows_out)


@pytest.mark.parametrize("M_r,T,H,rows_out", PACK_SHAPES)
def test_pack_gather_splits_back_into_the_gathered_states(oracle_mod, M_r, T, H, rows_out):
    """The page's symmetry: splitting the packed rows by H gives, for every state
    t, the ranks' state-t rows concatenated in rank order and cut to rows_out."""
    S = _random_states(M_r, T, H, seed=7 * T + H)
    P = oracle_mod.pack_gather(S, rows_out)
    for t in range(T):
        gathered = np.concatenate([S[r][t] for r in range(len(M_r))], axis=0)[:rows_out]
        assert np.array_equal(P[:, t * H:(t + 1) * H], gathered)


def test_pack_gather_special_cases(oracle_mod):
    S = _random_states([3, 2], 1, 8, seed=3)
    # T = 1: a plain all-gather of the hidden state
    assert np.array_equal(oracle_mod.pack_gather(S, 5), np.concatenate([S[0][0], S[1][0]]))
    # R = 1: a plain concatenation along the last dimension
    S1 = _random_states([4], 3, 8, seed=4)
    assert np.array_equal(oracle_mod.pack_gather(S1, 4), np.concatenate(S1[0], axis=1))
    # nothing kept
    assert oracle_mod.pack_gather(S, 0).shape == (0, 8)
    with pytest.raises(ValueError):
        oracle_mod.pack_gather(S, 6)


# ---------------------------------------------------------------- mutants

# Plausible slips in the oracle source; each must make at least one pin fail.
MUTANTS = {
    "drop_last_shard": ("for (int r = 1; r < R; ++r)", "for (int r = 1; r < R - 1; ++r)"),
    "short_k_loop": ("for (int64_t k = 0; k < K_r; ++k)", "for (int64_t k = 1; k < K_r; ++k)"),
    "transposed_weight_row": ("const uint16_t *w = W_r + n * K_r;", "const uint16_t *w = W_r + (m % (n + 1)) * K_r;"),
    "subtract_shard": ("y += shard_partial(X_r[r], W_r[r], K_r[r], m, n);",
                       "y -= shard_partial(X_r[r], W_r[r], K_r[r], m, n);"),
    "floor_rows_per_shard": ("int64_t rps = (M + R - 1) / R;", "int64_t rps = M / R + (M % R != 0) * (R > 2);"),
    "widen_shift": ("((uint32_t)bits) << 16", "((uint32_t)bits) << 15"),
    "ag_shard_order": ("const uint16_t *a = A_r[r] + (g - offset) * K;",
                       "const uint16_t *a = A_r[R - 1 - r] + (g - offset) * K;"),
    "pack_state_order": ("const uint16_t *src = S[r * T + t] + (g - offset) * H;",
                         "const uint16_t *src = S[r * T + (T - 1 - t)] + (g - offset) * H;"),
    "pack_rank_order": ("const uint16_t *src = S[r * T + t] + (g - offset) * H;",
                        "const uint16_t *src = S[(R - 1 - r) * T + t] + (g - offset) * H;"),
    "pack_reversed_columns": ("dst[h] = src[h];", "dst[h] = src[H - 1 - h];"),
}


def _pins_pass(oracle_mod) -> bool:
    try:
        test_bf16_decode_golden(oracle_mod)
        test_ar_hand_worked(oracle_mod)
        test_rs_hand_worked(oracle_mod)
        test_ag_hand_worked(oracle_mod)
        for M, N, K_r in AR_SHAPES:
            test_ar_bruteforce_integers(oracle_mod, M, N, K_r)
        for M, R in [(129, 2), (5, 3), (7, 16)]:
            test_rs_rows_and_values(oracle_mod, M, R)
        test_ag_bruteforce_integers(oracle_mod, [2, 7, 1, 5], 11, 16)
        # an AG case with equal shard sizes, so that a shard-order slip stays in bounds
        inp = gi.integer_ag([3, 3, 3], 5, 8, amp=3, seed=12)
        assert np.array_equal(oracle_mod.ag(inp.A_r, inp.W), py_ag(inp.A_r, inp.W))
        # packed gather: the hand-worked case first (equal shard sizes, so that a
        # rank-order slip stays in bounds), then the brute-force shapes
        test_pack_gather_hand_worked(oracle_mod)
        for M_r, T, H, rows_out in PACK_SHAPES:
            test_pack_gather_bruteforce(oracle_mod, M_r, T, H, rows_out)
    except AssertionError:
        return False
    return True


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(oracle_mod, tmp_path, monkeypatch, name):
    import ctypes
    src = open(os.path.join(os.path.dirname(oracle_mod.__file__), "gsr_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    str(mutant), "-o", str(so)], check=True)
    real = oracle_mod._load()
    lib = ctypes.CDLL(str(so))
    for fname in ("gsr_oracle_bf16_to_f64", "gsr_oracle_threads", "gsr_oracle_ar",
                  "gsr_oracle_ar_at", "gsr_oracle_rs_rows", "gsr_oracle_rs",
                  "gsr_oracle_ag", "gsr_oracle_ag_at", "gsr_oracle_pack_gather"):
        f, g = getattr(real, fname), getattr(lib, fname)
        g.argtypes, g.restype = f.argtypes, f.restype
    assert _pins_pass(oracle_mod), "pins must pass on the real oracle"
    monkeypatch.setattr(oracle_mod, "_lib", lib)
    assert not _pins_pass(oracle_mod), f"mutant {name} survived every pin"


def test_oracle_source_compiles_warning_free():
    """The oracle's C builds without warnings, with OpenMP and without it."""
    import subprocess
    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                       "gsr_oracle.c")
    for extra in (["-fopenmp"], ["-Wno-unknown-pragmas"]):
        r = subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                            *extra, src], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
