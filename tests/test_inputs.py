"""The seeded input recipe (shared by the tests, the benchmark and the smoke
check), checked on the CPU: deterministic per seed, shards that are slices of
one full draw in their own allocations, bf16 as the round-to-nearest-even cast
of the fp32 draw, integer variants inside their range, and the weight scale
1/sqrt(K) of the recipe."""
import math

import torch

from tensor_gemm_reduction_gb300 import inputs as gi


def test_same_seed_same_bits_and_shards_are_slices_of_one_draw():
    a = gi.gaussian_ar(33, 40, [8, 24, 16], seed=9)
    b = gi.gaussian_ar(33, 40, [8, 24, 16], seed=9)
    for x, y in zip(a.X_r + a.W_r, b.X_r + b.W_r):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    g = torch.Generator().manual_seed(9)
    X = torch.randn(33, 48, generator=g)
    W = torch.randn(40, 48, generator=g) / math.sqrt(48)
    assert torch.equal(torch.cat(a.X_r, 1).view(torch.int16), X.to(torch.bfloat16).view(torch.int16))
    assert torch.equal(torch.cat(a.W_r, 1).view(torch.int16), W.to(torch.bfloat16).view(torch.int16))
    ptrs = {t.data_ptr() for t in a.X_r + a.W_r}
    assert len(ptrs) == 6 and all(t.is_contiguous() for t in a.X_r + a.W_r)


def test_ag_shards_are_row_slices_and_empty_shards_exist():
    a = gi.gaussian_ag([5, 0, 7], 16, 24, seed=3)
    assert [t.shape for t in a.A_r] == [(5, 24), (0, 24), (7, 24)]
    g = torch.Generator().manual_seed(3)
    A = torch.randn(12, 24, generator=g).to(torch.bfloat16)
    assert torch.equal(torch.cat(a.A_r, 0).view(torch.int16), A.view(torch.int16))
    assert a.M == 12 and a.R == 3 and a.W.shape == (16, 24)


def test_default_seed_follows_the_pages_rule():
    w = gi.Workload("x", "ar", N=64, K=128, R=2, M=32)
    assert gi.default_seed(w.M, w.K) == 2000 + 32 + 128
    a = gi.make_inputs(w)
    b = gi.gaussian_ar(32, 64, [64, 64], seed=2000 + 32 + 128)
    assert torch.equal(a.X_r[1].view(torch.int16), b.X_r[1].view(torch.int16))


def test_integer_variants_stay_in_range_and_are_exact_in_bf16():
    a = gi.integer_ar(50, 30, [16, 8], amp=3, seed=2)
    for t in a.X_r + a.W_r:
        f = t.float()
        assert f.abs().max() <= 3 and torch.equal(f, f.round())
    s = set(torch.cat([t.flatten() for t in a.X_r]).float().tolist())
    assert s == {-3.0, -2.0, -1.0, 0.0, 1.0, 2.0, 3.0}
    g = gi.integer_ag([4, 9], 10, 16, amp=1, seed=4)
    assert set(torch.cat([t.flatten() for t in g.A_r]).float().tolist()) <= {-1.0, 0.0, 1.0}


def test_weight_scale_makes_outputs_unit_variance():
    """W ~ N(0, 1/K) with X ~ N(0, 1): each output has variance about 1, which
    the tolerance of the parity tests assumes (|ref| of order 1)."""
    a = gi.gaussian_ar(64, 256, [512, 512], seed=1)
    Y = torch.cat(a.X_r, 1).double() @ torch.cat(a.W_r, 1).double().t()
    assert 0.85 < Y.var().item() < 1.15


def test_states_are_separate_allocations():
    S = gi.gaussian_states([3, 0, 2], 4, 16, seed=5)
    assert [len(s) for s in S] == [4, 4, 4]
    assert all(t.shape == (m, 16) and t.dtype == torch.bfloat16 for s, m in zip(S, (3, 0, 2)) for t in s)
    ptrs = [t.data_ptr() for s in S for t in s if t.numel()]
    assert len(set(ptrs)) == len(ptrs)
