"""C-ABI checks that need no GPU: the library loads, exports every entry point
the header declares, and its host logic (argument validation, workspace sizing,
kernel configuration) behaves as documented. Calls go straight through ctypes
with made-up device addresses; a host plan never dereferences them."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from tensor_gemm_reduction_gb300 import binding as B
from tensor_gemm_reduction_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return B.load_library()


def header_functions():
    text = open(os.path.join(ROOT, "include", "gsr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in ("gemm_shard_plan_create", "gemm_shard_plan_destroy", "gemm_ar", "gemm_rs", "gemm_ag",
              "gemm_shard_workspace_size", "gemm_shard_check_status", "gsr_last_error_string"):
        assert n in names
    assert sorted(names) == sorted(B.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for n in header_functions():
        assert hasattr(lib, n), f"{n} declared in gsr.h but not exported"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU path")
def test_device_plan_without_gpu_is_unsupported(lib):
    h = ctypes.c_void_p(123)
    st = lib.gemm_shard_plan_create(ctypes.byref(h), 0, 128, 256, 256, 2)
    assert st == B.GSR_ERR_UNSUPPORTED
    assert h.value is None
    assert B.gsr_last_error_string()


def test_null_plan_is_rejected(lib):
    assert lib.gemm_shard_workspace_size(None) == 0
    assert lib.gemm_shard_plan_set_option(None, B.GSR_OPT_SPLIT_K, 2) == B.GSR_ERR_INVALID_VALUE
    assert "NULL" in B.gsr_last_error_string()
    assert lib.gemm_shard_plan_destroy(None) == B.GSR_OK


@pytest.mark.parametrize("args", [
    (0, 128, 256, 256, 2),      # sm_count
    (148, 0, 256, 256, 2),      # max_M
    (148, 128, 250, 256, 2),    # max_N not a multiple of 8
    (148, 128, 256, 12, 2),     # max_K not a multiple of 8
    (148, 128, 256, 256, 0),    # max_R
    (148, 128, 256, 256, 17),   # max_R > 16
    (148, 1 << 24, 1 << 20, 256, 2),   # 2^30 output tiles: past 32-bit piece counts
])
def test_host_plan_rejects_bad_maxima(lib, args):
    h = ctypes.c_void_p()
    assert lib.gemm_shard_plan_create_host(ctypes.byref(h), *args) == B.GSR_ERR_INVALID_VALUE
    assert h.value is None


def test_host_plan_accepts_the_largest_tile_count(lib):
    # (2^20 / 128 + 2 R) x (2^16 / 128) tiles = (8192 + 4) x 512, well inside 2^27;
    # one more factor of 32 in N crosses it.
    h = ctypes.c_void_p()
    assert lib.gemm_shard_plan_create_host(ctypes.byref(h), 148, 1 << 20, 1 << 16, 256, 2) == B.GSR_OK
    lib.gemm_shard_plan_destroy(h)
    assert lib.gemm_shard_plan_create_host(ctypes.byref(h), 148, 1 << 20, 1 << 21, 256, 2) \
        == B.GSR_ERR_INVALID_VALUE
    assert "output tiles" in B.gsr_last_error_string()


def _arr(ctype, vals):
    return (ctype * len(vals))(*vals)


class Host:
    """A host plan plus raw-pointer call helpers."""

    def __init__(self, lib, sm=148, max_M=32768, max_N=8192, max_K=8192, max_R=16):
        self.lib = lib
        self.plan = B.gemm_shard_plan_create_host(sm, max_M, max_N, max_K, max_R)
        self.ws_bytes = B.gemm_shard_workspace_size(self.plan)

    def ar(self, M, N, K_r, x=None, w=None, y=0x10000, ws=0x20000000, ws_bytes=None, mode="ar"):
        R = len(K_r)
        x = x if x is not None else [0x100000 * (r + 1) for r in range(R)]
        w = w if w is not None else [0x100000 * (r + 1) + 0x80000 for r in range(R)]
        ws_bytes = self.ws_bytes if ws_bytes is None else ws_bytes
        k = _arr(ctypes.c_int64, K_r)
        xa = _arr(ctypes.c_void_p, x)
        wa = _arr(ctypes.c_void_p, w)
        if mode == "ar":
            return self.lib.gemm_ar(self.plan.handle, M, N, R, k, xa, wa, ctypes.c_void_p(y),
                                    ctypes.c_void_p(ws), ws_bytes, None)
        ya = _arr(ctypes.c_void_p, y if isinstance(y, list) else [y + 0x1000 * r for r in range(R)])
        return self.lib.gemm_rs(self.plan.handle, M, N, R, k, xa, wa, ya, ctypes.c_void_p(ws),
                                ws_bytes, None)

    def ag(self, N, K, M_r, a=None, w=0x700000, y=0x10000, ws=0x20000000, ws_bytes=None):
        R = len(M_r)
        a = a if a is not None else [0x100000 * (r + 1) for r in range(R)]
        ws_bytes = self.ws_bytes if ws_bytes is None else ws_bytes
        return self.lib.gemm_ag(self.plan.handle, N, K, R, _arr(ctypes.c_int64, M_r),
                                _arr(ctypes.c_void_p, a), ctypes.c_void_p(w), ctypes.c_void_p(y),
                                ctypes.c_void_p(ws), ws_bytes, None)

    def describe(self, mode, M, N, K, sizes):
        return B.gemm_shard_describe(self.plan, mode, M, N, K, sizes)


@pytest.fixture()
def host(lib):
    return Host(lib)


def test_valid_calls_reach_the_launch_point(host):
    assert host.ar(128, 7168, [896] * 8) == B.GSR_ERR_UNSUPPORTED
    assert "arguments are valid" in B.gsr_last_error_string()
    assert host.ar(129, 7168, [896] * 8, mode="rs") == B.GSR_ERR_UNSUPPORTED
    assert host.ag(6288, 7168, [4096] * 8) == B.GSR_ERR_UNSUPPORTED


def test_empty_problems_return_ok_without_launch(host):
    assert host.ar(0, 256, [128, 128]) == B.GSR_OK
    assert host.ar(0, 256, [128, 128], mode="rs") == B.GSR_OK
    assert host.ag(256, 128, [0, 0, 0]) == B.GSR_OK


@pytest.mark.parametrize("kw,frag", [
    (dict(M=-1, N=256, K_r=[128]), "M must be"),
    (dict(M=40000, N=256, K_r=[128]), "max_M"),
    (dict(M=16, N=12, K_r=[128]), "multiple of 8"),
    (dict(M=16, N=0, K_r=[128]), "multiple of 8"),
    (dict(M=16, N=8200, K_r=[128]), "max_N"),
    (dict(M=16, N=256, K_r=[]), "R=0"),
    (dict(M=16, N=256, K_r=[8] * 17), "R=17"),
    (dict(M=16, N=256, K_r=[128, 20]), "K_r[1]"),
    (dict(M=16, N=256, K_r=[128, 0]), "K_r[1]"),
    (dict(M=16, N=256, K_r=[4096, 4104]), "max_K"),
    (dict(M=16, N=256, K_r=[128, 128], x=[0x100000, 0x100008]), "16-byte"),
    (dict(M=16, N=256, K_r=[128, 128], w=[0x100000, 0]), "NULL"),
    (dict(M=16, N=256, K_r=[128], y=0x10004), "16-byte"),
    (dict(M=16, N=256, K_r=[128], y=0), "Y must"),
])
def test_ar_argument_validation(host, kw, frag):
    assert host.ar(**kw) == B.GSR_ERR_INVALID_VALUE
    assert frag in B.gsr_last_error_string()


def test_rs_output_validation(host):
    assert host.ar(16, 256, [128, 128], y=[0x10000, 0x10008], mode="rs") == B.GSR_ERR_INVALID_VALUE
    assert host.ar(16, 256, [128, 128], y=[0x10000, 0], mode="rs") == B.GSR_ERR_INVALID_VALUE


@pytest.mark.parametrize("kw,frag", [
    (dict(N=256, K=100, M_r=[16]), "K must"),
    (dict(N=256, K=9000, M_r=[16]), "max_K"),
    (dict(N=252, K=128, M_r=[16]), "N must"),
    (dict(N=256, K=128, M_r=[16, -1]), "M_r[1]"),
    (dict(N=256, K=128, M_r=[16, 16], a=[0x100000, 0]), "A_r[1]"),
    (dict(N=256, K=128, M_r=[16], w=0x700008), "W must"),
    (dict(N=256, K=128, M_r=[20000, 20000]), "max_M"),
])
def test_ag_argument_validation(host, kw, frag):
    assert host.ag(**kw) == B.GSR_ERR_INVALID_VALUE
    assert frag in B.gsr_last_error_string()


@pytest.mark.parametrize("args,frag", [
    ((B.MODE_AR, -1, 256, 0, [128]), "M must"),
    ((B.MODE_AR, 16, 256, 0, [128, 20]), "K_r[1]"),
    ((B.MODE_RS, 16, 256, 0, [0]), "K_r[0]"),
    ((B.MODE_AG, 0, 256, 0, [16]), "K must"),
    ((B.MODE_AG, 0, 256, 100, [16]), "K must"),
    ((B.MODE_AG, 0, 256, 128, [16, -1]), "M_r[1]"),
    ((B.MODE_AR, 16, 250, 0, [128]), "N must"),
    ((3, 16, 256, 0, [128]), "mode"),
    ((B.MODE_AR, 16, 256, 0, []), "bad R"),
])
def test_describe_argument_validation(host, args, frag):
    with pytest.raises(B.GsrError) as e:
        host.describe(*args)
    assert e.value.status == B.GSR_ERR_INVALID_VALUE
    assert frag in str(e.value)


def test_ag_null_pointer_allowed_for_empty_shard(host):
    assert host.ag(256, 128, [16, 0, 8], a=[0x100000, 0, 0x300000]) == B.GSR_ERR_UNSUPPORTED


def test_workspace_checks(host):
    assert host.ar(128, 7168, [896] * 8, ws=0) == B.GSR_ERR_WORKSPACE
    assert host.ar(128, 7168, [896] * 8, ws=0x20000080) == B.GSR_ERR_WORKSPACE
    assert "256-byte" in B.gsr_last_error_string()
    assert host.ar(128, 7168, [896] * 8, ws_bytes=1024) == B.GSR_ERR_WORKSPACE
    assert "too small" in B.gsr_last_error_string()


def test_workspace_size_covers_every_heuristic_config(host):
    # The plan's bound must cover the per-call requirement of every shape.
    for M in (1, 7, 127, 128, 129, 257, 1000, 4096, 32768):
        for N in (8, 136, 3648, 6288, 7168, 8192):
            for K_r in ([896] * 8, [8], [4096, 4096], [448] * 16):
                d = host.describe(B.MODE_AR, M, N, 0, K_r)
                assert d["workspace_bytes"] <= host.ws_bytes
                assert host.ar(M, N, K_r) == B.GSR_ERR_UNSUPPORTED, B.gsr_last_error_string()
    for M_r in ([256] * 8, [384] * 8, [4096] * 8, [1, 130, 0, 257]):
        for N in (3648, 6288):
            d = host.describe(B.MODE_AG, 0, N, 7168, M_r)
            assert d["workspace_bytes"] <= host.ws_bytes


def test_config_is_independent_of_mode(host):
    for M in (1, 128, 129, 1000, 4096, 32768):
        for K_r in ([896] * 8, [3584] * 2, [448] * 16, [8, 72, 136]):
            a = host.describe(B.MODE_AR, M, 7168, 0, K_r)
            r = host.describe(B.MODE_RS, M, 7168, 0, K_r)
            assert a == r


def test_small_m_uses_the_pair_tile_kernel(host):
    # M <= 256 (AR/RS): the small-M kernel, one CTA pair per tile of W rows
    # (block_n, the pair MMA's N) over the whole K range, against all rows.
    # The tile height is the smallest multiple of 16 that spreads N over every
    # pair in the fewest waves: N = 7168 on 148 SMs (74 pairs) gives 112-row
    # tiles, 64 tiles on 128 CTAs, whatever M up to 256; on 152 SMs, 96 rows
    # and 75 tiles on 150 CTAs.
    for M in (1, 16, 127, 128, 129, 200, 256):
        d = host.describe(B.MODE_AR, M, 7168, 0, [896] * 8)
        assert (d["cta_group"], d["block_n"], d["schedule"], d["split"], d["tiles"], d["ctas"]) == \
            (2, 112, 3, 1, 64, 128), M
        # no split-K partials or counters: the workspace is the fixed minimum
        assert d["workspace_bytes"] <= host.describe(B.MODE_AR, 4096, 7168, 0, [896] * 8)["workspace_bytes"]
    d = Host(host.lib, sm=152).describe(B.MODE_AR, 64, 7168, 0, [896] * 8)
    assert (d["block_n"], d["tiles"], d["ctas"]) == (96, 75, 150)
    # more tiles than pairs: tiles walked in turn; N = 32640 needs two waves
    # of at most 256 rows: 224-row tiles
    d = host.describe(B.MODE_AR, 64, 32768 - 128, 0, [896] * 8)
    assert (d["schedule"], d["block_n"], d["tiles"], d["ctas"]) == (3, 224, 146, 148)
    # small N: one tile of 16 rows
    d = host.describe(B.MODE_AR, 64, 8, 0, [896] * 8)
    assert (d["block_n"], d["tiles"], d["ctas"]) == (16, 1, 2)
    # the tile height as an option: 128 rows, 56 tiles on 112 CTAs
    h = Host(host.lib)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SMALL_TILE_ROWS, 128)
    d = h.describe(B.MODE_AR, 128, 7168, 0, [896] * 8)
    assert (d["schedule"], d["block_n"], d["tiles"], d["ctas"]) == (3, 128, 56, 112)
    for bad in (-16, 8, 20, 136, 272):
        with pytest.raises(B.GsrError):
            B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SMALL_TILE_ROWS, bad)
    # k-blocks per copy: the largest of 4, 3, 2, 1 that leaves a ring of four
    # stages, unless a shard has a ragged k-block; a shard's last copy may run
    # past its k-blocks (14 per shard of 896: four copies of 4)
    assert host.describe(B.MODE_AR, 1, 7168, 0, [896] * 8)["kblocks"] == 4       # 4 x 9 KB stages
    assert host.describe(B.MODE_AR, 64, 7168, 0, [896] * 8)["kblocks"] == 4     # 32 rows a CTA
    assert host.describe(B.MODE_AR, 128, 7168, 0, [896] * 8)["kblocks"] == 3    # 4 x 15 KB: 3 fit
    assert Host(host.lib, sm=152).describe(B.MODE_AR, 128, 7168, 0, [896] * 8)["kblocks"] == 4
    assert host.describe(B.MODE_AR, 1, 7168, 0, [1024] * 7)["kblocks"] == 4
    assert host.describe(B.MODE_AR, 129, 7168, 0, [896] * 8)["kblocks"] == 3    # 80 rows a CTA
    assert host.describe(B.MODE_AR, 200, 7168, 0, [1024] * 7)["kblocks"] == 2   # 112 rows a CTA
    assert host.describe(B.MODE_AR, 64, 7168, 0, [8, 72, 136])["kblocks"] == 1  # ragged
    assert host.describe(B.MODE_AR, 4096, 7168, 0, [1024] * 7)["kblocks"] == 1  # the main kernel
    h = Host(host.lib)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SMALL_KBLOCKS, 1)
    assert h.describe(B.MODE_AR, 64, 7168, 0, [896] * 8)["kblocks"] == 1
    # a capped grid keeps whole pairs
    h = Host(host.lib)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_MAX_CTAS, 9)
    assert h.describe(B.MODE_AR, 64, 7168, 0, [896] * 8)["ctas"] == 8
    # above 256 rows, or in AG mode: the main kernel; a single k-block is fine
    assert host.describe(B.MODE_AR, 257, 7168, 0, [896] * 8)["schedule"] != 3
    assert host.describe(B.MODE_AR, 64, 7168, 0, [64])["schedule"] == 3
    assert host.describe(B.MODE_AR, 64, 7168, 0, [8])["schedule"] == 3
    assert host.describe(B.MODE_AR, 64, 7168, 0, [8, 8])["schedule"] == 3
    assert host.describe(B.MODE_AG, 0, 7168, 7168, [16] * 8)["schedule"] != 3
    # a forced configuration option selects the main kernel unless small_m = 2
    h = Host(host.lib)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_BLOCK_N, 256)
    assert h.describe(B.MODE_AR, 128, 7168, 0, [896] * 8)["schedule"] != 3
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SMALL_M, 2)
    assert h.describe(B.MODE_AR, 128, 7168, 0, [896] * 8)["schedule"] == 3
    with pytest.raises(B.GsrError):
        B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SMALL_M, 3)


def test_l2_hints_where_both_operands_fit_in_l2(host):
    # The main kernel asks for A evict-last / B evict-first where A and W fit
    # in the L2 together (126 MiB on a host plan), else for no hints; the
    # option overrides; the small-M kernel always takes them.
    assert host.describe(B.MODE_AG, 0, 3648, 7168, [256] * 8)["l2_hints"] == 2    # 81 MB
    assert host.describe(B.MODE_AG, 0, 3648, 7168, [512] * 8)["l2_hints"] == 2    # 111 MB
    assert host.describe(B.MODE_AG, 0, 3648, 7168, [1024] * 8)["l2_hints"] == 1   # 170 MB
    assert host.describe(B.MODE_AG, 0, 6288, 7168, [4096] * 8)["l2_hints"] == 1
    assert host.describe(B.MODE_AR, 1000, 7168, 0, [896] * 8)["l2_hints"] == 2    # 117 MB
    assert host.describe(B.MODE_RS, 1000, 7168, 0, [896] * 8)["l2_hints"] == 2
    assert host.describe(B.MODE_AR, 4096, 7168, 0, [896] * 8)["l2_hints"] == 1    # 162 MB
    assert host.describe(B.MODE_AR, 64, 7168, 0, [896] * 8)["l2_hints"] == 2      # small-M
    for v, want in ((1, 1), (2, 2), (3, 3)):
        h = Host(host.lib)
        B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_L2_HINTS, v)
        assert h.describe(B.MODE_AG, 0, 3648, 7168, [256] * 8)["l2_hints"] == want
        assert h.describe(B.MODE_AR, 4096, 7168, 0, [896] * 8)["l2_hints"] == want


def test_small_m_off_splits_tiles(lib):
    h = Host(lib)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SMALL_M, 1)
    # M = 128, one row tile: 56 single-CTA tiles of 128 x 128, each cut into
    # 148 // 56 = 2 pieces of 56 k-blocks: 112 CTAs
    d = h.describe(B.MODE_AR, 128, 7168, 0, [896] * 8)
    assert (d["cta_group"], d["block_n"], d["schedule"], d["split"], d["tiles"], d["ctas"]) == \
        (1, 128, 1, 2, 56, 112)
    # M = 129: one 256-row pair tile keeps W read once: 28 pair tiles x 2 pieces
    d = h.describe(B.MODE_AR, 129, 7168, 0, [896] * 8)
    assert (d["cta_group"], d["block_n"], d["schedule"], d["split"], d["tiles"], d["ctas"]) == \
        (2, 256, 1, 2, 28, 112)
    # stream-K on demand: every tile's 112 k-blocks shared out over all SMs
    plan2 = B.gemm_shard_plan_create_host(148, 32768, 8192, 8192, 16)
    B.gemm_shard_plan_set_option(plan2, B.GSR_OPT_SCHEDULE, 3)
    B.gemm_shard_plan_set_option(plan2, B.GSR_OPT_CTA_GROUP, 1)
    d = B.gemm_shard_describe(plan2, B.MODE_AR, 128, 7168, 0, [896] * 8)
    assert d["cta_group"] == 1 and d["schedule"] == 2 and d["tiles"] == 28
    assert d["dp_tiles"] == 0 and d["sk_iters"] == 28 * 112 and d["ctas"] == 148


def test_uniform_schedule_splits_small_m(lib):
    h = Host(lib)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SCHEDULE, 1)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_CTA_GROUP, 1)
    d = h.describe(B.MODE_AR, 128, 7168, 0, [896] * 8)
    assert (d["schedule"], d["split"], d["ctas"], d["cta_group"]) == (1, 5, 140, 1)
    assert d["workspace_bytes"] <= B.gemm_shard_workspace_size(h.plan)


def test_large_m_uses_cta_pairs_and_a_stream_k_tail(host):
    # 256 x 256 tiles per CTA pair: 128 x 28 = 3584 tiles on 74 pairs is 48.4
    # waves; the partial last wave (32 tiles, under half a wave) is cut into two
    # k-pieces per tile, one per worker (split tail)
    d = host.describe(B.MODE_AR, 32768, 7168, 0, [896] * 8)
    assert d["cta_group"] == 2 and d["schedule"] == 4 and d["ctas"] == 148
    assert d["tiles"] == 3584 and d["dp_tiles"] == 48 * 74 and d["split"] == 2 and d["sk_iters"] == 0
    # or shared out k-block by k-block (stream-K over the partial last wave)
    plan3 = B.gemm_shard_plan_create_host(148, 32768, 8192, 8192, 16)
    B.gemm_shard_plan_set_option(plan3, B.GSR_OPT_SCHEDULE, 3)
    d = B.gemm_shard_describe(plan3, B.MODE_AR, 32768, 7168, 0, [896] * 8)
    assert d["schedule"] == 2 and d["dp_tiles"] == 48 * 74 and d["sk_iters"] == 32 * 112
    plan2 = B.gemm_shard_plan_create_host(148, 32768, 8192, 8192, 16)
    B.gemm_shard_plan_set_option(plan2, B.GSR_OPT_SCHEDULE, 2)   # the last 1.4 waves
    d = B.gemm_shard_describe(plan2, B.MODE_AR, 32768, 7168, 0, [896] * 8)
    assert d["dp_tiles"] == 47 * 74 and d["sk_iters"] == 106 * 112
    d = host.describe(B.MODE_AG, 0, 6288, 7168, [4096] * 8)
    assert d["cta_group"] == 2 and d["tiles"] == 8 * 16 * 25
    # 448-row shards: 64-row granules, two per CTA and possibly from two
    # shards, so no rows are wasted: 3584 rows in 14 pair tiles (not 16)
    d = host.describe(B.MODE_AG, 0, 3648, 7168, [448] * 8)
    assert d["cta_group"] == 2 and d["tiles"] == 14 * 15
    # 384-row shards: 24 half-tiles of 128 rows, paired across shard boundaries
    d = host.describe(B.MODE_AG, 0, 3648, 7168, [384] * 8)
    assert d["cta_group"] == 2 and d["tiles"] == 12 * 15
    # an odd number of half-tiles leaves the last pair's second half idle
    d = host.describe(B.MODE_AG, 0, 6288, 7168, [384] * 7)
    assert d["cta_group"] == 2 and d["tiles"] == 11 * 25


def test_whole_waves_have_no_stream_k(lib):
    h = Host(lib, sm=16)
    d = h.describe(B.MODE_AR, 2048, 4096, 0, [256])   # 8 x 16 = 128 pair tiles on 8 pairs
    assert d["cta_group"] == 2 and d["dp_tiles"] == 128 and d["sk_iters"] == 0
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SCHEDULE, 2)
    d = h.describe(B.MODE_AR, 2304, 4096, 0, [256])   # 9 x 16 = 144 pair tiles on 8 pairs
    assert d["dp_tiles"] == 144 and d["sk_iters"] == 0
    d = h.describe(B.MODE_AR, 2560, 4096, 0, [256])   # 10 x 16 = 160 = 20 waves
    assert d["sk_iters"] == 0
    d = h.describe(B.MODE_AR, 2304, 4000, 0, [256])   # 9 x 16 tiles, 4000 wide: same tiles
    assert d["sk_iters"] == 0


def test_forced_options(lib):
    h = Host(lib, max_M=4096, max_N=1024, max_K=1024, max_R=4)
    base = h.ws_bytes
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SPLIT_K, 3)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_BLOCK_N, 128)
    assert B.gemm_shard_workspace_size(h.plan) > base
    d = h.describe(B.MODE_AR, 1000, 1024, 0, [256, 256])
    assert d["split"] == 3 and d["block_n"] == 128 and d["schedule"] == 1
    assert d["tiles"] == 8 * 8 and d["cta_group"] == 1
    # a forced split never exceeds the number of k-blocks
    d = h.describe(B.MODE_AR, 64, 256, 0, [64])
    assert d["split"] == 1
    for opt, bad in ((B.GSR_OPT_SPLIT_K, 17), (B.GSR_OPT_BLOCK_N, 64), (B.GSR_OPT_TIMEOUT_NS, -1),
                     (B.GSR_OPT_MAX_CTAS, -5), (B.GSR_OPT_SCHEDULE, 6), (B.GSR_OPT_CTA_GROUP, 3),
                     (99, 1)):
        with pytest.raises(B.GsrError) as e:
            B.gemm_shard_plan_set_option(h.plan, opt, bad)
        assert e.value.status == B.GSR_ERR_INVALID_VALUE
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_MAX_CTAS, 10)
    assert h.describe(B.MODE_AR, 4096, 1024, 0, [256])["ctas"] == 10
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_CTA_GROUP, 2)
    d = h.describe(B.MODE_AR, 1000, 1024, 0, [256, 256])
    assert d["cta_group"] == 2 and d["ctas"] == 10 and d["tiles"] == 4 * 8
    assert d["workspace_bytes"] <= B.gemm_shard_workspace_size(h.plan)


def test_host_plan_has_no_device_status(host):
    with pytest.raises(B.GsrError) as e:
        B.load_library()
        st = host.lib.gemm_shard_check_status(host.plan.handle, ctypes.c_void_p(0x20000000), None)
        B._check(st)
    assert e.value.status == B.GSR_ERR_UNSUPPORTED


def test_flagged_ag_and_signal_validation(host):
    lib = host.lib
    M_r = (ctypes.c_int64 * 2)(16, 16)
    A = (ctypes.c_void_p * 2)(0x100000, 0x200000)
    args = lambda ready: (host.plan.handle, 256, 128, 2, M_r, A, ctypes.c_void_p(0x700000),
                          ctypes.c_void_p(0x10000), ctypes.c_void_p(ready), ctypes.c_uint32(1),
                          ctypes.c_void_p(0x20000000), host.ws_bytes, None)
    assert lib.gemm_ag_flagged(*args(0)) == B.GSR_ERR_INVALID_VALUE
    assert lib.gemm_ag_flagged(*args(0x30000002)) == B.GSR_ERR_INVALID_VALUE
    assert lib.gemm_ag_flagged(*args(0x30000000)) == B.GSR_ERR_UNSUPPORTED   # host plan: valid
    assert lib.gemm_shard_signal(host.plan.handle, ctypes.c_void_p(0), 1, None) == B.GSR_ERR_INVALID_VALUE
    assert lib.gemm_shard_signal(host.plan.handle, ctypes.c_void_p(0x30000000), 1, None) == B.GSR_ERR_UNSUPPORTED


def _pack(lib, plan, M_r, T, H, rows_out, S=None, P=0x40000, ws=0x20000000, ws_bytes=4096):
    R = len(M_r)
    S = S if S is not None else [0x100000 * (i + 1) for i in range(R * T)]
    return lib.gemm_shard_pack_gather(plan.handle, R, _arr(ctypes.c_int64, M_r), T, H,
                                      _arr(ctypes.c_void_p, S), rows_out, ctypes.c_void_p(P),
                                      ctypes.c_void_p(ws), ws_bytes, None)


def test_pack_gather_validation(host):
    lib, plan = host.lib, host.plan
    # valid calls reach the launch point; nothing kept returns OK with no launch
    assert _pack(lib, plan, [4096] * 8, 4, 7168, 32765) == B.GSR_ERR_UNSUPPORTED
    assert "arguments are valid" in B.gsr_last_error_string()
    assert _pack(lib, plan, [3, 0, 5], 2, 8, 0) == B.GSR_OK
    # a shard with no kept row may have NULL states; a kept one may not
    S = [0x100000, 0x200000, 0, 0]
    assert _pack(lib, plan, [4, 4], 2, 8, 4, S=S) == B.GSR_ERR_UNSUPPORTED
    assert _pack(lib, plan, [4, 4], 2, 8, 5, S=S) == B.GSR_ERR_INVALID_VALUE
    assert "S[2]" in B.gsr_last_error_string()
    # an empty shard may have NULL states even before rows_out
    assert _pack(lib, plan, [4, 0, 4], 1, 8, 8, S=[0x100000, 0, 0x300000]) == B.GSR_ERR_UNSUPPORTED
    bad = [
        (dict(M_r=[4] * 17, T=1, H=8, rows_out=4), "R="),
        (dict(M_r=[4], T=0, H=8, rows_out=4), "T="),
        (dict(M_r=[4], T=17, H=8, rows_out=4), "T="),
        (dict(M_r=[4], T=1, H=12, rows_out=4), "multiple of 8"),
        (dict(M_r=[4], T=1, H=0, rows_out=4), "multiple of 8"),
        (dict(M_r=[4, -1], T=1, H=8, rows_out=3), "M_r[1]"),
        (dict(M_r=[4, 4], T=1, H=8, rows_out=9), "rows_out"),
        (dict(M_r=[4], T=1, H=8, rows_out=-1), "rows_out"),
        (dict(M_r=[4], T=1, H=8, rows_out=4, P=0x40008), "P must"),
        (dict(M_r=[4], T=1, H=8, rows_out=4, P=0), "P must"),
        (dict(M_r=[4], T=1, H=8, rows_out=4, S=[0x100008]), "16-byte"),
    ]
    for kw, frag in bad:
        assert _pack(lib, plan, **kw) == B.GSR_ERR_INVALID_VALUE, kw
        assert frag in B.gsr_last_error_string(), (kw, B.gsr_last_error_string())
    assert _pack(lib, plan, [4], 1, 8, 4, ws=0) == B.GSR_ERR_WORKSPACE
    assert _pack(lib, plan, [4], 1, 8, 4, ws=0x20000010) == B.GSR_ERR_WORKSPACE
    assert _pack(lib, plan, [4], 1, 8, 4, ws_bytes=128) == B.GSR_ERR_WORKSPACE
    assert lib.gemm_shard_pack_gather(None, 1, _arr(ctypes.c_int64, [4]), 1, 8,
                                      _arr(ctypes.c_void_p, [0x100000]), 4, ctypes.c_void_p(0x40000),
                                      ctypes.c_void_p(0x20000000), 4096, None) == B.GSR_ERR_INVALID_VALUE


def test_stream_k_range_stays_in_32_bit(lib):
    """The kernel walks the stream-K range in 32-bit arithmetic: a range with
    (sk_iters + 1) * (workers + 1) >= 2^32 runs as whole tiles instead."""
    K = (1 << 31) - 128
    h = Host(lib, max_M=32768, max_N=8192, max_K=K, max_R=1)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SCHEDULE, 3)   # stream-K tail
    d = h.describe(B.MODE_AR, 32768, 7168, 0, [K])
    assert d["cta_group"] == 2 and d["sk_iters"] == 0 and d["dp_tiles"] == d["tiles"]
    # an ordinary K keeps its stream-K tail
    d = h.describe(B.MODE_AR, 32768, 7168, 0, [7168])
    assert d["sk_iters"] == 32 * 112 and (d["sk_iters"] + 1) * (74 + 1) < 2 ** 32
    # the split tail (the default here) cuts each tail tile into k-pieces with
    # plain 32-bit products (at most 3 x 2^25 k-blocks)
    h2 = Host(lib, max_M=32768, max_N=8192, max_K=K, max_R=1)
    d = h2.describe(B.MODE_AR, 32768, 7168, 0, [K])
    assert d["schedule"] == 4 and d["split"] == 2 and d["dp_tiles"] == 48 * 74


def test_raster_options_are_validated_and_leave_the_configuration(host):
    """Raster order (by m-tile groups or by n-tile groups) changes only the
    order in which tiles are walked: tiles, pieces and grid stay the same."""
    base = host.describe(B.MODE_AR, 32768, 7168, 0, [896] * 8)
    for opt, v in ((B.GSR_OPT_RASTER_M, 4), (B.GSR_OPT_RASTER_N, 8), (B.GSR_OPT_RASTER_N, 64)):
        h = Host(host.lib)
        B.gemm_shard_plan_set_option(h.plan, opt, v)
        assert h.describe(B.MODE_AR, 32768, 7168, 0, [896] * 8) == base
    h = Host(host.lib)
    for opt in (B.GSR_OPT_RASTER_M, B.GSR_OPT_RASTER_N):
        for bad in (-1, 65):
            with pytest.raises(B.GsrError):
                B.gemm_shard_plan_set_option(h.plan, opt, bad)


def test_192_column_tiles_only_where_they_fill_few_whole_waves(host):
    """On 152 SMs (76 pairs): AG with N = 3648 (19 x 192, not a multiple of
    256) uses 192-column pair tiles at 2048, 3072 and 4096 rows (exactly two,
    three and four waves, no cut tile), 256 columns otherwise (3584 rows in
    64-row granules, 8192 rows: eight waves) and for other N."""
    h = Host(host.lib, sm=152)
    def bn(m_r, N):
        return h.describe(B.MODE_AG, 0, N, 7168, [m_r] * 8)["block_n"]
    assert bn(256, 3648) == 192 and bn(384, 3648) == 192
    assert h.describe(B.MODE_AG, 0, 3648, 7168, [256] * 8)["sk_iters"] == 0
    assert bn(512, 3648) == 192
    assert bn(448, 3648) == 256 and bn(1024, 3648) == 256 and bn(4096, 3648) == 256
    assert bn(256, 6288) == 256 and bn(256, 7168) == 256
    # AR and RS on the same shape get the same tiles
    d_ar = h.describe(B.MODE_AR, 2048, 3648, 0, [896] * 8)
    assert d_ar["block_n"] == 192 and h.describe(B.MODE_RS, 2048, 3648, 0, [896] * 8) == d_ar
    # an explicit tile width wins; so does another SM count
    h2 = Host(host.lib, sm=152)
    B.gemm_shard_plan_set_option(h2.plan, B.GSR_OPT_BLOCK_N, 256)
    assert h2.describe(B.MODE_AG, 0, 3648, 7168, [256] * 8)["block_n"] == 256
    assert host.describe(B.MODE_AG, 0, 3648, 7168, [256] * 8)["block_n"] == 256   # 148 SMs


def test_split_tail_where_the_partial_wave_is_at_most_half(lib):
    """On 152 SMs (76 pairs): AR M = 1000 (112 tiles: one wave plus 36) cuts
    each of the 36 tail tiles into two k-pieces on 72 workers; the headline
    shapes (partial waves of 8 and 12 tiles) keep the stream-K tail."""
    h = Host(lib, sm=152, max_M=34816)
    d = h.describe(B.MODE_AR, 1000, 7168, 0, [896] * 8)
    assert (d["schedule"], d["split"], d["tiles"], d["dp_tiles"], d["ctas"]) == (4, 2, 112, 76, 152)
    assert h.describe(B.MODE_RS, 1000, 7168, 0, [896] * 8) == d
    assert h.describe(B.MODE_AG, 0, 6288, 7168, [4096] * 8)["schedule"] == 2
    assert h.describe(B.MODE_AR, 32768, 7168, 0, [896] * 8)["schedule"] == 2
    # whole waves need no tail at all
    assert h.describe(B.MODE_AR, 2048, 4864, 0, [896] * 8)["sk_iters"] == 0


def test_nearly_full_partial_wave_runs_whole_tiles(lib):
    """On 152 SMs (76 pairs): a partial last wave of at least 70 % of the
    workers runs as whole tiles (AR M = 4096: 448 tiles, 68 in the last wave;
    AG KDA M = 3072: 300 tiles, 72; AG MLA M = 3584 in 448-row shards: 210
    tiles, 58), a fuller share-out stays stream-K (AG KDA M = 2048: 48 of 76),
    and an explicit schedule still gets stream-K."""
    h = Host(lib, sm=152, max_M=34816)
    d = h.describe(B.MODE_AR, 4096, 7168, 0, [896] * 8)
    assert (d["tiles"], d["dp_tiles"], d["sk_iters"], d["ctas"]) == (448, 448, 0, 152)
    d = h.describe(B.MODE_AG, 0, 6288, 7168, [384] * 8)
    assert (d["tiles"], d["dp_tiles"], d["sk_iters"]) == (300, 300, 0)
    d = h.describe(B.MODE_AG, 0, 3648, 7168, [448] * 8)
    assert (d["tiles"], d["dp_tiles"], d["sk_iters"]) == (210, 210, 0)
    d = h.describe(B.MODE_AG, 0, 6288, 7168, [256] * 8)
    assert d["schedule"] == 2 and d["sk_iters"] == 48 * 112
    h3 = Host(lib, sm=152, max_M=34816)
    B.gemm_shard_plan_set_option(h3.plan, B.GSR_OPT_SCHEDULE, 3)
    assert h3.describe(B.MODE_AR, 4096, 7168, 0, [896] * 8)["sk_iters"] == 68 * 112


@pytest.mark.parametrize("sm", [16, 148, 152])
@pytest.mark.parametrize("schedule", [0, 2, 3, 4, 5])
def test_workspace_and_schedule_invariants_over_shapes(lib, sm, schedule):
    """Every configuration, heuristic or forced, fits the plan's workspace; a
    split tail hands out at most one piece per worker, every piece at least
    one k-block; whole-tile runs need no partial slots."""
    h = Host(lib, sm=sm, max_M=34816)
    if schedule:
        B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SCHEDULE, schedule)
    rng = np.random.default_rng(100 * sm + schedule)
    shapes = [(1000, 7168, [896] * 8), (4096, 7168, [896] * 8), (2048, 3648, [896] * 8),
              (32768, 7168, [896] * 8), (3584, 6288, [7168])]
    for _ in range(40):
        M = int(rng.integers(1, 34817))
        N = int(rng.integers(1, 1025)) * 8
        R = int(rng.integers(1, 17))
        shapes.append((M, N, [int(rng.integers(1, 129)) * 8 for _ in range(R)]))
    for M, N, K_r in shapes:
        d = h.describe(B.MODE_AR, M, N, 0, K_r)
        assert d["workspace_bytes"] <= h.ws_bytes, (M, N, K_r)
        assert 1 <= d["ctas"] <= sm
        # RS rows equal AR rows bit for bit only because the configuration
        # never depends on the mode.
        assert h.describe(B.MODE_RS, M, N, 0, K_r) == d, (M, N, K_r)
        kb = sum((k + 63) // 64 for k in K_r)
        workers = d["ctas"] // d["cta_group"]
        if d["schedule"] == 4:
            tail = d["tiles"] - d["dp_tiles"]
            assert 0 < tail * d["split"] <= workers and 1 <= d["split"] <= min(3, kb), (M, N, K_r, d)
        if d["schedule"] in (2, 4) and d["dp_tiles"] == d["tiles"]:
            assert d["sk_iters"] == 0


@pytest.mark.parametrize("sm", [16, 148, 152])
@pytest.mark.parametrize("opts", [{}, {"cta_group": 4}, {"block_n": 192}, {"schedule": 5}],
                         ids=["heuristic", "cta_group4", "block_n192", "split_tail"])
def test_ag_workspace_and_grid_invariants_over_shapes(lib, sm, opts):
    """AG over random shard sizes (empty shards included), N and K: every
    configuration fits the plan's workspace, the grid fits the SMs in whole
    clusters, and the call reaches the launch point."""
    h = Host(lib, sm=sm, max_M=34816)
    for name, value in opts.items():
        B.gemm_shard_plan_set_option(h.plan, getattr(B, f"GSR_OPT_{name.upper()}"), value)
    rng = np.random.default_rng(sm + 7 * len(opts))
    shapes = [([4096] * 8, 6288, 7168), ([448] * 8, 3648, 7168), ([0, 0, 130], 136, 64)]
    for _ in range(40):
        R = int(rng.integers(1, 17))
        M_r = [int(rng.integers(0, 4097)) if rng.random() > 0.2 else 0 for _ in range(R)]
        if sum(M_r) > 34816 or sum(M_r) == 0:
            M_r = [int(rng.integers(1, 2049))]
        shapes.append((M_r, int(rng.integers(1, 1025)) * 8, int(rng.integers(1, 1025)) * 8))
    for M_r, N, K in shapes:
        d = h.describe(B.MODE_AG, 0, N, K, M_r)
        assert d["workspace_bytes"] <= h.ws_bytes, (M_r, N, K, d)
        assert 1 <= d["ctas"] <= sm and d["ctas"] % d["cta_group"] == 0, (M_r, N, K, d)
        assert d["dp_tiles"] <= d["tiles"] and d["sk_iters"] >= 0, (M_r, N, K, d)
        assert h.ag(N, K, M_r) == B.GSR_ERR_UNSUPPORTED, B.gsr_last_error_string()


def _build_in_child(q):
    from tensor_gemm_reduction_gb300 import build as b
    import oracle as o
    q.put((b.build(), o.build()))


def test_concurrent_builds_take_turns(lib):
    """Ranks that start together all call build(): with the library stale, they
    must take turns and leave one loadable library, not interleaved objects."""
    import multiprocessing as mp
    import oracle
    for src, built in ((os.path.join(ROOT, "include", "gsr.h"), B.library_path()),
                       (os.path.join(ROOT, "oracle", "gsr_oracle.c"), oracle.build())):
        st = os.stat(src)
        os.utime(src, (st.st_atime, max(st.st_mtime, os.path.getmtime(built)) + 1))
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_build_in_child, args=(q,)) for _ in range(3)]
    for p in procs:
        p.start()
    paths = [q.get(timeout=600) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert len(set(paths)) == 1
    assert not gbuild._stale() and oracle._fresh()
    again = ctypes.CDLL(paths[0][0])
    for n in header_functions():
        assert hasattr(again, n)
    for built in paths[0]:
        assert [f for f in os.listdir(os.path.dirname(built)) if f.endswith(".tmp")] == []


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "gsr.h"
int main(void) {
  gemm_shard_plan *p = NULL;
  if (gemm_shard_plan_create_host(&p, 152, 4096, 7168, 7168, 8) != GSR_OK) return 1;
  int64_t K_r[8] = {896, 896, 896, 896, 896, 896, 896, 896};
  gsr_config c;
  if (gemm_shard_describe(p, 0, 1000, 7168, 0, 8, K_r, &c) != GSR_OK) return 2;
  if (c.block_n != 256 || c.cta_group != 2 || c.tiles != 112) return 3;
  if (gemm_shard_workspace_size(p) < c.workspace_bytes) return 4;
  if (gemm_ar(p, 1000, 7168, 8, K_r, NULL, NULL, NULL, NULL, 0, NULL) != GSR_ERR_INVALID_VALUE)
    return 5;
  if (strstr(gsr_last_error_string(), "NULL") == NULL) return 6;
  if (gemm_shard_plan_destroy(p) != GSR_OK) return 7;
  return 0;
}
"""


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_is_plain_c_and_cxx(lang):
    import subprocess
    std = "-std=c99" if lang == "c" else "-std=c++17"
    r = subprocess.run(["gcc" if lang == "c" else "g++", std, "-Wall", "-Wextra", "-pedantic",
                        "-Werror", "-fsyntax-only", "-x", lang,
                        os.path.join(ROOT, "include", "gsr.h")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_a_plain_c_program_links_and_calls_the_library(lib, tmp_path):
    import subprocess
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(B.library_path())
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-lgsr", f"-Wl,-rpath,{libdir}", "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)


LOG_CLIENT = r"""
import ctypes, sys
sys.path.insert(0, sys.argv[1])
from tensor_gemm_reduction_gb300 import binding as B
lib = B.load_library()
p = B.gemm_shard_plan_create_host(152, 32768, 8192, 8192, 16)
ws = B.gemm_shard_workspace_size(p)
k = (ctypes.c_int64 * 8)(*([896] * 8))
ptr = lambda n, base: (ctypes.c_void_p * n)(*[base + 0x100000 * i for i in range(n)])
lib.gemm_ar(p.handle, 1000, 7168, 8, k, ptr(8, 0x1000000), ptr(8, 0x9000000), ctypes.c_void_p(0x10000),
            ctypes.c_void_p(0x20000000), ws, None)
lib.gemm_ar(p.handle, 128, 7168, 8, k, ptr(8, 0x1000000), ptr(8, 0x9000000), ctypes.c_void_p(0x10000),
            ctypes.c_void_p(0x20000000), ws, None)
m = (ctypes.c_int64 * 8)(*([4096] * 8))
lib.gemm_ag(p.handle, 6288, 7168, 8, m, ptr(8, 0x1000000), ctypes.c_void_p(0x9000000),
            ctypes.c_void_p(0x10000), ctypes.c_void_p(0x20000000), ws, None)
lib.gemm_ar(p.handle, 0, 7168, 8, k, ptr(8, 0x1000000), ptr(8, 0x9000000), ctypes.c_void_p(0x10000),
            ctypes.c_void_p(0x20000000), ws, None)
"""


@pytest.mark.parametrize("value,expect", [("1", 3), ("0", 0), (None, 0)])
def test_config_logging_env(lib, value, expect):
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items() if k != "GSR_LOG_CONFIG"}
    if value is not None:
        env["GSR_LOG_CONFIG"] = value
    r = subprocess.run([sys.executable, "-c", LOG_CLIENT, ROOT], capture_output=True, text=True,
                       env=env, timeout=120)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stderr.splitlines() if l.startswith("gsr: ")]
    assert len(lines) == expect, r.stderr
    if expect:
        assert lines[0].startswith("gsr: ar M=1000 N=7168 R=8 kernel=main block_n=256 cta_group=2 "
                                   "schedule=split_tail split=2 tiles=112")
        assert "kernel=small" in lines[1] and "schedule=small_m" in lines[1]
        assert lines[2].startswith("gsr: ag M=32768 N=6288 R=8 kernel=main") and "stream_k" in lines[2]


def test_last_error_string_is_per_thread(lib, host):
    """gsr_last_error_string is thread-local: another thread's failure in between
    does not replace this thread's message."""
    import threading
    barrier = threading.Barrier(2)
    seen = {}

    def worker(name, call):
        assert call() == B.GSR_ERR_INVALID_VALUE
        barrier.wait()           # both threads have failed, each its own way
        barrier.wait()
        seen[name] = B.gsr_last_error_string()

    t1 = threading.Thread(target=worker, args=("m", lambda: host.ar(-1, 256, [128])))
    t2 = threading.Thread(target=worker, args=("r", lambda: host.ar(16, 256, [8] * 17)))
    t1.start(); t2.start(); t1.join(); t2.join()
    assert "M must be" in seen["m"] and "R=17" in seen["r"]


@pytest.mark.parametrize("name,good,bad", [
    ("SPLIT_K", [0, 1, 16], [-1, 17]),
    ("BLOCK_N", [0, 128, 192, 256], [64, 200, 512]),
    ("TIMEOUT_NS", [0, 1, 10**12], [-1]),
    ("MAX_CTAS", [0, 1, 2**31 - 1], [-1, 2**31]),
    ("RASTER_M", [0, 1, 64], [-1, 65]),
    ("RASTER_N", [0, 1, 64], [-1, 65]),
    ("L2_HINTS", [0, 3], [-1, 4]),
    ("CTA_GROUP", [0, 1, 2, 4], [-1, 3, 5]),
    ("SCHEDULE", [0, 5], [-1, 6]),
    ("SMALL_M", [0, 2], [-1, 3]),
    ("SMALL_TILE_ROWS", [0, 16, 256], [-16, 8, 136, 272]),
    ("SMALL_KBLOCKS", [0, 1, 3, 4], [-1, 5, 8]),
])
def test_every_option_checks_its_range(host, name, good, bad):
    opt = getattr(B, "GSR_OPT_" + name)
    for v in good:
        assert host.lib.gemm_shard_plan_set_option(host.plan.handle, opt, v) == B.GSR_OK, (name, v)
    for v in bad:
        assert host.lib.gemm_shard_plan_set_option(host.plan.handle, opt, v) == \
            B.GSR_ERR_INVALID_VALUE, (name, v)


def test_unknown_option_is_rejected(host):
    assert host.lib.gemm_shard_plan_set_option(host.plan.handle, 99, 1) == B.GSR_ERR_INVALID_VALUE
    assert "unknown option" in B.gsr_last_error_string()


def _noalloc(h, M, N, K_r):
    R = len(K_r)
    return h.lib.gemm_ar_noalloc(h.plan.handle, M, N, R, _arr(ctypes.c_int64, K_r),
                                 _arr(ctypes.c_void_p, [0x100000 * (r + 1) for r in range(R)]),
                                 _arr(ctypes.c_void_p, [0x8000000 + 0x100000 * r for r in range(R)]),
                                 ctypes.c_void_p(0x10000), None)


def test_noalloc_fits_the_builtin_scratch_or_says_why(lib):
    h = Host(lib, sm=152)
    # Every heuristic shape fits (the uniform schedule where the plan's own
    # configuration would need more than 24 MiB): valid up to the launch point.
    for M in (0, 1, 128, 1000, 4096, 32768):
        assert _noalloc(h, M, 7168, [896] * 8) == (B.GSR_OK if M == 0 else B.GSR_ERR_UNSUPPORTED)
        if M:
            assert "arguments are valid" in B.gsr_last_error_string()
    # A forced 16-way split on 3584 tiles needs far more: rejected before any launch.
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_SPLIT_K, 16)
    assert _noalloc(h, 32768, 7168, [896] * 8) == B.GSR_ERR_WORKSPACE
    assert "built-in scratch" in B.gsr_last_error_string()
    # Argument errors come first, as for gemm_ar.
    assert _noalloc(h, 16, 252, [128]) == B.GSR_ERR_INVALID_VALUE


def test_noalloc_keeps_a_forced_schedule(lib):
    """M=2560, N=7168: the heuristic's stream-K tail needs more than the
    built-in 24 MiB, so an unforced plan falls back to the uniform schedule,
    but a plan that forces stream-K (schedule 2, or 4: stream-K with the
    whole tiles first) is rejected instead of silently summing in another
    order."""
    h = Host(lib, sm=152)
    d = B.gemm_shard_describe(h.plan, B.MODE_AR, 2560, 7168, 0, [896] * 8)
    assert d["schedule"] == 2 and d["workspace_bytes"] > 24 << 20
    assert _noalloc(h, 2560, 7168, [896] * 8) == B.GSR_ERR_UNSUPPORTED   # valid: falls back
    for sched in (2, 4):
        f = Host(lib, sm=152)
        B.gemm_shard_plan_set_option(f.plan, B.GSR_OPT_SCHEDULE, sched)
        d = B.gemm_shard_describe(f.plan, B.MODE_AR, 2560, 7168, 0, [896] * 8)
        assert d["workspace_bytes"] > 24 << 20
        assert _noalloc(f, 2560, 7168, [896] * 8) == B.GSR_ERR_WORKSPACE, sched
        assert "built-in scratch" in B.gsr_last_error_string()


def test_noalloc_status_query_on_a_host_plan(lib):
    h = Host(lib, sm=152)
    assert lib.gemm_ar_noalloc_check_status(h.plan.handle, None) == B.GSR_ERR_UNSUPPORTED
    assert lib.gemm_ar_noalloc_check_status(None, None) == B.GSR_ERR_INVALID_VALUE


def test_replicated_ar_validation(host):
    lib = host.lib

    def call(y, M=16):
        K = _arr(ctypes.c_int64, [128, 128])
        X = _arr(ctypes.c_void_p, [0x100000, 0x200000])
        W = _arr(ctypes.c_void_p, [0x300000, 0x400000])
        Y = None if y is None else _arr(ctypes.c_void_p, y)
        return lib.gemm_ar_replicated(host.plan.handle, M, 256, 2, K, X, W, Y,
                                      ctypes.c_void_p(0x20000000), host.ws_bytes, None)

    assert call([0x10000, 0x20000]) == B.GSR_ERR_UNSUPPORTED           # valid: stops at the launch
    assert call(None) == B.GSR_ERR_INVALID_VALUE
    assert call([0x10000, 0]) == B.GSR_ERR_INVALID_VALUE
    assert call([0x10000, 0x20008]) == B.GSR_ERR_INVALID_VALUE
    assert "16-byte" in B.gsr_last_error_string()
    assert call([0, 0], M=0) == B.GSR_OK                                # nothing to write


def test_workspace_init_checks(host):
    lib = host.lib
    need = host.ws_bytes
    assert lib.gemm_shard_workspace_init(host.plan.handle, None, need, None) == B.GSR_ERR_WORKSPACE
    assert lib.gemm_shard_workspace_init(host.plan.handle, ctypes.c_void_p(0x20000010), need,
                                         None) == B.GSR_ERR_WORKSPACE
    assert lib.gemm_shard_workspace_init(host.plan.handle, ctypes.c_void_p(0x20000000), 64,
                                         None) == B.GSR_ERR_WORKSPACE
    assert "too small" in B.gsr_last_error_string()
    assert lib.gemm_shard_workspace_init(host.plan.handle, ctypes.c_void_p(0x20000000), need,
                                         None) == B.GSR_ERR_UNSUPPORTED
    assert lib.gemm_shard_workspace_init(None, ctypes.c_void_p(0x20000000), need, None) == \
        B.GSR_ERR_INVALID_VALUE


def test_two_pairs_per_cluster_on_request(lib):
    """GSR_OPT_CTA_GROUP = 4: clusters of two CTA pairs, each cluster on two
    256-row tiles of the same columns (half as many work tiles), a grid of
    whole clusters; the configuration still does not depend on the mode, and
    every schedule fits the plan's workspace."""
    h = Host(lib, sm=152)
    B.gemm_shard_plan_set_option(h.plan, B.GSR_OPT_CTA_GROUP, 4)
    pairs = Host(lib, sm=152)
    B.gemm_shard_plan_set_option(pairs.plan, B.GSR_OPT_CTA_GROUP, 2)
    for M in (300, 1000, 4096, 32768):
        d = h.describe(B.MODE_AR, M, 7168, 0, [896] * 8)
        d2 = pairs.describe(B.MODE_AR, M, 7168, 0, [896] * 8)
        assert d["cta_group"] == 4 and d["ctas"] % 4 == 0 and d["ctas"] <= 152
        assert d["tiles"] == -(-(-(-M // 256)) // 2) * 28 and d2["tiles"] == -(-M // 256) * 28
        assert d == h.describe(B.MODE_RS, M, 7168, 0, [896] * 8)
        assert d["workspace_bytes"] <= h.ws_bytes
    d = h.describe(B.MODE_AG, 0, 6288, 7168, [4096] * 8)
    assert d["cta_group"] == 4 and d["tiles"] == 64 * 25
    # too few SMs for a cluster of four: CTA pairs
    small = Host(lib, sm=2)
    B.gemm_shard_plan_set_option(small.plan, B.GSR_OPT_CTA_GROUP, 4)
    assert small.describe(B.MODE_AR, 1000, 7168, 0, [896] * 8)["cta_group"] == 2
