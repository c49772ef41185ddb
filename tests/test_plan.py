"""The block GEMM's launch plan (host logic; no GPU needed).

Pins the decisions the measured results rest on: swap-AB tiles by token
count, the split-K choice, split-K inside clusters of two, 64-token swap-AB
tiles for mid-sized M where the 128x256 tiles would leave most SMs idle, and
the alternating MMA issuers; and checks the plan's invariants over a grid of
shapes."""
import itertools
import math

import pytest

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import binding

SMS = 152   # GB300


def plan(M, N, K, bk, sms=SMS):
    return sgq.sgq_gemm_plan(M, N, K, bk, sms)


def test_decode_block32_swap_ab_two_splits():
    p = plan(16, 7168, 2048, 32)
    assert p == {"swap": 1, "bn": 16, "splits": 2, "items": 112, "grid": 112, "alt": 0, "ck": 0, "pair": 0}


@pytest.mark.parametrize("M,bn", [(1, 16), (16, 16), (17, 32), (32, 32), (33, 64), (64, 64)])
def test_swap_ab_tile_width_follows_tokens(M, bn):
    p = plan(M, 7168, 2048, 32)
    assert p["swap"] == 1 and p["bn"] == bn


def test_cluster_split_k_only_with_several_items_per_cta():
    p = plan(16, 24576, 1536, 128)
    assert p["swap"] == 1 and p["splits"] == 2 and p["items"] > p["grid"] and p["ck"] == 1
    # one item per CTA: the global workspace path
    assert plan(16, 7168, 2048, 128)["ck"] == 0


def test_narrow_n_splits_k_across_the_grid():
    p = plan(1, 1536, 7168, 128)
    assert p["swap"] == 1 and p["splits"] == 12 and p["items"] == 144 and p["grid"] == 144


def test_mid_m_swap_ab_where_wide_tiles_leave_sms_idle():
    # 128 x 1536 x 7168: six 128x256 tiles for 152 SMs
    p = plan(128, 1536, 7168, 128)
    assert p["swap"] == 1 and p["bn"] == 64 and p["splits"] == 6
    # enough wide tiles: they stay
    assert plan(2048, 1536, 7168, 128)["swap"] == 0
    assert plan(128, 24576, 1536, 128)["swap"] == 0
    # above 1024 tokens the wide tiles always run
    assert plan(1025, 1536, 7168, 32)["swap"] == 0


def test_wide_tiles_one_split_alternating_issuers_for_long_k_block128():
    p = plan(4096, 7168, 7168, 128)
    assert p["swap"] == 0 and p["bn"] == 256 and p["splits"] == 1 and p["alt"] == 1 and p["pair"] == 0
    assert plan(4096, 4096, 7168, 32)["alt"] == 0     # [*,32]: one issuer, two scale warps
    assert plan(8192, 24576, 1536, 128)["alt"] == 0   # K < 4096


SHAPES = list(itertools.product([1, 5, 16, 33, 64, 65, 128, 300, 512, 1024, 1025, 4096],
                                [8, 264, 1536, 7168, 24576], [32, 96, 2048, 7168], [32, 128]))


@pytest.mark.parametrize("M,N,K,bk", [s for s in SHAPES if s[2] % s[3] == 0])
def test_plan_invariants(M, N, K, bk):
    p = plan(M, N, K, bk)
    if p["swap"]:
        tiles = math.ceil(N / 128) * math.ceil(M / p["bn"])
        assert p["bn"] in (16, 32, 64)
        if M <= 64:
            assert p["bn"] == (16 if M <= 16 else 32 if M <= 32 else 64)
        else:
            assert M <= 1024 and p["bn"] == 64
    else:
        tiles = math.ceil(M / 128) * math.ceil(N / 256)
        assert M > 64 and p["bn"] == 256 and p["splits"] == 1
    kb = math.ceil(K / 128)
    s = p["splits"]
    assert 1 <= s <= min(kb, 32)
    assert math.ceil(kb / math.ceil(kb / s)) == s          # every split non-empty
    assert p["items"] == tiles * s
    assert p["grid"] == min(p["items"], SMS)
    if p["ck"]:
        assert p["swap"] and s == 2 and p["bn"] <= 32 and p["items"] > p["grid"]
    if p["alt"]:
        assert not p["swap"] and bk == 128 and kb >= 32


def test_grid_follows_the_sm_count():
    assert plan(4096, 7168, 7168, 128, sms=76)["grid"] == 76
    # more SMs, more K splits, still one wave
    p = plan(16, 7168, 2048, 32, sms=1000)
    assert p["splits"] > 2 and p["items"] <= 1000 and p["grid"] == p["items"]


def test_plan_rejects_bad_arguments():
    lib = binding.load_library()
    import ctypes
    out = (ctypes.c_int32 * 8)()
    ptr = ctypes.cast(out, ctypes.c_void_p)
    assert lib.sgq_gemm_plan(16, 7168, 2048, 32, 152, None) == binding.SGQ_ERR_INVALID_ARG
    assert lib.sgq_gemm_plan(0, 7168, 2048, 32, 152, ptr) == binding.SGQ_ERR_INVALID_ARG
    assert lib.sgq_gemm_plan(16, 7168, 2048, 64, 152, ptr) == binding.SGQ_ERR_INVALID_ARG
    assert lib.sgq_gemm_plan(16, 7168, 2048, 32, 0, ptr) == binding.SGQ_ERR_INVALID_ARG
    assert lib.sgq_gemm_plan(16, 7168, 2048, 32, 152, ptr) == 0
