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


# ------------------------------------------- two-accumulator tiles (power-of-two scales)

def plan2(M, N, K, bk, e8=False, sms=SMS):
    return sgq.sgq_gemm_plan_pow2(M, N, K, bk, sms, e8)


def test_pow2_plan_widths_and_pairs():
    """Tile widths by rounds over the grid: 4096 x 7168 x 7168 on CTA pairs
    takes 192-wide tiles (304 tiles, exactly four rounds of 76 pairs, where
    224 would make 256 tiles in 3.4 rounds); 4096 x 4096 x 7168 on bytes 224
    (152 tiles, two rounds); 8192 x 24576 x 1536 single CTAs 224 wide."""
    p = plan2(4096, 7168, 7168, 128, e8=True)
    assert p == {"mode": 3, "bn": 192, "splits": 1, "items": 304, "grid": 152, "tiles": 304, "kps": 56}
    assert plan2(4096, 7168, 7168, 128) == p                       # fp32 [*,128] scales: the same plan
    p = plan2(4096, 4096, 7168, 32, e8=True)
    assert (p["mode"], p["bn"], p["items"], p["grid"]) == (3, 224, 152, 152)
    p = plan2(8192, 24576, 1536, 32, e8=True)
    assert (p["mode"], p["bn"], p["items"], p["grid"]) == (1, 224, 3520, 152)


def test_pow2_plan_modes():
    """Single CTAs for fp32 [*,32] scales and for short K, K split over CTAs
    at mid M with few tiles, and the 128-row kernel for decode-sized M."""
    assert plan2(4096, 4096, 7168, 32)["mode"] == 1              # fp32 [*,32]: no pairs
    assert plan2(8192, 24576, 1536, 128, e8=True)["mode"] == 1   # K < 4096
    p = plan2(1024, 1536, 7168, 128)
    assert p["mode"] == 2 and p["splits"] == 4 and p["items"] == p["tiles"] * 4
    assert plan2(16, 7168, 2048, 32, e8=True)["mode"] == 0
    assert plan2(64, 24576, 7168, 128)["mode"] == 0


POW2_SHAPES = list(itertools.product([65, 700, 1024, 2100, 4096, 6000, 8192, 16384], [448, 1536, 3000, 7168, 24576],
                                     [512, 1536, 4096, 5120, 7168], [32, 128], [False, True]))


@pytest.mark.parametrize("M,N,K,bk,e8", POW2_SHAPES)
def test_pow2_plan_invariants(M, N, K, bk, e8):
    p = plan2(M, N, K, bk, e8)
    if p["mode"] == 0:
        return
    rows = 512 if p["mode"] == 3 else 256
    units = SMS // 2 if p["mode"] == 3 else SMS
    kst = K // 128
    assert p["bn"] in (192, 224)
    assert p["tiles"] == math.ceil(M / rows) * math.ceil(N / p["bn"])
    s, kps = p["splits"], p["kps"]
    assert 1 <= s <= 16 and kps == math.ceil(kst / s) and (s - 1) * kps < kst   # every split non-empty
    if p["mode"] == 2:
        assert p["items"] == p["tiles"] * s <= units   # one item per CTA
    else:
        assert s == 1 and p["items"] == p["tiles"]
    assert p["grid"] == min(p["items"], units) * (2 if p["mode"] == 3 else 1)


def test_pow2_plan_rejects_bad_arguments():
    lib = binding.load_library()
    import ctypes
    out = (ctypes.c_int32 * 8)()
    ptr = ctypes.cast(out, ctypes.c_void_p)
    assert lib.sgq_gemm_plan_pow2(4096, 7168, 7168, 128, 152, 0, None) == binding.SGQ_ERR_INVALID_ARG
    assert lib.sgq_gemm_plan_pow2(4096, 7168, 7168, 64, 152, 0, ptr) == binding.SGQ_ERR_INVALID_ARG
    assert lib.sgq_gemm_plan_pow2(4096, 7168, 7168, 128, 1, 0, ptr) == binding.SGQ_ERR_INVALID_ARG
    assert lib.sgq_gemm_plan_pow2(4096, 7168, 7168, 128, 152, 2, ptr) == binding.SGQ_ERR_INVALID_ARG
    assert lib.sgq_gemm_plan_pow2(4096, 7168, 7168, 128, 152, 1, ptr) == 0 and out[0] == 3
