"""GPU block-scaled GEMM vs the CPU oracle under the stated tolerance:
||D - Dref||_F / ||Dref||_F <= 5e-3 and |D - Dref| <= 2^-7 |Dref| + 1e-4 sum_k |a||w|
(D read as fp64; Dref, the bound: fp64 oracle on the same codes and scales)."""
import functools

import numpy as np
import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import synth

import oracle
from common import check_gemm, tile_rows

pytestmark = pytest.mark.gpu

FLAGS = [sgq.SGQ_GEMM_DEFAULT, sgq.SGQ_GEMM_FORCE_PROMOTE]


@functools.lru_cache(maxsize=8)
def weights(N, K, bn, bk, ue, seed=0):
    w = synth.weight(N, K, seed)
    wq, ws = oracle.quant_weight_block(w, bn, bk, ue)
    return wq, ws


def run_gpu(aq, a_s, wq, ws, bn, bk, flags=0):
    d = sgq.fp8_block_gemm(torch.from_numpy(aq).cuda(), torch.from_numpy(a_s).cuda(),
                           torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda(), bn, bk, flags=flags)
    assert sgq.sgq_device_status() == 0
    return d


def case_check(c, flags_list=(0,), rows=None):
    """Quantise x with the oracle, run the GPU GEMM on the full problem, compare
    (all rows, or a sample of rows the oracle computes one by one)."""
    x = c.x()
    aq, a_s = oracle.quant_token_group(x, c.group, c.ue8m0)
    wq, ws = weights(c.N, c.K, c.blk_n, c.blk_k, c.ue8m0, c.seed)
    r = np.arange(c.M) if rows is None else rows
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, c.blk_n, c.blk_k)
    for fl in flags_list:
        d = run_gpu(aq, a_s, wq, ws, c.blk_n, c.blk_k, fl)
        check_gemm(d[torch.from_numpy(r).cuda()], dref, bound, f"{c.name} flags={fl}")


def test_tiny_fp32_scales():
    c = synth.WORKLOADS["tiny"][0]
    case_check(c, FLAGS)


@pytest.mark.parametrize("idx", range(4))
def test_decode_block32(idx):
    case_check(synth.WORKLOADS["decode_block32"][idx], FLAGS)


def test_prefill_block128_every_tile():
    """Full size; one row of every 64-row block (every M-tile of the wide
    plan) is compared over all N columns."""
    c = synth.WORKLOADS["prefill_block128"][0]
    case_check(c, FLAGS, rows=tile_rows(c.M, seed=1))


def test_prefill_block32_every_tile():
    c = synth.WORKLOADS["prefill_block32"][0]
    case_check(c, FLAGS, rows=tile_rows(c.M, seed=2))


SWEEP = synth.WORKLOADS["sweep"]


@pytest.mark.parametrize("idx", range(len(SWEEP)), ids=[c.name for c in SWEEP])
def test_sweep(idx):
    c = SWEEP[idx]
    rows = None if c.M <= 128 else tile_rows(c.M, seed=idx)
    case_check(c, (0,), rows=rows)


RAGGED = [(1, 8, 32, 32, 32), (3, 136, 96, 32, 32), (17, 264, 160, 32, 32), (65, 200, 256, 128, 128),
          (129, 136, 384, 128, 128), (200, 520, 2080, 32, 32), (64, 1032, 128, 128, 32),
          (300, 72, 640, 32, 128), (33, 256, 4096, 128, 128)]


@pytest.mark.parametrize("M,N,K,bn,bk", RAGGED)
@pytest.mark.parametrize("pow2", [True, False])
def test_ragged_shapes(M, N, K, bn, bk, pow2):
    c = synth.Case("ragged", M, N, K, bn, bk, pow2, seed=M + N + K)
    x = c.x()
    w = c.w()
    aq, a_s = oracle.quant_token_group(x, bk, pow2)
    wq, ws = oracle.quant_weight_block(w, bn, bk, pow2)
    dref, bound = oracle.gemm(aq, a_s, wq, ws, bn, bk)
    for fl in FLAGS:
        check_gemm(run_gpu(aq, a_s, wq, ws, bn, bk, fl), dref, bound, f"M={M} N={N} K={K} fl={fl}")


@pytest.mark.parametrize("M", [5, 200])
@pytest.mark.parametrize("bk", [32, 128])
def test_mixed_pow2_and_fp32_scales(M, bk):
    """Some K stages all power-of-two, others not: the kernel switches between
    the block-scale MMA and promotion inside one tile."""
    N, K, bn = 264, 1024, 128
    x = synth.activation(M, K, seed=11)
    w = synth.weight(N, K, seed=11)
    aq, a_s = oracle.quant_token_group(x, bk, True)
    wq, ws = oracle.quant_weight_block(w, bn, bk, True)
    rng = np.random.default_rng(M + bk)
    kcols = a_s.shape[1]
    stage_cols = 128 // bk
    for st in range(K // 128):
        if rng.random() < 0.5:   # make this stage's weight scales non-power-of-two
            ws[:, st * stage_cols:(st + 1) * stage_cols] *= np.float32(1.3)
    ws[0, kcols - 1] = np.float32(0.7) * ws[0, kcols - 1]   # last stage mixed too
    dref, bound = oracle.gemm(aq, a_s, wq, ws, bn, bk)
    check_gemm(run_gpu(aq, a_s, wq, ws, bn, bk), dref, bound, f"mixed M={M} bk={bk}")


@pytest.mark.parametrize("rows", [(130, 140), (3, 9), (250, 256)])
@pytest.mark.parametrize("bk", [32, 128])
def test_pair_tile_one_half_not_pow2(rows, bk):
    """Activation scales that are not powers of two in only part of the rows
    of a wide tile (rows 128-255 of the first 256-row span, or 0-127): the
    stage must take the promotion path for the rows that need it.  With CTA
    pairs (SGQ_PAIR=1, tested below in a child process) each CTA of the pair
    holds one half of a 256-row tile, and one half's non-power-of-two scales
    must send the whole tile's stage to the promotion path, for both halves."""
    M, N, K, bn = 300, 520, 1024, 128
    x = synth.activation(M, K, seed=5)
    w = synth.weight(N, K, seed=5)
    aq, a_s = oracle.quant_token_group(x, bk, True)
    wq, ws = oracle.quant_weight_block(w, bn, bk, True)
    stage_cols = 128 // bk
    for st in (1, 4, 5):
        a_s[rows[0]:rows[1], st * stage_cols:(st + 1) * stage_cols] *= np.float32(1.3)
    dref, bound = oracle.gemm(aq, a_s, wq, ws, bn, bk)
    check_gemm(run_gpu(aq, a_s, wq, ws, bn, bk), dref, bound, f"half rows={rows} bk={bk}")


@pytest.mark.parametrize("M", [1, 16, 64, 128, 4096])
def test_deterministic(M):
    """Split-K sums partials in a fixed order: repeated calls are bitwise equal."""
    N, K = 7168, 2048
    x = synth.activation(M, K, seed=3)
    aq, a_s = oracle.quant_token_group(x, 32, True)
    wq, ws = weights(N, K, 32, 32, True)
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
    d0 = sgq.fp8_block_gemm(*args, 32, 32)
    for _ in range(3):
        d1 = sgq.fp8_block_gemm(*args, 32, 32)
        assert torch.equal(d0, d1)


def test_linear_end_to_end_on_device():
    """Quant kernel feeding the GEMM on one stream (the programmatic-launch pair)."""
    c = synth.WORKLOADS["decode_block32"][2]
    x = c.x()
    wq, ws = weights(c.N, c.K, c.blk_n, c.blk_k, True)
    d = sgq.w8a8_linear(x.cuda(), torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda(), 32, 32, True)
    aq, a_s = oracle.quant_token_group(x, 32, True)
    dref, bound = oracle.gemm(aq, a_s, wq, ws, 32, 32)
    check_gemm(d, dref, bound, "w8a8_linear")
    assert sgq.sgq_device_status() == 0


def test_m_zero_is_noop():
    d = sgq.fp8_block_gemm(torch.empty((0, 256), dtype=torch.uint8, device="cuda"),
                           torch.empty((0, 2), dtype=torch.float32, device="cuda"),
                           torch.zeros((128, 256), dtype=torch.uint8, device="cuda"),
                           torch.ones((1, 2), dtype=torch.float32, device="cuda"), 128, 128)
    assert d.shape == (0, 128)


ISSUE = [(300, 520, 1024, 128, 128), (129, 136, 384, 128, 128), (200, 520, 2080, 32, 32),
         (257, 1032, 4128, 128, 32), (1000, 264, 8192, 32, 128), (300, 520, 2048, 32, 32),
         (257, 1032, 4096, 128, 32)]


@pytest.mark.parametrize("M,N,K,bn,bk", ISSUE)
@pytest.mark.parametrize("scales", ["pow2", "fp32", "mixed"])
def test_alternating_issuers_bit_identical(M, N, K, bn, bk, scales):
    """Wide tiles issued by two alternating MMA warps give the same bits as one
    issuer (the same MMA sequence into the one accumulator), and match the
    oracle; with power-of-two, fp32 and mixed scales (promotion segments
    closed by either warp), ragged M, N and K."""
    x = synth.activation(M, K, seed=M + K)
    w = synth.weight(N, K, seed=N + K)
    aq, a_s = oracle.quant_token_group(x, bk, scales != "fp32")
    wq, ws = oracle.quant_weight_block(w, bn, bk, scales != "fp32")
    if scales == "mixed":
        stage_cols = 128 // bk
        rng = np.random.default_rng(M + N)
        for st in range((K + 127) // 128):
            if rng.random() < 0.4:
                ws[:, st * stage_cols:(st + 1) * stage_cols] *= np.float32(1.3)
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
    d_alt = sgq.fp8_block_gemm(*args, bn, bk, flags=sgq.SGQ_GEMM_ISSUE_ALT)
    d_one = sgq.fp8_block_gemm(*args, bn, bk, flags=sgq.SGQ_GEMM_ISSUE_SINGLE)
    assert sgq.sgq_device_status() == 0
    assert torch.equal(d_alt, d_one)
    r = tile_rows(M, seed=M)
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, bn, bk)
    check_gemm(d_alt[torch.from_numpy(r).cuda()], dref, bound, f"alt M={M} N={N} K={K} {scales}")


def test_alternating_issuers_prefill_block128():
    """The full prefill [128,128] shape: alternating and single issuers agree bitwise."""
    c = synth.WORKLOADS["prefill_block128"][0]
    x = c.x()
    aq, a_s = oracle.quant_token_group(x, c.group, c.ue8m0)
    wq, ws = weights(c.N, c.K, c.blk_n, c.blk_k, c.ue8m0, c.seed)
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
    d_alt = sgq.fp8_block_gemm(*args, c.blk_n, c.blk_k, flags=sgq.SGQ_GEMM_ISSUE_ALT)
    d_one = sgq.fp8_block_gemm(*args, c.blk_n, c.blk_k, flags=sgq.SGQ_GEMM_ISSUE_SINGLE)
    assert sgq.sgq_device_status() == 0
    assert torch.equal(d_alt, d_one)


@pytest.mark.parametrize("M,N,K,bk", [(300, 1024, 1024, 128), (200, 512, 2048, 32)])
def test_wide_tile_store_alignment(M, N, K, bk):
    """Wide tiles store D rows with 32-byte stores when D's base and row pitch
    allow them, else with 16-byte ones: a D that starts 16 bytes past a 32-byte
    boundary must give the same result as an aligned one."""
    c = synth.Case("align", M, N, K, bk, bk, True, seed=M + K)
    aq, a_s = oracle.quant_token_group(c.x(), bk, True)
    wq, ws = weights(N, K, bk, bk, True)
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
    d0 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    buf = torch.empty(M * N + 16, dtype=torch.bfloat16, device="cuda")
    d1 = buf[8:8 + M * N].view(M, N)   # 16 bytes past the allocation's alignment
    assert d1.data_ptr() % 32 == 16
    for d in (d0, d1):
        sgq.sgq_fp8_block_gemm_ex(*args, d, M, N, K, bk, bk, sgq.SGQ_GEMM_ISSUE_SINGLE)
        assert sgq.sgq_device_status() == 0
    assert torch.equal(d0, d1)
    dref, bound = oracle.gemm(aq, a_s, wq, ws, bk, bk)
    check_gemm(d1, dref, bound, f"unaligned D M={M} N={N}")


_CK_CHILD = r"""
import sys, numpy as np, torch
import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import synth
import oracle
M, N, K, bk = (int(v) for v in sys.argv[1:5])
pow2, want_pair = sys.argv[6] == "1", int(sys.argv[7])
aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=31), bk, pow2)
wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=31), bk, bk, pow2)
if want_pair >= 0:
    assert sgq.sgq_gemm_plan(M, N, K, bk)["pair"] == want_pair
d = sgq.fp8_block_gemm(*(torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)), bk, bk)
assert sgq.sgq_device_status() == 0
np.save(sys.argv[5], d.view(torch.int16).cpu().numpy())
"""


def _child_gemm(tmp_path, name, env_extra, M, N, K, bk, pow2=True, want_pair=-1):
    """D of one GEMM computed in a fresh process whose launch plan reads the
    given environment switches (they are read once per process)."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.path.join(root, "tests"), **env_extra)
    out = str(tmp_path / f"{name}.npy")
    subprocess.run([sys.executable, "-c", _CK_CHILD, str(M), str(N), str(K), str(bk), out, "1" if pow2 else "0",
                    str(want_pair)], env=env, check=True, timeout=600, cwd=root)
    return np.load(out)


@pytest.mark.parametrize("M,N,K,bk,pow2", [(300, 520, 1024, 128, True), (300, 520, 1024, 128, False),
                                           (513, 264, 2048, 32, True), (1100, 520, 1024, 32, False),
                                           (4100, 1032, 1536, 128, True)])
def test_cta_pairs_match_oracle(tmp_path, M, N, K, bk, pow2):
    """The opt-in CTA-pair tiles (SGQ_PAIR=1: 256 x 256 tiles on two SMs,
    .cta_group::2): ragged M and N, both recipes, UE8M0 scales (block-scaled
    MMA) and fp32 scales (promotion).  SGQ_MIDSWAP=0 keeps M <= 1024 off the
    swap-AB tiles; the child process checks that its plan took pairs, and D is
    checked against the oracle here."""
    d = _child_gemm(tmp_path, "pair", {"SGQ_PAIR": "1", "SGQ_MIDSWAP": "0"}, M, N, K, bk, pow2, 1)
    aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=31), bk, pow2)
    wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=31), bk, bk, pow2)
    dref, bound = oracle.gemm(aq, a_s, wq, ws, bk, bk)
    check_gemm(torch.from_numpy(d).view(torch.bfloat16), dref, bound, f"pair M={M} N={N} K={K} bk={bk}")


@pytest.mark.parametrize("M,N,K,bk", [(16, 24576, 1536, 128), (8, 24576, 1536, 32)])
def test_cluster_split_k_bit_identical(tmp_path, M, N, K, bk):
    """Split-K inside clusters of two sums p0 + p1 as the global-workspace path
    does: D equals that path's bit for bit (the child process plans with the
    clusters off)."""
    assert sgq.sgq_gemm_plan(M, N, K, bk)["ck"] == 1
    d_global = _child_gemm(tmp_path, "global", {"SGQ_CK": "0"}, M, N, K, bk)
    aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=31), bk, True)
    wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=31), bk, bk, True)
    d = run_gpu(aq, a_s, wq, ws, bk, bk)
    assert np.array_equal(d.view(torch.int16).cpu().numpy(), d_global)


DECODE_SHAPES = [(1, 24576, 128, 128, 128), (3, 24576, 256, 32, 32), (17, 136, 1024, 128, 32), (31, 264, 640, 32, 128),
           (32, 1032, 7168, 32, 32), (2, 8, 2048, 128, 128), (5, 7168, 384, 32, 32), (24, 24576, 1536, 128, 32)]


@pytest.mark.parametrize("M,N,K,bn,bk", DECODE_SHAPES)
@pytest.mark.parametrize("pow2", [True, False])
def test_decode_shapes(M, N, K, bn, bk, pow2):
    """Decode-sized shapes of the swap-AB plans: one K stage (K = 128), long K
    split many ways (1032 x 7168), a single row tile split over 16 CTAs
    (N = 8, K = 2048), more row tiles than SMs (N = 24576), ragged N and M,
    both recipes, UE8M0 scales (block-scaled MMA) and fp32 scales
    (promotion); and the fixed split-K summation order: a second call gives
    the same bits."""
    c = synth.Case("decode", M, N, K, bn, bk, pow2, seed=M + N + K)
    aq, a_s = oracle.quant_token_group(c.x(), bk, pow2)
    wq, ws = oracle.quant_weight_block(c.w(), bn, bk, pow2)
    dref, bound = oracle.gemm(aq, a_s, wq, ws, bn, bk)
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
    d0 = sgq.fp8_block_gemm(*args, bn, bk)
    assert sgq.sgq_device_status() == 0
    check_gemm(d0, dref, bound, f"decode M={M} N={N} K={K} [{bn},{bk}] pow2={pow2}")
    assert torch.equal(d0, sgq.fp8_block_gemm(*args, bn, bk))


@pytest.mark.parametrize("M,N,K,bk,flags", [(16, 7168, 2048, 32, 0), (256, 256, 2048, 128, sgq.SGQ_GEMM_ISSUE_SINGLE)])
def test_bounded_wait_times_out_and_the_stream_recovers(M, N, K, bk, flags):
    """The bounded device-side waits: with SGQ_GEMM_TEST_TIMEOUT the first CTA
    never loads one of its weight tiles, so the wait for it runs out (after
    about 1 ms).  The kernel must return on its own, sgq_device_status must
    report SGQ_ERR_TIMEOUT (once: reading clears it), and a normal GEMM on the
    same stream right after must be correct -- for the swap-AB decode tiles
    with split-K (M = 16) and the wide tiles (M = 256)."""
    from fp8_block_scaled_sgq_gb300 import binding
    aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=41), bk, True)
    wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=41), bk, bk, True)
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
    d = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    sgq.sgq_fp8_block_gemm_ex(*args, d, M, N, K, bk, bk, flags | binding.SGQ_GEMM_TEST_TIMEOUT)
    assert sgq.sgq_device_status() == binding.SGQ_ERR_TIMEOUT
    assert sgq.sgq_device_status() == binding.SGQ_OK
    dref, bound = oracle.gemm(aq, a_s, wq, ws, bk, bk)
    for _ in range(2):
        d2 = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        sgq.sgq_fp8_block_gemm_ex(*args, d2, M, N, K, bk, bk, flags)
        assert sgq.sgq_device_status() == binding.SGQ_OK
        check_gemm(d2, dref, bound, f"after the time-out M={M}")


DUAL = [(300, 520, 1024, 128, 128), (513, 264, 2048, 32, 32), (4100, 7000, 1280, 128, 32), (257, 1032, 4096, 32, 128),
        (2048, 448, 7168, 32, 32), (4096, 7168, 512, 128, 128), (4200, 7000, 384, 32, 32),
        (1024, 1536, 7168, 128, 128), (1000, 1032, 7168, 32, 128), (700, 7168, 2048, 32, 32),
        (130, 24576, 1536, 128, 128)]


@pytest.mark.parametrize("M,N,K,bn,bk", DUAL)
def test_scales_pow2_tiles_match_oracle(M, N, K, bn, bk):
    """SGQ_GEMM_SCALES_POW2 (every scale a power of two): the wide-tile plans
    with a wave of tiles run on 256 x 224 or 256 x 192 tiles with two
    accumulators (4096 x 7168 and 4200 x 7000 take the 192-wide tiles; the
    small shapes keep the 128-row tiles); 700 x 7168 and 130 x 24576 (0.6 of a
    wave) take them with one K split; 2048 x 448, 1024 x 1536 and 1000 x 1032
    (fewer tiles, M >= 768) with K split over several CTAs that exchange
    their partials.  Ragged M and N (partial row and column tiles, N not a
    multiple of the width), both recipes and their mixes; every row (or one of
    every 64-row block) against the oracle, and against the default path
    within the same tolerance; a second call gives the same bits."""
    c = synth.Case("dual", M, N, K, bn, bk, True, seed=M + N)
    aq, a_s = oracle.quant_token_group(c.x(), bk, True)
    wq, ws = oracle.quant_weight_block(c.w(), bn, bk, True)
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
    d = sgq.fp8_block_gemm(*args, bn, bk, flags=sgq.SGQ_GEMM_SCALES_POW2)
    assert sgq.sgq_device_status() == 0
    assert torch.equal(d, sgq.fp8_block_gemm(*args, bn, bk, flags=sgq.SGQ_GEMM_SCALES_POW2))
    r = np.arange(M) if M <= 600 else tile_rows(M, seed=M)
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, bn, bk)
    rr = torch.from_numpy(r).cuda()
    check_gemm(d[rr], dref, bound, f"pow2 tiles M={M} N={N} K={K} [{bn},{bk}]")
    check_gemm(sgq.fp8_block_gemm(*args, bn, bk)[rr], dref, bound, "default path")


_DUAL_CHILD = r"""
import sys, numpy as np, torch
import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import synth
import oracle
M, N, K, bn, bk = (int(v) for v in sys.argv[1:6])
aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=43), bk, True)
wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=43), bn, bk, True)
args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
d = sgq.fp8_block_gemm(*args, bn, bk, flags=sgq.SGQ_GEMM_SCALES_POW2)
assert sgq.sgq_device_status() == 0
assert torch.equal(d, sgq.fp8_block_gemm(*args, bn, bk, flags=sgq.SGQ_GEMM_SCALES_POW2))
np.save(sys.argv[6], d.view(torch.int16).cpu().numpy())
"""


@pytest.mark.parametrize("splits", [2, 3, 5, 8, 16])
@pytest.mark.parametrize("M,N,K,bn,bk", [(1000, 1032, 7168, 32, 128), (300, 1032, 7168, 128, 32),
                                         (130, 448, 4096, 128, 128)])
def test_dual_split_counts_match_oracle(tmp_path, M, N, K, bn, bk, splits):
    """The two-accumulator tiles with K split over `splits` CTAs (forced with
    SGQ_DUAL=1 SGQ_DUAL_SPLITS in a child process; the host lowers counts
    beyond one wave of CTAs or whose exchange does not fit: 1000 x 1032 runs
    at most 6, 300 x 1032 at most 12, 130 x 448 all of them).  Each split
    count sums the partials in its own fixed order: D is checked against the
    oracle on every 64-row block, and the child checks that a second call
    gives the same bits."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.path.join(root, "tests"), SGQ_DUAL="1",
               SGQ_DUAL_SPLITS=str(splits))
    out = str(tmp_path / "d.npy")
    subprocess.run([sys.executable, "-c", _DUAL_CHILD, str(M), str(N), str(K), str(bn), str(bk), out], env=env,
                   check=True, timeout=600, cwd=root)
    d = torch.from_numpy(np.load(out)).view(torch.bfloat16)
    aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=43), bk, True)
    wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=43), bn, bk, True)
    r = tile_rows(M, seed=splits)
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, bn, bk)
    check_gemm(d[torch.from_numpy(r)], dref, bound, f"dual splits={splits} M={M} N={N} K={K}")


@pytest.mark.parametrize("M,N,K,bn,bk", [(4100, 7000, 1280, 128, 32), (4200, 7000, 384, 32, 32),
                                         (4096, 7168, 512, 128, 128), (2100, 14000, 768, 32, 128)])
def test_dual_cta_pairs_match_oracle(tmp_path, M, N, K, bn, bk):
    """The two-accumulator tiles on CTA pairs (512 rows x BN per cluster of
    two, .cta_group::2 MMAs issued by the leader over both CTAs' halves),
    forced with SGQ_DUAL_PAIR=1 in a child process on shapes the default plan
    keeps on single CTAs: ragged M and N (a partial 512-row tile, N not a
    multiple of the width), short K, both recipes; D against the oracle on
    every 64-row block, and a second call gives the same bits."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.path.join(root, "tests"), SGQ_DUAL_PAIR="1")
    out = str(tmp_path / "d.npy")
    subprocess.run([sys.executable, "-c", _DUAL_CHILD, str(M), str(N), str(K), str(bn), str(bk), out], env=env,
                   check=True, timeout=600, cwd=root)
    d = torch.from_numpy(np.load(out)).view(torch.bfloat16)
    aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=43), bk, True)
    wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=43), bn, bk, True)
    r = tile_rows(M, seed=M)
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, bn, bk)
    check_gemm(d[torch.from_numpy(r)], dref, bound, f"dual pairs M={M} N={N} K={K} [{bn},{bk}]")


@pytest.mark.parametrize("name", ["prefill_block128", "prefill_block32"])
def test_scales_pow2_prefill_every_tile(name):
    """The prefill configurations (UE8M0 on both operands) through the
    power-of-two tiles (block128: on CTA pairs, the default for [*,128] with
    long K), one row of every 64-row block over all N columns."""
    c = synth.WORKLOADS[name][0]
    aq, a_s = oracle.quant_token_group(c.x(), c.group, c.ue8m0)
    wq, ws = weights(c.N, c.K, c.blk_n, c.blk_k, c.ue8m0, c.seed)
    d = run_gpu(aq, a_s, wq, ws, c.blk_n, c.blk_k, sgq.SGQ_GEMM_SCALES_POW2)
    r = tile_rows(c.M, seed=3)
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, c.blk_n, c.blk_k)
    check_gemm(d[torch.from_numpy(r).cuda()], dref, bound, f"{name} pow2 tiles")


def test_scales_pow2_flag_reports_a_broken_promise():
    """fp32 scales with SGQ_GEMM_SCALES_POW2: the device status reports
    SGQ_ERR_INVALID_ARG (the promise was broken), and the next call is fine."""
    from fp8_block_scaled_sgq_gb300 import binding
    M, N, K, bk = 4096, 2240, 256, 128   # 16 x 10 tiles of 256 x 224: the power-of-two tiles run
    assert sgq.sgq_gemm_plan(M, N, K, bk)["swap"] == 0
    aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=9), bk, False)
    wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=9), bk, bk, False)
    args = [torch.from_numpy(t).cuda() for t in (aq, a_s, wq, ws)]
    d = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    sgq.sgq_fp8_block_gemm_ex(*args, d, M, N, K, bk, bk, binding.SGQ_GEMM_SCALES_POW2)
    assert sgq.sgq_device_status() == binding.SGQ_ERR_INVALID_ARG
    r = tile_rows(M, seed=9)
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, bk, bk)
    d2 = sgq.fp8_block_gemm(*args, bk, bk)
    check_gemm(d2[torch.from_numpy(r).cuda()], dref, bound, "default path after the broken promise")
    assert sgq.sgq_device_status() == 0
