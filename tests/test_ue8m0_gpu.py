"""UE8M0 scale bytes on the GPU: the byte-output quantiser and the fp32 -> byte
conversion against the oracle bit for bit, and the GEMM on byte scales against
the same GEMM on the fp32 scales 2^(e - 127) (bit for bit) and the oracle."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import binding, synth

import oracle
from common import check_gemm, tile_rows

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K,group", [(1, 128, 128), (5, 4096, 32), (257, 7168, 128), (1000, 2048, 32)])
def test_quant_token_group_ue8m0_matches_oracle(M, K, group):
    """Codes bit-identical to the ue8m0 = 1 quantiser (and the oracle); every
    scale byte the oracle's UE8M0 byte of its power-of-two group scale."""
    x = synth.activation(M, K, seed=M + K)
    aq_ref, as_ref = oracle.quant_token_group(x, group, True)
    xq, xe = sgq.quant_token_group_ue8m0(x.cuda(), group)
    assert np.array_equal(xq.cpu().numpy(), aq_ref)
    assert np.array_equal(xe.cpu().numpy(), oracle.ue8m0_bytes(as_ref))
    xq2, xs2 = sgq.quant_token_group(x.cuda(), group, True)
    assert torch.equal(xq, xq2)


def test_scales_to_ue8m0_matches_oracle_and_flags_bad_values():
    """Powers of two -> their bytes; anything else -> 255 and SGQ_ERR_INVALID_ARG."""
    rng = np.random.default_rng(3)
    good = np.ldexp(np.float32(1.0), rng.integers(-126, 128, 5000)).astype(np.float32)
    e = sgq.scales_to_ue8m0(torch.from_numpy(good).cuda())
    assert sgq.sgq_device_status() == binding.SGQ_OK
    assert np.array_equal(e.cpu().numpy(), oracle.ue8m0_bytes(good))
    bad = good.copy()
    bad[[0, 17, 4999]] = [3.0, 0.0, -0.5]
    e = sgq.scales_to_ue8m0(torch.from_numpy(bad).cuda())
    assert sgq.sgq_device_status() == binding.SGQ_ERR_INVALID_ARG
    assert np.array_equal(e.cpu().numpy(), oracle.ue8m0_bytes(bad))
    assert sgq.sgq_device_status() == binding.SGQ_OK


# the two-accumulator tiles (one CTA per tile; CTA pairs with K >= 4096; K
# split over CTAs), mid-M one split, and plans that widen the bytes first
# (decode, tiny, short K)
SHAPES = [(4096, 7168, 512, 128, 128), (4100, 7000, 4096, 128, 128), (4200, 7000, 384, 32, 32),
          (4100, 7000, 4096, 32, 32), (2100, 14000, 4096, 128, 32),
          (1024, 1536, 7168, 128, 128), (700, 7168, 2048, 32, 32), (16, 7168, 2048, 32, 32),
          (3, 520, 1024, 128, 32), (300, 1032, 640, 32, 128)]


@pytest.mark.parametrize("M,N,K,bn,bk", SHAPES)
def test_gemm_ue8m0_bit_identical_to_fp32_scales(M, N, K, bn, bk):
    """D from byte scales equals D from the fp32 scales 2^(e - 127) with the
    power-of-two promise bit for bit (the MMAs see the same factors) where
    both plans sum K in the same order -- no K splits (single CTAs or CTA
    pairs alike), or the same plan.  Both against the oracle on every 64-row
    block."""
    c = synth.Case("e8", M, N, K, bn, bk, True, seed=M + N + K)
    aq, a_s = oracle.quant_token_group(c.x(), bk, True)
    wq, ws = oracle.quant_weight_block(c.w(), bn, bk, True)
    ae, we = oracle.ue8m0_bytes(a_s), oracle.ue8m0_bytes(ws)
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
    d8 = sgq.fp8_block_gemm_ue8m0(t(aq), t(ae), t(wq), t(we), bn, bk)
    assert sgq.sgq_device_status() == 0
    d32 = sgq.fp8_block_gemm(t(aq), t(a_s), t(wq), t(ws), bn, bk, flags=sgq.SGQ_GEMM_SCALES_POW2)
    assert sgq.sgq_device_status() == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    p8, p32 = sgq.sgq_gemm_plan_pow2(M, N, K, bk, sms, True), sgq.sgq_gemm_plan_pow2(M, N, K, bk, sms, False)
    if (p8["splits"] <= 1 and p32["splits"] <= 1) or p8 == p32:
        assert torch.equal(d8, d32)
    r = np.arange(M) if M <= 600 else tile_rows(M, seed=M)
    rr = torch.from_numpy(r).cuda()
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, bn, bk)
    check_gemm(d8[rr], dref, bound, f"ue8m0 M={M} N={N} K={K} [{bn},{bk}]")
    check_gemm(d32[rr], dref, bound, f"fp32 pow2 M={M} N={N} K={K} [{bn},{bk}]")


def test_gemm_ue8m0_reports_a_nan_byte():
    """A scale byte of 255 (NaN) where the bytes are read directly: the call
    returns, sgq_device_status reports SGQ_ERR_INVALID_ARG once."""
    M, N, K, bk = 4096, 2240, 256, 128
    aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=9), bk, True)
    wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=9), bk, bk, True)
    ae, we = oracle.ue8m0_bytes(a_s), oracle.ue8m0_bytes(ws)
    ae[5, 1] = 255
    t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
    sgq.fp8_block_gemm_ue8m0(t(aq), t(ae), t(wq), t(we), bk, bk)
    assert sgq.sgq_device_status() == binding.SGQ_ERR_INVALID_ARG
    assert sgq.sgq_device_status() == binding.SGQ_OK


_PAIR_CHILD = r"""
import sys, numpy as np, torch
import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import synth
import oracle
M, N, K, bn, bk = (int(v) for v in sys.argv[1:6])
aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=47), bk, True)
wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=47), bn, bk, True)
t = lambda v: torch.from_numpy(np.ascontiguousarray(v)).cuda()
d8 = sgq.fp8_block_gemm_ue8m0(t(aq), t(oracle.ue8m0_bytes(a_s)), t(wq), t(oracle.ue8m0_bytes(ws)), bn, bk)
assert sgq.sgq_device_status() == 0
d32 = sgq.fp8_block_gemm(t(aq), t(a_s), t(wq), t(ws), bn, bk, flags=sgq.SGQ_GEMM_SCALES_POW2)
assert sgq.sgq_device_status() == 0
assert torch.equal(d8, d32)
np.save(sys.argv[6], d8.view(torch.int16).cpu().numpy())
"""


@pytest.mark.parametrize("M,N,K,bn,bk", [(4100, 7000, 1280, 128, 128), (4200, 7000, 2048, 32, 32),
                                         (4096, 7168, 4096, 128, 32)])
def test_gemm_ue8m0_on_forced_cta_pairs(tmp_path, M, N, K, bn, bk):
    """Byte scales on CTA pairs, forced with SGQ_DUAL_PAIR=1 in a child process
    (the default plan keeps K < 4096 on single CTAs): bit for bit the fp32
    path on pairs, and the oracle on every 64-row block."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.path.join(root, "tests"), SGQ_DUAL_PAIR="1")
    out = str(tmp_path / "d.npy")
    subprocess.run([sys.executable, "-c", _PAIR_CHILD, str(M), str(N), str(K), str(bn), str(bk), out], env=env,
                   check=True, timeout=600, cwd=root)
    d = torch.from_numpy(np.load(out)).view(torch.bfloat16)
    aq, a_s = oracle.quant_token_group(synth.activation(M, K, seed=47), bk, True)
    wq, ws = oracle.quant_weight_block(synth.weight(N, K, seed=47), bn, bk, True)
    r = tile_rows(M, seed=M)
    dref, bound = oracle.gemm(aq[r], a_s[r], wq, ws, bn, bk)
    check_gemm(d[torch.from_numpy(r)], dref, bound, f"ue8m0 pairs M={M} N={N} K={K} [{bn},{bk}]")
