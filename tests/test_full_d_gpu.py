"""Every element of D at the full sizes of the prefill configurations and of
the sweep cases with M > 128.

The CPU oracle computes sampled rows (one of every 64-row block, all columns)
in seconds; all of D would take it minutes.  Here a second fp64 reference of
the same definition -- dequantise (E4M3 code x its block scales), then an fp64
product -- is built with library operations on the GPU (torch's E4M3
conversion, repeat_interleave, cuBLAS DGEMM), with no code shared with the
library under test.  It is pinned to the oracle first: on the sampled rows the
two references agree to fp64 rounding (and the bound Sum_k |a||w| with them).
Then every element of D, from each path the configuration runs on (fp32
scales on the 128 x 256 tiles, the power-of-two promise on the two-accumulator
tiles, UE8M0 bytes), must meet the GEMM tolerance against it:
|D - Dref| <= 2^-7 |Dref| + 1e-4 Sum_k |a||w|, and ||D - Dref||_F <= 5e-3 ||Dref||_F.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import synth

import oracle
from common import ABS_BOUND, REL_ELEM, REL_FRO, tile_rows

pytestmark = pytest.mark.gpu


def dequant(q, s, rows_per_scale, cols_per_scale):
    """fp64 [R, K] = E4M3 code x its scale (scale blocks of rows_per_scale x cols_per_scale)."""
    v = q.view(torch.float8_e4m3fn).to(torch.float32).to(torch.float64)   # exact
    s = s.to(torch.float64).repeat_interleave(cols_per_scale, dim=1)
    s = s.repeat_interleave(rows_per_scale, dim=0)[: q.shape[0]]
    return v * s


def fp64_reference(aq, a_s, wq, ws, bn, bk):
    a = dequant(aq, a_s, 1, bk)
    w = dequant(wq, ws, bn, bk)
    return a @ w.T, a.abs() @ w.abs().T


def check_full(d, ref, bound, what):
    d = d.to(torch.float64)
    assert bool(torch.isfinite(d).all()), f"{what}: non-finite output"
    err = (d - ref).abs()
    bad = err > REL_ELEM * ref.abs() + ABS_BOUND * bound
    n_bad = int(bad.sum())
    assert n_bad == 0, f"{what}: {n_bad} of {d.numel()} elements out of tolerance"
    rel = float(torch.linalg.norm(d - ref) / torch.linalg.norm(ref))
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel}"


# The prefill configurations, and every sweep case the oracle compares on
# sampled rows only (M > 128; M <= 128 it compares all of D itself).
CASES = [("prefill_block128", 0), ("prefill_block32", 0)] + [
    ("sweep", c.name[len("sweep_"):]) for c in synth.WORKLOADS["sweep"] if c.M > 128]


@pytest.mark.parametrize("name,which", CASES)
def test_every_element_of_d(name, which):
    cs = synth.WORKLOADS[name]
    c = cs[which] if isinstance(which, int) else next(k for k in cs if k.name == "sweep_" + which)
    aq, a_s = oracle.quant_token_group(c.x(), c.group, c.ue8m0)
    wq, ws = oracle.quant_weight_block(c.w(), c.blk_n, c.blk_k, c.ue8m0)
    t = [torch.from_numpy(np.ascontiguousarray(v)).cuda() for v in (aq, a_s, wq, ws)]
    ref, bound = fp64_reference(*t, c.blk_n, c.blk_k)
    # the GPU reference against the oracle on the sampled rows
    r = tile_rows(c.M, seed=5)
    o_ref, o_bound = oracle.gemm(aq[r], a_s[r], wq, ws, c.blk_n, c.blk_k)
    rr = torch.from_numpy(r).cuda()
    # (fp64 sums in two orders: within K * 2^-53 of the bound)
    np.testing.assert_allclose(ref[rr].cpu().numpy(), o_ref, rtol=0, atol=1e-10 * float(o_bound.max()))
    np.testing.assert_allclose(bound[rr].cpu().numpy(), o_bound, rtol=1e-11)
    paths = [("fp32 scales", lambda: sgq.fp8_block_gemm(*t, c.blk_n, c.blk_k))]
    if c.ue8m0:
        paths.append(("power-of-two promise",
                      lambda: sgq.fp8_block_gemm(*t, c.blk_n, c.blk_k, flags=sgq.SGQ_GEMM_SCALES_POW2)))
        e = [torch.from_numpy(oracle.ue8m0_bytes(v)).cuda() for v in (a_s, ws)]
        paths.append(("UE8M0 bytes", lambda: sgq.fp8_block_gemm_ue8m0(t[0], e[0], t[2], e[1], c.blk_n, c.blk_k)))
    for what, run in paths:
        d = run()
        assert sgq.sgq_device_status() == 0
        check_full(d, ref, bound, f"{c.name} {what}")
        del d
    del ref, bound
    torch.cuda.empty_cache()


def scaled_mm_reference(aq, sa, wq, sb, bias):
    """fp64 (Aq Wq^T) * sa (per row or one) * sb (per column or one) + bias, and its bound."""
    a = aq.view(torch.float8_e4m3fn).to(torch.float32).to(torch.float64)
    w = wq.view(torch.float8_e4m3fn).to(torch.float32).to(torch.float64)
    s = sa.to(torch.float64).reshape(-1, 1) * sb.to(torch.float64).reshape(1, -1)
    d = (a @ w.T) * s
    if bias is not None:
        d = d + bias.to(torch.float64).reshape(1, -1)
    return d, (a.abs() @ w.abs().T) * s.abs()


def test_every_element_of_scaled_mm_d():
    """fp8_scaled_mm at the prefill size (4096 x 7168 x 7168), per-token
    activation scales, per-channel weight scales and a bias: all of D against
    the fp64 reference, itself pinned to the oracle on the sampled rows."""
    M, N, K = 4096, 7168, 7168
    x, w = synth.activation(M, K, seed=9), synth.weight(N, K, seed=10)
    aq, sa = oracle.quant_per_token(x)
    wq, sb = oracle.quant_per_token(w)
    bias = synth.activation(1, N, seed=N).reshape(N)
    t = [torch.from_numpy(np.ascontiguousarray(v)).cuda() for v in (aq, sa, wq, sb)]
    ref, bound = scaled_mm_reference(*t, bias.cuda())
    r = tile_rows(M, seed=9)
    o_ref, o_bound = oracle.scaled_mm(aq[r], sa[r], wq, sb, bias)
    rr = torch.from_numpy(r).cuda()
    np.testing.assert_allclose(ref[rr].cpu().numpy(), o_ref, rtol=0, atol=1e-10 * float(o_bound.max()) + 1e-12)
    np.testing.assert_allclose(bound[rr].cpu().numpy(), o_bound, rtol=1e-11)
    d = sgq.fp8_scaled_mm(*t, bias.cuda())
    assert sgq.sgq_device_status() == 0
    check_full(d, ref, bound, "fp8_scaled_mm 4096 x 7168 x 7168")
