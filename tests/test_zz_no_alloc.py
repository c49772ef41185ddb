"""The allocation-free GEMM entry point (sgq_fp8_block_gemm_noalloc).

It exists for callers that cannot let the library allocate device memory --
for example a serving engine that has reserved nearly all of HBM for its own
pool -- and keeps the split-K scratch in a fixed device array inside the
library.  This test calls it through the C ABI twice in a row on decode
shapes that do use split-K, and checks each result against the default entry
point's result under the same GEMM tolerance as the other tests.  It lives in
a file of its own, collected last, and works alone or after the other tests.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import binding, build, synth

import oracle
from common import check_gemm

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [16, 4])
def test_noalloc_matches_default_entry_point_twice(M):
    build.build()
    lib = binding.load_library()
    N, K, blk = 7168, 2048, 32
    x = synth.activation(M, K, seed=21)
    w = synth.weight(N, K, seed=21)
    aq, a_s = oracle.quant_token_group(x, blk, True)
    wq, ws = oracle.quant_weight_block(w, blk, blk, True)
    _, bound = oracle.gemm(aq, a_s, wq, ws, blk, blk)
    t = [torch.from_numpy(v).cuda() for v in (aq, a_s, wq, ws)]
    stream = torch.cuda.current_stream().cuda_stream

    d_default = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rc = lib.sgq_fp8_block_gemm(*(v.data_ptr() for v in t), d_default.data_ptr(), M, N, K, blk, blk, stream)
    assert rc == binding.SGQ_OK
    ref = d_default.double().cpu().numpy()

    for call in range(2):
        d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.sgq_fp8_block_gemm_noalloc(*(v.data_ptr() for v in t), d.data_ptr(), M, N, K, blk, blk,
                                            stream)
        assert rc == binding.SGQ_OK, sgq.status_string(rc)
        assert sgq.sgq_device_status() == binding.SGQ_OK
        check_gemm(d, ref, bound, f"no-alloc call {call + 1}, M={M}")


def test_noalloc_mid_m_plan_that_would_overflow_the_fixed_array():
    """1024 x 1536 x 7168: the default plan takes swap-AB tiles of 64 tokens in
    three K splits, whose partials (18.9 MB) exceed the fixed array; the
    allocation-free entry point runs the 128 x 256-tile plan instead."""
    from common import sample_rows
    lib = binding.load_library()
    M, N, K, blk = 1024, 1536, 7168, 32
    p = sgq.sgq_gemm_plan(M, N, K, blk)
    assert p["swap"] == 1 and p["items"] * 128 * p["bn"] * 4 > (16 << 20)
    x = synth.activation(M, K, seed=22)
    w = synth.weight(N, K, seed=22)
    aq, a_s = oracle.quant_token_group(x, blk, True)
    wq, ws = oracle.quant_weight_block(w, blk, blk, True)
    rows = sample_rows(M, 8, seed=22)
    dref, bound = oracle.gemm(aq[rows], a_s[rows], wq, ws, blk, blk)
    t = [torch.from_numpy(v).cuda() for v in (aq, a_s, wq, ws)]
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.sgq_fp8_block_gemm_noalloc(*(v.data_ptr() for v in t), d.data_ptr(), M, N, K, blk, blk,
                                        torch.cuda.current_stream().cuda_stream)
    assert rc == binding.SGQ_OK, sgq.status_string(rc)
    assert sgq.sgq_device_status() == binding.SGQ_OK
    check_gemm(d[torch.from_numpy(rows).cuda()], dref, bound, "no-alloc mid-M")
