"""The allocation-free GEMM entry point (sgq_fp8_block_gemm_noalloc).

It exists for callers that cannot let the library allocate device memory --
for example a serving engine that has reserved nearly all of HBM for its own
pool up front, where a later cudaMalloc would fail or fragment that pool -- and
keeps the split-K scratch in a fixed device array inside the library instead
of the workspace sgq_fp8_block_gemm allocates on first use.

These tests call it through the C ABI, twice in a row, on decode shapes that
use split-K, and compare it with the default entry point: bit for bit where
both take the same launch plan, within the GEMM tolerance where the fixed
array makes it take fewer K splits.  One test runs it first in a fresh process
and checks that the library allocated nothing.  The file is collected last,
and works alone or after the other tests.
"""
import os
import subprocess
import sys

import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import binding, build, synth

import oracle
from common import check_gemm, tile_rows

pytestmark = pytest.mark.gpu

NOALLOC_PARTIAL_BYTES = 16 << 20   # the fixed array's fp32 partials


def _operands(M, N, K, blk, seed):
    x = synth.activation(M, K, seed=seed)
    w = synth.weight(N, K, seed=seed)
    aq, a_s = oracle.quant_token_group(x, blk, True)
    wq, ws = oracle.quant_weight_block(w, blk, blk, True)
    return aq, a_s, wq, ws


def _plan_fits(M, N, K, blk):
    """Whether the default plan's split-K partials fit the fixed array."""
    p = sgq.sgq_gemm_plan(M, N, K, blk)
    return p["splits"] == 1 or p["items"] * 128 * p["bn"] * 4 <= NOALLOC_PARTIAL_BYTES


@pytest.mark.parametrize("M,N,K", [(16, 1536, 7168), (4, 1536, 7168), (64, 7168, 2048)])
def test_noalloc_matches_default_entry_point_twice(M, N, K):
    """Decode shapes whose plans split K, so the fixed array is used."""
    build.build()
    lib = binding.load_library()
    blk = 32
    assert sgq.sgq_gemm_plan(M, N, K, blk)["splits"] > 1   # the case exercises the fixed array
    assert _plan_fits(M, N, K, blk)                        # ... under the default plan
    aq, a_s, wq, ws = _operands(M, N, K, blk, 21)
    dref, bound = oracle.gemm(aq, a_s, wq, ws, blk, blk)
    t = [torch.from_numpy(v).cuda() for v in (aq, a_s, wq, ws)]
    stream = torch.cuda.current_stream().cuda_stream

    d_default = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    rc = lib.sgq_fp8_block_gemm(*(v.data_ptr() for v in t), d_default.data_ptr(), M, N, K, blk, blk, stream)
    assert rc == binding.SGQ_OK

    for call in range(2):
        d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.sgq_fp8_block_gemm_noalloc(*(v.data_ptr() for v in t), d.data_ptr(), M, N, K, blk, blk,
                                            stream)
        assert rc == binding.SGQ_OK, sgq.status_string(rc)
        assert sgq.sgq_device_status() == binding.SGQ_OK
        # same plan, same summation order: the same bits as the default entry point
        assert torch.equal(d, d_default), f"no-alloc call {call + 1}, M={M}"
        check_gemm(d, dref, bound, f"no-alloc call {call + 1}, M={M}")


@pytest.mark.parametrize("M,N,K", [(1024, 1536, 7168), (64, 24576, 7168)])
def test_noalloc_plans_within_the_fixed_array(M, N, K):
    """Shapes whose default plan needs more split-K partials than the fixed
    array holds (1024 x 1536 x 7168: swap-AB tiles of 64 tokens in three K
    splits, 18.9 MB; 64 x 24576 x 7168: three splits, 18.9 MB) still run: the
    allocation-free entry point plans fewer splits (or the 128 x 256 tiles)
    within the array.  Checked against the oracle on one row of every 64-row
    block, and against the default entry point within the tolerance, twice."""
    lib = binding.load_library()
    blk = 32
    assert not _plan_fits(M, N, K, blk)
    aq, a_s, wq, ws = _operands(M, N, K, blk, 22)
    rows = tile_rows(M, seed=22)
    dref, bound = oracle.gemm(aq[rows], a_s[rows], wq, ws, blk, blk)
    t = [torch.from_numpy(v).cuda() for v in (aq, a_s, wq, ws)]
    stream = torch.cuda.current_stream().cuda_stream
    r = torch.from_numpy(rows).cuda()
    d_default = sgq.fp8_block_gemm(*t, blk, blk)
    check_gemm(d_default[r], dref, bound, f"default {M}x{N}x{K}")
    for call in range(2):
        d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.sgq_fp8_block_gemm_noalloc(*(v.data_ptr() for v in t), d.data_ptr(), M, N, K, blk, blk,
                                            stream)
        assert rc == binding.SGQ_OK, sgq.status_string(rc)
        assert sgq.sgq_device_status() == binding.SGQ_OK
        assert bool(torch.isfinite(d).all())   # every element written
        check_gemm(d[r], dref, bound, f"no-alloc {M}x{N}x{K} call {call + 1}")


_FRESH_CHILD = r"""
import numpy as np, torch
import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import binding, synth
import oracle
from common import check_gemm
lib = binding.load_library()
M, N, K, blk = 16, 1536, 7168, 32
assert sgq.sgq_gemm_plan(M, N, K, blk)["splits"] > 1
x, w = synth.activation(M, K, seed=23), synth.weight(N, K, seed=23)
aq, a_s = oracle.quant_token_group(x, blk, True)
wq, ws = oracle.quant_weight_block(w, blk, blk, True)
dref, bound = oracle.gemm(aq, a_s, wq, ws, blk, blk)
t = [torch.from_numpy(v).cuda() for v in (aq, a_s, wq, ws)]
st = torch.cuda.current_stream().cuda_stream
for call in range(2):
    d = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    rc = lib.sgq_fp8_block_gemm_noalloc(*(v.data_ptr() for v in t), d.data_ptr(), M, N, K, blk, blk, st)
    assert rc == 0, sgq.status_string(rc)
    assert sgq.sgq_device_status() == 0
    check_gemm(d, dref, bound, f"fresh process, call {call + 1}")
assert sgq.sgq_allocated_bytes() == 0, sgq.sgq_allocated_bytes()
d2 = sgq.fp8_block_gemm(*t, blk, blk)          # the default entry point does allocate
assert sgq.sgq_allocated_bytes() > 0
print("fresh ok")
"""


def test_noalloc_first_call_in_fresh_process_allocates_nothing():
    """In a fresh process the allocation-free call comes first: its result
    matches the oracle, and the library reports no device allocation until the
    default entry point runs."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, PYTHONPATH=root + os.pathsep + os.path.join(root, "tests"))
    r = subprocess.run([sys.executable, "-c", _FRESH_CHILD], env=env, cwd=root, timeout=600,
                       capture_output=True, text=True)
    assert r.returncode == 0 and "fresh ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
