"""GPU quantisers vs the CPU oracle: codes and scale bits must match exactly."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import synth

import oracle

pytestmark = pytest.mark.gpu


def gpu_quant(x, group, ue8m0):
    xq, xs = sgq.quant_token_group(x.cuda(), group, ue8m0)
    torch.cuda.synchronize()
    return xq.cpu().numpy(), xs.cpu().numpy()


def assert_same(xq, xs, rq, rs, what):
    assert xs.view(np.uint32).shape == rs.view(np.uint32).shape
    bad_s = np.nonzero(xs.view(np.uint32) != rs.view(np.uint32))
    assert bad_s[0].size == 0, f"{what}: {bad_s[0].size} scales differ, first at {bad_s[0][0], bad_s[1][0]}: " \
                                f"{xs[bad_s[0][0], bad_s[1][0]]} vs {rs[bad_s[0][0], bad_s[1][0]]}"
    bad = np.nonzero(xq != rq)
    assert bad[0].size == 0, f"{what}: {bad[0].size} codes differ, first at {bad[0][0], bad[1][0]}: " \
                              f"{xq[bad[0][0], bad[1][0]]:#x} vs {rq[bad[0][0], bad[1][0]]:#x}"


CASES = [("tiny", 0), ("decode_block32", 0), ("decode_block32", 3), ("prefill_block128", 0),
         ("prefill_block32", 0), ("sweep", 8), ("sweep", 17), ("sweep", 26), ("sweep", 35)]


@pytest.mark.parametrize("workload,idx", CASES)
def test_quant_token_group_configs(workload, idx):
    c = synth.WORKLOADS[workload][idx]
    x = c.x()
    for ue in sorted({c.ue8m0, False}):
        xq, xs = gpu_quant(x, c.group, ue)
        rq, rs = oracle.quant_token_group(x, c.group, ue)
        assert_same(xq, xs, rq, rs, f"{c.name} ue8m0={ue}")


@pytest.mark.parametrize("group", [32, 128])
@pytest.mark.parametrize("ue8m0", [False, True])
def test_quant_edge_rows(group, ue8m0):
    K = 4 * group
    rows = []
    rows.append(np.zeros(K, np.float32))                                  # all-zero groups
    r = np.zeros(K, np.float32); r[::3] = -0.0; rows.append(r)
    r = -np.zeros(K, np.float32); rows.append(r)                          # -0.0 everywhere
    r = np.zeros(K, np.float32); r[5] = 3.0; r[group + 1] = -7.5; r[2 * group] = 1e-30; rows.append(r)
    # values on E4M3 tie midpoints after scaling by 1 (amax 448)
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2)
    r = np.resize(mids, K).astype(np.float32); r[::group] = 448.0; rows.append(r)
    r = -r; rows.append(r)
    # bf16 subnormals and extremes
    tiny = np.float32(2.0 ** -133)
    r = np.full(K, tiny, np.float32); r[::7] = -tiny * 5; rows.append(r)
    r = np.full(K, 3.0e38, np.float32); r[1::2] = -1.0; rows.append(r)
    r = np.linspace(-1e-3, 1e-3, K).astype(np.float32); rows.append(r)
    rng = np.random.default_rng(7)
    rows.append((rng.standard_normal(K) * 10.0 ** rng.integers(-30, 30)).astype(np.float32))
    x = torch.from_numpy(np.stack(rows)).to(torch.bfloat16)
    xq, xs = gpu_quant(x, group, ue8m0)
    rq, rs = oracle.quant_token_group(x, group, ue8m0)
    assert_same(xq, xs, rq, rs, f"edge rows g={group} ue8m0={ue8m0}")


@pytest.mark.parametrize("M,K,group", [(1, 32, 32), (3, 96, 32), (5, 384, 128), (129, 4096, 128),
                                       (257, 224, 32), (1000, 7168, 32)])
def test_quant_ragged_shapes(M, K, group):
    x = synth.activation(M, K, seed=M + K)
    for ue in (False, True):
        xq, xs = gpu_quant(x, group, ue)
        rq, rs = oracle.quant_token_group(x, group, ue)
        assert_same(xq, xs, rq, rs, f"M={M} K={K} g={group} ue={ue}")


def test_quant_m_zero_is_noop():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    xq, xs = sgq.quant_token_group(x, 128, True)
    assert xq.shape == (0, 256) and xs.shape == (0, 2)


WCASES = [(256, 512, 128, 128, False), (7168, 2048, 32, 32, True), (200, 256, 128, 128, True),
          (40, 96, 32, 32, False), (1536, 7168, 32, 32, True), (136, 384, 128, 32, True),
          (96, 256, 32, 128, False)]


@pytest.mark.parametrize("N,K,bn,bk,ue", WCASES)
def test_quant_weight_block(N, K, bn, bk, ue):
    w = synth.weight(N, K, seed=N)
    w[N - 1, K - 1] = 2.5           # lands in the (possibly ragged) last block
    wq, ws = sgq.quant_weight_block(w.cuda(), bn, bk, ue)
    torch.cuda.synchronize()
    rq, rs = oracle.quant_weight_block(w, bn, bk, ue)
    assert_same(wq.cpu().numpy(), ws.cpu().numpy(), rq, rs, f"weights N={N} K={K} [{bn},{bk}] ue={ue}")


@pytest.mark.parametrize("M,K", [(147, 7168), (1639, 640), (2049, 1536), (3, 384)])
@pytest.mark.parametrize("ue8m0", [False, True])
@pytest.mark.parametrize("group", [32, 128])
def test_both_access_widths(M, K, ue8m0, group):
    """The quantiser runs with 32-byte accesses when x has at least 2^20
    elements and starts on a 32-byte boundary, and with 16-byte ones otherwise
    (smaller x, or another alignment): both give the oracle's codes and scale
    bits (ragged last warp chunk included: M x K / 16 not a multiple of 32),
    fp32 scales and UE8M0 bytes."""
    x = synth.activation(M, K, seed=M + K)
    rq, rs = oracle.quant_token_group(x, group, ue8m0)
    buf = torch.empty(M * K + 16, dtype=torch.bfloat16, device="cuda")
    for off in (0, 8):   # elements: byte offsets 0 (32-byte aligned) and 16
        xd = buf[off:off + M * K].view(M, K)
        xd.copy_(x.cuda())
        assert (xd.data_ptr() % 32 == 0) == (off == 0)
        xq, xs = sgq.quant_token_group(xd, group, ue8m0)
        torch.cuda.synchronize()
        assert sgq.sgq_device_status() == 0
        assert_same(xq.cpu().numpy(), xs.cpu().numpy(), rq, rs, f"M={M} K={K} group={group} offset={off}")
        if ue8m0:
            xq8, xe = sgq.quant_token_group_ue8m0(xd, group)
            assert np.array_equal(xq8.cpu().numpy(), rq)
            assert np.array_equal(xe.cpu().numpy(), oracle.ue8m0_bytes(rs))
