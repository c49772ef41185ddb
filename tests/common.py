"""Shared helpers for the GPU parity tests (oracle on the CPU, library on the GPU)."""
import numpy as np
import torch

import oracle

REL_FRO = 5e-3          # ||D - Dref||_F / ||Dref||_F
REL_ELEM = 2.0 ** -7    # elementwise: |D - Dref| <= REL_ELEM*|Dref| + ABS_BOUND*sum_k|a||w|
ABS_BOUND = 1e-4


def u8(t):
    return t.detach().cpu().numpy()


def f32(t):
    return t.detach().cpu().numpy()


def check_gemm(d_gpu, d_ref, bound, what=""):
    """The GEMM acceptance criterion, on fp64 copies."""
    d = d_gpu.detach().float().cpu().numpy().astype(np.float64)
    assert d.shape == d_ref.shape, (d.shape, d_ref.shape)
    assert np.all(np.isfinite(d)), f"{what}: non-finite output"
    err = np.abs(d - d_ref)
    tol = REL_ELEM * np.abs(d_ref) + ABS_BOUND * bound
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance, e.g. at {i.tolist()}: "
                             f"got {d[tuple(i[0])]}, want {d_ref[tuple(i[0])]}")
    nrm = np.linalg.norm(d_ref)
    rel = np.linalg.norm(d - d_ref) / nrm if nrm > 0 else np.linalg.norm(d)
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel}"
    return rel


def oracle_weights(w_bf16, blk_n, blk_k, ue8m0):
    wq, ws = oracle.quant_weight_block(w_bf16, blk_n, blk_k, ue8m0)
    return wq, ws


def sample_rows(M, n=12, seed=0):
    """Rows that cover the first/last tile and tile borders, plus random ones."""
    if M <= 2 * n:
        return np.arange(M)
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, M // 2, M - 129, M - 128, M - 1]
    rows = set(r for r in fixed if 0 <= r < M)
    while len(rows) < n:
        rows.add(int(rng.integers(0, M)))
    return np.array(sorted(rows))


def tile_rows(M, block=64, seed=0):
    """One row in every `block`-row block of [0, M) -- with block = 64 that is
    every 128-row tile of the wide GEMM plan and every 64-token tile of the
    swap-AB plans -- at an offset inside the block that changes from block to
    block, plus the first and last row of every 128-row tile boundary pair and
    of the whole range."""
    rows = set()
    nblk = (M + block - 1) // block
    for b in range(nblk):
        off = (b * 37 + seed * 11 + 5) % block
        rows.add(min(b * block + off, M - 1))
    for r in (0, 1, 127, 128, M // 2, M - 129, M - 128, M - 1):
        if 0 <= r < M:
            rows.add(r)
    return np.array(sorted(rows))
