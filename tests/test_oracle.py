"""Pins for the CPU oracle, against what the pages and the mathematics fix.

Each test is chosen so that a plausible slip in the oracle (wrong rounding,
a dropped term, a transposed operand, an off-by-one block index) fails it.
No GPU, no CUDA library.
"""
import os
import struct

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def to_bf16_bits(vals):
    t = torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def parse_golden(name):
    sections, cur = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("["):
                cur = sections.setdefault(line.strip("[]"), {})
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            tgt = cur if cur is not None else sections.setdefault("", {})
            tgt.setdefault(k, []).append(v.split())
    return sections


# ---------------------------------------------------------------- E4M3 codec

def test_e4m3_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert codes.size == 254
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    back = oracle.e4m3_encode(vals)
    np.testing.assert_array_equal(back, codes)


def test_e4m3_decode_known_points():
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert dec[0x7E] == 448.0 and dec[0xFE] == -448.0          # largest finite
    assert dec[0x01] == 2.0 ** -9                              # smallest subnormal
    assert dec[0x08] == 2.0 ** -6                              # smallest normal
    assert dec[0x38] == 1.0 and dec[0x40] == 2.0
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert dec[0x80] == 0.0 and np.signbit(dec[0x80])


def test_e4m3_monotone():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)


def test_e4m3_ties_to_even_and_saturation():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.all(mids.astype(np.float64) == (pos[:-1] + pos[1:]) / 2)   # exact in fp32
    got = oracle.e4m3_encode(mids).astype(np.int64)
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1)                    # even code wins the tie
    np.testing.assert_array_equal(got, want)
    # just above / below a midpoint goes to the nearer code
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    np.testing.assert_array_equal(oracle.e4m3_encode(up), lo + 1)
    np.testing.assert_array_equal(oracle.e4m3_encode(dn[1:]), lo[1:])
    sat = oracle.e4m3_encode(np.array([448, 463.9, 464, 480, 1e30, np.inf,
                                       -448, -500, -np.inf], dtype=np.float32))
    np.testing.assert_array_equal(sat, [0x7E] * 6 + [0xFE] * 3)
    z = oracle.e4m3_encode(np.array([0.0, -0.0, 2.0 ** -10, -(2.0 ** -10), 1e-30, -1e-30],
                                    dtype=np.float32))
    np.testing.assert_array_equal(z, [0x00, 0x80, 0x00, 0x80, 0x00, 0x80])


def test_e4m3_matches_torch_dense_sweep():
    """Library special case: torch.float8_e4m3fn rounds to nearest even.

    Every fp32 on the 2^-12 lattice with |v| < 464 (torch does not saturate,
    so stay below the point where RNE would leave the finite range), plus
    random fp32 values of all magnitudes in that range.
    """
    lat = (np.arange(-464 * 4096 + 1, 464 * 4096, dtype=np.int64) / 4096.0).astype(np.float32)
    rng = np.random.default_rng(1)
    mant = rng.uniform(1.0, 2.0, 400000)
    expo = rng.integers(-40, 9, 400000)
    rnd = (rng.choice([-1.0, 1.0], 400000) * mant * np.exp2(expo)).astype(np.float32)
    rnd = rnd[np.abs(rnd) < 464]
    for v in (lat, rnd):
        ours = oracle.e4m3_encode(v)
        ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        np.testing.assert_array_equal(ours, ref)


# ---------------------------------------------------------------- scales

def test_ue8m0_is_minimal_power_of_two():
    rng = np.random.default_rng(2)
    amax = np.concatenate([
        (rng.uniform(1, 2, 20000) * np.exp2(rng.integers(-60, 60, 20000))),
        448.0 * np.exp2(rng.integers(-30, 30, 200)),               # amax/448 is a power of two
    ]).astype(np.float32)
    for a in amax:
        s32 = oracle.group_scale(a, ue8m0=False)
        s = oracle.group_scale(a, ue8m0=True)
        b = int(f32_bits(s))
        assert b & 0x7FFFFF == 0 and (b >> 31) == 0                # exact power of two
        assert float(s) >= float(s32) >= float(a) / 448.0 * (1 - 2 ** -23)
        if int(f32_bits(s32)) & 0x7FFFFF:
            assert float(s) / 2 < float(s32)                       # minimal
        else:
            assert float(s) == float(s32)


def test_ue8m0_bytes_closed_forms_and_round_trip():
    """UE8M0 byte of a power-of-two scale: the 8-bit biased exponent (value
    2^(e - 127)).  Closed forms, every byte 1 .. 254 through ldexp and back,
    the NaN byte (255) for everything that is not a positive normal power of
    two, and log2 of the power-of-two rounding (ue8m0_ceil) for random scales."""
    f32 = np.float32
    known = {1.0: 127, 0.5: 126, 2.0: 128, 2.0 ** -126: 1, 2.0 ** 127: 254, 2.0 ** -7: 120, 448.0 / 448.0: 127}
    for v, e in known.items():
        assert int(oracle.ue8m0_bytes(np.array([v], f32))[0]) == e
    e = np.arange(1, 255, dtype=np.uint8)
    v = np.ldexp(np.float32(1.0), e.astype(np.int32) - 127).astype(f32)
    assert np.array_equal(oracle.ue8m0_bytes(v), e)
    assert np.array_equal(oracle.ue8m0_values(e), v)
    bad = np.array([3.0, -1.0, 0.0, -0.0, 2.0 ** -130, np.inf, np.nan, 1.5, 448.0], f32)
    assert np.all(oracle.ue8m0_bytes(bad) == 255)
    assert np.isnan(oracle.ue8m0_values(np.array([255], np.uint8))[0])
    rng = np.random.default_rng(7)
    s = (rng.random(2000) * 10.0 ** rng.integers(-30, 30, 2000)).astype(f32)
    s = s[(s > np.finfo(f32).tiny) & (s < 2.0 ** 126)]
    p = oracle.ue8m0_ceil(s)
    assert np.array_equal(oracle.ue8m0_bytes(p).astype(np.int64), np.ceil(np.log2(s.astype(np.float64))).astype(np.int64) + 127)


def test_fp32_scale_is_correctly_rounded_division():
    rng = np.random.default_rng(3)
    a = rng.uniform(1e-3, 1e3, 5000).astype(np.float32)
    got = np.array([oracle.group_scale(x, False) for x in a], dtype=np.float32)
    # correctly rounded: the nearest fp32 to the exact quotient
    exact = a.astype(np.float64) / 448.0
    np.testing.assert_array_equal(got, exact.astype(np.float32))


def test_eps_floor_on_zero_group():
    x = np.zeros((2, 64), dtype=np.uint16)
    x[1, :32] = 0x8000                                              # -0.0
    q, s = oracle.quant_token_group(x, 32, ue8m0=False)
    assert np.all(s == np.float32(np.float32(1e-10) / np.float32(448.0)))
    assert np.all(q[0] == 0) and np.all(q[1, :32] == 0x80) and np.all(q[1, 32:] == 0)
    q, s = oracle.quant_token_group(x, 32, ue8m0=True)
    # 1e-10/448 = 2.23e-13 lies in (2^-43, 2^-42]
    assert np.all(s == np.float32(2.0 ** -42))


# ---------------------------------------------------------------- group quant

@pytest.mark.parametrize("case", ["scale_one", "half_steps_ue8m0", "half_steps_fp32"])
def test_golden_worked_examples(case):
    g = parse_golden("quant_group32_worked.txt")[case]
    x = to_bf16_bits([float(v) for v in g["x"][0]])
    assert np.all(torch.tensor([float(v) for v in g["x"][0]]).to(torch.bfloat16).float().numpy()
                  == np.array([float(v) for v in g["x"][0]]))
    want_codes = np.array([int(c, 16) for c in g["codes"][0]], dtype=np.uint8)
    want_scale = int(g["scale_bits"][0][0], 16)
    for ue in (int(u) for u in g["ue8m0"][0]):
        q, s = oracle.quant_token_group(x.reshape(1, 32), 32, ue8m0=bool(ue))
        assert int(f32_bits(s[0, 0])) == want_scale
        np.testing.assert_array_equal(q[0], want_codes)


def test_constant_and_one_hot_groups():
    vals = [0.75, -3.0, 1e-3, 12.5]
    x = np.concatenate([np.full(32, v, dtype=np.float32) for v in vals])
    q, s = oracle.quant_token_group(to_bf16_bits(x).reshape(1, -1), 32, ue8m0=False)
    for j, v in enumerate(vals):
        vb = float(torch.tensor(v).to(torch.bfloat16).float())
        assert s[0, j] == np.float32(np.float32(abs(vb)) / np.float32(448))
        assert np.all(q[0, 32 * j:32 * j + 32] == (0xFE if v < 0 else 0x7E))
    hot = np.zeros(128, dtype=np.float32)
    hot[5], hot[32 + 31], hot[64], hot[127] = 3.0, -0.5, 100.0, -7.0
    for ue in (False, True):
        q, s = oracle.quant_token_group(to_bf16_bits(hot).reshape(1, -1), 32, ue8m0=ue)
        nz = np.nonzero(q[0] & 0x7F)[0]
        np.testing.assert_array_equal(nz, [5, 63, 64, 127])
        mag = oracle.e4m3_decode(q[0, nz] & 0x7F)
        if ue:
            assert np.all((mag > 224) & (mag <= 448))        # amax/s in (224, 448]
        else:
            assert np.all(mag == 448)                        # the amax element maps to fp8_max
        assert np.all(np.signbit(oracle.e4m3_decode(q[0, nz])) == (hot[nz] < 0))


def test_lossless_roundtrip_pow2_grid():
    """x = c * S with c E4M3 codes and one power of two S per group is recovered."""
    rng = np.random.default_rng(4)
    for group in (32, 128):
        G = 64
        codes = rng.integers(0, 256, (G, group)).astype(np.uint8)
        codes[(codes & 0x7F) == 0x7F] = 0x3C
        c = oracle.e4m3_decode(codes)
        S = np.exp2(rng.integers(-20, 20, (G, 1))).astype(np.float64)
        x = (c * S).astype(np.float32)
        xb = to_bf16_bits(x).reshape(1, -1)
        assert np.all(torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).float().numpy()
                      == x.reshape(1, -1))
        q, s = oracle.quant_token_group(xb, group, ue8m0=True)
        s = s.reshape(G, 1).astype(np.float64)
        assert np.all(s <= S)
        back = oracle.e4m3_decode(q.reshape(G, group)) * s
        np.testing.assert_array_equal(back, x.astype(np.float64))
        # fp32-scale quantiser is lossless when amax/448 is a power of two
        codes[:, 0] = 0x7E
        x = (oracle.e4m3_decode(codes) * S).astype(np.float32)
        q, s = oracle.quant_token_group(to_bf16_bits(x).reshape(1, -1), group, ue8m0=False)
        assert np.all(s.reshape(G, 1) == S)
        back = oracle.e4m3_decode(q.reshape(G, group)) * s.reshape(G, 1)
        np.testing.assert_array_equal(back, x.astype(np.float64))


def test_quant_brute_force_random():
    """Group quant equals the elementwise rule written with numpy/torch pieces."""
    rng = np.random.default_rng(5)
    x = torch.from_numpy(rng.standard_normal((7, 256)).astype(np.float32) *
                         np.exp2(rng.integers(-8, 8, (7, 1))).astype(np.float32)).to(torch.bfloat16)
    for group in (32, 128):
        for ue in (False, True):
            q, s = oracle.quant_token_group(x, group, ue)
            xf = x.float().numpy().reshape(7, -1, group)
            amax = np.abs(xf).max(axis=2)
            s_ref = (np.maximum(amax, np.float32(1e-10)) / np.float32(448)).astype(np.float32)
            if ue:
                s_ref = np.exp2(np.ceil(np.log2(s_ref.astype(np.float64)))).astype(np.float32)
            np.testing.assert_array_equal(s, s_ref)
            quot = np.clip((xf / s_ref[:, :, None]).astype(np.float32), -448, 448)
            ref = torch.from_numpy(quot.reshape(7, -1)).to(torch.float8_e4m3fn)
            np.testing.assert_array_equal(q, ref.view(torch.uint8).numpy())


# ---------------------------------------------------------------- weight quant

def test_weight_block_quant_ragged_and_consistent():
    rng = np.random.default_rng(6)
    N, K = 40, 96
    w = torch.from_numpy(rng.standard_normal((N, K)).astype(np.float32) * 0.02).to(torch.bfloat16)
    w[39, 5] = 3.0                      # only in the ragged second N-block
    wq, ws = oracle.quant_weight_block(w, 32, 32, ue8m0=False)
    assert ws.shape == (2, 3)
    wf = w.float().numpy()
    for nb in range(2):
        for kb in range(3):
            blk = wf[nb * 32:(nb + 1) * 32, kb * 32:(kb + 1) * 32]
            assert ws[nb, kb] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448))
    assert ws[1, 0] == np.float32(np.float32(3.0) / np.float32(448))
    # a [1, g] weight block is exactly a token group
    for ue in (False, True):
        wq1, ws1 = oracle.quant_weight_block(w, 1, 32, ue)
        xq, xs = oracle.quant_token_group(w, 32, ue)
        np.testing.assert_array_equal(wq1, xq)
        np.testing.assert_array_equal(ws1, xs)


def test_page_fact_shapes():
    facts = parse_golden("page_facts.txt")[""]
    assert [int(v) for v in facts["recipe_block32"][0]] == [1, 32, 32]
    for row in facts["ws_shape"]:
        N, K, bn, bk, r, c = (int(v) for v in row)
        w = np.zeros((N, K), dtype=np.uint16)
        _, ws = oracle.quant_weight_block(w, bn, bk, True)
        assert ws.shape == (r, c)


# ---------------------------------------------------------------- GEMM

def _rand_operands(rng, M, N, K, bn, bk, pow2):
    aq = rng.integers(0, 256, (M, K)).astype(np.uint8)
    wq = rng.integers(0, 256, (N, K)).astype(np.uint8)
    aq[(aq & 0x7F) == 0x7F] = 0x40
    wq[(wq & 0x7F) == 0x7F] = 0x38
    NB = -(-N // bn)
    if pow2:
        a_s = np.exp2(rng.integers(-10, 10, (M, K // bk))).astype(np.float32)
        ws = np.exp2(rng.integers(-10, 10, (NB, K // bk))).astype(np.float32)
    else:
        a_s = rng.uniform(0.01, 2, (M, K // bk)).astype(np.float32)
        ws = rng.uniform(0.01, 2, (NB, K // bk)).astype(np.float32)
    return aq, a_s, wq, ws


@pytest.mark.parametrize("M,N,K,bn,bk", [(5, 70, 64, 32, 32), (3, 130, 256, 128, 128),
                                          (4, 96, 256, 32, 128), (1, 8, 32, 32, 32)])
def test_gemm_brute_force_and_broadcast_formula(M, N, K, bn, bk):
    rng = np.random.default_rng(M * 1000 + N)
    aq, a_s, wq, ws = _rand_operands(rng, M, N, K, bn, bk, pow2=(bk == 32))
    d, bound = oracle.gemm(aq, a_s, wq, ws, bn, bk)
    dec = oracle.e4m3_decode
    # brute force triple loop
    ref = np.zeros((M, N))
    refb = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = accb = 0.0
            for k in range(K):
                t = (float(dec(aq[m, k])) * float(a_s[m, k // bk])) * \
                    (float(dec(wq[n, k])) * float(ws[n // bn, k // bk]))
                acc += t
                accb += abs(t)
            ref[m, n], refb[m, n] = acc, accb
    np.testing.assert_allclose(d, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    np.testing.assert_allclose(bound, refb, rtol=1e-12)
    # mm(scale_a * a, scale_b * b) with numpy-style broadcasting of the scales
    sa = np.repeat(a_s.astype(np.float64), bk, axis=1)
    sb = np.repeat(np.repeat(ws.astype(np.float64), bn, axis=0)[:N], bk, axis=1)
    mm = (sa * dec(aq)) @ (sb * dec(wq)).T
    np.testing.assert_allclose(d, mm, rtol=1e-12, atol=1e-12 * np.abs(mm).max())


def test_gemm_constant_closed_form():
    M, N, K = 3, 40, 96
    aq = np.full((M, K), 0x38, np.uint8)      # 1.0
    wq = np.full((N, K), 0x40, np.uint8)      # 2.0
    a_s = np.full((M, K // 32), 0.5, np.float32)
    ws = np.full((2, K // 32), 0.25, np.float32)
    d = oracle.gemm(aq, a_s, wq, ws, 32, 32, with_bound=False)
    assert np.all(d == K * 0.5 * 0.5)


def test_gemm_block_index_mapping():
    """Distinct power-of-two scale per block: D picks up exactly the right ones."""
    M, N, K, bn, bk = 2, 96, 128, 32, 32
    aq = np.full((M, K), 0x38, np.uint8)
    wq = np.full((N, K), 0x38, np.uint8)
    a_s = np.exp2(np.arange(M * 4).reshape(M, 4)).astype(np.float32)
    ws = np.exp2(10 + np.arange(3 * 4).reshape(3, 4)).astype(np.float32)
    d = oracle.gemm(aq, a_s, wq, ws, bn, bk, with_bound=False)
    for m in range(M):
        for n in range(N):
            want = sum(32 * a_s[m, kb] * ws[n // bn, kb] for kb in range(4))
            assert d[m, n] == want


# ---------------------------------------------------------------- per-token / per-tensor / fp8_scaled_mm
# ("Sgl project Sglang GEMM Interface": sgl_per_token_quant_fp8, sgl_per_tensor_quant_fp8, fp8_scaled_mm)

def _rand_bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def test_per_token_is_group_quant_over_the_whole_row():
    x = _rand_bf16((7, 96), 1)
    x[3] = 0.0                                     # an all-zero row: eps scale, zero codes
    q, s = oracle.quant_per_token(x)
    qg, sg = oracle.quant_token_group(x, 96, False)
    assert np.array_equal(q, qg) and np.array_equal(s, sg[:, 0])
    xf = x.float().numpy()
    amax = np.abs(xf).max(axis=1).astype(np.float32)
    want = np.maximum(amax, np.float32(oracle.EPS)) / np.float32(448.0)   # one fp32 division
    assert np.array_equal(f32_bits(s), f32_bits(want))
    assert not q[3].any()


def test_per_token_rows_are_independent():
    x = _rand_bf16((5, 64), 2)
    q, s = oracle.quant_per_token(x)
    x2 = x.clone()
    x2[1] *= 8                                     # changes only row 1
    q2, s2 = oracle.quant_per_token(x2)
    keep = [0, 2, 3, 4]
    assert np.array_equal(q[keep], q2[keep]) and np.array_equal(s[keep], s2[keep])
    assert np.array_equal(q[1], q2[1]) and s2[1] == np.float32(8) * s[1]   # exact power-of-two rescale


def test_per_tensor_dynamic_is_one_group_over_everything():
    x = _rand_bf16((6, 32), 3)
    q, s = oracle.quant_per_tensor(x)
    flat = x.reshape(1, -1)
    qg, sg = oracle.quant_token_group(flat, flat.shape[1], False)
    assert np.array_equal(q.reshape(1, -1), qg) and s[0] == sg[0, 0]


def test_per_tensor_static_uses_the_given_scale():
    x = _rand_bf16((4, 48), 4, scale=3.0)
    s = np.float32(0.0213)
    q, s_out = oracle.quant_per_tensor(x, scale=float(s))
    assert s_out[0] == s
    xf = x.float().numpy()
    want = oracle.e4m3_encode(np.clip(xf / s, -448.0, 448.0).astype(np.float32))   # fp32 division, clip, RNE
    assert np.array_equal(q, want)
    # lossless on an E4M3 grid with a power-of-two scale
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    grid = oracle.e4m3_decode(codes) * 0.25
    xb = torch.tensor(grid, dtype=torch.float32).to(torch.bfloat16)
    assert np.array_equal(xb.float().numpy(), grid.astype(np.float32))   # representable in bf16
    q2, _ = oracle.quant_per_tensor(xb.reshape(1, -1), scale=0.25)
    assert np.array_equal(oracle.e4m3_decode(q2.reshape(-1)) * 0.25, grid)


@pytest.mark.parametrize("per_row,per_col,with_bias", [(True, True, True), (False, False, False),
                                                       (True, False, True), (False, True, False)])
def test_scaled_mm_brute_force(per_row, per_col, with_bias):
    rng = np.random.default_rng(7)
    M, N, K = 3, 5, 8                              # M != N: a swapped scale vector fails
    aq = rng.integers(0, 256, size=(M, K), dtype=np.uint8)
    wq = rng.integers(0, 256, size=(N, K), dtype=np.uint8)
    aq[(aq & 0x7F) == 0x7F] = 0x10                 # no NaN codes
    wq[(wq & 0x7F) == 0x7F] = 0x22
    sa = rng.uniform(0.5, 2.0, size=M if per_row else 1).astype(np.float32)
    sb = rng.uniform(0.5, 2.0, size=N if per_col else 1).astype(np.float32)
    bias = torch.tensor(rng.uniform(-3, 3, size=N), dtype=torch.float32).to(torch.bfloat16) if with_bias else None
    d, b = oracle.scaled_mm(aq, sa, wq, sb, bias)
    dec = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    for m in range(M):
        for n in range(N):
            acc = sum(float(dec[aq[m, k]]) * float(dec[wq[n, k]]) for k in range(K))
            ref = acc * float(sa[m if per_row else 0]) * float(sb[n if per_col else 0])
            if with_bias:
                ref += float(bias[n].float())
            assert d[m, n] == pytest.approx(ref, rel=1e-13, abs=1e-13)
            bb = sum(abs(float(dec[aq[m, k]])) * abs(float(dec[wq[n, k]])) for k in range(K))
            assert b[m, n] == pytest.approx(bb * abs(float(sa[m if per_row else 0]) * float(sb[n if per_col else 0])),
                                            rel=1e-13)


def test_scaled_mm_per_tensor_equals_block_gemm_with_constant_scales():
    x = _rand_bf16((4, 64), 8)
    w = _rand_bf16((6, 64), 9, scale=0.02)
    aq, sa = oracle.quant_per_tensor(x)
    wq, sb = oracle.quant_per_tensor(w)
    d, _ = oracle.scaled_mm(aq, sa, wq, sb)
    d2, _ = oracle.gemm(aq, np.full((4, 2), sa[0], np.float32), wq, np.full((1, 2), sb[0], np.float32), 32, 32)
    assert np.allclose(d, d2, rtol=1e-12, atol=0)
    bias = _rand_bf16((6,), 10)
    db, _ = oracle.scaled_mm(aq, sa, wq, sb, bias)
    assert np.allclose(db - d, np.broadcast_to(bias.float().numpy().astype(np.float64), d.shape), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- V2 quantiser: fused SiLU-and-mul, masked M
# ("Sgl project Sglang GEMM Interface", Quantization Routines: the V2 variant of
# sgl_per_token_group_quant_8bit; Signature: fuse_silu_and_mul, masked_m)

def _ulp_diff(a, b):
    ai = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    bi = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(ai - bi)


def test_exp_within_two_ulp_and_monotone():
    xs = np.linspace(-87.0, 88.5, 20001, dtype=np.float32)
    e = oracle.exp_tc(xs)
    ref = np.exp(xs.astype(np.float64)).astype(np.float32)          # correctly rounded to fp32 (almost always)
    assert _ulp_diff(e, ref).max() <= 2
    assert np.all(np.diff(e.astype(np.float64)) >= 0)
    assert oracle.exp_tc(np.float32(0.0)) == np.float32(1.0)
    assert oracle.exp_tc(np.float32(-100.0)) == 0.0 and np.isinf(oracle.exp_tc(np.float32(100.0)))


def test_silu_identities():
    g = np.linspace(-30, 30, 4001, dtype=np.float32)
    s = oracle.silu_mul(g, 1.0)
    ref = (g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64))))
    assert np.allclose(s, ref, rtol=3e-7, atol=1e-30)
    sm = oracle.silu_mul(-g, 1.0)
    assert np.allclose(s.astype(np.float64) - sm, g.astype(np.float64), rtol=1e-6, atol=1e-6)   # silu(x)-silu(-x)=x
    big = np.array([17.0, 20.0, 100.0, 3.0e4], np.float32)
    assert np.array_equal(oracle.silu_mul(big, 1.0), big)                   # e^-g below half an ulp of 1
    assert oracle.silu_mul(np.float32(0.0), np.float32(5.0)) == 0.0
    u = np.array([0.5, -2.0, 3.0, 7.0], np.float32)
    assert np.array_equal(oracle.silu_mul(big, u), big * u)                 # exact products


def _v2_input(E, T, H, fuse, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((E, T, 2 * H if fuse else H), generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("group,ue", [(32, True), (128, False)])
def test_v2_without_fusion_or_mask_is_the_group_quantiser(group, ue):
    x = _v2_input(3, 5, 256, False, 11)
    q, s = oracle.quant_token_group_v2(x, group, ue, fuse=False)
    qg, sg = oracle.quant_token_group(x.reshape(15, 256), group, ue)
    assert np.array_equal(q.reshape(15, 256), qg) and np.array_equal(s.reshape(15, -1), sg)


def test_v2_fused_with_saturated_gate_is_the_group_quantiser_of_the_gate():
    H = 128
    gate = (torch.rand((2, 4, H), generator=torch.Generator().manual_seed(12)) * 30 + 17).to(torch.bfloat16)
    x = torch.cat([gate, torch.ones_like(gate)], dim=-1)
    q, s = oracle.quant_token_group_v2(x, 32, True, fuse=True)
    qg, sg = oracle.quant_token_group(gate.reshape(8, H), 32, True)
    assert np.array_equal(q.reshape(8, H), qg) and np.array_equal(s.reshape(8, -1), sg)


def test_v2_fused_matches_fp64_silu_mul_then_the_pinned_quantiser():
    """y from an fp64 silu(gate) * up (rounded to fp32) quantised by the pinned
    group rule: the codes agree except where the fp32 pipeline's last-ulp
    difference moves a value across an E4M3 rounding boundary (none here)."""
    E, T, H, group = 2, 3, 64, 32
    x = _v2_input(E, T, H, True, 13)
    q, s = oracle.quant_token_group_v2(x, group, False, fuse=True)
    xf = x.float().numpy().astype(np.float64)
    y = (xf[..., :H] / (1.0 + np.exp(-xf[..., :H])) * xf[..., H:]).astype(np.float32)
    for e in range(E):
        for t in range(T):
            for j in range(H // group):
                grp = y[e, t, j * group:(j + 1) * group]
                sc = oracle.group_scale(np.abs(grp).max(), False)
                assert _ulp_diff(s[e, t, j], sc) <= 2
                want = oracle.e4m3_encode(np.clip(grp / s[e, t, j], -448, 448).astype(np.float32))
                assert (q[e, t, j * group:(j + 1) * group] != want).sum() <= 1


def test_v2_masked_rows_untouched():
    E, T, H = 3, 6, 128
    x = _v2_input(E, T, H, True, 14)
    masked = np.array([0, 4, 6], np.int32)
    sentinel_q = np.full((E, T, H), 0x5A, np.uint8)
    sentinel_s = np.full((E, T, H // 32), -1.0, np.float32)
    q, s = oracle.quant_token_group_v2(x, 32, True, fuse=True, masked_m=masked, xq=sentinel_q, xs=sentinel_s)
    qa, sa = oracle.quant_token_group_v2(x, 32, True, fuse=True)
    for e in range(E):
        m = masked[e]
        assert np.array_equal(q[e, :m], qa[e, :m]) and np.array_equal(s[e, :m], sa[e, :m])
        assert (q[e, m:] == 0x5A).all() and (s[e, m:] == -1.0).all()
