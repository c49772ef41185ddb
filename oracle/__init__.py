"""CPU oracle for the W8A8 FP8 block-scaled linear layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and it imports nothing from the product.

The arithmetic lives in ``sgq_oracle.c`` (plain C, fp64 GEMM); this module
builds it with gcc on first use and wraps it with numpy arrays:

* ``e4m3_encode`` / ``e4m3_decode`` / ``ue8m0_ceil`` -- the bit-level codec.
* ``quant_token_group`` -- per-token-group quantisation ("Sgl project Sglang
  GEMM Interface", Quantization Routines: sgl_per_token_group_quant_8bit).
* ``quant_weight_block`` -- one scale per [blk_n, blk_k] weight tile, stored
  [n_blocks, k_blocks] (vLLM scaled_mm page, XPUFp8BlockScaledMMKernel).
* ``gemm`` -- D = mm(As*Aq, (Ws*Wq)^T) in fp64 (vLLM scaled_mm page,
  AiterInt8ScaledMMLinearKernel.apply_weights docstring) plus the bound
  sum_k |a_deq||w_deq| used by the error criterion.
* ``quant_token_group_v2`` (with ``exp_tc`` / ``silu_mul``) -- the V2
  per-token-group quantiser: fused SiLU-and-mul and masked M (same page,
  Quantization Routines and Signature).
* ``ue8m0_bytes`` / ``ue8m0_values`` -- power-of-two scales as UE8M0 bytes
  (8-bit biased exponent, value 2^(e - 127), 255 = NaN), the format of the
  scale buffers the sglang PR #42604 path prepares (Modifications: "prepares
  block32 scale buffers", with UE8M0 activation rounding).
* ``quant_per_token`` / ``quant_per_tensor`` / ``scaled_mm`` -- the
  per-token and per-tensor quantisers and fp8_scaled_mm (per-tensor or per-row
  A scales, per-tensor or per-column B scales, optional bias) of "Sgl project
  Sglang GEMM Interface", Quantization Routines and Signature.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

EPS = 1e-10          # reading: the pages name eps without a value
FP8_MAX = 448.0      # OCP E4M3FN largest finite value

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgq_oracle.c")
_LIB = os.path.join(_HERE, "libsgq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available). Returns the .so path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    base = ["gcc", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-std=c11", _SRC,
            "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        cf = ctypes.c_float
        lib.sgqo_e4m3_encode.argtypes = [cf]
        lib.sgqo_e4m3_encode.restype = ctypes.c_uint8
        lib.sgqo_e4m3_encode_array.argtypes = [P, i64, P]
        lib.sgqo_e4m3_encode_array.restype = None
        lib.sgqo_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.sgqo_e4m3_decode.restype = ctypes.c_double
        lib.sgqo_ue8m0_ceil.argtypes = [cf]
        lib.sgqo_ue8m0_ceil.restype = cf
        lib.sgqo_group_scale.argtypes = [cf, cf, ci]
        lib.sgqo_group_scale.restype = cf
        lib.sgqo_quant_token_group.argtypes = [P, i64, i64, ci, ci, cf, P, P]
        lib.sgqo_quant_token_group.restype = None
        lib.sgqo_quant_weight_block.argtypes = [P, i64, i64, ci, ci, ci, cf, P, P]
        lib.sgqo_quant_weight_block.restype = None
        lib.sgqo_gemm.argtypes = [P, P, P, P, i64, i64, i64, ci, ci, ci, P, P]
        lib.sgqo_gemm.restype = None
        lib.sgqo_quant_per_token.argtypes = [P, i64, i64, cf, P, P]
        lib.sgqo_quant_per_token.restype = None
        lib.sgqo_quant_per_tensor.argtypes = [P, i64, ci, cf, P, P]
        lib.sgqo_quant_per_tensor.restype = None
        lib.sgqo_scaled_mm.argtypes = [P, P, i64, P, P, i64, P, i64, i64, i64, P, P]
        lib.sgqo_scaled_mm.restype = None
        lib.sgqo_exp_tc.argtypes = [cf]
        lib.sgqo_exp_tc.restype = cf
        lib.sgqo_silu_mul.argtypes = [cf, cf]
        lib.sgqo_silu_mul.restype = cf
        lib.sgqo_quant_token_group_v2.argtypes = [P, i64, i64, i64, ci, P, ci, ci, cf, P, P]
        lib.sgqo_quant_token_group_v2.restype = None
        lib.sgqo_num_threads.argtypes = []
        lib.sgqo_num_threads.restype = ci
        lib.sgqo_set_num_threads.argtypes = [ci]
        lib.sgqo_set_num_threads.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().sgqo_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops (n < 1: all processors); timing only."""
    _load().sgqo_set_num_threads(int(n))


def e4m3_encode(v) -> np.ndarray:
    """fp32 values -> E4M3 codes (uint8), elementwise, by the bit-level encoder."""
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    _load().sgqo_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_decode(c) -> np.ndarray:
    """E4M3 codes -> fp64 values."""
    lib = _load()
    c = np.asarray(c, dtype=np.uint8)
    table = np.array([lib.sgqo_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[c]


def ue8m0_ceil(s) -> np.ndarray:
    lib = _load()
    s = np.asarray(s, dtype=np.float32)
    return np.array([lib.sgqo_ue8m0_ceil(float(x)) for x in s.reshape(-1)],
                    dtype=np.float32).reshape(s.shape)


def ue8m0_bytes(s) -> np.ndarray:
    """fp32 scales -> UE8M0 bytes, elementwise: the biased exponent field of a
    positive normal power of two (value 2^(e - 127), e in 1 .. 254); any other
    value (not a power of two, zero, negative, subnormal, inf, NaN) -> 255,
    the format's NaN."""
    s = np.ascontiguousarray(s, dtype=np.float32)
    bits = s.view(np.uint32)
    e = (bits >> np.uint32(23)) & np.uint32(0xFF)
    exact = ((bits & np.uint32(0x807FFFFF)) == 0) & (e >= 1) & (e <= 254)
    return np.where(exact, e, 255).astype(np.uint8)


def ue8m0_values(e) -> np.ndarray:
    """UE8M0 bytes -> fp32 values 2^(e - 127); 255 -> NaN."""
    e = np.asarray(e, dtype=np.uint8).astype(np.int64)
    v = np.ldexp(np.float64(1.0), (e - 127).astype(np.int32))
    return np.where(e == 255, np.nan, v).astype(np.float32)


def group_scale(amax: float, ue8m0: bool, eps: float = EPS) -> np.float32:
    return np.float32(_load().sgqo_group_scale(float(amax), float(eps), int(ue8m0)))


def _as_bf16_bits(x) -> np.ndarray:
    """Accept a torch bf16 tensor or a uint16 array of bf16 bits."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.asarray(x)
    if a.dtype != np.uint16:
        raise TypeError("expected bf16 bits as uint16 or a torch.bfloat16 tensor")
    return np.ascontiguousarray(a)


def quant_token_group(x, group: int, ue8m0: bool, eps: float = EPS):
    """x: bf16 [M, K] -> (codes uint8 [M, K], scales fp32 [M, K/group])."""
    xb = _as_bf16_bits(x)
    M, K = xb.shape
    if K % group:
        raise ValueError("K must be a multiple of group")
    xq = np.empty((M, K), dtype=np.uint8)
    xs = np.empty((M, K // group), dtype=np.float32)
    _load().sgqo_quant_token_group(_ptr(xb), M, K, group, int(ue8m0), eps, _ptr(xq), _ptr(xs))
    return xq, xs


def quant_weight_block(w, blk_n: int, blk_k: int, ue8m0: bool, eps: float = EPS):
    """w: bf16 [N, K] -> (codes uint8 [N, K], scales fp32 [ceil(N/blk_n), K/blk_k])."""
    wb = _as_bf16_bits(w)
    N, K = wb.shape
    if K % blk_k:
        raise ValueError("K must be a multiple of blk_k")
    wq = np.empty((N, K), dtype=np.uint8)
    ws = np.empty(((N + blk_n - 1) // blk_n, K // blk_k), dtype=np.float32)
    _load().sgqo_quant_weight_block(_ptr(wb), N, K, blk_n, blk_k, int(ue8m0), eps,
                                    _ptr(wq), _ptr(ws))
    return wq, ws


def gemm(aq, a_s, wq, ws, blk_n: int, blk_k: int, a_group: int | None = None,
         with_bound: bool = True):
    """fp64 D [M, N] (and bound [M, N]) of the block-scaled product."""
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    a_s = np.ascontiguousarray(a_s, dtype=np.float32)
    ws = np.ascontiguousarray(ws, dtype=np.float32)
    M, K = aq.shape
    N = wq.shape[0]
    if a_group is None:
        a_group = K // a_s.shape[1]
    d = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64) if with_bound else None
    _load().sgqo_gemm(_ptr(aq), _ptr(a_s), _ptr(wq), _ptr(ws), M, N, K, a_group,
                      blk_n, blk_k, _ptr(d), _ptr(b) if b is not None else None)
    return (d, b) if with_bound else d


def quant_per_token(x, eps: float = EPS):
    """x: bf16 [M, K] -> (codes uint8 [M, K], scales fp32 [M]), one scale per row."""
    xb = _as_bf16_bits(x)
    M, K = xb.shape
    xq = np.empty((M, K), dtype=np.uint8)
    xs = np.empty((M,), dtype=np.float32)
    _load().sgqo_quant_per_token(_ptr(xb), M, K, eps, _ptr(xq), _ptr(xs))
    return xq, xs


def quant_per_tensor(x, scale=None, eps: float = EPS):
    """x: bf16 [...] -> (codes uint8 [...], scale fp32 [1]).  scale=None:
    dynamic (amax over the tensor); else the given static scale."""
    xb = _as_bf16_bits(x)
    xq = np.empty(xb.shape, dtype=np.uint8)
    s = np.array([0.0 if scale is None else scale], dtype=np.float32)
    _load().sgqo_quant_per_tensor(_ptr(xb), xb.size, 0 if scale is None else 1, eps, _ptr(xq), _ptr(s))
    return xq, s


def scaled_mm(aq, sa, wq, sb, bias=None, with_bound: bool = True):
    """fp64 D [M, N] = (Aq Wq^T) * sa * sb + bias (sa: 1 or M values, sb: 1 or N,
    bias: bf16 [N] or None), and the bound [M, N]."""
    aq = np.ascontiguousarray(aq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32).reshape(-1)
    sb = np.ascontiguousarray(sb, dtype=np.float32).reshape(-1)
    M, K = aq.shape
    N = wq.shape[0]
    if sa.size not in (1, M) or sb.size not in (1, N):
        raise ValueError("sa must have 1 or M values, sb 1 or N")
    bb = None if bias is None else _as_bf16_bits(bias).reshape(-1)
    d = np.empty((M, N), dtype=np.float64)
    b = np.empty((M, N), dtype=np.float64) if with_bound else None
    _load().sgqo_scaled_mm(_ptr(aq), _ptr(sa), sa.size, _ptr(wq), _ptr(sb), sb.size,
                           _ptr(bb) if bb is not None else None, M, N, K, _ptr(d),
                           _ptr(b) if b is not None else None)
    return (d, b) if with_bound else d


def exp_tc(x) -> np.ndarray:
    """fp32 exp by Cody-Waite reduction and a degree-7 Taylor polynomial (elementwise)."""
    lib = _load()
    x = np.asarray(x, dtype=np.float32)
    return np.array([lib.sgqo_exp_tc(float(v)) for v in x.reshape(-1)], dtype=np.float32).reshape(x.shape)


def silu_mul(g, u) -> np.ndarray:
    lib = _load()
    g = np.asarray(g, dtype=np.float32)
    u = np.broadcast_to(np.asarray(u, dtype=np.float32), g.shape)
    return np.array([lib.sgqo_silu_mul(float(a), float(b)) for a, b in zip(g.reshape(-1), u.reshape(-1))],
                    dtype=np.float32).reshape(g.shape)


def quant_token_group_v2(x, group: int, ue8m0: bool, fuse: bool, masked_m=None, eps: float = EPS,
                         xq=None, xs=None):
    """x: bf16 [E, T, W] (W = 2H when fuse, else H) -> (codes [E, T, H], scales [E, T, H/group]).
    Rows t >= masked_m[e] keep the contents of the given xq/xs (zeros when not given)."""
    xb = _as_bf16_bits(x)
    E, T, W = xb.shape
    H = W // 2 if fuse else W
    if H % group:
        raise ValueError("H must be a multiple of group")
    xq = np.zeros((E, T, H), dtype=np.uint8) if xq is None else np.ascontiguousarray(xq, dtype=np.uint8).copy()
    xs = np.zeros((E, T, H // group), dtype=np.float32) if xs is None else \
        np.ascontiguousarray(xs, dtype=np.float32).copy()
    mm = None if masked_m is None else np.ascontiguousarray(masked_m, dtype=np.int32)
    _load().sgqo_quant_token_group_v2(_ptr(xb), E, T, H, int(fuse), _ptr(mm) if mm is not None else None,
                                      group, int(ue8m0), eps, _ptr(xq), _ptr(xs))
    return xq, xs
