"""Host-side checks of the C ABI: the library builds, loads and exports every
declared symbol, and argument validation answers before anything touches a
GPU.  Runs without a GPU (validation never reaches the CUDA runtime)."""
import os
import re

import pytest

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "sgq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sgq_[a-z0-9_]+)\s*\(", text)))


def test_exports_match_header(lib):
    decl = declared_symbols()
    assert set(decl) == set(binding.EXPORTS)
    for name in decl:
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in [(0, "SGQ_OK"), (1, "SGQ_ERR_INVALID_ARG"), (2, "SGQ_ERR_UNSUPPORTED"),
                       (3, "SGQ_ERR_MISALIGNED"), (4, "SGQ_ERR_CUDA"), (5, "SGQ_ERR_TIMEOUT")]:
        assert sgq.status_string(code) == name
    assert sgq.status_string(99) == "SGQ_ERR_UNKNOWN"
    assert sgq.sgq_version() == 104


A = 0x10000      # fake, 16-byte aligned device addresses: never dereferenced
B = 0x20000
C = 0x30000
D = 0x40000
E = 0x50000
S = 1            # fake stream handle; validation fails before it is used


def q(*args):
    return binding.load_library().sgq_quant_token_group(*args)


def g(*args):
    return binding.load_library().sgq_fp8_block_gemm_ex(*args)


def w(*args):
    return binding.load_library().sgq_quant_weight_block(*args)


def test_quant_validation(lib):
    INV, MIS, OK = binding.SGQ_ERR_INVALID_ARG, binding.SGQ_ERR_MISALIGNED, binding.SGQ_OK
    assert q(A, 4, 256, 64, 0, B, C, S) == INV          # group not 32/128
    assert q(A, 4, 96, 128, 0, B, C, S) == INV          # K % group
    assert q(A, -1, 256, 128, 0, B, C, S) == INV        # M < 0
    assert q(A, 4, 0, 128, 0, B, C, S) == INV           # K == 0
    assert q(A, 4, 256, 128, 2, B, C, S) == INV         # ue8m0 not 0/1
    assert q(None, 4, 256, 128, 0, B, C, S) == INV      # null
    assert q(A, 4, 256, 128, 0, None, C, S) == INV
    assert q(A + 8, 4, 256, 128, 0, B, C, S) == MIS     # misaligned
    assert q(A, 4, 256, 32, 1, B, C + 4, S) == MIS
    assert q(A, 0, 256, 128, 0, None, None, S) == OK    # M == 0: no-op


def test_weight_quant_validation(lib):
    INV, MIS, OK = binding.SGQ_ERR_INVALID_ARG, binding.SGQ_ERR_MISALIGNED, binding.SGQ_OK
    assert w(A, 256, 256, 64, 128, 1, B, C, S) == INV
    assert w(A, 256, 256, 128, 64, 1, B, C, S) == INV
    assert w(A, 256, 96, 128, 128, 1, B, C, S) == INV
    assert w(A, -3, 256, 128, 128, 1, B, C, S) == INV
    assert w(A, 256, 256, 128, 128, 1, B + 2, C, S) == MIS
    assert w(A, 0, 256, 128, 128, 1, None, None, S) == OK


def test_gemm_validation(lib):
    INV, MIS, OK = binding.SGQ_ERR_INVALID_ARG, binding.SGQ_ERR_MISALIGNED, binding.SGQ_OK
    args = lambda **k: [k.get("Aq", A), k.get("As", B), k.get("Wq", C), k.get("Ws", D), k.get("D", E),
                        k.get("M", 16), k.get("N", 256), k.get("K", 512), k.get("bn", 128),
                        k.get("bk", 128), k.get("flags", 0), S]
    assert g(*args(bn=64)) == INV
    assert g(*args(bk=256)) == INV
    assert g(*args(K=96)) == INV                 # K % blk_k
    assert g(*args(N=260)) == INV                # N % 8
    assert g(*args(N=0)) == INV
    assert g(*args(M=-1)) == INV
    assert g(*args(flags=32)) == INV             # unknown flag
    assert g(*args(flags=6)) == INV              # both issue modes at once
    assert g(*args(M=1 << 31)) == INV
    assert g(*args(Aq=None)) == INV
    assert g(*args(Ws=None)) == INV
    assert g(*args(As=B + 4)) == MIS
    assert g(*args(D=E + 8)) == MIS
    assert g(*args(M=0, Aq=None, As=None, D=None)) == OK   # M == 0: no-op
    lib = binding.load_library()
    assert lib.sgq_fp8_block_gemm(A, B, C, D, E, 16, 256, 512, 128, 64, S) == INV


def test_linear_validation(lib):
    INV, MIS, OK = binding.SGQ_ERR_INVALID_ARG, binding.SGQ_ERR_MISALIGNED, binding.SGQ_OK
    f = binding.load_library().sgq_fp8_block_linear
    args = lambda **k: [k.get("x", A), k.get("ue", 1), k.get("Wq", C), k.get("Ws", D), k.get("D", E),
                        k.get("M", 16), k.get("N", 256), k.get("K", 512), k.get("bn", 128), k.get("bk", 128),
                        k.get("xq", None), k.get("xs", None), S]
    assert f(*args(ue=2)) == INV                 # ue8m0 not 0/1
    assert f(*args(bk=64)) == INV
    assert f(*args(K=96)) == INV                 # K % blk_k
    assert f(*args(N=260)) == INV                # N % 8
    assert f(*args(xq=B)) == INV                 # xq without xs
    assert f(*args(xs=B)) == INV                 # xs without xq
    assert f(*args(x=None)) == INV
    assert f(*args(Ws=None)) == INV
    assert f(*args(x=A + 2)) == MIS
    assert f(*args(xq=B + 8, xs=B)) == MIS
    assert f(*args(M=0, x=None, D=None)) == OK   # M == 0: no-op


def test_per_token_per_tensor_scaled_mm_validation(lib):
    INV, MIS, OK = binding.SGQ_ERR_INVALID_ARG, binding.SGQ_ERR_MISALIGNED, binding.SGQ_OK
    L = binding.load_library()
    assert L.sgq_quant_per_token(A, 4, 40, B, C, S) == INV          # K % 16
    assert L.sgq_quant_per_token(A, -1, 64, B, C, S) == INV
    assert L.sgq_quant_per_token(None, 4, 64, B, C, S) == INV
    assert L.sgq_quant_per_token(A + 8, 4, 64, B, C, S) == MIS
    assert L.sgq_quant_per_token(A, 0, 64, None, None, S) == OK      # M == 0: no-op
    assert L.sgq_quant_per_tensor(A, 40, 0, B, C, S) == INV          # n % 16
    assert L.sgq_quant_per_tensor(A, 64, 2, B, C, S) == INV          # is_static not 0/1
    assert L.sgq_quant_per_tensor(A, 64, 0, B, None, S) == INV
    assert L.sgq_quant_per_tensor(A, 64, 1, B + 4, C, S) == MIS
    assert L.sgq_quant_per_tensor(A, 0, 0, None, None, S) == OK
    mm = lambda **k: L.sgq_fp8_scaled_mm(k.get("Aq", A), k.get("sa", B), k.get("sa_n", 16), k.get("Wq", C),
                                         k.get("sb", D), k.get("sb_n", 1), k.get("bias", None), k.get("D", E),
                                         k.get("M", 16), k.get("N", 256), k.get("K", 512), S)
    assert mm(K=48) == INV                       # K % 32
    assert mm(N=260) == INV                      # N % 8
    assert mm(sa_n=3) == INV                     # neither 1 nor M
    assert mm(sb_n=255) == INV                   # neither 1 nor N
    assert mm(sa=None) == INV
    assert mm(bias=E + 4) == MIS
    assert mm(M=0, Aq=None, sa=None, D=None, sa_n=1) == OK


def test_v2_quant_validation(lib):
    INV, MIS, OK = binding.SGQ_ERR_INVALID_ARG, binding.SGQ_ERR_MISALIGNED, binding.SGQ_OK
    f = binding.load_library().sgq_quant_token_group_v2
    args = lambda **k: [k.get("x", A), k.get("E", 2), k.get("T", 4), k.get("H", 256), k.get("group", 128),
                        k.get("ue", 0), k.get("fuse", 1), k.get("mask", None), k.get("xq", B), k.get("xs", C), S]
    assert f(*args(group=64)) == INV
    assert f(*args(H=80, group=32)) == INV       # H % group
    assert f(*args(ue=2)) == INV
    assert f(*args(fuse=2)) == INV
    assert f(*args(E=-1)) == INV
    assert f(*args(x=None)) == INV
    assert f(*args(mask=D + 4)) == MIS
    assert f(*args(T=0, x=None, xq=None, xs=None)) == OK


def test_binding_raises(lib):
    with pytest.raises(sgq.SgqError) as ei:
        sgq.sgq_quant_token_group(A, 4, 96, 128, 0, B, C, stream=S)
    assert ei.value.status == binding.SGQ_ERR_INVALID_ARG


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "fp8_block_scaled_sgq_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "sgq_oracle" not in src and "sgqo_" not in src, f


def test_ue8m0_entry_validation(lib):
    """The UE8M0-byte entry points check their arguments on the host before
    anything is launched (fake, never dereferenced addresses)."""
    INV, MIS, OK = binding.SGQ_ERR_INVALID_ARG, binding.SGQ_ERR_MISALIGNED, binding.SGQ_OK
    lib = binding.load_library()
    qe = lib.sgq_quant_token_group_ue8m0
    assert qe(A, 4, 256, 64, B, C, S) == INV            # group not 32/128
    assert qe(A, 4, 96, 128, B, C, S) == INV            # K % group
    assert qe(A, -1, 256, 128, B, C, S) == INV          # M < 0
    assert qe(None, 4, 256, 128, B, C, S) == INV        # null
    assert qe(A, 4, 256, 128, B, None, S) == INV
    assert qe(A, 4, 256, 32, B, C + 4, S) == MIS        # byte scales 16-byte aligned too
    assert qe(A + 8, 4, 256, 32, B, C, S) == MIS
    assert qe(A, 0, 256, 128, None, None, S) == OK      # M == 0: no-op
    se = lib.sgq_scales_to_ue8m0
    assert se(A, -1, B, S) == INV
    assert se(None, 16, B, S) == INV
    assert se(A, 16, None, S) == INV
    assert se(None, 0, None, S) == OK                   # n == 0: no-op
    ge = lib.sgq_fp8_block_gemm_ue8m0
    args = lambda **k: [k.get("Aq", A), k.get("Ae", B), k.get("Wq", C), k.get("We", D), k.get("D", E),
                        k.get("M", 16), k.get("N", 256), k.get("K", 512), k.get("bn", 128),
                        k.get("bk", 128), k.get("flags", 0), S]
    assert ge(*args(bn=64)) == INV
    assert ge(*args(K=96)) == INV                # K % blk_k
    assert ge(*args(N=260)) == INV               # N % 8
    assert ge(*args(flags=32)) == INV            # unknown flag
    assert ge(*args(flags=6)) == INV             # both issue modes at once
    assert ge(*args(M=1 << 31)) == INV
    assert ge(*args(We=None)) == INV
    assert ge(*args(Ae=B + 4)) == MIS
    assert ge(*args(D=E + 8)) == MIS
    assert ge(*args(M=0, Aq=None, Ae=None, D=None)) == OK
