"""ctypes binding of ``libsgq.so`` -- argument marshalling only.

Each function has the name and argument order of the C call in
``include/sgq.h``.  Tensor arguments may be torch CUDA tensors (their
``data_ptr()`` is passed) or raw integer device addresses; ``stream`` may be a
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None for the current
torch stream.  A non-OK status raises :class:`SgqError`.  There is no
fallback: if the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsgq.so")

SGQ_OK = 0
SGQ_ERR_INVALID_ARG = 1
SGQ_ERR_UNSUPPORTED = 2
SGQ_ERR_MISALIGNED = 3
SGQ_ERR_CUDA = 4
SGQ_ERR_TIMEOUT = 5

SGQ_GEMM_DEFAULT = 0
SGQ_GEMM_FORCE_PROMOTE = 1
SGQ_GEMM_ISSUE_ALT = 2
SGQ_GEMM_ISSUE_SINGLE = 4
SGQ_GEMM_TEST_TIMEOUT = 8
SGQ_GEMM_SCALES_POW2 = 16

# Symbols declared in include/sgq.h (checked by the tests).
EXPORTS = (
    "sgq_quant_token_group",
    "sgq_quant_weight_block",
    "sgq_fp8_block_gemm",
    "sgq_fp8_block_gemm_ex",
    "sgq_fp8_block_gemm_noalloc",
    "sgq_fp8_block_gemm_ue8m0",
    "sgq_quant_token_group_ue8m0",
    "sgq_scales_to_ue8m0",
    "sgq_fp8_block_linear",
    "sgq_quant_token_group_v2",
    "sgq_quant_per_token",
    "sgq_quant_per_tensor",
    "sgq_fp8_scaled_mm",
    "sgq_status_string",
    "sgq_device_status",
    "sgq_launch_count",
    "sgq_allocated_bytes",
    "sgq_gemm_plan",
    "sgq_gemm_plan_pow2",
    "sgq_version",
)


class SgqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libsgq.so (built by ``fp8_block_scaled_sgq_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA extension not built: {path} is missing "
                               "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        lib = ctypes.CDLL(path)
        P, i64, ci, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
        lib.sgq_quant_token_group.argtypes = [P, i64, i64, ci, ci, P, P, P]
        lib.sgq_quant_weight_block.argtypes = [P, i64, i64, ci, ci, ci, P, P, P]
        lib.sgq_fp8_block_gemm.argtypes = [P, P, P, P, P, i64, i64, i64, ci, ci, P]
        lib.sgq_fp8_block_gemm_ex.argtypes = [P, P, P, P, P, i64, i64, i64, ci, ci, u32, P]
        lib.sgq_fp8_block_gemm_noalloc.argtypes = [P, P, P, P, P, i64, i64, i64, ci, ci, P]
        lib.sgq_fp8_block_gemm_ue8m0.argtypes = [P, P, P, P, P, i64, i64, i64, ci, ci, u32, P]
        lib.sgq_quant_token_group_ue8m0.argtypes = [P, i64, i64, ci, P, P, P]
        lib.sgq_scales_to_ue8m0.argtypes = [P, i64, P, P]
        lib.sgq_fp8_block_linear.argtypes = [P, ci, P, P, P, i64, i64, i64, ci, ci, P, P, P]
        lib.sgq_quant_token_group_v2.argtypes = [P, i64, i64, i64, ci, ci, ci, P, P, P, P]
        lib.sgq_quant_per_token.argtypes = [P, i64, i64, P, P, P]
        lib.sgq_quant_per_tensor.argtypes = [P, i64, ci, P, P, P]
        lib.sgq_fp8_scaled_mm.argtypes = [P, P, i64, P, P, i64, P, P, i64, i64, i64, P]
        for f in ("sgq_quant_token_group", "sgq_quant_weight_block", "sgq_fp8_block_gemm",
                  "sgq_fp8_block_gemm_ex", "sgq_fp8_block_gemm_noalloc", "sgq_fp8_block_linear",
                  "sgq_fp8_block_gemm_ue8m0", "sgq_quant_token_group_ue8m0", "sgq_scales_to_ue8m0",
                  "sgq_quant_per_token", "sgq_quant_per_tensor", "sgq_fp8_scaled_mm", "sgq_quant_token_group_v2"):
            getattr(lib, f).restype = ci
        lib.sgq_status_string.argtypes = [ci]
        lib.sgq_status_string.restype = ctypes.c_char_p
        lib.sgq_device_status.argtypes = [P]
        lib.sgq_device_status.restype = ci
        lib.sgq_launch_count.argtypes = []
        lib.sgq_launch_count.restype = ctypes.c_uint64
        lib.sgq_allocated_bytes.argtypes = []
        lib.sgq_allocated_bytes.restype = ctypes.c_uint64
        lib.sgq_gemm_plan.argtypes = [i64, i64, i64, ci, ci, P]
        lib.sgq_gemm_plan.restype = ci
        lib.sgq_gemm_plan_pow2.argtypes = [i64, i64, i64, ci, ci, ci, P]
        lib.sgq_gemm_plan_pow2.restype = ci
        lib.sgq_version.argtypes = []
        lib.sgq_version.restype = ci
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    raise TypeError(f"expected a tensor or an int address, got {type(t)!r}")


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int, what: str):
    if rc != SGQ_OK:
        raise SgqError(rc, what)


def status_string(status: int) -> str:
    return load_library().sgq_status_string(status).decode()


def sgq_quant_token_group(x, M, K, group, ue8m0, xq, xs, stream=None):
    _check(load_library().sgq_quant_token_group(_ptr(x), M, K, group, int(ue8m0), _ptr(xq), _ptr(xs),
                                                _stream(stream)), "sgq_quant_token_group")


def sgq_quant_weight_block(w, N, K, blk_n, blk_k, ue8m0, wq, ws, stream=None):
    _check(load_library().sgq_quant_weight_block(_ptr(w), N, K, blk_n, blk_k, int(ue8m0), _ptr(wq),
                                                 _ptr(ws), _stream(stream)), "sgq_quant_weight_block")


def sgq_fp8_block_gemm(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k, stream=None):
    _check(load_library().sgq_fp8_block_gemm(_ptr(Aq), _ptr(As), _ptr(Wq), _ptr(Ws), _ptr(D), M, N, K,
                                             blk_n, blk_k, _stream(stream)), "sgq_fp8_block_gemm")


def sgq_fp8_block_gemm_ex(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k, flags, stream=None):
    _check(load_library().sgq_fp8_block_gemm_ex(_ptr(Aq), _ptr(As), _ptr(Wq), _ptr(Ws), _ptr(D), M, N,
                                                K, blk_n, blk_k, flags, _stream(stream)),
           "sgq_fp8_block_gemm_ex")


def sgq_fp8_block_gemm_noalloc(Aq, As, Wq, Ws, D, M, N, K, blk_n, blk_k, stream=None):
    """The GEMM with its split-K scratch in the library's fixed device array
    (for callers that cannot let the library allocate device memory)."""
    _check(load_library().sgq_fp8_block_gemm_noalloc(_ptr(Aq), _ptr(As), _ptr(Wq), _ptr(Ws), _ptr(D), M, N,
                                                     K, blk_n, blk_k, _stream(stream)),
           "sgq_fp8_block_gemm_noalloc")


def sgq_fp8_block_gemm_ue8m0(Aq, Ae, Wq, We, D, M, N, K, blk_n, blk_k, flags=0, stream=None):
    """The GEMM with UE8M0 scale bytes (uint8 tensors) in place of fp32 scales."""
    _check(load_library().sgq_fp8_block_gemm_ue8m0(_ptr(Aq), _ptr(Ae), _ptr(Wq), _ptr(We), _ptr(D), M, N, K,
                                                   blk_n, blk_k, flags, _stream(stream)),
           "sgq_fp8_block_gemm_ue8m0")


def sgq_quant_token_group_ue8m0(x, M, K, group, xq, xe, stream=None):
    _check(load_library().sgq_quant_token_group_ue8m0(_ptr(x), M, K, group, _ptr(xq), _ptr(xe), _stream(stream)),
           "sgq_quant_token_group_ue8m0")


def sgq_scales_to_ue8m0(s, n, e, stream=None):
    _check(load_library().sgq_scales_to_ue8m0(_ptr(s), n, _ptr(e), _stream(stream)), "sgq_scales_to_ue8m0")


def sgq_fp8_block_linear(x, ue8m0, Wq, Ws, D, M, N, K, blk_n, blk_k, xq=None, xs=None, stream=None):
    """Quantise-and-multiply (one kernel at decode-sized M); xq/xs optional outputs."""
    _check(load_library().sgq_fp8_block_linear(_ptr(x), int(ue8m0), _ptr(Wq), _ptr(Ws), _ptr(D), M, N, K,
                                               blk_n, blk_k, _ptr(xq), _ptr(xs), _stream(stream)),
           "sgq_fp8_block_linear")


def sgq_quant_token_group_v2(x, E, T, H, group, ue8m0, fuse, masked_m, xq, xs, stream=None):
    _check(load_library().sgq_quant_token_group_v2(_ptr(x), E, T, H, group, int(ue8m0), int(fuse), _ptr(masked_m),
                                                   _ptr(xq), _ptr(xs), _stream(stream)),
           "sgq_quant_token_group_v2")


def sgq_quant_per_token(x, M, K, xq, xs, stream=None):
    _check(load_library().sgq_quant_per_token(_ptr(x), M, K, _ptr(xq), _ptr(xs), _stream(stream)),
           "sgq_quant_per_token")


def sgq_quant_per_tensor(x, n, is_static, xq, xs, stream=None):
    _check(load_library().sgq_quant_per_tensor(_ptr(x), n, int(is_static), _ptr(xq), _ptr(xs), _stream(stream)),
           "sgq_quant_per_tensor")


def sgq_fp8_scaled_mm(Aq, sa, sa_n, Wq, sb, sb_n, bias, D, M, N, K, stream=None):
    _check(load_library().sgq_fp8_scaled_mm(_ptr(Aq), _ptr(sa), sa_n, _ptr(Wq), _ptr(sb), sb_n, _ptr(bias),
                                            _ptr(D), M, N, K, _stream(stream)),
           "sgq_fp8_scaled_mm")


def sgq_device_status(stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device status code."""
    return int(load_library().sgq_device_status(_stream(stream)))


def sgq_launch_count() -> int:
    return int(load_library().sgq_launch_count())


def sgq_allocated_bytes() -> int:
    return int(load_library().sgq_allocated_bytes())


def sgq_version() -> int:
    return int(load_library().sgq_version())


PLAN_FIELDS = ("swap", "bn", "splits", "items", "grid", "alt", "ck", "pair")


def sgq_gemm_plan(M, N, K, blk_k, sm_count=152) -> dict:
    """The GEMM's launch plan for this problem (host only; see include/sgq.h)."""
    out = (ctypes.c_int32 * 8)()
    _check(load_library().sgq_gemm_plan(M, N, K, blk_k, sm_count, ctypes.cast(out, ctypes.c_void_p)),
           "sgq_gemm_plan")
    return dict(zip(PLAN_FIELDS, (int(v) for v in out)))


PLAN_POW2_FIELDS = ("mode", "bn", "splits", "items", "grid", "tiles", "kps")


def sgq_gemm_plan_pow2(M, N, K, blk_k, sm_count=152, e8=False) -> dict:
    """The two-accumulator plan under the power-of-two promise (host only; see include/sgq.h)."""
    out = (ctypes.c_int32 * 8)()
    _check(load_library().sgq_gemm_plan_pow2(M, N, K, blk_k, sm_count, int(bool(e8)), ctypes.cast(out, ctypes.c_void_p)),
           "sgq_gemm_plan_pow2")
    return dict(zip(PLAN_POW2_FIELDS, (int(v) for v in out)))
