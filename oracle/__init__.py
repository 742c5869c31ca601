"""CPU oracle for the W4A8 packed-linear GEMM (test infrastructure only).

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import this package. The product path (the CUDA library and its
binding) never loads it and shares no code with it.

The arithmetic lives in `egopq_oracle.c` (plain C: int64 accumulation, fp64
combination, one bf16 rounding from fp64). This module compiles it with gcc and
marshals numpy arrays; it adds no arithmetic of its own.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "egopq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libegopq_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (gcc, OpenMP, no fast-math, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, u16, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_uint16, ctypes.c_double
            lib.oracle_fp16_to_double.restype = dbl
            lib.oracle_fp16_to_double.argtypes = [u16]
            lib.oracle_bf16_to_double.restype = dbl
            lib.oracle_bf16_to_double.argtypes = [u16]
            lib.oracle_bf16_from_double.restype = u16
            lib.oracle_bf16_from_double.argtypes = [dbl]
            lib.oracle_quant_act.restype = None
            lib.oracle_quant_act.argtypes = [vp, i64, i64, i64, vp, vp, vp]
            lib.oracle_group_partials.restype = None
            lib.oracle_group_partials.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp]
            lib.oracle_w4a8.restype = None
            lib.oracle_w4a8.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, vp]
            lib.oracle_w4a16.restype = None
            lib.oracle_w4a16.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp, vp]
            lib.oracle_w8a16.restype = None
            lib.oracle_w8a16.argtypes = [vp, vp, vp, i64, i64, i64, vp, vp]
            lib.oracle_w8a8.restype = None
            lib.oracle_dequant_w4_bf16.restype = None
            lib.oracle_gptq_unpack.restype = i64
            lib.oracle_gptq_unpack.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, vp, vp]
            lib.oracle_dequant_w4_bf16.argtypes = [vp, vp, vp, i64, i64, i64, vp]
            lib.oracle_w8a8.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, vp]
            lib.oracle_packed_w4_bytes.restype = i64
            lib.oracle_packed_w4_bytes.argtypes = [i64, i64, i64]
            lib.oracle_code_location.restype = None
            lib.oracle_code_location.argtypes = [i64, i64, i64, i64, vp, vp]
            lib.oracle_pack_w4.restype = ctypes.c_int
            lib.oracle_pack_w4.argtypes = [vp, vp, vp, i64, i64, i64, vp]
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.dtype(dtype), (a.dtype, dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data


def fp16_to_double(bits: int) -> float:
    return float(_load().oracle_fp16_to_double(int(bits)))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits)))


def bf16_from_double(x: float) -> int:
    return int(_load().oracle_bf16_from_double(float(x)))


def quant_act(x_bf16: np.ndarray, group: int = 128):
    """Per-token int8 quantization: returns (a_q int8 [M,K], a_s f32 [M], asum i32 [M,G])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    a_q = np.empty((M, K), np.int8)
    a_s = np.empty((M,), np.float32)
    asum = np.empty((M, K // group), np.int32)
    _load().oracle_quant_act(_p(x), M, K, group, _p(a_q), _p(a_s), _p(asum))
    return a_q, a_s, asum


def group_partials(a_q: np.ndarray, w_q: np.ndarray, z: np.ndarray, group: int = 128):
    """Q[m,n,g] (int64)."""
    a_q, w_q, z = _c(a_q, np.int8), _c(w_q, np.uint8), _c(z, np.uint8)
    M, K = a_q.shape
    N = w_q.shape[0]
    Q = np.empty((M, N, K // group), np.int64)
    _load().oracle_group_partials(_p(a_q), _p(w_q), _p(z), M, N, K, group, _p(Q))
    return Q


def w4a8(a_q, a_s, w_q, s_f16, z, group: int = 128):
    """Returns (y64 float64 [M,N], y bf16 bits uint16 [M,N])."""
    a_q, a_s = _c(a_q, np.int8), _c(a_s, np.float32)
    w_q, s_f16, z = _c(w_q, np.uint8), _c(s_f16, np.uint16), _c(z, np.uint8)
    M, K = a_q.shape
    N = w_q.shape[0]
    y64 = np.empty((M, N), np.float64)
    y = np.empty((M, N), np.uint16)
    _load().oracle_w4a8(_p(a_q), _p(a_s), _p(w_q), _p(s_f16), _p(z), M, N, K, group,
                        _p(y64), _p(y))
    return y64, y


def w4a16(x_bf16, w_q, s_f16, z, group: int = 128):
    x, w_q, s_f16, z = _c(x_bf16, np.uint16), _c(w_q, np.uint8), _c(s_f16, np.uint16), _c(z, np.uint8)
    M, K = x.shape
    N = w_q.shape[0]
    y64 = np.empty((M, N), np.float64)
    y = np.empty((M, N), np.uint16)
    _load().oracle_w4a16(_p(x), _p(w_q), _p(s_f16), _p(z), M, N, K, group, _p(y64), _p(y))
    return y64, y


def dequant_w4_bf16(w_q, s_f16, z, group: int = 128):
    """bf16 bits [N][K] of s[n,g] * (w_q[n,k] - z[n,g]) (the dense twin's weight)."""
    w_q, s_f16, z = _c(w_q, np.uint8), _c(s_f16, np.uint16), _c(z, np.uint8)
    N, K = w_q.shape
    out = np.empty((N, K), np.uint16)
    _load().oracle_dequant_w4_bf16(_p(w_q), _p(s_f16), _p(z), N, K, group, _p(out))
    return out


def gptq_unpack(qweight, qzeros, scales, N: int, K: int, group: int = 128,
                zero_offset: int = 1):
    """GPTQ checkpoint tensors -> (w_q [N][K], s [N][G] fp16 bits, z [N][G], number of
    zero points outside [0, 15])."""
    qweight, qzeros = _c(qweight, np.int32), _c(qzeros, np.int32)
    scales = _c(scales, np.uint16)
    G = K // group
    w_q = np.empty((N, K), np.uint8)
    s = np.empty((N, G), np.uint16)
    z = np.empty((N, G), np.uint8)
    bad = _load().oracle_gptq_unpack(_p(qweight), _p(qzeros), _p(scales), N, K, group,
                                     zero_offset, _p(w_q), _p(s), _p(z))
    return w_q, s, z, int(bad)


def w8a16(x_bf16, w_q, s_f16):
    x, w_q, s_f16 = _c(x_bf16, np.uint16), _c(w_q, np.int8), _c(s_f16, np.uint16)
    M, K = x.shape
    N = w_q.shape[0]
    y64 = np.empty((M, N), np.float64)
    y = np.empty((M, N), np.uint16)
    _load().oracle_w8a16(_p(x), _p(w_q), _p(s_f16), M, N, K, _p(y64), _p(y))
    return y64, y


def w8a8(a_q, a_s, w_q, s_f16):
    """W8A8 int8-dynamic: (int64 dot [M][N], fp64 y, bf16 bits y)."""
    a_q, a_s = _c(a_q, np.int8), _c(a_s, np.float32)
    w_q, s_f16 = _c(w_q, np.int8), _c(s_f16, np.uint16)
    M, K = a_q.shape
    N = w_q.shape[0]
    dot = np.empty((M, N), np.int64)
    y64 = np.empty((M, N), np.float64)
    y = np.empty((M, N), np.uint16)
    _load().oracle_w8a8(_p(a_q), _p(a_s), _p(w_q), _p(s_f16), M, N, K, _p(dot), _p(y64), _p(y))
    return dot, y64, y


def packed_w4_bytes(N: int, K: int, group: int = 128) -> int:
    return int(_load().oracle_packed_w4_bytes(N, K, group))


def code_location(N: int, K: int, n: int, k: int):
    off = ctypes.c_int64()
    sh = ctypes.c_int()
    _load().oracle_code_location(N, K, n, k, ctypes.addressof(off), ctypes.addressof(sh))
    return off.value, sh.value


def pack_w4(w_q, s_f16, z, group: int = 128) -> np.ndarray:
    w_q, s_f16, z = _c(w_q, np.uint8), _c(s_f16, np.uint16), _c(z, np.uint8)
    N, K = w_q.shape
    nbytes = packed_w4_bytes(N, K, group)
    if nbytes == 0:
        raise ValueError(f"unsupported shape N={N} K={K} group={group}")
    out = np.empty(nbytes, np.uint8)
    rc = _load().oracle_pack_w4(_p(w_q), _p(s_f16), _p(z), N, K, group, _p(out))
    if rc:
        raise ValueError(f"oracle_pack_w4 returned {rc}")
    return out
