"""Seeded synthetic inputs shared by the CPU oracle and the CUDA path.

Test and benchmark infrastructure only. This module draws codes, zero points,
scales and activations; it holds none of the method's arithmetic. The C source
(`synth.c`) states every stream and distribution. Shapes follow the
Qwen2.5-7B-sized linears and DiT-sized blocks the benchmark uses.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lock = threading.Lock()
_lib = None

# linear index per projection, used in the per-tensor seed
LINEARS = {"q": 0, "k": 1, "v": 2, "o": 3, "gate": 4, "up": 5, "down": 6, "head": 7}
# tensor ids inside one linear
T_CODES, T_ZEROS, T_SCALES, T_ACT, T_W8, T_S8 = 0, 1, 2, 3, 4, 5


def build(force: bool = False) -> str:
    """Compile synth.c into a shared library next to it (gcc, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.synth_mix.restype = u64
            lib.synth_mix.argtypes = [u64]
            lib.synth_tensor_seed.restype = u64
            lib.synth_tensor_seed.argtypes = [i64, i64, i64, i64]
            for name, extra in [("synth_u4", []), ("synth_i8_sym", []), ("synth_normal", [])]:
                getattr(lib, name).restype = None
                getattr(lib, name).argtypes = [u64, i64, vp]
            lib.synth_scales_f16.restype = None
            lib.synth_scales_f16.argtypes = [u64, i64, dbl, dbl, dbl, vp]
            lib.synth_outlier_count.restype = i64
            lib.synth_outlier_count.argtypes = [i64, dbl]
            lib.synth_outlier_channels.restype = None
            lib.synth_outlier_channels.argtypes = [u64, i64, i64, vp]
            lib.synth_act_bf16.restype = None
            lib.synth_act_bf16.argtypes = [u64, i64, i64, dbl, dbl, vp]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def tensor_seed(config: int, layer: int, linear: int, tensor_id: int) -> int:
    return int(_load().synth_tensor_seed(config, layer, linear, tensor_id))


def mix(x: int) -> int:
    return int(_load().synth_mix(x & 0xFFFFFFFFFFFFFFFF))


def u4(seed: int, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.uint8)
    _load().synth_u4(seed, out.size, _ptr(out))
    return out


def i8_sym(seed: int, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.int8)
    _load().synth_i8_sym(seed, out.size, _ptr(out))
    return out


def normal(seed: int, shape) -> np.ndarray:
    out = np.empty(shape, dtype=np.float64)
    _load().synth_normal(seed, out.size, _ptr(out))
    return out


def scales_f16(seed: int, shape, sigma: float = 0.02, div: float = 7.0,
               add: float = 1e-4) -> np.ndarray:
    """fp16 bit patterns of |N(0, sigma)| / div + add."""
    out = np.empty(shape, dtype=np.uint16)
    _load().synth_scales_f16(seed, out.size, sigma, div, add, _ptr(out))
    return out


def outlier_count(K: int, frac: float = 0.02) -> int:
    return int(_load().synth_outlier_count(K, frac))


def outlier_channels(seed: int, K: int, frac: float = 0.02) -> np.ndarray:
    n = outlier_count(K, frac)
    out = np.empty(n, dtype=np.int64)
    if n:
        _load().synth_outlier_channels(seed, K, n, _ptr(out))
    return out


def act_bf16(seed: int, M: int, K: int, frac: float = 0.02, mult: float = 20.0) -> np.ndarray:
    """bf16 bit patterns of N(0,1) activations with outlier channels x mult."""
    out = np.empty((M, K), dtype=np.uint16)
    _load().synth_act_bf16(seed, M, K, frac, mult, _ptr(out))
    return out


class W4Weights:
    """Logical int4 group-wise asymmetric weights of one linear."""

    def __init__(self, w_q: np.ndarray, scale_f16: np.ndarray, zero: np.ndarray, group: int):
        self.w_q, self.scale_f16, self.zero, self.group = w_q, scale_f16, zero, group

    @property
    def N(self):
        return self.w_q.shape[0]

    @property
    def K(self):
        return self.w_q.shape[1]


def w4_weights(config: int, layer: int, linear: int, N: int, K: int, group: int = 128,
               sigma: float = 0.02, div: float = 7.0, add: float = 1e-4) -> W4Weights:
    """Codes and zeros uniform in [0,15]; scales fp16(|N(0,sigma)|/div + add)."""
    G = K // group
    return W4Weights(
        u4(tensor_seed(config, layer, linear, T_CODES), (N, K)),
        scales_f16(tensor_seed(config, layer, linear, T_SCALES), (N, G), sigma, div, add),
        u4(tensor_seed(config, layer, linear, T_ZEROS), (N, G)),
        group,
    )


def w8_weights(config: int, layer: int, linear: int, N: int, K: int):
    """int8 symmetric per-output-channel weights: codes uniform in [-127,127];
    scales fp16(|N(0,0.02)|/127 + 1e-4)."""
    w = i8_sym(tensor_seed(config, layer, linear, T_W8), (N, K))
    s = scales_f16(tensor_seed(config, layer, linear, T_S8), (N,), 0.02, 127.0, 1e-4)
    return w, s


def activations(config: int, layer: int, linear: int, M: int, K: int,
                outliers: bool = True) -> np.ndarray:
    seed = tensor_seed(config, layer, linear, T_ACT)
    return act_bf16(seed, M, K, 0.02 if outliers else 0.0, 20.0)
