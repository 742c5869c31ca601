"""Shared test helpers: device transfer of bit patterns and the output bar.

Output bar (bf16 results): |y_gpu - y_ref| <= 1e-2 * max|y_ref| + ulp(y_ref[m,n]),
y_ref being the oracle's fp64 result rounded once to bf16 and ulp the bf16
spacing at y_ref[m,n]. Integer outputs are compared bit for bit.
"""
import numpy as np

import synth


def bf16_bits_to_f64(b) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(a)).astype(np.int64) - 7)


def check_bf16_output(y_gpu_bits: np.ndarray, y_ref_bits: np.ndarray, what: str = ""):
    """Assert the output bar; returns (max_abs_err, bound_scale)."""
    g = bf16_bits_to_f64(y_gpu_bits)
    r = bf16_bits_to_f64(y_ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    scale = np.abs(r).max() if r.size else 0.0
    tol = 1e-2 * scale + bf16_ulp(r)
    err = np.abs(g - r)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} elements over the bar; first {idx.tolist()} "
                             f"gpu={g[bad][:5]} ref={r[bad][:5]} max|ref|={scale}")
    return float(err.max()) if err.size else 0.0, scale


def to_dev(a: np.ndarray, torch_dtype=None, device="cuda"):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    t = torch.from_numpy(a).to(device)
    return t.view(torch_dtype) if torch_dtype is not None else t


def to_host_bits(t) -> np.ndarray:
    """bf16/fp16 tensor -> uint16 bit patterns."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def w4_case(config, M, N, K, layer=0, linear=0, outliers=True):
    w = synth.w4_weights(config, layer, linear, N, K)
    x = synth.activations(config, layer, linear, M, K, outliers)
    return x, w


def e4m3_to_f64(b) -> np.ndarray:
    """OCP FP8 E4M3 bytes -> float64 (bias 7, 3 mantissa bits; NaN not used here)."""
    b = np.asarray(b, np.uint8).astype(np.int64)
    sign = np.where(b >> 7, -1.0, 1.0)
    e, m = (b >> 3) & 15, b & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return sign * mag


# byte q of each aligned 8-run of the e4m3 operand planes holds K offset ORDER[q]
TC_PLANE_ORDER = np.array([0, 2, 4, 6, 1, 3, 5, 7])


def decode_tc_operand(buf: np.ndarray, M: int, K: int, e4m3_planes: bool) -> np.ndarray:
    """Integer codes [M][K] held by the tensor-core operand buffer (2*M*K bytes)
    in the form include/egopq.h documents: two e4m3 planes (a >> 4, a & 15) in
    the packed weights' nibble order when e4m3_planes, fp16 [M][K] otherwise.
    Raises if a plane value is not the integer range it must be."""
    buf = np.ascontiguousarray(buf).view(np.uint8).reshape(-1)
    assert buf.size == 2 * M * K
    if not e4m3_planes:
        return buf.view(np.float16).reshape(M, K).astype(np.float64)
    hi = e4m3_to_f64(buf[:M * K]).reshape(M, K // 8, 8)
    lo = e4m3_to_f64(buf[M * K:]).reshape(M, K // 8, 8)
    assert np.all((hi >= -8) & (hi <= 7) & (hi == np.round(hi)))
    assert np.all((lo >= 0) & (lo <= 15) & (lo == np.round(lo)))
    codes = np.empty((M, K // 8, 8))
    codes[:, :, TC_PLANE_ORDER] = 16 * hi + lo
    return codes.reshape(M, K)
