"""GB300 (sm_103a) W4A8 packed-linear GEMM: thin Python binding of libegopq.

Argument marshalling only: every step of the path runs in the CUDA kernels of
`libegopq.so` (built in-tree by `w4a8_quantized_gemm_gb300.builder`). PyTorch
provides device memory and the current stream. There is no CPU fallback: if the
library is missing or the device is not sm_103, calls raise.

Typical use (one linear, W4A8):

    packed = pack_w4(w_q, scale_f16, zero)            # once per weight
    a = quant_act(x)                                  # per token batch
    y = w4a8_gemm(a, packed, N, K)                    # bf16 [M, N]
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import NamedTuple, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libegopq.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "egopq.h")

PATH_AUTO, PATH_GEMV, PATH_TC = 0, 1, 2
VARIANT_W4A8, VARIANT_W4A16, VARIANT_W8A16, VARIANT_W8A8 = 0, 1, 2, 3
STATUS = {0: "OK", -1: "INVALID_ARG", -2: "UNSUPPORTED_SHAPE", -3: "MISALIGNED",
          -4: "ARCH", -5: "CUDA", -6: "TIMEOUT", -7: "DEVICE_INDEX"}
DEBUG_LIB_PATH = os.path.join(_HERE, "_build", "libegopq_debug.so")
GROUP = 128

_lock = threading.Lock()
_lib = None


class EgopqError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"egopq error {code} ({STATUS.get(code, '?')}): {msg}")
        self.code = code


def build(force: bool = False) -> str:
    from . import builder
    return builder.build(force=force)


def load() -> ctypes.CDLL:
    """Load libegopq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m w4a8_quantized_gemm_gb300.builder`")
        lib = ctypes.CDLL(LIB_PATH)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        sig = {
            "egopq_version": (i32, []),
            "egopq_last_error_string": (ctypes.c_char_p, []),
            "egopq_packed_w4_bytes": (sz, [i64, i64, i32]),
            "egopq_pack_w4": (i32, [vp, vp, vp, i64, i64, i32, vp, vp]),
            "egopq_unpack_w4": (i32, [vp, i64, i64, i32, vp, vp, vp, vp]),
            "egopq_dequant_w4": (i32, [vp, i64, i64, i32, vp, vp]),
            "egopq_pack_w4_gptq": (i32, [vp, vp, vp, i64, i64, i32, i32, vp, vp]),
            "egopq_quant_act_i8": (i32, [vp, i64, i64, i32, vp, vp, vp, vp, vp]),
            "egopq_w4a8_gemm": (i32, [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, vp]),
            "egopq_w4a8_gemm_ex": (i32, [vp, vp, vp, vp, vp, i64, i64, i64, i32, vp, i32, vp]),
            "egopq_w4a8_group_partials": (i32, [vp, vp, vp, vp, i64, i64, i64, i32, vp, i32, vp]),
            "egopq_w4a16_gemm": (i32, [vp, vp, i64, i64, i64, i32, vp, vp]),
            "egopq_w4a16_gemm_ex": (i32, [vp, vp, i64, i64, i64, i32, vp, i32, vp]),
            "egopq_w8a16_gemm": (i32, [vp, vp, vp, i64, i64, i64, vp, vp]),
            "egopq_w8a16_gemm_ex": (i32, [vp, vp, vp, i64, i64, i64, vp, i32, vp]),
            "egopq_w8a8_gemm": (i32, [vp, vp, vp, vp, vp, i64, i64, i64, vp, vp]),
            "egopq_w8a8_gemm_ex": (i32, [vp, vp, vp, vp, vp, i64, i64, i64, vp, i32, vp]),
            "egopq_w4a8_linear_workspace_bytes": (sz, [i64, i64, i32, i32]),
            "egopq_w4a8_linear": (i32, [vp, vp, i64, i64, i64, i32, vp, vp, sz, i32, vp]),
            "egopq_w4a8_linear_noalloc": (i32, [vp, vp, i64, i64, i64, i32, vp, i32, vp]),
            "egopq_w4a8_gemm_grouped": (i32, [vp, vp, vp, vp, i32, vp, vp, i64, i64, i32, vp,
                                              i32, vp]),
            "egopq_w4a8_linear_grouped": (i32, [vp, i32, vp, vp, i64, i64, i32, vp, vp, sz, i32,
                                                vp]),
            "egopq_bf16_gemm_twin": (i32, [vp, vp, i64, i64, i64, vp, vp]),
            "egopq_supported": (i32, [i64, i64, i64, i32, i32]),
            "egopq_auto_path": (i32, [i64, i32]),
            "egopq_tc_operand_bytes": (sz, [i64, i64, i32]),
            "egopq_tc_operand_form": (i32, [i64]),
            "egopq_tc_token_tile": (i32, [i64, i64, i64, i32]),
            "egopq_tc_launches": (i32, [i64, i64, i64, i32]),
            "egopq_device_status": (i32, [vp]),
            "egopq_selftest_timeout": (i32, [i32, vp]),
            "egopq_debug_build": (i32, []),
            "egopq_debug_set_record_limit": (i32, [ctypes.c_uint64]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def header_functions() -> list:
    """Names of the functions include/egopq.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(egopq_[a-z0-9_]+)\s*\(", text)))


# ------------------------------------------------------------------ helpers --

def _check(rc: int):
    if rc != 0:
        raise EgopqError(rc, load().egopq_last_error_string().decode(errors="replace"))


def _stream(stream: Optional[torch.cuda.Stream] = None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _dtype(t: torch.Tensor, *dtypes):
    if t.dtype not in dtypes:
        raise TypeError(f"expected dtype in {dtypes}, got {t.dtype}")


# --------------------------------------------------------------------- API ---

def packed_w4_bytes(N: int, K: int, group: int = GROUP) -> int:
    return int(load().egopq_packed_w4_bytes(N, K, group))


def pack_w4(w_q: torch.Tensor, scale_f16: torch.Tensor, zero: torch.Tensor,
            out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """w_q uint8 [N,K] codes 0..15, scale fp16 [N,G], zero uint8 [N,G] -> packed uint8."""
    _dtype(w_q, torch.uint8)
    _dtype(scale_f16, torch.float16, torch.int16, torch.uint16)
    _dtype(zero, torch.uint8)
    N, K = w_q.shape
    nbytes = packed_w4_bytes(N, K)
    if nbytes == 0:
        raise EgopqError(-2, f"shape N={N} K={K} is not packable (K, N multiples of 128)")
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=w_q.device)
    _check(load().egopq_pack_w4(_ptr(w_q), _ptr(scale_f16), _ptr(zero), N, K, GROUP,
                                _ptr(out), _stream(stream)))
    return out


def unpack_w4(packed: torch.Tensor, N: int, K: int, stream=None):
    G = K // GROUP
    dev = packed.device
    w = torch.empty((N, K), dtype=torch.uint8, device=dev)
    s = torch.empty((N, G), dtype=torch.float16, device=dev)
    z = torch.empty((N, G), dtype=torch.uint8, device=dev)
    _check(load().egopq_unpack_w4(_ptr(packed), N, K, GROUP, _ptr(w), _ptr(s), _ptr(z),
                                  _stream(stream)))
    return w, s, z


def pack_w4_gptq(qweight: torch.Tensor, qzeros: torch.Tensor, scales: torch.Tensor,
                 zero_offset: int = 1, stream=None) -> torch.Tensor:
    """Packed weight from a GPTQ checkpoint's qweight int32 [K/8, N], qzeros
    int32 [G, N/8] and scales fp16 [G, N] (layout in include/egopq.h)."""
    _dtype(qweight, torch.int32)
    _dtype(qzeros, torch.int32)
    K, N = qweight.shape[0] * 8, qweight.shape[1]
    packed = torch.empty(packed_w4_bytes(N, K), dtype=torch.uint8, device=qweight.device)
    _check(load().egopq_pack_w4_gptq(_ptr(qweight), _ptr(qzeros), _ptr(scales), N, K, GROUP,
                                     zero_offset, _ptr(packed), _stream(stream)))
    return packed


def dequant_w4(packed: torch.Tensor, N: int, K: int, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """The packed weight dequantized once to dense bf16 [N, K]."""
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=packed.device)
    _check(load().egopq_dequant_w4(_ptr(packed), N, K, GROUP, _ptr(out), _stream(stream)))
    return out


class QuantAct(NamedTuple):
    # int8 [M, K], or None when the codes were written only in the tensor-core
    # operand form (all the tensor-core path reads)
    a_q: Optional[torch.Tensor]
    a_s: torch.Tensor      # fp32 [M]
    a_gsum: torch.Tensor   # int32 [M, G]
    # uint8: the codes in the tensor-core operand form the library picks for
    # this M (tc_operand_form; layout in include/egopq.h), or None
    a_tc: Optional[torch.Tensor]


TC_FORM_E4M3_PLANES, TC_FORM_F16 = 1, 2


def auto_path(M: int, variant: int = VARIANT_W4A8) -> int:
    """The path (PATH_GEMV or PATH_TC) the library's AUTO choice takes for M
    tokens of `variant`."""
    rc = int(load().egopq_auto_path(M, variant))
    if rc < 0:
        _check(rc)
    return rc


def tc_token_tile(M: int, N: int, K: int, variant: int = VARIANT_W4A8) -> int:
    """Tokens per output tile (the MMA's N) the tensor-core path runs an
    M x N x K call of `variant` with on the current device."""
    rc = int(load().egopq_tc_token_tile(M, N, K, variant))
    if rc < 0:
        _check(rc)
    return rc


def tc_launches(M: int, N: int, K: int, variant: int = VARIANT_W4A8) -> int:
    """Kernel launches (1 or 2) the tensor-core path makes for an M x N x K
    call of `variant` on the current device."""
    rc = int(load().egopq_tc_launches(M, N, K, variant))
    if rc < 0:
        _check(rc)
    return rc


def tc_operand_form(M: int) -> int:
    """TC_FORM_E4M3_PLANES or TC_FORM_F16: the form quant_act writes the
    tensor-core operand in for M tokens."""
    rc = int(load().egopq_tc_operand_form(M))
    if rc < 0:
        _check(rc)
    return rc


def tc_operand(M: int, K: int, device) -> torch.Tensor:
    """A buffer for the tensor-core operand form of M x K codes (empty for an
    empty batch)."""
    if M == 0:
        return torch.empty((0,), dtype=torch.uint8, device=device)
    nbytes = int(load().egopq_tc_operand_bytes(M, K, GROUP))
    if nbytes == 0:
        raise EgopqError(-2, f"no tensor-core operand for M={M} K={K}")
    return torch.empty((nbytes,), dtype=torch.uint8, device=device)


def quant_act(x: torch.Tensor, with_tc: bool = True, out: Optional[QuantAct] = None,
              stream=None, with_codes: bool = True) -> QuantAct:
    """Per-token symmetric int8 quantization of bf16 x [M, K]. with_codes=False
    leaves the int8 codes out (a_q None): only the tensor-core path can read
    the result."""
    _dtype(x, torch.bfloat16, torch.int16, torch.uint16)
    M, K = x.shape
    if out is None:
        dev = x.device
        out = QuantAct(torch.empty((M, K), dtype=torch.int8, device=dev) if with_codes else None,
                       torch.empty((M,), dtype=torch.float32, device=dev),
                       torch.empty((M, max(K // GROUP, 1)), dtype=torch.int32, device=dev),
                       tc_operand(M, K, dev) if with_tc else None)
    _check(load().egopq_quant_act_i8(_ptr(x), M, K, GROUP, _ptr(out.a_q), _ptr(out.a_s),
                                     _ptr(out.a_gsum), _ptr(out.a_tc), _stream(stream)))
    return out


def w4a8_gemm(a: QuantAct, packed: torch.Tensor, N: int, K: int, path: int = PATH_AUTO,
              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    M = a.a_s.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.a_s.device)
    _check(load().egopq_w4a8_gemm_ex(_ptr(a.a_q), _ptr(a.a_tc), _ptr(a.a_s), _ptr(a.a_gsum),
                                     _ptr(packed), M, N, K, GROUP, _ptr(out), path,
                                     _stream(stream)))
    return out


def w4a8_linear_workspace_bytes(M: int, K: int, path: int = PATH_AUTO) -> int:
    return int(load().egopq_w4a8_linear_workspace_bytes(M, K, GROUP, path))


def w4a8_linear(x: torch.Tensor, packed: torch.Tensor, N: int, path: int = PATH_AUTO,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """One-call W4A8 linear from bf16 x [M, K]: per-token int8 quantization into
    a workspace, then the W4A8 GEMM (two kernels, one call)."""
    _dtype(x, torch.bfloat16)
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    need = w4a8_linear_workspace_bytes(M, K, path)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().egopq_w4a8_linear(_ptr(x), _ptr(packed), M, N, K, GROUP, _ptr(out),
                                    _ptr(workspace), ws_bytes, path, _stream(stream)))
    return out


class _Group:
    """Host arrays (packed pointers, row counts, output pointers) of sibling
    linears for the grouped calls; built once, reused by every call."""

    def __init__(self, packed, N, outs):
        n = len(packed)
        if not (1 <= n <= 8) or len(N) != n or len(outs) != n:
            raise ValueError("1 to 8 linears, with one N and one output each")
        self.count = n
        self.packed = (ctypes.c_void_p * n)(*[_ptr(p) for p in packed])
        self.N = (ctypes.c_int64 * n)(*[int(v) for v in N])
        self.y = (ctypes.c_void_p * n)(*[_ptr(o) for o in outs])


def _grouped_outputs(M, N, device, out):
    if out is None:
        out = [torch.empty((M, n), dtype=torch.bfloat16, device=device) for n in N]
    for o, n in zip(out, N):
        _dtype(o, torch.bfloat16)
        if tuple(o.shape) != (M, n):
            raise ValueError(f"output of shape {tuple(o.shape)}, expected {(M, n)}")
    return out


def w4a8_gemm_grouped(a: QuantAct, packed: list, N: list, K: int, path: int = PATH_AUTO,
                      out: Optional[list] = None, stream=None) -> list:
    """Sibling linears sharing the activations `a` (q|k|v, gate|up) in one
    launch: returns [y_j bf16 [M, N_j]]."""
    M = a.a_s.shape[0]
    out = _grouped_outputs(M, N, a.a_s.device, out)
    g = _Group(packed, N, out)
    _check(load().egopq_w4a8_gemm_grouped(_ptr(a.a_q), _ptr(a.a_tc), _ptr(a.a_s), _ptr(a.a_gsum),
                                          g.count, g.packed, g.N, M, K, GROUP, g.y, path,
                                          _stream(stream)))
    return out


def w4a8_linear_grouped(x: torch.Tensor, packed: list, N: list, path: int = PATH_AUTO,
                        out: Optional[list] = None, workspace: Optional[torch.Tensor] = None,
                        stream=None) -> list:
    """One quantization of bf16 x [M, K] and one grouped GEMM over the sibling
    weights: returns [y_j bf16 [M, N_j]]."""
    _dtype(x, torch.bfloat16)
    M, K = x.shape
    out = _grouped_outputs(M, N, x.device, out)
    need = w4a8_linear_workspace_bytes(M, K, path)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    g = _Group(packed, N, out)
    _check(load().egopq_w4a8_linear_grouped(_ptr(x), g.count, g.packed, g.N, M, K, GROUP, g.y,
                                            _ptr(workspace), workspace.numel(), path,
                                            _stream(stream)))
    return out


def w4a8_group_partials(a: QuantAct, packed: torch.Tensor, N: int, K: int,
                        path: int = PATH_TC, stream=None) -> torch.Tensor:
    M = a.a_s.shape[0]
    Q = torch.empty((M, N, K // GROUP), dtype=torch.int32, device=a.a_s.device)
    _check(load().egopq_w4a8_group_partials(_ptr(a.a_q), _ptr(a.a_tc), _ptr(a.a_gsum),
                                            _ptr(packed), M, N, K, GROUP, _ptr(Q), path,
                                            _stream(stream)))
    return Q


def w4a16_gemm(x: torch.Tensor, packed: torch.Tensor, N: int, K: int, path: int = PATH_AUTO,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    _dtype(x, torch.bfloat16)
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().egopq_w4a16_gemm_ex(_ptr(x), _ptr(packed), M, N, K, GROUP, _ptr(out), path,
                                      _stream(stream)))
    return out


def w8a16_gemm(x: torch.Tensor, w_q: torch.Tensor, scale_f16: torch.Tensor,
               path: int = PATH_AUTO, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    _dtype(x, torch.bfloat16)
    _dtype(w_q, torch.int8)
    M, K = x.shape
    N = w_q.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().egopq_w8a16_gemm_ex(_ptr(x), _ptr(w_q), _ptr(scale_f16), M, N, K, _ptr(out),
                                      path, _stream(stream)))
    return out


def w8a8_gemm(a: QuantAct, w_q: torch.Tensor, scale_f16: torch.Tensor, path: int = PATH_AUTO,
              out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """W8A8 int8-dynamic GEMM: per-token int8 activations (from quant_act; a_tc
    is read on the tensor-core path only) times int8 weights [N, K] with fp16
    per-channel scales [N]."""
    _dtype(w_q, torch.int8)
    M = a.a_s.shape[0]
    N, K = w_q.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.a_s.device)
    _check(load().egopq_w8a8_gemm_ex(_ptr(a.a_q), _ptr(a.a_tc), _ptr(a.a_s), _ptr(w_q),
                                     _ptr(scale_f16), M, N, K, _ptr(out), path,
                                     _stream(stream)))
    return out


def bf16_gemm_twin(x: torch.Tensor, w: torch.Tensor, out: Optional[torch.Tensor] = None,
                   stream=None) -> torch.Tensor:
    """Dense bf16 x [M, K] times w [N, K] through the W4A16 tensor-core
    pipeline with a copy in place of the int4 unpack (comparison kernel)."""
    _dtype(x, torch.bfloat16)
    _dtype(w, torch.bfloat16)
    M, K = x.shape
    N = w.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().egopq_bf16_gemm_twin(_ptr(x), _ptr(w), M, N, K, _ptr(out), _stream(stream)))
    return out


def supported(M: int, N: int, K: int, variant: int = VARIANT_W4A8, group: int = GROUP) -> bool:
    return bool(load().egopq_supported(M, N, K, group, variant))


def device_status(stream=None) -> int:
    """Synchronize and return (and clear) the device error status code."""
    return int(load().egopq_device_status(_stream(stream)))


def selftest_timeout(timeout_us: int, stream=None) -> None:
    _check(load().egopq_selftest_timeout(timeout_us, _stream(stream)))


def version() -> int:
    return int(load().egopq_version())
