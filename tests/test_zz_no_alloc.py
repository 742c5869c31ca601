"""The allocation-free one-call linear, checked against the allocating one.

egopq_w4a8_linear_noalloc exists for callers with no device allocator (a
plugin inside a framework that owns every device buffer, a serving loop that
must never enter cudaMalloc); it stages the quantized activations in a static
device array instead of a caller workspace. This file is collected last so
that a run stopping at its first failure has run everything else already; it
passes alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest

import synth
from helpers import check_bf16_output, to_dev, to_host_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

import w4a8_quantized_gemm_gb300 as eg  # noqa: E402


def _noalloc(lib, x, packed, N, y, path):
    M, K = x.shape
    return lib.egopq_w4a8_linear_noalloc(x.data_ptr(), packed.data_ptr(), M, N, K, 128,
                                         y.data_ptr(), path,
                                         torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("path,M", [(eg.PATH_AUTO, 4), (eg.PATH_TC, 48), (eg.PATH_AUTO, 130)])
def test_noalloc_matches_workspace_linear_twice(path, M):
    """Two calls in a row (different inputs, the same static array) against
    egopq_w4a8_linear with a workspace: identical bits, hence within the bar."""
    lib = eg.load()
    torch.cuda.set_device(0)
    N, K = 256, 3584
    w = synth.w4_weights(9, 0, 0, N, K)
    packed = eg.pack_w4(to_dev(w.w_q), to_dev(w.scale_f16, torch.float16), to_dev(w.zero))
    for call in range(2):
        x = to_dev(synth.activations(9, call, 0, M, K), torch.bfloat16)
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, x, packed, N, y, path) == 0, lib.egopq_last_error_string()
        ref = eg.w4a8_linear(x, packed, N, path=path)
        torch.cuda.synchronize()
        assert torch.equal(y, ref), f"call {call}"
        check_bf16_output(to_host_bits(y), to_host_bits(ref), f"noalloc call {call}")
    assert eg.device_status() == 0


def test_noalloc_refuses_staging_beyond_its_array():
    lib = eg.load()
    M, N, K = 512, 128, 18944  # about 2*M*K = 19.4 MB of staging on the tensor-core path
    assert eg.w4a8_linear_workspace_bytes(M, K, eg.PATH_TC) > 16 << 20
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    packed = torch.zeros(eg.packed_w4_bytes(N, K), dtype=torch.uint8, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, x, packed, N, y, eg.PATH_TC) == -2
    assert b"16 MiB" in lib.egopq_last_error_string()
    assert eg.device_status() == 0
