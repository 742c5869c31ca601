"""The dense bf16 twin (egopq_bf16_gemm_twin): the W4A16 tensor-core pipeline
with a copy in place of the int4 unpack, a comparison kernel ("OSCAR PR #20",
commit message: a bf16 twin of identical structure as the speed baseline).

Checked against a float64 product of the same bf16 values rounded once to
bf16 (the plain definition of a dense GEMM), and, on weights dequantized once
by egopq_dequant_w4, against the W4A16 oracle within the output bar."""
import numpy as np
import pytest

import oracle
import synth
from helpers import bf16_bits_to_f64, check_bf16_output, to_dev, to_host_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

import w4a8_quantized_gemm_gb300 as eg  # noqa: E402


def _bf16_round(v: np.ndarray) -> np.ndarray:
    return np.vectorize(oracle.bf16_from_double, otypes=[np.uint16])(v)


@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (17, 384, 1024), (130, 256, 512),
                                   (300, 128 * 80, 384)])
def test_twin_matches_dense_definition(M, N, K):
    rng = np.random.default_rng(M + N)
    x = synth.activations(13, 0, 0, M, K, outliers=False)
    # weights: bf16 values of N(0, 0.05)
    w = (rng.standard_normal((N, K)).astype(np.float32) * 0.05).view(np.uint32)
    w = ((w + 0x7FFF + ((w >> 16) & 1)) >> 16).astype(np.uint16)
    y = eg.bf16_gemm_twin(to_dev(x, torch.bfloat16), to_dev(w, torch.bfloat16))
    cols = np.arange(N) if N <= 512 else np.unique(np.concatenate(
        [np.arange(128), np.arange(N - 128, N), rng.choice(N, 256, replace=False)]))
    ref = bf16_bits_to_f64(x) @ bf16_bits_to_f64(w[cols]).T
    check_bf16_output(to_host_bits(y)[:, cols], _bf16_round(ref), f"twin M={M} N={N}")
    assert eg.device_status() == 0


@pytest.mark.parametrize("M", [65, 256])
def test_twin_on_dequantized_weights_meets_the_w4a16_bar(M):
    N, K = 512, 1024
    w = synth.w4_weights(13, 1, 0, N, K)
    x = synth.activations(13, 1, 0, M, K, outliers=False)
    packed = eg.pack_w4(to_dev(w.w_q), to_dev(w.scale_f16, torch.float16), to_dev(w.zero))
    dense = eg.dequant_w4(packed, N, K)
    y = eg.bf16_gemm_twin(to_dev(x, torch.bfloat16), dense)
    _, y_ref = oracle.w4a16(x, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, f"twin on dequantized weights M={M}")


def test_twin_refusals():
    lib = eg.load()
    x = torch.zeros((4, 512), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((256, 512), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((4, 256), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    assert lib.egopq_bf16_gemm_twin(x.data_ptr(), w.data_ptr(), 4, 256, 500, y.data_ptr(), st) == -2
    assert lib.egopq_bf16_gemm_twin(None, w.data_ptr(), 4, 256, 512, y.data_ptr(), st) == -1
    assert lib.egopq_bf16_gemm_twin(x.data_ptr(), w.data_ptr(), 0, 256, 512, y.data_ptr(), st) == 0
    assert eg.device_status() == 0
