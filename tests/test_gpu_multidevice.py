"""Launch state kept per device: the W4A8 linear on each visible device in turn.

The shared-memory opt-ins of the large kernels, the SM counts that size their
grids and the arch check are cached per device ordinal. A process that runs the
library on device 0 and then on device 1 must get the opt-in and the grid sizing
of device 1 there (a process-wide cache would leave device 1's large-smem
launches without their opt-in). Skipped where fewer than two devices are
visible.
"""
import numpy as np
import pytest

import oracle
from helpers import check_bf16_output, to_dev, to_host_bits, w4_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

import w4a8_quantized_gemm_gb300 as eg  # noqa: E402


def _dev_weights(w, dev):
    return (to_dev(w.w_q).to(dev), to_dev(w.scale_f16, torch.float16).to(dev),
            to_dev(w.zero).to(dev))


@pytest.mark.skipif(torch.cuda.device_count() < 2, reason="needs two visible devices")
def test_w4a8_linear_on_two_devices_in_turn():
    eg.load()
    M, K = 300, 512
    for ordinal in (0, 1, 0):
        dev = torch.device(f"cuda:{ordinal}")
        torch.cuda.set_device(dev)
        sms = torch.cuda.get_device_properties(ordinal).multi_processor_count
        N = 128 * (sms // 2)   # a wide-tile grid: the large shared-memory kernel
        x, w = w4_case(15, M, N, K)
        packed = eg.pack_w4(*_dev_weights(w, dev))
        xd = to_dev(x, torch.bfloat16).to(dev)
        y = eg.w4a8_linear(xd, packed, N, path=eg.PATH_TC)
        a_q, a_s, _ = oracle.quant_act(x)
        _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
        check_bf16_output(to_host_bits(y), y_ref, f"device {ordinal}")
        assert eg.device_status() == 0
    torch.cuda.set_device(0)
