"""The debug build (libegopq_debug.so, EGOPQ_DEBUG): the same kernels with
device-side read-index checks on the packed-record copies, the per-group scale
reads and the activation and group-sum reads.

The small oracle cases run clean under it (no check fires) on both kernel
paths. Then the packed-record checks are made to fire without any read
leaving a real buffer: egopq_debug_set_record_limit declares the packed
weight shorter than its allocation, so a failed check is seen in
egopq_device_status while every redirected read still lands inside the real
buffer."""
import numpy as np
import pytest

import oracle
import synth
from helpers import check_bf16_output, to_dev, to_host_bits, w4_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

import w4a8_quantized_gemm_gb300 as eg  # noqa: E402


@pytest.fixture()
def dbg(monkeypatch):
    """The binding bound to the debug library for one test."""
    monkeypatch.setattr(eg, "LIB_PATH", eg.DEBUG_LIB_PATH)
    monkeypatch.setattr(eg, "_lib", None)
    lib = eg.load()
    assert lib.egopq_debug_build() == 1
    lib.egopq_debug_set_record_limit(0)
    yield lib
    lib.egopq_debug_set_record_limit(0)
    eg.device_status()


def _pack(w):
    return eg.pack_w4(to_dev(w.w_q), to_dev(w.scale_f16, torch.float16), to_dev(w.zero))


@pytest.mark.parametrize("path", [eg.PATH_GEMV, eg.PATH_TC])
@pytest.mark.parametrize("M", [1, 17, 129])
def test_oracle_cases_run_clean_under_the_checks(dbg, path, M):
    N, K = 256, 512
    x, w = w4_case(0, M, N, K)
    packed = _pack(w)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    y = eg.w4a8_gemm(a, packed, N, K, path=path)
    Q = eg.w4a8_group_partials(a, packed, N, K, path=path)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, f"debug build path={path} M={M}")
    assert np.array_equal(Q.cpu().numpy(), oracle.group_partials(a_q, w.w_q, w.zero))
    y16 = eg.w4a16_gemm(to_dev(x, torch.bfloat16), packed, N, K, path=path)
    _, y16_ref = oracle.w4a16(x, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y16), y16_ref, f"debug build W4A16 path={path} M={M}")
    assert eg.device_status() == 0


@pytest.mark.parametrize("path,M", [(eg.PATH_GEMV, 2), (eg.PATH_TC, 16), (eg.PATH_TC, 130)])
def test_record_checks_fire_inside_the_real_buffer(dbg, path, M):
    N, K = 256, 512          # two row blocks x four groups = eight records
    x, w = w4_case(0, M, N, K)
    packed = _pack(w)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    eg.w4a8_gemm(a, packed, N, K, path=path)
    assert eg.device_status() == 0
    # declare only the first row block's four records: the second block's
    # reads fail their check and are redirected to record 0
    assert dbg.egopq_debug_set_record_limit(4 * 8512) == 0
    eg.w4a8_gemm(a, packed, N, K, path=path)
    assert eg.device_status() == -7
    assert b"index check" in dbg.egopq_last_error_string()
    dbg.egopq_debug_set_record_limit(0)
    y = eg.w4a8_gemm(a, packed, N, K, path=path)
    assert eg.device_status() == 0
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, "after the limit is lifted")
