"""GPU parity of the 192-token tensor-core tiles (the full-rate wide tile: two
TMEM accumulators; two converter sets splitting each group's K, two
alternating MMA issuers and the drain warps meeting on hardware named
barriers) against the CPU oracle.

The library picks 192 or 128 tokens per tile from the grid each makes on the
device's SMs (egopq_tc_token_tile). The shapes below are built from the SM
count so that the 192-token grid has fewer rounds and is chosen: a persistent
grid of exactly one round with a ragged token tail, a persistent grid of two
rounds (several tiles per CTA: the double-buffered epilogue staging), and a
split-K grid (cluster reduction of 192 x 128 partial sums). Outputs are
compared in full; group partials bit for bit, worst-case magnitudes included.
"""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    eg.load()
    torch.cuda.set_device(0)
    yield
    assert eg.device_status() == 0


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _shape(case):
    """(M, N, K) whose 192-token grid needs fewer rounds than the 128-token one."""
    sms = _sms()
    if case == "one_round":      # 2 x sms/2 tiles of 192 (1 round) against 3 x sms/2 of 128
        return 300, 128 * (sms // 2), 512
    if case == "two_rounds":     # 6 m-tiles of 192 (last: 40 tokens) against 8 of 128
        return 1000, 128 * (sms // 3), 1024
    if case == "split_k":        # 2 m-tiles of 192 small enough to split K in two
        return 384, 128 * (sms * 2 // 9), 1024
    raise ValueError(case)


def _dev_weights(w):
    return (to_dev(w.w_q), to_dev(w.scale_f16, torch.float16), to_dev(w.zero))


@pytest.mark.parametrize("case", ["one_round", "two_rounds", "split_k"])
def test_w4a8_full_tile_output(case):
    M, N, K = _shape(case)
    assert eg.tc_token_tile(M, N, K) == 192, (case, M, N, K)
    x, w = w4_case(11, M, N, K)
    packed = eg.pack_w4(*_dev_weights(w))
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    y = eg.w4a8_gemm(a, packed, N, K, path=eg.PATH_TC)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, f"192-token tiles {case} M={M} N={N} K={K}")


@pytest.mark.parametrize("M", [384, 256])    # 192-token tiles; 128-token tiles
def test_w4a8_split_tail_output(M):
    """Persistent grids whose last round would hold a few tiles of a long K:
    those tiles run as a second launch with K split over clusters (each rank
    reducing a slice of the tile's columns). 2 m-tiles x (SMs + 2 or + 3)
    n-tiles, 64 groups each: two full rounds, then the last n-tiles (every
    m-tile) of the banded order split 8 ways; compared on the first, some
    middle and the last 384 output columns (the split tiles)."""
    sms = _sms()
    N, K = 128 * (sms + (2 if M == 384 else 3)), 8192
    assert eg.tc_token_tile(M, N, K) == (192 if M == 384 else 128)
    assert eg.tc_launches(M, N, K) == 2
    x, w = w4_case(17, M, N, K)
    packed = eg.pack_w4(*_dev_weights(w))
    y = eg.w4a8_linear(to_dev(x, torch.bfloat16), packed, N, path=eg.PATH_TC)
    rng = np.random.default_rng(M)
    cols = np.unique(np.concatenate([np.arange(128), rng.choice(N, 256, replace=False),
                                     np.arange(N - 384, N)]))
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q[cols], w.scale_f16[cols], w.zero[cols])
    check_bf16_output(to_host_bits(y)[:, cols], y_ref, f"split tail M={M} N={N} K={K}")


@pytest.mark.parametrize("case", ["one_round", "split_k"])
def test_w4a8_full_tile_group_partials(case):
    M, N, K = _shape(case)
    x, w = w4_case(12, M, N, K)
    packed = eg.pack_w4(*_dev_weights(w))
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    Q = eg.w4a8_group_partials(a, packed, N, K, path=eg.PATH_TC).cpu().numpy()
    a_q, _, _ = oracle.quant_act(x)
    rows = np.array([0, 1, 190, 191, 192, 193, M - 1])
    assert np.array_equal(Q[rows], oracle.group_partials(a_q[rows], w.w_q, w.zero))


@pytest.mark.parametrize("case", ["max_pos", "alternating"])
def test_w4a8_full_tile_worst_case_magnitudes(case):
    """|Q| = 128 * 127 * 15 = 243840 in 192-token tiles: still exact in fp32."""
    M, N, K = _shape("one_round")
    G = K // 128
    x = np.full((M, K), 0x3F80, np.uint16)                     # 1.0 -> a_q = 127
    w_q = np.full((N, K), 15, np.uint8)
    z = np.zeros((N, G), np.uint8)
    if case == "alternating":
        x[:, 1::2] = 0xBF80                                    # -1.0 -> a_q = -127
        w_q[:, 1::2] = 0
        w_q[::2, :] = 15 - w_q[::2, :]
        z[:, :] = np.arange(N)[:, None] % 16
    s = np.full((N, G), 0x3C00, np.uint16)
    w = synth.W4Weights(w_q, s, z, 128)
    packed = eg.pack_w4(*_dev_weights(w))
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    Q = eg.w4a8_group_partials(a, packed, N, K, path=eg.PATH_TC).cpu().numpy()
    a_q, _, _ = oracle.quant_act(x)
    rows = np.array([0, 191, 192, M - 1])
    ref = oracle.group_partials(a_q[rows], w_q, z)
    if case == "max_pos":
        assert ref.max() == 243840
    assert np.array_equal(Q[rows], ref)


def test_w4a16_full_tile_output():
    M, N, K = _shape("one_round")
    assert eg.tc_token_tile(M, N, K, eg.VARIANT_W4A16) == 192
    x = synth.activations(13, 0, 0, M, K, outliers=False)
    w = synth.w4_weights(13, 0, 0, N, K)
    y = eg.w4a16_gemm(to_dev(x, torch.bfloat16), eg.pack_w4(*_dev_weights(w)), N, K,
                      path=eg.PATH_TC)
    _, y_ref = oracle.w4a16(x, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, "W4A16 192-token tiles")


@pytest.mark.parametrize("case", ["one_round", "two_rounds", "split_k"])
def test_w8a16_full_tile_output(case):
    """W8A16 on 192-token tiles (all of K accumulated in a 192-column TMEM
    accumulator, two accumulators and two A buffers): one persistent round with
    a ragged token tail, two rounds, and a split-K grid (cluster reduction)."""
    M, N, K = _shape(case)
    assert eg.tc_token_tile(M, N, K, eg.VARIANT_W8A16) == 192, (case, M, N, K)
    x = synth.activations(18, 0, 0, M, K, outliers=False)
    w8, s8 = synth.w8_weights(18, 0, 0, N, K)
    y = eg.w8a16_gemm(to_dev(x, torch.bfloat16), to_dev(w8), to_dev(s8, torch.float16),
                      path=eg.PATH_TC)
    _, y_ref = oracle.w8a16(x, w8, s8)
    check_bf16_output(to_host_bits(y), y_ref, f"W8A16 192-token tiles {case}")


@pytest.mark.parametrize("case", ["one_round", "two_rounds", "split_k"])
def test_w8a8_full_tile_output(case):
    """W8A8 on 192-token tiles (partials of 8 groups exact in fp32, added as
    int32): the same three grid forms."""
    M, N, K = _shape(case)
    assert eg.tc_token_tile(M, N, K, eg.VARIANT_W8A8) == 192, (case, M, N, K)
    x = synth.activations(19, 0, 0, M, K)
    w8, s8 = synth.w8_weights(19, 0, 0, N, K)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    y = eg.w8a8_gemm(a, to_dev(w8), to_dev(s8, torch.float16), path=eg.PATH_TC)
    a_q, a_s, _ = oracle.quant_act(x)
    _, _, y_ref = oracle.w8a8(a_q, a_s, w8, s8)
    check_bf16_output(to_host_bits(y), y_ref, f"W8A8 192-token tiles {case}")


def test_w8a8_full_tile_integer_case_bit_exact():
    """Codes that quantize to themselves and unit scales: each output is an
    integer dot product below 2^24, rounded once to bf16 on both sides."""
    M, N, K = _shape("one_round")
    assert eg.tc_token_tile(M, N, K, eg.VARIANT_W8A8) == 192
    rng = np.random.default_rng(20)
    xi = rng.integers(-127, 128, size=(M, K))
    xi[:, 0] = 127
    x = torch.tensor(xi, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
    x = x.view(np.uint16)
    w8 = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    s8 = np.full(N, 0x3C00, dtype=np.uint16)  # fp16 1.0
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    y = to_host_bits(eg.w8a8_gemm(a, to_dev(w8), to_dev(s8, torch.float16), path=eg.PATH_TC))
    a_q, a_s, _ = oracle.quant_act(x)
    dot, _, y_ref = oracle.w8a8(a_q, a_s, w8, s8)
    assert np.abs(dot).max() < 2 ** 24
    assert np.array_equal(y, y_ref)


def test_token_tile_choice():
    """Decode-sized tiles by M; 128 where 192 gains no round; the int8-weight
    variants take 192 too."""
    assert [eg.tc_token_tile(m, 3584, 3584) for m in (5, 16, 17, 32, 33, 64)] == \
        [16, 16, 32, 32, 64, 64]
    assert eg.tc_token_tile(256, 256, 512) == 128        # 2 m-tiles at either width
    assert eg.tc_token_tile(4096, 152064, 3584) == 192   # the untied head at 4096 tokens
    assert eg.tc_token_tile(4096, 12288, 3072, eg.VARIANT_W8A16) == 192
    assert eg.tc_token_tile(4096, 12288, 3072, eg.VARIANT_W8A8) == 192


def test_bf16_twin_full_tile():
    """The structure twin (dense bf16 weights through the same pipeline) on a
    192-token grid: each converter set copies its half of the group's K."""
    from helpers import bf16_bits_to_f64
    M, N, K = _shape("one_round")
    assert eg.tc_token_tile(M, N, K, eg.VARIANT_W4A16) == 192   # the twin's rule
    rng = np.random.default_rng(21)
    x = synth.activations(14, 0, 0, M, K, outliers=False)
    w = (rng.standard_normal((N, K)).astype(np.float32) * 0.05).view(np.uint32)
    w = ((w + 0x7FFF + ((w >> 16) & 1)) >> 16).astype(np.uint16)   # bf16, round to even
    y = eg.bf16_gemm_twin(to_dev(x, torch.bfloat16), to_dev(w, torch.bfloat16))
    cols = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N),
                                     rng.choice(N, 256, replace=False)]))
    ref = bf16_bits_to_f64(x) @ bf16_bits_to_f64(w[cols]).T
    ref_bits = np.vectorize(oracle.bf16_from_double, otypes=[np.uint16])(ref)
    check_bf16_output(to_host_bits(y)[:, cols], ref_bits, "twin, 192-token tiles")
