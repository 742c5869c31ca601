"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Integer stages (activation codes, scales, group sums, packing, group partials)
are compared bit for bit; bf16 outputs against the bar in tests/helpers.py.
Sizes span several 128-row tiles and ragged token tails; the full Qwen2.5-7B and
DiT shapes are checked on sampled rows/columns the oracle computes directly.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import check_bf16_output, decode_tc_operand, to_dev, to_host_bits, w4_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

import w4a8_quantized_gemm_gb300 as eg  # noqa: E402

PATHS = [eg.PATH_GEMV, eg.PATH_TC]
SHAPES_7B = {"q": (3584, 3584), "k": (3584, 512), "gate": (3584, 18944), "down": (18944, 3584)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    eg.load()
    torch.cuda.set_device(0)
    yield
    assert eg.device_status() == 0


def dev_weights(w):
    return (to_dev(w.w_q), to_dev(w.scale_f16, torch.float16), to_dev(w.zero))


def run_w4a8(x, w, path, M, N, K):
    packed = eg.pack_w4(*dev_weights(w))
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    y = eg.w4a8_gemm(a, packed, N, K, path=path)
    return a, packed, y


# ------------------------------------------------------------ activation quant

@pytest.mark.parametrize("M,K", [(16, 512), (1, 3584), (5, 18944), (64, 640), (65, 1024), (129, 1024),
                                 (300, 384),
                                 # rows split over clusters of 3, 5 and 8 CTAs
                                 (1, 8320), (4, 18944), (64, 18944), (7, 32768)])
def test_quant_act_bit_exact(M, K):
    x = synth.activations(0, 1, 0, M, K)
    if M > 3:
        x[2] = 0                                     # an all-zero token
        x[3] = 0
        x[3, K // 3] = 0xC47A                        # a single outlier (-1000)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    a_q, a_s, asum = oracle.quant_act(x)
    assert np.array_equal(a.a_q.cpu().numpy(), a_q)
    assert np.array_equal(a.a_s.cpu().numpy().view(np.uint32), a_s.view(np.uint32))
    assert np.array_equal(a.a_gsum.cpu().numpy(), asum)
    form = eg.tc_operand_form(M)
    assert form == (eg.TC_FORM_E4M3_PLANES if M <= 64 else eg.TC_FORM_F16)
    got = decode_tc_operand(a.a_tc.cpu().numpy(), M, K, form == eg.TC_FORM_E4M3_PLANES)
    assert np.array_equal(got, a_q.astype(np.float64))


def test_quant_act_ties_from_golden_rows():
    # rows whose quotients x / a_s sit exactly on .5 (round-half-even decides)
    rows = [[254, 1, 3, -5, 0, 7, -1, 100], [-254, 3, 5, -3, -1, 1, 9, 11]]
    x = np.zeros((2, 128), np.float32)
    x[:, :8] = rows
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    a = eg.quant_act(to_dev(xb, torch.bfloat16))
    got = a.a_q.cpu().numpy()[:, :8]
    assert got.tolist() == [[127, 0, 2, -2, 0, 4, 0, 50], [-127, 2, 2, -2, 0, 0, 4, 6]]


def _misrounding_rows(M, K, seed):
    """bf16 rows each holding values x whose product with the reciprocal of
    the row's scale, x * fl(1 / a_s), rounds to another integer than the fp32
    quotient x / a_s (found by search over every bf16 value below the row's
    absmax, in numpy's IEEE fp32 arithmetic); random values elsewhere. The
    quantizer computes codes from that product and divides exactly where the
    product lies near a half-integer: these are the values that check it."""
    rng = np.random.default_rng(seed)
    pos = (np.arange(0x0080, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    x = np.zeros((M, K), np.float32)
    m = 0
    while m < M:
        amax = pos[rng.integers(0x2F00, 0x4780)]     # absmax 2^-33 .. 2^16
        s = np.float32(amax) / np.float32(127)
        inv = np.float32(1) / s
        cand = pos[pos <= amax]
        bad = cand[np.rint(cand * inv) != np.rint(cand / s)]
        if len(bad) == 0:
            continue
        row = (rng.uniform(-1.0, 1.0, K) * 0.99 * float(amax)).astype(np.float32)
        row[0] = amax
        where = rng.choice(np.arange(1, K), size=min(K // 4, 64), replace=False)
        row[where] = rng.choice(np.concatenate([bad, -bad]), size=len(where))
        x[m] = row
        m += 1
    bits = x.view(np.uint32)
    return ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("M,K", [(3, 3584),      # few tokens: 512 threads a row
                                 (5, 18944),     # few tokens: a cluster splits the row
                                 (2, 33024),     # few tokens, row too long for both: two passes
                                 # many tokens: persistent CTAs streaming rows through
                                 # shared memory -- one row each, then several rows each
                                 # (more rows than resident CTAs: double-buffered staging)
                                 (70, 8192), (2600, 1024), (101, 4096), (1000, 16384),
                                 (400, 32768),
                                 (66, 33024)])   # many tokens, rows too long to stage: two passes
@pytest.mark.parametrize("with_codes", [True, False])
def test_quant_act_misrounding_products_bit_exact(M, K, with_codes):
    """Every quantization kernel, on rows built from the values where the
    reciprocal product alone would round wrong: codes, scales, group sums and
    the operand form bit for bit against the oracle, with the int8 codes
    written or left out."""
    x = _misrounding_rows(M, K, 40 + M + K % 97)
    a = eg.quant_act(to_dev(x, torch.bfloat16), with_codes=with_codes)
    a_q, a_s, asum = oracle.quant_act(x)
    if with_codes:
        assert np.array_equal(a.a_q.cpu().numpy(), a_q)
    else:
        assert a.a_q is None
    assert np.array_equal(a.a_s.cpu().numpy().view(np.uint32), a_s.view(np.uint32))
    assert np.array_equal(a.a_gsum.cpu().numpy(), asum)
    got = decode_tc_operand(a.a_tc.cpu().numpy(), M, K, M <= 64)
    assert np.array_equal(got, a_q.astype(np.float64))


@pytest.mark.parametrize("M", [16, 130])
def test_w4a8_gemm_without_int8_codes(M):
    """Codes kept only in the operand form: the tensor-core path gives the
    bits it gives with the int8 codes present; the GEMV path, which reads
    them, refuses."""
    N, K = 256, 1024
    x, w = w4_case(16, M, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    xd = to_dev(x, torch.bfloat16)
    y1 = eg.w4a8_gemm(eg.quant_act(xd), packed, N, K, path=eg.PATH_TC)
    lean = eg.quant_act(xd, with_codes=False)
    y2 = eg.w4a8_gemm(lean, packed, N, K, path=eg.PATH_TC)
    assert torch.equal(y1, y2)
    ys1 = eg.w4a8_gemm_grouped(eg.quant_act(xd), [packed, packed], [N, N], K, path=eg.PATH_TC)
    ys2 = eg.w4a8_gemm_grouped(lean, [packed, packed], [N, N], K, path=eg.PATH_TC)
    assert all(torch.equal(u, v) for u, v in zip(ys1, ys2))
    with pytest.raises(eg.EgopqError) as err:
        eg.w4a8_gemm(lean, packed, N, K, path=eg.PATH_GEMV)
    assert err.value.code == -1
    assert eg.device_status() == 0


# -------------------------------------------------------------------- packing

@pytest.mark.parametrize("N,K", [(128, 128), (256, 512), (512, 3584)])
def test_pack_bit_exact_and_roundtrip(N, K):
    w = synth.w4_weights(0, 2, 0, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    ref = oracle.pack_w4(w.w_q, w.scale_f16, w.zero)
    assert np.array_equal(packed.cpu().numpy(), ref)
    w2, s2, z2 = eg.unpack_w4(packed, N, K)
    assert np.array_equal(w2.cpu().numpy(), w.w_q)
    assert np.array_equal(to_host_bits(s2), w.scale_f16)
    assert np.array_equal(z2.cpu().numpy(), w.zero)


# ------------------------------------------------------------- group partials

@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 3, 4, 5, 16, 17, 33, 48, 64, 65, 129])
def test_w4a8_group_partials_bit_exact(path, M):
    N, K = 256, 512
    x, w = w4_case(0, M, N, K)
    a, packed, _ = run_w4a8(x, w, path, M, N, K)
    Q = eg.w4a8_group_partials(a, packed, N, K, path=path).cpu().numpy()
    a_q, _, _ = oracle.quant_act(x)
    assert np.array_equal(Q, oracle.group_partials(a_q, w.w_q, w.zero))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("case", ["max_pos", "max_neg", "alternating", "neg_act"])
@pytest.mark.parametrize("M", [16, 100])
def test_w4a8_group_partials_worst_case_magnitudes(path, case, M):
    """|Q| up to 128*127*15 = 243840: the tensor-core path must stay exact
    (integer products accumulated in fp32 within one group; e4m3 operands for
    M = 16, fp16 for M = 100)."""
    N, K = 128, 512
    G = K // 128
    x = np.full((M, K), 0x3F80, np.uint16)                     # 1.0 -> a_q = 127
    w_q = np.full((N, K), 15, np.uint8)
    z = np.zeros((N, G), np.uint8)
    if case == "max_neg":
        w_q[:] = 0
        z[:] = 15
    elif case == "alternating":
        x[:, 1::2] = 0xBF80                                    # -1.0 -> a_q = -127
        w_q[:, 1::2] = 0
        w_q[::2, :] = 15 - w_q[::2, :]                         # half the rows flipped
        z[:, :] = np.arange(N)[:, None] % 16
    elif case == "neg_act":
        x[:] = 0xBF80                                          # a_q = -127 = 16*(-8) + 1
    s = np.full((N, G), 0x3C00, np.uint16)                     # 1.0
    w = synth.W4Weights(w_q, s, z, 128)
    a, packed, _ = run_w4a8(x, w, path, M, N, K)
    Q = eg.w4a8_group_partials(a, packed, N, K, path=path).cpu().numpy()
    a_q, _, _ = oracle.quant_act(x)
    ref = oracle.group_partials(a_q, w_q, z)
    if case == "max_pos":
        assert ref.max() == 243840
    if case in ("max_neg", "neg_act"):
        assert ref.min() == -243840
    assert np.array_equal(Q, ref)


# ------------------------------------------------------------------ W4A8 output

@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8, 15, 16, 17, 31, 64, 100, 127, 128, 129, 256])
def test_w4a8_output_sweep_small(path, M):
    N, K = 256, 512
    x, w = w4_case(0, M, N, K)
    a, packed, y = run_w4a8(x, w, path, M, N, K)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, f"W4A8 path={path} M={M}")


@pytest.mark.parametrize("path", PATHS)
def test_w4a8_output_many_tiles(path):
    # several 128-row weight tiles, 28 groups, ragged token tail, split-K clusters
    M, N, K = 37, 1024, 3584
    x, w = w4_case(0, M, N, K, layer=3)
    a, packed, y = run_w4a8(x, w, path, M, N, K)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, f"W4A8 path={path}")


def test_w4a8_paths_agree_and_deterministic():
    M, N, K = 4, 512, 3584
    x, w = w4_case(1, M, N, K)
    _, _, y1 = run_w4a8(x, w, eg.PATH_GEMV, M, N, K)
    _, _, y2 = run_w4a8(x, w, eg.PATH_GEMV, M, N, K)
    _, _, y3 = run_w4a8(x, w, eg.PATH_TC, M, N, K)
    _, _, y4 = run_w4a8(x, w, eg.PATH_TC, M, N, K)
    assert torch.equal(y1, y2) and torch.equal(y3, y4)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y1), y_ref, "gemv")
    check_bf16_output(to_host_bits(y3), y_ref, "tc")


def _sampled_check(x, w, y_bits, rows, cols, what):
    a_q, a_s, _ = oracle.quant_act(x[rows])
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q[cols], w.scale_f16[cols], w.zero[cols])
    check_bf16_output(y_bits[np.ix_(rows, cols)], y_ref, what)


@pytest.mark.parametrize("name", list(SHAPES_7B))
@pytest.mark.parametrize("M", [1, 4, 16])
def test_w4a8_decode_7b_shapes(name, M):
    K, N = SHAPES_7B[name]
    x, w = w4_case(1, M, N, K, linear=synth.LINEARS[name])
    a, packed, y = run_w4a8(x, w, eg.PATH_AUTO, M, N, K)
    a_q, a_s, asum = oracle.quant_act(x)
    assert np.array_equal(a.a_q.cpu().numpy(), a_q)
    cols = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N),
                                     np.random.default_rng(M).choice(N, 256, replace=False)]))
    _sampled_check(x, w, to_host_bits(y), np.arange(M), cols, f"decode {name} M={M}")


@pytest.mark.parametrize("name,M", [("q", 512), ("gate", 2048), ("down", 4096), ("k", 4096)])
def test_w4a8_prefill_7b_shapes_sampled(name, M):
    K, N = SHAPES_7B[name]
    x, w = w4_case(2, M, N, K, linear=synth.LINEARS[name])
    a, packed, y = run_w4a8(x, w, eg.PATH_AUTO, M, N, K)
    a_q, a_s, asum = oracle.quant_act(x)
    assert np.array_equal(a.a_q.cpu().numpy(), a_q)
    assert np.array_equal(a.a_gsum.cpu().numpy(), asum)
    rng = np.random.default_rng(M + N)
    rows = np.unique(np.concatenate([np.arange(4), np.arange(M - 4, M), rng.choice(M, 8, replace=False)]))
    cols = np.unique(np.concatenate([np.arange(64), np.arange(N - 64, N), rng.choice(N, 128, replace=False)]))
    _sampled_check(x, w, to_host_bits(y), rows, cols, f"prefill {name} M={M}")


def test_w4a8_head_prefill_sampled():
    """Untied quantized output head, K=3584, N=152064, at M=512."""
    M, K, N = 512, 3584, 152064
    x, w = w4_case(2, M, N, K, linear=synth.LINEARS["head"])
    a, packed, y = run_w4a8(x, w, eg.PATH_AUTO, M, N, K)
    rng = np.random.default_rng(7)
    rows = np.array([0, 1, 255, 256, 510, 511])
    cols = np.unique(np.concatenate([np.arange(32), np.arange(N - 32, N), rng.choice(N, 192, replace=False)]))
    _sampled_check(x, w, to_host_bits(y), rows, cols, "head M=512")


# ------------------------------------------------------- W4A16 and W8A16 output

@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 3, 16, 17, 130])
def test_w4a16_output(path, M):
    N, K = 384, 1024
    x, w = w4_case(4, M, N, K, outliers=False)
    packed = eg.pack_w4(*dev_weights(w))
    y = eg.w4a16_gemm(to_dev(x, torch.bfloat16), packed, N, K, path=path)
    _, y_ref = oracle.w4a16(x, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, f"W4A16 path={path} M={M}")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("M", [1, 3, 16, 17, 130])
def test_w8a16_output(path, M):
    N, K = 384, 1024
    w8, s8 = synth.w8_weights(4, 0, 0, N, K)
    x = synth.activations(4, 0, 0, M, K, outliers=False)
    y = eg.w8a16_gemm(to_dev(x, torch.bfloat16), to_dev(w8), to_dev(s8, torch.float16), path=path)
    _, y_ref = oracle.w8a16(x, w8, s8)
    check_bf16_output(to_host_bits(y), y_ref, f"W8A16 path={path} M={M}")


@pytest.mark.parametrize("K,N", [(3072, 3072), (3072, 12288), (12288, 3072)])
@pytest.mark.parametrize("M", [1, 16, 4096])
def test_weight_only_dit_shapes_sampled(K, N, M):
    x = synth.activations(4, 1, 0, M, K, outliers=False)
    w = synth.w4_weights(4, 1, 0, N, K)
    w8, s8 = synth.w8_weights(4, 1, 0, N, K)
    xd = to_dev(x, torch.bfloat16)
    y4 = to_host_bits(eg.w4a16_gemm(xd, eg.pack_w4(*dev_weights(w)), N, K))
    y8 = to_host_bits(eg.w8a16_gemm(xd, to_dev(w8), to_dev(s8, torch.float16)))
    rng = np.random.default_rng(K + N + M)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, min(M, 6), replace=False)]))
    cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 160, replace=False)]))
    _, r4 = oracle.w4a16(x[rows], w.w_q[cols], w.scale_f16[cols], w.zero[cols])
    _, r8 = oracle.w8a16(x[rows], w8[cols], s8[cols])
    check_bf16_output(y4[np.ix_(rows, cols)], r4, f"W4A16 DiT K={K} N={N} M={M}")
    check_bf16_output(y8[np.ix_(rows, cols)], r8, f"W8A16 DiT K={K} N={N} M={M}")


# ------------------------------------------------------------ GPTQ import

def to_gptq(w_q, s_f16, z, zero_offset):
    """Logical codes [N][K], scales and zero points [N][G] as GPTQ checkpoint
    tensors (qweight [K/8][N], qzeros [G][N/8], scales [G][N]); the zero
    points are stored minus the offset."""
    N, K = w_q.shape
    cw = w_q.astype(np.uint32).T.reshape(K // 8, 8, N)             # [r][i][n]
    qweight = np.zeros((K // 8, N), np.uint32)
    for i in range(8):
        qweight |= (cw[:, i, :] & 0xF) << (4 * i)
    zs = (z.astype(np.int64) - zero_offset).T.reshape(-1, N // 8, 8)  # [g][c][j]
    qzeros = np.zeros(zs.shape[:2], np.uint32)
    for j in range(8):
        qzeros |= (zs[:, :, j].astype(np.uint32) & 0xF) << (4 * j)
    return qweight.view(np.int32), qzeros.view(np.int32), np.ascontiguousarray(s_f16.T)


@pytest.mark.parametrize("N,K,off", [(128, 128, 1), (384, 1024, 0), (3584, 18944, 1)])
def test_gptq_import_equals_pack(N, K, off):
    w = synth.w4_weights(8, 0, 0, N, K)
    z = np.maximum(w.zero, off).astype(np.uint8)   # representable after the offset
    qweight, qzeros, scales = to_gptq(w.w_q, w.scale_f16, z, off)
    # the helper's words decode (by the oracle) to the logical tensors
    wq2, s2, z2, bad = oracle.gptq_unpack(qweight, qzeros, scales, N, K, 128, off)
    assert bad == 0 and np.array_equal(wq2, w.w_q) and np.array_equal(s2, w.scale_f16)
    assert np.array_equal(z2, z)
    got = eg.pack_w4_gptq(to_dev(qweight), to_dev(qzeros), to_dev(scales, torch.float16), off)
    ref = eg.pack_w4(to_dev(w.w_q), to_dev(w.scale_f16, torch.float16), to_dev(z))
    assert torch.equal(got, ref)
    assert eg.device_status() == 0


def test_gptq_import_flags_unrepresentable_zero():
    """With offset 1 a stored zero nibble of 15 means z = 16, which the 4-bit
    record cannot hold: the import completes, and the next egopq_device_status
    reports EGOPQ_ERR_INVALID_ARG (once: the word is cleared)."""
    N, K = 128, 256
    w = synth.w4_weights(8, 1, 0, N, K)
    z = np.ones_like(w.zero)                       # stored as 0 with offset 1
    qweight, qzeros, scales = to_gptq(w.w_q, w.scale_f16, z, 1)
    qz = qzeros.view(np.uint32).copy()
    qz[1, 3] |= np.uint32(0xF << 8)                # output 8*3 + 2 = 26, group 1: stored 15
    qz = qz.view(np.int32)
    assert oracle.gptq_unpack(qweight, qz, scales, N, K, 128, 1)[3] == 1
    eg.pack_w4_gptq(to_dev(qweight), to_dev(qz), to_dev(scales, torch.float16), 1)
    assert eg.device_status() == -1
    assert eg.device_status() == 0


# ------------------------------------------- dense bf16 twin: dequantize once

@pytest.mark.parametrize("N,K", [(128, 128), (384, 1024), (3584, 18944)])
def test_dequant_w4_bit_exact(N, K):
    """egopq_dequant_w4 against the oracle, every element, bit for bit."""
    w = synth.w4_weights(6, 0, 0, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    got = to_host_bits(eg.dequant_w4(packed, N, K))
    assert np.array_equal(got, oracle.dequant_w4_bf16(w.w_q, w.scale_f16, w.zero))


def test_dequant_w4_head_sampled_rows():
    """The 152064 x 3584 output head (1.09 GB of bf16): sampled rows from the
    first, last and random 128-row blocks."""
    N, K = 152064, 3584
    w = synth.w4_weights(6, 1, synth.LINEARS["head"], N, K)
    dq = eg.dequant_w4(eg.pack_w4(*dev_weights(w)), N, K)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, N - 1], rng.choice(N, 64, replace=False)]))
    got = to_host_bits(dq[torch.from_numpy(rows).cuda()])
    ref = oracle.dequant_w4_bf16(w.w_q[rows], w.scale_f16[rows], w.zero[rows])
    assert np.array_equal(got, ref)


# ------------------------------------------------- W8A8 int8-dynamic output

def run_w8a8(x, w8, s8, path):
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    return eg.w8a8_gemm(a, to_dev(w8), to_dev(s8, torch.float16), path=path)


@pytest.mark.parametrize("path,M", [(eg.PATH_GEMV, m) for m in (1, 2, 3, 5, 8, 9, 16, 17, 64)]
                         + [(eg.PATH_TC, m) for m in (65, 130, 300)]
                         + [(eg.PATH_AUTO, m) for m in (1, 64, 65, 129)])
def test_w8a8_output(path, M):
    """GEMV (up to 8 tokens a launch, ragged tails) and the tensor-core path
    (128-token tiles, ragged tails) against the int8-dynamic oracle."""
    N, K = 384, 1024
    w8, s8 = synth.w8_weights(5, 0, 0, N, K)
    x = synth.activations(5, 0, 0, M, K)
    y = run_w8a8(x, w8, s8, path)
    a_q, a_s, _ = oracle.quant_act(x)
    _, _, y_ref = oracle.w8a8(a_q, a_s, w8, s8)
    check_bf16_output(to_host_bits(y), y_ref, f"W8A8 path={path} M={M}")


@pytest.mark.parametrize("path,M", [(eg.PATH_GEMV, 7), (eg.PATH_TC, 200)])
def test_w8a8_integer_case_bit_exact(path, M):
    """Tokens whose absmax is 127 quantize to themselves with scale 1; with unit
    weight scales every output is an integer dot product below 2^24, which the
    kernel and the oracle both round once to bf16: identical bits."""
    N, K = 256, 768
    rng = np.random.default_rng(M)
    xi = rng.integers(-127, 128, size=(M, K))
    xi[:, 0] = 127
    x = torch.tensor(xi, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w8 = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
    s8 = np.full(N, 0x3C00, dtype=np.uint16)  # fp16 1.0
    y = to_host_bits(run_w8a8(x, w8, s8, path))
    a_q, a_s, _ = oracle.quant_act(x)
    assert np.array_equal(a_q, xi.astype(np.int8)) and np.all(a_s == 1.0)
    dot, _, y_ref = oracle.w8a8(a_q, a_s, w8, s8)
    assert np.abs(dot).max() < 2 ** 24
    assert np.array_equal(y, y_ref)


@pytest.mark.parametrize("path,M", [(eg.PATH_GEMV, 4), (eg.PATH_TC, 130)])
def test_w8a8_extreme_magnitudes(path, M):
    """Every code at +-127 over K = 18944: dot products of +-305,547,776 stay
    exact in the int32 accumulators (and in the tensor-core path's per-group
    fp32 partials, each at most 128*127*127 < 2^24)."""
    N, K = 128, 18944
    rng = np.random.default_rng(3)
    sign_a = rng.choice([-1, 1], size=(M, K))
    sign_a[1] = 1
    x = torch.tensor(sign_a * 2.0, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    w8 = (rng.choice([-1, 1], size=(N, K)) * 127).astype(np.int8)
    w8[0] = 127
    s8 = np.full(N, 0x2C00, dtype=np.uint16)  # fp16 1/16
    y = run_w8a8(x, w8, s8, path)
    a_q, a_s, _ = oracle.quant_act(x)
    dot, _, y_ref = oracle.w8a8(a_q, a_s, w8, s8)
    assert dot[1, 0] == 127 * 127 * K
    check_bf16_output(to_host_bits(y), y_ref, f"W8A8 extreme path={path}")


def test_w8a8_refusals():
    """The tensor-core path takes the fp16 operand form only (M > 64): forced
    TC below it is an unsupported shape; TC without a_tc is an invalid argument."""
    N, K = 128, 256
    w8, s8 = synth.w8_weights(5, 1, 0, N, K)
    a = eg.quant_act(to_dev(synth.activations(5, 1, 0, 64, K), torch.bfloat16))
    with pytest.raises(eg.EgopqError) as e:
        eg.w8a8_gemm(a, to_dev(w8), to_dev(s8, torch.float16), path=eg.PATH_TC)
    assert e.value.code == -2
    a2 = eg.quant_act(to_dev(synth.activations(5, 1, 0, 130, K), torch.bfloat16), with_tc=False)
    with pytest.raises(eg.EgopqError) as e:
        eg.w8a8_gemm(a2, to_dev(w8), to_dev(s8, torch.float16), path=eg.PATH_TC)
    assert e.value.code == -1
    y = eg.w8a8_gemm(a2, to_dev(w8), to_dev(s8, torch.float16), path=eg.PATH_GEMV)
    assert y.shape == (130, N)


@pytest.mark.parametrize("K,N", [(3072, 3072), (3072, 12288), (12288, 3072)])
@pytest.mark.parametrize("M", [16, 4096])
def test_w8a8_dit_shapes_sampled(K, N, M):
    """The DiT linears at a decode-sized and a 4096-token batch (GEMV and
    tensor cores under AUTO), checked on sampled rows and columns."""
    x = synth.activations(5, 2, 0, M, K, outliers=False)
    w8, s8 = synth.w8_weights(5, 2, 0, N, K)
    y = to_host_bits(run_w8a8(x, w8, s8, eg.PATH_AUTO))
    rng = np.random.default_rng(K + N + M)
    rows = np.unique(np.concatenate([[0, M - 1], rng.choice(M, min(M, 6), replace=False)]))
    cols = np.unique(np.concatenate([[0, N - 1], rng.choice(N, 160, replace=False)]))
    a_q, a_s, _ = oracle.quant_act(x[rows])
    _, _, r = oracle.w8a8(a_q, a_s, w8[cols], s8[cols])
    check_bf16_output(y[np.ix_(rows, cols)], r, f"W8A8 DiT K={K} N={N} M={M}")


# ----------------------------------------------------------------- edge cases

def test_empty_batch_is_a_noop():
    K, N = 512, 256
    w = synth.w4_weights(0, 0, 0, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    a = eg.quant_act(x)
    y = eg.w4a8_gemm(a, packed, N, K)
    assert y.shape == (0, N)


def test_empty_batches_other_variants_are_noops():
    """M = 0 through every GEMM entry point: an empty result, nothing launched,
    no error."""
    K, N = 512, 256
    w = synth.w4_weights(0, 0, 0, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    w8, s8 = synth.w8_weights(0, 0, 0, N, K)
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    a = eg.quant_act(x)
    for path in (eg.PATH_AUTO, eg.PATH_GEMV, eg.PATH_TC):
        assert eg.w4a16_gemm(x, packed, N, K, path=path).shape == (0, N)
        assert eg.w8a16_gemm(x, to_dev(w8), to_dev(s8, torch.float16), path=path).shape == (0, N)
        assert eg.w8a8_gemm(a, to_dev(w8), to_dev(s8, torch.float16), path=path).shape == (0, N)
    assert eg.device_status() == 0


def test_rejections_new_entry_points():
    """Host-side refusals of the W8A8, GPTQ-import and dequantization calls:
    untiled N, a group other than 128, a bad zero offset, misaligned pointers;
    nothing is launched and the status names the cause."""
    lib = eg.load()
    st = torch.cuda.current_stream().cuda_stream
    K, N = 512, 256
    w8, s8 = synth.w8_weights(0, 0, 0, N, K)
    w8d, s8d = to_dev(w8), to_dev(s8, torch.float16)
    a = eg.quant_act(to_dev(synth.activations(0, 0, 0, 4, K), torch.bfloat16))
    y = torch.empty((4, N), dtype=torch.bfloat16, device="cuda")
    # W8A8: N = 192 untiled; misaligned output
    assert lib.egopq_w8a8_gemm_ex(a.a_q.data_ptr(), None, a.a_s.data_ptr(), w8d.data_ptr(),
                                  s8d.data_ptr(), 4, 192, K, y.data_ptr(), 0, st) == -2
    assert lib.egopq_w8a8_gemm_ex(a.a_q.data_ptr(), None, a.a_s.data_ptr(), w8d.data_ptr(),
                                  s8d.data_ptr(), 4, N, K, y.data_ptr() + 2, 0, st) == -3
    # GPTQ import: group 64, zero offset 2, misaligned qweight
    qweight = torch.zeros((K // 8, N), dtype=torch.int32, device="cuda")
    qzeros = torch.zeros((K // 128, N // 8), dtype=torch.int32, device="cuda")
    scales = torch.ones((K // 128, N), dtype=torch.float16, device="cuda")
    packed = torch.empty(eg.packed_w4_bytes(N, K), dtype=torch.uint8, device="cuda")
    args = (qzeros.data_ptr(), scales.data_ptr(), N, K)
    assert lib.egopq_pack_w4_gptq(qweight.data_ptr(), *args, 64, 1, packed.data_ptr(), st) == -2
    assert lib.egopq_pack_w4_gptq(qweight.data_ptr(), *args, 128, 2, packed.data_ptr(), st) == -1
    assert lib.egopq_pack_w4_gptq(qweight.data_ptr() + 4, *args, 128, 1, packed.data_ptr(),
                                  st) == -3
    # dequantization: untiled K, misaligned output
    wd = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    assert lib.egopq_dequant_w4(packed.data_ptr(), N, K - 64, 128, wd.data_ptr(), st) == -2
    assert lib.egopq_dequant_w4(packed.data_ptr(), N, K, 128, wd.data_ptr() + 2, st) == -3
    assert eg.device_status() == 0


def test_guard_bands_new_outputs():
    """The W8A8 (GEMV and tensor-core) and dequantization kernels write
    exactly their outputs: sentinel bands on both sides stay intact."""
    pad = 4096
    K, N = 1024, 256
    w8, s8 = synth.w8_weights(0, 1, 0, N, K)
    for M, path in [(9, eg.PATH_GEMV), (130, eg.PATH_TC)]:
        a = eg.quant_act(to_dev(synth.activations(0, 1, 0, M, K), torch.bfloat16))
        buf = torch.full((M * N + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
        out = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
        eg.w8a8_gemm(a, to_dev(w8), to_dev(s8, torch.float16), path=path, out=out)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + M * N:] == 12345), path
    w = synth.w4_weights(0, 1, 0, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    buf = torch.full((N * K + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
    eg.dequant_w4(packed, N, K, out=buf[pad:pad + N * K].view(torch.bfloat16).view(N, K))
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + N * K:] == 12345)
    assert eg.device_status() == 0


def test_output_guard_bands_untouched():
    M, N, K = 17, 256, 512
    x, w = w4_case(0, M, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    for path in PATHS:
        pad = 4096
        buf = torch.full((M * N + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
        out = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
        eg.w4a8_gemm(a, packed, N, K, path=path, out=out)
        torch.cuda.synchronize()
        assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + M * N:] == 12345)


def test_rejections():
    K, N = 512, 256
    w = synth.w4_weights(0, 0, 0, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    a = eg.quant_act(to_dev(synth.activations(0, 0, 0, 4, K), torch.bfloat16))
    lib = eg.load()
    s = torch.cuda.current_stream().cuda_stream
    y = torch.empty((4, N), dtype=torch.bfloat16, device="cuda")
    # N not a multiple of 128, misaligned output, missing fp16 codes on the TC path
    assert lib.egopq_w4a8_gemm_ex(a.a_q.data_ptr(), a.a_tc.data_ptr(), a.a_s.data_ptr(),
                                  a.a_gsum.data_ptr(), packed.data_ptr(), 4, 192, K, 128,
                                  y.data_ptr(), 0, s) == -2
    assert lib.egopq_w4a8_gemm_ex(a.a_q.data_ptr(), a.a_tc.data_ptr(), a.a_s.data_ptr(),
                                  a.a_gsum.data_ptr(), packed.data_ptr(), 4, N, K, 128,
                                  y.data_ptr() + 2, 0, s) == -3
    assert lib.egopq_w4a8_gemm_ex(a.a_q.data_ptr(), None, a.a_s.data_ptr(),
                                  a.a_gsum.data_ptr(), packed.data_ptr(), 4, N, K, 128,
                                  y.data_ptr(), eg.PATH_TC, s) == -1
    assert lib.egopq_w4a8_gemm_ex(a.a_q.data_ptr(), a.a_tc.data_ptr(), a.a_s.data_ptr(),
                                  a.a_gsum.data_ptr(), packed.data_ptr(), 4, N, K, 64,
                                  y.data_ptr(), 0, s) == -2
    assert eg.supported(4, N, K) and not eg.supported(4, 80, K)
    assert eg.device_status() == 0


def test_bounded_wait_reports_timeout_without_fault():
    eg.selftest_timeout(2000)          # 2 ms deadline, nothing ever arrives
    assert eg.device_status() == -6    # reported, then cleared
    assert eg.device_status() == 0
    # the context is still usable
    M, N, K = 4, 256, 512
    x, w = w4_case(0, M, N, K)
    a, packed, y = run_w4a8(x, w, eg.PATH_TC, M, N, K)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, "after timeout self-test")


@pytest.mark.parametrize("M", [1, 4, 16, 200])
def test_fused_sibling_linears_equal_separate(M):
    """q|k|v packed as one weight (N = 3584+512+512): the fused GEMM's column
    blocks are the separate linears' outputs."""
    K = 3584
    parts = [("q", 3584), ("k", 512), ("v", 512)]
    ws = [synth.w4_weights(5, 0, synth.LINEARS[nm], n, K) for nm, n in parts]
    fused = synth.W4Weights(np.concatenate([w.w_q for w in ws]),
                            np.concatenate([w.scale_f16 for w in ws]),
                            np.concatenate([w.zero for w in ws]), 128)
    x = synth.activations(5, 0, 0, M, K)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    N = sum(n for _, n in parts)
    yf = to_host_bits(eg.w4a8_gemm(a, eg.pack_w4(*dev_weights(fused)), N, K))
    off = 0
    a_q, a_s, _ = oracle.quant_act(x)
    cols = np.random.default_rng(M).choice(N, 96, replace=False)
    _, y_ref = oracle.w4a8(a_q, a_s, fused.w_q[cols], fused.scale_f16[cols], fused.zero[cols])
    check_bf16_output(yf[:, cols], y_ref, f"fused qkv M={M}")
    for (nm, n), w in zip(parts, ws):
        ys = to_host_bits(eg.w4a8_gemm(a, eg.pack_w4(*dev_weights(w)), n, K))
        if M <= 4:  # GEMV: each row's sum is formed the same way whatever N is
            assert np.array_equal(yf[:, off:off + n], ys), nm
        else:
            check_bf16_output(yf[:, off:off + n], ys, f"fused vs {nm}")
        off += n


@pytest.mark.parametrize("n_tiles", [76, 78, 77])
def test_w4a8_persistent_grid_full(n_tiles):
    """Grids with at least one tile per SM run persistently, striding over the
    tiles in bands of m-tiles; n-tile counts around one and two per SM, a
    ragged token tail (M=200 over two 128-token tiles), full oracle
    comparison."""
    M, K, N = 200, 512, 128 * n_tiles
    x, w = w4_case(6, M, N, K)
    a, packed, y = run_w4a8(x, w, eg.PATH_TC, M, N, K)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, f"persistent n_tiles={n_tiles}")
    Q = eg.w4a8_group_partials(a, packed, N, K, path=eg.PATH_TC).cpu().numpy()
    rows = [0, 127, 128, 199]
    assert np.array_equal(Q[rows], oracle.group_partials(a_q[rows], w.w_q, w.zero))


@pytest.mark.parametrize("per_sm", [(2, 0), (2, 1), (3, 0)])
def test_w4a8_persistent_grid_small_token_tile(per_sm):
    """Token tiles of 16 (e4m3 form) run two CTAs per SM, so their grid goes
    persistent from two tiles per SM on: tile counts of exactly two per SM, one
    more, and three per SM, with a ragged token count (13 of 16)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n_tiles = per_sm[0] * sms + per_sm[1]
    M, K, N = 13, 256, 128 * n_tiles
    x, w = w4_case(10, M, N, K)
    a, packed, y = run_w4a8(x, w, eg.PATH_TC, M, N, K)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y), y_ref, f"persistent 16-token tiles n_tiles={n_tiles}")
    Q = eg.w4a8_group_partials(a, packed, N, K, path=eg.PATH_TC).cpu().numpy()
    assert np.array_equal(Q, oracle.group_partials(a_q, w.w_q, w.zero))


@pytest.mark.parametrize("variant", ["w4a16", "w8a16"])
def test_weight_only_persistent_grid_full(variant):
    M, K, N = 256, 384, 128 * 76
    x = synth.activations(7, 0, 0, M, K, outliers=False)
    if variant == "w4a16":
        w = synth.w4_weights(7, 0, 0, N, K)
        y = eg.w4a16_gemm(to_dev(x, torch.bfloat16), eg.pack_w4(*dev_weights(w)), N, K,
                          path=eg.PATH_TC)
        _, y_ref = oracle.w4a16(x, w.w_q, w.scale_f16, w.zero)
    else:
        w8, s8 = synth.w8_weights(7, 0, 0, N, K)
        y = eg.w8a16_gemm(to_dev(x, torch.bfloat16), to_dev(w8), to_dev(s8, torch.float16),
                          path=eg.PATH_TC)
        _, y_ref = oracle.w8a16(x, w8, s8)
    check_bf16_output(to_host_bits(y), y_ref, f"{variant} persistent")


# ------------------------------------------------------- one-call W4A8 linear

@pytest.mark.parametrize("path", [eg.PATH_AUTO, eg.PATH_GEMV, eg.PATH_TC])
@pytest.mark.parametrize("M", [1, 3, 4, 8, 16, 17, 129])
def test_w4a8_linear_equals_quant_then_gemm(path, M):
    """The one-call linear (quantization staged in a caller workspace, then the
    GEMM) is bit-identical to the two-call sequence on the same path, and meets
    the bar against the oracle."""
    N, K = 384, 3584
    x, w = w4_case(8, M, N, K)
    x[min(2, M - 1)] = 0  # an all-zero token
    packed = eg.pack_w4(*dev_weights(w))
    xd = to_dev(x, torch.bfloat16)
    y1 = eg.w4a8_linear(xd, packed, N, path=path)
    two_step_path = path if path != eg.PATH_AUTO else eg.auto_path(M)
    y2 = eg.w4a8_gemm(eg.quant_act(xd), packed, N, K, path=two_step_path)
    assert torch.equal(y1, y2)
    a_q, a_s, _ = oracle.quant_act(x)
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
    check_bf16_output(to_host_bits(y1), y_ref, f"linear path={path} M={M}")


def test_w4a8_linear_workspace_checks():
    M, N, K = 32, 256, 512
    x, w = w4_case(8, M, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    need = eg.w4a8_linear_workspace_bytes(M, K, eg.PATH_TC)
    assert need > eg.w4a8_linear_workspace_bytes(M, K, eg.PATH_GEMV) > 0
    lib = eg.load()
    xd = to_dev(x, torch.bfloat16)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (xd.data_ptr(), packed.data_ptr(), M, N, K, 128, y.data_ptr())
    assert lib.egopq_w4a8_linear(*args, None, 0, eg.PATH_TC, s) == -1
    assert lib.egopq_w4a8_linear(*args, ws.data_ptr(), need - 1, eg.PATH_TC, s) == -1
    assert lib.egopq_w4a8_linear(*args, ws.data_ptr(), need, eg.PATH_TC, s) == 0
    assert lib.egopq_w4a8_linear(*args, None, 0, eg.PATH_GEMV, s) == -1
    assert eg.device_status() == 0


def _tie_rows(M, K, seed):
    """bf16 rows whose quotients x / a_s sit on or within a few fp32 ulps of
    half-integers (the cases the fused quantizer divides exactly), plus an
    all-zero row and a plain random row."""
    rng = np.random.default_rng(seed)
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        if m == 1:
            continue                                   # an all-zero token
        if m == 2:
            x[m] = rng.standard_normal(K)
            continue
        # amax = 254 -> a_s = 2: integers k give k / 2, odd k exact ties
        x[m] = rng.integers(-254, 255, size=K).astype(np.float32)
        x[m, 0] = 254.0
        # values one bf16 ulp off the ties (above 128 a bf16 ulp is 1.0, so
        # take them below: 2*j + 1 +- 1/128 for small j)
        j = rng.integers(0, 60, size=K // 8)
        x[m, 1:K // 8 + 1] = 2.0 * j + 1.0 + rng.choice([-1.0, 1.0], size=K // 8) / 128.0
    bits = x.view(np.uint32)
    return ((bits + 0x7FFF + ((bits >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("N", [384, 128 * 300])    # split-K clusters; one CTA per tile
@pytest.mark.parametrize("M", [1, 4, 16])
def test_fused_quant_gemv_ties_bit_identical(N, M):
    """Rows full of exact and near half-integer quotients: the quantization
    (round half to even of the fp32 quotient) matches the oracle bit for bit,
    and the one-call linear on the GEMV path gives the bits of
    egopq_quant_act_i8 followed by the GEMV, on split-K clusters and on grids
    of one CTA per tile."""
    K = 3584
    x = _tie_rows(M, K, 30 + M)
    w = synth.w4_weights(14, M, 0, N, K)
    packed = eg.pack_w4(*dev_weights(w))
    xd = to_dev(x, torch.bfloat16)
    y1 = eg.w4a8_linear(xd, packed, N, path=eg.PATH_GEMV)
    a = eg.quant_act(xd)
    y2 = eg.w4a8_gemm(a, packed, N, K, path=eg.PATH_GEMV)
    assert torch.equal(y1, y2)
    a_q, a_s, _ = oracle.quant_act(x)
    assert np.array_equal(a.a_q.cpu().numpy(), a_q)
    cols = np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N)]))
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q[cols], w.scale_f16[cols], w.zero[cols])
    check_bf16_output(to_host_bits(y1)[:, cols], y_ref, f"fused quant GEMV N={N} M={M}")
