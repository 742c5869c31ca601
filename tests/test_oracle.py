"""Pins for the CPU oracle, independent of the oracle itself.

Each check ties the oracle to something it cannot agree with by construction:
values fixed by number-format definitions (tests/golden/), exact rational
brute force on a hand-sized example, dequantize-then-fp64-matmul, an int64
library matmul, special cases that reduce to a simpler method (the symmetric
grid, zero point = 8), and invariants. A dropped term, a wrong sign or index, or
a transposed operand in the oracle fails at least one of them.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers ---

def bf16_bits_to_float(b):
    return np.asarray(b, np.uint16).astype(np.uint32).__lshift__(16).view(np.float32)


def fp16_bits_to_double(b):
    return np.asarray(b, np.uint16).view(np.float16).astype(np.float64)


def frac_to_bf16_bits(fr: Fraction) -> int:
    """Nearest bf16 to an exact rational, ties to even, by bracketing with
    exact rationals (independent of the oracle's floating-point route)."""
    if fr == 0:
        return 0
    sign = 0x8000 if fr < 0 else 0
    a = abs(fr)
    E = math.floor(math.log2(a))
    while Fraction(2) ** E > a:
        E -= 1
    while Fraction(2) ** (E + 1) <= a:
        E += 1
    E = max(E, -126)
    q = Fraction(2) ** (E - 7)
    t = a / q
    fl = t.numerator // t.denominator
    rem = t - fl
    r = fl + 1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1) else fl
    val = r * q
    bits = np.array([float(val)], np.float32).view(np.uint32)[0] >> 16
    return sign | int(bits)


def rne_frac(fr: Fraction) -> int:
    fl = fr.numerator // fr.denominator
    rem = fr - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def to_bf16_bits_exact_ints(vals):
    """bf16 bit patterns of small integers (exact in bf16)."""
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def random_case(seed, M, N, K, group=128, outliers=True):
    w = synth.w4_weights(90 + seed, 0, 0, N, K, group)
    x = synth.activations(90 + seed, 0, 0, M, K, outliers)
    return x, w


def dequant_matmul_w4a8(a_q, a_s, w_q, s, z, group):
    """Brute force: X = a_s*a_q, W = s*(w_q - z) per group, Y = X @ W^T (fp64)."""
    N, K = w_q.shape
    X = a_s.astype(np.float64)[:, None] * a_q.astype(np.float64)
    sd = np.repeat(fp16_bits_to_double(s), group, axis=1)
    zd = np.repeat(z.astype(np.float64), group, axis=1)
    W = sd * (w_q.astype(np.float64) - zd)
    return X @ W.T


# ------------------------------------------------------- number formats ----

def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def test_bf16_from_double_golden():
    n = 0
    for line in _golden_rows("bf16_rounding.txt"):
        parts = line.split()
        # value expression may contain spaces; the bits field is the first 0x token
        idx = next(i for i, p in enumerate(parts) if p.startswith("0x"))
        expr, bits = " ".join(parts[:idx]), int(parts[idx], 16)
        value = eval(expr, {"__builtins__": {}}, {})
        got = oracle.bf16_from_double(value)
        assert got == bits, f"{expr}: got {got:#06x} want {bits:#06x}"
        n += 1
    assert n >= 20


def test_bf16_from_double_matches_torch_for_float_exact_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    f = (rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))).astype(np.float32)
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_from_double(float(v)) for v in f], np.uint16)
    assert np.array_equal(got, want)


def test_fp16_and_bf16_decoders_match_numpy():
    bits = np.arange(65536, dtype=np.uint16)
    ref16 = bits.view(np.float16).astype(np.float64)
    got16 = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    finite = np.isfinite(ref16)
    assert np.array_equal(got16[finite], ref16[finite])
    assert np.all(np.isinf(got16[np.isinf(ref16)]))
    with np.errstate(invalid="ignore"):
        refb = bf16_bits_to_float(bits).astype(np.float64)
    gotb = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    finite = np.isfinite(refb)
    assert np.array_equal(gotb[finite], refb[finite])


# ------------------------------------------------- activation quantization ----

def test_act_quant_golden_ties():
    for line in _golden_rows("act_quant_ties.txt"):
        xs, s, qs = [p.strip() for p in line.split("|")]
        x = np.array([int(v) for v in xs.split(",")], np.float32)
        want_q = np.array([int(v) for v in qs.split(",")], np.int8)
        xb = to_bf16_bits_exact_ints(x)[None, :]
        a_q, a_s, asum = oracle.quant_act(xb, group=4)
        assert a_s[0] == np.float32(float(s))
        assert np.array_equal(a_q[0], want_q)
        assert np.array_equal(asum[0], want_q.astype(np.int64).reshape(2, 4).sum(1))


def test_act_quant_properties_and_library_rounding():
    x, _ = random_case(1, 37, 64, 1024)
    a_q, a_s, asum = oracle.quant_act(x, 128)
    xf = bf16_bits_to_float(x)
    amax = np.abs(xf).max(axis=1)
    # a_s is the fp32 quotient amax / 127
    assert np.array_equal(a_s, (amax / np.float32(127)).astype(np.float32))
    # the absmax element lands on +-127
    arg = np.abs(xf).argmax(axis=1)
    assert np.all(np.abs(a_q[np.arange(37), arg]) == 127)
    assert np.all(np.abs(a_q.astype(np.int32)) <= 127)
    # round-half-even of the fp32 quotient, via numpy's rint (a library routine)
    lib = np.clip(np.rint((xf / a_s[:, None]).astype(np.float32)), -127, 127).astype(np.int8)
    assert np.array_equal(a_q, lib)
    # reconstruction error is at most half a step (plus the fp32 quotient's rounding)
    err = np.abs(a_q.astype(np.float64) * a_s[:, None] - xf)
    assert np.all(err <= a_s[:, None].astype(np.float64) * (0.5 + 1e-6))
    # group sums
    assert np.array_equal(asum, a_q.astype(np.int64).reshape(37, 8, 128).sum(2))


def test_act_quant_zero_row_and_outlier_row():
    x = np.zeros((2, 256), np.uint16)
    x[1, 7] = to_bf16_bits_exact_ints([-1000.0])[0]
    a_q, a_s, asum = oracle.quant_act(x, 128)
    assert a_s[0] == 0 and not a_q[0].any() and not asum[0].any()
    assert a_q[1, 7] == -127 and np.count_nonzero(a_q[1]) == 1
    assert asum[1, 0] == -127 and asum[1, 1] == 0


# ---------------------------------------------------------------- W4A8 ------

def hand_example():
    """M=2, K=8, N=8, group 4: integer activations (a_s = 1 and 2), codes
    w_q[n][k] = (3n+5k+1) mod 16, zeros z[n][g] = (2n+7g+3) mod 16 and scales
    s[n][g] = (n+1)/8 + g/4, all exact in their formats."""
    x = np.array([[127, -3, 5, 0, 64, -127, 1, 2],
                  [254, 1, 3, -5, 0, 7, -1, 100]], np.float32)
    N, K, grp = 8, 8, 4
    G = K // grp
    w = np.array([[(3 * n + 5 * k + 1) % 16 for k in range(K)] for n in range(N)], np.uint8)
    z = np.array([[(2 * n + 7 * g + 3) % 16 for g in range(G)] for n in range(N)], np.uint8)
    s_exact = [[Fraction(n + 1, 8) + Fraction(g, 4) for g in range(G)] for n in range(N)]
    s = np.array([[float(v) for v in row] for row in s_exact], np.float16).view(np.uint16)
    return x, w, z, s, s_exact, grp


def test_hand_example_exact_rationals():
    x, w, z, s, s_exact, grp = hand_example()
    xb = to_bf16_bits_exact_ints(x)
    a_q, a_s, asum = oracle.quant_act(xb, grp)
    # hand-derived: row0 has amax 127 (a_s = 1), row1 amax 254 (a_s = 2) with
    # ties 1/2 -> 0, -5/2 -> -2, -1/2 -> 0
    assert list(a_s) == [1.0, 2.0]
    assert a_q[1].tolist() == [127, 0, 2, -2, 0, 4, 0, 50]
    assert asum.tolist() == [[129, -60], [127, 54]]
    Q = oracle.group_partials(a_q, w, z, grp)
    assert Q[0, 0].tolist() == [-223, -327] and Q[1, 7].tolist() == [625, 78]
    y64, y = oracle.w4a8(a_q, a_s, w, s, z, grp)
    # exact rational brute force of y = a_s * sum_g s * sum_k a_q * (w_q - z)
    M, K = x.shape
    N, G = w.shape[0], K // grp
    for m in range(M):
        amax = max(abs(Fraction(int(v))) for v in x[m])
        a = amax / 127
        aq = [max(-127, min(127, rne_frac(Fraction(int(v)) / a))) for v in x[m]]
        assert aq == a_q[m].tolist()
        for n in range(N):
            acc = Fraction(0)
            for g in range(G):
                acc += s_exact[n][g] * sum(aq[k] * (int(w[n, k]) - int(z[n, g]))
                                           for k in range(g * grp, (g + 1) * grp))
            exact = a * acc
            assert Fraction(y64[m, n]) == exact
            assert y[m, n] == frac_to_bf16_bits(exact)
    # a few values worked by hand
    assert float(y64[0, 0]) == -150.5 and float(y64[1, 3]) == 1110.0
    assert bf16_bits_to_float(y[0]).tolist() == [-150, -225, 964, 454, -332, -1856, -2112, -354]
    assert bf16_bits_to_float(y[1]).tolist() == [-284, -298, -328, 1112, 158, -2544, -2576, 1448]


def test_hand_example_w4a16_equals_w4a8_for_integer_row():
    # row0 is integer with amax 127, so a_q = x and a_s = 1: W4A16 == W4A8
    x, w, z, s, _, grp = hand_example()
    xb = to_bf16_bits_exact_ints(x[:1])
    a_q, a_s, _ = oracle.quant_act(xb, grp)
    y64a, ya = oracle.w4a8(a_q, a_s, w, s, z, grp)
    y64b, yb = oracle.w4a16(xb, w, s, z, grp)
    assert np.array_equal(y64a, y64b) and np.array_equal(ya, yb)


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (5, 64, 256), (16, 256, 512), (3, 8, 384)])
def test_w4a8_matches_dequant_then_matmul(M, N, K):
    x, w = random_case(M + N, M, N, K)
    a_q, a_s, _ = oracle.quant_act(x, 128)
    y64, y = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero, 128)
    ref = dequant_matmul_w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero, 128)
    scale = np.abs(ref).max()
    assert np.max(np.abs(y64 - ref)) <= 1e-12 * scale
    # bf16 rounding of the fp64 result, checked against the exact-rational route
    for (m, n) in [(0, 0), (M - 1, N - 1), (M // 2, N // 3)]:
        assert y[m, n] == frac_to_bf16_bits(Fraction(float(y64[m, n])))


def test_group_partials_match_int64_library_matmul():
    x, w = random_case(3, 6, 40, 512)
    a_q, _, asum = oracle.quant_act(x, 128)
    Q = oracle.group_partials(a_q, w.w_q, w.zero, 128)
    A = a_q.astype(np.int64).reshape(6, 4, 128)
    W = w.w_q.astype(np.int64).reshape(40, 4, 128) - w.zero.astype(np.int64)[:, :, None]
    ref = np.einsum("mgk,ngk->mng", A, W)
    assert np.array_equal(Q, ref)
    # worst-case magnitude stays far inside int32
    assert np.abs(Q).max() <= 128 * 127 * 15


def test_zero_point_8_is_the_symmetric_grid():
    """With z = 8 everywhere the method is the symmetric int4 grid c = w_q - 8
    in [-8, 7] ("The 4-bit CPU path", section "W4A8": the exporter's constant 8)."""
    x, w = random_case(4, 9, 64, 384)
    z8 = np.full_like(w.zero, 8)
    a_q, a_s, _ = oracle.quant_act(x, 128)
    y64, _ = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, z8, 128)
    c = w.w_q.astype(np.int64) - 8
    assert c.min() >= -8 and c.max() <= 7
    A = a_q.astype(np.int64).reshape(9, 3, 128)
    P = np.einsum("mgk,ngk->mng", A, c.reshape(64, 3, 128))  # no zero-point term at all
    ref = a_s.astype(np.float64)[:, None] * (P * fp16_bits_to_double(w.scale_f16)[None]).sum(2)
    assert np.max(np.abs(y64 - ref)) <= 1e-13 * np.abs(ref).max()


def test_zero_activation_group_contributes_nothing():
    x, w = random_case(5, 4, 32, 512)
    a_q, a_s, _ = oracle.quant_act(x, 128)
    a_q[:, 256:384] = 0
    Q = oracle.group_partials(a_q, w.w_q, w.zero, 128)
    assert not Q[:, :, 2].any()
    y1, _ = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero, 128)
    w2 = w.w_q.copy()
    w2[:, 256:384] = (w2[:, 256:384] + 7) % 16
    z2 = w.zero.copy()
    z2[:, 2] = (z2[:, 2] + 3) % 16
    y2, _ = oracle.w4a8(a_q, a_s, w2, w.scale_f16, z2, 128)
    assert np.array_equal(y1, y2)


def test_codes_equal_zero_give_zero_and_scale_doubling_is_exact():
    x, w = random_case(6, 3, 16, 256)
    a_q, a_s, _ = oracle.quant_act(x, 128)
    wz = np.repeat(w.zero, 128, axis=1)
    y64, y = oracle.w4a8(a_q, a_s, wz, w.scale_f16, w.zero, 128)
    assert not y64.any() and not (y & 0x7FFF).any()
    s2 = (fp16_bits_to_double(w.scale_f16) * 2).astype(np.float16).view(np.uint16)
    ya, _ = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero, 128)
    yb, _ = oracle.w4a8(a_q, a_s, w.w_q, s2, w.zero, 128)
    assert np.array_equal(yb, 2 * ya)


def test_swapping_rows_and_columns_permutes_outputs():
    # catches transposed operands / mixed-up indices
    x, w = random_case(7, 4, 24, 256)
    a_q, a_s, _ = oracle.quant_act(x, 128)
    y, _ = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero, 128)
    pm, pn = np.array([2, 0, 3, 1]), np.random.default_rng(0).permutation(24)
    yp, _ = oracle.w4a8(a_q[pm], a_s[pm], w.w_q[pn], w.scale_f16[pn], w.zero[pn], 128)
    assert np.array_equal(yp, y[pm][:, pn])


# ------------------------------------------------------ W4A16 and W8A16 -----

@pytest.mark.parametrize("M,N,K", [(1, 64, 256), (7, 32, 384)])
def test_w4a16_matches_dequant_then_matmul(M, N, K):
    x, w = random_case(10 + M, M, N, K, outliers=False)
    y64, y = oracle.w4a16(x, w.w_q, w.scale_f16, w.zero, 128)
    X = bf16_bits_to_float(x).astype(np.float64)
    W = np.repeat(fp16_bits_to_double(w.scale_f16), 128, 1) * (
        w.w_q.astype(np.float64) - np.repeat(w.zero.astype(np.float64), 128, 1))
    ref = X @ W.T
    assert np.max(np.abs(y64 - ref)) <= 1e-12 * np.abs(ref).max()


@pytest.mark.parametrize("M,N,K", [(1, 64, 256), (6, 48, 512)])
def test_w8a16_matches_dequant_then_matmul(M, N, K):
    w8, s8 = synth.w8_weights(4, 0, 0, N, K)
    x = synth.activations(4, 0, 0, M, K, outliers=False)
    y64, y = oracle.w8a16(x, w8, s8)
    ref = bf16_bits_to_float(x).astype(np.float64) @ (
        w8.astype(np.float64) * fp16_bits_to_double(s8)[:, None]).T
    assert np.max(np.abs(y64 - ref)) <= 1e-12 * np.abs(ref).max()
    assert w8.min() >= -127 and w8.max() <= 127


# ------------------------------------------------------------ GPTQ import --

def _i32(u):
    return np.array(u, dtype=np.uint32).view(np.int32)


def test_gptq_unpack_hand_words():
    """Words written by hand from the format (codes of k = 8r + i in bits
    4i..4i+3 of qweight[r][n]; zero points of n = 8c + j in bits 4j..4j+3 of
    qzeros[g][c]): 0x87654321 is codes 1..8 in K order, 0x0FEDCBA9 is
    9..15, 0; words with the sign bit set (0xF0000000, 0x80000000) give a top
    code of 15 and 8. A reversed nibble order, a transposed qweight, an
    arithmetic-shift sign smear or a dropped offset fails one of them."""
    N, K = 8, 128
    qweight = np.zeros((K // 8, N), np.uint32)
    qweight[0, 0] = 0x87654321
    qweight[1, 0] = 0x0FEDCBA9
    qweight[0, 1] = 0x11111111
    qweight[2, 1] = 0xF0000000
    qweight[3, 7] = 0x80000000
    qzeros = np.array([[0x76543210]], np.uint32)
    scales = (0x3C00 + np.arange(N, dtype=np.uint16)).reshape(1, N)
    for off in (0, 1):
        w_q, sc, z, bad = oracle.gptq_unpack(_i32(qweight), _i32(qzeros), scales, N, K, 128, off)
        assert bad == 0
        assert list(w_q[0, :16]) == [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 0]
        assert list(w_q[1, :8]) == [1] * 8 and list(w_q[1, 16:24]) == [0] * 7 + [15]
        assert list(w_q[7, 24:32]) == [0] * 7 + [8]
        assert w_q[2:7].max() == 0 and w_q[0, 16:].max() == 0
        assert list(z[:, 0]) == [n + off for n in range(N)]
        assert list(sc[:, 0]) == list(scales[0])


def test_gptq_unpack_counts_unrepresentable_zeros():
    """Offset 1 (stored z - 1): a stored 15 is z = 16, outside the 4-bit
    range; each such entry is counted."""
    N, K = 16, 256
    qweight = np.zeros((K // 8, N), np.int32)
    qzeros = np.zeros((2, N // 8), np.uint32)
    qzeros[1, 1] = 0xF00000F0  # n = 9 and n = 15 of group 1
    scales = np.full((2, N), 0x3C00, np.uint16)
    _, _, z, bad = oracle.gptq_unpack(qweight, _i32(qzeros), scales, N, K, 128, 1)
    assert bad == 2
    _, _, z0, bad0 = oracle.gptq_unpack(qweight, _i32(qzeros), scales, N, K, 128, 0)
    assert bad0 == 0 and z0[9, 1] == 15 and z0[15, 1] == 15 and z0[8, 1] == 0


# ------------------------------------------------- dequantized bf16 weight -

def test_dequant_w4_bf16_hand_values():
    """One 1x128 group per case, worked by hand (fp16 scale bits, code, zero ->
    bf16 bits): 0.5*(3-1) = 1.0; 0.5*(0-15) = -7.5; (1+2^-10)*3 = 3.0029296875
    rounds down to 3.0; q == z gives +0."""
    cases = [(0x3800, 3, 1, 0x3F80), (0x3800, 0, 15, 0xC0F0),
             (0x3C01, 3, 0, 0x4040), (0x3C00, 7, 7, 0x0000)]
    for sb, q, z, want in cases:
        w = np.full((1, 128), q, np.uint8)
        got = oracle.dequant_w4_bf16(w, np.array([[sb]], np.uint16), np.array([[z]], np.uint8))
        assert np.all(got == want), (hex(sb), q, z, hex(int(got[0, 0])))


def test_dequant_w4_bf16_ties_to_even():
    """Products exactly halfway between two bf16 values: 1 + 2^-8 lies between
    1.0 (0x3F80, even) and 1 + 2^-7 (0x3F81); 1 + 3*2^-8 between 0x3F81 and
    0x3F82 (even). A truncating or round-half-up conversion fails one of them."""
    for sb, want in [(0x3C04, 0x3F80), (0x3C0C, 0x3F82)]:
        w = np.full((1, 128), 1, np.uint8)
        got = oracle.dequant_w4_bf16(w, np.array([[sb]], np.uint16), np.zeros((1, 1), np.uint8))
        assert np.all(got == want), hex(int(got[0, 0]))


def test_dequant_w4_bf16_matches_library_conversion():
    """Random codes, zeros and scales over several groups: the fp32 product is
    exact, so torch's fp32 -> bf16 conversion (round to nearest even) of it
    gives the same bits; a transposed scale index or a sign slip would not."""
    torch = pytest.importorskip("torch")
    N, K = 256, 512
    w = synth.w4_weights(11, 0, 0, N, K)
    got = oracle.dequant_w4_bf16(w.w_q, w.scale_f16, w.zero)
    s32 = torch.from_numpy(w.scale_f16.view(np.float16).astype(np.float32))
    q = torch.from_numpy(w.w_q.astype(np.float32))
    z = torch.from_numpy(w.zero.astype(np.float32))
    ref = (s32.repeat_interleave(128, 1) * (q - z.repeat_interleave(128, 1))).to(torch.bfloat16)
    assert np.array_equal(got, ref.view(torch.int16).numpy().view(np.uint16))


def test_dequant_w4_bf16_reproduces_w4a16_on_a_basis_vector():
    """x = e_k (a one at column k): the W4A16 oracle's fp64 output is exactly
    the unrounded dequantized weight column, which rounds to the same bits."""
    N, K = 128, 256
    w = synth.w4_weights(12, 0, 0, N, K)
    dq = oracle.dequant_w4_bf16(w.w_q, w.scale_f16, w.zero)
    for k in (0, 127, 128, 255):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        _, y = oracle.w4a16(x, w.w_q, w.scale_f16, w.zero)
        assert np.array_equal(y[0], dq[:, k])


# ---------------------------------------------------------------- W8A8 -----

def test_w8a8_hand_example():
    """2 tokens x 3 channels x K = 4, worked by hand.
    a = [[1, 2, -3, 4], [-127, 0, 0, 4]], w = [[3, -1, 2, 1], [1, 0, 0, 0],
    [0, 0, 0, 1]]: dots [[3-2-6+4, 1, 4], [-381+4, -127, 4]] = [[-1, 1, 4],
    [-377, -127, 4]]. With a_s = [0.5, 2] and s = [1, 0.25, -2]:
    y = [[-0.5, 0.125, -4], [-754, -63.5, -16]]; in bf16 -754 lies halfway
    between -752 and -756 and rounds to the even mantissa, -752 (0xC43C)."""
    a = np.array([[1, 2, -3, 4], [-127, 0, 0, 4]], np.int8)
    w = np.array([[3, -1, 2, 1], [1, 0, 0, 0], [0, 0, 0, 1]], np.int8)
    a_s = np.array([0.5, 2.0], np.float32)
    s = np.array([0x3C00, 0x3400, 0xC000], np.uint16)  # fp16 1, 0.25, -2
    dot, y64, y = oracle.w8a8(a, a_s, w, s)
    assert dot.tolist() == [[-1, 1, 4], [-377, -127, 4]]
    assert y64.tolist() == [[-0.5, 0.125, -4.0], [-754.0, -63.5, -16.0]]
    assert y.tolist() == [[0xBF00, 0x3E00, 0xC080], [0xC43C, 0xC27E, 0xC180]]


def test_w8a8_extreme_dot_is_exact():
    """All +-127 over K = 18944: the dot is +-18944 * 16129 = +-305547776,
    beyond 2^24 (a float accumulator would round) and inside int32."""
    K = 18944
    a = np.full((2, K), 127, np.int8)
    a[1] = -127
    w = np.full((1, K), 127, np.int8)
    dot, _, _ = oracle.w8a8(a, np.ones(2, np.float32), w, np.array([0x3C00], np.uint16))
    assert dot[:, 0].tolist() == [305547776, -305547776]


def test_w8a8_reduces_to_w8a16_on_integer_activations():
    """When every activation is an integer in [-127, 127] and each row's
    absmax is 127, quantization is the identity (a_s = 1), so W8A8 equals the
    separately pinned W8A16 on the same data."""
    rng = np.random.default_rng(5)
    M, N, K = 3, 5, 256
    xi = rng.integers(-127, 128, size=(M, K))
    xi[:, 7] = 127
    x = (xi.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    w8, s8 = synth.w8_weights(6, 0, 0, N, K)
    a_q, a_s, _ = oracle.quant_act(x)
    assert np.array_equal(a_q, xi.astype(np.int8)) and np.all(a_s == 1.0)
    _, y64, _ = oracle.w8a8(a_q, a_s, w8, s8)
    y64_ref, _ = oracle.w8a16(x, w8, s8)
    assert np.array_equal(y64, y64_ref)


@pytest.mark.parametrize("M,N,K", [(1, 8, 128), (5, 16, 640)])
def test_w8a8_matches_dequant_then_matmul(M, N, K):
    """Against fp64 dequantized operands: (a_s * a_q) @ (s * w_q)^T."""
    x = synth.activations(7, 0, 0, M, K)
    a_q, a_s, _ = oracle.quant_act(x)
    w8, s8 = synth.w8_weights(7, 0, 0, N, K)
    _, y64, _ = oracle.w8a8(a_q, a_s, w8, s8)
    ref = (a_q.astype(np.float64) * a_s.astype(np.float64)[:, None]) @ (
        w8.astype(np.float64) * fp16_bits_to_double(s8)[:, None]).T
    assert np.max(np.abs(y64 - ref)) <= 1e-12 * np.abs(ref).max()
    _, y64n, _ = oracle.w8a8(a_q, a_s, -w8, s8)                    # sign symmetry
    assert np.array_equal(y64n, -y64)


# ------------------------------------------------------------- packing ------

def unpack_reference(packed, N, K):
    """Decode the packed layout by reshaping (an independent route from the
    oracle's per-code location function)."""
    G, T = K // 128, N // 128
    rec = packed.reshape(T, G, 8512)
    codes = rec[:, :, :8192].reshape(T, G, 4, 128, 4, 4)   # t, g, c, r, j, byte
    b = codes.astype(np.uint32)
    word = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)  # t,g,c,r,j
    nib = np.stack([(word >> (4 * p)) & 0xF for p in range(8)], axis=-1)  # ...,p
    e = np.array([0, 2, 4, 6, 1, 3, 5, 7])  # nibble p -> k offset e(p)
    vals = np.empty_like(nib)
    vals[..., e] = nib  # vals[..., e(p)] = nib[..., p]
    # axes: t, g, c, r, j, e -> n = 128t + r, k = 128g + 32c + 8j + e
    w = vals.transpose(0, 3, 1, 2, 4, 5).reshape(N, K).astype(np.uint8)
    s = np.ascontiguousarray(rec[:, :, 8192:8448]).view(np.uint16)  # t, g, r
    s = s.transpose(0, 2, 1).reshape(N, G)
    zb = rec[:, :, 8448:8512]                                        # t, g, r/2
    z = np.empty((T, 128, G), np.uint8)
    z[:, 0::2, :] = (zb & 0xF).transpose(0, 2, 1)
    z[:, 1::2, :] = (zb >> 4).transpose(0, 2, 1)
    return w, np.ascontiguousarray(s), z.reshape(N, G)


def test_pack_roundtrip_and_index_pattern():
    N, K = 256, 384
    n = np.arange(N)[:, None]
    k = np.arange(K)[None, :]
    w = ((7 * n + 3 * k + (k // 128)) % 16).astype(np.uint8)
    G = K // 128
    s = (np.arange(N * G).reshape(N, G) % 60000).astype(np.uint16)
    z = ((n[:, :G] * 5 + np.arange(G)[None]) % 16).astype(np.uint8)
    packed = oracle.pack_w4(w, s, z)
    assert packed.size == N * K // 2 + 2 * G * N + G * N // 2
    w2, s2, z2 = unpack_reference(packed, N, K)
    assert np.array_equal(w2, w) and np.array_equal(s2, s) and np.array_equal(z2, z)


def test_pack_layout_spot_locations():
    # index-pattern probe: one code set, all others zero, see where it lands
    N, K = 256, 256
    for (nn, kk, want_byte, want_shift) in [
        (0, 0, 0, 0),                      # tile 0, chunk 0, row 0, word 0, nibble 0
        (0, 1, 2, 0),                      # k0+1 is nibble 4 -> byte 2, low
        (0, 2, 0, 4),                      # k0+2 is nibble 1 -> byte 0, high
        (0, 7, 3, 4),                      # k0+7 is nibble 7 -> byte 3, high
        (0, 8, 4, 0),                      # next word
        (0, 32, 128 * 16, 0),              # chunk 1 starts after 128 rows x 16 B
        (1, 0, 16, 0),                     # row 1
        (0, 128, 8512, 0),                 # group 1 of row block 0 (8512-byte records)
        (128, 0, 2 * 8512, 0),             # row block 1 (G = 2 groups per row block)
    ]:
        w = np.zeros((N, K), np.uint8)
        w[nn, kk] = 0xF
        packed = oracle.pack_w4(w, np.zeros((N, 2), np.uint16), np.zeros((N, 2), np.uint8))
        nz = np.flatnonzero(packed)
        assert nz.tolist() == [want_byte], (nn, kk, nz)
        assert packed[want_byte] == (0xF << want_shift)
        assert oracle.code_location(N, K, nn, kk) == (want_byte, want_shift)


def test_pack_rejects_unsupported_shapes():
    assert oracle.packed_w4_bytes(80, 128) == 0        # N does not tile 128 rows
    assert oracle.packed_w4_bytes(128, 200) == 0       # K not a multiple of the group
    assert oracle.packed_w4_bytes(128, 256, 64) == 0   # only group 128 is packed
    assert oracle.packed_w4_bytes(128, 256) == 128 * 128 + 2 * 2 * 128 + 128
    assert oracle.packed_w4_bytes(128, 256) == 2 * 8512
