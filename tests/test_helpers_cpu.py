"""Pins of the test-side decoders (they read kernel operand buffers, so a slip
in them would hide or fake a kernel error)."""
import numpy as np

from helpers import TC_PLANE_ORDER, decode_tc_operand, e4m3_to_f64


def test_e4m3_decoder_known_codes():
    # OCP FP8 E4M3: 1.0 = 0x38, 15 = 1.875 * 2^3 = 0x57, -8 = 0xD0, 448 = 0x7E,
    # smallest subnormal 2^-9 = 0x01, -0 = 0x80
    codes = [0x00, 0x38, 0x40, 0x44, 0x57, 0xD0, 0xB8, 0x7E, 0x01, 0x80]
    want = [0.0, 1.0, 2.0, 3.0, 15.0, -8.0, -1.0, 448.0, 2.0 ** -9, -0.0]
    assert e4m3_to_f64(codes).tolist() == want


def test_decode_tc_operand_planes_roundtrip():
    # encode by hand with an independent table and permutation, then decode
    enc = {v: c for v, c in zip(range(-8, 16), [0xD0, 0xCE, 0xCC, 0xCA, 0xC8, 0xC4, 0xC0, 0xB8,
                                                 0x00, 0x38, 0x40, 0x44, 0x48, 0x4A, 0x4C, 0x4E,
                                                 0x50, 0x51, 0x52, 0x53, 0x54, 0x55, 0x56, 0x57])}
    rng = np.random.default_rng(3)
    M, K = 3, 16
    a = rng.integers(-127, 128, size=(M, K))
    buf = np.zeros(2 * M * K, np.uint8)
    for m in range(M):
        for k in range(K):
            run, off = divmod(k, 8)
            q = int(np.nonzero(TC_PLANE_ORDER == off)[0][0])
            buf[m * K + run * 8 + q] = enc[int(a[m, k]) >> 4]
            buf[M * K + m * K + run * 8 + q] = enc[int(a[m, k]) & 15]
    assert np.array_equal(decode_tc_operand(buf, M, K, e4m3_planes=True), a)
    # the other form holds fp16 codes
    f16 = a.astype(np.float16).view(np.uint8).reshape(-1)
    assert np.array_equal(decode_tc_operand(f16, M, K, e4m3_planes=False), a)
