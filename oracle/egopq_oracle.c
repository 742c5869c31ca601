/*
 * egopq_oracle.c -- plain CPU oracle for the W4A8 packed-linear GEMM and its
 * W4A16 / W8A16 / W8A8 variants.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load or call this file. The product path
 * never does; it shares no code, header or table with it.
 *
 * Integers accumulate in int64; every floating-point combination is fp64; the
 * final bf16 rounding is taken directly from the fp64 value (ties to even).
 * No blocking, fusion or reordering beyond the definitions below.
 *
 * Sources (page title, section):
 *  - "The 4-bit CPU path", section "W4A8 - _C::int4_scaled_mm_cpu": the W4A8
 *    kernel consumes GPTQ-packed int4 weights and quantizes activations to
 *    int8; the exporter uses the checkpoint's zero points, or the constant 8
 *    when none are set (the symmetric grid).
 *  - "EgoPQ Real-Serving Handoff", section 2 "External Artifacts": native
 *    W4A8 serving needs exact per-group _gptq_scale and _gptq_zero metadata.
 *  - "The 4-bit CPU path", sections "W4A16 - PyTorch tinygemm" and "Building
 *    a checkpoint": weight-only int4 with bf16 activations, group size 128.
 *  - "Serve a pre-quantized int8 weight-only DiT via compressed-tensors ...",
 *    sections "Context" and "Plan": int8 weight-only (W8A16) linears; sections
 *    "Directive after the int8-wo result" and "Round two": W8A8 int8-dynamic.
 *  - "The 4-bit CPU path", section "W4A16 - PyTorch tinygemm": the
 *    dequantize-once bf16 weight of the dense comparison path.
 *  - GPTQ checkpoint tensors (qweight / qzeros / scales): the pages name the
 *    metadata only; the byte layout read here is the common export
 *    convention, stated at oracle_gptq_unpack.
 *  - The combination y = a_s * sum_g s * (sum_k a_q*w_q - z * sum_k a_q) is
 *    the plainest reading of those pieces: dequantized weight s*(w_q - z),
 *    dequantized activation a_s*a_q.
 *
 * Readings where the pages are silent: a_s = absmax/127 as an fp32 quotient;
 * a_q = clamp(round_half_even(x / a_s), -127, 127) with an fp32 quotient; an
 * all-zero row has a_s = 0 and a_q = 0; absmax is taken over the whole row.
 *
 * Parity pins: every function here is checked by the CPU tests against brute
 * force (dequantize-then-fp64-matmul, exact rationals), library routines and
 * invariants; none is marked parity-unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ---- number formats, from their bit definitions ------------------------- */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_fp16_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)f, -24);                 /* subnormal / zero */
  else if (e == 31) v = f ? NAN : INFINITY;
  else v = ldexp(1.0 + (double)f / 1024.0, e - 15);
  return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* double -> bfloat16, round to nearest, ties to even, in one step from the
 * double (no intermediate float). bf16 keeps 7 fraction bits and binary32's
 * exponent range: quantum 2^(E-7) for |x| in [2^E, 2^(E+1)), E >= -126, and
 * 2^-133 below (subnormals). Values that round past the largest finite bf16
 * become infinity. */
uint16_t oracle_bf16_from_double(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(a)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);       /* a = f * 2^e, f in [0.5, 1) */
  int E = e - 1;      /* a in [2^E, 2^(E+1)) */
  if (E < -126) E = -126;
  double q = ldexp(1.0, E - 7);
  double r = nearbyint(a / q) * q; /* exact scaling by a power of two */
  if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, 4);
  return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ---- per-token symmetric int8 activation quantization ------------------- */

/* For each row m: amax = max_k |x|; a_s = amax / 127 (fp32 quotient);
 * a_q = clamp(round_half_even(x / a_s), -127, 127) (fp32 quotient);
 * asum[m][g] = sum of a_q over group g. asum may be NULL. */
void oracle_quant_act(const uint16_t* x_bf16, int64_t M, int64_t K, int64_t group,
                      int8_t* a_q, float* a_s, int32_t* asum) {
  int64_t G = K / group;
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    const uint16_t* xr = x_bf16 + m * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      float v = fabsf((float)oracle_bf16_to_double(xr[k]));
      if (v > amax) amax = v;
    }
    float s = amax / 127.0f;
    a_s[m] = s;
    for (int64_t k = 0; k < K; ++k) {
      int q = 0;
      if (amax != 0.0f) {
        float t = (float)oracle_bf16_to_double(xr[k]) / s;
        float r = nearbyintf(t); /* default rounding: to nearest, ties to even */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q = (int)r;
      }
      a_q[m * K + k] = (int8_t)q;
    }
    if (asum) {
      for (int64_t g = 0; g < G; ++g) {
        int64_t acc = 0;
        for (int64_t k = g * group; k < (g + 1) * group; ++k) acc += a_q[m * K + k];
        asum[m * G + g] = (int32_t)acc;
      }
    }
  }
}

/* ---- W4A8 ----------------------------------------------------------------- */

/* Group partials Q[m][n][g] = sum_{k in g} a_q[m,k]*w_q[n,k]
 *                            - z[n,g] * sum_{k in g} a_q[m,k]   (int64). */
void oracle_group_partials(const int8_t* a_q, const uint8_t* w_q, const uint8_t* z,
                           int64_t M, int64_t N, int64_t K, int64_t group, int64_t* Q) {
  int64_t G = K / group;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n)
      for (int64_t g = 0; g < G; ++g) {
        int64_t dot = 0, sa = 0;
        for (int64_t k = g * group; k < (g + 1) * group; ++k) {
          dot += (int64_t)a_q[m * K + k] * (int64_t)w_q[n * K + k];
          sa += (int64_t)a_q[m * K + k];
        }
        Q[(m * N + n) * G + g] = dot - (int64_t)z[n * G + g] * sa;
      }
}

/* y[m][n] = a_s[m] * sum_g s[n,g] * Q[m][n][g], fp64, then bf16.
 * y64 (fp64 result) and y_bf16 may each be NULL. */
void oracle_w4a8(const int8_t* a_q, const float* a_s, const uint8_t* w_q,
                 const uint16_t* s_f16, const uint8_t* z, int64_t M, int64_t N,
                 int64_t K, int64_t group, double* y64, uint16_t* y_bf16) {
  int64_t G = K / group;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t g = 0; g < G; ++g) {
        int64_t dot = 0, sa = 0;
        for (int64_t k = g * group; k < (g + 1) * group; ++k) {
          dot += (int64_t)a_q[m * K + k] * (int64_t)w_q[n * K + k];
          sa += (int64_t)a_q[m * K + k];
        }
        int64_t q = dot - (int64_t)z[n * G + g] * sa;
        acc += oracle_fp16_to_double(s_f16[n * G + g]) * (double)q;
      }
      double y = (double)a_s[m] * acc;
      if (y64) y64[m * N + n] = y;
      if (y_bf16) y_bf16[m * N + n] = oracle_bf16_from_double(y);
    }
}

/* ---- W4A16: bf16 activations, int4 group-wise weights -------------------- */

/* y[m][n] = sum_g s[n,g] * sum_{k in g} x[m,k] * (w_q[n,k] - z[n,g]). */
void oracle_w4a16(const uint16_t* x_bf16, const uint8_t* w_q, const uint16_t* s_f16,
                  const uint8_t* z, int64_t M, int64_t N, int64_t K, int64_t group,
                  double* y64, uint16_t* y_bf16) {
  int64_t G = K / group;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t g = 0; g < G; ++g) {
        double part = 0.0;
        int64_t zz = z[n * G + g];
        for (int64_t k = g * group; k < (g + 1) * group; ++k)
          part += oracle_bf16_to_double(x_bf16[m * K + k]) *
                  (double)((int64_t)w_q[n * K + k] - zz);
        acc += oracle_fp16_to_double(s_f16[n * G + g]) * part;
      }
      if (y64) y64[m * N + n] = acc;
      if (y_bf16) y_bf16[m * N + n] = oracle_bf16_from_double(acc);
    }
}

/* ---- GPTQ checkpoint tensors -> logical codes, scales and zero points ---- */

/* Reading of the checkpoint format (the pages name the _gptq_scale and
 * _gptq_zero metadata -- "EgoPQ Real-Serving Handoff", section 2 "External
 * Artifacts"; "The 4-bit CPU path", section "W4A8" -- but print no byte
 * layout; this is the common GPTQ export convention):
 *   qweight int32 [K/8][N]: word (r, n) holds the codes of rows k = 8r + i,
 *           i = 0..7, of output n in bits 4i .. 4i+3 (low nibble first);
 *   qzeros  int32 [G][N/8]: word (g, c) holds the zero points of outputs
 *           n = 8c + j in bits 4j .. 4j+3;
 *   scales  fp16  [G][N].
 * The zero point is the stored nibble plus zero_offset (1 for exporters that
 * store z - 1). Outputs in the logical layout: w_q [N][K], s [N][G], z [N][G].
 * Returns how many zero points fall outside [0, 15] (not representable in the
 * 4-bit record; those entries of z hold the value modulo 16). */
int64_t oracle_gptq_unpack(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales,
                           int64_t N, int64_t K, int64_t group, int64_t zero_offset,
                           uint8_t* w_q, uint16_t* s_f16, uint8_t* z) {
  int64_t G = K / group, bad = 0;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      uint32_t word = (uint32_t)qweight[(k / 8) * N + n];
      w_q[n * K + k] = (uint8_t)((word >> (4 * (k % 8))) & 0xFu);
    }
  for (int64_t g = 0; g < G; ++g)
    for (int64_t n = 0; n < N; ++n) {
      uint32_t word = (uint32_t)qzeros[g * (N / 8) + n / 8];
      int64_t zz = (int64_t)((word >> (4 * (n % 8))) & 0xFu) + zero_offset;
      if (zz < 0 || zz > 15) ++bad;
      z[n * G + g] = (uint8_t)(zz & 0xF);
      s_f16[n * G + g] = scales[g * N + n];
    }
  return bad;
}

/* ---- dense twin operand: the int4 weight dequantized once to bf16 -------- */

/* w[n][k] = bf16( s[n,g] * (w_q[n,k] - z[n,g]) ), g = k / group. The product
 * is exact in fp64 (an 11-bit fp16 significand times an integer of magnitude
 * at most 15); the one rounding is fp64 -> bf16, ties to even. ("The 4-bit
 * CPU path", section "W4A16 - PyTorch tinygemm": large batches dequantize the
 * weight to bf16 once and hand it to an ordinary dense GEMM.) */
void oracle_dequant_w4_bf16(const uint8_t* w_q, const uint16_t* s_f16, const uint8_t* z,
                            int64_t N, int64_t K, int64_t group, uint16_t* w_bf16) {
  int64_t G = K / group;
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      int64_t g = k / group;
      double v = oracle_fp16_to_double(s_f16[n * G + g]) *
                 (double)((int64_t)w_q[n * K + k] - (int64_t)z[n * G + g]);
      w_bf16[n * K + k] = oracle_bf16_from_double(v);
    }
}

/* ---- W8A16: bf16 activations, int8 per-output-channel weights ------------ */

/* y[m][n] = s[n] * sum_k x[m,k] * w_q[n,k]. */
void oracle_w8a16(const uint16_t* x_bf16, const int8_t* w_q, const uint16_t* s_f16,
                  int64_t M, int64_t N, int64_t K, double* y64, uint16_t* y_bf16) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k)
        acc += oracle_bf16_to_double(x_bf16[m * K + k]) * (double)w_q[n * K + k];
      double y = oracle_fp16_to_double(s_f16[n]) * acc;
      if (y64) y64[m * N + n] = y;
      if (y_bf16) y_bf16[m * N + n] = oracle_bf16_from_double(y);
    }
}

/* ---- W8A8: int8 per-token activations, int8 per-output-channel weights --- */

/* "Serve a pre-quantized int8 weight-only DiT via compressed-tensors ...",
 * sections "Directive after the int8-wo result" and "Round two": W8A8
 * int8-dynamic -- activations quantized per token at run time (the same
 * quantizer as above), weights int8 per output channel, int8 products summed
 * as integers, then both scales applied:
 *   y[m][n] = a_s[m] * s[n] * sum_k a_q[m,k] * w_q[n,k].
 * dot (int64 [M][N]), y64 and y_bf16 may each be NULL. */
void oracle_w8a8(const int8_t* a_q, const float* a_s, const int8_t* w_q, const uint16_t* s_f16,
                 int64_t M, int64_t N, int64_t K, int64_t* dot, double* y64,
                 uint16_t* y_bf16) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      int64_t d = 0;
      for (int64_t k = 0; k < K; ++k) d += (int64_t)a_q[m * K + k] * (int64_t)w_q[n * K + k];
      double y = (double)a_s[m] * oracle_fp16_to_double(s_f16[n]) * (double)d;
      if (dot) dot[m * N + n] = d;
      if (y64) y64[m * N + n] = y;
      if (y_bf16) y_bf16[m * N + n] = oracle_bf16_from_double(y);
    }
}

/* ---- packed int4 weight layout ------------------------------------------- */
/*
 * The packed buffer for an N x K weight with group 128 (K % 128 == 0,
 * N % 128 == 0; G = K/128, T = N/128) is one 8512-byte record per (row block
 * t, group g) -- rows n = 128t..128t+127, columns k = 128g..128g+127 -- at
 * ((t*G + g) * 8512), records of one row block consecutive in g:
 *
 *  codes   bytes [0, 8192): the 16-byte unit for chunk c (0..3) of row r
 *          (0..127) sits at (c*128 + r) * 16; chunk c holds k = 128g + 32c ..
 *          +31. Inside the unit, little-endian 32-bit word j (0..3) holds the
 *          eight codes k0 = 128g + 32c + 8j .. k0+7; nibble p (bits 4p..4p+3)
 *          carries k0 + 2p for p < 4 and k0 + 2(p-4) + 1 for p >= 4.
 *  scales  bytes [8192, 8448): s[n,g] as fp16 at 8192 + 2r.
 *  zeros   bytes [8448, 8512): z[n,g] in byte 8448 + r/2, low nibble for even
 *          r, high nibble for odd r.
 *
 * Total T*G*8512 = N*K/2 + 2.5*N*G bytes.
 */
int64_t oracle_packed_w4_bytes(int64_t N, int64_t K, int64_t group) {
  if (group != 128 || K <= 0 || N <= 0 || K % 128 || N % 128) return 0;
  return (N / 128) * (K / 128) * 8512;
}

/* Byte offset and nibble shift of code (n, k). */
void oracle_code_location(int64_t N, int64_t K, int64_t n, int64_t k,
                          int64_t* byte_offset, int* shift) {
  (void)N;
  int64_t G = K / 128;
  int64_t t = n / 128, r = n % 128, g = k / 128, kk = k % 128;
  int64_t c = kk / 32, j = (kk % 32) / 8, e = kk % 8;
  int p = (e % 2 == 0) ? (int)(e / 2) : (int)(4 + e / 2);
  *byte_offset = (t * G + g) * 8512 + (c * 128 + r) * 16 + j * 4 + p / 2;
  *shift = (p % 2) * 4;
}

int oracle_pack_w4(const uint8_t* w_q, const uint16_t* s_f16, const uint8_t* z,
                   int64_t N, int64_t K, int64_t group, uint8_t* packed) {
  int64_t total = oracle_packed_w4_bytes(N, K, group);
  if (!total) return -2;
  int64_t G = K / 128;
  memset(packed, 0, (size_t)total);
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) {
      int64_t off;
      int sh;
      oracle_code_location(N, K, n, k, &off, &sh);
      packed[off] |= (uint8_t)((w_q[n * K + k] & 0xF) << sh);
    }
  for (int64_t n = 0; n < N; ++n)
    for (int64_t g = 0; g < G; ++g) {
      uint8_t* rec = packed + ((n / 128) * G + g) * 8512;
      int64_t r = n % 128;
      uint16_t v = s_f16[n * G + g];
      rec[8192 + 2 * r] = (uint8_t)(v & 0xFF);
      rec[8192 + 2 * r + 1] = (uint8_t)(v >> 8);
      rec[8448 + r / 2] |= (uint8_t)((z[n * G + g] & 0xF) << ((r % 2) * 4));
    }
  return 0;
}
