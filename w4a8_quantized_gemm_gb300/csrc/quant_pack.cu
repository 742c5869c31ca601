// quant_pack.cu -- per-token int8 activation quantization and int4 weight
// packing kernels.
//
// Activation quantization follows "The 4-bit CPU path", section "W4A8 -
// _C::int4_scaled_mm_cpu" (activations are quantized to int8 at run time):
// symmetric per token, a_s = absmax / 127, a_q = round_half_even(x / a_s)
// clamped to +-127, both quotients IEEE fp32 (so the integer codes match any
// correctly rounded implementation bit for bit). The same pass emits the
// per-group sums of a_q that fold the zero points into the GEMM epilogue, and
// optionally the codes in the tensor-core operand form (two exact e4m3 planes
// for small token counts, exact fp16 integers otherwise).
//
// Weight packing lays GPTQ-style int4 codes (per-group _gptq_scale /
// _gptq_zero, "EgoPQ Real-Serving Handoff", section 2) out in 8512-byte
// records of 128 rows x 128 K -- codes, scales and zero points together -- so
// that one 1-D bulk copy stages everything a (row block, group) needs, and so
// that one AND/OR per 32-bit word yields two consecutive K values as an fp16
// pair. The layout is documented in include/egopq.h.
//
// Also here: rows longer than 8192 for up to 64 tokens are quantized by a
// cluster of CTAs (partial absmax through distributed shared memory); GPTQ
// checkpoint tensors (qweight / qzeros / scales) are packed directly; and a
// packed weight can be dequantized once to dense bf16.
#include "egopq_internal.h"

namespace egopq {

constexpr int kQuantThreads = 256;

// e4m3 code of an integer in [-16, 16] (exact: the conversion does not
// round).
__device__ __forceinline__ uint32_t e4m3_exact(int v) {
  return __nv_cvt_float_to_fp8((float)v, __NV_SATFINITE, __NV_E4M3);
}

// Writes the tensor-core operand form of the 8 codes q[0..7] (K = 8*vec ..
// 8*vec+7) of token m, as documented for a_tc in include/egopq.h: with
// fp8 = true two e4m3 planes [2][M][K] (high part a >> 4 in [-8, 7], low
// part a & 15, a = 16 * high + low) with each 8-run in the packed weights' nibble order (even offsets,
// then odd); otherwise fp16 [M][K].
__device__ __forceinline__ void store_tc_operand(void* a_tc, bool fp8, int64_t M, int64_t K,
                                                 int64_t m, int64_t vec, const int (&q)[8]) {
  if (fp8) {
    constexpr int kOrder[8] = {0, 2, 4, 6, 1, 3, 5, 7};
    uint32_t hi[2] = {0, 0}, lo[2] = {0, 0};
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      const int a = q[kOrder[b]];
      hi[b >> 2] |= e4m3_exact(a >> 4) << (8 * (b & 3));
      lo[b >> 2] |= e4m3_exact(a & 15) << (8 * (b & 3));
    }
    uint8_t* base = static_cast<uint8_t*>(a_tc);
    *reinterpret_cast<uint2*>(base + m * K + 8 * vec) = make_uint2(hi[0], hi[1]);
    *reinterpret_cast<uint2*>(base + M * K + m * K + 8 * vec) = make_uint2(lo[0], lo[1]);
  } else {
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 hv = __halves2half2(__int2half_rn(q[2 * i]), __int2half_rn(q[2 * i + 1]));
      h[i] = *reinterpret_cast<uint32_t*>(&hv);
    }
    reinterpret_cast<uint4*>(static_cast<uint16_t*>(a_tc) + m * K)[vec] =
        make_uint4(h[0], h[1], h[2], h[3]);
  }
}

__global__ void __launch_bounds__(kQuantThreads)
quant_act_kernel(const uint16_t* __restrict__ x, int64_t K, int8_t* __restrict__ a_q,
                 float* __restrict__ a_s, int32_t* __restrict__ a_gsum,
                 void* __restrict__ a_tc, bool tc_fp8) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int64_t m = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + m * K);
  const int64_t nvec = K / 8;  // 8 bf16 per 16-byte vector; K % 128 == 0
  __shared__ float warp_max[kQuantThreads / 32];

  float amax = 0.f;
  for (int64_t v = threadIdx.x; v < nvec; v += kQuantThreads) {
    uint4 p = __ldg(xr + v);
    uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[i] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int i = 1; i < kQuantThreads / 32; ++i) amax = fmaxf(amax, warp_max[i]);

  const float s = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) a_s[m] = s;
  const bool zero_row = (amax == 0.f);

  for (int64_t v = threadIdx.x; v < nvec; v += kQuantThreads) {
    uint4 p = __ldg(xr + v);
    uint32_t w[4] = {p.x, p.y, p.z, p.w};
    int q[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo = __uint_as_float(w[i] << 16);
      float hi = __uint_as_float(w[i] & 0xFFFF0000u);
      int ql = zero_row ? 0 : __float2int_rn(__fdiv_rn(lo, s));
      int qh = zero_row ? 0 : __float2int_rn(__fdiv_rn(hi, s));
      q[2 * i] = max(-127, min(127, ql));
      q[2 * i + 1] = max(-127, min(127, qh));
    }
    uint2 packed;
    packed.x = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
               ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
    packed.y = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) |
               ((uint32_t)(q[6] & 0xFF) << 16) | ((uint32_t)(q[7] & 0xFF) << 24);
    reinterpret_cast<uint2*>(a_q + m * K)[v] = packed;
    if (a_tc) store_tc_operand(a_tc, tc_fp8, gridDim.x, K, m, v, q);
    // 16 consecutive vectors make one 128-wide group; kQuantThreads % 16 == 0
    // K % 128 == 0, so the 16 lanes of a half-warp are all inside the loop or
    // all outside it; reduce within the half-warp only.
    int sum = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
    const unsigned half_mask = 0xFFFFu << (threadIdx.x & 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(half_mask, sum, o);
    if ((threadIdx.x & 15) == 0) a_gsum[m * (K / 128) + v / 16] = sum;
  }
}

// Single-pass variant: the whole row stays in registers (up to kRegVec 16-byte
// vectors per thread, K <= kQuantRegThreads * kRegVec * 8), so x is read from
// memory once. It waits for the preceding kernel only when the launch carried a
// programmatic dependency.
constexpr int kQuantRegThreads = 512;
constexpr int kRegVec = 8;

__global__ void __launch_bounds__(kQuantRegThreads)
quant_act_reg_kernel(const uint16_t* __restrict__ x, int64_t K, int8_t* __restrict__ a_q,
                     float* __restrict__ a_s, int32_t* __restrict__ a_gsum,
                     void* __restrict__ a_tc, bool tc_fp8) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int64_t m = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + m * K);
  const int nvec = (int)(K / 8);
  __shared__ float warp_max[kQuantRegThreads / 32];
  uint4 v[kRegVec];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kRegVec; ++i) {
    const int idx = threadIdx.x + i * kQuantRegThreads;
    v[i] = idx < nvec ? __ldg(xr + idx) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int i = 1; i < kQuantRegThreads / 32; ++i) amax = fmaxf(amax, warp_max[i]);
  const float s = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) a_s[m] = s;
  const bool zero_row = (amax == 0.f);
#pragma unroll
  for (int i = 0; i < kRegVec; ++i) {
    const int idx = threadIdx.x + i * kQuantRegThreads;
    if (idx >= nvec) break;  // whole half-warps leave together (nvec % 16 == 0)
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    int q[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16);
      const float hi = __uint_as_float(w[j] & 0xFFFF0000u);
      q[2 * j] = zero_row ? 0 : max(-127, min(127, __float2int_rn(__fdiv_rn(lo, s))));
      q[2 * j + 1] = zero_row ? 0 : max(-127, min(127, __float2int_rn(__fdiv_rn(hi, s))));
    }
    uint2 packed;
    packed.x = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
               ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
    packed.y = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) |
               ((uint32_t)(q[6] & 0xFF) << 16) | ((uint32_t)(q[7] & 0xFF) << 24);
    reinterpret_cast<uint2*>(a_q + m * K)[idx] = packed;
    if (a_tc) store_tc_operand(a_tc, tc_fp8, gridDim.x, K, m, idx, q);
    int sum = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
    const unsigned half_mask = 0xFFFFu << (threadIdx.x & 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(half_mask, sum, o);
    if ((threadIdx.x & 15) == 0) a_gsum[m * (K / 128) + idx / 16] = sum;
  }
}

// Long rows for few tokens: one token's row is split over a cluster of CTAs
// (whole 128-wide groups each, at most kSplitVec 16-byte vectors per thread),
// so that the per-element divisions spread over several SMs; the CTAs combine
// their partial absmax through distributed shared memory. Same arithmetic as
// the kernels above, element for element.
constexpr int kSplitThreads = 256;
constexpr int kSplitVec = 2;
constexpr int kSplitMaxVec = kSplitThreads * kSplitVec;  // vectors one CTA holds

__global__ void __launch_bounds__(kSplitThreads)
quant_act_split_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                       int8_t* __restrict__ a_q, float* __restrict__ a_s,
                       int32_t* __restrict__ a_gsum, void* __restrict__ a_tc, bool tc_fp8) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int C = (int)cluster_nctarank();
  const int rank = (int)cluster_ctarank();
  const int64_t m = blockIdx.x / C;
  const int G = (int)(K / 128);
  const int v0 = (int)((int64_t)rank * G / C) * 16, v1 = (int)((int64_t)(rank + 1) * G / C) * 16;
  const uint4* xr = reinterpret_cast<const uint4*>(x + m * K);
  __shared__ float warp_max[kSplitThreads / 32];
  __shared__ float cta_max;
  uint4 v[kSplitVec];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < kSplitVec; ++i) {
    const int idx = v0 + threadIdx.x + i * kSplitThreads;
    v[i] = idx < v1 ? __ldg(xr + idx) : make_uint4(0, 0, 0, 0);
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = warp_max[0];
#pragma unroll
    for (int i = 1; i < kSplitThreads / 32; ++i) a = fmaxf(a, warp_max[i]);
    cta_max = a;
  }
  cluster_sync_all();  // every CTA's partial maximum is in its shared memory
  amax = 0.f;
  for (int r = 0; r < C; ++r) amax = fmaxf(amax, ld_dsmem_f32(map_to_rank(smem_u32(&cta_max), r)));
  cluster_sync_all();  // no CTA leaves while another still reads its partial
  const float s = __fdiv_rn(amax, 127.0f);
  if (rank == 0 && threadIdx.x == 0) a_s[m] = s;
  const bool zero_row = (amax == 0.f);
#pragma unroll
  for (int i = 0; i < kSplitVec; ++i) {
    const int idx = v0 + threadIdx.x + i * kSplitThreads;
    if (idx >= v1) break;  // whole half-warps leave together (v0, v1 multiples of 16)
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    int q[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = __uint_as_float(w[j] << 16);
      const float hi = __uint_as_float(w[j] & 0xFFFF0000u);
      q[2 * j] = zero_row ? 0 : max(-127, min(127, __float2int_rn(__fdiv_rn(lo, s))));
      q[2 * j + 1] = zero_row ? 0 : max(-127, min(127, __float2int_rn(__fdiv_rn(hi, s))));
    }
    uint2 packed;
    packed.x = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
               ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
    packed.y = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) |
               ((uint32_t)(q[6] & 0xFF) << 16) | ((uint32_t)(q[7] & 0xFF) << 24);
    reinterpret_cast<uint2*>(a_q + m * K)[idx] = packed;
    if (a_tc) store_tc_operand(a_tc, tc_fp8, M, K, m, idx, q);
    int sum = q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7];
    const unsigned half_mask = 0xFFFFu << (threadIdx.x & 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(half_mask, sum, o);
    if ((threadIdx.x & 15) == 0) a_gsum[m * G + idx / 16] = sum;
  }
}

// nibble p of a packed word carries K offset kNibbleK[p] inside its 8-wide run
__device__ __constant__ int kNibbleK[8] = {0, 2, 4, 6, 1, 3, 5, 7};

// Packed records: one 8512-byte record per (row block t, group g) at
// (t*G + g) * 8512 -- codes [0, 8192), fp16 scales [8192, 8448), zero nibbles
// [8448, 8512) -- so one bulk copy stages everything a group of 128 rows needs.
constexpr int64_t kRecBytes = 8512;

__global__ void pack_codes_kernel(const uint8_t* __restrict__ w_q, int64_t N, int64_t K,
                                  uint8_t* __restrict__ out) {
  const int64_t G = K / 128;
  const int64_t nwords = N * K / 8;
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < nwords;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rec = w / 2048, u = w % 2048;
    const int64_t t = rec / G, g = rec % G;
    const int64_t unit = u / 4, j = u % 4;
    const int64_t c = unit / 128, r = unit % 128;
    const int64_t n = t * 128 + r, k0 = g * 128 + c * 32 + j * 8;
    const uint2 src = *reinterpret_cast<const uint2*>(w_q + n * K + k0);
    const uint8_t* b = reinterpret_cast<const uint8_t*>(&src);
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) word |= (uint32_t)(b[kNibbleK[p]] & 0xF) << (4 * p);
    *reinterpret_cast<uint32_t*>(out + rec * kRecBytes + u * 4) = word;
  }
}

__global__ void unpack_codes_kernel(const uint8_t* __restrict__ in, int64_t N, int64_t K,
                                    uint8_t* __restrict__ w_q) {
  const int64_t G = K / 128;
  const int64_t nwords = N * K / 8;
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < nwords;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rec = w / 2048, u = w % 2048;
    const int64_t t = rec / G, g = rec % G;
    const int64_t unit = u / 4, j = u % 4;
    const int64_t c = unit / 128, r = unit % 128;
    const int64_t n = t * 128 + r, k0 = g * 128 + c * 32 + j * 8;
    const uint32_t word = *reinterpret_cast<const uint32_t*>(in + rec * kRecBytes + u * 4);
    uint2 dst;
    uint8_t* b = reinterpret_cast<uint8_t*>(&dst);
#pragma unroll
    for (int p = 0; p < 8; ++p) b[kNibbleK[p]] = (word >> (4 * p)) & 0xF;
    *reinterpret_cast<uint2*>(w_q + n * K + k0) = dst;
  }
}

// scales [N][G] and zeros [N][G] into (and out of) the records
__global__ void pack_meta_kernel(const uint16_t* __restrict__ s, const uint8_t* __restrict__ z,
                                 int64_t N, int64_t G, uint8_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < G * N;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t g = i / N, n = i % N;
    uint8_t* rec = out + ((n / 128) * G + g) * kRecBytes;
    const int64_t r = n % 128;
    *reinterpret_cast<uint16_t*>(rec + 8192 + 2 * r) = s[n * G + g];
    if ((r & 1) == 0)
      rec[8448 + r / 2] = (uint8_t)((z[n * G + g] & 0xF) | ((z[(n + 1) * G + g] & 0xF) << 4));
  }
}

__global__ void unpack_meta_kernel(const uint8_t* __restrict__ in, int64_t N, int64_t G,
                                   uint16_t* __restrict__ s, uint8_t* __restrict__ z) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < G * N;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t g = i / N, n = i % N;
    const uint8_t* rec = in + ((n / 128) * G + g) * kRecBytes;
    const int64_t r = n % 128;
    s[n * G + g] = *reinterpret_cast<const uint16_t*>(rec + 8192 + 2 * r);
    const uint8_t b = rec[8448 + r / 2];
    z[n * G + g] = (r & 1) ? (b >> 4) : (b & 0xF);
  }
}

// Dequantize once: w[n][k] = bf16(s[n,g] * (w_q[n,k] - z[n,g])). One CTA per
// packed record (a 128-row x 128-K block); thread (c, r) reads the 16 code
// bytes of row r, K offsets c*32 .. c*32+31 (consecutive threads, consecutive
// 16-byte units) and writes those 32 values as 64 contiguous bytes of row n.
// The fp32 product is exact (11-bit scale significand times |q - z| <= 15),
// so the one rounding is the bf16 conversion (nearest, ties to even).
constexpr int kDequantThreads = 512;

__global__ void __launch_bounds__(kDequantThreads)
dequant_w4_kernel(const uint8_t* __restrict__ in, int64_t G, int64_t K, uint16_t* __restrict__ w) {
  const int64_t rec = blockIdx.x;
  const int64_t t = rec / G, g = rec % G;
  const int c = threadIdx.x / 128, r = threadIdx.x % 128;
  const uint8_t* rp = in + rec * kRecBytes;
  const uint4 v = *reinterpret_cast<const uint4*>(rp + (c * 128 + r) * 16);
  const float s = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(rp + 8192 + 2 * r)));
  const uint8_t zb = rp[8448 + r / 2];
  const int z = (r & 1) ? (zb >> 4) : (zb & 0xF);
  const uint32_t words[4] = {v.x, v.y, v.z, v.w};
  uint16_t* dst = w + (t * 128 + r) * K + g * 128 + c * 32;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t o[4] = {0u, 0u, 0u, 0u};  // bf16 pairs in K order
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      const int q = (int)((words[j] >> (4 * p)) & 0xF);
      // nibble p of a word: K offset 2p (p < 4) or 2(p - 4) + 1
      const int kk = p < 4 ? 2 * p : 2 * (p - 4) + 1;
      const uint32_t bits = __bfloat16_as_ushort(__float2bfloat16_rn(s * (float)(q - z)));
      o[kk >> 1] |= bits << (16 * (kk & 1));
    }
    *reinterpret_cast<uint4*>(dst + j * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// GPTQ checkpoint tensors straight into the packed records. qweight int32
// [K/8][N]: word (r, n) holds the codes of rows k = 8r + i of output n in bits
// 4i..4i+3, so the 8 codes of one packed word (K offsets k0 .. k0+7, k0 a
// multiple of 8) are one qweight word, its nibbles permuted to the record's
// order.
__global__ void pack_gptq_codes_kernel(const int32_t* __restrict__ qweight, int64_t N, int64_t K,
                                       uint8_t* __restrict__ out) {
  const int64_t G = K / 128;
  const int64_t nwords = N * K / 8;
  for (int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; w < nwords;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t rec = w / 2048, u = w % 2048;
    const int64_t t = rec / G, g = rec % G;
    const int64_t unit = u / 4, j = u % 4;
    const int64_t c = unit / 128, r = unit % 128;
    const int64_t n = t * 128 + r, k0 = g * 128 + c * 32 + j * 8;
    const uint32_t in = static_cast<uint32_t>(qweight[(k0 / 8) * N + n]);
    uint32_t word = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) word |= ((in >> (4 * kNibbleK[p])) & 0xFu) << (4 * p);
    *reinterpret_cast<uint32_t*>(out + rec * kRecBytes + u * 4) = word;
  }
}

// scales fp16 [G][N] and qzeros int32 [G][N/8] (zero point of output n = 8c + j
// in bits 4j..4j+3 of word (g, c), plus zero_offset) into the records; a zero
// point outside [0, 15] raises kErrRange (and is stored modulo 16).
__global__ void pack_gptq_meta_kernel(const int32_t* __restrict__ qzeros,
                                      const uint16_t* __restrict__ scales, int64_t N, int64_t G,
                                      int zero_offset, uint8_t* __restrict__ out) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < G * N;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t g = i / N, n = i % N;
    uint8_t* rec = out + ((n / 128) * G + g) * kRecBytes;
    const int64_t r = n % 128;
    *reinterpret_cast<uint16_t*>(rec + 8192 + 2 * r) = scales[g * N + n];
    if ((r & 1) == 0) {
      // n is even, so n and n + 1 share a qzeros word
      const uint32_t word = static_cast<uint32_t>(qzeros[g * (N / 8) + n / 8]);
      const int z0 = (int)((word >> (4 * (n % 8))) & 0xFu) + zero_offset;
      const int z1 = (int)((word >> (4 * (n % 8 + 1))) & 0xFu) + zero_offset;
      if (z0 < 0 || z0 > 15 || z1 < 0 || z1 > 15) raise_error(kErrRange);
      rec[8448 + r / 2] = (uint8_t)((z0 & 0xF) | ((z1 & 0xF) << 4));
    }
  }
}

static unsigned grid_for(int64_t work, int threads) {
  int64_t b = (work + threads - 1) / threads;
  return (unsigned)(b < 1 ? 1 : (b > 65535 * 8 ? 65535 * 8 : b));
}

cudaError_t launch_quant_act(const uint16_t* x, int64_t M, int64_t K, int8_t* a_q, float* a_s,
                             int32_t* a_gsum, void* a_tc, cudaStream_t st) {
  // few tokens: one wide CTA per row, one read of x (latency); many tokens:
  // narrower CTAs, several resident per SM (throughput)
  const bool reg = (M <= 64 && K <= (int64_t)kQuantRegThreads * kRegVec * 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, 1, 1);
  cfg.blockDim = dim3(reg ? kQuantRegThreads : kQuantThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool tc_fp8 = M <= kTcFp8MaxM;
  // rows longer than 1024 vectors for few tokens: split over a cluster of up
  // to 8 CTAs, each holding whole groups and at most kSplitMaxVec vectors
  const int64_t nvec = K / 8;
  if (M <= 64 && nvec > 1024) {
    const int64_t G = K / 128;
    int split = (int)((nvec + kSplitMaxVec - 1) / kSplitMaxVec);
    if (split < 2) split = 2;
    // each CTA's share, ceil(G / split) groups, must fit its registers
    if (split <= 8 && (G + split - 1) / split * 16 <= kSplitMaxVec) {
      cudaLaunchAttribute cattr[2];
      cattr[0] = attr[0];
      cattr[1].id = cudaLaunchAttributeClusterDimension;
      cattr[1].val.clusterDim.x = (unsigned)split;
      cattr[1].val.clusterDim.y = 1;
      cattr[1].val.clusterDim.z = 1;
      cfg.attrs = cattr;
      cfg.numAttrs = 2;
      cfg.gridDim = dim3((unsigned)(M * split), 1, 1);
      cfg.blockDim = dim3(kSplitThreads, 1, 1);
      return cudaLaunchKernelEx(&cfg, quant_act_split_kernel, x, M, K, a_q, a_s, a_gsum, a_tc,
                                tc_fp8);
    }
  }
  if (reg)
    return cudaLaunchKernelEx(&cfg, quant_act_reg_kernel, x, K, a_q, a_s, a_gsum, a_tc, tc_fp8);
  return cudaLaunchKernelEx(&cfg, quant_act_kernel, x, K, a_q, a_s, a_gsum, a_tc, tc_fp8);
}

cudaError_t launch_pack_w4(const uint8_t* w_q, const uint16_t* s, const uint8_t* z, int64_t N,
                           int64_t K, void* packed, cudaStream_t st) {
  const int64_t G = K / 128;
  uint8_t* base = static_cast<uint8_t*>(packed);
  pack_codes_kernel<<<grid_for(N * K / 8, 256), 256, 0, st>>>(w_q, N, K, base);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pack_meta_kernel<<<grid_for(G * N, 256), 256, 0, st>>>(s, z, N, G, base);
  return cudaGetLastError();
}

cudaError_t launch_unpack_w4(const void* packed, int64_t N, int64_t K, uint8_t* w_q, uint16_t* s,
                             uint8_t* z, cudaStream_t st) {
  const int64_t G = K / 128;
  const uint8_t* base = static_cast<const uint8_t*>(packed);
  unpack_codes_kernel<<<grid_for(N * K / 8, 256), 256, 0, st>>>(base, N, K, w_q);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  unpack_meta_kernel<<<grid_for(G * N, 256), 256, 0, st>>>(base, N, G, s, z);
  return cudaGetLastError();
}

cudaError_t launch_pack_w4_gptq(const int32_t* qweight, const int32_t* qzeros,
                               const uint16_t* scales, int64_t N, int64_t K, int zero_offset,
                               void* packed, cudaStream_t st) {
  const int64_t G = K / 128;
  uint8_t* out = static_cast<uint8_t*>(packed);
  pack_gptq_codes_kernel<<<grid_for(N * K / 8, 256), 256, 0, st>>>(qweight, N, K, out);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  pack_gptq_meta_kernel<<<grid_for(G * N, 256), 256, 0, st>>>(qzeros, scales, N, G, zero_offset,
                                                               out);
  return cudaGetLastError();
}

cudaError_t launch_dequant_w4(const void* packed, int64_t N, int64_t K, uint16_t* w,
                              cudaStream_t st) {
  const int64_t G = K / 128;
  const int64_t recs = (N / 128) * G;
  if (recs <= 0) return cudaSuccess;
  if (recs > 0x7FFFFFFF) return cudaErrorInvalidValue;
  dequant_w4_kernel<<<(unsigned)recs, kDequantThreads, 0, st>>>(
      static_cast<const uint8_t*>(packed), G, K, w);
  return cudaGetLastError();
}

cudaError_t take_error_word_quant_pack(unsigned* out) { return take_local_error_word(out); }

}  // namespace egopq
