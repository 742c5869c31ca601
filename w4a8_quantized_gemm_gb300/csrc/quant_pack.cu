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
// part a & 15, a = 16 * high + low) with each 8-run in the packed weights'
// nibble order (even offsets, then odd); otherwise fp16 [M][K] (the codes
// qf as fp32 integers, exact in fp16).
__device__ __forceinline__ void store_tc_operand(void* a_tc, bool fp8, int64_t M, int64_t K,
                                                 int64_t m, int64_t vec, const int (&q)[8],
                                                 const float (&qf)[8]) {
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
      const __half2 hv = __floats2half2_rn(qf[2 * i], qf[2 * i + 1]);
      h[i] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    reinterpret_cast<uint4*>(static_cast<uint16_t*>(a_tc) + m * K)[vec] =
        make_uint4(h[0], h[1], h[2], h[3]);
  }
}

// Reciprocal of the row scale s for quant_code's product form, or NaN where
// that form is not used (s zero, below 2^-100, above 2^126 or not finite): a
// NaN product sends every element of the row to the IEEE quotient.
__device__ __forceinline__ float quant_recip(float s) {
  return (s >= 0x1p-100f && s <= 0x1p+126f) ? __frcp_rn(s) : __int_as_float(0x7fc00000);
}

// clamp(round_half_even(fp32 quotient x / s), -127, 127) as an fp32 integer,
// equal to __float2int_rn(__fdiv_rn(x, s)) clamped. With inv the correctly
// rounded 1/s, r = fl(x * inv) is within |x / s| * 2^-23 of the exact quotient
// q (two roundings of at most 2^-24 relative), and fl(q) within |q| * 2^-24 of
// q; as |q| <= 127 * (1 + 2^-23), r and fl(q) lie within 2.3e-5 of each other.
// So they round to the same integer unless r lies within that distance of a
// half-integer; where r lies within 1e-4 of one (|r - rint(r)| >= 0.4999, or r
// NaN) the IEEE quotient decides. On the product's side |r| < 127.5, so its
// integer needs no clamp.
__device__ __forceinline__ float quant_code(float x, float s, float inv) {
  const float r = x * inv;
  const float rf = rintf(r);
  if (fabsf(r - rf) < 0.4999f) return rf;
  return (float)max(-127, min(127, __float2int_rn(__fdiv_rn(x, s))));
}

// Quantizes the 8 bf16 values of one 16-byte vector v (K = 8*idx .. 8*idx+7
// of token m, scale s, inv = quant_recip(s)) and writes their codes: to a_q
// when given, to the tensor-core operand form when a_tc is given, and, summed
// over the 16 vectors of a 128-wide group that one half-warp holds, to a_gsum.
// All 16 lanes of the calling half-warp take part.
__device__ __forceinline__ void quant_store_vec(const uint4& v, float s, float inv, bool zero_row,
                                                int8_t* a_q, int32_t* a_gsum, void* a_tc,
                                                bool tc_fp8, int64_t M, int64_t K, int64_t m,
                                                int64_t idx) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float qf[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    qf[2 * j] = zero_row ? 0.f : quant_code(__uint_as_float(w[j] << 16), s, inv);
    qf[2 * j + 1] = zero_row ? 0.f : quant_code(__uint_as_float(w[j] & 0xFFFF0000u), s, inv);
  }
  int q[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) q[j] = (int)qf[j];  // exact: integers in [-127, 127]
  if (a_q) {
    uint2 packed;
    packed.x = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
               ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
    packed.y = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) |
               ((uint32_t)(q[6] & 0xFF) << 16) | ((uint32_t)(q[7] & 0xFF) << 24);
    reinterpret_cast<uint2*>(a_q + m * K)[idx] = packed;
  }
  if (a_tc) store_tc_operand(a_tc, tc_fp8, M, K, m, idx, q, qf);
  // the group sum in fp32: |sum| <= 128 * 127, exact
  float sum = ((qf[0] + qf[1]) + (qf[2] + qf[3])) + ((qf[4] + qf[5]) + (qf[6] + qf[7]));
  const unsigned half_mask = 0xFFFFu << (threadIdx.x & 16);
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(half_mask, sum, o);
  if ((threadIdx.x & 15) == 0) a_gsum[m * (K / 128) + idx / 16] = (int32_t)sum;
}

// max |x| over the 8 bf16 values of v folded into acc, a bf16 pair of running
// maxima (max is exact in bf16; a NaN operand gives the other, as fmaxf)
__device__ __forceinline__ __nv_bfloat162 vec_absmax(const uint4& v, __nv_bfloat162 acc) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t a = w[j] & 0x7FFF7FFFu;  // |x| of both halves
    acc = __hmax2(acc, *reinterpret_cast<const __nv_bfloat162*>(&a));
  }
  return acc;
}

__device__ __forceinline__ float absmax_f32(__nv_bfloat162 acc) {
  return fmaxf(__low2float(acc), __high2float(acc));
}

// Maximum of v over the block's threads (T of them); every thread gets it.
template <int T>
__device__ __forceinline__ float block_max(float v, float* warp_max) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = v;
  __syncthreads();
  v = warp_max[0];
#pragma unroll
  for (int i = 1; i < T / 32; ++i) v = fmaxf(v, warp_max[i]);
  return v;
}

// Rows of any length: one CTA per token row, two passes over x (the row's
// absmax, then the codes; the second pass reads the row from L2).
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
  __nv_bfloat162 acc = __float2bfloat162_rn(0.f);
  for (int64_t v = threadIdx.x; v < nvec; v += kQuantThreads) acc = vec_absmax(__ldg(xr + v), acc);
  const float amax = block_max<kQuantThreads>(absmax_f32(acc), warp_max);
  const float s = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) a_s[m] = s;
  const float inv = quant_recip(s);
  // 16 consecutive vectors make one 128-wide group; kQuantThreads % 16 == 0
  // and nvec % 16 == 0, so the 16 lanes of a half-warp are all inside the
  // loop or all outside it
  for (int64_t v = threadIdx.x; v < nvec; v += kQuantThreads)
    quant_store_vec(__ldg(xr + v), s, inv, amax == 0.f, a_q, a_gsum, a_tc, tc_fp8, gridDim.x, K,
                    m, v);
}

// Few tokens, rows up to kRowThreads * kRowVec * 8 values: one 512-thread CTA
// a row holding the whole row in registers (up to kRowVec 16-byte vectors a
// thread, every load issued before the first is used), so x is read once and
// the row's latency is short. It waits for the preceding kernel only when the
// launch carried a programmatic dependency.
constexpr int kRowThreads = 512;
constexpr int kRowVec = 8;

__global__ void __launch_bounds__(kRowThreads, 1)
quant_act_row_kernel(const uint16_t* __restrict__ x, int64_t K, int8_t* __restrict__ a_q,
                     float* __restrict__ a_s, int32_t* __restrict__ a_gsum,
                     void* __restrict__ a_tc, bool tc_fp8) {
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int64_t m = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + m * K);
  const int nvec = (int)(K / 8);
  __shared__ float warp_max[kRowThreads / 32];
  uint4 v[kRowVec];
#pragma unroll
  for (int i = 0; i < kRowVec; ++i) {
    const int idx = threadIdx.x + i * kRowThreads;
    v[i] = idx < nvec ? __ldg(xr + idx) : make_uint4(0, 0, 0, 0);
  }
  __nv_bfloat162 acc = __float2bfloat162_rn(0.f);
#pragma unroll
  for (int i = 0; i < kRowVec; ++i) acc = vec_absmax(v[i], acc);
  const float amax = block_max<kRowThreads>(absmax_f32(acc), warp_max);
  const float s = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) a_s[m] = s;
  const float inv = quant_recip(s);
#pragma unroll
  for (int i = 0; i < kRowVec; ++i) {
    const int idx = threadIdx.x + i * kRowThreads;
    if (idx >= nvec) break;  // whole half-warps leave together (nvec % 16 == 0)
    quant_store_vec(v[i], s, inv, amax == 0.f, a_q, a_gsum, a_tc, tc_fp8, gridDim.x, K, m, idx);
  }
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Many tokens, rows up to kStreamMaxK values: persistent CTAs walk the rows
// m = blockIdx.x, blockIdx.x + gridDim.x, ...; each row is staged whole in
// shared memory by asynchronous copies while the previous one is quantized
// (two buffers), so x streams from HBM once with a row always in flight, and
// the row's absmax and codes are read from shared memory. T = 256 threads,
// 512 for rows longer than 8192 (fewer CTAs fit beside their buffers).
constexpr int64_t kStreamMaxK = 32768;

template <int T>
__global__ void __launch_bounds__(T)
quant_act_stream_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                        int8_t* __restrict__ a_q, float* __restrict__ a_s,
                        int32_t* __restrict__ a_gsum, void* __restrict__ a_tc, bool tc_fp8) {
  extern __shared__ __align__(16) uint4 rows[];  // [2][K / 8]
  __shared__ float warp_max[T / 32];
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch_dependents();
  const int nvec = (int)(K / 8);
  auto stage = [&](int64_t m, int buf) {
    const uint4* src = reinterpret_cast<const uint4*>(x + m * K);
    uint4* dst = rows + buf * nvec;
    for (int i = threadIdx.x; i < nvec; i += T) cp_async16(dst + i, src + i);
    cp_async_commit();
  };
  int64_t m = blockIdx.x;
  if (m < M) stage(m, 0);
  for (int j = 0; m < M; ++j, m += gridDim.x) {
    if (m + gridDim.x < M) {
      stage(m + gridDim.x, (j + 1) & 1);
      cp_async_wait<1>();  // this thread's copies of row m have landed
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();  // ... and every thread's
    const uint4* row = rows + (j & 1) * nvec;
    __nv_bfloat162 acc = __float2bfloat162_rn(0.f);
    for (int i = threadIdx.x; i < nvec; i += T) acc = vec_absmax(row[i], acc);
    const float amax = block_max<T>(absmax_f32(acc), warp_max);
    const float s = __fdiv_rn(amax, 127.0f);
    if (threadIdx.x == 0) a_s[m] = s;
    const float inv = quant_recip(s);
    // nvec % 16 == 0 and T % 16 == 0: whole half-warps iterate
    for (int i = threadIdx.x; i < nvec; i += T)
      quant_store_vec(row[i], s, inv, amax == 0.f, a_q, a_gsum, a_tc, tc_fp8, M, K, m, i);
    __syncthreads();  // row buffer and warp_max are reused by the next row
  }
}

// Long rows for few tokens: one token's row is split over a cluster of CTAs
// (whole 128-wide groups each, at most kSplitVec 16-byte vectors per thread),
// so that the per-element work spreads over several SMs; the CTAs combine
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
#pragma unroll
  for (int i = 0; i < kSplitVec; ++i) {
    const int idx = v0 + threadIdx.x + i * kSplitThreads;
    v[i] = idx < v1 ? __ldg(xr + idx) : make_uint4(0, 0, 0, 0);
  }
  __nv_bfloat162 acc = __float2bfloat162_rn(0.f);
#pragma unroll
  for (int i = 0; i < kSplitVec; ++i) acc = vec_absmax(v[i], acc);
  if (const float part = block_max<kSplitThreads>(absmax_f32(acc), warp_max); threadIdx.x == 0)
    cta_max = part;
  cluster_sync_all();  // every CTA's partial maximum is in its shared memory
  float amax = 0.f;
  for (int r = 0; r < C; ++r) amax = fmaxf(amax, ld_dsmem_f32(map_to_rank(smem_u32(&cta_max), r)));
  cluster_sync_all();  // no CTA leaves while another still reads its partial
  const float s = __fdiv_rn(amax, 127.0f);
  if (rank == 0 && threadIdx.x == 0) a_s[m] = s;
  const float inv = quant_recip(s);
#pragma unroll
  for (int i = 0; i < kSplitVec; ++i) {
    const int idx = v0 + threadIdx.x + i * kSplitThreads;
    if (idx >= v1) break;  // whole half-warps leave together (v0, v1 multiples of 16)
    quant_store_vec(v[i], s, inv, amax == 0.f, a_q, a_gsum, a_tc, tc_fp8, M, K, m, idx);
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
  const int64_t nvec = K / 8;
  const bool tc_fp8 = M <= kTcFp8MaxM;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)M, 1, 1);
  cfg.blockDim = dim3(kQuantThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (M > 64) {
    // many tokens: persistent CTAs streaming rows through shared memory, as
    // many as are resident at once with two row buffers each
    if (K <= kStreamMaxK) {
      const bool wide = K > 8192;
      auto kern = wide ? quant_act_stream_kernel<512> : quant_act_stream_kernel<256>;
      const int threads = wide ? 512 : 256;
      const size_t smem = (size_t)(2 * K * 2);
      static SmemOptIn opt_in[2];
      if (cudaError_t e = opt_in[wide].ensure(kern, smem); e != cudaSuccess) return e;
      int per_sm = 0;
      if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
          e != cudaSuccess)
        return e;
      const int sms = device_sm_count();
      if (per_sm < 1 || sms < 1) return cudaErrorInvalidConfiguration;
      const int64_t ctas = (int64_t)sms * per_sm;
      cfg.gridDim = dim3((unsigned)(M < ctas ? M : ctas), 1, 1);
      cfg.blockDim = dim3(threads, 1, 1);
      cfg.dynamicSmemBytes = smem;
      return cudaLaunchKernelEx(&cfg, kern, x, M, K, a_q, a_s, a_gsum, a_tc, tc_fp8);
    }
    return cudaLaunchKernelEx(&cfg, quant_act_kernel, x, K, a_q, a_s, a_gsum, a_tc, tc_fp8);
  }
  // few tokens: rows longer than 1024 vectors split over a cluster of up to 8
  // CTAs, each holding whole groups and at most kSplitMaxVec vectors
  if (nvec > 1024) {
    const int64_t G = K / 128;
    int split = (int)((nvec + kSplitMaxVec - 1) / kSplitMaxVec);
    if (split < 2) split = 2;
    // each CTA's share, ceil(G / split) groups, must fit its registers
    if (split <= 8 && (G + split - 1) / split * 16 <= kSplitMaxVec) {
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = (unsigned)split;
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      cfg.numAttrs = 2;
      cfg.gridDim = dim3((unsigned)(M * split), 1, 1);
      cfg.blockDim = dim3(kSplitThreads, 1, 1);
      return cudaLaunchKernelEx(&cfg, quant_act_split_kernel, x, M, K, a_q, a_s, a_gsum, a_tc,
                                tc_fp8);
    }
  }
  if (nvec <= (int64_t)kRowThreads * kRowVec) {
    cfg.blockDim = dim3(kRowThreads, 1, 1);
    return cudaLaunchKernelEx(&cfg, quant_act_row_kernel, x, K, a_q, a_s, a_gsum, a_tc, tc_fp8);
  }
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
