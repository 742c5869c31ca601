// egopq_internal.h -- launchers shared between the kernel files and the C ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "egopq_common.cuh"

namespace egopq {

enum Variant { kW4A8 = 0, kW4A16 = 1, kW8A16 = 2, kW8A8 = 3 };

// Operands of one GEMM call, already validated by the ABI layer.
struct GemmArgs {
  int variant;
  int64_t M, N, K;
  // activation codes (W4A8, W8A8; a_gsum W4A8 only)
  const int8_t* a_q;
  const void* a_tc;  // tensor-core operand form of a_q (see kTcFp8MaxM)
  const float* a_s;
  const int32_t* a_gsum;
  // W4A16 / W8A16
  const uint16_t* x;
  // packed int4 weight (W4A8, W4A16)
  const uint8_t* packed;
  // int8 weight and per-channel scale (W8A16, W8A8)
  const int8_t* w8;
  const uint16_t* s8;
  // outputs
  uint16_t* y;
  int32_t* partials;  // non-null: write group partials instead of y (W4A8 only)
  uint64_t timeout_ns;
};

cudaError_t launch_quant_act(const uint16_t* x, int64_t M, int64_t K, int8_t* a_q, float* a_s,
                             int32_t* a_gsum, void* a_tc, cudaStream_t st);
cudaError_t launch_pack_w4(const uint8_t* w_q, const uint16_t* s, const uint8_t* z, int64_t N,
                           int64_t K, void* packed, cudaStream_t st);
cudaError_t launch_unpack_w4(const void* packed, int64_t N, int64_t K, uint8_t* w_q, uint16_t* s,
                             uint8_t* z, cudaStream_t st);
cudaError_t launch_pack_w4_gptq(const int32_t* qweight, const int32_t* qzeros,
                               const uint16_t* scales, int64_t N, int64_t K, int zero_offset,
                               void* packed, cudaStream_t st);
cudaError_t launch_dequant_w4(const void* packed, int64_t N, int64_t K, uint16_t* w,
                              cudaStream_t st);

// Each kernel unit's device error word, read and cleared (see egopq_common.cuh).
cudaError_t take_error_word_quant_pack(unsigned* out);
cudaError_t take_error_word_gemv(unsigned* out);
cudaError_t take_error_word_tc_gemm(unsigned* out);

// CUDA-core GEMV (small M). Returns cudaErrorNotSupported for shapes it does
// not take.
cudaError_t launch_gemv(const GemmArgs& a, cudaStream_t st);
// tcgen05 tensor-core GEMM (any M).
cudaError_t launch_tc_gemm(const GemmArgs& a, cudaStream_t st);
// Bounded-wait self test.
cudaError_t launch_selftest_timeout(uint64_t timeout_ns, cudaStream_t st);

// Tensor-core W4A8 operand form: up to this many tokens the activation codes
// are staged as two e4m3 planes (a_q >> 4, a_q & 15) and the MMAs run
// kind::f8f6f4 at K = 32 (token tiles of at most 64); above it as fp16 codes
// for kind::f16 MMAs (128-token tiles).
constexpr int kTcFp8MaxM = 64;
// Largest M per W4A8 GEMV launch (larger M run as several launches).
constexpr int kGemvMaxRows = 16;
// AUTO path: W4A8 batches up to this many tokens take the GEMV.
constexpr int kGemvAutoMaxM = 4;

}  // namespace egopq
