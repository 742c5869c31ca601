// egopq_internal.h -- launchers shared between the kernel files and the C ABI.
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/egopq.h"
#include "egopq_common.cuh"

namespace egopq {

// kW16A16: dense bf16 weights through the W4A16 tensor-core pipeline (the
// same roles, buffers and per-group drains; the converters copy instead of
// unpacking) -- a yardstick, not a quantized path.
enum Variant { kW4A8 = 0, kW4A16 = 1, kW8A16 = 2, kW8A8 = 3, kW16A16 = 4 };

// Launch state that depends on the device (shared-memory opt-ins, SM counts)
// is kept per device ordinal, up to this many devices.
constexpr int kMaxDevices = 64;

// Host-side checks shared by the entry points; each records its message as the
// calling thread's last error and returns a negative egopq_status on failure.
// Shape gate of the packed int4 weight (and the size limit of every call).
int check_w4_shape(int64_t M, int64_t N, int64_t K, int group);
// The current device is an sm_103 (cached per device).
int check_arch();

// Ordinal of the calling thread's current device, or -1 if cudaGetDevice
// fails or the ordinal is kMaxDevices or more.
int current_device();
// SM count of the current device (cached per device; 0 if it cannot be read).
int device_sm_count();

// A kernel's dynamic shared-memory opt-in, kept per device: cudaFuncSetAttribute
// applies to the current device only, so each device gets its own call. ensure()
// raises the opt-in to at least `bytes` (never lowers it); thread-safe.
class SmemOptIn {
 public:
  template <typename Kernel>
  cudaError_t ensure(Kernel kern, size_t bytes) {
    const int dev = current_device();
    if (dev < 0) return cudaErrorInvalidDevice;
    if (done_[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    std::lock_guard<std::mutex> lock(mu_);
    if (done_[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    done_[dev].store(bytes, std::memory_order_release);
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  std::atomic<size_t> done_[kMaxDevices] = {};
};

// Sibling linears that read the same activations, run as one launch: the
// output tiles (128 weight rows each) of linear j are the global tiles
// [tile0[j], tile0[j + 1]); a single linear is the table with count 1.
constexpr int kMaxSegs = 8;
struct SegTable {
  int count;
  int tile0[kMaxSegs + 1];
  const uint8_t* packed[kMaxSegs];  // packed int4 weight of linear j
  uint16_t* y[kMaxSegs];            // its bf16 output [M][N[j]]
  int64_t N[kMaxSegs];
};

// Global tile `nt` resolved to its linear: the packed record (tile, group 0)
// (records of one tile are consecutive, 8512 bytes apart), the output, its row
// count and the tile's first output row. Compile-time indexes only, so the
// table stays in the parameter space.
struct TileRef {
  const uint8_t* rec0;
  uint16_t* y;
  int64_t N;
  int64_t n0;
  int seg;  // which linear
};
__device__ __forceinline__ TileRef tile_ref(const SegTable& s, int nt, int G) {
  const uint8_t* pk = s.packed[0];
  uint16_t* y = s.y[0];
  int64_t N = s.N[0];
  int t0 = 0, seg = 0;
#pragma unroll
  for (int j = 1; j < kMaxSegs; ++j) {
    if (j < s.count && nt >= s.tile0[j]) {
      pk = s.packed[j];
      y = s.y[j];
      N = s.N[j];
      t0 = s.tile0[j];
      seg = j;
    }
  }
  const int64_t lt = nt - t0;
  return TileRef{pk + lt * G * 8512, y, N, lt * 128, seg};
}

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
  // dense bf16 weight [N][K] (W16A16)
  const uint16_t* w16;
  // outputs
  uint16_t* y;
  int32_t* partials;  // non-null: write group partials instead of y (W4A8 only)
  uint64_t timeout_ns;
  // packed int4 variants: sibling linears sharing the activations (null: one
  // linear, packed / y / N above)
  const SegTable* segs;
};

// The segment table of a call: `a.segs`, or the one linear of packed / y / N.
inline SegTable seg_table(const GemmArgs& a) {
  if (a.segs) return *a.segs;
  SegTable t{};
  t.count = 1;
  t.tile0[0] = 0;
  t.tile0[1] = (int)(a.N / 128);
  t.packed[0] = a.packed;
  t.y[0] = a.y;
  t.N[0] = a.N;
  return t;
}

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
// Debug builds: the packed-record read limit of each unit that reads records
// (cudaErrorNotSupported in release builds).
cudaError_t set_record_limit_gemv(unsigned long long bytes);
cudaError_t set_record_limit_tc_gemm(unsigned long long bytes);

// Byte size of the packed records of one linear with N rows and G groups.
__host__ __device__ inline uint64_t packed_record_bytes(int64_t N, int G) {
  return (uint64_t)(N / 128) * (uint64_t)G * 8512u;
}

// CUDA-core GEMV (small M). Returns cudaErrorNotSupported for shapes it does
// not take.
cudaError_t launch_gemv(const GemmArgs& a, cudaStream_t st);
// tcgen05 tensor-core GEMM (any M).
cudaError_t launch_tc_gemm(const GemmArgs& a, cudaStream_t st);
// Token tile (MMA N) the tensor-core GEMM runs an M x N x K call of `variant`
// with: 16, 32 or 64 up to 64 tokens; above, 128 or 192 (per-group variants,
// chosen from the grid each makes) or 128.
int tc_token_tile(int variant, int64_t M, int64_t N, int64_t K);
// Kernel launches of the tensor-core GEMM of that shape: 1, or 2 when the
// persistent grid's short last round runs as a split-K second launch.
int tc_launches(int variant, int64_t M, int64_t N, int64_t K);
// Bounded-wait self test.
cudaError_t launch_selftest_timeout(uint64_t timeout_ns, cudaStream_t st);

// Tensor-core W4A8 operand form: up to this many tokens the activation codes
// are staged as two e4m3 planes (a_q >> 4, a_q & 15) and the MMAs run
// kind::f8f6f4 at K = 32 (token tiles of at most 64); above it as fp16 codes
// for kind::f16 MMAs (128-token tiles).
constexpr int kTcFp8MaxM = 64;
// Largest M per W4A8 GEMV launch (larger M run as several launches).
constexpr int kGemvMaxRows = 16;
// AUTO path: W4A8, W4A16 and W8A16 batches up to this many tokens take the GEMV.
constexpr int kGemvAutoMaxM = 4;

// The kernel path a call takes: `path` itself unless it is EGOPQ_PATH_AUTO,
// which resolves by token count -- W4A8, W4A16 and W8A16 on the CUDA-core
// GEMVs up to kGemvAutoMaxM tokens, W8A8 on its GEMV up to kTcFp8MaxM (its
// tensor-core form exists only above), everything else on the tensor cores.
inline int auto_path(int64_t M, int variant, int path) {
  if (path != EGOPQ_PATH_AUTO) return path;
  if (variant == kW8A8) return M <= kTcFp8MaxM ? EGOPQ_PATH_GEMV : EGOPQ_PATH_TC;
  if (variant == kW16A16) return EGOPQ_PATH_TC;  // (no GEMV form)
  // W4A8, W4A16, W8A16: the GEMV up to kGemvAutoMaxM tokens (measured on
  // GB300: W4A16 3072 x 3072 at one token 5.5 us on the GEMV, 12.3 us on
  // 16-token tensor-core tiles; from 8 tokens the tiles win on every shape)
  return M <= kGemvAutoMaxM ? EGOPQ_PATH_GEMV : EGOPQ_PATH_TC;
}

}  // namespace egopq
