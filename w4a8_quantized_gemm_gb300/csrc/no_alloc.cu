// no_alloc.cu -- the one-call W4A8 linear for callers that cannot allocate
// device memory.
//
// egopq_w4a8_linear stages the quantized activations in a workspace the caller
// allocates. Some callers have no allocator to call: a plugin or custom
// operator running inside a host framework that owns every device buffer and
// hands kernels only their inputs and outputs, or a latency-critical serving
// loop that must never enter cudaMalloc (which can synchronize the device and
// take milliseconds). This entry point serves them: its staging buffer is a
// file-scope device array that exists for as long as the library is loaded,
// so the call allocates nothing.
//
// Costs and limits, stated for the caller:
//  - every GPU that loads the library holds kStaticScratchBytes (16 MiB) of
//    device memory for this array until the process exits;
//  - a call whose staged activations exceed that size is refused;
//  - all calls share the one array: calls that overlap on the GPU (different
//    streams, or different host threads without ordering) race on it;
//  - the first call on each device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current); make that first call
//    before any stream capture.
#include <mutex>

#include "../../include/egopq.h"
#include "egopq_internal.h"

namespace egopq {
int run_linear(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N, int64_t K,
               uint16_t* y_bf16, uint8_t* ws, int use, cudaStream_t st);
int set_last_error(int code, const char* msg);
}

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

// Staging buffer of egopq_w4a8_linear_noalloc. Host code must not use this
// name as an address (it denotes a host-side stand-in); the device address
// comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) uint8_t g_linear_scratch[kStaticScratchBytes];

std::mutex g_addr_mu;
void* g_addr[kMaxDevices] = {};

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace

extern "C" int egopq_w4a8_linear_noalloc(const uint16_t* x_bf16, const void* packed, int64_t M,
                                         int64_t N, int64_t K, int group, uint16_t* y_bf16,
                                         int path, egopq_stream_t stream) {
  using egopq::set_last_error;
  if (path != EGOPQ_PATH_AUTO && path != EGOPQ_PATH_GEMV && path != EGOPQ_PATH_TC)
    return set_last_error(EGOPQ_ERR_INVALID_ARG, "egopq_w4a8_linear_noalloc: unknown path");
  if (M < 0 || N <= 0 || K <= 0)
    return set_last_error(EGOPQ_ERR_INVALID_ARG, "egopq_w4a8_linear_noalloc: bad sizes");
  if (group != 128 || K % 128 || N % 128)
    return set_last_error(EGOPQ_ERR_UNSUPPORTED_SHAPE,
                          "egopq_w4a8_linear_noalloc: group must be 128 and K, N multiples of 128");
  if (M == 0) return EGOPQ_OK;
  if (!x_bf16 || !packed || !y_bf16)
    return set_last_error(EGOPQ_ERR_INVALID_ARG, "egopq_w4a8_linear_noalloc: NULL pointer");
  if (misaligned(x_bf16) || misaligned(packed) || misaligned(y_bf16))
    return set_last_error(EGOPQ_ERR_MISALIGNED,
                          "egopq_w4a8_linear_noalloc: a pointer is not 16-byte aligned");
  const size_t need = egopq_w4a8_linear_workspace_bytes(M, K, group, path);
  if (need == 0 || need > kStaticScratchBytes)
    return set_last_error(EGOPQ_ERR_UNSUPPORTED_SHAPE,
                          "egopq_w4a8_linear_noalloc: the staged activations (about 3*M*K bytes "
                          "on the tensor-core path, M*K on the GEMV path) exceed its 16 MiB "
                          "static scratch; use egopq_w4a8_linear with a workspace");
  if (!egopq_supported(M, N, K, group, EGOPQ_VARIANT_W4A8))
    return set_last_error(EGOPQ_ERR_ARCH, "egopq_w4a8_linear_noalloc: device is not sm_103");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return set_last_error(EGOPQ_ERR_CUDA, "egopq_w4a8_linear_noalloc: cudaGetDevice failed");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_addr_mu);
    if (!g_addr[dev]) {
      // set-up, once per device, with that device current
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_linear_scratch);
      if (e != cudaSuccess || !ptr)
        return set_last_error(EGOPQ_ERR_CUDA,
                              "egopq_w4a8_linear_noalloc: cudaGetSymbolAddress failed");
      g_addr[dev] = ptr;
    }
    scratch = g_addr[dev];
  }
  // the quantization kernel overwrites every staged byte the GEMM then reads,
  // so nothing in the shared array needs clearing between calls
  const int use = (path == EGOPQ_PATH_AUTO) ? (M <= egopq::kGemvAutoMaxM ? EGOPQ_PATH_GEMV : EGOPQ_PATH_TC)
                                            : path;
  return egopq::run_linear(x_bf16, packed, M, N, K, y_bf16, static_cast<uint8_t*>(scratch), use,
                           (cudaStream_t)stream);
}
