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
//  - the first call in each CUDA context looks up the array's device address
//    (cudaGetSymbolAddress, with that context's device current); make that
//    first call before any stream capture. The address is kept per device and
//    tagged with the context it was read in, so a call after a device reset
//    (a new primary context, where the array may have moved) looks it up
//    again.
#include <mutex>

#include "../../include/egopq.h"
#include "egopq_internal.h"

namespace egopq {
int run_linear(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N, int64_t K,
               uint16_t* y_bf16, uint8_t* ws, int use, cudaStream_t st);
int set_last_error(int code, const char* msg);
}  // namespace egopq

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;

// Staging buffer of egopq_w4a8_linear_noalloc. Host code must not use this
// name as an address (it denotes a host-side stand-in); the device address
// comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) uint8_t g_linear_scratch[kStaticScratchBytes];

// Identity of the calling thread's current context (cuCtxGetId through the
// runtime's driver entry points); 0 when there is none or it cannot be read.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

struct ScratchAddr {
  void* ptr = nullptr;
  unsigned long long ctx = 0;  // context the address was read in (0: unknown)
};
std::mutex g_addr_mu;
ScratchAddr g_addr[egopq::kMaxDevices];

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

}  // namespace

extern "C" int egopq_w4a8_linear_noalloc(const uint16_t* x_bf16, const void* packed, int64_t M,
                                         int64_t N, int64_t K, int group, uint16_t* y_bf16,
                                         int path, egopq_stream_t stream) {
  using egopq::set_last_error;
  if (path != EGOPQ_PATH_AUTO && path != EGOPQ_PATH_GEMV && path != EGOPQ_PATH_TC)
    return set_last_error(EGOPQ_ERR_INVALID_ARG, "egopq_w4a8_linear_noalloc: unknown path");
  // the same shape gate as egopq_w4a8_linear, before any size arithmetic
  if (const int rc = egopq::check_w4_shape(M, N, K, group)) return rc;
  if (M == 0) return EGOPQ_OK;
  if (!x_bf16 || !packed || !y_bf16)
    return set_last_error(EGOPQ_ERR_INVALID_ARG, "egopq_w4a8_linear_noalloc: NULL pointer");
  if (misaligned(x_bf16) || misaligned(packed) || misaligned(y_bf16))
    return set_last_error(EGOPQ_ERR_MISALIGNED,
                          "egopq_w4a8_linear_noalloc: a pointer is not 16-byte aligned");
  const size_t need = egopq_w4a8_linear_workspace_bytes(M, K, group, path);
  if (need > kStaticScratchBytes)
    return set_last_error(EGOPQ_ERR_UNSUPPORTED_SHAPE,
                          "egopq_w4a8_linear_noalloc: the staged activations (about 2*M*K bytes "
                          "on the tensor-core path, M*K on the GEMV path) exceed its 16 MiB "
                          "static scratch; use egopq_w4a8_linear with a workspace");
  if (const int rc = egopq::check_arch()) return rc;
  const int dev = egopq::current_device();
  if (dev < 0)
    return set_last_error(EGOPQ_ERR_CUDA, "egopq_w4a8_linear_noalloc: cudaGetDevice failed");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_addr_mu);
    ScratchAddr& a = g_addr[dev];
    const unsigned long long ctx = current_context_id();
    if (!a.ptr || ctx == 0 || ctx != a.ctx) {
      // set-up, once per device and context, with that device current
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_linear_scratch);
      if (e != cudaSuccess || !ptr)
        return set_last_error(EGOPQ_ERR_CUDA,
                              "egopq_w4a8_linear_noalloc: cudaGetSymbolAddress failed");
      a.ptr = ptr;
      a.ctx = current_context_id();  // the lookup made the context current if it was not
    }
    scratch = a.ptr;
  }
  // the quantization kernel overwrites every staged byte the GEMM then reads,
  // so nothing in the shared array needs clearing between calls
  return egopq::run_linear(x_bf16, packed, M, N, K, y_bf16, static_cast<uint8_t*>(scratch),
                           egopq::auto_path(M, egopq::kW4A8, path), (cudaStream_t)stream);
}
