// egopq_api.cu -- the C ABI declared in include/egopq.h: argument validation,
// path dispatch, the device error words and error strings. No allocation
// happens here; every buffer belongs to the caller.
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "../../include/egopq.h"
#include "egopq_internal.h"

namespace egopq {

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

int device_sm_count() {
  static std::atomic<int> cached[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return 0;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace egopq

using namespace egopq;

namespace {

thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(EGOPQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per bounded wait
constexpr int64_t kMaxDim = (int64_t)1 << 31;

}  // namespace

namespace egopq {

// sm_103 check, cached per device
int check_arch() {
  static std::atomic<int> cached[kMaxDevices] = {};  // 0 unknown, 1 ok, 2 bad
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(EGOPQ_ERR_CUDA, "device ordinal %d is beyond the %d this library tracks", dev,
                kMaxDevices);
  const int c = cached[dev].load(std::memory_order_relaxed);
  if (c) {
    if (c == 1) return EGOPQ_OK;
    return fail(EGOPQ_ERR_ARCH, "device %d is not sm_103; this library is built for sm_103a", dev);
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  const bool ok = (major == 10 && minor == 3);
  cached[dev].store(ok ? 1 : 2, std::memory_order_relaxed);
  if (!ok) return fail(EGOPQ_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a", dev,
                       major, minor);
  return EGOPQ_OK;
}

int check_w4_shape(int64_t M, int64_t N, int64_t K, int group) {
  if (M < 0 || N <= 0 || K <= 0)
    return fail(EGOPQ_ERR_INVALID_ARG, "bad sizes M=%lld N=%lld K=%lld", (long long)M,
                (long long)N, (long long)K);
  if (M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
    return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "sizes M=%lld N=%lld K=%lld exceed 2^31 - 1",
                (long long)M, (long long)N, (long long)K);
  if (group != 128) return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "group must be 128 (got %d)", group);
  if (K % 128 || N % 128)
    return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE,
                "K (%lld) and N (%lld) must be multiples of 128", (long long)K, (long long)N);
  return EGOPQ_OK;
}

}  // namespace egopq

namespace {

int check_ptrs(int n, ...) {
  va_list ap;
  va_start(ap, n);
  for (int i = 0; i < n; ++i) {
    const char* name = va_arg(ap, const char*);
    const void* p = va_arg(ap, const void*);
    if (!p) {
      va_end(ap);
      return fail(EGOPQ_ERR_INVALID_ARG, "%s is NULL", name);
    }
    if (!aligned16(p)) {
      va_end(ap);
      return fail(EGOPQ_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    }
  }
  va_end(ap);
  return EGOPQ_OK;
}

int run_gemm(const GemmArgs& a, int path, cudaStream_t st) {
  if (path != EGOPQ_PATH_AUTO && path != EGOPQ_PATH_GEMV && path != EGOPQ_PATH_TC)
    return fail(EGOPQ_ERR_INVALID_ARG, "unknown path %d", path);
  int rc = check_arch();
  if (rc) return rc;
  if (a.M == 0) return EGOPQ_OK;
  const int use = auto_path(a.M, a.variant, path);
  if (use == EGOPQ_PATH_TC && (a.variant == kW4A8 || a.variant == kW8A8) && !a.a_tc)
    return fail(EGOPQ_ERR_INVALID_ARG, "a_tc is required by the tensor-core path");
  if (use == EGOPQ_PATH_GEMV && (a.variant == kW4A8 || a.variant == kW8A8) && !a.a_q)
    return fail(EGOPQ_ERR_INVALID_ARG, "a_q is required by the GEMV path");
  cudaError_t e = (use == EGOPQ_PATH_GEMV) ? launch_gemv(a, st) : launch_tc_gemm(a, st);
  if (e == cudaErrorNotSupported)
    return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "shape not supported by the requested path");
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return EGOPQ_OK;
}

}  // namespace

extern "C" {

int egopq_version(void) { return 1 * 10000 + 0 * 100 + 0; }

const char* egopq_last_error_string(void) { return g_msg; }

size_t egopq_packed_w4_bytes(int64_t N, int64_t K, int group) {
  if (group != 128 || N <= 0 || K <= 0 || N % 128 || K % 128 || N >= kMaxDim || K >= kMaxDim)
    return 0;
  const int64_t G = K / 128;
  return (size_t)(N * K / 2 + 2 * G * N + G * N / 2);
}

int egopq_pack_w4(const uint8_t* w_q, const uint16_t* scale_f16, const uint8_t* zero, int64_t N,
                  int64_t K, int group, void* packed, egopq_stream_t stream) {
  int rc = check_w4_shape(0, N, K, group);
  if (rc) return rc;
  rc = check_ptrs(4, "w_q", w_q, "scale_f16", scale_f16, "zero", zero, "packed", packed);
  if (rc) return rc;
  if ((rc = check_arch())) return rc;
  cudaError_t e = launch_pack_w4(w_q, scale_f16, zero, N, K, packed, (cudaStream_t)stream);
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "pack_w4 launch");
}

int egopq_unpack_w4(const void* packed, int64_t N, int64_t K, int group, uint8_t* w_q,
                    uint16_t* scale_f16, uint8_t* zero, egopq_stream_t stream) {
  int rc = check_w4_shape(0, N, K, group);
  if (rc) return rc;
  rc = check_ptrs(4, "packed", packed, "w_q", w_q, "scale_f16", scale_f16, "zero", zero);
  if (rc) return rc;
  if ((rc = check_arch())) return rc;
  cudaError_t e = launch_unpack_w4(packed, N, K, w_q, scale_f16, zero, (cudaStream_t)stream);
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "unpack_w4 launch");
}

int egopq_pack_w4_gptq(const int32_t* qweight, const int32_t* qzeros, const uint16_t* scales_f16,
                       int64_t N, int64_t K, int group, int zero_offset, void* packed,
                       egopq_stream_t stream) {
  int rc = check_w4_shape(0, N, K, group);
  if (rc) return rc;
  if (zero_offset != 0 && zero_offset != 1)
    return fail(EGOPQ_ERR_INVALID_ARG, "zero_offset must be 0 or 1 (got %d)", zero_offset);
  rc = check_ptrs(4, "qweight", qweight, "qzeros", qzeros, "scales_f16", scales_f16, "packed",
                  packed);
  if (rc) return rc;
  if ((rc = check_arch())) return rc;
  cudaError_t e =
      launch_pack_w4_gptq(qweight, qzeros, scales_f16, N, K, zero_offset, packed, (cudaStream_t)stream);
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "pack_w4_gptq launch");
}

int egopq_dequant_w4(const void* packed, int64_t N, int64_t K, int group, uint16_t* w_bf16,
                     egopq_stream_t stream) {
  int rc = check_w4_shape(0, N, K, group);
  if (rc) return rc;
  rc = check_ptrs(2, "packed", packed, "w_bf16", w_bf16);
  if (rc) return rc;
  if ((rc = check_arch())) return rc;
  cudaError_t e = launch_dequant_w4(packed, N, K, w_bf16, (cudaStream_t)stream);
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "dequant_w4 launch");
}

int egopq_quant_act_i8(const uint16_t* x_bf16, int64_t M, int64_t K, int group, int8_t* a_q,
                       float* a_s, int32_t* a_gsum, void* a_tc, egopq_stream_t stream) {
  if (M < 0 || K <= 0)
    return fail(EGOPQ_ERR_INVALID_ARG, "bad sizes M=%lld K=%lld", (long long)M, (long long)K);
  if (M >= kMaxDim || K >= kMaxDim)
    return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "sizes M=%lld K=%lld exceed 2^31 - 1", (long long)M,
                (long long)K);
  if (group != 128) return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "group must be 128 (got %d)", group);
  if (K % 128) return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "K must be a multiple of 128");
  if (M == 0) return EGOPQ_OK;
  int rc = check_ptrs(3, "x_bf16", x_bf16, "a_s", a_s, "a_gsum", a_gsum);
  if (rc) return rc;
  if (!a_q && !a_tc) return fail(EGOPQ_ERR_INVALID_ARG, "a_q and a_tc are both NULL");
  if (a_tc && !aligned16(a_tc)) return fail(EGOPQ_ERR_MISALIGNED, "a_tc is not 16-byte aligned");
  if (a_q && !aligned16(a_q)) return fail(EGOPQ_ERR_MISALIGNED, "a_q is not 16-byte aligned");
  if ((rc = check_arch())) return rc;
  cudaError_t e = launch_quant_act(x_bf16, M, K, a_q, a_s, a_gsum, a_tc, (cudaStream_t)stream);
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "quant_act launch");
}

int egopq_w4a8_gemm_ex(const int8_t* a_q, const void* a_tc, const float* a_s,
                       const int32_t* a_gsum, const void* packed, int64_t M, int64_t N,
                       int64_t K, int group, uint16_t* y_bf16, int path, egopq_stream_t stream) {
  int rc = check_w4_shape(M, N, K, group);
  if (rc) return rc;
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(4, "a_s", a_s, "a_gsum", a_gsum, "packed", packed, "y_bf16", y_bf16);
  if (rc) return rc;
  if (a_tc && !aligned16(a_tc)) return fail(EGOPQ_ERR_MISALIGNED, "a_tc is not 16-byte aligned");
  if (a_q && !aligned16(a_q)) return fail(EGOPQ_ERR_MISALIGNED, "a_q is not 16-byte aligned");
  GemmArgs a{};
  a.variant = kW4A8;
  a.M = M;
  a.N = N;
  a.K = K;
  a.a_q = a_q;
  a.a_tc = a_tc;
  a.a_s = a_s;
  a.a_gsum = a_gsum;
  a.packed = static_cast<const uint8_t*>(packed);
  a.y = y_bf16;
  a.timeout_ns = kDefaultTimeoutNs;
  return run_gemm(a, path, (cudaStream_t)stream);
}

}  // extern "C"

namespace {

// Validate a sibling-linear list and build its segment table (total output
// rows in *n_total).
int build_segs(int count, const void* const* packed, const int64_t* N, uint16_t* const* y,
               SegTable* t, int64_t* n_total) {
  if (count < 1 || count > kMaxSegs)
    return fail(EGOPQ_ERR_INVALID_ARG, "count must be in [1, %d] (got %d)", kMaxSegs, count);
  if (!packed || !N || !y) return fail(EGOPQ_ERR_INVALID_ARG, "packed, N and y_bf16 must be non-NULL");
  *t = SegTable{};
  t->count = count;
  int64_t tiles = 0;
  for (int j = 0; j < count; ++j) {
    if (N[j] <= 0) return fail(EGOPQ_ERR_INVALID_ARG, "N[%d] = %lld", j, (long long)N[j]);
    if (N[j] % 128)
      return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "N[%d] = %lld is not a multiple of 128", j,
                  (long long)N[j]);
    if (!packed[j] || !y[j]) return fail(EGOPQ_ERR_INVALID_ARG, "packed[%d] or y_bf16[%d] is NULL", j, j);
    if (!aligned16(packed[j]) || !aligned16(y[j]))
      return fail(EGOPQ_ERR_MISALIGNED, "packed[%d] or y_bf16[%d] is not 16-byte aligned", j, j);
    t->tile0[j] = (int)tiles;
    t->packed[j] = static_cast<const uint8_t*>(packed[j]);
    t->y[j] = y[j];
    t->N[j] = N[j];
    tiles += N[j] / 128;
    if (tiles * 128 >= kMaxDim)
      return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "the linears' outputs exceed 2^31 - 1 rows");
  }
  t->tile0[count] = (int)tiles;
  *n_total = tiles * 128;
  return EGOPQ_OK;
}

}  // namespace

extern "C" {

int egopq_w4a8_gemm_grouped(const int8_t* a_q, const void* a_tc, const float* a_s,
                            const int32_t* a_gsum, int count, const void* const* packed,
                            const int64_t* N, int64_t M, int64_t K, int group,
                            uint16_t* const* y_bf16, int path, egopq_stream_t stream) {
  SegTable segs;
  int64_t n_total = 0;
  int rc = build_segs(count, packed, N, y_bf16, &segs, &n_total);
  if (rc) return rc;
  if ((rc = check_w4_shape(M, n_total, K, group))) return rc;
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(2, "a_s", a_s, "a_gsum", a_gsum);
  if (rc) return rc;
  if (a_tc && !aligned16(a_tc)) return fail(EGOPQ_ERR_MISALIGNED, "a_tc is not 16-byte aligned");
  if (a_q && !aligned16(a_q)) return fail(EGOPQ_ERR_MISALIGNED, "a_q is not 16-byte aligned");
  GemmArgs a{};
  a.variant = kW4A8;
  a.M = M;
  a.N = n_total;
  a.K = K;
  a.a_q = a_q;
  a.a_tc = a_tc;
  a.a_s = a_s;
  a.a_gsum = a_gsum;
  a.packed = segs.packed[0];
  a.y = segs.y[0];
  a.segs = &segs;
  a.timeout_ns = kDefaultTimeoutNs;
  return run_gemm(a, path, (cudaStream_t)stream);
}

int egopq_w4a8_gemm(const int8_t* a_q, const void* a_tc, const float* a_s,
                    const int32_t* a_gsum, const void* packed, int64_t M, int64_t N, int64_t K,
                    int group, uint16_t* y_bf16, egopq_stream_t stream) {
  return egopq_w4a8_gemm_ex(a_q, a_tc, a_s, a_gsum, packed, M, N, K, group, y_bf16,
                            EGOPQ_PATH_AUTO, stream);
}

// Workspace of the one-call linear: the quantized activations it stages
// between its two kernels, in 256-byte aligned regions -- scales fp32 [M],
// group sums int32 [M][G], then the codes in the form the path reads: int8
// [M][K] for the GEMV, the 2*M*K-byte operand form for the tensor cores.
static size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
static int linear_path(int64_t M, int path) { return auto_path(M, kW4A8, path); }

size_t egopq_w4a8_linear_workspace_bytes(int64_t M, int64_t K, int group, int path) {
  if (M <= 0 || K <= 0 || group != 128 || K % 128 || M >= kMaxDim || K >= kMaxDim) return 0;
  if (path != EGOPQ_PATH_AUTO && path != EGOPQ_PATH_GEMV && path != EGOPQ_PATH_TC) return 0;
  const bool tc = linear_path(M, path) == EGOPQ_PATH_TC;
  return align256((size_t)(4 * M)) + align256((size_t)(4 * M * (K / 128))) +
         align256((size_t)((tc ? 2 : 1) * M * K));
}

}  // extern "C"

namespace egopq {
// Record `msg` as the calling thread's last error (read back through
// egopq_last_error_string) and return `code`.
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }

// Quantize x into `ws` (layout above) and run the W4A8 GEMM of the linears in
// `segs` (N output rows in all) on `use`.
int run_linear_segs(const uint16_t* x_bf16, const SegTable& segs, int64_t M, int64_t N, int64_t K,
                    uint8_t* ws, int use, cudaStream_t st) {
  float* a_s = reinterpret_cast<float*>(ws);
  int32_t* asum = reinterpret_cast<int32_t*>(ws + align256((size_t)(4 * M)));
  uint8_t* codes = reinterpret_cast<uint8_t*>(asum) + align256((size_t)(4 * M * (K / 128)));
  int8_t* a_q = use == EGOPQ_PATH_TC ? nullptr : reinterpret_cast<int8_t*>(codes);
  void* a_tc = use == EGOPQ_PATH_TC ? codes : nullptr;
  cudaError_t e = launch_quant_act(x_bf16, M, K, a_q, a_s, asum, a_tc, st);
  if (e != cudaSuccess) return cuda_fail(e, "quant_act launch");
  GemmArgs a{};
  a.variant = kW4A8;
  a.M = M;
  a.N = N;
  a.K = K;
  a.a_q = a_q;
  a.a_tc = a_tc;
  a.a_s = a_s;
  a.a_gsum = asum;
  a.packed = segs.packed[0];
  a.y = segs.y[0];
  a.segs = &segs;
  a.timeout_ns = kDefaultTimeoutNs;
  e = (use == EGOPQ_PATH_GEMV) ? launch_gemv(a, st) : launch_tc_gemm(a, st);
  if (e == cudaErrorNotSupported)
    return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "shape not supported by the requested path");
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "gemm launch");
}

// The one-call linear of a single weight.
int run_linear(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N, int64_t K,
               uint16_t* y_bf16, uint8_t* ws, int use, cudaStream_t st) {
  SegTable segs{};
  segs.count = 1;
  segs.tile0[0] = 0;
  segs.tile0[1] = (int)(N / 128);
  segs.packed[0] = static_cast<const uint8_t*>(packed);
  segs.y[0] = y_bf16;
  segs.N[0] = N;
  return run_linear_segs(x_bf16, segs, M, N, K, ws, use, st);
}
}  // namespace egopq

extern "C" {

int egopq_w4a8_linear(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N, int64_t K,
                      int group, uint16_t* y_bf16, void* workspace, size_t workspace_bytes,
                      int path, egopq_stream_t stream) {
  int rc = check_w4_shape(M, N, K, group);
  if (rc) return rc;
  if (path != EGOPQ_PATH_AUTO && path != EGOPQ_PATH_GEMV && path != EGOPQ_PATH_TC)
    return fail(EGOPQ_ERR_INVALID_ARG, "unknown path %d", path);
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(4, "x_bf16", x_bf16, "packed", packed, "y_bf16", y_bf16, "workspace", workspace);
  if (rc) return rc;
  const size_t need = egopq_w4a8_linear_workspace_bytes(M, K, group, path);
  if (workspace_bytes < need)
    return fail(EGOPQ_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than %zu", workspace_bytes,
                need);
  if ((rc = check_arch())) return rc;
  return run_linear(x_bf16, packed, M, N, K, y_bf16, static_cast<uint8_t*>(workspace),
                    linear_path(M, path), (cudaStream_t)stream);
}

int egopq_w4a8_linear_grouped(const uint16_t* x_bf16, int count, const void* const* packed,
                              const int64_t* N, int64_t M, int64_t K, int group,
                              uint16_t* const* y_bf16, void* workspace, size_t workspace_bytes,
                              int path, egopq_stream_t stream) {
  SegTable segs;
  int64_t n_total = 0;
  int rc = build_segs(count, packed, N, y_bf16, &segs, &n_total);
  if (rc) return rc;
  if ((rc = check_w4_shape(M, n_total, K, group))) return rc;
  if (path != EGOPQ_PATH_AUTO && path != EGOPQ_PATH_GEMV && path != EGOPQ_PATH_TC)
    return fail(EGOPQ_ERR_INVALID_ARG, "unknown path %d", path);
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(2, "x_bf16", x_bf16, "workspace", workspace);
  if (rc) return rc;
  const size_t need = egopq_w4a8_linear_workspace_bytes(M, K, group, path);
  if (workspace_bytes < need)
    return fail(EGOPQ_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than %zu", workspace_bytes,
                need);
  if ((rc = check_arch())) return rc;
  return run_linear_segs(x_bf16, segs, M, n_total, K, static_cast<uint8_t*>(workspace),
                         linear_path(M, path), (cudaStream_t)stream);
}

int egopq_w4a8_group_partials(const int8_t* a_q, const void* a_tc, const int32_t* a_gsum,
                              const void* packed, int64_t M, int64_t N, int64_t K, int group,
                              int32_t* Q, int path, egopq_stream_t stream) {
  int rc = check_w4_shape(M, N, K, group);
  if (rc) return rc;
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(3, "a_gsum", a_gsum, "packed", packed, "Q", Q);
  if (rc) return rc;
  if (a_tc && !aligned16(a_tc)) return fail(EGOPQ_ERR_MISALIGNED, "a_tc is not 16-byte aligned");
  if (a_q && !aligned16(a_q)) return fail(EGOPQ_ERR_MISALIGNED, "a_q is not 16-byte aligned");
  GemmArgs a{};
  a.variant = kW4A8;
  a.M = M;
  a.N = N;
  a.K = K;
  a.a_q = a_q;
  a.a_tc = a_tc;
  a.a_gsum = a_gsum;
  a.packed = static_cast<const uint8_t*>(packed);
  a.partials = Q;
  a.timeout_ns = kDefaultTimeoutNs;
  return run_gemm(a, path, (cudaStream_t)stream);
}

int egopq_w4a16_gemm_ex(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N,
                        int64_t K, int group, uint16_t* y_bf16, int path,
                        egopq_stream_t stream) {
  int rc = check_w4_shape(M, N, K, group);
  if (rc) return rc;
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(3, "x_bf16", x_bf16, "packed", packed, "y_bf16", y_bf16);
  if (rc) return rc;
  GemmArgs a{};
  a.variant = kW4A16;
  a.M = M;
  a.N = N;
  a.K = K;
  a.x = x_bf16;
  a.packed = static_cast<const uint8_t*>(packed);
  a.y = y_bf16;
  a.timeout_ns = kDefaultTimeoutNs;
  return run_gemm(a, path, (cudaStream_t)stream);
}

int egopq_w4a16_gemm(const uint16_t* x_bf16, const void* packed, int64_t M, int64_t N,
                     int64_t K, int group, uint16_t* y_bf16, egopq_stream_t stream) {
  return egopq_w4a16_gemm_ex(x_bf16, packed, M, N, K, group, y_bf16, EGOPQ_PATH_AUTO, stream);
}

int egopq_w8a16_gemm_ex(const uint16_t* x_bf16, const int8_t* w_q, const uint16_t* scale_f16,
                        int64_t M, int64_t N, int64_t K, uint16_t* y_bf16, int path,
                        egopq_stream_t stream) {
  int rc = check_w4_shape(M, N, K, 128);
  if (rc) return rc;
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(4, "x_bf16", x_bf16, "w_q", w_q, "scale_f16", scale_f16, "y_bf16", y_bf16);
  if (rc) return rc;
  GemmArgs a{};
  a.variant = kW8A16;
  a.M = M;
  a.N = N;
  a.K = K;
  a.x = x_bf16;
  a.w8 = w_q;
  a.s8 = scale_f16;
  a.y = y_bf16;
  a.timeout_ns = kDefaultTimeoutNs;
  return run_gemm(a, path, (cudaStream_t)stream);
}

int egopq_w8a16_gemm(const uint16_t* x_bf16, const int8_t* w_q, const uint16_t* scale_f16,
                     int64_t M, int64_t N, int64_t K, uint16_t* y_bf16, egopq_stream_t stream) {
  return egopq_w8a16_gemm_ex(x_bf16, w_q, scale_f16, M, N, K, y_bf16, EGOPQ_PATH_AUTO, stream);
}

int egopq_w8a8_gemm_ex(const int8_t* a_q, const void* a_tc, const float* a_s, const int8_t* w_q,
                       const uint16_t* scale_f16, int64_t M, int64_t N, int64_t K,
                       uint16_t* y_bf16, int path, egopq_stream_t stream) {
  int rc = check_w4_shape(M, N, K, 128);
  if (rc) return rc;
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(4, "a_s", a_s, "w_q", w_q, "scale_f16", scale_f16, "y_bf16", y_bf16);
  if (rc) return rc;
  if (a_tc && !aligned16(a_tc)) return fail(EGOPQ_ERR_MISALIGNED, "a_tc is not 16-byte aligned");
  if (a_q && !aligned16(a_q)) return fail(EGOPQ_ERR_MISALIGNED, "a_q is not 16-byte aligned");
  GemmArgs a{};
  a.variant = kW8A8;
  a.M = M;
  a.N = N;
  a.K = K;
  a.a_q = a_q;
  a.a_tc = a_tc;
  a.a_s = a_s;
  a.w8 = w_q;
  a.s8 = scale_f16;
  a.y = y_bf16;
  a.timeout_ns = kDefaultTimeoutNs;
  return run_gemm(a, path, (cudaStream_t)stream);
}

int egopq_w8a8_gemm(const int8_t* a_q, const void* a_tc, const float* a_s, const int8_t* w_q,
                    const uint16_t* scale_f16, int64_t M, int64_t N, int64_t K, uint16_t* y_bf16,
                    egopq_stream_t stream) {
  return egopq_w8a8_gemm_ex(a_q, a_tc, a_s, w_q, scale_f16, M, N, K, y_bf16, EGOPQ_PATH_AUTO,
                            stream);
}

int egopq_bf16_gemm_twin(const uint16_t* x_bf16, const uint16_t* w_bf16, int64_t M, int64_t N,
                         int64_t K, uint16_t* y_bf16, egopq_stream_t stream) {
  int rc = check_w4_shape(M, N, K, 128);
  if (rc) return rc;
  if (M == 0) return EGOPQ_OK;
  rc = check_ptrs(3, "x_bf16", x_bf16, "w_bf16", w_bf16, "y_bf16", y_bf16);
  if (rc) return rc;
  if ((rc = check_arch())) return rc;
  GemmArgs a{};
  a.variant = kW16A16;
  a.M = M;
  a.N = N;
  a.K = K;
  a.x = x_bf16;
  a.w16 = w_bf16;
  a.y = y_bf16;
  a.timeout_ns = kDefaultTimeoutNs;
  cudaError_t e = launch_tc_gemm(a, (cudaStream_t)stream);
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "bf16 twin launch");
}

int egopq_supported(int64_t M, int64_t N, int64_t K, int group, int variant) {
  if (variant < EGOPQ_VARIANT_W4A8 || variant > EGOPQ_VARIANT_W8A8) return 0;
  if (variant == EGOPQ_VARIANT_W8A16 || variant == EGOPQ_VARIANT_W8A8) group = 128;
  if (M < 0 || N <= 0 || K <= 0 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim) return 0;
  if (group != 128 || K % 128 || N % 128) return 0;
  if (check_arch() != EGOPQ_OK) return 0;
  return 1;
}

int egopq_auto_path(int64_t M, int variant) {
  if (variant < EGOPQ_VARIANT_W4A8 || variant > EGOPQ_VARIANT_W8A8 || M < 0)
    return fail(EGOPQ_ERR_INVALID_ARG, "bad variant %d or M %lld", variant, (long long)M);
  return auto_path(M, variant, EGOPQ_PATH_AUTO);
}

int egopq_tc_token_tile(int64_t M, int64_t N, int64_t K, int variant) {
  if (variant < EGOPQ_VARIANT_W4A8 || variant > EGOPQ_VARIANT_W8A8 || M <= 0)
    return fail(EGOPQ_ERR_INVALID_ARG, "bad variant %d or M %lld", variant, (long long)M);
  if (N <= 0 || K <= 0 || N % 128 || K % 128 || M >= kMaxDim || N >= kMaxDim || K >= kMaxDim)
    return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "shape %lld x %lld x %lld", (long long)M,
                (long long)N, (long long)K);
  if (variant == EGOPQ_VARIANT_W8A8 && M <= kTcFp8MaxM)
    return fail(EGOPQ_ERR_UNSUPPORTED_SHAPE, "W8A8 has no tensor-core form for M <= %d",
                kTcFp8MaxM);
  return tc_token_tile(variant, M, N, K);
}

int egopq_tc_launches(int64_t M, int64_t N, int64_t K, int variant) {
  const int bt = egopq_tc_token_tile(M, N, K, variant);
  return bt < 0 ? bt : tc_launches(variant, M, N, K);
}

size_t egopq_tc_operand_bytes(int64_t M, int64_t K, int group) {
  if (M <= 0 || K <= 0 || M >= kMaxDim || K >= kMaxDim || group != 128 || K % 128) return 0;
  return (size_t)(2 * M * K);
}

int egopq_tc_operand_form(int64_t M) {
  if (M <= 0 || M >= kMaxDim) return fail(EGOPQ_ERR_INVALID_ARG, "bad M %lld", (long long)M);
  return M <= kTcFp8MaxM ? EGOPQ_TC_FORM_E4M3_PLANES : EGOPQ_TC_FORM_F16;
}

int egopq_device_status(egopq_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0;
  cudaError_t (*const take[])(unsigned*) = {take_error_word_quant_pack, take_error_word_gemv,
                                            take_error_word_tc_gemm};
  for (auto fn : take) {
    unsigned int w = 0;
    e = fn(&w);
    if (e != cudaSuccess) return cuda_fail(e, "read and clear a device error word");
    word |= w;
  }
  if (word & kErrTimeout) return fail(EGOPQ_ERR_TIMEOUT, "a kernel's bounded wait expired");
  if (word & kErrIndex)
    return fail(EGOPQ_ERR_DEVICE_INDEX, "a device-side index check of the debug build failed");
  if (word & kErrRange)
    return fail(EGOPQ_ERR_INVALID_ARG, "an imported zero point is outside [0, 15]");
  return EGOPQ_OK;
}

int egopq_debug_build(void) {
#ifdef EGOPQ_DEBUG
  return 1;
#else
  return 0;
#endif
}

int egopq_debug_set_record_limit(uint64_t bytes) {
#ifdef EGOPQ_DEBUG
  int rc = check_arch();
  if (rc) return rc;
  cudaError_t e = set_record_limit_gemv(bytes);
  if (e == cudaSuccess) e = set_record_limit_tc_gemm(bytes);
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "set the record limit");
#else
  (void)bytes;
  return fail(EGOPQ_ERR_INVALID_ARG, "egopq_debug_set_record_limit needs the debug build");
#endif
}

int egopq_selftest_timeout(int timeout_us, egopq_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000)
    return fail(EGOPQ_ERR_INVALID_ARG, "timeout_us must be in [1, 1000000]");
  int rc = check_arch();
  if (rc) return rc;
  cudaError_t e = launch_selftest_timeout((uint64_t)timeout_us * 1000ull, (cudaStream_t)stream);
  return e == cudaSuccess ? EGOPQ_OK : cuda_fail(e, "selftest launch");
}

}  // extern "C"
