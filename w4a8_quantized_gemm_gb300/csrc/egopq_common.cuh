// egopq_common.cuh -- device helpers shared by the egopq kernels (sm_103a).
//
// Thin inline-PTX wrappers for mbarriers, TMA (cp.async.bulk[.tensor]),
// Tensor Memory (tcgen05.alloc/ld/st) and the fifth-generation tensor-core MMA
// (tcgen05.mma kind::f16), plus the library's device error word. Every wait
// is bounded by a %globaltimer deadline: on expiry it raises the CTA's abort
// flag and the device error word instead of spinning forever.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace egopq {

// ---- device error word ----------------------------------------------------
// Bit 0: a bounded wait expired (EGOPQ_ERR_TIMEOUT on the host side).
// Bit 1: an imported value the packed format cannot hold (a GPTQ zero point
// outside [0, 15] after its offset; EGOPQ_ERR_INVALID_ARG).
// One word per translation unit: the library compiles every unit as a whole
// program (no relocatable device code), which is what lets ptxas honour
// per-warpgroup register budgets (setmaxnreg). Each unit with kernels exports
// a take_error_word_* function; the host ORs and clears them all.
constexpr unsigned kErrTimeout = 1u;
constexpr unsigned kErrRange = 2u;
// Bit 2: a debug build's device-side index check failed (EGOPQ_ERR_DEVICE_INDEX).
constexpr unsigned kErrIndex = 4u;
static __device__ unsigned int g_error_word = 0;

// Host: read this unit's word and clear it if set.
static inline cudaError_t take_local_error_word(unsigned* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_error_word, sizeof(unsigned));
  if (e != cudaSuccess || *out == 0) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned));
}

__device__ __forceinline__ void raise_error(unsigned bits) { atomicOr(&g_error_word, bits); }

// ---- debug builds (EGOPQ_DEBUG): device-side read-index checks ---------------
// dbg_ok(off, len, size): the read [off, off + len) lies inside a buffer of
// `size` elements or bytes. A failed check records kErrIndex and returns
// false; the caller then reads a known-valid address instead, so the check
// never becomes a fault. dbg_record_ok() checks reads of packed weight records
// against the buffer's size or, when a test has set it lower, against
// g_dbg_record_limit: the checks can then be made to fire while every read
// stays inside the real buffer. Release builds compile the checks away.
#ifdef EGOPQ_DEBUG
static __device__ unsigned long long g_dbg_record_limit = 0;  // 0: the buffer's size
__device__ __forceinline__ bool dbg_ok(uint64_t off, uint64_t len, uint64_t size) {
  if (off + len <= size) return true;
  raise_error(kErrIndex);
  return false;
}
__device__ __forceinline__ bool dbg_record_ok(uint64_t off, uint64_t len, uint64_t size) {
  const unsigned long long lim = *reinterpret_cast<volatile unsigned long long*>(&g_dbg_record_limit);
  return dbg_ok(off, len, (lim != 0 && lim < size) ? lim : size);
}
static inline cudaError_t set_local_record_limit(unsigned long long bytes) {
  return cudaMemcpyToSymbol(g_dbg_record_limit, &bytes, sizeof(bytes));
}
#else
__device__ __forceinline__ constexpr bool dbg_ok(uint64_t, uint64_t, uint64_t) { return true; }
__device__ __forceinline__ constexpr bool dbg_record_ok(uint64_t, uint64_t, uint64_t) {
  return true;
}
static inline cudaError_t set_local_record_limit(unsigned long long) {
  return cudaErrorNotSupported;
}
#endif

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t elect_lane0() { return (threadIdx.x & 31) == 0; }

// ---- mbarrier -------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of phase `parity` (a cheaper round trip than try_wait,
// which may hold the thread for a while before reporting failure).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on phase `parity`. Returns false (and raises the abort flag and
// the error word) once `timeout_ns` has passed, or as soon as another thread
// of the CTA has raised the abort flag, or once any CTA has recorded a timeout
// in the device error word (so one failure ends the whole grid quickly; the
// word stays set until the host reads it with egopq_device_status).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t timeout_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((it & 63) == 0) {
      if (*reinterpret_cast<volatile unsigned int*>(&g_error_word) & kErrTimeout) {
        *abort_flag = 1;
        return false;
      }
      if (globaltimer() - t0 > timeout_ns) {
        *abort_flag = 1;
        raise_error(kErrTimeout);
        return false;
      }
    }
  }
}

// ---- packed fp32 arithmetic (sm_100 and later) ------------------------------
// {r0, r1} += s * {v0, v1} as one fma.rn.f32x2: two independent
// round-to-nearest FMAs, bit for bit what fmaf gives each lane, in one issue.
// s2 holds s in both halves (f32x2_splat).
__device__ __forceinline__ uint64_t f32x2_splat(float s) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %1};" : "=l"(d) : "f"(s));
  return d;
}
__device__ __forceinline__ void fma_f32x2(float& r0, float& r1, uint64_t s2, uint32_t v0,
                                          uint32_t v1) {
  uint64_t r, v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(r0), "f"(r1));
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(v0), "r"(v1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(r) : "l"(s2), "l"(v));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r0), "=f"(r1) : "l"(r));
}

// ---- TMA --------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// 1-D bulk copy: both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Tiled bulk store shared -> global (2-D), tracked by the issuing thread's
// bulk async-groups; rows or columns past the tensor's extent are not written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until every committed bulk store of this thread has finished reading
// its shared-memory source (the buffer may then be rewritten).
__device__ __forceinline__ void bulk_wait_group_read0() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_group0() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA) before a bulk store reads them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- Tensor Memory and tcgen05 ---------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T, A is M x K (lanes = rows), B is N x K.
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with kind::f8f6f4 (A and B e4m3, K = 32 per instruction).
__device__ __forceinline__ void tc_mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 16 consecutive 32-bit columns, one lane per thread of the warp.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 8 consecutive columns (results in r[0..7]).
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// Per-warpgroup register budget (all four warps execute the same one; R a
// multiple of 8 in [24, 256]). An increase waits until other warpgroups of
// the block have released enough, so the budgets must add up to at most what
// the block was launched with.
template <int R>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

// Shared-memory matrix descriptor (tcgen05 form) for a K-major operand staged
// by TMA with 128-byte swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes
// (stride byte offset), version field 1, layout type 2 (SWIZZLE_128B). The
// leading byte offset is unused for swizzled K-major layouts. Atom bases must
// be 1024-byte aligned; a K step inside an atom advances the start address.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with f32 accumulation, both operands
// K-major. ab_bf16 selects bf16 (1) or fp16 (0) for A and B alike. With
// ab_bf16 = 0 it is also the kind::f8f6f4 descriptor for e4m3 A and B (format
// code 0 in the same fields).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int ab_bf16) {
  return (1u << 4) | (static_cast<uint32_t>(ab_bf16) << 7) |
         (static_cast<uint32_t>(ab_bf16) << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---- programmatic dependent launch ---------------------------------------------
// Wait until the preceding grid in the stream has completed and its writes are
// visible (a no-op when the launch carried no programmatic dependency).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Allow the next grid in the stream to begin launching.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- cluster helpers -----------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ---- small numeric helpers -------------------------------------------------------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t magic) {
  uint32_t r;
  // (a & mask) | magic
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(mask), "r"(magic));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ float f16_bits_to_f32(uint16_t h) {
  return __half2float(__ushort_as_half(h));
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

}  // namespace egopq
