// gemv.cu -- CUDA-core decode kernels for small M (up to 16 token rows per launch).
//
// Decode is a weight-streaming problem: every packed weight byte is read once
// per token batch, so the kernels below are built to keep HBM busy. Each CTA
// owns one 128-row tile of the output (one consumer thread per weight row,
// four consumer warps) and a contiguous range of K groups; a producer warp
// streams the range's packed records through a shared-memory ring, one bulk
// copy per group. When the tiles do not fill the GPU, a cluster of up to 8
// CTAs splits a tile's groups and reduces the partial sums through
// distributed shared memory -- no global scratch, fixed summation order,
// deterministic output.
//
// W4A8: per (row n, group g) the integer partial
//   Q = sum_{k in g} a_q*w_q - z[n,g] * a_gsum[m,g]
// is formed exactly with dp4a on the raw codes (zero point folded through the
// per-group activation sums), then acc += s[n,g] * Q in fp32 and
// y = bf16(a_s[m] * acc). The packed nibble order puts K offsets
// {0,4,1,5} and {2,6,3,7} of each 8-wide run in the low/high nibbles of the
// four bytes of a word, so the activations are permuted the same way when
// staged. ("The 4-bit CPU path", section "W4A16 - PyTorch tinygemm": a
// per-row weight kernel is the right tool for decode-sized batches.)
//
// W4A16: the same skeleton with fp32 FMAs of bf16 activations against exact
// (w_q - z) values, scaled per group.
//
// W8A8: the same walk on int8 activation codes, dp4a into exact int32 sums.
//
// W8A16: int8 row-major weights, one warp per 4 rows, 16-byte coalesced loads
// along K and a warp-shuffle reduction; y = bf16(s[n] * sum_k x*w_q).
#include "egopq_internal.h"

namespace egopq {

constexpr int kGemvConsumers = 128;                 // one thread per weight row of a tile
constexpr int kGemvThreads = kGemvConsumers + 32;   // + one producer warp
constexpr int kGemvStages = 8;
constexpr int kGemvStageBytes = 8512;               // one packed record: codes, scales, zeros
constexpr int kGemvMaxGroupsPerCta = 64;

struct GemvParams {
  int64_t M, N, K;  // N: output rows of all linears together
  int G, ks, rows;
  const int8_t* a_q;
  const float* a_s;
  const int32_t* a_gsum;
  const uint16_t* x;
  int32_t* partials;
  uint64_t timeout_ns;
  SegTable seg;  // packed weight and output of each linear (outputs offset to this row chunk)
};

// Decode kernel for the packed int4 weight (W4A8 and W4A16). CTA = one
// 128-row tile x a contiguous range of groups; a producer lane streams each
// group's 8512-byte packed record (codes, 128 scales, 64 bytes of zero
// nibbles) into an 8-stage shared-memory ring with one 1-D bulk copy per
// group -- few, large copies keep the copy engine's per-copy cost out of the
// way -- starting before the preceding kernel has finished; each consumer
// thread owns one weight row.
template <int VARIANT, int MT, bool PARTIALS>
__global__ void __launch_bounds__(kGemvThreads)
gemv_w4_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x, t = blockIdx.y;
  const int G = p.G;
  const int g0 = (int)((int64_t)ks * G / p.ks), g1 = (int)((int64_t)(ks + 1) * G / p.ks);
  const int ng = g1 - g0;
  const int64_t K = p.K;
  const TileRef tile = tile_ref(p.seg, t, G);  // this tile's linear
  const int64_t N = tile.N;

  // smem: ring | barriers | abort flag | reduction buffer | staged activations
  uint8_t* ring = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kGemvStages * kGemvStageBytes);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kGemvStages);
  float* red = reinterpret_cast<float*>(smem + kGemvStages * kGemvStageBytes + 256);
  uint8_t* act = reinterpret_cast<uint8_t*>(red + MT * 128);
  auto full_bar = [&](int s) { return smem_u32(bars + s); };
  auto empty_bar = [&](int s) { return smem_u32(bars + kGemvStages + s); };
  const uint64_t tmo = p.timeout_ns;

  float red_scale[MT];  // (consumers) token scales for the split-K epilogue
#pragma unroll
  for (int m = 0; m < MT; ++m) red_scale[m] = 1.f;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGemvStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      // one copy per group: the packed record holds codes, scales and zeros
      auto issue = [&](int i) {
        const int s = i % kGemvStages, g = g0 + i;
        mbar_arrive_expect_tx(full_bar(s), kGemvStageBytes);
        const uint8_t* seg_base = p.seg.packed[tile.seg];
        const uint8_t* src = tile.rec0 + (int64_t)g * kGemvStageBytes;
        if (!dbg_record_ok((uint64_t)(src - seg_base), kGemvStageBytes,
                           packed_record_bytes(tile.N, G)))
          src = seg_base;
        bulk_load(smem_u32(ring + s * kGemvStageBytes), src, kGemvStageBytes, full_bar(s));
      };
      int issued = 0;
      for (int i = 0; i < ng; ++i) {
        if (i >= kGemvStages &&
            !mbar_wait(empty_bar(i % kGemvStages), ((i / kGemvStages) & 1) ^ 1, abort_flag, tmo))
          break;
        issue(i);
        ++issued;
      }
      for (int i = (issued > kGemvStages ? issued - kGemvStages : 0); i < issued; ++i) {
        volatile int no_abort = 0;
        mbar_wait(full_bar(i % kGemvStages), (i / kGemvStages) & 1, &no_abort, tmo);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- consumers
    const int r = threadIdx.x;  // row in the tile
    const int64_t n = tile.n0 + r;
    griddep_wait();             // activations come from the preceding kernel
    if (threadIdx.x == 0) griddep_launch_dependents();
    // the tokens' scales, needed only by the epilogue: loaded now so that
    // their latency overlaps the group loop
    float asc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m)
      asc[m] = (VARIANT == kW4A8 && !PARTIALS && m < p.rows) ? __ldg(p.a_s + m) : 1.f;
    // stage this CTA's activations, permuted to the nibble order
    if constexpr (VARIANT == kW4A8) {
      uint2* aw = reinterpret_cast<uint2*>(act);
      int32_t* as = reinterpret_cast<int32_t*>(act + (size_t)ng * MT * 16 * sizeof(uint2));
      for (int i = threadIdx.x; i < ng * MT * 16; i += kGemvConsumers) {
        const int gl = i / (MT * 16), m = (i / 16) % MT, cj = i % 16;
        uint2 v = make_uint2(0, 0);
        if (m < p.rows && dbg_ok((uint64_t)(m * K + (int64_t)(g0 + gl) * 128 + cj * 8), 8,
                                 (uint64_t)p.rows * K)) {
          const int64_t k0 = (int64_t)(g0 + gl) * 128 + cj * 8;
          const uint2 X = *reinterpret_cast<const uint2*>(p.a_q + m * K + k0);
          v.x = prmt(X.x, X.y, 0x5140);  // K offsets {0,4,1,5}
          v.y = prmt(X.x, X.y, 0x7362);  // K offsets {2,6,3,7}
        }
        aw[i] = v;
      }
      for (int i = threadIdx.x; i < ng * MT; i += kGemvConsumers) {
        const int gl = i / MT, m = i % MT;
        as[i] = (m < p.rows && dbg_ok((uint64_t)(m * G + g0 + gl), 1, (uint64_t)p.rows * G))
                    ? p.a_gsum[m * G + g0 + gl]
                    : 0;
      }
    } else {
      float* xs = reinterpret_cast<float*>(act);
      for (int i = threadIdx.x; i < ng * MT * 128; i += kGemvConsumers) {
        const int gl = i / (MT * 128), m = (i / 128) % MT, kk = i % 128;
        // position kk = 32c + 8j + nib holds K offset 32c + 8j + e(nib)
        const int nib = kk & 7;
        const int e = (nib < 4) ? 2 * nib : 2 * (nib - 4) + 1;
        float v = 0.f;
        if (m < p.rows &&
            dbg_ok((uint64_t)(m * K + (int64_t)(g0 + gl) * 128 + (kk & ~7) + e), 1,
                   (uint64_t)p.rows * K))
          v = bf16_bits_to_f32(p.x[m * K + (int64_t)(g0 + gl) * 128 + (kk & ~7) + e]);
        xs[i] = v;
      }
    }
    asm volatile("bar.sync 2, %0;" ::"n"(kGemvConsumers) : "memory");

    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    for (int i = 0; i < ng; ++i) {
      const int s = i % kGemvStages, g = g0 + i;
      if (!mbar_wait(full_bar(s), (i / kGemvStages) & 1, abort_flag, tmo)) break;
      const uint8_t* st = ring + s * kGemvStageBytes;
      uint4 cur[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) cur[c] = *reinterpret_cast<const uint4*>(st + (c * 128 + r) * 16);
      const float sc = f16_bits_to_f32(reinterpret_cast<const uint16_t*>(st + 8192)[r]);
      const uint8_t zb = st[8192 + 256 + (r >> 1)];
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
      const int z = (r & 1) ? (zb >> 4) : (zb & 0xF);
      if constexpr (VARIANT == kW4A8) {
        const uint4* aw = reinterpret_cast<const uint4*>(act) + (size_t)i * MT * 8;
        const int32_t* as =
            reinterpret_cast<const int32_t*>(act + (size_t)ng * MT * 16 * sizeof(uint2));
        int dot[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) dot[m] = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t wv[4] = {cur[c].x, cur[c].y, cur[c].z, cur[c].w};
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const uint32_t lo0 = wv[2 * jj] & 0x0F0F0F0Fu, hi0 = (wv[2 * jj] >> 4) & 0x0F0F0F0Fu;
            const uint32_t lo1 = wv[2 * jj + 1] & 0x0F0F0F0Fu,
                           hi1 = (wv[2 * jj + 1] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const uint4 a = aw[m * 8 + c * 2 + jj];
              dot[m] = __dp4a((int)lo0, (int)a.x, dot[m]);
              dot[m] = __dp4a((int)hi0, (int)a.y, dot[m]);
              dot[m] = __dp4a((int)lo1, (int)a.z, dot[m]);
              dot[m] = __dp4a((int)hi1, (int)a.w, dot[m]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const int q = dot[m] - z * as[i * MT + m];
          if constexpr (PARTIALS) {
            if (m < p.rows) p.partials[((int64_t)m * N + n) * G + g] = q;
          } else {
            acc[m] = fmaf(sc, (float)q, acc[m]);
          }
        }
      } else {
        const float* xs = reinterpret_cast<const float*>(act) + (size_t)i * MT * 128;
        const float zf = 8388608.0f + (float)z;
        float part[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) part[m] = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t wv[4] = {cur[c].x, cur[c].y, cur[c].z, cur[c].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float v[8];
#pragma unroll
            for (int nib = 0; nib < 8; ++nib)
              v[nib] = __uint_as_float(0x4B000000u | ((wv[j] >> (4 * nib)) & 0xFu)) - zf;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
              const float4 xa = *reinterpret_cast<const float4*>(xs + m * 128 + c * 32 + j * 8);
              const float4 xb =
                  *reinterpret_cast<const float4*>(xs + m * 128 + c * 32 + j * 8 + 4);
              part[m] = fmaf(xa.x, v[0], part[m]);
              part[m] = fmaf(xa.y, v[1], part[m]);
              part[m] = fmaf(xa.z, v[2], part[m]);
              part[m] = fmaf(xa.w, v[3], part[m]);
              part[m] = fmaf(xb.x, v[4], part[m]);
              part[m] = fmaf(xb.y, v[5], part[m]);
              part[m] = fmaf(xb.z, v[6], part[m]);
              part[m] = fmaf(xb.w, v[7], part[m]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = fmaf(sc, part[m], acc[m]);
      }
    }
    if constexpr (!PARTIALS) {
      if (p.ks > 1) {
#pragma unroll
        for (int m = 0; m < MT; ++m) red[m * 128 + r] = acc[m];
      } else {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < p.rows) {
            float v = acc[m];
            if constexpr (VARIANT == kW4A8) v = asc[m] * v;
            tile.y[m * N + n] = f32_to_bf16_bits(v);
          }
        }
      }
      if (p.ks > 1) {  // rank 0 applies the scales after the reduction
#pragma unroll
        for (int m = 0; m < MT; ++m) red_scale[m] = asc[m];
      }
    }
  }
  // ---- split-K: reduce the cluster's partial sums through DSMEM (all threads)
  if constexpr (!PARTIALS) {
    if (p.ks > 1) {
      cluster_sync_all();
      if (cluster_ctarank() == 0 && warp < 4) {
        const int r = threadIdx.x;
        const int64_t n = tile.n0 + r;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = red[m * 128 + r];
        const uint32_t local = smem_u32(red);
        // every rank's partials of a chunk of tokens are loaded before any is
        // added (one DSMEM round trip a chunk, not one a rank); the sums keep
        // rank order
        constexpr int MC = MT < 4 ? MT : 4;
#pragma unroll
        for (int m0 = 0; m0 < MT; m0 += MC) {
          float v[7][MC];
#pragma unroll
          for (int rk = 1; rk < 8; ++rk) {
            if (rk < p.ks) {
              const uint32_t remote = map_to_rank(local, rk);
#pragma unroll
              for (int mm = 0; mm < MC; ++mm)
                v[rk - 1][mm] = ld_dsmem_f32(remote + ((m0 + mm) * 128 + r) * 4);
            }
          }
#pragma unroll
          for (int rk = 1; rk < 8; ++rk) {
            if (rk < p.ks) {
#pragma unroll
              for (int mm = 0; mm < MC; ++mm) acc[m0 + mm] += v[rk - 1][mm];
            }
          }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < p.rows) {
            float v = acc[m];
            if constexpr (VARIANT == kW4A8) v = red_scale[m] * v;
            tile.y[m * N + n] = f32_to_bf16_bits(v);
          }
        }
      }
      cluster_sync_all();
    }
  }
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---- W8A16 ------------------------------------------------------------------
constexpr int kW8Threads = 256;
constexpr int kW8RowsPerWarp = 4;

// One lane's 16 bytes of each of a warp's rows at K offset kc (zeros past N or
// K), so that all the warp's row loads of a slice are in flight together.
__device__ __forceinline__ void load_w8_rows(uint4 (&w)[kW8RowsPerWarp], const int8_t* w8,
                                             int64_t n0, int64_t N, int64_t K, int64_t kc) {
#pragma unroll
  for (int i = 0; i < kW8RowsPerWarp; ++i)
    w[i] = (n0 + i < N && kc < K) ? ldg_stream(w8 + (n0 + i) * K + kc) : make_uint4(0, 0, 0, 0);
}

template <int MT>
__global__ void __launch_bounds__(kW8Threads)
gemv_w8_kernel(const uint16_t* __restrict__ x, const int8_t* __restrict__ w8,
               const uint16_t* __restrict__ s8, int64_t N, int64_t K, int rows,
               uint16_t* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * kW8Threads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kW8Threads) >> 5;
  for (int64_t n0 = gw * kW8RowsPerWarp; n0 < N; n0 += nwarps * kW8RowsPerWarp) {
    float acc[kW8RowsPerWarp][MT];
#pragma unroll
    for (int i = 0; i < kW8RowsPerWarp; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[i][m] = 0.f;
    // the next slice's weights are requested before the current slice is used
    uint4 wcur[kW8RowsPerWarp], wnext[kW8RowsPerWarp];
    load_w8_rows(wcur, w8, n0, N, K, (int64_t)lane * 16);
    for (int64_t kc = (int64_t)lane * 16; kc < K; kc += 512) {
      load_w8_rows(wnext, w8, n0, N, K, kc + 512);
      float xv[MT][16];
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m < rows) {
          const uint4 a = __ldg(reinterpret_cast<const uint4*>(x + m * K + kc));
          const uint4 b = __ldg(reinterpret_cast<const uint4*>(x + m * K + kc + 8));
          const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            xv[m][2 * i] = __uint_as_float(u[i] << 16);
            xv[m][2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) xv[m][i] = 0.f;
        }
      }
#pragma unroll
      for (int i = 0; i < kW8RowsPerWarp; ++i) {
        if (n0 + i < N) {
          const uint4 wv = wcur[i];
          const uint32_t ww[4] = {wv.x ^ 0x80808080u, wv.y ^ 0x80808080u, wv.z ^ 0x80808080u,
                                  wv.w ^ 0x80808080u};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              // 2^23 + (w + 128) as fp32 bits, minus 2^23 + 128: exactly w
              const float wf =
                  __uint_as_float(prmt(ww[q], 0x4B000000u, 0x7650u | b)) - 8388736.0f;
#pragma unroll
              for (int m = 0; m < MT; ++m) acc[i][m] = fmaf(xv[m][4 * q + b], wf, acc[i][m]);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kW8RowsPerWarp; ++i) wcur[i] = wnext[i];
    }
#pragma unroll
    for (int i = 0; i < kW8RowsPerWarp; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[i][m] += __shfl_xor_sync(0xffffffffu, acc[i][m], o);
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < kW8RowsPerWarp; ++i) {
        if (n0 + i >= N) break;
        const float sc = f16_bits_to_f32(s8[n0 + i]);
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < rows) y[m * N + n0 + i] = f32_to_bf16_bits(sc * acc[i][m]);
      }
    }
  }
}

// ---- W8A8 ---------------------------------------------------------------------
// Same warp-per-4-rows walk as W8A16, on int8 activation codes: dp4a products
// summed exactly in int32 (|sum| <= K * 127 * 127 < 2^31 for K < 133144),
// then y = bf16(a_s[m] * s[n] * sum).
template <int MT>
__global__ void __launch_bounds__(kW8Threads)
gemv_w8a8_kernel(const int8_t* __restrict__ a_q, const float* __restrict__ a_s,
                 const int8_t* __restrict__ w8, const uint16_t* __restrict__ s8, int64_t N,
                 int64_t K, int rows, uint16_t* __restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t gw = ((int64_t)blockIdx.x * kW8Threads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kW8Threads) >> 5;
  for (int64_t n0 = gw * kW8RowsPerWarp; n0 < N; n0 += nwarps * kW8RowsPerWarp) {
    int acc[kW8RowsPerWarp][MT];
#pragma unroll
    for (int i = 0; i < kW8RowsPerWarp; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[i][m] = 0;
    // the next slice's weights are requested before the current slice is used
    uint4 wcur[kW8RowsPerWarp], wnext[kW8RowsPerWarp];
    load_w8_rows(wcur, w8, n0, N, K, (int64_t)lane * 16);
    for (int64_t kc = (int64_t)lane * 16; kc < K; kc += 512) {
      load_w8_rows(wnext, w8, n0, N, K, kc + 512);
      uint4 av[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m)
        av[m] = (m < rows) ? __ldg(reinterpret_cast<const uint4*>(a_q + m * K + kc))
                           : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int i = 0; i < kW8RowsPerWarp; ++i) {
        if (n0 + i < N) {
          const uint4 wv = wcur[i];
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            int d = acc[i][m];
            d = __dp4a((int)wv.x, (int)av[m].x, d);
            d = __dp4a((int)wv.y, (int)av[m].y, d);
            d = __dp4a((int)wv.z, (int)av[m].z, d);
            d = __dp4a((int)wv.w, (int)av[m].w, d);
            acc[i][m] = d;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kW8RowsPerWarp; ++i) wcur[i] = wnext[i];
    }
#pragma unroll
    for (int i = 0; i < kW8RowsPerWarp; ++i)
#pragma unroll
      for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc[i][m] += __shfl_xor_sync(0xffffffffu, acc[i][m], o);
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < kW8RowsPerWarp; ++i) {
        if (n0 + i >= N) break;
        const float sc = f16_bits_to_f32(s8[n0 + i]);
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < rows) y[m * N + n0 + i] = f32_to_bf16_bits(a_s[m] * sc * (float)acc[i][m]);
      }
    }
  }
}

// ---- launchers ----------------------------------------------------------------
static int sm_count() {
  const int n = device_sm_count();
  return n > 0 ? n : 148;
}

template <int VARIANT, int MT, bool PARTIALS>
static cudaError_t launch_w4_slice(const GemvParams& p, cudaStream_t st) {
  const int ng_max = (p.G + p.ks - 1) / p.ks;
  const size_t act_bytes = (VARIANT == kW4A8) ? (size_t)ng_max * MT * (16 * 8 + 4)
                                              : (size_t)ng_max * MT * 128 * 4;
  const size_t smem = (size_t)kGemvStages * kGemvStageBytes + 256 + MT * 128 * 4 + act_bytes;
  auto kern = gemv_w4_kernel<VARIANT, MT, PARTIALS>;
  static SmemOptIn opt_in;  // largest carve-out requested so far, per device
  if (cudaError_t e = opt_in.ensure(kern, smem); e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.ks, (unsigned)(p.N / 128), 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int VARIANT, bool PARTIALS>
static cudaError_t launch_w4_rows(const GemvParams& p, cudaStream_t st) {
  if (p.rows == 1) return launch_w4_slice<VARIANT, 1, PARTIALS>(p, st);
  if (p.rows == 2) return launch_w4_slice<VARIANT, 2, PARTIALS>(p, st);
  if (p.rows <= 4 || VARIANT != kW4A8) return launch_w4_slice<VARIANT, 4, PARTIALS>(p, st);
  if (p.rows <= 8) return launch_w4_slice<kW4A8, 8, PARTIALS>(p, st);
  return launch_w4_slice<kW4A8, 16, PARTIALS>(p, st);
}

cudaError_t launch_gemv(const GemmArgs& a, cudaStream_t st) {
  if (a.M == 0) return cudaSuccess;
  if (a.variant == kW8A8) {
    const int64_t warps_needed = (a.N + kW8RowsPerWarp - 1) / kW8RowsPerWarp;
    int64_t blocks = (warps_needed * 32 + kW8Threads - 1) / kW8Threads;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    constexpr int kW8A8MaxRows = 8;  // token rows per W8A8 GEMV launch
    for (int64_t m0 = 0; m0 < a.M; m0 += kW8A8MaxRows) {
      const int rows = (int)((a.M - m0) < kW8A8MaxRows ? (a.M - m0) : kW8A8MaxRows);
      const int8_t* aq = a.a_q + m0 * a.K;
      const float* as = a.a_s + m0;
      uint16_t* y = a.y + m0 * a.N;
      if (rows == 1)
        gemv_w8a8_kernel<1><<<(unsigned)blocks, kW8Threads, 0, st>>>(aq, as, a.w8, a.s8, a.N, a.K, rows, y);
      else if (rows == 2)
        gemv_w8a8_kernel<2><<<(unsigned)blocks, kW8Threads, 0, st>>>(aq, as, a.w8, a.s8, a.N, a.K, rows, y);
      else if (rows <= 4)
        gemv_w8a8_kernel<4><<<(unsigned)blocks, kW8Threads, 0, st>>>(aq, as, a.w8, a.s8, a.N, a.K, rows, y);
      else
        gemv_w8a8_kernel<8><<<(unsigned)blocks, kW8Threads, 0, st>>>(aq, as, a.w8, a.s8, a.N, a.K, rows, y);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  if (a.variant == kW8A16) {
    const int64_t warps_needed = (a.N + kW8RowsPerWarp - 1) / kW8RowsPerWarp;
    int64_t blocks = (warps_needed * 32 + kW8Threads - 1) / kW8Threads;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    constexpr int kW8MaxRows = 4;  // token rows per W8A16 GEMV launch
    for (int64_t m0 = 0; m0 < a.M; m0 += kW8MaxRows) {
      const int rows = (int)((a.M - m0) < kW8MaxRows ? (a.M - m0) : kW8MaxRows);
      const uint16_t* x = a.x + m0 * a.K;
      uint16_t* y = a.y + m0 * a.N;
      if (rows == 1)
        gemv_w8_kernel<1><<<(unsigned)blocks, kW8Threads, 0, st>>>(x, a.w8, a.s8, a.N, a.K, rows, y);
      else if (rows == 2)
        gemv_w8_kernel<2><<<(unsigned)blocks, kW8Threads, 0, st>>>(x, a.w8, a.s8, a.N, a.K, rows, y);
      else
        gemv_w8_kernel<4><<<(unsigned)blocks, kW8Threads, 0, st>>>(x, a.w8, a.s8, a.N, a.K, rows, y);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  const int G = (int)(a.K / 128);
  const int64_t tiles = a.N / 128;
  const SegTable seg = seg_table(a);
  // split the groups of each tile over a cluster so that about two CTAs per
  // SM stream weights, keeping at most kGemvMaxGroupsPerCta groups per CTA
  const int64_t slots = 2LL * sm_count();
  int ks = 1;
  double best = 1e30;
  for (int c = 1; c <= 8 && c <= G; ++c) {
    if ((G + c - 1) / c > kGemvMaxGroupsPerCta) continue;
    const int64_t rounds = (tiles * c + slots - 1) / slots;
    const double cost = (double)rounds * ((G + c - 1) / c) * (c > 1 ? 1.03 : 1.0);
    if (cost < best - 1e-9) {
      best = cost;
      ks = c;
    }
  }
  if ((G + ks - 1) / ks > kGemvMaxGroupsPerCta) return cudaErrorNotSupported;
  // token rows per launch: up to 16 for W4A8 (dp4a), 4 for W4A16 (fp32 FMA)
  const int max_rows = (a.variant == kW4A8) ? kGemvMaxRows : 4;
  for (int64_t m0 = 0; m0 < a.M; m0 += max_rows) {
    GemvParams p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G = G;
    p.ks = ks;
    p.rows = (int)((a.M - m0) < max_rows ? (a.M - m0) : max_rows);
    p.seg = seg;
    for (int j = 0; j < seg.count; ++j) p.seg.y[j] = seg.y[j] + m0 * seg.N[j];
    p.timeout_ns = a.timeout_ns;
    cudaError_t e;
    if (a.variant == kW4A8) {
      p.a_q = a.a_q + m0 * a.K;
      p.a_s = a.a_s + m0;
      p.a_gsum = a.a_gsum + m0 * G;
      if (a.partials) {
        p.partials = a.partials + m0 * a.N * G;
        e = launch_w4_rows<kW4A8, true>(p, st);
      } else {
        e = launch_w4_rows<kW4A8, false>(p, st);
      }
    } else {
      p.x = a.x + m0 * a.K;
      e = launch_w4_rows<kW4A16, false>(p, st);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t take_error_word_gemv(unsigned* out) { return take_local_error_word(out); }
cudaError_t set_record_limit_gemv(unsigned long long bytes) { return set_local_record_limit(bytes); }

}  // namespace egopq
