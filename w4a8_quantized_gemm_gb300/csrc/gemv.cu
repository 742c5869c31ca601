// gemv.cu -- CUDA-core decode kernels for small M (M <= 4 per launch slice).
//
// Decode is a weight-streaming problem: every packed weight byte is read once
// per token batch, so the kernels below are built to keep HBM busy. Each CTA
// (4 warps) owns a 32-row slab of the output and a contiguous range of K
// groups; its warps take every fourth group of that range, so a warp's loads
// are 512 contiguous bytes per 16-byte chunk (32 rows x 16 B). A cluster of
// up to 8 CTAs splits the groups of one slab further and reduces the partial
// sums through distributed shared memory -- no global scratch, fixed
// summation order, deterministic output.
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
// W8A16: int8 row-major weights, one warp per 4 rows, 16-byte coalesced loads
// along K and a warp-shuffle reduction; y = bf16(s[n] * sum_k x*w_q).
#include "egopq_internal.h"

namespace egopq {

constexpr int kGemvThreads = 128;
constexpr int kGemvMaxGroupsPerCta = 64;

struct GemvParams {
  int64_t M, N, K;
  int G, ks, rows;
  const int8_t* a_q;
  const float* a_s;
  const int32_t* a_gsum;
  const uint16_t* x;
  const uint8_t* packed;
  uint16_t* y;
  int32_t* partials;
};

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int VARIANT, int MT, bool PARTIALS>
__global__ void __launch_bounds__(kGemvThreads)
gemv_w4_kernel(const GemvParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ks = blockIdx.x, slab = blockIdx.y;
  const int G = p.G;
  const int g0 = (int)((int64_t)ks * G / p.ks), g1 = (int)((int64_t)(ks + 1) * G / p.ks);
  const int ng = g1 - g0;
  const int64_t N = p.N, K = p.K;
  const int64_t n = (int64_t)slab * 32 + lane;
  const int64_t t = slab >> 2;
  const int r = (slab & 3) * 32 + lane;
  const uint8_t* codes = p.packed;
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(p.packed + N * K / 2);
  const uint8_t* zeros = p.packed + N * K / 2 + 2 * (int64_t)G * N;

  // ---- stage this CTA's activations (permuted to the nibble order) ----------
  // W4A8: per (group, row m, chunk c, word j) a uint2 {lo, hi} of int8 quads;
  // then int32 group sums. W4A16: 128 floats per (group, row), nibble order.
  float* red = reinterpret_cast<float*>(smem);  // [4 warps][MT][32], reused below
  uint8_t* act = smem + 4 * MT * 32 * sizeof(float);
  if constexpr (VARIANT == kW4A8) {
    uint2* aw = reinterpret_cast<uint2*>(act);
    int32_t* as = reinterpret_cast<int32_t*>(act + (size_t)ng * MT * 16 * sizeof(uint2));
    for (int i = threadIdx.x; i < ng * MT * 16; i += kGemvThreads) {
      const int gl = i / (MT * 16), m = (i / 16) % MT, cj = i % 16;
      uint2 v = make_uint2(0, 0);
      if (m < p.rows) {
        const int64_t k0 = (int64_t)(g0 + gl) * 128 + cj * 8;
        const uint2 X = *reinterpret_cast<const uint2*>(p.a_q + m * K + k0);
        v.x = prmt(X.x, X.y, 0x5140);  // K offsets {0,4,1,5}
        v.y = prmt(X.x, X.y, 0x7362);  // K offsets {2,6,3,7}
      }
      aw[i] = v;
    }
    for (int i = threadIdx.x; i < ng * MT; i += kGemvThreads) {
      const int gl = i / MT, m = i % MT;
      as[i] = (m < p.rows) ? p.a_gsum[m * G + g0 + gl] : 0;
    }
  } else {
    float* xs = reinterpret_cast<float*>(act);
    for (int i = threadIdx.x; i < ng * MT * 128; i += kGemvThreads) {
      const int gl = i / (MT * 128), m = (i / 128) % MT, kk = i % 128;
      // position kk = 32c + 8j + nib holds K offset 32c + 8j + e(nib)
      const int nib = kk & 7;
      const int e = (nib < 4) ? 2 * nib : 2 * (nib - 4) + 1;
      float v = 0.f;
      if (m < p.rows)
        v = bf16_bits_to_f32(p.x[m * K + (int64_t)(g0 + gl) * 128 + (kk & ~7) + e]);
      xs[i] = v;
    }
  }
  __syncthreads();

  float acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0.f;

  auto load_tile = [&](int g, uint4 (&w)[4]) {
    const uint8_t* base = codes + ((t * G + g) * 8192) + (int64_t)r * 16;
#pragma unroll
    for (int c = 0; c < 4; ++c) w[c] = ldg_stream(base + c * 2048);
  };

  int g = g0 + warp;
  uint4 cur[4], nxt[4];
  if (g < g1) load_tile(g, cur);
  for (; g < g1; g += 4) {
    const int gn = g + 4;
    if (gn < g1) load_tile(gn, nxt);
    const uint8_t zb = __ldg(zeros + (int64_t)g * (N / 2) + (n >> 1));
    const int z = (n & 1) ? (zb >> 4) : (zb & 0xF);
    const float s = f16_bits_to_f32(__ldg(scales + (int64_t)g * N + n));
    const int gl = g - g0;
    if constexpr (VARIANT == kW4A8) {
      const uint4* aw = reinterpret_cast<const uint4*>(act) + (size_t)gl * MT * 8;
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
        const int q = dot[m] - z * as[gl * MT + m];
        if constexpr (PARTIALS) {
          if (m < p.rows) p.partials[((int64_t)m * N + n) * G + g] = q;
        } else {
          acc[m] = fmaf(s, (float)q, acc[m]);
        }
      }
    } else {
      const float* xs = reinterpret_cast<const float*>(act) + (size_t)gl * MT * 128;
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
            const float4 xb = *reinterpret_cast<const float4*>(xs + m * 128 + c * 32 + j * 8 + 4);
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
      for (int m = 0; m < MT; ++m) acc[m] = fmaf(s, part[m], acc[m]);
    }
    if (gn < g1) {
#pragma unroll
      for (int c = 0; c < 4; ++c) cur[c] = nxt[c];
    }
  }
  if constexpr (!PARTIALS) {
  // ---- reduce: the 4 warps of the CTA, then the CTAs of the cluster --------
#pragma unroll
  for (int m = 0; m < MT; ++m) red[(warp * MT + m) * 32 + lane] = acc[m];
  __syncthreads();
  float* cta_sum = red + 4 * MT * 32;  // [MT][32], inside the staging area
  if (warp == 0) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      float v = red[(0 * MT + m) * 32 + lane];
      v += red[(1 * MT + m) * 32 + lane];
      v += red[(2 * MT + m) * 32 + lane];
      v += red[(3 * MT + m) * 32 + lane];
      acc[m] = v;
    }
  }
  if (p.ks > 1) {
    if (warp == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m) cta_sum[m * 32 + lane] = acc[m];
    }
    cluster_sync_all();
    if (cluster_ctarank() == 0 && warp == 0) {
      const uint32_t local = smem_u32(cta_sum);
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = cta_sum[m * 32 + lane];
      for (int rk = 1; rk < p.ks; ++rk) {
        const uint32_t remote = map_to_rank(local, rk);
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] += ld_dsmem_f32(remote + (m * 32 + lane) * 4);
      }
    }
    cluster_sync_all();
    if (cluster_ctarank() != 0) return;
  }
  if (warp == 0) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < p.rows) {
        float v = acc[m];
        if constexpr (VARIANT == kW4A8) v = p.a_s[m] * v;
        p.y[m * N + n] = f32_to_bf16_bits(v);
      }
    }
  }
  }  // !PARTIALS
}

// ---- W8A16 ------------------------------------------------------------------
constexpr int kW8Threads = 256;
constexpr int kW8RowsPerWarp = 4;

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
    for (int64_t kc = (int64_t)lane * 16; kc < K; kc += 512) {
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
          const uint4 wv = ldg_stream(w8 + (n0 + i) * K + kc);
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

// ---- launchers ----------------------------------------------------------------
static int sm_count() {
  static int count = 0;
  if (!count) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev);
    if (count <= 0) count = 148;
  }
  return count;
}

template <int VARIANT, int MT, bool PARTIALS>
static cudaError_t launch_w4_slice(const GemvParams& p, cudaStream_t st) {
  const int ng_max = (p.G + p.ks - 1) / p.ks;
  size_t act_bytes = (VARIANT == kW4A8) ? (size_t)ng_max * MT * (16 * 8 + 4)
                                        : (size_t)ng_max * MT * 128 * 4;
  size_t smem = 4 * MT * 32 * 4 + act_bytes;
  // the reduction buffers (4*MT*32 + MT*32 floats) must fit in front of and
  // inside the staging area
  const size_t red_need = (4 * MT * 32 + MT * 32) * 4;
  if (smem < red_need) smem = red_need;
  auto kern = gemv_w4_kernel<VARIANT, MT, PARTIALS>;
  static size_t attr_smem = 0;  // largest carve-out requested so far for this instantiation
  if (smem > attr_smem) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    attr_smem = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.ks, (unsigned)(p.N / 32), 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.ks;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int VARIANT, bool PARTIALS>
static cudaError_t launch_w4_rows(const GemvParams& p, cudaStream_t st) {
  if (p.rows == 1) return launch_w4_slice<VARIANT, 1, PARTIALS>(p, st);
  if (p.rows == 2) return launch_w4_slice<VARIANT, 2, PARTIALS>(p, st);
  return launch_w4_slice<VARIANT, 4, PARTIALS>(p, st);
}

cudaError_t launch_gemv(const GemmArgs& a, cudaStream_t st) {
  if (a.M == 0) return cudaSuccess;
  if (a.variant == kW8A16) {
    const int64_t warps_needed = (a.N + kW8RowsPerWarp - 1) / kW8RowsPerWarp;
    int64_t blocks = (warps_needed * 32 + kW8Threads - 1) / kW8Threads;
    const int64_t cap = (int64_t)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    for (int64_t m0 = 0; m0 < a.M; m0 += kGemvMaxRows) {
      const int rows = (int)((a.M - m0) < kGemvMaxRows ? (a.M - m0) : kGemvMaxRows);
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
  const int64_t slabs = a.N / 32;
  // split K across a cluster so the grid covers the GPU a few times over,
  // keeping at least two groups per warp and at most kGemvMaxGroupsPerCta per CTA
  int ks = (int)((4LL * sm_count() + slabs - 1) / slabs);
  const int ks_cap = G / 8 > 0 ? G / 8 : 1;
  if (ks > ks_cap) ks = ks_cap;
  const int ks_min = (G + kGemvMaxGroupsPerCta - 1) / kGemvMaxGroupsPerCta;
  if (ks < ks_min) ks = ks_min;
  if (ks > 8) ks = 8;
  if (ks < 1) ks = 1;
  if ((G + ks - 1) / ks > kGemvMaxGroupsPerCta) return cudaErrorNotSupported;
  for (int64_t m0 = 0; m0 < a.M; m0 += kGemvMaxRows) {
    GemvParams p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.G = G;
    p.ks = ks;
    p.rows = (int)((a.M - m0) < kGemvMaxRows ? (a.M - m0) : kGemvMaxRows);
    p.packed = a.packed;
    p.y = a.y + m0 * a.N;
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

}  // namespace egopq
