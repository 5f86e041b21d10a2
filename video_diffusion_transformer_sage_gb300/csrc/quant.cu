// quant.cu -- HBM-bound kernels of the quantised-attention path: K mean, V column
// absolute maxima, INT8 quantisation of Q and K - mean, FP8 E4M3 quantisation of V.
//
// These are the qk_quantize, v_quantize and k-smoothing stages of the Sage2 attention
// call in "gb10-sampling-component-profile-1344x768-124f-seed440420.json"
// (attention_internal_p50_milliseconds.sage2).  Every kernel reads the bf16 inputs as
// strided [N, H, D] views with 16-byte vector loads: no transposed copy is made (the
// strided-NHD dataflow of "gb10-sage-strided-nhd-summary-...json", dataflow.qkv_input).
//
// Arithmetic contract (shared with nothing; the CPU oracle restates it independently):
//  * K mean: fp32 sum of each 128-token chunk in ascending token order; the chunk sums are
//    split into 8 groups of ceil(chunks / 8) consecutive chunks, each group summed in fp64 in
//    ascending order, the 8 group sums added in fp64 in ascending order; divided by N in
//    fp64, rounded once to fp32.
//  * INT8: scale = fl32(amax / 127), code = clamp(rint(fl32(x / scale)), -127, 127), IEEE
//    division; all-zero block -> scale 0, codes 0.  K uses fl32(k - mean).
//  * E4M3: scale = fl32(amax / 448), code = cvt.rn.satfinite.e4m3(fl32(v / scale)).
// The per-element quotient fl32(x / scale) is formed from one IEEE reciprocal per scale and
// Markstein's FMA correction (div_rn2), which yields the same correctly rounded value.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <type_traits>

#include "qk_row.cuh"
#include "sage_internal.h"
#include "sm103_ptx.cuh"

namespace sage {
namespace {

__device__ __forceinline__ uint4 ld_stream(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void unpack8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// ---------------------------------------------------------------------------- kernel R
// One thread per (chunk of 128 tokens, 8 consecutive columns of one head).  Sum mode adds
// the chunk's tokens in ascending order in fp32; absmax mode keeps max |x|, or with kSubMean
// max |fl32(x - mean[h][c])| (the maxima of smoothed V).  partials[chunk][h*D + c].
template <bool kAbsMax, bool kSubMean = false>
__device__ __forceinline__ void colreduce_block(const uint16_t* __restrict__ x, int64_t st, int64_t sh, int n, int h,
                                                int d, const float* __restrict__ mean, float* __restrict__ partials) {
  const int vpr = d >> 3;  // 16-byte vectors per (token, head) row
  const int g = blockIdx.y * blockDim.x + threadIdx.x;
  if (g >= h * vpr) return;
  const int hh = g / vpr, c8 = g - hh * vpr;
  const int t0 = blockIdx.x * 128;
  const int t1 = min(t0 + 128, n);
  const uint16_t* base = x + hh * sh + c8 * 8;
  float acc[8], mu[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    acc[j] = 0.0f;
    mu[j] = kSubMean ? mean[hh * d + c8 * 8 + j] : 0.0f;
  }
  for (int t = t0; t < t1; t += 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (t + u < t1) v[u] = ld_stream(base + static_cast<int64_t>(t + u) * st);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (t + u < t1) {
        float f[8];
        unpack8(v[u], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (kSubMean) f[j] = __fsub_rn(f[j], mu[j]);
          acc[j] = kAbsMax ? fmaxf(acc[j], fabsf(f[j])) : acc[j] + f[j];
        }
      }
    }
  }
  float4* dst = reinterpret_cast<float4*>(partials + static_cast<int64_t>(blockIdx.x) * h * d + hh * d + c8 * 8);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

template <bool kAbsMax, bool kSubMean = false>
__global__ void __launch_bounds__(128) colreduce_kernel(const uint16_t* __restrict__ x, int64_t st, int64_t sh,
                                                        int n, int h, int d, const float* __restrict__ mean,
                                                        float* __restrict__ partials) {
  colreduce_block<kAbsMax, kSubMean>(x, st, sh, n, h, d, mean, partials);
}

// The K sums (z = 0) and the V maxima (z = 1) of the whole path in one launch.
__global__ void __launch_bounds__(128) colreduce_kv_kernel(const uint16_t* __restrict__ k, int64_t kst, int64_t ksh,
                                                           const uint16_t* __restrict__ v, int64_t vst, int64_t vsh,
                                                           int n, int h, int d, float* __restrict__ part_k,
                                                           float* __restrict__ part_v) {
  if (blockIdx.z == 0)
    colreduce_block<false>(k, kst, ksh, n, h, d, nullptr, part_k);
  else
    colreduce_block<true>(v, vst, vsh, n, h, d, nullptr, part_v);
}

// ---------------------------------------------------------------------------- finalise
// 32 columns per CTA.  The chunk partials are split into 8 groups of G = ceil(nchunk / 8)
// consecutive chunks; warp w folds group w in ascending chunk order (fp64 for sums), then
// warp 0 folds the 8 group results in ascending group order.  Mean = fp32(total / N); in
// absmax mode out = fl32(max / amax_div) (448 for E4M3 scales, 127 for INT8), IEEE division.
template <bool kAbsMax>
__device__ __forceinline__ void colfinal_block(const float* __restrict__ partials, int nchunk, int cols, int n,
                                               float amax_div, float* __restrict__ out) {
  __shared__ double gsum[8][32];
  __shared__ float gmax[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int col = blockIdx.x * 32 + lane;
  const int g = (nchunk + 7) / 8;
  const int c0 = warp * g, c1 = min(nchunk, c0 + g);
  double total = 0.0;
  float amax = 0.0f;
  if (col < cols) {
    for (int c = c0; c < c1; c += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = c + u < c1 ? partials[static_cast<int64_t>(c + u) * cols + col] : 0.0f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c + u < c1) {
          if (kAbsMax)
            amax = fmaxf(amax, v[u]);
          else
            total += static_cast<double>(v[u]);
        }
      }
    }
  }
  gsum[warp][lane] = total;
  gmax[warp][lane] = amax;
  __syncthreads();
  if (warp == 0 && col < cols) {
    double t = 0.0;
    float m = 0.0f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      t += gsum[w][lane];
      m = fmaxf(m, gmax[w][lane]);
    }
    out[col] = kAbsMax ? __fdiv_rn(m, amax_div) : static_cast<float>(t / static_cast<double>(n));
  }
}

template <bool kAbsMax>
__global__ void __launch_bounds__(256) colfinal_kernel(const float* __restrict__ partials, int nchunk, int cols,
                                                       int n, float amax_div, float* __restrict__ out) {
  colfinal_block<kAbsMax>(partials, nchunk, cols, n, amax_div, out);
}

// The K mean (z = 0) and the E4M3 V scales (z = 1) of the whole path in one launch.
__global__ void __launch_bounds__(256) colfinal_kv_kernel(const float* __restrict__ part_k,
                                                          const float* __restrict__ part_v, int nchunk, int cols,
                                                          int n, float* __restrict__ k_mean,
                                                          float* __restrict__ v_scales) {
  grid_dep_wait();   // launched as a dependent of the column pass (small calls)
  grid_dep_launch();
  if (blockIdx.z == 0)
    colfinal_block<false>(part_k, nchunk, cols, n, 0.0f, k_mean);
  else
    colfinal_block<true>(part_v, nchunk, cols, n, 448.0f, v_scales);
}

// ---------------------------------------------------------------------------- transform
// The qk_transform of the NP rows a thread holds (rows row_first + p * RPP, 8 channels each):
// every lane of the block takes part (the row sum is a butterfly over the row's lanes); rows
// past n stay zero (their table index is clamped into range and the result dropped).
template <int D, int NP, int RPP>
__device__ __forceinline__ void transform_rows(uint4 (&v)[NP], const float* gamma, int row_first, int n, int c8,
                                               const RowTransform& tr) {
  float g[8];
  load_gamma8(gamma, c8, g);
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int row = row_first + p * RPP;
    const uint4 y = transform_row8<D>(v[p], min(row, n - 1), c8, g, tr.rope_cos, tr.rope_sin, tr.eps);
    v[p] = row < n ? y : make_uint4(0, 0, 0, 0);
  }
}

// Column sums of the transformed K, per 128-token chunk, in the order of colreduce_kernel's
// sum mode (ascending tokens, fp32): the partials of the mean of the transformed K.  The
// transformed rows themselves (bf16) go to kt, head-major [H][npad][D], so that K is
// transformed once and its quantisation reads them back.
// One CTA per (128-token chunk, 128 columns = 128 / D heads).  Phase 1: the 256 threads
// transform the chunk's rows in parallel, 8 row vectors each (a row's D/8 vectors are
// consecutive lanes, for the row sum's butterfly), store them to kt and to a shared-memory
// tile.  Phase 2: one thread per column adds the chunk's values from the tile in ascending token
// order.  Columns of heads past h are neither stored nor summed.  Capped at 64 registers, 4 CTAs
// per SM (the shared tile's limit): 0.712 ms for the fused call on the video workload, against
// 0.725 at 80 registers and 3 CTAs per SM.
template <int D>
__global__ void __launch_bounds__(256, 4) colsum_transform_kernel(const uint16_t* __restrict__ x, int64_t st, int64_t sh,
                                                               int n, int npad, int h, const RowTransform tr,
                                                               float* __restrict__ partials,
                                                               uint16_t* __restrict__ kt) {
  constexpr int VPR = D / 8;            // 16-byte vectors per row
  constexpr int HG = 128 / D;           // heads per CTA
  __shared__ __align__(16) uint16_t tile[128][128];
  const int t0 = blockIdx.x * 128, t1 = min(t0 + 128, n);
  const int h0 = blockIdx.y * HG;
  const int c16 = threadIdx.x & 15;     // 8-column vector within the CTA's 128 columns
  const int head = h0 + c16 / VPR, c8 = c16 % VPR;
  const bool hv = head < h;
  float gam[8];
  load_gamma8(tr.gamma_k, c8, gam);
  const uint16_t* base = x + static_cast<int64_t>(hv ? head : 0) * sh + c8 * 8;
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = t0 + (threadIdx.x >> 4) + 16 * i;
    v[i] = (hv && t < t1) ? ld_stream(base + static_cast<int64_t>(t) * st) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = (threadIdx.x >> 4) + 16 * i, t = t0 + r;
    // Every lane transforms (the row sum is a butterfly); rows past n are dropped.
    const uint4 y = transform_row8<D>(v[i], min(t, n - 1), c8, gam, tr.rope_cos, tr.rope_sin, tr.eps);
    if (t < t1) {
      if (hv) *reinterpret_cast<uint4*>(kt + (static_cast<int64_t>(head) * npad + t) * D + c8 * 8) = y;
      *reinterpret_cast<uint4*>(&tile[r][c16 * 8]) = y;
    }
  }
  __syncthreads();
  if (threadIdx.x < 128 && h0 + static_cast<int>(threadIdx.x) / D < h) {
    const int c = threadIdx.x;
    float acc = 0.0f;
    for (int r = 0; r < t1 - t0; ++r) acc = acc + __uint_as_float(static_cast<uint32_t>(tile[r][c]) << 16);
    partials[static_cast<int64_t>(blockIdx.x) * h * D + h0 * D + c] = acc;
  }
}

// ---------------------------------------------------------------------------- kernel Q
// Correctly rounded x / s from r = RN(1 / s): y = RN(x r) is within 2 ulp of x / s, the FMA
// gives the exact remainder x - y s, and one FMA correction y + r (x - y s) rounds to
// RN(x / s) (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  Two quotients per call, on the
// packed fp32x2 pipe; `neg_s2` holds -s twice and `r2` holds r twice.
__device__ __forceinline__ uint64_t div_rn2(uint64_t x2, uint64_t neg_s2, uint64_t r2) {
  const uint64_t y2 = f2_mul(x2, r2);
  const uint64_t e2 = f2_fma(y2, neg_s2, x2);
  return f2_fma(e2, r2, y2);
}

// A nonzero scale below the smallest normal float has no finite reciprocal, so the
// reciprocal route of div_rn2 does not apply; it needs a block of values below ~2^-119.
// Kernels test it once per block and take a separate, directly dividing loop for it.
__device__ __forceinline__ bool subnormal_scale(float s) { return s != 0.0f && s < 1.17549435e-38f; }

// Two INT8 codes (held as fp16) of x0, x1 for block scale s (r = RN(1/s)):
// clamp(rint(RN(x / s)), -127, 127), or 0 when s == 0.  kDivide: IEEE division instead of
// the reciprocal route (for a subnormal s).
template <bool kDivide = false>
__device__ __forceinline__ uint32_t i8codes_f16x2(float x0, float x1, float s, uint64_t neg_s2, uint64_t r2) {
  if (s == 0.0f) return 0u;
  float q0, q1;
  if (!kDivide) {
    f2_unpack(div_rn2(f2_pack(x0, x1), neg_s2, r2), q0, q1);
  } else {
    q0 = __fdiv_rn(x0, s);
    q1 = __fdiv_rn(x1, s);
  }
  // rint, then the clamp to [-127, 127] on the fp16 pair: integers up to 2048 convert exactly,
  // anything larger (or infinite) becomes at least 2048 in magnitude and clamps to +-127 as it
  // would in fp32, and a NaN gives -127 in both (max returns the non-NaN operand, as fmaxf).
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(rintf(q1)), "f"(rintf(q0)));
  asm("max.f16x2 %0, %0, %1;" : "+r"(h) : "r"(0xD7F0D7F0u));   // -127, -127
  asm("min.f16x2 %0, %0, %1;" : "+r"(h) : "r"(0x57F057F0u));   // 127, 127
  return h;
}

// Codes and scales of one (head hh, 128-row block b) whose rows the block holds in v (the thread's
// NP rows row0 + p * RPP + rin, 8 channels c8 each; already transformed when the qk_transform
// applies): Q's |x| maximum over the block, or K's |k - mean| maximum per 64-row half; the block
// reduction through red; the codes; the scales.  Pad rows (>= n) are excluded from the maxima and
// written as code 0.  Every thread of the block must call it.
template <int D, int NP, int RPP>
__device__ __forceinline__ void quant_block(uint4 (&v)[NP], bool is_k, const float* __restrict__ k_mean, int hh, int b,
                                            int n, int npad, int c8, int rin, float (&red)[2][8],
                                            uint16_t* __restrict__ q_codes, float* __restrict__ q_scales,
                                            uint16_t* __restrict__ k_codes, float* __restrict__ k_scales) {
  const int row0 = b * 128;
  float mu[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mu[j] = is_k ? k_mean[hh * D + c8 * 8 + j] : 0.0f;

  // Q: |x| max on the bf16 bit patterns (for finite values magnitude order = unsigned order
  // of the bits without the sign).  K: max |k - mean| per 64-row half, over valid rows.
  float am[2] = {0.0f, 0.0f};
  if (!is_k) {
    uint32_t qbits = 0;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      qbits = __vmaxu2(qbits, v[p].x & 0x7FFF7FFFu);
      qbits = __vmaxu2(qbits, v[p].y & 0x7FFF7FFFu);
      qbits = __vmaxu2(qbits, v[p].z & 0x7FFF7FFFu);
      qbits = __vmaxu2(qbits, v[p].w & 0x7FFF7FFFu);
    }
    am[0] = am[1] = fmaxf(__uint_as_float((qbits & 0xFFFFu) << 16), __uint_as_float(qbits & 0xFFFF0000u));
  } else {
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      if (row0 + p * RPP + rin < n) {
        float f[8];
        unpack8(v[p], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) am[p >= NP / 2] = fmaxf(am[p >= NP / 2], fabsf(f[j] - mu[j]));
      }
    }
  }
  float a0 = am[0], a1 = am[1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, o));
    a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, o));
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    red[0][warp] = a0;
    red[1][warp] = a1;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    a0 = fmaxf(a0, red[0][w]);
    a1 = fmaxf(a1, red[1][w]);
  }
  // Q: one scale (a0 == a1); K: one per 64-row half.
  const float s0 = a0 / 127.0f, s1 = a1 / 127.0f;
  const float r0 = 1.0f / s0, r1 = 1.0f / s1;   // IEEE; unused when a scale is 0
  const uint64_t ns02 = f2_pack(-s0, -s0), r02 = f2_pack(r0, r0);
  const uint64_t ns12 = f2_pack(-s1, -s1), r12 = f2_pack(r1, r1);
  uint16_t* dst = is_k ? k_codes : q_codes;
  auto write_codes = [&](auto divide) {
    constexpr bool kDiv = decltype(divide)::value;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const int row = row0 + p * RPP + rin;
      const bool lo = p < NP / 2;
      const float sc = lo ? s0 : s1;
      const uint64_t ns2 = lo ? ns02 : ns12, rr2 = lo ? r02 : r12;
      uint32_t w[4] = {0, 0, 0, 0};
      if (row < n) {
        float f[8];
        unpack8(v[p], f);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          w[j] = i8codes_f16x2<kDiv>(f[2 * j] - mu[2 * j], f[2 * j + 1] - mu[2 * j + 1], sc, ns2, rr2);
      }
      *reinterpret_cast<uint4*>(dst + (static_cast<int64_t>(hh) * npad + row) * D + c8 * 8) =
          make_uint4(w[0], w[1], w[2], w[3]);
    }
  };
  if (!subnormal_scale(s0) && !subnormal_scale(s1))   // uniform over the CTA
    write_codes(std::false_type{});
  else
    write_codes(std::true_type{});
  if (threadIdx.x == 0) {
    if (is_k) {
      k_scales[hh * (npad / 64) + 2 * b] = s0;
      k_scales[hh * (npad / 64) + 2 * b + 1] = s1;
    } else {
      q_scales[hh * (npad / 128) + b] = s0;
    }
  }
}

// One CTA per (head h, 128-row block b, operand): z = 0 quantises the Q block with one
// scale; z = 1 quantises the same rows of K - mean as two 64-row blocks, one scale each.
// only_k: every CTA does K (Q is quantised by another kernel).  Pad rows (>= n) are excluded
// from the maxima and written as code 0.  Each thread issues all its loads before any
// arithmetic; the maxima share one block reduction.
// Capped at 64 registers (4 CTAs per SM): at 70 the lost fourth CTA cost 9 % of its time.
template <int D>
__global__ void __launch_bounds__(256, 4) quant_qk_kernel(const uint16_t* __restrict__ q, int64_t qst, int64_t qsh,
                                                          const uint16_t* __restrict__ k, int64_t kst, int64_t ksh,
                                                          const float* __restrict__ k_mean, int n, int npad,
                                                          int only_k, uint16_t* __restrict__ q_codes,
                                                          float* __restrict__ q_scales, uint16_t* __restrict__ k_codes,
                                                          float* __restrict__ k_scales) {
  constexpr int VPR = D / 8;            // vectors per row
  constexpr int RPP = 256 / VPR;        // rows per pass
  constexpr int NP = 128 / RPP;         // passes per 128-row block
  __shared__ float red[2][8];
  const int hh = blockIdx.x, b = blockIdx.y;   // heads fastest: co-resident CTAs read adjacent columns
  const bool is_k = only_k || blockIdx.z != 0;
  const int c8 = threadIdx.x % VPR, rin = threadIdx.x / VPR;
  const int row0 = b * 128;
  const uint16_t* src = is_k ? k : q;
  const int64_t st = is_k ? kst : qst, sh = is_k ? ksh : qsh;

  uint4 v[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int row = row0 + p * RPP + rin;
    v[p] = row < n ? ld_stream(src + static_cast<int64_t>(row) * st + hh * sh + c8 * 8) : make_uint4(0, 0, 0, 0);
  }
  quant_block<D, NP, RPP>(v, is_k, k_mean, hh, b, n, npad, c8, rin, red, q_codes, q_scales, k_codes, k_scales);
}

// The rows [row0, row0 + 128) of the rotary table (cos and sin of D/2 angles per token, the same
// for every head) into shared memory: tab[r * D/8 + i] holds cos of pairs 4i .. 4i + 3 of token
// row0 + r, tab[128 * D/8 + ...] the sines.  Rows past n are clamped into range (their results
// are dropped).  Every thread of the block must call it; a __syncthreads must follow.
template <int D>
__device__ __forceinline__ void stage_rope_table(float4* tab, int row0, int n, const RowTransform& tr) {
  constexpr int VPR = D / 8;
  for (int i = threadIdx.x; i < 128 * VPR; i += blockDim.x) {
    const int64_t off = static_cast<int64_t>(min(row0 + i / VPR, n - 1)) * (D / 2) + (i % VPR) * 4;
    tab[i] = __ldg(reinterpret_cast<const float4*>(tr.rope_cos + off));
    tab[128 * VPR + i] = __ldg(reinterpret_cast<const float4*>(tr.rope_sin + off));
  }
}

// Heads [h0, h0 + g) of one 128-row block b of Q, with the qk_transform applied to each row as
// it is loaded, the rotary factors taken from the staged table; done in turn: the next head's
// rows are loaded while the current one is transformed and quantised (quant_block).
template <int D>
__device__ __forceinline__ void tab_quant_heads(const uint16_t* __restrict__ src, int64_t st, int64_t sh, int h0,
                                                int g, int h, int b, int n, int npad, const float4* tab,
                                                const RowTransform& tr, float (&red)[2][2][8],
                                                uint16_t* __restrict__ q_codes, float* __restrict__ q_scales) {
  constexpr int VPR = D / 8;            // vectors per row (and float4s of cos or sin per token)
  constexpr int RPP = 256 / VPR;        // rows per pass
  constexpr int NP = 128 / RPP;         // passes per 128-row block
  const int c8 = threadIdx.x % VPR, rin = threadIdx.x / VPR;
  const int row0 = b * 128;
  float gam[8];
  load_gamma8(tr.gamma_q, c8, gam);
  uint4 nxt[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int row = row0 + p * RPP + rin;
    nxt[p] = row < n ? ld_stream(src + static_cast<int64_t>(row) * st + h0 * sh + c8 * 8) : make_uint4(0, 0, 0, 0);
  }
  for (int gi = 0; gi < g && h0 + gi < h; ++gi) {   // uniform over the block
    const int hh = h0 + gi;
    uint4 v[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) v[p] = nxt[p];
    if (gi + 1 < g && hh + 1 < h) {
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        const int row = row0 + p * RPP + rin;
        nxt[p] = row < n ? ld_stream(src + static_cast<int64_t>(row) * st + (hh + 1) * sh + c8 * 8)
                         : make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      const int r = p * RPP + rin;
      float f[8];
      unpack_bf16x8(v[p], f);
      const float ss = row_sumsq<VPR>(f);
      const uint4 y = norm_rotate8<D>(f, ss, tr.eps, gam, tab[r * VPR + c8], tab[128 * VPR + r * VPR + c8]);
      v[p] = row0 + r < n ? y : make_uint4(0, 0, 0, 0);
    }
    quant_block<D, NP, RPP>(v, false, nullptr, hh, b, n, npad, c8, rin, red[gi & 1], q_codes, q_scales, nullptr,
                            nullptr);
  }
}

// The quantisation of Q (one scale per 128 rows) with the qk_transform applied to each row as it
// is loaded, for g heads of one 128-row block per CTA.  The block's rows of the rotary table are
// staged in shared memory once and serve all G heads, instead of being read again from L2 by
// one CTA per head.  Dynamic shared memory: 2 x 128 x D/2 floats.
template <int D>
__global__ void __launch_bounds__(256, 2) quant_q_tab_kernel(const uint16_t* __restrict__ q, int64_t qst, int64_t qsh,
                                                            int n, int h, int g, int npad, uint16_t* __restrict__ q_codes,
                                                            float* __restrict__ q_scales, const RowTransform tr) {
  extern __shared__ float4 tab[];
  __shared__ float red[2][2][8];        // by head parity: a head's reduction never meets the next one's
  stage_rope_table<D>(tab, blockIdx.y * 128, n, tr);
  __syncthreads();
  tab_quant_heads<D>(q, qst, qsh, blockIdx.x * g, g, h, blockIdx.y, n, npad, tab, tr, red, q_codes, q_scales);
}

// One CTA per (head h, 128-row block b) of Q when one scale covers q_block < 128 rows
// (q_block a power of two).  The |q| maximum of each row is taken over the VPR threads that
// hold it (on bf16 bit patterns, as above), then over each group of q_block rows: shuffles
// within a warp (thread t < 128 holds row t), shared memory across warps for 64-row groups.
// Pad rows count as 0, so a group wholly in the padding gets scale 0 and codes 0.
template <int D, bool kTransform>
__global__ void __launch_bounds__(256) quant_q_grouped_kernel(const uint16_t* __restrict__ q, int64_t qst,
                                                              int64_t qsh, int n, int npad, int q_block,
                                                              uint16_t* __restrict__ q_codes,
                                                              float* __restrict__ q_scales, const RowTransform tr) {
  constexpr int VPR = D / 8;            // vectors per row
  constexpr int RPP = 256 / VPR;        // rows per pass
  constexpr int NP = 128 / RPP;         // passes per 128-row block
  __shared__ float rmax[128];
  __shared__ float wmax[4];
  const int hh = blockIdx.x, b = blockIdx.y;
  const int c8 = threadIdx.x % VPR, rin = threadIdx.x / VPR;
  const int row0 = b * 128;

  uint4 v[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int row = row0 + p * RPP + rin;
    v[p] = row < n ? ld_stream(q + static_cast<int64_t>(row) * qst + hh * qsh + c8 * 8) : make_uint4(0, 0, 0, 0);
  }
  if (kTransform) transform_rows<D, NP, RPP>(v, tr.gamma_q, row0 + rin, n, c8, tr);
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    uint32_t bits = __vmaxu2(__vmaxu2(v[p].x & 0x7FFF7FFFu, v[p].y & 0x7FFF7FFFu),
                             __vmaxu2(v[p].z & 0x7FFF7FFFu, v[p].w & 0x7FFF7FFFu));
    float a = fmaxf(__uint_as_float((bits & 0xFFFFu) << 16), __uint_as_float(bits & 0xFFFF0000u));
#pragma unroll
    for (int o = VPR / 2; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    if (c8 == 0) rmax[p * RPP + rin] = a;
  }
  __syncthreads();
  float g = 0.0f;
  if (threadIdx.x < 128) {                 // warps 0-3, whole warps
    g = rmax[threadIdx.x];
    const int span = q_block < 32 ? q_block : 32;
    for (int o = 1; o < span; o <<= 1) g = fmaxf(g, __shfl_xor_sync(0xffffffffu, g, o));
    if (q_block > 32 && (threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = g;
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    if (q_block > 32) {
      const int wpg = q_block / 32, w0 = (threadIdx.x >> 5) / wpg * wpg;
      g = wmax[w0];
      for (int i = 1; i < wpg; ++i) g = fmaxf(g, wmax[w0 + i]);
    }
    rmax[threadIdx.x] = g;                 // now the maximum of row threadIdx.x's group
    if ((threadIdx.x & (q_block - 1)) == 0)
      q_scales[static_cast<int64_t>(hh) * (npad / q_block) + (row0 + threadIdx.x) / q_block] = g / 127.0f;
  }
  __syncthreads();
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int row = row0 + p * RPP + rin;
    const float sc = rmax[p * RPP + rin] / 127.0f;
    const float rr = 1.0f / sc;            // IEEE; unused when the scale is 0
    const uint64_t ns2 = f2_pack(-sc, -sc), rr2 = f2_pack(rr, rr);
    uint32_t w[4] = {0, 0, 0, 0};
    if (row < n) {
      float f[8];
      unpack8(v[p], f);
      if (!subnormal_scale(sc)) {
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = i8codes_f16x2(f[2 * j], f[2 * j + 1], sc, ns2, rr2);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = i8codes_f16x2<true>(f[2 * j], f[2 * j + 1], sc, ns2, rr2);
      }
    }
    *reinterpret_cast<uint4*>(q_codes + (static_cast<int64_t>(hh) * npad + row) * D + c8 * 8) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// ---------------------------------------------------------------------------- kernel V
// One CTA per (head, 128-token block).  Phase 1: each work item loads 4 tokens x 8 channels,
// encodes them and stores, per channel, the codes of its 4 consecutive tokens into a
// [D][kWords + 1]-word shared tile (kWords words hold a channel's 128 codes).  Phase 2: each
// channel's 128 contiguous codes of v_codes[h][c][block] leave with 16-byte stores.
//   kI8 = false: E4M3 bytes, scale = max / 448.  kI8 = true: INT8 codes held as fp16 (the INT8
//   P.V variant), scale = max / 127, code = clamp(rint(x / scale), -127, 127).
//   kMean: the codes of x = fl32(v - v_mean[h][c]) (V smoothing); otherwise x = v.
// The codes of a channel with a subnormal scale (no finite reciprocal) come out wrong here and
// are rewritten by quant_v_fixup_kernel, so the loop below stays free of that case.
// Capped at 64 registers (4 CTAs per SM; 75 uncapped gave 3): 144 us instead of 159 at the
// video shape (0.81 GB read and written).
template <int D, bool kI8, bool kMean>
__global__ void __launch_bounds__(256, 4) quant_v_kernel(const uint16_t* __restrict__ v, int64_t st, int64_t sh,
                                                      const float* __restrict__ v_scales,
                                                      const float* __restrict__ v_mean, int n, int npad,
                                                      void* __restrict__ v_codes) {
  constexpr int VPR = D / 8;
  constexpr int kWords = kI8 ? 64 : 32;
  __shared__ uint32_t tile[D][kWords + 1];
  const int hh = blockIdx.x, b = blockIdx.y;   // heads fastest: co-resident CTAs read adjacent columns
  const int t_base = b * 128;
  constexpr int kItems = VPR * 32 / 256;   // work items per thread: 2 at D = 128, 1 at D = 64
  uint4 raw[kItems][4];
#pragma unroll
  for (int i = 0; i < kItems; ++i) {
    const int it = threadIdx.x + i * 256;
    const int c8 = it % VPR, tg = it / VPR;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t_base + tg * 4 + u;
      raw[i][u] = t < n ? ld_stream(v + static_cast<int64_t>(t) * st + hh * sh + c8 * 8) : make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int i = 0; i < kItems; ++i) {
    const int it = threadIdx.x + i * 256;
    const int c8 = it % VPR, tg = it / VPR;
    uint64_t ns2[4], r2[4];
    bool zero[8];
    float mu[8];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float s0 = v_scales[hh * D + c8 * 8 + j], s1 = v_scales[hh * D + c8 * 8 + j + 1];
      zero[j] = s0 == 0.0f;
      zero[j + 1] = s1 == 0.0f;
      ns2[j / 2] = f2_pack(-s0, -s1);
      r2[j / 2] = f2_pack(1.0f / s0, 1.0f / s1);   // IEEE; unused when the scale is 0
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) mu[j] = kMean ? v_mean[hh * D + c8 * 8 + j] : 0.0f;
    uint32_t bytes[4][8];   // E4M3 codes
    float cq[4][8];         // INT8 codes
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t_base + tg * 4 + u;
      float f[8];
      unpack8(raw[i][u], f);
      if (kMean) {
#pragma unroll
        for (int j = 0; j < 8; ++j) f[j] = __fsub_rn(f[j], mu[j]);
      }
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        float y0, y1;
        f2_unpack(div_rn2(f2_pack(f[j], f[j + 1]), ns2[j / 2], r2[j / 2]), y0, y1);
        // The correction step turns x = -0 into +0 (-0 + +0); a positive divisor keeps the sign
        // of x, and E4M3 has a signed zero (0x80), so take the sign from x.
        y0 = copysignf(y0, f[j]);
        y1 = copysignf(y1, f[j + 1]);
        if (t >= n || zero[j]) y0 = 0.0f;
        if (t >= n || zero[j + 1]) y1 = 0.0f;
        if (kI8) {
          cq[u][j] = fminf(fmaxf(rintf(y0), -127.0f), 127.0f);
          cq[u][j + 1] = fminf(fmaxf(rintf(y1), -127.0f), 127.0f);
        } else {
          const uint32_t pr = e4m3x2(y0, y1);
          bytes[u][j] = pr & 0xFFu;
          bytes[u][j + 1] = pr >> 8;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (kI8) {
        uint32_t w0, w1;   // integers |c| <= 127: exact in fp16; the earlier token in the low half
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w0) : "f"(cq[1][j]), "f"(cq[0][j]));
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(w1) : "f"(cq[3][j]), "f"(cq[2][j]));
        tile[c8 * 8 + j][tg * 2] = w0;
        tile[c8 * 8 + j][tg * 2 + 1] = w1;
      } else {
        tile[c8 * 8 + j][tg] = bytes[0][j] | (bytes[1][j] << 8) | (bytes[2][j] << 16) | (bytes[3][j] << 24);
      }
    }
  }
  __syncthreads();
  constexpr int kSegs = kWords / 4;   // 16-byte segments per channel
  for (int o = threadIdx.x; o < D * kSegs; o += 256) {
    const int c = o / kSegs, seg = o % kSegs;
    const uint4 w = make_uint4(tile[c][seg * 4], tile[c][seg * 4 + 1], tile[c][seg * 4 + 2], tile[c][seg * 4 + 3]);
    const int64_t row = (static_cast<int64_t>(hh) * D + c) * npad + t_base;
    if (kI8)
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(v_codes) + row + seg * 8) = w;
    else
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(v_codes) + row + seg * 16) = w;
  }
}

// One CTA per head: if a channel of the head has a subnormal scale (all |x| of the channel
// below ~2^-117), its codes are recomputed with IEEE division; otherwise the CTA exits at once.
template <int D, bool kI8, bool kMean>
__global__ void __launch_bounds__(256) quant_v_fixup_kernel(const uint16_t* __restrict__ v, int64_t st, int64_t sh,
                                                            const float* __restrict__ v_scales,
                                                            const float* __restrict__ v_mean, int n, int npad,
                                                            void* __restrict__ v_codes) {
  grid_dep_wait();   // launched as a dependent of quant_v (small calls)
  grid_dep_launch();
  const int hh = blockIdx.x;
  bool sub = false;
  for (int c = threadIdx.x; c < D; c += 256) sub = sub || subnormal_scale(v_scales[hh * D + c]);
  if (!__syncthreads_or(sub)) return;
  for (int c = 0; c < D; ++c) {
    const float sc = v_scales[hh * D + c];
    if (!subnormal_scale(sc)) continue;
    const float mu = kMean ? v_mean[hh * D + c] : 0.0f;
    for (int t = threadIdx.x; t < n; t += 256) {
      float x = __uint_as_float(static_cast<uint32_t>(v[static_cast<int64_t>(t) * st + hh * sh + c]) << 16);
      if (kMean) x = __fsub_rn(x, mu);
      const float q = __fdiv_rn(x, sc);
      const int64_t idx = (static_cast<int64_t>(hh) * D + c) * npad + t;
      if (kI8)
        static_cast<uint16_t*>(v_codes)[idx] = __half_as_ushort(__float2half_rn(fminf(fmaxf(rintf(q), -127.0f), 127.0f)));
      else
        static_cast<uint8_t*>(v_codes)[idx] = static_cast<uint8_t>(e4m3x2(q, 0.0f) & 0xFFu);
    }
  }
}

template <int D, bool kI8, bool kMean>
cudaError_t launch_quant_v_t(const StridedView& v, const float* v_scales, const float* v_mean, int n, int h,
                             void* v_codes, cudaStream_t s) {
  const int npad = static_cast<int>(pad128(n));
  quant_v_kernel<D, kI8, kMean><<<dim3(h, npad / 128), 256, 0, s>>>(v.data, v.st, v.sh, v_scales, v_mean, n, npad,
                                                                     v_codes);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // The fix-up (one CTA per head, nearly always exiting at once) launches as a dependent of
  // quant_v in small calls, which hides its launch.
  return launch_dependent(dependent_launches(n, h, D), quant_v_fixup_kernel<D, kI8, kMean>, dim3(h), dim3(256), 0, s,
                          v.data, v.st, v.sh, v_scales, v_mean, n, npad, v_codes);
}

template <int D>
cudaError_t launch_quant_v_d(const StridedView& v, const float* v_scales, const float* v_mean, int v_format, int n,
                             int h, void* v_codes, cudaStream_t s) {
  if (v_format == 1)
    return v_mean ? launch_quant_v_t<D, true, true>(v, v_scales, v_mean, n, h, v_codes, s)
                  : launch_quant_v_t<D, true, false>(v, v_scales, v_mean, n, h, v_codes, s);
  return v_mean ? launch_quant_v_t<D, false, true>(v, v_scales, v_mean, n, h, v_codes, s)
                : launch_quant_v_t<D, false, false>(v, v_scales, v_mean, n, h, v_codes, s);
}

}  // namespace

cudaError_t launch_colreduce(const StridedView& x, int n, int h, int d, bool absmax, const float* mean,
                             float* partials, cudaStream_t s) {
  const int nchunk = (n + 127) / 128;
  const int groups = h * (d / 8);
  dim3 grid(nchunk, (groups + 127) / 128);
  if (absmax && mean)
    colreduce_kernel<true, true><<<grid, 128, 0, s>>>(x.data, x.st, x.sh, n, h, d, mean, partials);
  else if (absmax)
    colreduce_kernel<true><<<grid, 128, 0, s>>>(x.data, x.st, x.sh, n, h, d, nullptr, partials);
  else
    colreduce_kernel<false><<<grid, 128, 0, s>>>(x.data, x.st, x.sh, n, h, d, nullptr, partials);
  return cudaGetLastError();
}

cudaError_t launch_colreduce_kv(const StridedView& k, const StridedView& v, int n, int h, int d, float* part_k,
                               float* part_v, cudaStream_t s) {
  const int nchunk = (n + 127) / 128;
  const int groups = h * (d / 8);
  colreduce_kv_kernel<<<dim3(nchunk, (groups + 127) / 128, 2), 128, 0, s>>>(k.data, k.st, k.sh, v.data, v.st, v.sh,
                                                                           n, h, d, part_k, part_v);
  return cudaGetLastError();
}

cudaError_t launch_colfinal_kv(const float* part_k, const float* part_v, int nchunk, int cols, int n, float* k_mean,
                               float* v_scales, cudaStream_t s) {
  // A dependent of the column pass in small calls, which hides its launch.
  return launch_dependent(dependent_launches(n, 1, cols), colfinal_kv_kernel, dim3((cols + 31) / 32, 1, 2), dim3(256), 0,
                          s, part_k, part_v, nchunk, cols, n, k_mean, v_scales);
}

cudaError_t launch_colfinal(const float* partials, int nchunk, int cols, int n, float amax_div, float* out,
                            cudaStream_t s) {
  dim3 grid((cols + 31) / 32);
  if (amax_div != 0.0f)
    colfinal_kernel<true><<<grid, 256, 0, s>>>(partials, nchunk, cols, n, amax_div, out);
  else
    colfinal_kernel<false><<<grid, 256, 0, s>>>(partials, nchunk, cols, n, 0.0f, out);
  return cudaGetLastError();
}

namespace {

// Heads per CTA of quant_q_tab_kernel.  Two CTAs fit on an SM (its shared-memory table), and a
// CTA's time is about (heads + 1) head-steps (the +1: staging the table), so the call takes
// about ceil(CTAs / (2 SMs)) x (g + 1) head-steps; g minimises that, the larger g on a tie.  At
// the video shape (296 row blocks, 56 heads) it picks 56 (one wave); the fused call took 0.752
// ms at 8 heads per CTA, 0.745 at 14, 0.741 at 28 and 0.740 at 56.  At N = 8192 (64 row blocks)
// a fixed 28 left 128 CTAs for 152 SMs, and 12 made 320 CTAs, one wave and a 16-CTA tail.
int tab_heads_per_cta(int h, int blocks) {
  static std::atomic<int> sms_of[64];   // SM count per device, looked up once
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int sms = sms_of[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 152;
    sms_of[dev].store(sms, std::memory_order_relaxed);
  }
  const int64_t slots = 2 * static_cast<int64_t>(sms);
  int best = h;
  int64_t best_cost = -1;
  for (int g = h; g >= 1; --g) {
    const int64_t ctas = static_cast<int64_t>(blocks) * ((h + g - 1) / g);
    const int64_t cost = (ctas + slots - 1) / slots * (g + 1);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = g;
    }
  }
  return best;
}

template <int D>
cudaError_t launch_quant_qk_t(const StridedView& q, const StridedView& k, const float* k_mean, int n, int h,
                              int q_block, uint16_t* q_codes, float* q_scales, uint16_t* k_codes, float* k_scales,
                              cudaStream_t s) {
  const int npad = static_cast<int>(pad128(n));
  const int only_k = q_block != 128;
  quant_qk_kernel<D><<<dim3(h, npad / 128, only_k ? 1 : 2), 256, 0, s>>>(
      q.data, q.st, q.sh, k.data, k.st, k.sh, k_mean, n, npad, only_k, q_codes, q_scales, k_codes, k_scales);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !only_k) return e;
  quant_q_grouped_kernel<D, false><<<dim3(h, npad / 128), 256, 0, s>>>(q.data, q.st, q.sh, n, npad, q_block, q_codes,
                                                                       q_scales, RowTransform{});
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_quant_k_t(const StridedView& k, const float* k_mean, int n, int h, uint16_t* k_codes,
                             float* k_scales, cudaStream_t s) {
  const int npad = static_cast<int>(pad128(n));
  quant_qk_kernel<D><<<dim3(h, npad / 128, 1), 256, 0, s>>>(k.data, k.st, k.sh, k.data, k.st, k.sh, k_mean, n, npad,
                                                            1, nullptr, nullptr, k_codes, k_scales);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_quant_q_transform_t(const StridedView& q, int n, int h, int q_block, uint16_t* q_codes,
                                       float* q_scales, const RowTransform& tr, cudaStream_t s) {
  const int npad = static_cast<int>(pad128(n));
  if (q_block == 128) {
    constexpr int kTab = 2 * 128 * (D / 2) * 4;
    // The dynamic shared-memory limit is a per-device attribute of the function: set it on every
    // call (a host-side call, no device synchronisation).
    cudaError_t e = cudaFuncSetAttribute(quant_q_tab_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTab);
    if (e != cudaSuccess) return e;
    const int g = tab_heads_per_cta(h, npad / 128);
    quant_q_tab_kernel<D><<<dim3((h + g - 1) / g, npad / 128), 256, kTab, s>>>(q.data, q.st, q.sh, n, h, g, npad,
                                                                              q_codes, q_scales, tr);
  } else {
    quant_q_grouped_kernel<D, true><<<dim3(h, npad / 128), 256, 0, s>>>(q.data, q.st, q.sh, n, npad, q_block, q_codes,
                                                                        q_scales, tr);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_qk(const StridedView& q, const StridedView& k, const float* k_mean, int n, int h, int d,
                            int q_block, uint16_t* q_codes, float* q_scales, uint16_t* k_codes, float* k_scales,
                            cudaStream_t s) {
  if (d == 128)
    return launch_quant_qk_t<128>(q, k, k_mean, n, h, q_block, q_codes, q_scales, k_codes, k_scales, s);
  return launch_quant_qk_t<64>(q, k, k_mean, n, h, q_block, q_codes, q_scales, k_codes, k_scales, s);
}

cudaError_t launch_quant_k(const StridedView& k, const float* k_mean, int n, int h, int d, uint16_t* k_codes,
                           float* k_scales, cudaStream_t s) {
  if (d == 128) return launch_quant_k_t<128>(k, k_mean, n, h, k_codes, k_scales, s);
  return launch_quant_k_t<64>(k, k_mean, n, h, k_codes, k_scales, s);
}

cudaError_t launch_quant_q_transform(const StridedView& q, int n, int h, int d, int q_block, uint16_t* q_codes,
                                     float* q_scales, const RowTransform& tr, cudaStream_t s) {
  if (d == 128) return launch_quant_q_transform_t<128>(q, n, h, q_block, q_codes, q_scales, tr, s);
  return launch_quant_q_transform_t<64>(q, n, h, q_block, q_codes, q_scales, tr, s);
}

cudaError_t launch_colsum_transform(const StridedView& k, int n, int h, int d, const RowTransform& tr,
                                    float* partials, uint16_t* kt, cudaStream_t s) {
  const int nchunk = (n + 127) / 128;
  const int npad = static_cast<int>(pad128(n));
  const dim3 grid(nchunk, (h * d + 127) / 128);
  if (d == 128)
    colsum_transform_kernel<128><<<grid, 256, 0, s>>>(k.data, k.st, k.sh, n, npad, h, tr, partials, kt);
  else
    colsum_transform_kernel<64><<<grid, 256, 0, s>>>(k.data, k.st, k.sh, n, npad, h, tr, partials, kt);
  return cudaGetLastError();
}

cudaError_t launch_quant_v(const StridedView& v, const float* v_scales, const float* v_mean, int v_format, int n,
                           int h, int d, void* v_codes, cudaStream_t s) {
  return d == 128 ? launch_quant_v_d<128>(v, v_scales, v_mean, v_format, n, h, v_codes, s)
                  : launch_quant_v_d<64>(v, v_scales, v_mean, v_format, n, h, v_codes, s);
}

}  // namespace sage
