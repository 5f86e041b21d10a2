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
//  * K mean: fp32 sum of each 128-token chunk in ascending token order, chunk sums added in
//    fp64 in ascending chunk order, divided by N in fp64, rounded once to fp32.
//  * INT8: scale = fl32(amax / 127), code = clamp(rint(fl32(x / scale)), -127, 127), IEEE
//    division; all-zero block -> scale 0, codes 0.  K uses fl32(k - mean).
//  * E4M3: scale = fl32(amax / 448), code = cvt.rn.satfinite.e4m3(fl32(v / scale)).
// The per-element quotient fl32(x / scale) is formed from one IEEE reciprocal per scale and
// Markstein's FMA correction (div_rn2), which yields the same correctly rounded value.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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
// the chunk's tokens in ascending order in fp32; absmax mode keeps max |x|.
// partials[chunk][h*D + c].
template <bool kAbsMax>
__global__ void __launch_bounds__(128) colreduce_kernel(const uint16_t* __restrict__ x, int64_t st, int64_t sh,
                                                        int n, int h, int d, float* __restrict__ partials) {
  const int vpr = d >> 3;  // 16-byte vectors per (token, head) row
  const int g = blockIdx.y * blockDim.x + threadIdx.x;
  if (g >= h * vpr) return;
  const int hh = g / vpr, c8 = g - hh * vpr;
  const int t0 = blockIdx.x * 128;
  const int t1 = min(t0 + 128, n);
  const uint16_t* base = x + hh * sh + c8 * 8;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
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
        for (int j = 0; j < 8; ++j) acc[j] = kAbsMax ? fmaxf(acc[j], fabsf(f[j])) : acc[j] + f[j];
      }
    }
  }
  float4* dst = reinterpret_cast<float4*>(partials + static_cast<int64_t>(blockIdx.x) * h * d + hh * d + c8 * 8);
  dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// ---------------------------------------------------------------------------- finalise
// 32 columns per CTA: 8 warps stage chunk partials in shared memory (coalesced), then
// warp 0 folds them per column in ascending chunk order.
template <bool kAbsMax>
__global__ void __launch_bounds__(256) colfinal_kernel(const float* __restrict__ partials, int nchunk, int cols,
                                                       int n, float* __restrict__ out) {
  constexpr int kBatch = 128;
  __shared__ float stage[kBatch][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int col = blockIdx.x * 32 + lane;
  double total = 0.0;
  float amax = 0.0f;
  for (int c0 = 0; c0 < nchunk; c0 += kBatch) {
    const int cb = min(kBatch, nchunk - c0);
    for (int c = warp; c < cb; c += 8)
      stage[c][lane] = col < cols ? partials[static_cast<int64_t>(c0 + c) * cols + col] : 0.0f;
    __syncthreads();
    if (warp == 0) {
      for (int c = 0; c < cb; ++c) {
        if (kAbsMax)
          amax = fmaxf(amax, stage[c][lane]);
        else
          total += static_cast<double>(stage[c][lane]);
      }
    }
    __syncthreads();
  }
  if (warp == 0 && col < cols) out[col] = kAbsMax ? amax / 448.0f : static_cast<float>(total / static_cast<double>(n));
}

// ---------------------------------------------------------------------------- kernel Q
template <int kThreads>
__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
  __syncthreads();
  return r;
}

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

// Two INT8 codes (held as fp16) of x0, x1 for block scale s (r = RN(1/s)):
// clamp(rint(RN(x / s)), -127, 127), or 0 when s == 0.
__device__ __forceinline__ uint32_t i8codes_f16x2(float x0, float x1, float s, uint64_t neg_s2, uint64_t r2) {
  if (s == 0.0f) return 0u;
  float q0, q1;
  f2_unpack(div_rn2(f2_pack(x0, x1), neg_s2, r2), q0, q1);
  q0 = fminf(fmaxf(rintf(q0), -127.0f), 127.0f);
  q1 = fminf(fmaxf(rintf(q1), -127.0f), 127.0f);
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(q1), "f"(q0));   // integers |q| <= 127: exact
  return h;
}

// One CTA per (128-row block b, head h): Q block -> one scale; the same rows of K - mean ->
// two 64-row blocks, one scale each.  Pad rows (>= n) are excluded from the maxima and
// written as code 0.  All Q and K loads of the block are issued before any arithmetic so
// that 32 KB per CTA are in flight; the three maxima share one block reduction.
template <int D>
__global__ void __launch_bounds__(256) quant_qk_kernel(const uint16_t* __restrict__ q, int64_t qst, int64_t qsh,
                                                       const uint16_t* __restrict__ k, int64_t kst, int64_t ksh,
                                                       const float* __restrict__ k_mean, int n, int npad,
                                                       uint16_t* __restrict__ q_codes, float* __restrict__ q_scales,
                                                       uint16_t* __restrict__ k_codes,
                                                       float* __restrict__ k_scales) {
  constexpr int VPR = D / 8;            // vectors per row
  constexpr int RPP = 256 / VPR;        // rows per pass
  constexpr int NP = 128 / RPP;         // passes per 128-row block
  __shared__ float red[3][8];
  const int hh = blockIdx.x, b = blockIdx.y;   // heads fastest: co-resident CTAs read adjacent columns
  const int c8 = threadIdx.x % VPR, rin = threadIdx.x / VPR;
  const int row0 = b * 128;

  uint4 vq[NP], vk[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int row = row0 + p * RPP + rin;
    vq[p] = row < n ? ld_stream(q + static_cast<int64_t>(row) * qst + hh * qsh + c8 * 8) : make_uint4(0, 0, 0, 0);
    vk[p] = row < n ? ld_stream(k + static_cast<int64_t>(row) * kst + hh * ksh + c8 * 8) : make_uint4(0, 0, 0, 0);
  }
  float mu[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mu[j] = k_mean[hh * D + c8 * 8 + j];

  // |q| max on the bf16 bit patterns: for finite values, magnitude order = unsigned order
  // of the bits without the sign.
  uint32_t qbits = 0;
  float am[2] = {0.0f, 0.0f};
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    qbits = __vmaxu2(qbits, vq[p].x & 0x7FFF7FFFu);
    qbits = __vmaxu2(qbits, vq[p].y & 0x7FFF7FFFu);
    qbits = __vmaxu2(qbits, vq[p].z & 0x7FFF7FFFu);
    qbits = __vmaxu2(qbits, vq[p].w & 0x7FFF7FFFu);
    const int row = row0 + p * RPP + rin;
    if (row < n) {
      float f[8];
      unpack8(vk[p], f);
#pragma unroll
      for (int j = 0; j < 8; ++j) am[p >= NP / 2] = fmaxf(am[p >= NP / 2], fabsf(f[j] - mu[j]));
    }
  }
  float aq = fmaxf(__uint_as_float((qbits & 0xFFFFu) << 16), __uint_as_float(qbits & 0xFFFF0000u));
  float a0 = am[0], a1 = am[1];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    aq = fmaxf(aq, __shfl_xor_sync(0xffffffffu, aq, o));
    a0 = fmaxf(a0, __shfl_xor_sync(0xffffffffu, a0, o));
    a1 = fmaxf(a1, __shfl_xor_sync(0xffffffffu, a1, o));
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    red[0][warp] = aq;
    red[1][warp] = a0;
    red[2][warp] = a1;
  }
  __syncthreads();
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    aq = fmaxf(aq, red[0][w]);
    a0 = fmaxf(a0, red[1][w]);
    a1 = fmaxf(a1, red[2][w]);
  }
  const float qs = aq / 127.0f, ks0 = a0 / 127.0f, ks1 = a1 / 127.0f;
  const float rq = 1.0f / qs, rk0 = 1.0f / ks0, rk1 = 1.0f / ks1;   // IEEE; unused when a scale is 0
  const uint64_t nq2 = f2_pack(-qs, -qs), rq2 = f2_pack(rq, rq);
  const uint64_t nk02 = f2_pack(-ks0, -ks0), rk02 = f2_pack(rk0, rk0);
  const uint64_t nk12 = f2_pack(-ks1, -ks1), rk12 = f2_pack(rk1, rk1);
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    const int row = row0 + p * RPP + rin;
    float f[8];
    unpack8(vq[p], f);
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = i8codes_f16x2(f[2 * j], f[2 * j + 1], qs, nq2, rq2);
    *reinterpret_cast<uint4*>(q_codes + (static_cast<int64_t>(hh) * npad + row) * D + c8 * 8) =
        make_uint4(w[0], w[1], w[2], w[3]);
    const bool lo = p < NP / 2;
    const float ks = lo ? ks0 : ks1;
    const uint64_t nk2 = lo ? nk02 : nk12, rk2 = lo ? rk02 : rk12;
    uint32_t u[4] = {0, 0, 0, 0};
    if (row < n) {
      unpack8(vk[p], f);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        u[j] = i8codes_f16x2(f[2 * j] - mu[2 * j], f[2 * j + 1] - mu[2 * j + 1], ks, nk2, rk2);
    }
    *reinterpret_cast<uint4*>(k_codes + (static_cast<int64_t>(hh) * npad + row) * D + c8 * 8) =
        make_uint4(u[0], u[1], u[2], u[3]);
  }
  if (threadIdx.x == 0) {
    q_scales[hh * (npad / 128) + b] = qs;
    k_scales[hh * (npad / 64) + 2 * b] = ks0;
    k_scales[hh * (npad / 64) + 2 * b + 1] = ks1;
  }
}

// ---------------------------------------------------------------------------- kernel V
// One CTA per (128-token block, head).  Phase 1: each work item loads 4 tokens x 8 channels,
// encodes them and stores, per channel, one 32-bit word of 4 consecutive tokens into a
// [D][33]-word shared tile.  Phase 2: 8 threads write each channel's 128 contiguous bytes
// of v_codes[h][c][block] with 16-byte stores.
template <int D>
__global__ void __launch_bounds__(256) quant_v_kernel(const uint16_t* __restrict__ v, int64_t st, int64_t sh,
                                                      const float* __restrict__ v_scales, int n, int npad,
                                                      uint8_t* __restrict__ v_codes) {
  constexpr int VPR = D / 8;
  __shared__ uint32_t tile[D][33];
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
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float s0 = v_scales[hh * D + c8 * 8 + j], s1 = v_scales[hh * D + c8 * 8 + j + 1];
      zero[j] = s0 == 0.0f;
      zero[j + 1] = s1 == 0.0f;
      ns2[j / 2] = f2_pack(-s0, -s1);
      r2[j / 2] = f2_pack(1.0f / s0, 1.0f / s1);   // IEEE; unused when the scale is 0
    }
    uint32_t bytes[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t_base + tg * 4 + u;
      float f[8];
      unpack8(raw[i][u], f);
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        float y0, y1;
        f2_unpack(div_rn2(f2_pack(f[j], f[j + 1]), ns2[j / 2], r2[j / 2]), y0, y1);
        if (t >= n || zero[j]) y0 = 0.0f;
        if (t >= n || zero[j + 1]) y1 = 0.0f;
        const uint32_t pr = e4m3x2(y0, y1);
        bytes[u][j] = pr & 0xFFu;
        bytes[u][j + 1] = pr >> 8;
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      tile[c8 * 8 + j][tg] = bytes[0][j] | (bytes[1][j] << 8) | (bytes[2][j] << 16) | (bytes[3][j] << 24);
  }
  __syncthreads();
  for (int o = threadIdx.x; o < D * 8; o += 256) {
    const int c = o >> 3, seg = o & 7;
    const uint4 w = make_uint4(tile[c][seg * 4], tile[c][seg * 4 + 1], tile[c][seg * 4 + 2], tile[c][seg * 4 + 3]);
    *reinterpret_cast<uint4*>(v_codes + (static_cast<int64_t>(hh) * D + c) * npad + t_base + seg * 16) = w;
  }
}

}  // namespace

cudaError_t launch_colreduce(const StridedView& x, int n, int h, int d, bool absmax, float* partials,
                             cudaStream_t s) {
  const int nchunk = (n + 127) / 128;
  const int groups = h * (d / 8);
  dim3 grid(nchunk, (groups + 127) / 128);
  if (absmax)
    colreduce_kernel<true><<<grid, 128, 0, s>>>(x.data, x.st, x.sh, n, h, d, partials);
  else
    colreduce_kernel<false><<<grid, 128, 0, s>>>(x.data, x.st, x.sh, n, h, d, partials);
  return cudaGetLastError();
}

cudaError_t launch_colfinal(const float* partials, int nchunk, int cols, int n, bool absmax, float* out,
                            cudaStream_t s) {
  dim3 grid((cols + 31) / 32);
  if (absmax)
    colfinal_kernel<true><<<grid, 256, 0, s>>>(partials, nchunk, cols, n, out);
  else
    colfinal_kernel<false><<<grid, 256, 0, s>>>(partials, nchunk, cols, n, out);
  return cudaGetLastError();
}

cudaError_t launch_quant_qk(const StridedView& q, const StridedView& k, const float* k_mean, int n, int h, int d,
                            uint16_t* q_codes, float* q_scales, uint16_t* k_codes, float* k_scales,
                            cudaStream_t s) {
  const int npad = static_cast<int>(pad128(n));
  dim3 grid(h, npad / 128);
  if (d == 128)
    quant_qk_kernel<128><<<grid, 256, 0, s>>>(q.data, q.st, q.sh, k.data, k.st, k.sh, k_mean, n, npad, q_codes,
                                              q_scales, k_codes, k_scales);
  else
    quant_qk_kernel<64><<<grid, 256, 0, s>>>(q.data, q.st, q.sh, k.data, k.st, k.sh, k_mean, n, npad, q_codes,
                                             q_scales, k_codes, k_scales);
  return cudaGetLastError();
}

cudaError_t launch_quant_v(const StridedView& v, const float* v_scales, int n, int h, int d, uint8_t* v_codes,
                           cudaStream_t s) {
  const int npad = static_cast<int>(pad128(n));
  dim3 grid(h, npad / 128);
  if (d == 128)
    quant_v_kernel<128><<<grid, 256, 0, s>>>(v.data, v.st, v.sh, v_scales, n, npad, v_codes);
  else
    quant_v_kernel<64><<<grid, 256, 0, s>>>(v.data, v.st, v.sh, v_scales, n, npad, v_codes);
  return cudaGetLastError();
}

}  // namespace sage
