// qk_transform.cu -- in-place RMSNorm + rotary embedding of Q and K on strided views.
//
// The qk_transform stage of the strided-NHD dataflow in
// "gb10-sage-strided-nhd-summary-1344x768-124f-seed440420.json" (key dataflow.qk_transform:
// RMSNorm and RoPE applied in place on the projection's strided views; timed as rms_rope in
// the block-24 profile of "gb10-sampling-component-profile-1344x768-124f-seed440420.json").
// It runs upstream of the K mean and the quantisation, on the same bf16 [N, H, D] views.
//
// Per (token t, head h), in fp32 with every product and sum rounded on its own (no
// contraction into fused multiply-adds), IEEE square root and division:
//   ms = (sum_c x_c^2) / D       the sum as D/8 partial sums of 8 consecutive channels, each
//                                in channel order, folded pairwise by a butterfly over the
//                                row's D/8 threads (partial g + partial g^s, s = D/16 .. 1)
//   r  = 1 / sqrt(ms + eps),     y_c = (x_c * r) * gamma[c]
//   z_2i = y_2i cos - y_2i+1 sin,   z_2i+1 = y_2i sin + y_2i+1 cos    (cos, sin of [t][i])
//   x_c <- bf16_rne(z_c)
// The pages fix no precision or order; this one is stated so that the result is reproducible
// bit for bit.
//
// HBM-bound: each row is read once and written once (8 N H D bytes for Q and K together).
// Two kernels, the same row arithmetic (the inline functions below), identical results:
//  * rmsnorm_rope_bulk_kernel, when the heads of a token are contiguous (head stride D): whole
//    token slices move between HBM and shared memory by bulk copy (458 us on the video
//    workload, 4.77 TB/s);
//  * rmsnorm_rope_kernel, for any strides: D/8 threads hold a row, 16 bytes each; a persistent
//    grid strides over batches of rows, each thread loading its rows of the next batch before
//    it computes and stores those of the current one (474 us, 4.61 TB/s).
// Neither may load through the read-only (non-coherent) path: they write what they read.
#include <cuda_bf16.h>

#include <algorithm>

#include "qk_row.cuh"
#include "sage_internal.h"
#include "sm103_ptx.cuh"

namespace sage {
namespace {

constexpr int kRows = 4;   // rows per batch per thread (two batches in flight)

__device__ __forceinline__ uint4 ld_rows(const uint16_t* p) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// blockIdx.z: 0 = Q, 1 = K.  Rows (t, h) are numbered t * H + h, heads fastest; batch b holds
// rows [b * kBatch, (b + 1) * kBatch), thread (rin, c8) rows b * kBatch + rin * kRows + i, so
// a thread's rows are mostly heads of one token and it loads that token's cos / sin once for
// them.  Persistent: gridDim.x CTAs stride over the batches.  Stores stream (st.global.cs):
// the rows are not read again here.
template <int D>
__global__ void __launch_bounds__(256) rmsnorm_rope_kernel(uint16_t* q, int64_t qst, int64_t qsh, uint16_t* k,
                                                           int64_t kst, int64_t ksh, int n, int h,
                                                           const float* __restrict__ gamma_q,
                                                           const float* __restrict__ gamma_k,
                                                           const float* __restrict__ rope_cos,
                                                           const float* __restrict__ rope_sin, float eps) {
  constexpr int VPR = D / 8;
  constexpr int RPP = 256 / VPR;
  constexpr uint32_t kBatch = RPP * kRows;
  const bool is_k = blockIdx.z != 0;
  uint16_t* x = is_k ? k : q;
  const int64_t st = is_k ? kst : qst, sh = is_k ? ksh : qsh;
  const float* gamma = is_k ? gamma_k : gamma_q;
  const int c8 = threadIdx.x % VPR, rin = threadIdx.x / VPR;
  const uint32_t nrows = static_cast<uint32_t>(n) * static_cast<uint32_t>(h);
  const uint32_t nbatch = (nrows + kBatch - 1) / kBatch;
  float g[8];
  load_gamma8(gamma, c8, g);
  uint4 v[kRows];
  auto load = [&](uint32_t b) {
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const uint32_t r = b * kBatch + rin * kRows + i;
      v[i] = make_uint4(0, 0, 0, 0);
      if (r < nrows) {
        const uint32_t t = r / static_cast<uint32_t>(h);
        v[i] = ld_rows(x + t * st + (r - t * h) * sh + c8 * 8);
      }
    }
  };
  uint32_t b = blockIdx.x;
  if (b < nbatch) load(b);
  for (; b < nbatch; b += gridDim.x) {
    uint4 cur[kRows];
    uint32_t t_tab = 0xFFFFFFFFu;
    float4 cs = make_float4(0.f, 0.f, 0.f, 0.f), sn = cs;
#pragma unroll
    for (int i = 0; i < kRows; ++i) cur[i] = v[i];
    if (b + gridDim.x < nbatch) load(b + gridDim.x);
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const uint32_t r = b * kBatch + rin * kRows + i;
      float f[8];
      unpack_bf16x8(cur[i], f);
      const float acc = row_sumsq<VPR>(f);
      if (r >= nrows) continue;           // whole rows only: the shuffles above ran in every lane
      const uint32_t t = r / static_cast<uint32_t>(h);
      if (t != t_tab) {                 // the thread's rows are mostly heads of one token
        cs = __ldg(reinterpret_cast<const float4*>(rope_cos + static_cast<size_t>(t) * (D / 2) + c8 * 4));
        sn = __ldg(reinterpret_cast<const float4*>(rope_sin + static_cast<size_t>(t) * (D / 2) + c8 * 4));
        t_tab = t;
      }
      const uint4 o = norm_rotate8<D>(f, acc, eps, g, cs, sn);
      {
        uint16_t* dst = x + t * st + (r - t * h) * sh + c8 * 8;
        asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(dst), "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                     : "memory");
      }
    }
  }
}

// Token slices through shared memory, for views whose heads lie contiguously in a token
// (head stride D, as in the projection buffer): unit u < N is Q's token u, unit N + t is K's
// token t, each H * D bf16 contiguous.  A persistent CTA takes units blockIdx.x + i gridDim.x;
// thread 0 streams them in with bulk copies kBulkAhead units ahead into a ring of kBulkSlots
// slots and writes each transformed slice back with a bulk store.  The bulk copies move whole
// slices at DMA rates, which the in-place loads of the kernel above cannot (they may not take
// the read-only path).  A slot is reloaded only after the store of its previous unit has
// finished reading it; the compute of that unit ended at the barrier before that store.
constexpr int kBulkSlots = 4, kBulkAhead = 2;
constexpr int kBulkMaxBytes = 28672;   // H * D * 2 up to 28 KB (H <= 112 at D = 128)
constexpr uint64_t kBulkWaitNs = 2000000000ull;

template <int D>
__global__ void __launch_bounds__(256) rmsnorm_rope_bulk_kernel(uint16_t* q, int64_t qst, uint16_t* k, int64_t kst,
                                                                int n, int h, const float* __restrict__ gamma_q,
                                                                const float* __restrict__ gamma_k,
                                                                const float* __restrict__ rope_cos,
                                                                const float* __restrict__ rope_sin, float eps) {
  constexpr int VPR = D / 8, RPP = 256 / VPR;
  extern __shared__ __align__(128) uint8_t slices[];
  __shared__ __align__(8) uint64_t full[kBulkSlots];
  const uint32_t bytes = static_cast<uint32_t>(h) * D * 2;
  const uint32_t slot_bytes = (bytes + 127u) & ~127u;
  const int units = 2 * n;
  const int count = static_cast<int>(blockIdx.x) < units ? (units - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  auto unit_ptr = [&](int i) -> uint16_t* {
    const int u = blockIdx.x + i * gridDim.x;
    return u < n ? q + static_cast<int64_t>(u) * qst : k + static_cast<int64_t>(u - n) * kst;
  };
  auto issue_load = [&](int i) {
    const int sl = i % kBulkSlots;
    mbar_arrive_expect_tx(full + sl, bytes);
    bulk_load(slices + sl * slot_bytes, unit_ptr(i), bytes, full + sl);
  };
  if (threadIdx.x == 0) {
    for (int sl = 0; sl < kBulkSlots; ++sl) mbar_init(full + sl, 1);
    fence_mbar_init();
    for (int i = 0; i < kBulkAhead && i < count; ++i) issue_load(i);
  }
  __syncthreads();
  const int c8 = threadIdx.x % VPR, rin = threadIdx.x / VPR;
  float gq[8], gk[8];
  load_gamma8(gamma_q, c8, gq);
  load_gamma8(gamma_k, c8, gk);
  for (int i = 0; i < count; ++i) {
    if (threadIdx.x == 0 && i + kBulkAhead < count) {
      bulk_wait_read<kBulkSlots - kBulkAhead - 1>();   // the store of unit i + kBulkAhead - kBulkSlots
      issue_load(i + kBulkAhead);
    }
    const int sl = i % kBulkSlots;
    const bool landed = mbar_wait(full + sl, (i / kBulkSlots) & 1, kBulkWaitNs);
    if (!__syncthreads_and(landed)) break;   // a copy that never lands (a failing device): stop
    const int u = blockIdx.x + i * gridDim.x;
    const bool is_k = u >= n;
    const int64_t t = is_k ? u - n : u;
    const float4 cs = __ldg(reinterpret_cast<const float4*>(rope_cos + t * (D / 2) + c8 * 4));
    const float4 sn = __ldg(reinterpret_cast<const float4*>(rope_sin + t * (D / 2) + c8 * 4));
    uint16_t* base = reinterpret_cast<uint16_t*>(slices + sl * slot_bytes);
    for (int r0 = 0; r0 < h; r0 += RPP) {
      const int r = r0 + rin;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < h) v = *reinterpret_cast<const uint4*>(base + r * D + c8 * 8);
      float f[8];
      unpack_bf16x8(v, f);
      const float acc = row_sumsq<VPR>(f);
      if (r < h) *reinterpret_cast<uint4*>(base + r * D + c8 * 8) = norm_rotate8<D>(f, acc, eps, is_k ? gk : gq, cs, sn);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      bulk_store(unit_ptr(i), base, bytes);
      bulk_commit();
    }
  }
  if (threadIdx.x == 0) bulk_wait_all();
}

}  // namespace

cudaError_t launch_rmsnorm_rope(const StridedView& q, const StridedView& k, int n, int h, int d,
                                const float* gamma_q, const float* gamma_k, const float* rope_cos,
                                const float* rope_sin, float eps, cudaStream_t s) {
  const int64_t slice = static_cast<int64_t>(h) * d * 2;
  if (q.sh == d && k.sh == d && slice <= kBulkMaxBytes) {
    // Heads contiguous in each token: whole token slices by bulk copy.
    const int slot = static_cast<int>((slice + 127) / 128 * 128);
    const int smem = kBulkSlots * slot;
    int sms = 0, dev = 0, occ = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
      e = d == 128 ? cudaFuncSetAttribute(rmsnorm_rope_bulk_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                   : cudaFuncSetAttribute(rmsnorm_rope_bulk_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess)
      e = d == 128 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rmsnorm_rope_bulk_kernel<128>, 256, smem)
                   : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rmsnorm_rope_bulk_kernel<64>, 256, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(int64_t(2) * n, int64_t(sms) * std::max(occ, 1)));
    uint16_t* qd = const_cast<uint16_t*>(q.data);
    uint16_t* kd = const_cast<uint16_t*>(k.data);
    if (d == 128)
      rmsnorm_rope_bulk_kernel<128><<<static_cast<unsigned>(grid), 256, smem, s>>>(qd, q.st, kd, k.st, n, h, gamma_q,
                                                                                  gamma_k, rope_cos, rope_sin, eps);
    else
      rmsnorm_rope_bulk_kernel<64><<<static_cast<unsigned>(grid), 256, smem, s>>>(qd, q.st, kd, k.st, n, h, gamma_q,
                                                                                 gamma_k, rope_cos, rope_sin, eps);
    return cudaGetLastError();
  }
  const int64_t nrows = static_cast<int64_t>(n) * h;
  const int vpr = d / 8, rows_per_cta = (256 / vpr) * kRows;
  const int64_t blocks = (nrows + rows_per_cta - 1) / rows_per_cta;
  if (nrows >= (int64_t(1) << 30)) return cudaErrorInvalidValue;
  int sms = 0, dev = 0, occ = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = d == 128 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rmsnorm_rope_kernel<128>, 256, 0)
                 : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, rmsnorm_rope_kernel<64>, 256, 0);
  if (e != cudaSuccess) return e;
  // Every resident CTA slot, split between Q and K; never more CTAs than batches.
  const int64_t per_z = std::max<int64_t>(1, std::min<int64_t>(blocks, int64_t(sms) * std::max(occ, 1) / 2));
  dim3 grid(static_cast<unsigned>(per_z), 1, 2);
  uint16_t* qd = const_cast<uint16_t*>(q.data);
  uint16_t* kd = const_cast<uint16_t*>(k.data);
  if (d == 128)
    rmsnorm_rope_kernel<128><<<grid, 256, 0, s>>>(qd, q.st, q.sh, kd, k.st, k.sh, n, h, gamma_q, gamma_k, rope_cos,
                                                  rope_sin, eps);
  else
    rmsnorm_rope_kernel<64><<<grid, 256, 0, s>>>(qd, q.st, q.sh, kd, k.st, k.sh, n, h, gamma_q, gamma_k, rope_cos,
                                                 rope_sin, eps);
  return cudaGetLastError();
}

}  // namespace sage
