// mma_rate.cu -- measures the tensor-core rate of the tcgen05.mma shapes the fused attention
// issues, so that its roofline has a measured ceiling for each instruction kind.
//
// One CTA per SM.  Each CTA zeroes its shared-memory operand tiles and the tensor-memory
// columns it reads as an operand, then one thread issues `iters` rounds of MMAs back to back
// (tcgen05.mma issue blocks while the pipe is busy, so the loop runs at the pipe's rate), and
// the CTA waits for the last one.  Modes (per round):
//   0  QK^T step: kind::f16, A and B from shared memory, 128 x 128 x 16, into two
//      accumulators in turn (as the two Q tiles' S_0 and S_1)                      (8 MMAs)
//   1  P.V step:  kind::f8f6f4 E4M3, A from tensor memory, B from shared memory,
//                 128 x 128 x 32, into two accumulators in turn (O_0, O_1)          (8 MMAs)
//   2  one key tile of one 128-row Q tile as the fused kernel issues it: 8 of mode 0 into an
//      S accumulator, then 4 of mode 1 reading P from the other S accumulator     (12 MMAs)
//   3  kind::f8f6f4 E4M3, both operands from shared memory, 128 x 256 x 32         (8 MMAs)
//   4  kind::f16, both operands from shared memory, 128 x 256 x 16                 (8 MMAs)
//   5  P.V step at D = 64: as mode 1 with 128 x 64 x 32                            (8 MMAs)
//   6  one key tile of one 128-row Q tile at D = 64: 4 of mode 0 into an S accumulator,
//      then 4 of mode 5 reading P from the other S accumulator                     (8 MMAs)
// The operands are zeros: the rate of these instructions does not depend on the values.
#include <cuda_runtime.h>

#include "sage_internal.h"
#include "sm103_ptx.cuh"

namespace sage {
namespace {

constexpr int kATileBytes = 128 * 128;    // 128 rows x 128 B (128-byte swizzle), 1024-B aligned
constexpr int kBTileBytes = 256 * 128;    // up to 256 rows x 128 B
constexpr int kSmemBytes = kATileBytes + kBTileBytes + 1024;

__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int mode, int iters, int32_t* status, uint64_t limit) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t tmem_slot;
  __shared__ uint64_t bar_done;
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < (kATileBytes + kBTileBytes) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&bar_done, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  {
    // Zero the first 32 columns of both S accumulators (the P operand of modes 1 and 2).
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    SAGE_TMEM_ST32(tmem + lane_base + 0, z);
    SAGE_TMEM_ST32(tmem + lane_base + 128, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) {
    const uint32_t sa = smem_u32(smem), sb = smem_u32(smem + kATileBytes);
    const uint64_t da = sdesc_k_sw128(sa), db = sdesc_k_sw128(sb);
    constexpr uint32_t id128 = idesc_f32acc(128, 128), id256 = idesc_f32acc(128, 256);
    constexpr uint32_t id64 = idesc_f32acc(128, 64);
    // One loop per mode, 8 MMAs (mode 2: 12) unrolled per round, so the issuing thread's loop
    // overhead stays far below the MMAs' execution time.
    switch (mode) {
      case 0:   // two accumulators in turn, as the kernel's two Q tiles use S_0 and S_1
        for (int it = 0; it < iters; ++it) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            mma_f16_ss(tmem + (u & 1) * 128, sdesc_k_sw128(sa + (u >> 1) * 32), sdesc_k_sw128(sb + (u >> 1) * 32),
                       id128, (it > 0 || u > 1) ? 1u : 0u);
        }
        break;
      case 1:   // two accumulators in turn (O_0, O_1), P read from S_0 and S_1
        for (int it = 0; it < iters; ++it) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            mma_f8_ts(tmem + 256 + (u & 1) * 128, tmem + (u & 1) * 128 + (u >> 1) * 8,
                      sdesc_k_sw128(sb + (u >> 1) * 32), id128, (it > 0 || u > 1) ? 1u : 0u);
        }
        break;
      case 2:
        for (int it = 0; it < iters; ++it) {
          const uint32_t s_acc = tmem + (it & 1) * 128, s_p = tmem + ((it + 1) & 1) * 128;
          const uint32_t o_acc = tmem + 256 + (it & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_f16_ss(s_acc, sdesc_k_sw128(sa + (kk & 3) * 32), sdesc_k_sw128(sb + (kk & 3) * 32), id128,
                       kk > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8_ts(o_acc, s_p + kk * 8, sdesc_k_sw128(sb + kk * 32), id128, (it > 1 || kk > 0) ? 1u : 0u);
        }
        break;
      case 5:   // two accumulators in turn (O_0, O_1 at D = 64), P read from S_0 and S_1
        for (int it = 0; it < iters; ++it) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            mma_f8_ts(tmem + 256 + (u & 1) * 64, tmem + (u & 1) * 128 + (u >> 1) * 8,
                      sdesc_k_sw128(sb + (u >> 1) * 32), id64, (it > 0 || u > 1) ? 1u : 0u);
        }
        break;
      case 6:
        for (int it = 0; it < iters; ++it) {
          const uint32_t s_acc = tmem + (it & 1) * 128, s_p = tmem + ((it + 1) & 1) * 128;
          const uint32_t o_acc = tmem + 256 + (it & 1) * 64;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16_ss(s_acc, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sb + kk * 32), id128, kk > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8_ts(o_acc, s_p + kk * 8, sdesc_k_sw128(sb + kk * 32), id64, (it > 1 || kk > 0) ? 1u : 0u);
        }
        break;
      case 3:
        for (int it = 0; it < iters; ++it) {
#pragma unroll
          for (int u = 0; u < 8; ++u) mma_f8_ss(tmem + (u & 1) * 256, da, db, id256, (it > 0 || u > 1) ? 1u : 0u);
        }
        break;
      default:
        for (int it = 0; it < iters; ++it) {
#pragma unroll
          for (int u = 0; u < 8; ++u) mma_f16_ss(tmem + (u & 1) * 256, da, db, id256, (it > 0 || u > 1) ? 1u : 0u);
        }
        break;
    }
    tc_commit(&bar_done);
    if (!mbar_wait(&bar_done, 0, limit) && atomicCAS(status, 0, 1) == 0) status[1] = kWhereDebugMma;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_mma_rate(int mode, int iters, int ctas, int32_t* status, uint64_t limit_ns, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  mma_rate_kernel<<<ctas, 128, kSmemBytes, s>>>(mode, iters, status, limit_ns);
  return cudaGetLastError();
}

}  // namespace sage
