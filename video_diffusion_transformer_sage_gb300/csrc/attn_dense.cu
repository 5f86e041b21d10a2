// attn_dense.cu -- unquantised attention in fp32 arithmetic on bf16 inputs: the dense
// quality anchor that the pages compare the quantised path against
// ("gb10-sampling-component-profile-1344x768-124f-seed440420.json",
// quality_gates.sol_fully_dense_tau_minus_100_relative_l2_vs_sage2).  A correctness path:
// plain CUDA cores, one pass of online softmax, no tensor cores.
//
// CTA = 8 warps x (8 rows at D = 64, 4 rows at D = 128) of one head.  Per 64-key tile, K is staged
// transposed ([D][64] fp32) so that lane j reads key j without bank conflicts, and V as
// [64][D] fp32.  Lane j scores keys j and j + 32 for its warp's 8 rows; P is broadcast
// with warp shuffles into the O accumulation, where lane owns channels lane + 32 i.
//
// Also here: the V transpose of the tensor-core dense path (attn_fwd.cu, attn_dense_tc_kernel),
// whose P.V takes V with the keys of each channel contiguous.
#include <cuda_bf16.h>

#include "sage_internal.h"

namespace sage {
namespace {

constexpr int kKeys = 64;
// Rows per warp: 4 at D = 128 keeps the accumulators in registers.
template <int D> __host__ __device__ constexpr int rows_per_warp() { return D == 128 ? 4 : 8; }

template <int D>
__global__ void __launch_bounds__(256) attn_dense_kernel(const uint16_t* __restrict__ q, int64_t qst, int64_t qsh,
                                                         const uint16_t* __restrict__ k, int64_t kst, int64_t ksh,
                                                         const uint16_t* __restrict__ v, int64_t vst, int64_t vsh,
                                                         int n, float scale_log2, uint16_t* __restrict__ out,
                                                         int64_t ost, int64_t osh) {
  constexpr int RPW = rows_per_warp<D>(), kRows = 8 * RPW;
  extern __shared__ float sm[];
  float* sq = sm;                       // [kRows][D]
  float* skt = sq + kRows * D;          // [D][kKeys]
  float* sv = skt + D * kKeys;          // [kKeys][D]
  const int hh = blockIdx.y, r0 = blockIdx.x * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bf = [](uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); };

  for (int i = threadIdx.x; i < kRows * D; i += 256) {
    const int r = i / D, c = i % D;
    sq[i] = (r0 + r < n) ? bf(q[static_cast<int64_t>(r0 + r) * qst + hh * qsh + c]) * scale_log2 : 0.0f;
  }
  constexpr int CI = D / 32;
  float o[RPW][CI];
  float m[RPW], l[RPW];
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0f;
#pragma unroll
    for (int i = 0; i < CI; ++i) o[r][i] = 0.0f;
  }
  for (int j0 = 0; j0 < n; j0 += kKeys) {
    __syncthreads();
    for (int i = threadIdx.x; i < kKeys * D; i += 256) {
      const int j = i / D, c = i % D;
      const bool ok = j0 + j < n;
      skt[c * kKeys + j] = ok ? bf(k[static_cast<int64_t>(j0 + j) * kst + hh * ksh + c]) : 0.0f;
      sv[i] = ok ? bf(v[static_cast<int64_t>(j0 + j) * vst + hh * vsh + c]) : 0.0f;
    }
    __syncthreads();
    float s[RPW][2];
#pragma unroll
    for (int r = 0; r < RPW; ++r) s[r][0] = s[r][1] = 0.0f;
    for (int c = 0; c < D; ++c) {
      const float k0 = skt[c * kKeys + lane], k1 = skt[c * kKeys + lane + 32];
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        const float qv = sq[(warp * RPW + r) * D + c];
        s[r][0] = fmaf(qv, k0, s[r][0]);
        s[r][1] = fmaf(qv, k1, s[r][1]);
      }
    }
    const bool v0 = j0 + lane < n, v1 = j0 + lane + 32 < n;
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
      if (!v0) s[r][0] = -INFINITY;
      if (!v1) s[r][1] = -INFINITY;
      float mx = fmaxf(s[r][0], s[r][1]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mn = fmaxf(m[r], mx);
      const float alpha = exp2f(m[r] - mn);
      const float p0 = exp2f(s[r][0] - mn), p1 = exp2f(s[r][1] - mn);
      float ps = p0 + p1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l[r] = l[r] * alpha + ps;
      m[r] = mn;
#pragma unroll
      for (int i = 0; i < CI; ++i) o[r][i] *= alpha;
      for (int j = 0; j < kKeys; ++j) {
        const float pj = __shfl_sync(0xffffffffu, j < 32 ? p0 : p1, j & 31);
#pragma unroll
        for (int i = 0; i < CI; ++i) o[r][i] = fmaf(pj, sv[j * D + lane + 32 * i], o[r][i]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int row = r0 + warp * RPW + r;
    if (row >= n) continue;
    uint16_t* orow = out + static_cast<int64_t>(row) * ost + static_cast<int64_t>(hh) * osh;
#pragma unroll
    for (int i = 0; i < CI; ++i) orow[lane + 32 * i] = __bfloat16_as_ushort(__float2bfloat16_rn(o[r][i] / l[r]));
  }
}

// V^T for the tensor-core dense path: vt[h][c][t] = v[t][h][c] (bf16 bits), t < N_pad, zero for
// t >= N.  CTA = (head, 128 tokens): the tokens' rows are read as 16-byte vectors (4 tokens x 8
// channels per work item), each channel's 128 tokens gathered in shared memory as 64 bf16 pairs
// (the earlier token in the low half), then written as 16-byte runs of 8 tokens.
template <int D>
__global__ void __launch_bounds__(256) transpose_v_kernel(const uint16_t* __restrict__ v, int64_t st, int64_t sh,
                                                          int n, int npad, uint16_t* __restrict__ vt) {
  constexpr int VPR = D / 8;
  __shared__ uint32_t tile[D][64 + 1];
  const int hh = blockIdx.x, t_base = blockIdx.y * 128;
  for (int it = threadIdx.x; it < VPR * 32; it += 256) {
    const int c8 = it % VPR, tg = it / VPR;
    uint4 raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = t_base + tg * 4 + u;
      raw[u] = t < n ? *reinterpret_cast<const uint4*>(v + static_cast<int64_t>(t) * st + hh * sh + c8 * 8)
                     : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t h16[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t w = (&raw[u].x)[j >> 1];
        h16[u] = (j & 1) ? (w >> 16) : (w & 0xFFFFu);
      }
      tile[c8 * 8 + j][tg * 2] = h16[0] | (h16[1] << 16);
      tile[c8 * 8 + j][tg * 2 + 1] = h16[2] | (h16[3] << 16);
    }
  }
  __syncthreads();
  for (int o = threadIdx.x; o < D * 16; o += 256) {
    const int c = o / 16, seg = o % 16;
    const uint4 w = make_uint4(tile[c][seg * 4], tile[c][seg * 4 + 1], tile[c][seg * 4 + 2], tile[c][seg * 4 + 3]);
    *reinterpret_cast<uint4*>(vt + (static_cast<int64_t>(hh) * D + c) * npad + t_base + seg * 8) = w;
  }
}

}  // namespace

cudaError_t launch_transpose_v(const StridedView& v, int n, int h, int d, uint16_t* vt, cudaStream_t s) {
  const int npad = static_cast<int>((n + 127) / 128 * 128);
  const dim3 grid(h, npad / 128);
  if (d == 128)
    transpose_v_kernel<128><<<grid, 256, 0, s>>>(v.data, v.st, v.sh, n, npad, vt);
  else
    transpose_v_kernel<64><<<grid, 256, 0, s>>>(v.data, v.st, v.sh, n, npad, vt);
  return cudaGetLastError();
}

cudaError_t launch_attn_dense(const StridedView& q, const StridedView& k, const StridedView& v, int n, int h,
                              int d, float sm_scale, void* out, int64_t ost, int64_t osh, cudaStream_t s) {
  const float scale_log2 = sm_scale * 1.4426950408889634f;
  const int rows = 8 * (d == 128 ? rows_per_warp<128>() : rows_per_warp<64>());
  dim3 grid((n + rows - 1) / rows, h);
  const int smem = (rows * d + d * kKeys + kKeys * d) * 4;
  cudaError_t e;
  if (d == 128) {
    e = cudaFuncSetAttribute(attn_dense_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attn_dense_kernel<128><<<grid, 256, smem, s>>>(q.data, q.st, q.sh, k.data, k.st, k.sh, v.data, v.st, v.sh, n,
                                                   scale_log2, static_cast<uint16_t*>(out), ost, osh);
  } else {
    e = cudaFuncSetAttribute(attn_dense_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attn_dense_kernel<64><<<grid, 256, smem, s>>>(q.data, q.st, q.sh, k.data, k.st, k.sh, v.data, v.st, v.sh, n,
                                                  scale_log2, static_cast<uint16_t*>(out), ost, osh);
  }
  return cudaGetLastError();
}

}  // namespace sage
