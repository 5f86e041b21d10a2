// qk_row.cuh -- the row arithmetic of the qk_transform stage (RMSNorm with weight gamma, then
// the rotary embedding of channel pairs), shared by the in-place kernels of qk_transform.cu and
// the quantise kernels of quant.cu that apply it as they load a row.  One definition, so both
// paths give the same bf16 values bit for bit.
//
// Per (token t, head h), in fp32 with every product and sum rounded on its own, IEEE square
// root and division:
//   ms = (sum_c x_c^2) / D       the sum as D/8 partial sums of 8 consecutive channels, each
//                                in channel order, folded pairwise by a butterfly over the
//                                row's D/8 lanes (partial g + partial g^s, s = D/16 .. 1)
//   r  = 1 / sqrt(ms + eps),     y_c = (x_c * r) * gamma[c]
//   z_2i = y_2i cos - y_2i+1 sin,   z_2i+1 = y_2i sin + y_2i+1 cos    (cos, sin of [t][i])
//   x_c <- bf16_rne(z_c)
// A row is held by D/8 consecutive lanes of a warp, 8 channels (16 bytes) each.
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace sage {

__device__ __forceinline__ uint32_t bf16x2_rne(float lo, float hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(lo))) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(hi))) << 16);
}

// ---- the row arithmetic, shared by both kernels ----------------------------------------
__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
}

// sum_c x_c^2 of the row: the thread's 8 channels in channel order, then the butterfly over
// the row's VPR consecutive lanes.  Every lane of the warp must call it.
template <int VPR>
__device__ __forceinline__ float row_sumsq(const float f[8]) {
  float acc = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) acc = __fadd_rn(acc, __fmul_rn(f[j], f[j]));
#pragma unroll
  for (int s = VPR / 2; s > 0; s >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, s));
  return acc;
}

// The thread's 8 channels after the norm (1 / sqrt(sum / D + eps), weight g) and the rotation
// of its 4 channel pairs by (cs, sn), as 4 bf16x2 words.
template <int D>
__device__ __forceinline__ uint4 norm_rotate8(const float f[8], float sumsq, float eps, const float g[8],
                                              const float4& cs, const float4& sn) {
  const float ms = __fmul_rn(sumsq, 1.0f / D);
  const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
  const float cc[4] = {cs.x, cs.y, cs.z, cs.w}, ss[4] = {sn.x, sn.y, sn.z, sn.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float y0 = __fmul_rn(__fmul_rn(f[2 * j], rs), g[2 * j]);
    const float y1 = __fmul_rn(__fmul_rn(f[2 * j + 1], rs), g[2 * j + 1]);
    const float z0 = __fsub_rn(__fmul_rn(y0, cc[j]), __fmul_rn(y1, ss[j]));
    const float z1 = __fadd_rn(__fmul_rn(y0, ss[j]), __fmul_rn(y1, cc[j]));
    o[j] = bf16x2_rne(z0, z1);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void load_gamma8(const float* gamma, int c8, float g[8]) {
  const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma + c8 * 8));
  const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma + c8 * 8 + 4));
  g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
  g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
}

// The same transform of one lane's 8 channels of row (token t) in place: loads the lane's cos /
// sin pairs of token t.  Every lane of the warp must call it (the row sum is a butterfly).
template <int D>
__device__ __forceinline__ uint4 transform_row8(const uint4& v, int t, int c8, const float g[8],
                                                const float* __restrict__ rope_cos,
                                                const float* __restrict__ rope_sin, float eps) {
  float f[8];
  unpack_bf16x8(v, f);
  const float ss = row_sumsq<D / 8>(f);
  const int64_t off = static_cast<int64_t>(t) * (D / 2) + c8 * 4;
  const float4 cs = __ldg(reinterpret_cast<const float4*>(rope_cos + off));
  const float4 sn = __ldg(reinterpret_cast<const float4*>(rope_sin + off));
  return norm_rotate8<D>(f, ss, eps, g, cs, sn);
}

}  // namespace sage
