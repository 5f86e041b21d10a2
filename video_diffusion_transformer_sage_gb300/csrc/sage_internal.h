// sage_internal.h -- launchers shared between the C-ABI layer and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "sage.h"

namespace sage {

// Device-side status codes recorded in the status block (first int32: nonzero on error,
// second int32: where the error was detected).
enum DeviceWhere : int32_t {
  kWhereNone = 0,
  kWhereQFull = 1,
  kWhereKvFull = 2,
  kWhereKvEmpty = 3,
  kWhereSFull = 4,
  kWherePFull = 5,
  kWherePvDone = 6,
  kWhereDebugTma = 7,
  kWhereDebugMma = 8,
  kWhereDebugTimeout = 10,
};

struct StridedView {
  const uint16_t* data;  // bf16 bits
  int64_t st, sh;        // token and head strides in elements
};

inline int64_t pad128(int64_t n) { return (n + 127) / 128 * 128; }

// sage_api.cu: the argument checks of sage_smooth_quant_qk (views, shapes, output buffers),
// everything but the workspace.
sage_status check_smooth_quant_qk_args(const sage_view* q, const sage_view* k, const sage_quantized* qz);

// quant.cu
// Per-128-token column partials: sums, or maxima of |x| (of |fl32(x - mean)| when mean is set).
cudaError_t launch_colreduce(const StridedView& x, int n, int h, int d, bool absmax, const float* mean,
                             float* partials, cudaStream_t s);
// The whole path's K sums and V maxima in one launch (part_k, part_v as for launch_colreduce).
cudaError_t launch_colreduce_kv(const StridedView& k, const StridedView& v, int n, int h, int d, float* part_k,
                               float* part_v, cudaStream_t s);
// The K mean and the E4M3 V scales (max / 448) from those partials in one launch.
cudaError_t launch_colfinal_kv(const float* part_k, const float* part_v, int nchunk, int cols, int n, float* k_mean,
                               float* v_scales, cudaStream_t s);
// amax_div == 0: out = the column mean; otherwise out = fl32(column max / amax_div).
cudaError_t launch_colfinal(const float* partials, int nchunk, int cols, int n, float amax_div, float* out,
                            cudaStream_t s);
// The qk_transform of a row (RMSNorm with weight gamma, rotary embedding by the [N][D/2] cos /
// sin table), applied by the fused quantise path to each row as it loads it.
struct RowTransform {
  const float* gamma_q;
  const float* gamma_k;
  const float* rope_cos;
  const float* rope_sin;
  float eps;
};
// Per-128-token column sums of the transformed K rows (the partials of the K mean); the
// transformed rows themselves (bf16) go to kt, head-major [H][pad128(n)][D].
cudaError_t launch_colsum_transform(const StridedView& k, int n, int h, int d, const RowTransform& tr,
                                    float* partials, uint16_t* kt, cudaStream_t s);
// Codes and scales of Q and of K - k_mean.  q_block: rows per Q scale, a power of two <= 128.
cudaError_t launch_quant_qk(const StridedView& q, const StridedView& k, const float* k_mean, int n, int h, int d,
                            int q_block, uint16_t* q_codes, float* q_scales, uint16_t* k_codes, float* k_scales,
                            cudaStream_t s);
// Codes and scales of K - k_mean alone.
cudaError_t launch_quant_k(const StridedView& k, const float* k_mean, int n, int h, int d, uint16_t* k_codes,
                           float* k_scales, cudaStream_t s);
// Codes and scales of Q with the qk_transform applied to each row as it is loaded.
cudaError_t launch_quant_q_transform(const StridedView& q, int n, int h, int d, int q_block, uint16_t* q_codes,
                                     float* q_scales, const RowTransform& tr, cudaStream_t s);
// v_format 0: E4M3 bytes; 1: INT8 codes held as fp16.  v_mean: NULL or the mean to subtract.
cudaError_t launch_quant_v(const StridedView& v, const float* v_scales, const float* v_mean, int v_format, int n,
                           int h, int d, void* v_codes, cudaStream_t s);

// qk_transform.cu: in place on the Q and K views.
cudaError_t launch_rmsnorm_rope(const StridedView& q, const StridedView& k, int n, int h, int d,
                                const float* gamma_q, const float* gamma_k, const float* rope_cos,
                                const float* rope_sin, float eps, cudaStream_t s);

// attn_fwd.cu
cudaError_t launch_attn_fwd(int n, int h, int d, const sage_quantized& qz, int q_block, float sm_scale, void* out,
                            int64_t ost, int64_t osh, int32_t* status, cudaStream_t s);
cudaError_t launch_debug_qk(int n, int h, int d, const sage_quantized& qz, int head, int i0, int j0, int row_tiles,
                            int col_tiles, int32_t* out, int32_t* status, cudaStream_t s);

cudaError_t launch_debug_wait_timeout(int32_t* status, uint64_t limit_ns, cudaStream_t s);
// The tensor-core dense path: Q, K as bf16 views, V transposed to vt [H][D][N_pad] bf16.
cudaError_t launch_attn_dense_tc(const StridedView& q, const StridedView& k, const uint16_t* vt, int n, int h, int d,
                                 float sm_scale, void* out, int64_t ost, int64_t osh, int32_t* status, cudaStream_t s);

// mma_rate.cu: `ctas` CTAs each issue `iters` rounds of the tensor-core MMAs of `mode` (0-4).
cudaError_t launch_mma_rate(int mode, int iters, int ctas, int32_t* status, uint64_t limit_ns, cudaStream_t s);

// attn_dense.cu
cudaError_t launch_attn_dense(const StridedView& q, const StridedView& k, const StridedView& v, int n, int h,
                              int d, float sm_scale, void* out, int64_t ost, int64_t osh, cudaStream_t s);
// vt[h][c][t] = v[t][h][c] for t < N_pad (zero for t >= N): the V operand of the tensor-core dense path.
cudaError_t launch_transpose_v(const StridedView& v, int n, int h, int d, uint16_t* vt, cudaStream_t s);

// Calls of at most this many Q (or K, V) elements launch their short kernels (the column
// finalise, the V fix-up) as dependents of the kernel before them, which hides those launches
// (tiny: 0.056 -> 0.050 ms per whole call); larger calls gain nothing measurable and launch
// every kernel in plain stream order.
constexpr int64_t kDependentLaunchMaxElements = int64_t(1) << 26;
inline bool dependent_launches(int64_t n, int64_t h, int64_t d) { return n * h * d <= kDependentLaunchMaxElements; }

// Launches `kernel`; with `dependent`, with programmatic stream serialization: it may launch while
// the previous kernel of the stream drains, and must call grid_dep_wait before touching memory
// that kernel writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(bool dependent, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace sage
