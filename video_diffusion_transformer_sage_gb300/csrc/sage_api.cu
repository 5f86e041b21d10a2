// sage_api.cu -- the extern "C" entry points declared in include/sage.h: argument and
// alignment checks, workspace carving, and the launch sequence of the quantised
// attention path.  No entry point allocates device memory.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "sage_internal.h"

namespace {

using sage::pad128;

constexpr int64_t kMaxTokens = int64_t(1) << 22;     // keeps every TMA row coordinate in int32
constexpr size_t kStatusBytes = 256;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

sage_status check_shape(int64_t n, int64_t h, int64_t d) {
  if (n <= 0 || h <= 0 || d <= 0) return SAGE_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SAGE_ERR_UNSUPPORTED;
  if (n > kMaxTokens || h > 4096 || h * pad128(n) >= (int64_t(1) << 31) / 2) return SAGE_ERR_UNSUPPORTED;
  return SAGE_OK;
}

sage_status check_view(const sage_view* v) {
  if (!v || !v->data) return SAGE_ERR_INVALID_ARG;
  sage_status st = check_shape(v->n_tokens, v->n_heads, v->head_dim);
  if (st != SAGE_OK) return st;
  if (v->stride_token < 0 || v->stride_head < 0) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(v->data) || (v->stride_token % 8) != 0 || (v->stride_head % 8) != 0) return SAGE_ERR_ALIGNMENT;
  return SAGE_OK;
}

bool same_shape(const sage_view* a, const sage_view* b) {
  return a->n_tokens == b->n_tokens && a->n_heads == b->n_heads && a->head_dim == b->head_dim;
}

sage::StridedView sv(const sage_view* v) {
  return sage::StridedView{static_cast<const uint16_t*>(v->data), v->stride_token, v->stride_head};
}

sage_status check_out(const void* out, int64_t ost, int64_t osh) {
  if (!out) return SAGE_ERR_INVALID_ARG;
  if (ost < 0 || osh < 0) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(out) || (ost % 8) != 0 || (osh % 8) != 0) return SAGE_ERR_ALIGNMENT;
  return SAGE_OK;
}

// Rows per Q scale: 0 stands for the default 128; otherwise a power of two up to 128.
int q_block_of(const sage_quantized* qz) { return qz->q_block == 0 ? 128 : static_cast<int>(qz->q_block); }
bool q_block_ok(int64_t qb) { return qb == 0 || (qb >= 1 && qb <= 128 && (qb & (qb - 1)) == 0); }

sage_status check_qz(const sage_quantized* qz, bool need_qk, bool need_v) {
  if (!qz) return SAGE_ERR_INVALID_ARG;
  if (need_qk) {
    if (!q_block_ok(qz->q_block)) return SAGE_ERR_INVALID_ARG;
    if (!qz->q_codes || !qz->q_scales || !qz->k_codes || !qz->k_scales || !qz->k_mean) return SAGE_ERR_INVALID_ARG;
    if (qz->q_codes == qz->k_codes) return SAGE_ERR_INVALID_ARG;   // one buffer for both code sets
    if (!aligned16(qz->q_codes) || !aligned16(qz->k_codes) || !aligned16(qz->q_scales) ||
        !aligned16(qz->k_scales) || !aligned16(qz->k_mean))
      return SAGE_ERR_ALIGNMENT;
  }
  if (need_v) {
    if (!qz->v_codes || !qz->v_scales) return SAGE_ERR_INVALID_ARG;
    if (qz->v_format != 0 && qz->v_format != 1) return SAGE_ERR_INVALID_ARG;
    if (!aligned16(qz->v_codes) || !aligned16(qz->v_scales) || !aligned16(qz->v_mean)) return SAGE_ERR_ALIGNMENT;
  }
  return SAGE_OK;
}

inline sage_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA; }

size_t scratch_bytes(int64_t n, int64_t h, int64_t d) {
  return up256(static_cast<size_t>((n + 127) / 128) * h * d * sizeof(float));
}

// Carves the sage_attn_fwd workspace: status | q_codes | k_codes | v_codes | q_scales |
// k_scales | k_mean | v_scales | scratch (K partials) | scratch_v (V partials), each 256-byte
// aligned.
struct Carve {
  void* status;
  sage_quantized qz;
  float* scratch;
  float* scratch_v;
  size_t total;
};
Carve carve(void* base, int64_t n, int64_t h, int64_t d) {
  const int64_t np = pad128(n);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += up256(bytes);
    return static_cast<char*>(base) + o;
  };
  Carve c;
  c.status = take(kStatusBytes);
  c.qz.q_codes = reinterpret_cast<uint16_t*>(take(size_t(h) * np * d * 2));
  c.qz.k_codes = reinterpret_cast<uint16_t*>(take(size_t(h) * np * d * 2));
  c.qz.v_codes = reinterpret_cast<uint8_t*>(take(size_t(h) * d * np));
  c.qz.q_scales = reinterpret_cast<float*>(take(size_t(h) * (np / 128) * 4));
  c.qz.q_block = 128;
  c.qz.k_scales = reinterpret_cast<float*>(take(size_t(h) * (np / 64) * 4));
  c.qz.k_mean = reinterpret_cast<float*>(take(size_t(h) * d * 4));
  c.qz.v_scales = reinterpret_cast<float*>(take(size_t(h) * d * 4));
  c.qz.v_format = 0;
  c.qz.v_mean = nullptr;
  c.scratch = reinterpret_cast<float*>(take(scratch_bytes(n, h, d)));
  c.scratch_v = reinterpret_cast<float*>(take(scratch_bytes(n, h, d)));
  c.total = off;
  return c;
}

}  // namespace

namespace sage {
sage_status check_smooth_quant_qk_args(const sage_view* q, const sage_view* k, const sage_quantized* qz) {
  sage_status st;
  if ((st = check_view(q)) != SAGE_OK || (st = check_view(k)) != SAGE_OK) return st;
  if (!same_shape(q, k)) return SAGE_ERR_INVALID_ARG;
  return check_qz(qz, true, false);
}
}  // namespace sage

extern "C" {

const char* sage_status_string(sage_status status) {
  switch (status) {
    case SAGE_OK: return "SAGE_OK";
    case SAGE_ERR_INVALID_ARG: return "SAGE_ERR_INVALID_ARG: null pointer, bad size or mismatched shapes";
    case SAGE_ERR_ALIGNMENT: return "SAGE_ERR_ALIGNMENT: pointer not 16-byte aligned or stride not a multiple of 8";
    case SAGE_ERR_UNSUPPORTED: return "SAGE_ERR_UNSUPPORTED: head_dim must be 64 or 128; sizes within limits";
    case SAGE_ERR_WORKSPACE: return "SAGE_ERR_WORKSPACE: workspace missing or too small";
    case SAGE_ERR_CUDA: return "SAGE_ERR_CUDA: a CUDA call or kernel launch failed";
    case SAGE_ERR_DEVICE_TIMEOUT: return "SAGE_ERR_DEVICE_TIMEOUT: a bounded device wait expired";
  }
  return "unknown sage_status";
}

size_t sage_quant_scratch_bytes(int64_t n, int64_t h, int64_t d) {
  if (check_shape(n, h, d) != SAGE_OK) return 0;
  return scratch_bytes(n, h, d) + 256;
}

size_t sage_workspace_bytes(int64_t n, int64_t h, int64_t d) {
  if (check_shape(n, h, d) != SAGE_OK) return 0;
  return carve(nullptr, n, h, d).total;
}

size_t sage_status_block_bytes(void) { return kStatusBytes; }

sage_status sage_smooth_quant_qk(const sage_view* q, const sage_view* k, const sage_quantized* qz, void* ws,
                                 size_t ws_bytes, void* stream) {
  sage_status st;
  if ((st = sage::check_smooth_quant_qk_args(q, k, qz)) != SAGE_OK) return st;
  const int64_t n = q->n_tokens, h = q->n_heads, d = q->head_dim;
  if (!ws || !aligned16(ws)) return ws ? SAGE_ERR_ALIGNMENT : SAGE_ERR_WORKSPACE;
  if (ws_bytes < scratch_bytes(n, h, d)) return SAGE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(ws);
  const int nchunk = static_cast<int>((n + 127) / 128);
  cudaError_t e = sage::launch_colreduce(sv(k), int(n), int(h), int(d), false, nullptr, part, s);
  if (e == cudaSuccess) e = sage::launch_colfinal(part, nchunk, int(h * d), int(n), 0.0f, qz->k_mean, s);
  if (e == cudaSuccess)
    e = sage::launch_quant_qk(sv(q), sv(k), qz->k_mean, int(n), int(h), int(d), q_block_of(qz), qz->q_codes,
                              qz->q_scales, qz->k_codes, qz->k_scales, s);
  return cuda_status(e);
}

sage_status sage_smooth_quant_qk_rmsnorm_rope(const sage_view* q, const sage_view* k, const float* gamma_q,
                                              const float* gamma_k, const float* rope_cos, const float* rope_sin,
                                              float eps, const sage_quantized* qz, void* ws, size_t ws_bytes,
                                              void* stream) {
  sage_status st;
  if ((st = check_view(q)) != SAGE_OK || (st = check_view(k)) != SAGE_OK) return st;
  if (!same_shape(q, k)) return SAGE_ERR_INVALID_ARG;
  if ((st = check_qz(qz, true, false)) != SAGE_OK) return st;
  if (!gamma_q || !gamma_k || !rope_cos || !rope_sin) return SAGE_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !(eps < INFINITY)) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(gamma_q) || !aligned16(gamma_k) || !aligned16(rope_cos) || !aligned16(rope_sin))
    return SAGE_ERR_ALIGNMENT;
  const int64_t n = q->n_tokens, h = q->n_heads, d = q->head_dim;
  if (!ws || !aligned16(ws)) return ws ? SAGE_ERR_ALIGNMENT : SAGE_ERR_WORKSPACE;
  if (ws_bytes < scratch_bytes(n, h, d)) return SAGE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(ws);
  const int nchunk = static_cast<int>((n + 127) / 128);
  const sage::RowTransform tr{gamma_q, gamma_k, rope_cos, rope_sin, eps};
  // K is transformed once: the K-mean pass leaves the transformed rows in the Q code buffer
  // (same [H][pad128(N)][D] 16-bit shape), K is quantised from there, and only then are the Q
  // codes written, from Q transformed as it is loaded.
  const sage::StridedView kt{qz->q_codes, d, pad128(n) * d};
  cudaError_t e = sage::launch_colsum_transform(sv(k), int(n), int(h), int(d), tr, part, qz->q_codes, s);
  if (e == cudaSuccess) e = sage::launch_colfinal(part, nchunk, int(h * d), int(n), 0.0f, qz->k_mean, s);
  if (e == cudaSuccess)
    e = sage::launch_quant_k(kt, qz->k_mean, int(n), int(h), int(d), qz->k_codes, qz->k_scales, s);
  if (e == cudaSuccess)
    e = sage::launch_quant_q_transform(sv(q), int(n), int(h), int(d), q_block_of(qz), qz->q_codes, qz->q_scales, tr,
                                       s);
  return cuda_status(e);
}

sage_status sage_quant_v(const sage_view* v, const sage_quantized* qz, void* ws, size_t ws_bytes, void* stream) {
  sage_status st;
  if ((st = check_view(v)) != SAGE_OK) return st;
  if ((st = check_qz(qz, false, true)) != SAGE_OK) return st;
  const int64_t n = v->n_tokens, h = v->n_heads, d = v->head_dim;
  if (!ws || !aligned16(ws)) return ws ? SAGE_ERR_ALIGNMENT : SAGE_ERR_WORKSPACE;
  if (ws_bytes < scratch_bytes(n, h, d)) return SAGE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* part = static_cast<float*>(ws);
  const int nchunk = static_cast<int>((n + 127) / 128);
  cudaError_t e = cudaSuccess;
  if (qz->v_mean) {   // V smoothing: the channel mean first, as for K
    e = sage::launch_colreduce(sv(v), int(n), int(h), int(d), false, nullptr, part, s);
    if (e == cudaSuccess) e = sage::launch_colfinal(part, nchunk, int(h * d), int(n), 0.0f, qz->v_mean, s);
  }
  // Maxima of |v| (or |v - mean|), then scale = max / 448 (E4M3) or max / 127 (INT8).
  if (e == cudaSuccess) e = sage::launch_colreduce(sv(v), int(n), int(h), int(d), true, qz->v_mean, part, s);
  if (e == cudaSuccess)
    e = sage::launch_colfinal(part, nchunk, int(h * d), int(n), qz->v_format ? 127.0f : 448.0f, qz->v_scales, s);
  if (e == cudaSuccess)
    e = sage::launch_quant_v(sv(v), qz->v_scales, qz->v_mean, int(qz->v_format), int(n), int(h), int(d),
                             qz->v_codes, s);
  return cuda_status(e);
}

sage_status sage_qk_rmsnorm_rope(const sage_view* q, const sage_view* k, const float* gamma_q,
                                 const float* gamma_k, const float* rope_cos, const float* rope_sin,
                                 float eps, void* stream) {
  sage_status st;
  if ((st = check_view(q)) != SAGE_OK || (st = check_view(k)) != SAGE_OK) return st;
  if (!same_shape(q, k)) return SAGE_ERR_INVALID_ARG;
  if (!gamma_q || !gamma_k || !rope_cos || !rope_sin) return SAGE_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !(eps < INFINITY)) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(gamma_q) || !aligned16(gamma_k) || !aligned16(rope_cos) || !aligned16(rope_sin))
    return SAGE_ERR_ALIGNMENT;
  return cuda_status(sage::launch_rmsnorm_rope(sv(q), sv(k), int(q->n_tokens), int(q->n_heads), int(q->head_dim),
                                               gamma_q, gamma_k, rope_cos, rope_sin, eps,
                                               static_cast<cudaStream_t>(stream)));
}

sage_status sage_attn_fwd_quantized(int64_t n, int64_t h, int64_t d, const sage_quantized* qz, float sm_scale,
                                    void* out, int64_t ost, int64_t osh, void* status_block, void* stream) {
  sage_status st;
  if ((st = check_shape(n, h, d)) != SAGE_OK) return st;
  if ((st = check_qz(qz, true, true)) != SAGE_OK) return st;
  if ((st = check_out(out, ost, osh)) != SAGE_OK) return st;
  if (!status_block) return SAGE_ERR_INVALID_ARG;
  if (!(sm_scale > 0.0f) || sm_scale != sm_scale) return SAGE_ERR_INVALID_ARG;
  return cuda_status(sage::launch_attn_fwd(int(n), int(h), int(d), *qz, q_block_of(qz), sm_scale, out, ost, osh,
                                           static_cast<int32_t*>(status_block), static_cast<cudaStream_t>(stream)));
}

sage_status sage_quant_qkv(const sage_view* q, const sage_view* k, const sage_view* v, const sage_quantized* qz,
                           void* ws, size_t ws_bytes, void* stream) {
  sage_status st;
  if ((st = sage::check_smooth_quant_qk_args(q, k, qz)) != SAGE_OK) return st;
  if ((st = check_view(v)) != SAGE_OK) return st;
  if (!same_shape(q, v)) return SAGE_ERR_INVALID_ARG;
  if ((st = check_qz(qz, false, true)) != SAGE_OK) return st;
  const int64_t n = q->n_tokens, h = q->n_heads, d = q->head_dim;
  const size_t sb = scratch_bytes(n, h, d);
  if (!ws || !aligned16(ws)) return ws ? SAGE_ERR_ALIGNMENT : SAGE_ERR_WORKSPACE;
  if (ws_bytes < 2 * sb) return SAGE_ERR_WORKSPACE;
  if (q_block_of(qz) != 128 || qz->v_format != 0 || qz->v_mean) {
    // The options: the two stage calls, in turn (the first scratch region serves both).
    if ((st = sage_smooth_quant_qk(q, k, qz, ws, sb, stream)) != SAGE_OK) return st;
    return sage_quant_v(v, qz, ws, sb, stream);
  }
  // The default path: the kernels of the two stage calls, except that the K sums and the V
  // maxima share one launch, and so do the K mean and the V scales (5 launches instead of 7).
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* part_k = static_cast<float*>(ws);
  float* part_v = reinterpret_cast<float*>(static_cast<char*>(ws) + sb);
  const int nchunk = static_cast<int>((n + 127) / 128);
  cudaError_t e = sage::launch_colreduce_kv(sv(k), sv(v), int(n), int(h), int(d), part_k, part_v, s);
  if (e == cudaSuccess)
    e = sage::launch_colfinal_kv(part_k, part_v, nchunk, int(h * d), int(n), qz->k_mean, qz->v_scales, s);
  if (e == cudaSuccess)
    e = sage::launch_quant_qk(sv(q), sv(k), qz->k_mean, int(n), int(h), int(d), 128, qz->q_codes, qz->q_scales,
                              qz->k_codes, qz->k_scales, s);
  if (e == cudaSuccess)
    e = sage::launch_quant_v(sv(v), qz->v_scales, nullptr, 0, int(n), int(h), int(d), qz->v_codes, s);
  return cuda_status(e);
}

sage_status sage_attn_fwd(const sage_view* q, const sage_view* k, const sage_view* v, float sm_scale, void* out,
                          int64_t ost, int64_t osh, void* ws, size_t ws_bytes, void* stream) {
  sage_status st;
  if ((st = check_view(q)) != SAGE_OK || (st = check_view(k)) != SAGE_OK || (st = check_view(v)) != SAGE_OK)
    return st;
  if (!same_shape(q, k) || !same_shape(q, v)) return SAGE_ERR_INVALID_ARG;
  if ((st = check_out(out, ost, osh)) != SAGE_OK) return st;
  if (!(sm_scale > 0.0f)) return SAGE_ERR_INVALID_ARG;
  const int64_t n = q->n_tokens, h = q->n_heads, d = q->head_dim;
  if (!ws) return SAGE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SAGE_ERR_ALIGNMENT;
  Carve c = carve(ws, n, h, d);
  if (ws_bytes < c.total) return SAGE_ERR_WORKSPACE;
  // The two scratch regions are adjacent: 2 * scratch_bytes, as sage_quant_qkv takes them.
  if ((st = sage_quant_qkv(q, k, v, &c.qz, c.scratch, 2 * scratch_bytes(n, h, d), stream)) != SAGE_OK) return st;
  return sage_attn_fwd_quantized(n, h, d, &c.qz, sm_scale, out, ost, osh, c.status, stream);
}

sage_status sage_attn_dense_bf16(const sage_view* q, const sage_view* k, const sage_view* v, float sm_scale,
                                 void* out, int64_t ost, int64_t osh, void* stream) {
  sage_status st;
  if ((st = check_view(q)) != SAGE_OK || (st = check_view(k)) != SAGE_OK || (st = check_view(v)) != SAGE_OK)
    return st;
  if (!same_shape(q, k) || !same_shape(q, v)) return SAGE_ERR_INVALID_ARG;
  if ((st = check_out(out, ost, osh)) != SAGE_OK) return st;
  if (!(sm_scale > 0.0f)) return SAGE_ERR_INVALID_ARG;
  return cuda_status(sage::launch_attn_dense(sv(q), sv(k), sv(v), int(q->n_tokens), int(q->n_heads),
                                             int(q->head_dim), sm_scale, out, ost, osh,
                                             static_cast<cudaStream_t>(stream)));
}

size_t sage_dense_workspace_bytes(int64_t n, int64_t h, int64_t d) {
  if (check_shape(n, h, d) != SAGE_OK) return 0;
  return kStatusBytes + up256(static_cast<size_t>(h) * d * pad128(n) * 2);
}

sage_status sage_attn_dense_bf16_tc(const sage_view* q, const sage_view* k, const sage_view* v, float sm_scale,
                                    void* out, int64_t ost, int64_t osh, void* ws, size_t ws_bytes, void* stream) {
  sage_status st;
  if ((st = check_view(q)) != SAGE_OK || (st = check_view(k)) != SAGE_OK || (st = check_view(v)) != SAGE_OK)
    return st;
  if (!same_shape(q, k) || !same_shape(q, v)) return SAGE_ERR_INVALID_ARG;
  if ((st = check_out(out, ost, osh)) != SAGE_OK) return st;
  if (!(sm_scale > 0.0f)) return SAGE_ERR_INVALID_ARG;
  const int64_t n = q->n_tokens, h = q->n_heads, d = q->head_dim;
  if (!ws) return SAGE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return SAGE_ERR_ALIGNMENT;
  if (ws_bytes < sage_dense_workspace_bytes(n, h, d)) return SAGE_ERR_WORKSPACE;
  auto* status = static_cast<int32_t*>(ws);
  auto* vt = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) + kStatusBytes);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = sage::launch_transpose_v(sv(v), int(n), int(h), int(d), vt, s);
  if (e == cudaSuccess)
    e = sage::launch_attn_dense_tc(sv(q), sv(k), vt, int(n), int(h), int(d), sm_scale, out, ost, osh, status, s);
  return cuda_status(e);
}

sage_status sage_debug_qk_int32(int64_t n, int64_t h, int64_t d, const sage_quantized* qz, int64_t head, int64_t i0,
                                int64_t j0, int64_t row_tiles, int64_t col_tiles, int32_t* out, void* status_block,
                                void* stream) {
  sage_status st;
  if ((st = check_shape(n, h, d)) != SAGE_OK) return st;
  if ((st = check_qz(qz, true, false)) != SAGE_OK) return st;
  const int64_t np = pad128(n);
  if (!out || !status_block || head < 0 || head >= h || i0 < 0 || j0 < 0 || (i0 % 128) || (j0 % 128) ||
      row_tiles <= 0 || col_tiles <= 0 || i0 + 128 * row_tiles > np || j0 + 128 * col_tiles > np ||
      row_tiles > 65535 || col_tiles > 65535)
    return SAGE_ERR_INVALID_ARG;
  return cuda_status(sage::launch_debug_qk(int(n), int(h), int(d), *qz, int(head), int(i0), int(j0), int(row_tiles),
                                           int(col_tiles), out, static_cast<int32_t*>(status_block),
                                           static_cast<cudaStream_t>(stream)));
}

sage_status sage_measure_mma_rate(int64_t mode, int64_t iters, int64_t ctas, void* status_block, void* stream) {
  if (mode < 0 || mode > 6 || iters < 1 || iters > 100000000 || ctas < 1 || ctas > 65535 || !status_block)
    return SAGE_ERR_INVALID_ARG;
  return cuda_status(sage::launch_mma_rate(int(mode), int(iters), int(ctas), static_cast<int32_t*>(status_block),
                                           2000000000ull, static_cast<cudaStream_t>(stream)));
}

sage_status sage_debug_wait_timeout(void* status_block, int64_t limit_ns, void* stream) {
  if (!status_block || limit_ns <= 0 || limit_ns > 10000000000LL) return SAGE_ERR_INVALID_ARG;
  return cuda_status(sage::launch_debug_wait_timeout(static_cast<int32_t*>(status_block),
                                                     static_cast<uint64_t>(limit_ns),
                                                     static_cast<cudaStream_t>(stream)));
}

sage_status sage_check_device_status(void* status_block, void* stream, int32_t* where) {
  if (!status_block) return SAGE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t host[2] = {0, 0};
  if (cudaStreamSynchronize(s) != cudaSuccess) return SAGE_ERR_CUDA;
  if (cudaMemcpy(host, status_block, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return SAGE_ERR_CUDA;
  if (where) *where = host[1];
  if (host[0] != 0) {
    if (cudaMemset(status_block, 0, sizeof(host)) != cudaSuccess) return SAGE_ERR_CUDA;
    return SAGE_ERR_DEVICE_TIMEOUT;
  }
  return SAGE_OK;
}

sage_status sage_get_device_status(void* status_block, void* stream, int32_t* where) {
  return sage_check_device_status(status_block, stream, where);
}

}  // extern "C"
