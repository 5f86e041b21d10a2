// noalloc.cu -- sage_smooth_quant_qk_noalloc: the K-mean / Q,K quantisation entry point for
// callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers: plugin and custom-operator
// interfaces of host frameworks that own every device allocation and offer no workspace,
// and code that must not call cudaMalloc / cudaFree because those calls can synchronise
// the whole device.  sage_smooth_quant_qk needs a caller-provided scratch buffer for its
// per-128-token column partials; this variant takes that scratch from a fixed array in the
// library's own device memory instead, so it needs nothing beyond the caller's inputs and
// outputs.
//
// The array lives for as long as the library is loaded, on every GPU that loads it.  Its
// size bounds the problem: ceil(N / 128) * H * D <= kNoAllocScratchFloats.
#include <cuda_runtime.h>

#include <mutex>

#include "sage_internal.h"

namespace {

// 16 MiB: enough for the pages' call (ceil(37810/128) * 56 * 128 = 2,121,728 floats).
constexpr size_t kNoAllocScratchFloats = size_t(4) << 20;

// Per-128-token column partials of K.  Every element a call reads is written earlier in the
// same call, so nothing needs clearing between calls.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
float* g_scratch_ptr[kMaxDevices] = {};
cudaError_t g_setup_err[kMaxDevices] = {};

// The host-side name g_noalloc_scratch is not a device address; the kernels must be given the
// address cudaGetSymbolAddress returns, looked up once per device with that device current.
float* device_scratch(int dev, cudaError_t* err) {
  std::call_once(g_once[dev], [dev] {
    void* p = nullptr;
    g_setup_err[dev] = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    g_scratch_ptr[dev] = g_setup_err[dev] == cudaSuccess ? static_cast<float*>(p) : nullptr;
  });
  *err = g_setup_err[dev];
  return g_scratch_ptr[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

sage_status sage_smooth_quant_qk_noalloc(const sage_view* q, const sage_view* k, const sage_quantized* qz,
                                         void* stream) {
  if (!q || !k || !qz || !q->data || !k->data) return SAGE_ERR_INVALID_ARG;
  const int64_t n = q->n_tokens, h = q->n_heads, d = q->head_dim;
  if (n <= 0 || h <= 0 || d <= 0) return SAGE_ERR_INVALID_ARG;
  if (k->n_tokens != n || k->n_heads != h || k->head_dim != d) return SAGE_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SAGE_ERR_UNSUPPORTED;
  // Beyond the fixed array: refuse before touching the device.
  if (static_cast<size_t>((n + 127) / 128) * static_cast<size_t>(h) * static_cast<size_t>(d) >
      kNoAllocScratchFloats)
    return SAGE_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SAGE_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  float* scratch = device_scratch(dev, &e);
  if (e != cudaSuccess || !scratch) return SAGE_ERR_CUDA;
  if (!aligned16(scratch)) return SAGE_ERR_ALIGNMENT;
  // The argument checks and the three launches of sage_smooth_quant_qk, with the scratch
  // pointer above in place of a caller workspace.
  return sage_smooth_quant_qk(q, k, qz, scratch, kNoAllocScratchFloats * sizeof(float), stream);
}

}  // extern "C"
