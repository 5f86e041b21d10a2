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

#include "sage_internal.h"

namespace {

// 16 MiB: enough for the pages' call (ceil(37810/128) * 56 * 128 = 2,121,728 floats).
constexpr size_t kNoAllocScratchFloats = size_t(4) << 20;

// Per-128-token column partials of K.  Every element a call reads is written earlier in the
// same call, so nothing needs clearing between calls.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

sage_status sage_smooth_quant_qk_noalloc(const sage_view* q, const sage_view* k, const sage_quantized* qz,
                                         void* stream) {
  // The argument checks of sage_smooth_quant_qk first, so a bad view or shape gets the same
  // status from both entry points; then the limit of the fixed array, before touching the device.
  sage_status st = sage::check_smooth_quant_qk_args(q, k, qz);
  if (st != SAGE_OK) return st;
  const int64_t n = q->n_tokens, h = q->n_heads, d = q->head_dim;
  if (static_cast<size_t>((n + 127) / 128) * static_cast<size_t>(h) * static_cast<size_t>(d) >
      kNoAllocScratchFloats)
    return SAGE_ERR_WORKSPACE;
  // The host-side name g_noalloc_scratch is not a device address: the kernels get the address
  // cudaGetSymbolAddress returns with the caller's device current.  It is looked up on every
  // call (a host-side query that does not synchronise), so a pointer from an earlier context --
  // before a cudaDeviceReset, say -- is never reused, and a failed lookup is not remembered.
  // The first call in a process may load the library's device code: make it before any stream
  // capture on that device.
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SAGE_ERR_CUDA;
  if (!aligned16(p)) return SAGE_ERR_ALIGNMENT;
  // The three launches of sage_smooth_quant_qk, with the array in place of a caller workspace.
  return sage_smooth_quant_qk(q, k, qz, p, kNoAllocScratchFloats * sizeof(float), stream);
}

}  // extern "C"
