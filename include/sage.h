/*
 * sage.h -- C ABI of the GB300 (sm_103a) quantised-attention library `libsage_gb300.so`.
 *
 * The library computes SageAttention2-style non-causal multi-head attention over one
 * packed token sequence: per-head K mean smoothing, symmetric INT8 quantisation of Q
 * (one scale per head and 128-row block) and of K - mean (per head and 64-row block),
 * FP8 E4M3 quantisation of V (per head and channel), then a fused kernel that forms the
 * exact integer QK^T on the tensor cores, runs an fp32 online softmax, multiplies E4M3 P
 * by E4M3 V with fp32 accumulation and writes bf16 O.
 *
 * Page references: the call is the Sage2 attention of block 24 profiled in
 * "gb10-sampling-component-profile-1344x768-124f-seed440420.json"
 * (attention_internal_p50_milliseconds.sage2: qk_quantize, v_quantize, attention_forward,
 * framework_and_k_smoothing_estimate) at q_shape [1, 37810, 56, 128]
 * ("gb10-sage2-p0-interleave-softmax-latency.json", key q_shape), and it reads Q, K, V as
 * strided NHD views of the token-major QKV projection with no transposed copies and
 * writes a contiguous NHD output that the next projection reads as [N, H*D]
 * ("gb10-sage-strided-nhd-summary-1344x768-124f-seed440420.json", key dataflow).
 *
 * General rules for every entry point:
 *  - All pointers are DEVICE pointers unless a parameter says "host".  The caller owns
 *    every buffer (inputs, outputs, code buffers, workspace); the library allocates no
 *    device memory and keeps no per-call state.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL means the legacy default stream)
 *    and the call returns without waiting, except sage_check_device_status.
 *  - Arguments are checked before anything is launched; a failed check returns a status
 *    and launches nothing.  Nothing aborts or throws.  SAGE_ERR_CUDA wraps a failed launch
 *    (cudaGetLastError after the launch).
 *  - Batch is 1 (the pages' call has batch 1).  head_dim must be 64 or 128.  Q, K and V
 *    must agree in n_tokens, n_heads and head_dim.
 *  - N_pad = ceil(n_tokens / 128) * 128.  Code buffers hold N_pad rows; pad rows get code 0.
 */
#ifndef SAGE_GB300_H
#define SAGE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sage_status {
  SAGE_OK = 0,
  SAGE_ERR_INVALID_ARG = 1,     /* null pointer, non-positive size, mismatched shapes */
  SAGE_ERR_ALIGNMENT = 2,       /* pointer not 16-byte aligned or stride not a multiple of 8 elements */
  SAGE_ERR_UNSUPPORTED = 3,     /* head_dim not in {64, 128}; n_tokens > 2^22, n_heads > 4096 or
                                   n_heads * N_pad >= 2^30 (every TMA row coordinate in int32) */
  SAGE_ERR_WORKSPACE = 4,       /* workspace pointer null or smaller than required */
  SAGE_ERR_CUDA = 5,            /* a CUDA runtime call or kernel launch failed */
  SAGE_ERR_DEVICE_TIMEOUT = 6   /* a bounded device-side wait expired (see sage_check_device_status) */
} sage_status;

/* A bf16 [n_tokens, n_heads, head_dim] view with unit channel stride: element (t, h, c)
 * lives at ((const uint16_t*)data)[t * stride_token + h * stride_head + c].
 * data must be 16-byte aligned and both strides multiples of 8 elements (16 bytes), so
 * that every (t, h) row can be read with 16-byte vector loads.  Examples: a contiguous
 * NHD tensor has strides (H*D, D); a Q/K/V slice of a token-major [N, 3*H*D] projection
 * buffer has strides (3*H*D, D); an HND-contiguous tensor has strides (D, N*D). */
typedef struct sage_view {
  const void* data;
  int64_t n_tokens;
  int64_t n_heads;
  int64_t head_dim;
  int64_t stride_token;
  int64_t stride_head;
} sage_view;

/* Quantised operands produced by sage_smooth_quant_qk / sage_quant_v and consumed by
 * sage_attn_fwd_quantized.  Layouts (all row-major):
 *   q_codes  [H][N_pad][D]  INT8 codes in [-127, 127] held as IEEE fp16 (uint16 bits).
 *            sm_103a has no 8-bit integer MMA kind; every integer |c| <= 2048 is exact
 *            in fp16, and the fp16 MMA with fp32 accumulation reproduces the integer dot
 *            products exactly (|QK^T| <= 128 * 127^2 < 2^21).
 *   q_scales [H][N_pad/q_block] fp32: one scale per q_block consecutive rows
 *   k_codes  [H][N_pad][D]  as q_codes, codes of K - k_mean
 *   k_scales [H][N_pad/64]  fp32
 *   k_mean   [H][D]         fp32
 *   v_codes  [H][D][N_pad]  keys contiguous (the K-major B operand of P.V): FP8 E4M3 bytes
 *            (v_format 0), or INT8 codes in [-127, 127] held as fp16 (v_format 1; the buffer
 *            then holds 2 * H * D * N_pad bytes)
 *   v_scales [H][D]         fp32
 *   q_block  rows per Q scale: 0 or 128 (the method's default, one scale per 128-row block
 *            as in the pages' call), or 64, 32, 16, 8, 4, 2, 1.  32 is the per-warp
 *            granularity of the pages' recorded kernel configuration ("warp_q": 32 in the
 *            scheduler of "gb10-sage2-p0-interleave-softmax-latency.json"); 1 is one scale
 *            per row.  Finer blocks cost nothing in the attention kernel (each softmax
 *            thread owns one row) and lower the quantisation error of Q on inputs with
 *            outlier rows.  Any other value: SAGE_ERR_INVALID_ARG.  sage_attn_fwd always
 *            uses 128.
 *   v_format 0: the method's FP8 path (E4M3 V, P = E4M3(448 p), kind::f8f6f4 P.V).
 *            1: the INT8 P.V variant timed on the sampling-component page
 *            (sol_int8_qk_pv_*, v_int8_quantize): V as INT8 codes with scale amax / 127 and
 *            P = rint(127 p) in [0, 127], both held as fp16 and multiplied with the fp16 MMA;
 *            every integer product sum of one 16-key step is exact in the fp32 accumulator.
 *            Any other value: SAGE_ERR_INVALID_ARG.  sage_attn_fwd always uses 0.
 *   v_mean   NULL: V is quantised as it is.  Otherwise [H][D] fp32, written by sage_quant_v:
 *            V smoothing -- the channel mean of V (summed in the order of the K mean) is
 *            taken out of V before its scales and codes are formed, and the attention adds it
 *            back to every output row (softmax rows sum to 1).  It lowers the quantisation
 *            error of V with a large per-channel offset.  sage_attn_fwd leaves it NULL.
 * All of these pointers must be 16-byte aligned, and the buffers must not overlap one another
 * (the calls write several of them at once); equal q_codes and k_codes pointers are refused
 * with SAGE_ERR_INVALID_ARG. */
typedef struct sage_quantized {
  uint16_t* q_codes;
  float* q_scales;
  uint16_t* k_codes;
  float* k_scales;
  float* k_mean;
  uint8_t* v_codes;
  float* v_scales;
  int64_t q_block;
  int64_t v_format;
  float* v_mean;
} sage_quantized;

/* Human-readable name of a status code (static storage, never NULL). */
const char* sage_status_string(sage_status status);

/* Bytes of scratch that sage_smooth_quant_qk and sage_quant_v need in `ws`: per-128-token
 * column partials of K (sums) or V (absolute maxima), 4 * ceil(N/128) * H * D bytes each,
 * plus alignment slack. */
size_t sage_quant_scratch_bytes(int64_t n_tokens, int64_t n_heads, int64_t head_dim);

/* Bytes of workspace sage_attn_fwd needs: the sage_quantized buffers above, the scratch of
 * sage_quant_scratch_bytes and a 256-byte device status block, each 256-byte aligned. */
size_t sage_workspace_bytes(int64_t n_tokens, int64_t n_heads, int64_t head_dim);

/* Bytes of the status block that sage_attn_fwd_quantized takes. */
size_t sage_status_block_bytes(void);

/* K smoothing and INT8 quantisation of Q and K (the pages' framework_and_k_smoothing and
 * qk_quantize stages).
 *   k_mean[h][c] = fp32(total / N) in fp64: each 128-token chunk summed in fp32 in
 *                  ascending token order; the chunk sums summed in fp64 in 8 groups of
 *                  ceil(chunks / 8) consecutive chunks, the groups added in ascending order;
 *   Q: per (h, q_block-row block; 128 when qz->q_block is 0) scale = fl32(amax / 127),
 *      code = clamp(rint(fl32(x / scale)), -127, 127) with IEEE division; an all-zero
 *      block (also one wholly in the padding) has scale 0 and codes 0;
 *   K: the same on fl32(k - k_mean[h][c]) per (h, 64-row block).
 * Writes qz->q_codes, q_scales, k_codes, k_scales, k_mean.  ws: >= sage_quant_scratch_bytes,
 * 16-byte aligned, contents ignored and overwritten. */
sage_status sage_smooth_quant_qk(const sage_view* q, const sage_view* k, const sage_quantized* qz,
                                 void* ws, size_t ws_bytes, void* stream);

/* Same computation and outputs as sage_smooth_quant_qk, for callers that cannot allocate
 * device memory: plugin or custom-operator interfaces that receive only their input and
 * output buffers from a host framework owning all device memory, and code that must not call
 * cudaMalloc / cudaFree because those calls can synchronise the whole device.  The pages
 * have no counterpart; it exists for such callers only.
 *   - Scratch comes from a fixed 16 MiB array (4,194,304 floats) in the library's own device
 *     memory, which every GPU that loads the library holds until the process exits.  Nothing
 *     is allocated: no cudaMalloc, no cudaFree, no allocating library call.
 *   - Limit: ceil(n_tokens / 128) * n_heads * head_dim <= 4,194,304 (the pages' call uses
 *     2,121,728).  Larger problems return SAGE_ERR_WORKSPACE and nothing is launched.
 *   - Each call looks up the array's device address with the caller's device current (a
 *     host-side query that does not synchronise), so the address stays right after a device
 *     reset.  The first call in a process may load the library's device code: make the first
 *     call on each device before any stream capture begins.
 *   - Every call on a device uses the same array, so calls that can overlap on the GPU (other
 *     streams, other host threads) race: serialise them.  No element needs to start at zero:
 *     each call writes every scratch element it reads.
 * Errors: the argument checks of sage_smooth_quant_qk come first and give the same statuses
 * (e.g. SAGE_ERR_UNSUPPORTED for n_tokens > 2^22); then the limit above (SAGE_ERR_WORKSPACE);
 * SAGE_ERR_CUDA if the address lookup or a launch fails. */
sage_status sage_smooth_quant_qk_noalloc(const sage_view* q, const sage_view* k, const sage_quantized* qz,
                                         void* stream);

/* Quantisation of V (the pages' v_quantize stage), per (h, c) over the N tokens, of
 * x = v (qz->v_mean NULL) or x = fl32(v - mean[h][c]) (V smoothing: qz->v_mean receives the
 * mean first, computed exactly as k_mean is):
 *   v_format 0: scale = fl32(max_t |x| / 448), code = E4M3 round-to-nearest-even, saturating,
 *               of fl32(x / scale);
 *   v_format 1: scale = fl32(max_t |x| / 127), code = clamp(rint(fl32(x / scale)), -127, 127)
 *               held as fp16;
 * an all-zero channel has scale 0 and codes 0; IEEE division.  Writes qz->v_codes (transposed
 * to [H][D][N_pad]), qz->v_scales and, with smoothing, qz->v_mean.  ws as for
 * sage_smooth_quant_qk. */
sage_status sage_quant_v(const sage_view* v, const sage_quantized* qz, void* ws, size_t ws_bytes,
                         void* stream);

/* K smoothing, qk_quantize and v_quantize in one call: the outputs of sage_smooth_quant_qk
 * followed by sage_quant_v, bit for bit, for any options in qz.  With the default options
 * (q_block 0 or 128, v_format 0, v_mean NULL) the K sums and the V maxima share one launch, and
 * so do the K mean and the V scales: 5 launches instead of 7, the launches of the pages'
 * framework_and_k_smoothing_estimate, qk_quantize and v_quantize stages together.  Other
 * options run the two calls in turn.  q, k, v: views of one shape.  ws: 16-byte aligned device
 * scratch of ws_bytes >= 2 * sage_quant_scratch_bytes(N, H, D), caller-owned, contents
 * irrelevant.  Errors as for the two calls. */
sage_status sage_quant_qkv(const sage_view* q, const sage_view* k, const sage_view* v, const sage_quantized* qz,
                           void* ws, size_t ws_bytes, void* stream);

/* Fused attention on quantised operands (the pages' attention_forward stage):
 *   s_ij = S_ij * q_scales[h][i/128] * k_scales[h][j/64] * sm_scale,  S = exact integer QK^T
 *   running row max m over 128-key tiles; p = exp(s - m); P8 = E4M3(448 p);
 *   l = sum of fp32 p; O and l are multiplied by exp(m_old - m_new) whenever m rises;
 *   out[i][h][c] = bf16_rn( (sum_j P8_ij * v_codes[h][c][j]) * v_scales[h][c] / (448 l) ).
 * With v_format 1: P8 = rint(127 p) and the division is by 127 l.  With v_mean set:
 * + v_mean[h][c] inside the rounding.
 * out: bf16, element (t, h, c) at out[t * out_stride_token + h * out_stride_head + c];
 * 16-byte aligned, strides multiples of 8 elements; rows >= n_tokens are never written.
 * status_block: >= sage_status_block_bytes() bytes of device memory, zeroed by the caller
 * once; the kernel records expired device waits there (sage_check_device_status). */
sage_status sage_attn_fwd_quantized(int64_t n_tokens, int64_t n_heads, int64_t head_dim,
                                    const sage_quantized* qz, float sm_scale, void* out,
                                    int64_t out_stride_token, int64_t out_stride_head,
                                    void* status_block, void* stream);

/* The qk_transform stage upstream of the quantisation: RMSNorm and a rotary embedding of Q
 * and K, in place on their strided views (the strided-NHD dataflow of
 * "gb10-sage-strided-nhd-summary-1344x768-124f-seed440420.json", key dataflow.qk_transform;
 * timed as rms_rope in the block-24 profile of the sampling-component page).  Per token t
 * and head h of each of Q and K, in fp32, every product and sum rounded on its own:
 *   ms = (sum_c x_c^2) / D, the sum as D/8 partial sums of 8 consecutive channels (each in
 *        channel order) folded pairwise, partial g + partial g + s for s = D/16, ..., 1;
 *   r  = 1 / sqrt(ms + eps) (IEEE sqrt and division);  y_c = (x_c * r) * gamma[c];
 *   z_2i = y_2i cos[t][i] - y_2i+1 sin[t][i],  z_2i+1 = y_2i sin[t][i] + y_2i+1 cos[t][i];
 *   x_c <- bf16 round-to-nearest-even(z_c).
 * The pages give neither the norm weights nor the rotary table: both are caller inputs.
 *   q, k: views as above (same shape); their data is WRITTEN in place.
 *   gamma_q, gamma_k: device fp32 [D] norm weights of Q and K.
 *   rope_cos, rope_sin: device fp32 [n_tokens][D/2]: cos and sin of the angle that turns
 *     channel pair (2i, 2i+1) of token t (the caller's rotary table, e.g. 3-D positions).
 *   eps: >= 0 and finite (a row of zeros with eps = 0 gives NaN, as the formula does).
 * All device pointers 16-byte aligned.  Q and K may be slices of one projection buffer; they
 * must not overlap each other. */
sage_status sage_qk_rmsnorm_rope(const sage_view* q, const sage_view* k, const float* gamma_q,
                                 const float* gamma_k, const float* rope_cos, const float* rope_sin,
                                 float eps, void* stream);

/* The qk_transform fused into the K smoothing and Q / K quantisation: the same outputs, bit for
 * bit, as sage_qk_rmsnorm_rope(q, k, ...) followed by sage_smooth_quant_qk(q, k, qz, ...), but
 * q and k are only READ -- the fusion of the rms_rope stage into the quantisation prologue.
 * K is transformed once, by the K-mean pass, which leaves the transformed rows in qz->q_codes
 * for K's quantisation to read back; Q is transformed as its quantise kernel loads it, and
 * its codes then replace that scratch content.  The transformed Q is never written, and Q and
 * K are not written back in place.  Arguments: q, k, gamma_*, rope_*, eps as for
 * sage_qk_rmsnorm_rope; qz, ws, ws_bytes as for sage_smooth_quant_qk (any q_block).  Errors
 * as for both; after an error qz->q_codes may hold transformed K rows. */
sage_status sage_smooth_quant_qk_rmsnorm_rope(const sage_view* q, const sage_view* k, const float* gamma_q,
                                              const float* gamma_k, const float* rope_cos, const float* rope_sin,
                                              float eps, const sage_quantized* qz, void* ws, size_t ws_bytes,
                                              void* stream);

/* The whole path: the Sage2 call whose stages "gb10-sampling-component-profile-1344x768-124f-
 * seed440420.json" times under attention_internal_p50_milliseconds.sage2 (K smoothing,
 * qk_quantize, v_quantize, attention_forward; total_excluding_external_layout), as
 * sage_quant_qkv and sage_attn_fwd_quantized (6 launches) on buffers carved from ws
 * (>= sage_workspace_bytes, 256-byte aligned, caller-owned; the status block at its start must
 * be zeroed once by the caller before first use).  Arguments, layouts and errors as for those
 * three calls; a device timeout is reported through the status block at the start of ws. */
sage_status sage_attn_fwd(const sage_view* q, const sage_view* k, const sage_view* v, float sm_scale,
                          void* out, int64_t out_stride_token, int64_t out_stride_head, void* ws,
                          size_t ws_bytes, void* stream);

/* Unquantised reference attention in bf16 inputs / fp32 arithmetic:
 * out = bf16_rn(softmax(sm_scale * q k^T) v), the dense attention the pages use as the
 * quality anchor (quality_gates.sol_fully_dense_tau_minus_100_relative_l2_vs_sage2).
 * A correctness path, not tuned. */
sage_status sage_attn_dense_bf16(const sage_view* q, const sage_view* k, const sage_view* v,
                                 float sm_scale, void* out, int64_t out_stride_token,
                                 int64_t out_stride_head, void* stream);

/* Bytes of workspace sage_attn_dense_bf16_tc needs: a 256-byte device status block and V
 * transposed, H * D * N_pad bf16 values (N_pad = N rounded up to 128), 256-byte aligned.
 * 0 for a shape the library does not take. */
size_t sage_dense_workspace_bytes(int64_t n_tokens, int64_t n_heads, int64_t head_dim);

/* The same dense attention on the tensor cores, for timing the quantised path against
 * unquantised attention on the same GPU (the pages time their dense path:
 * "gb10-sampling-component-profile-1344x768-124f-seed440420.json",
 * quality_gates.sol_fully_dense_tau_minus_100_p50_milliseconds).  Flash-attention schedule of the fused kernel: 128-key tiles,
 * S = q k^T from bf16 operands with fp32 accumulation; m the running row max of S;
 * p = exp2(S * sm_scale * log2 e - m); P = bf16_rn(p); l = sum of the unrounded p;
 * O = sum P v with fp32 accumulation (rescaled by exp2(m_old - m_new) when m rises);
 * out = bf16_rn(O / l).  Rounding P to bf16 makes it less exact than sage_attn_dense_bf16:
 * per element |out - exact| <= 2^-8 max_t |v[t][h][c]| plus fp32 rounding.
 * Views, output and errors as for sage_attn_dense_bf16.  ws: caller-owned, 256-byte aligned,
 * >= sage_dense_workspace_bytes (sage_workspace_bytes is enough); the status block at its
 * start must be zeroed once by the caller before first use, and reports a device timeout
 * (read it with sage_check_device_status).  Two launches: V's transpose into ws, then the
 * attention. */
sage_status sage_attn_dense_bf16_tc(const sage_view* q, const sage_view* k, const sage_view* v,
                                    float sm_scale, void* out, int64_t out_stride_token,
                                    int64_t out_stride_head, void* ws, size_t ws_bytes, void* stream);

/* Test hook: the integer S = Qc Kc^T (the QK^T product inside attention_forward of the call
 * above) of head `head`, query rows [i0, i0 + 128 * row_tiles)
 * and keys [j0, j0 + 128 * col_tiles), produced by the same tensor-core QK^T code path
 * as sage_attn_fwd_quantized and converted to int32.  i0, j0 multiples of 128 and inside
 * N_pad.  out: int32 [128 * row_tiles][128 * col_tiles] row-major. */
sage_status sage_debug_qk_int32(int64_t n_tokens, int64_t n_heads, int64_t head_dim,
                                const sage_quantized* qz, int64_t head, int64_t i0, int64_t j0,
                                int64_t row_tiles, int64_t col_tiles, int32_t* out,
                                void* status_block, void* stream);

/* Test hook for the failure path: one thread waits, with the kernels' bounded mbarrier wait,
 * on a barrier nothing arrives on.  After limit_ns (1 .. 1e10) nanoseconds the wait gives up
 * and records SAGE_ERR_DEVICE_TIMEOUT (where = 10) in the status block; nothing faults or
 * hangs.  Read the result with sage_check_device_status. */
sage_status sage_debug_wait_timeout(void* status_block, int64_t limit_ns, void* stream);

/* Measurement hook: the tensor-core rate of the MMA instructions the fused attention issues,
 * i.e. the ceiling its roofline is read against.  `ctas` CTAs (one per SM: 128 threads, 512 TMEM
 * columns, ~49 KB shared memory) each issue `iters` rounds of `mode` back to back on zero operands
 * and wait for the last; the caller times the call (e.g. CUDA events on `stream`).  FLOPs per CTA
 * and round, 2 M N K per MMA:
 *   mode 0  8 x kind::f16 128x128x16, both operands in shared memory (QK^T steps)  4,194,304
 *   mode 1  8 x kind::f8f6f4 E4M3 128x128x32, A in tensor memory (P.V steps)       8,388,608
 *   mode 2  8 QK^T steps then 4 P.V steps: one key tile of one 128-row Q tile      8,388,608
 *   mode 3  8 x kind::f8f6f4 E4M3 128x256x32, both in shared memory (E4M3 peak)  16,777,216
 *   mode 4  8 x kind::f16 128x256x16, both in shared memory (16-bit peak)          8,388,608
 *   mode 5  8 x kind::f8f6f4 E4M3 128x64x32, A in tensor memory (P.V at D = 64)    4,194,304
 *   mode 6  4 QK^T steps then 4 P.V steps at D = 64: one key tile of one Q tile    4,194,304
 * iters 1 .. 1e8, ctas 1 .. 65535.  A wait that exceeds 2 s is recorded in status_block as for
 * the other kernels (read it with sage_check_device_status).  Not part of the attention path. */
sage_status sage_measure_mma_rate(int64_t mode, int64_t iters, int64_t ctas, void* status_block, void* stream);

/* Waits for `stream`, reads the status block (device pointer) and returns SAGE_OK,
 * SAGE_ERR_DEVICE_TIMEOUT (a bounded wait expired; the block is then cleared) or
 * SAGE_ERR_CUDA.  If where != NULL (host), *where receives the code of the wait that
 * expired: 1 Q tile, 2 K/V tile loaded, 3 K/V slot free, 4 S ready, 5 P ready, 6 P.V done,
 * 7/8 the S-tile hook's load / MMA, 10 the timeout hook; 0 if none.  This is the one call that
 * synchronises. */
sage_status sage_check_device_status(void* status_block, void* stream, int32_t* where);

/* The same call as sage_check_device_status, under the name "get device status": reads (and on a
 * recorded timeout clears) the device status word of status_block after `stream` drains. */
sage_status sage_get_device_status(void* status_block, void* stream, int32_t* where);

#ifdef __cplusplus
}
#endif

#endif /* SAGE_GB300_H */
