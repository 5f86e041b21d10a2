// attn_fwd.cu -- fused quantised attention forward for sm_103a (tcgen05 + TMEM + TMA).
//
// Computes the attention_forward stage of the Sage2 call profiled in
// "gb10-sampling-component-profile-1344x768-124f-seed440420.json"
// (attention_internal_p50_milliseconds.sage2.attention_forward) on operands made by
// quant.cu: S = exact integer QK^T (INT8 codes held in fp16, kind::f16 MMA, fp32
// accumulator), an fp32 online softmax on S * s_q * s_k * sm_scale, P = E4M3(448 p) kept in
// tensor memory, O += P.V with E4M3 V (kind::f8f6f4 MMA, fp32 accumulator), and a bf16
// epilogue O * s_v / l.  The pages' kernel (an sm_89 build, cta_q 128 / cta_k 64 / 128
// threads per CTA; "gb10-sage2-p0-interleave-softmax-latency.json", key scheduler) is prior
// art only: this kernel is organised around Blackwell's tensor memory instead.
//
// CTA = 256 query rows of one head (two 128-row tiles t = 0, 1) and every 128-key tile of
// that head.  Warp roles (384 threads):
//   warp 0      TMA producer: Q tiles once, then K/V tiles into a kStages-deep ring
//   warp 1      MMA issuer (one thread): S_t = Q_t K^T, O_t += P_t V
//   warp 2      TMEM allocator
//   warps 4-7   softmax + epilogue of tile 0 (thread = row = TMEM lane)
//   warps 8-11  softmax + epilogue of tile 1
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256, 256+D), O_1 [256+D, 256+2D).
// P_t (E4M3, 4 keys per 32-bit column) overwrites columns [0,32) of S_t and is the A
// operand of the P.V MMA straight from TMEM.  At D = 64 the columns from 384 on are free and
// P_t has its own there (P_0 at 384, P_1 after it): S_t of the next key tile is then issued as
// soon as the softmax has read S_t, and P.V no longer sits between a softmax and the next S.
//
// The INT8 P.V variant (kPv16; the sampling-component page's sol_int8_qk_pv_* /
// v_int8_quantize) keeps the same schedule with V as INT8 codes and P = rint(127 p), both held
// as fp16 (integers |c| <= 127 are exact): P_t takes columns [0,64) of S_t, P.V is 8 kind::f16
// MMAs of K = 16 per tile (each 16-key partial sum <= 16 * 127^2 is exact in fp32), and a V
// tile is two 64-key panels, so the K/V ring holds 2 stages at D = 128.
//
// V smoothing (v_mean set): the epilogue adds the channel mean taken out of V.
//
// Online softmax with P in E4M3: P is encoded against the current running max, so p <= 1
// and 448 p never overflows; whenever a row's max rises, O and l of that row are
// multiplied by exp2(m_old - m_new) before the next P.V is issued (an exact rescale on
// every increase).
//
// Every mbarrier wait is bounded (global-timer limit); on expiry the thread records the
// wait in the status block, raises the CTA's abort flag and every role unwinds to the
// common exit, which frees the tensor memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "sage_internal.h"
#include "sm103_ptx.cuh"

namespace sage {
namespace {

constexpr int kBM = 128;   // query rows per tile
// Register split of the 384-thread CTA, launched at 168 registers per thread (384 x 168 =
// 64512): the role warpgroup (warps 0-3) drops, the two softmax warpgroups rise.  Every split
// below compiles without spills; among the splits that do, these measured fastest (D = 128:
// 80 / 200, 21.90 ms against 21.97 for 56 / 224 on the video shape; D = 64: 72 / 216, 1.592
// against 1.611 ms on strided64).  The 16-bit P.V schedule's producer (two V panels) and issuer
// (eight P.V MMAs) spill at 56: the INT8 P.V variant takes 80 / 208 at D = 128 (24.95 ms against
// 25.31 for 72 / 208) and 72 / 208 at D = 64; the dense bf16 kernel 72 / 216 (25.28 against 25.38).
constexpr int kRegsLaunch = 168;
template <int D, bool kPv16, bool kDense = false> constexpr int regs_roles() {
  return kDense ? 72 : (kPv16 ? (D == 128 ? 80 : 72) : (D == 128 ? 80 : 72));
}
template <int D, bool kPv16, bool kDense = false> constexpr int regs_softmax() {
  return kDense ? 216 : (kPv16 ? 208 : (D == 128 ? 200 : 216));
}
static_assert(128 * regs_roles<128, false>() + 256 * regs_softmax<128, false>() <= 384 * kRegsLaunch,
              "register split exceeds launch");
static_assert(128 * regs_roles<64, false>() + 256 * regs_softmax<64, false>() <= 384 * kRegsLaunch,
              "register split exceeds launch");
static_assert(128 * regs_roles<128, true>() + 256 * regs_softmax<128, true>() <= 384 * kRegsLaunch,
              "register split exceeds launch");
static_assert(128 * regs_roles<64, true>() + 256 * regs_softmax<64, true>() <= 384 * kRegsLaunch,
              "register split exceeds launch");
static_assert(128 * regs_roles<128, true, true>() + 256 * regs_softmax<128, true, true>() <= 384 * kRegsLaunch,
              "register split exceeds launch");
constexpr int kBN = 128;   // keys per tile
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLog2_448 = 8.807354922057604f;     // log2(448): P is encoded as E4M3(448 p)
constexpr float kLog2_127 = 6.988684686772166f;     // log2(127): INT8 P = rint(127 p)
// 2^23 + 0x6400: in [2^23, 2^24) the fp32 ulp is 1, so fl32(x + kRintMagic) = kRintMagic +
// rint(x) for 0 <= x < 2^15 (ties to even: kRintMagic is even), and its low 16 bits are then
// 0x6400 + rint(x), the fp16 number 1024 + rint(x) for rint(x) < 1024.
constexpr float kRintMagic = 8414208.0f;

// kPv16: the INT8 P.V variant -- V codes held as fp16 (2 bytes per key), P as fp16 codes.
template <int D, bool kPv16 = false>
struct Cfg {
  static constexpr int kPanels = D / 64;                 // 128-byte swizzle panels per fp16 row
  static constexpr int kPanelBytes = 128 * 128;          // 128 rows x 128 B
  static constexpr int kQTileBytes = kBM * D * 2;
  static constexpr int kKTileBytes = kBN * D * 2;
  static constexpr int kVPanelBytes = D * 128;           // D channel rows x 128 B (64 fp16 keys)
  static constexpr int kVTileBytes = D * kBN * (kPv16 ? 2 : 1);
  static constexpr int kStageBytes = kKTileBytes + kVTileBytes;
  static constexpr int kStages = D == 128 ? (kPv16 ? 2 : 3) : 4;
  static constexpr int kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  // At D = 64 the O accumulators end at column 384 and [384, 512) is free: P_t gets its own
  // columns there (32 for E4M3, 64 for fp16 codes) instead of overwriting S_t, so the next S_t
  // may be computed as soon as the softmax has read S_t into registers.
  static constexpr bool kSepP = D == 64;
  static constexpr int kColP0 = 384, kColP1 = 384 + (kPv16 ? 64 : 32);
  static constexpr int kTmemCols = 512;
  static constexpr int kBarOffset = 2 * kQTileBytes + kStages * kStageBytes;
  // q_full, kv_full[S], kv_empty[S], s_full[2], p_full[2], pv_done[2], s_free[2], mma_final
  static constexpr int kNumBars = 1 + 2 * kStages + 2 + 2 + 2 + 2 + 1;
  static constexpr int kSmemBytes = kBarOffset + kNumBars * 8 + 16 + 1024;   // + slack for 1024-B alignment
};

struct AttnParams {
  int n, npad, h;
  int q_shift;             // log2 of the rows per Q scale
  const float* q_scales;   // [H][npad >> q_shift]
  const float* k_scales;   // [H][npad/64]
  const float* v_scales;   // [H][D]
  const float* v_mean;     // [H][D] or null: added to every output row (V smoothing)
  float sm_scale_log2;     // sm_scale * log2(e)
  uint16_t* out;           // bf16
  int64_t ost, osh;
  int tma_out;             // 1: the epilogue stores through the output tensor map
  int32_t* status;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void record_error(int32_t* status, int32_t where, volatile int* abort_flag) {
  if (atomicCAS(status, 0, 1) == 0) status[1] = where;
  *abort_flag = 1;
}

// Bounded wait usable by a whole warp: every lane waits, and the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t limit) {
  bool ok = mbar_wait(bar, parity, limit);
  return __all_sync(0xffffffffu, ok);
}

// Max of 64 consecutive fp32 values (as bits): four independent chains of 3-input maxima
// covering s[0..11], then s[12..59] eight at a time, then s[60..63].
__device__ __forceinline__ float block_max64(const uint32_t* s) {
  auto f = [s](int i) { return __uint_as_float(s[i]); };
  float a = fmax3(f(0), f(1), f(2)), b = fmax3(f(3), f(4), f(5));
  float c = fmax3(f(6), f(7), f(8)), d = fmax3(f(9), f(10), f(11));
#pragma unroll
  for (int k = 12; k < 60; k += 8) {
    a = fmax3(a, f(k), f(k + 1));
    b = fmax3(b, f(k + 2), f(k + 3));
    c = fmax3(c, f(k + 4), f(k + 5));
    d = fmax3(d, f(k + 6), f(k + 7));
  }
  a = fmax3(a, f(60), f(61));
  b = fmax3(b, f(62), f(63));
  return fmaxf(fmax3(a, b, c), d);
}

// kind::f16 operand format bf16 (code 1) for A and B; the default code 0 is fp16.
constexpr uint32_t kIdescBf16 = (1u << 7) | (1u << 10);

// S[tmem d_col] = Q_tile(sq) . K_tile(sk)^T over D channels: D/16 MMAs of 128x128x16 (fp16
// operands, or bf16 with kBf16).
// ql, kl: the descriptor low words (sdesc_lo) of the Q and K tiles.
template <int D, bool kBf16 = false>
__device__ __forceinline__ void issue_qk_lo(uint32_t d_tmem, uint32_t ql, uint32_t kl) {
  constexpr uint32_t idesc = idesc_f32acc(kBM, kBN) | (kBf16 ? kIdescBf16 : 0u);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off16 = ((kk >> 2) * Cfg<D>::kPanelBytes + (kk & 3) * 32) >> 4;
    mma_f16_ss(d_tmem, sdesc_of_lo(ql + off16), sdesc_of_lo(kl + off16), idesc, kk > 0 ? 1u : 0u);
  }
}
template <int D, bool kBf16 = false>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t sq, uint32_t sk) {
  issue_qk_lo<D, kBf16>(d_tmem, sdesc_lo(sq), sdesc_lo(sk));
}

// O[tmem] (+)= P[tmem] . V_tile(sv): 4 MMAs of 128 x D x 32 (E4M3), or with kPv16 8 MMAs of
// 128 x D x 16 on 16-bit values, fp16 codes or with kBf16 bf16 (P: 16 keys per 8 TMEM
// columns; V: two 64-key panels).
// vl: the descriptor low word (sdesc_lo) of the V tile.
template <int D, bool kPv16, bool kBf16 = false>
__device__ __forceinline__ void issue_pv_lo(uint32_t o_tmem, uint32_t p_tmem, uint32_t vl, bool first) {
  constexpr uint32_t idesc = idesc_f32acc(kBM, D) | (kBf16 ? kIdescBf16 : 0u);
  if (kPv16) {
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk)
      mma_f16_ts(o_tmem, p_tmem + kk * 8,
                 sdesc_of_lo(vl + (((kk >> 2) * Cfg<D, true>::kVPanelBytes + (kk & 3) * 32) >> 4)), idesc,
                 (first && kk == 0) ? 0u : 1u);
  } else {
#pragma unroll
    for (int kk = 0; kk < kBN / 32; ++kk)
      mma_f8_ts(o_tmem, p_tmem + kk * 8, sdesc_of_lo(vl + ((kk * 32) >> 4)), idesc, (first && kk == 0) ? 0u : 1u);
  }
}

// Four INT8 P codes rint(p'_k) (p' = 127 p) as two fp16x2 words, the lower key in the low half.
__device__ __forceinline__ void p_codes_f16(const float pp[4], uint64_t magic2, uint32_t& w01, uint32_t& w23) {
  float a0, a1, a2, a3;
  f2_unpack(f2_add(f2_pack(pp[0], pp[1]), magic2), a0, a1);
  f2_unpack(f2_add(f2_pack(pp[2], pp[3]), magic2), a2, a3);
  uint32_t h01, h23;
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(h01) : "r"(__float_as_uint(a0)), "r"(__float_as_uint(a1)));
  asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(h23) : "r"(__float_as_uint(a2)), "r"(__float_as_uint(a3)));
  // (1024 + c) - 1024 in fp16: exact.
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(w01) : "r"(h01), "r"(0x64006400u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(w23) : "r"(h23), "r"(0x64006400u));
}

// Four probabilities p_k as two bf16x2 words (round to nearest even), the lower key in the low half.
__device__ __forceinline__ void p_bf16(const float pp[4], uint32_t& w01, uint32_t& w23) {
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w01) : "f"(pp[1]), "f"(pp[0]));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w23) : "f"(pp[3]), "f"(pp[2]));
}

// One 128-key tile j of the online softmax for the calling thread's row (= TMEM lane):
//   reads S from TMEM; forms the tile max on raw S per 64-key half (c >= 0 and rounding is
//   monotone, so max_k fl(S_k c) = fl(c max_k S_k)); writes P = E4M3(448 p) with
//   p = exp2(S c - m_new) into the first 32 columns of S (kPv16: P = rint(127 p) as fp16 into
//   the first 64); l = alpha l + sum p; and, if any row of the warp saw its max rise,
//   multiplies that row's O by alpha = exp2(m_old - m_new).
// With separate P columns (Cfg::kSepP, D = 64): S_t is released to the MMA issuer (s_free) as
//   soon as it is in registers; P goes to its own columns tP, written, like O's rescale, only
//   once P.V of tile j - 1 has finished with them (pv_done, phase (j - 1) & 1).  Returns false
//   if that wait expired.
// kTail: keys >= kvalid are excluded from the max and get p = 0.
// kDense (with kPv16): unquantised attention, P = bf16_rn(p) with p = exp2(S c - m_new) itself.
template <int D, bool kTail, bool kPv16, bool kDense = false>
__device__ __forceinline__ bool softmax_step(uint32_t tS, uint32_t tO, uint32_t tP, float c0, float c1, int kvalid,
                                             bool first, float& m, float& l, uint64_t* s_free, uint64_t* pv_done,
                                             int j, uint64_t limit) {
  constexpr bool kSep = Cfg<D, kPv16>::kSepP;
  uint32_t sr[128];
  SAGE_TMEM_LD32(tS + 0, (sr + 0));
  SAGE_TMEM_LD32(tS + 32, (sr + 32));
  SAGE_TMEM_LD32(tS + 64, (sr + 64));
  SAGE_TMEM_LD32(tS + 96, (sr + 96));
  tmem_wait_ld();
  if (kSep) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(s_free);
  }
  float mx0, mx1;
  if (!kTail) {
    mx0 = block_max64(sr);
    mx1 = block_max64(sr + 64);
  } else {
    mx0 = mx1 = -INFINITY;
#pragma unroll
    for (int k = 0; k < 64; ++k)
      if (k < kvalid) mx0 = fmaxf(mx0, __uint_as_float(sr[k]));
#pragma unroll
    for (int k = 64; k < 128; ++k)
      if (k < kvalid) mx1 = fmaxf(mx1, __uint_as_float(sr[k]));
  }
  // fmaxf drops the NaN of (-inf) * 0 for an empty half.
  const float m_new = fmaxf(m, fmaxf(mx0 * c0, mx1 * c1));
  const bool rise = !first && (m_new > m);
  const float alpha = rise ? ex2_approx(m - m_new) : 1.0f;
  m = m_new;
  // p' = 448 p = exp2(S c + log2(448) - m) (127 p with kPv16, p with kDense), two keys per fp32x2 FMA.
  constexpr float kLog2P = kDense ? 0.0f : (kPv16 ? kLog2_127 : kLog2_448);
  const uint64_t bias2 = f2_pack(kLog2P - m_new, kLog2P - m_new);
  const uint64_t magic2 = f2_pack(kRintMagic, kRintMagic);
  // Partial sums of p': one per (32-key chunk, key pair parity), so no add waits on more than
  // eight earlier ones.
  uint64_t l2[4][2];
  // With separate P columns the P words wait in registers until P.V of tile j - 1 is done.
  uint32_t pkeep[kSep ? (kPv16 ? 64 : 32) : 1];
#pragma unroll
  for (int cch = 0; cch < 4; ++cch) {
    const float cb = cch < 2 ? c0 : c1;
    const uint64_t cb2 = f2_pack(cb, cb);
    uint32_t pw[kPv16 ? 16 : 8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int k = cch * 32 + w * 4;
      float pp[4];
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), cb2, bias2), pp[0], pp[1]);
      f2_unpack(f2_fma(f2_pack(__uint_as_float(sr[k + 2]), __uint_as_float(sr[k + 3])), cb2, bias2), pp[2], pp[3]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        pp[u] = ex2_approx(pp[u]);
        if (kTail && k + u >= kvalid) pp[u] = 0.0f;
      }
      if (w == 0) {
        l2[cch][0] = f2_pack(pp[0], pp[1]);
        l2[cch][1] = f2_pack(pp[2], pp[3]);
      } else {
        l2[cch][0] = f2_add(l2[cch][0], f2_pack(pp[0], pp[1]));
        l2[cch][1] = f2_add(l2[cch][1], f2_pack(pp[2], pp[3]));
      }
      if (kDense)
        p_bf16(pp, pw[2 * w], pw[2 * w + 1]);
      else if (kPv16)
        p_codes_f16(pp, magic2, pw[2 * w], pw[2 * w + 1]);
      else
        pw[w] = pack_h2(e4m3x2(pp[0], pp[1]), e4m3x2(pp[2], pp[3]));
    }
    if (kSep) {
#pragma unroll
      for (int i = 0; i < (kPv16 ? 16 : 8); ++i) pkeep[cch * (kPv16 ? 16 : 8) + i] = pw[i];
    } else if (kPv16) {
      // All of S is in registers (tmem_wait_ld above), so P may overwrite its columns.
      SAGE_TMEM_ST16(tS + cch * 16, pw);
    } else {
      SAGE_TMEM_ST8(tS + cch * 8, pw);
    }
  }
  const uint64_t la = f2_add(f2_add(l2[0][0], l2[0][1]), f2_add(l2[1][0], l2[1][1]));
  const uint64_t lb = f2_add(f2_add(l2[2][0], l2[2][1]), f2_add(l2[3][0], l2[3][1]));
  float llo, lhi;
  f2_unpack(f2_add(la, lb), llo, lhi);
  l = l * alpha + (llo + lhi);
  if (kSep) {
    if (!first) {
      if (!warp_wait(pv_done, (j - 1) & 1, limit)) return false;
      tc_fence_after();
    }
    SAGE_TMEM_ST32(tP, pkeep);
    if (kPv16) SAGE_TMEM_ST32(tP + 32, (pkeep + 32));
  }
  // O is rescaled after P is formed, when S no longer occupies registers.  P.V of this tile
  // is issued only after p_full, so O still holds the previous tiles' sum here (with separate P
  // columns, P.V of tile j - 1 has completed: the wait above).
  if (__any_sync(0xffffffffu, rise)) {
    // The whole O row in one TMEM round trip: S no longer occupies registers here.
    const uint64_t a2 = f2_pack(alpha, alpha);
    uint32_t o[D];
#pragma unroll
    for (int c = 0; c < D; c += 32) SAGE_TMEM_LD32(tO + c, (o + c));
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < D; k += 2) {
      float lo, hi;
      f2_unpack(f2_mul(f2_pack(__uint_as_float(o[k]), __uint_as_float(o[k + 1])), a2), lo, hi);
      o[k] = __float_as_uint(lo);
      o[k + 1] = __float_as_uint(hi);
    }
#pragma unroll
    for (int c = 0; c < D; c += 32) SAGE_TMEM_ST32(tO + c, (o + c));
  }
  tmem_wait_st();
  return true;
}

// kRowQ: Q scales per 2^q_shift < 128 rows, so each softmax thread reads its own row's scale;
// otherwise one scale per 128-row tile.  Two instantiations keep the default one's code as it
// was: the per-row lookup alone measured 0.7 % slower there.
// kMean: V was smoothed, the epilogue adds p.v_mean (a separate instantiation keeps the
// default epilogue free of the extra loads).
// kDense (with kPv16, not kRowQ / kMean): unquantised attention on bf16 Q, K and V.  Q and K come
// straight from the caller's [N][H][D] views through 3-D tensor maps (rows past N read as
// zeros), V from its transpose [H][D][N_pad]; there are no Q, K or V scales (c = sm_scale log2 e,
// out = O / l), P is bf16 and both MMAs take bf16 operands.
template <int D, bool kRowQ, bool kPv16, bool kMean, bool kDense>
__device__ __forceinline__ void attn_body(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                          const CUtensorMap& omap, const AttnParams& p) {
  static_assert(!kDense || (kPv16 && !kRowQ && !kMean), "the dense path is the 16-bit P.V schedule alone");
  using C = Cfg<D, kPv16>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_skip;
  __shared__ volatile int s_abort;
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + 2 * C::kQTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOffset);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + C::kStages;
  uint64_t* s_full = kv_empty + C::kStages;
  uint64_t* p_full = s_full + 2;
  uint64_t* pv_done = p_full + 2;
  uint64_t* s_free = pv_done + 2;
  uint64_t* mma_final = s_free + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hh = blockIdx.y;
  const int q0 = blockIdx.x * 2 * kBM;
  const int ntiles = p.npad / kBN;

  if (threadIdx.x == 0) {
    s_skip = *reinterpret_cast<volatile int32_t*>(p.status);
    s_abort = 0;
    mbar_init(q_full, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(kv_full + s, 1);
      mbar_init(kv_empty + s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(s_full + t, 1);
      mbar_init(p_full + t, 128);
      mbar_init(pv_done + t, 1);
      mbar_init(s_free + t, 4);
    }
    mbar_init(mma_final, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (s_skip) return;   // an earlier CTA already failed: do no work
  if (warp == 2) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint64_t limit = p.wait_limit_ns;
  if (warp < 4) {
    regs_dec<regs_roles<D, kPv16, kDense>()>();
    if (warp == 0) {
      // ------------------------------------------------------------ TMA producer
      if (lane == 0) {
        tma_prefetch_desc(&qmap);
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&vmap);
        const int qrow = hh * p.npad + q0;
        mbar_arrive_expect_tx(q_full, 2 * C::kQTileBytes);
        for (int t = 0; t < 2; ++t)
          for (int pn = 0; pn < C::kPanels; ++pn) {
            if (kDense)
              tma_load_3d(sQ + t * C::kQTileBytes + pn * C::kPanelBytes, &qmap, q_full, pn * 64, hh, q0 + t * kBM);
            else
              tma_load_2d(sQ + t * C::kQTileBytes + pn * C::kPanelBytes, &qmap, q_full, pn * 64, qrow + t * kBM);
          }
        for (int j = 0; j < ntiles; ++j) {
          const int s = j % C::kStages;
          if (j >= C::kStages && !mbar_wait(kv_empty + s, ((j / C::kStages) - 1) & 1, limit)) {
            record_error(p.status, kWhereKvEmpty, &s_abort);
            break;
          }
          if (s_abort) break;
          uint8_t* sk = sKV + s * C::kStageBytes;
          mbar_arrive_expect_tx(kv_full + s, C::kStageBytes);
          for (int pn = 0; pn < C::kPanels; ++pn) {
            if (kDense)
              tma_load_3d(sk + pn * C::kPanelBytes, &kmap, kv_full + s, pn * 64, hh, j * kBN);
            else
              tma_load_2d(sk + pn * C::kPanelBytes, &kmap, kv_full + s, pn * 64, hh * p.npad + j * kBN);
          }
          if (kPv16) {
            for (int pn = 0; pn < 2; ++pn)
              tma_load_2d(sk + C::kKTileBytes + pn * C::kVPanelBytes, &vmap, kv_full + s, j * kBN + pn * 64, hh * D);
          } else {
            tma_load_2d(sk + C::kKTileBytes, &vmap, kv_full + s, j * kBN, hh * D);
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        const uint32_t sq = smem_u32(sQ);
        const uint32_t skv = smem_u32(sKV);
        const uint32_t colS[2] = {tmem + C::kColS0, tmem + C::kColS1};
        const uint32_t colO[2] = {tmem + C::kColO0, tmem + C::kColO1};
        const uint32_t colP[2] = {tmem + (C::kSepP ? C::kColP0 : C::kColS0), tmem + (C::kSepP ? C::kColP1 : C::kColS1)};
        // Descriptor low words: Q tile t at q_lo + t * kQLo, ring stage s's K tile at kv_lo + s * kStageLo,
        // its V tile kVLo further.
        const uint32_t q_lo = sdesc_lo(sq), kv_lo = sdesc_lo(skv);
        constexpr uint32_t kQLo = C::kQTileBytes >> 4, kStageLo = C::kStageBytes >> 4, kVLo = C::kKTileBytes >> 4;
        bool ok = mbar_wait(q_full, 0, limit) && mbar_wait(kv_full, 0, limit);
        if (!ok) record_error(p.status, kWhereQFull, &s_abort);
        if (ok) {
          tc_fence_after();
          issue_qk_lo<D, kDense>(colS[0], q_lo, kv_lo);
          tc_commit(s_full + 0);
          issue_qk_lo<D, kDense>(colS[1], q_lo + kQLo, kv_lo);
          tc_commit(s_full + 1);
        }
        // Ring stage of tile j (s) and of tile j + 1 (sn) with the kv_full phase of tile j + 1,
        // advanced once per tile.
        int s = 0, sn = 1 % C::kStages;
        uint32_t phn = 0;
        // Separate P columns: S_t of tile j + 1 is issued as soon as the softmax has read S_t of tile
        // j (s_free), P.V of tile j once P_t is written (p_full).  A softmax writes P_t of tile j + 1
        // only after P.V of tile j is done, so it never runs two tiles ahead of these waits.
        for (int j = 0; C::kSepP && ok && j < ntiles; ++j) {
          if (j + 1 < ntiles) {
            if (!mbar_wait(kv_full + sn, phn, limit)) {
              record_error(p.status, kWhereKvFull, &s_abort);
              break;
            }
            const uint32_t k_next = kv_lo + sn * kStageLo;
            int t = 0;
            for (; t < 2; ++t) {
              if (!mbar_wait(s_free + t, j & 1, limit)) {
                record_error(p.status, kWhereSFull, &s_abort);
                break;
              }
              tc_fence_after();
              issue_qk_lo<D, kDense>(colS[t], q_lo + t * kQLo, k_next);
              tc_commit(s_full + t);
            }
            if (t < 2) break;
          }
          int t = 0;
          for (; t < 2; ++t) {
            if (!mbar_wait(p_full + t, j & 1, limit)) {
              record_error(p.status, kWherePFull, &s_abort);
              break;
            }
            tc_fence_after();
            issue_pv_lo<D, kPv16, kDense>(colO[t], colP[t], kv_lo + s * kStageLo + kVLo, j == 0);
            tc_commit(pv_done + t);
          }
          if (t < 2) break;
          tc_commit(kv_empty + s);
          s = sn;
          if (++sn == C::kStages) {
            sn = 0;
            phn ^= 1u;
          }
        }
        for (int j = 0; !C::kSepP && ok && j < ntiles; ++j) {
          const uint32_t k_next = kv_lo + sn * kStageLo;
          for (int t = 0; t < 2 && ok; ++t) {
            if (!mbar_wait(p_full + t, j & 1, limit)) {
              record_error(p.status, kWherePFull, &s_abort);
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv_lo<D, kPv16, kDense>(colO[t], colS[t], kv_lo + s * kStageLo + kVLo, j == 0);
            tc_commit(pv_done + t);
            if (t == 1) tc_commit(kv_empty + s);
            if (j + 1 < ntiles) {
              if (t == 0 && !mbar_wait(kv_full + sn, phn, limit)) {
                record_error(p.status, kWhereKvFull, &s_abort);
                ok = false;
                break;
              }
              // P_t lives in S_t's columns: the next S_t may be written only after P_t.V is done.
              if (!mbar_wait(pv_done + t, j & 1, limit)) {
                record_error(p.status, kWherePvDone, &s_abort);
                ok = false;
                break;
              }
              tc_fence_after();
              issue_qk_lo<D, kDense>(colS[t], q_lo + t * kQLo, k_next);
              tc_commit(s_full + t);
            }
          }
          s = sn;
          if (++sn == C::kStages) {
            sn = 0;
            phn ^= 1u;
          }
        }
        // Drain: every MMA issued above has finished before the CTA frees its tensor memory.
        tc_commit(mma_final);
        mbar_wait(mma_final, 0, limit);
      }
    }
  } else {
    regs_inc<regs_softmax<D, kPv16, kDense>()>();
    // ------------------------------------------------------------ softmax + epilogue
    const int t = (warp - 4) >> 2;
    const int wq = warp & 3;                     // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;                // row within the tile = TMEM lane
    const int row = q0 + t * kBM + r;            // query row
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + (t == 0 ? C::kColS0 : C::kColS1);
    const uint32_t tO = tmem + lane_base + (t == 0 ? C::kColO0 : C::kColO1);
    const uint32_t tP = C::kSepP ? tmem + lane_base + (t == 0 ? C::kColP0 : C::kColP1) : tS;
    const int nbk = p.npad / 64;
    float qscale;
    if (kDense) {
      qscale = 1.0f;
    } else if (kRowQ) {
      // The scale of this thread's own row (its block of 2^q_shift rows); none past the padding.
      qscale = row < p.npad ? p.q_scales[hh * (p.npad >> p.q_shift) + (row >> p.q_shift)] : 0.0f;
    } else {
      const int nbq = p.npad / 128, qblk = (q0 + t * kBM) / 128;
      qscale = qblk < nbq ? p.q_scales[hh * nbq + qblk] : 0.0f;
    }
    const float cq = qscale * p.sm_scale_log2;
    const float* ks = kDense ? nullptr : p.k_scales + hh * nbk;
    float m = -INFINITY, l = 0.0f;
    float ksn0 = kDense ? 1.0f : ks[0], ksn1 = kDense ? 1.0f : ks[1];   // k scales of the next tile, loaded one tile ahead
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const float ks0 = ksn0, ks1 = ksn1;
      if (!kDense && j + 1 < ntiles) {
        ksn0 = ks[2 * j + 2];
        ksn1 = ks[2 * j + 3];
      }
      if (!warp_wait(s_full + t, j & 1, limit)) {
        if (lane == 0) record_error(p.status, kWhereSFull, &s_abort);
        ok = false;
        break;
      }
      tc_fence_after();
      const float c0 = cq * ks0, c1 = cq * ks1;
      const int kvalid = min(kBN, p.n - j * kBN);
      const bool stepped =
          kvalid == kBN
              ? softmax_step<D, false, kPv16, kDense>(tS, tO, tP, c0, c1, kBN, j == 0, m, l, s_free + t, pv_done + t,
                                                      j, limit)
              : softmax_step<D, true, kPv16, kDense>(tS, tO, tP, c0, c1, kvalid, j == 0, m, l, s_free + t, pv_done + t,
                                                     j, limit);
      if (!stepped) {
        if (lane == 0) record_error(p.status, kWherePvDone, &s_abort);
        ok = false;
        break;
      }
      tc_fence_before();
      mbar_arrive(p_full + t);
    }
    if (ok && warp_wait(pv_done + t, (ntiles - 1) & 1, limit)) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const float* vs = kDense ? nullptr : p.v_scales + hh * D;
      const float* vm = kMean ? p.v_mean + hh * D : nullptr;
      uint16_t* orow = p.out + static_cast<int64_t>(row) * p.ost + static_cast<int64_t>(hh) * p.osh;
      // With the output map, the rows go through Q tile t's shared memory (every Q.K^T that read it
      // was issued before this tile's last P.V, so it has completed) in the map's 128-byte
      // swizzled layout, and each warp stores its 32 rows with one bulk tensor copy per 64
      // channels: whole lines, instead of 16 bytes per row and instruction.
      uint8_t* stage = sQ + t * C::kQTileBytes;
      // The staged store exists only at D = 128 (at D = 64 it measured slower); the D = 64
      // instantiations keep the row stores alone.
      const bool tma_out = D == 128 && p.tma_out;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        SAGE_TMEM_LD32(tO + c, o);
        tmem_wait_ld();
        if (tma_out || row < p.n) {
#pragma unroll
          for (int v8 = 0; v8 < 4; ++v8) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int k = v8 * 8 + u * 2;
              float a = kDense ? __uint_as_float(o[k]) * inv_l : __uint_as_float(o[k]) * vs[c + k] * inv_l;
              float b = kDense ? __uint_as_float(o[k + 1]) * inv_l : __uint_as_float(o[k + 1]) * vs[c + k + 1] * inv_l;
              if (kMean) {
                a += vm[c + k];
                b += vm[c + k + 1];
              }
              w[u] = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a))) |
                     (static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(b))) << 16);
            }
            if (tma_out) {
              const int col = c + v8 * 8, chunk = (col & 63) >> 3;
              *reinterpret_cast<uint4*>(stage + (col >> 6) * C::kPanelBytes + r * 128 + ((chunk ^ (r & 7)) << 4)) =
                  make_uint4(w[0], w[1], w[2], w[3]);
            } else {
              *reinterpret_cast<uint4*>(orow + c + v8 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
      if (tma_out) {
        fence_proxy_async_smem();
        __syncwarp();
        const int row0 = q0 + t * kBM + wq * 32;
        if (lane == 0 && row0 < p.n) {   // rows past n are not written (a box wholly past n is skipped)
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_store_3d(&omap, stage + pn * C::kPanelBytes + wq * 32 * 128, pn * 64, hh, row0);
          bulk_commit();
          bulk_wait_read<0>();
        }
        __syncwarp();
      }
    } else if (ok) {
      if (lane == 0) record_error(p.status, kWherePvDone, &s_abort);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, bool kRowQ, bool kPv16, bool kMean>
__global__ void __launch_bounds__(384, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                    const AttnParams p) {
  attn_body<D, kRowQ, kPv16, kMean, false>(qmap, kmap, vmap, omap, p);
}

template <int D>
__global__ void __launch_bounds__(384, 1)
    attn_dense_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
                         const AttnParams p) {
  attn_body<D, false, true, false, true>(qmap, kmap, vmap, omap, p);
}

// --------------------------------------------------------------------------- debug: S tiles
// One CTA per (128-row, 128-key) tile: the same TMA loads and issue_qk as the fused kernel,
// then S is read back from TMEM and written as int32.
template <int D>
__global__ void __launch_bounds__(128, 1)
    debug_qk_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap, int npad,
                    int head, int i0, int j0, int32_t* out, int ldo, int32_t* status, uint64_t limit) {
  using C = Cfg<D, false>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ volatile int s_abort;
  __shared__ uint32_t tmem_slot;
  __shared__ uint64_t bar_tma, bar_mma;
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;
  uint8_t* sK = smem + C::kQTileBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bar_tma, 1);
    mbar_init(&bar_mma, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 128);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int qrow = head * npad + i0 + blockIdx.x * kBM;
  const int krow = head * npad + j0 + blockIdx.y * kBN;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bar_tma, C::kQTileBytes + C::kKTileBytes);
    for (int pn = 0; pn < C::kPanels; ++pn) {
      tma_load_2d(sQ + pn * C::kPanelBytes, &qmap, &bar_tma, pn * 64, qrow);
      tma_load_2d(sK + pn * C::kPanelBytes, &kmap, &bar_tma, pn * 64, krow);
    }
    if (mbar_wait(&bar_tma, 0, limit)) {
      tc_fence_after();
      issue_qk<D>(tmem, smem_u32(sQ), smem_u32(sK));
    } else {
      record_error(status, kWhereDebugTma, &s_abort);
    }
    tc_commit(&bar_mma);
  }
  __syncwarp();
  if (warp_wait(&bar_mma, 0, limit)) {
    tc_fence_after();
    const int r = warp * 32 + lane;
    const uint32_t ta = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    int32_t* orow = out + static_cast<int64_t>(blockIdx.x * kBM + r) * ldo + blockIdx.y * kBN;
    for (int c = 0; c < kBN; c += 32) {
      uint32_t v[32];
      SAGE_TMEM_LD32(ta + c, v);
      tmem_wait_ld();
      if (!s_abort)
        for (int k = 0; k < 32; ++k) orow[c + k] = __float2int_rn(__uint_as_float(v[k]));
    }
  } else if (lane == 0) {
    record_error(status, kWhereDebugMma, &s_abort);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 128);
  }
}

// --------------------------------------------------------------------------- debug: timeout
// One thread waits, with the same bounded wait as the kernels above, on an mbarrier that
// nothing ever arrives on.  The wait must give up after `limit` ns and record the timeout
// in the status block: the test of the failure path, with no fault and no hang.
__global__ void debug_wait_timeout_kernel(int32_t* status, uint64_t limit) {
  __shared__ uint64_t bar;
  __shared__ volatile int s_abort;
  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, limit)) record_error(status, kWhereDebugTimeout, &s_abort);
  }
}

// --------------------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// The bf16 output as a [N][H][D] tensor with the caller's token and head strides (elements),
// 128-byte swizzled boxes of 32 rows x 1 head x 64 channels.  False if the strides do not suit a
// tensor map (the epilogue then stores row by row).
bool make_out_map(CUtensorMap* m, void* out, int n, int h, int d, int64_t ost, int64_t osh) {
  auto fn = encode_fn();
  if (!fn || ost <= 0 || osh <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(n)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(osh) * 2, static_cast<cuuint64_t>(ost) * 2};
  cuuint32_t box[3] = {64, 1, 32};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A bf16 [N][H][D] view with the caller's token and head strides (elements) as a 3-D map
// {D, H, N}, 128-byte swizzled boxes of 64 channels x 1 head x 128 rows: in shared memory the
// same panel layout as a 128-row tile of codes.  A stride of a dimension of extent 1 is never
// stepped, so any valid value stands in for it.  False if the map cannot be built (the strides
// must be multiples of 8 elements).
bool make_view_map(CUtensorMap* m, const void* base, int n, int h, int d, int64_t st, int64_t sh) {
  auto fn = encode_fn();
  if (!fn) return false;
  if (h == 1 && sh <= 0) sh = d;
  if (n == 1 && st <= 0) st = static_cast<int64_t>(h) * d;
  if (st <= 0 || sh <= 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(h), static_cast<cuuint64_t>(n)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(sh) * 2, static_cast<cuuint64_t>(st) * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major [rows][inner] matrix, 128-byte swizzled boxes of box_rows x box_inner elements.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
              uint64_t rows, uint32_t box_inner, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * elem_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool kRowQ, bool kPv16, bool kMean>
cudaError_t launch_variant(dim3 grid, const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& omap, const AttnParams& p, cudaStream_t s) {
  constexpr int kSmem = Cfg<D, kPv16>::kSmemBytes;
  // The shared-memory limit is an attribute of the function in the current context: set it on
  // every call (a host-side call, no device synchronisation), so that a new context -- on
  // another device, or after a cudaDeviceReset -- gets it too.
  cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<D, kRowQ, kPv16, kMean>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<D, kRowQ, kPv16, kMean><<<grid, 384, kSmem, s>>>(qmap, kmap, vmap, omap, p);
  return cudaGetLastError();
}

template <int D, bool kRowQ, bool kPv16>
cudaError_t launch_mean(dim3 grid, const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                        const CUtensorMap& omap, const AttnParams& p, cudaStream_t s) {
  return p.v_mean ? launch_variant<D, kRowQ, kPv16, true>(grid, qmap, kmap, vmap, omap, p, s)
                  : launch_variant<D, kRowQ, kPv16, false>(grid, qmap, kmap, vmap, omap, p, s);
}

template <int D>
cudaError_t launch_attn_fwd_t(int n, int h, const sage_quantized& qz, int q_block, float sm_scale, void* out,
                              int64_t ost, int64_t osh, int32_t* status, cudaStream_t s) {
  const int npad = static_cast<int>(pad128(n));
  const bool pv16 = qz.v_format == 1;
  CUtensorMap qmap, kmap, vmap;
  const bool vmap_ok =
      pv16 ? make_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, qz.v_codes, npad, static_cast<uint64_t>(h) * D, 64, D)
           : make_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qz.v_codes, npad, static_cast<uint64_t>(h) * D, 128, D);
  if (!make_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, qz.q_codes, D, static_cast<uint64_t>(h) * npad, 64, 128) ||
      !make_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, qz.k_codes, D, static_cast<uint64_t>(h) * npad, 64, 128) ||
      !vmap_ok)
    return cudaErrorInvalidValue;
  AttnParams p;
  p.n = n;
  p.npad = npad;
  p.h = h;
  p.q_scales = qz.q_scales;
  p.q_shift = 0;
  while ((1 << p.q_shift) < q_block) ++p.q_shift;
  p.k_scales = qz.k_scales;
  p.v_scales = qz.v_scales;
  p.v_mean = qz.v_mean;
  p.sm_scale_log2 = sm_scale * kLog2e;
  p.out = static_cast<uint16_t*>(out);
  p.ost = ost;
  p.osh = osh;
  CUtensorMap omap;
  memset(&omap, 0, sizeof(omap));
  // At D = 64 the staged store measured slower (strided64 1.623 ms against 1.612 storing row by
  // row); at D = 128 faster (video 21.96 against 21.99 ms).
  p.tma_out = (D == 128 && make_out_map(&omap, out, n, h, D, ost, osh)) ? 1 : 0;
  p.status = status;
  p.wait_limit_ns = kWaitLimitNs;
  const dim3 grid((npad + 2 * kBM - 1) / (2 * kBM), h);
  const bool row_q = q_block != 128;
  if (pv16)
    return row_q ? launch_mean<D, true, true>(grid, qmap, kmap, vmap, omap, p, s)
                 : launch_mean<D, false, true>(grid, qmap, kmap, vmap, omap, p, s);
  return row_q ? launch_mean<D, true, false>(grid, qmap, kmap, vmap, omap, p, s)
               : launch_mean<D, false, false>(grid, qmap, kmap, vmap, omap, p, s);
}

template <int D>
cudaError_t launch_attn_dense_tc_t(const StridedView& q, const StridedView& k, const uint16_t* vt, int n, int h,
                                   float sm_scale, void* out, int64_t ost, int64_t osh, int32_t* status,
                                   cudaStream_t s) {
  using C = Cfg<D, true>;
  const int npad = static_cast<int>(pad128(n));
  CUtensorMap qmap, kmap, vmap, omap;
  if (!make_view_map(&qmap, q.data, n, h, D, q.st, q.sh) || !make_view_map(&kmap, k.data, n, h, D, k.st, k.sh) ||
      !make_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, vt, npad, static_cast<uint64_t>(h) * D, 64, D))
    return cudaErrorInvalidValue;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.n = n;
  p.npad = npad;
  p.h = h;
  p.sm_scale_log2 = sm_scale * kLog2e;
  p.out = static_cast<uint16_t*>(out);
  p.ost = ost;
  p.osh = osh;
  memset(&omap, 0, sizeof(omap));
  p.tma_out = (D == 128 && make_out_map(&omap, out, n, h, D, ost, osh)) ? 1 : 0;
  p.status = status;
  p.wait_limit_ns = kWaitLimitNs;
  cudaError_t e = cudaFuncSetAttribute(attn_dense_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const dim3 grid((npad + 2 * kBM - 1) / (2 * kBM), h);
  attn_dense_tc_kernel<D><<<grid, 384, C::kSmemBytes, s>>>(qmap, kmap, vmap, omap, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_debug_qk_t(int n, int h, const sage_quantized& qz, int head, int i0, int j0, int row_tiles,
                              int col_tiles, int32_t* out, int32_t* status, cudaStream_t s) {
  using C = Cfg<D, false>;
  const int npad = static_cast<int>(pad128(n));
  CUtensorMap qmap, kmap;
  if (!make_map(&qmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, qz.q_codes, D, static_cast<uint64_t>(h) * npad, 64, 128) ||
      !make_map(&kmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, qz.k_codes, D, static_cast<uint64_t>(h) * npad, 64, 128))
    return cudaErrorInvalidValue;
  const int smem = C::kQTileBytes + C::kKTileBytes + 1024;
  cudaError_t e = cudaFuncSetAttribute(debug_qk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  debug_qk_kernel<D><<<dim3(row_tiles, col_tiles), 128, smem, s>>>(qmap, kmap, npad, head, i0, j0, out,
                                                                    col_tiles * kBN, status, kWaitLimitNs);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(int n, int h, int d, const sage_quantized& qz, int q_block, float sm_scale, void* out,
                            int64_t ost, int64_t osh, int32_t* status, cudaStream_t s) {
  return d == 128 ? launch_attn_fwd_t<128>(n, h, qz, q_block, sm_scale, out, ost, osh, status, s)
                  : launch_attn_fwd_t<64>(n, h, qz, q_block, sm_scale, out, ost, osh, status, s);
}

cudaError_t launch_attn_dense_tc(const StridedView& q, const StridedView& k, const uint16_t* vt, int n, int h, int d,
                                 float sm_scale, void* out, int64_t ost, int64_t osh, int32_t* status, cudaStream_t s) {
  return d == 128 ? launch_attn_dense_tc_t<128>(q, k, vt, n, h, sm_scale, out, ost, osh, status, s)
                  : launch_attn_dense_tc_t<64>(q, k, vt, n, h, sm_scale, out, ost, osh, status, s);
}

cudaError_t launch_debug_wait_timeout(int32_t* status, uint64_t limit_ns, cudaStream_t s) {
  debug_wait_timeout_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_debug_qk(int n, int h, int d, const sage_quantized& qz, int head, int i0, int j0, int row_tiles,
                            int col_tiles, int32_t* out, int32_t* status, cudaStream_t s) {
  return d == 128 ? launch_debug_qk_t<128>(n, h, qz, head, i0, j0, row_tiles, col_tiles, out, status, s)
                  : launch_debug_qk_t<64>(n, h, qz, head, i0, j0, row_tiles, col_tiles, out, status, s);
}

}  // namespace sage
