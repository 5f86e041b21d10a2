/*
 * sage_oracle.c -- plain, slow, obviously-correct CPU oracle for SageAttention2-style
 * quantised attention.  TEST INFRASTRUCTURE ONLY: it is linked by the tests, by the
 * package's smoke() check and by the CPU-baseline leg of bench.py, never by the product
 * path.  It shares no source, header or table with the CUDA library.
 *
 * What it computes, in the order of the quantised attention call timed in
 * "gb10-sampling-component-profile-1344x768-124f-seed440420.json"
 * (key attention_internal_p50_milliseconds.sage2: framework_and_k_smoothing_estimate,
 * qk_quantize, v_quantize, attention_forward):
 *
 *   1. K mean       mu[h,c] = mean over tokens of K[t,h,c]                 oracle_k_mean
 *   2. Q quantise   per (head, 128-row block) symmetric INT8, fp32 scale   oracle_quant_q
 *                   (or per (head, qb-row block), qb | 128: the per-warp variant with the
 *                   recorded warp_q of 32 rows, down to per row)           oracle_quant_q_blk
 *   3. K quantise   K~ = K - mu, per (head, 64-row block) INT8             oracle_quant_k
 *   4. V quantise   per (head, channel) FP8 E4M3, fp32 scale               oracle_quant_v
 *                   (or INT8, and optionally of V - mean(V))                oracle_quant_v_fmt
 *   5. S = Qc Kc^T  exact integer dot products                             oracle_qk_int32
 *   6-8. softmax(S * s_q * s_k * sm_scale) with P held in E4M3, times V    oracle_attn_sq(_blk)
 *        (P in INT8 when V is INT8; + mean(V) when V was smoothed)         oracle_attn_sq_v
 *   9. exact fp64 softmax attention of the bf16 inputs                     oracle_attn_exact
 *   0. (upstream of 1-4) in-place RMSNorm + rotary embedding of Q / K       oracle_rmsnorm_rope
 *
 * The shapes are those of the attention call profiled in
 * "gb10-sage2-p0-interleave-softmax-latency.json" (q_shape [1, 37810, 56, 128]).
 * Readings where the pages are silent (the summation order of the mean, division rather
 * than reciprocal multiplication, the clamp at +-127, the static 448 scale of P, ...) are
 * stated at each function.
 *
 * Inputs are bf16 bit patterns (uint16) addressed as data[t*st + h*sh + c]: a strided
 * [N, H, D] view with unit channel stride.  Code buffers use N_pad = ceil(N/128)*128 rows,
 * and the pad rows hold code 0.
 *
 * Build: plain C99, no fast-math, no FMA contraction (-ffp-contract=off), OpenMP optional.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Test hook: a nonzero value plants one deliberate mistake (see the MUT_* list) so that
 * the tests can show that the pins catch it.  Always 0 outside those tests. */
enum { MUT_NONE = 0, MUT_NO_SMOOTH = 1, MUT_RESCALE_SIGN = 2, MUT_SCALE_255 = 3,
       MUT_KEY_INDEX = 4, MUT_V_SCALE_CHANNEL = 5, MUT_DROP_LAST_KEY = 6,
       MUT_E4M3_TRUNC = 7, MUT_MEAN_N_PAD = 8, MUT_Q_BLOCK_INDEX = 9, MUT_ROPE_SIGN = 10,
       MUT_RMS_SUM = 11, MUT_V_MEAN_SIGN = 12, MUT_P_I8_255 = 13, MUT_V_I8_448 = 14,
       MUT_F32_HALF_SCALE = 15, MUT_F32_KSCALE_TILE = 16, MUT_F32_L_CODES = 17, MUT_F32_EXP_BASE = 18 };
static int g_mutation = 0;
void oracle_set_mutation(int m) { g_mutation = m; }

static inline float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static inline int64_t pad128(int64_t n) { return (n + 127) / 128 * 128; }

/* ------------------------------------------------------------------------------------
 * FP8 E4M3 (OCP 8-bit floating point specification, E4M3 variant): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals m * 2^-9; there
 * are no infinities and S.1111.111 is NaN, so the largest finite magnitude is
 * 1.110b * 2^8 = 448.  Encoding rounds to nearest with ties to even and saturates finite
 * values beyond 448 to +-448 ("satfinite").
 * ---------------------------------------------------------------------------------- */
double oracle_e4m3_decode(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return s ? -v : v;
}

uint8_t oracle_e4m3_encode(double x) {
  uint8_t s = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (isnan(x)) return (uint8_t)(s | 0x7F);
  if (a > 448.0) a = 448.0;                    /* satfinite */
  if (a == 0.0) return s;
  int e2;
  frexp(a, &e2);                               /* a in [2^(e2-1), 2^e2) */
  int E = e2 - 1;                              /* unbiased exponent of a */
  if (E < -6) E = -6;                          /* subnormals share the 2^-6 binade's spacing */
  double q = ldexp(1.0, E - 3);                /* spacing of E4M3 values in this binade */
  double n = nearbyint(a / q);                 /* a/q exact; ties to even */
  if (g_mutation == MUT_E4M3_TRUNC) n = floor(a / q);
  if (n >= 16.0) { E += 1; n = 8.0; }          /* carried into the next binade */
  /* n*2^(E-3): for E = -6 the code is n itself (n < 8 subnormal, n = 8.. normal with
   * exponent field 1); otherwise exponent field E+7 and mantissa n-8. */
  uint8_t mag = (E == -6) ? (uint8_t)n : (uint8_t)(((E + 7) << 3) | ((int)n - 8));
  return (uint8_t)(s | mag);
}

/* ------------------------------------------------------------------------------------
 * 1. K mean.  The pages fold it into "framework_and_k_smoothing_estimate" and give no
 * order of summation.  Reading used here (and in the CUDA path, so that the INT8 K codes
 * can be compared bit for bit): tokens are split into consecutive chunks of 128; each
 * chunk is summed in fp32 in ascending token order starting from 0; the chunk sums are
 * split into 8 groups of G = ceil(chunks / 8) consecutive chunks; each group is summed in
 * fp64 in ascending chunk order starting from 0; the 8 group sums are added in fp64 in
 * ascending group order; the total is divided by N in fp64 and rounded once to fp32.
 * ---------------------------------------------------------------------------------- */
void oracle_k_mean(const uint16_t* k, int64_t n, int64_t h, int64_t d, int64_t st, int64_t sh,
                   float* mu) {
  int64_t nchunk = (n + 127) / 128;
  int64_t g = (nchunk + 7) / 8;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t hh = 0; hh < h; ++hh) {
    for (int64_t c = 0; c < d; ++c) {
      double total = 0.0;
      for (int64_t grp = 0; grp < 8; ++grp) {
        double gsum = 0.0;
        for (int64_t ch = grp * g; ch < (grp + 1) * g && ch < nchunk; ++ch) {
          float part = 0.0f;
          int64_t t1 = (ch + 1) * 128 < n ? (ch + 1) * 128 : n;
          for (int64_t t = ch * 128; t < t1; ++t) part = part + bf16_to_f32(k[t * st + hh * sh + c]);
          gsum += (double)part;
        }
        total += gsum;
      }
      double denom = (g_mutation == MUT_MEAN_N_PAD) ? (double)pad128(n) : (double)n;
      mu[hh * d + c] = (float)(total / denom);
    }
  }
}

/* ------------------------------------------------------------------------------------
 * Symmetric INT8 quantisation of one block (rows [r0, r1) of one head, all D channels).
 * scale = fl32(amax / 127); code = clamp(round_half_even(fl32(x / scale)), -127, 127),
 * with IEEE fp32 division.  An all-zero block has scale 0 and codes 0.  Pad rows (>= N)
 * are not part of the block's max and get code 0.
 * ---------------------------------------------------------------------------------- */
static float quant_block_i8(const float* x, int64_t rows, int64_t d, int8_t* codes) {
  float amax = 0.0f;
  for (int64_t i = 0; i < rows * d; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float scale = (g_mutation == MUT_SCALE_255) ? amax / 255.0f : amax / 127.0f;
  for (int64_t i = 0; i < rows * d; ++i) {
    if (scale == 0.0f) { codes[i] = 0; continue; }
    float y = x[i] / scale;
    float r = rintf(y);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    codes[i] = (int8_t)r;
  }
  return scale;
}

/* 2. Q: one scale per (head, qb-row block), qb a power of two dividing 128 (the method's
 * default is qb = 128; qb = 32 is the per-warp granularity of the recorded kernel's warp_q).
 * codes [H][N_pad][D], scales [H][N_pad/qb].  A block that lies wholly in the padding has
 * scale 0. */
void oracle_quant_q_blk(const uint16_t* q, int64_t n, int64_t h, int64_t d, int64_t st, int64_t sh,
                        int64_t qb, int8_t* codes, float* scales) {
  int64_t np = pad128(n), nb = np / qb;
  memset(codes, 0, (size_t)(h * np * d));
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t hh = 0; hh < h; ++hh)
    for (int64_t b = 0; b < nb; ++b) {
      float* buf = (float*)malloc(sizeof(float) * (size_t)(qb * d));
      int64_t r0 = b * qb, r1 = r0 + qb < n ? r0 + qb : n;
      for (int64_t t = r0; t < r1; ++t)
        for (int64_t c = 0; c < d; ++c) buf[(t - r0) * d + c] = bf16_to_f32(q[t * st + hh * sh + c]);
      scales[hh * nb + b] = quant_block_i8(buf, r1 - r0, d, codes + (hh * np + r0) * d);
      free(buf);
    }
}

void oracle_quant_q(const uint16_t* q, int64_t n, int64_t h, int64_t d, int64_t st, int64_t sh,
                    int8_t* codes, float* scales) {
  oracle_quant_q_blk(q, n, h, d, st, sh, 128, codes, scales);
}

/* 3. K smoothing then quantisation: K~ = fl32(K - mu) (one fp32 subtraction), one scale per
 * (head, 64-row block). codes [H][N_pad][D], scales [H][N_pad/64]. */
void oracle_quant_k(const uint16_t* k, int64_t n, int64_t h, int64_t d, int64_t st, int64_t sh,
                    const float* mu, int8_t* codes, float* scales) {
  int64_t np = pad128(n), nb = np / 64;
  memset(codes, 0, (size_t)(h * np * d));
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t hh = 0; hh < h; ++hh)
    for (int64_t b = 0; b < nb; ++b) {
      int64_t r0 = b * 64, r1 = r0 + 64 < n ? r0 + 64 : n;
      if (r1 <= r0) { scales[hh * nb + b] = 0.0f; continue; }
      float* buf = (float*)malloc(sizeof(float) * 64 * d);
      for (int64_t t = r0; t < r1; ++t)
        for (int64_t c = 0; c < d; ++c) {
          float m = (g_mutation == MUT_NO_SMOOTH) ? 0.0f : mu[hh * d + c];
          buf[(t - r0) * d + c] = bf16_to_f32(k[t * st + hh * sh + c]) - m;
        }
      scales[hh * nb + b] = quant_block_i8(buf, r1 - r0, d, codes + (hh * np + r0) * d);
      free(buf);
    }
}

/* 4. V: one scale per (head, channel), scale = fl32(amax over tokens / 448), code =
 * E4M3(fl32(v / scale)); written transposed as [H][D][N_pad] (keys contiguous). */
void oracle_quant_v(const uint16_t* v, int64_t n, int64_t h, int64_t d, int64_t st, int64_t sh,
                    uint8_t* codes, float* scales) {
  int64_t np = pad128(n);
  memset(codes, 0, (size_t)(h * d * np));
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t hh = 0; hh < h; ++hh)
    for (int64_t c = 0; c < d; ++c) {
      float amax = 0.0f;
      for (int64_t t = 0; t < n; ++t) {
        float a = fabsf(bf16_to_f32(v[t * st + hh * sh + c]));
        if (a > amax) amax = a;
      }
      float scale = amax / 448.0f;
      int64_t sc = (g_mutation == MUT_V_SCALE_CHANNEL) ? (c + 1) % d : c;
      scales[hh * d + sc] = scale;
      for (int64_t t = 0; t < n; ++t) {
        if (scale == 0.0f) continue;
        float y = bf16_to_f32(v[t * st + hh * sh + c]) / scale;
        codes[(hh * d + c) * np + t] = oracle_e4m3_encode((double)y);
      }
    }
}

/* 4'. The V path's two options.
 *  mu != NULL: V smoothing.  x = fl32(v - mu[h][c]) (one fp32 subtraction, mu the channel mean
 *    of V over the tokens, taken as oracle_k_mean takes the mean of K); softmax rows sum to 1,
 *    so the attention adds mu back to its output (oracle_attn_sq_v).  mu == NULL: x = v.
 *  fmt 0: E4M3 as oracle_quant_v: scale = fl32(amax / 448), code = E4M3(fl32(x / scale)).
 *  fmt 1: INT8: scale = fl32(amax / 127), code = clamp(rint(fl32(x / scale)), -127, 127),
 *    stored as the int8 byte (two's complement) -- the INT8 P.V variant timed on the
 *    sampling-component page (v_int8_quantize), quantised like Q and K.
 * amax over the N tokens of |x|; an all-zero channel has scale 0 and codes 0.
 * codes [H][D][N_pad] (keys contiguous), scales [H][D]. */
void oracle_quant_v_fmt(const uint16_t* v, int64_t n, int64_t h, int64_t d, int64_t st, int64_t sh,
                        const float* mu, int64_t fmt, uint8_t* codes, float* scales) {
  int64_t np = pad128(n);
  memset(codes, 0, (size_t)(h * d * np));
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t hh = 0; hh < h; ++hh)
    for (int64_t c = 0; c < d; ++c) {
      float m = mu ? mu[hh * d + c] : 0.0f;
      float amax = 0.0f;
      for (int64_t t = 0; t < n; ++t) {
        float a = fabsf(bf16_to_f32(v[t * st + hh * sh + c]) - m);
        if (a > amax) amax = a;
      }
      float scale = fmt ? amax / (g_mutation == MUT_V_I8_448 ? 448.0f : 127.0f) : amax / 448.0f;
      scales[hh * d + c] = scale;
      if (scale == 0.0f) continue;
      for (int64_t t = 0; t < n; ++t) {
        float y = (bf16_to_f32(v[t * st + hh * sh + c]) - m) / scale;
        uint8_t code;
        if (fmt) {
          float r = rintf(y);
          if (r > 127.0f) r = 127.0f;
          if (r < -127.0f) r = -127.0f;
          code = (uint8_t)(int8_t)r;
        } else {
          code = oracle_e4m3_encode((double)y);
        }
        codes[(hh * d + c) * np + t] = code;
      }
    }
}

/* 5. S[i][j] = sum_c qc[h][i0+i][c] * kc[h][j0+j][c], exact in int64, stored as int32
 * (|S| <= 128 * 127^2 < 2^31). */
void oracle_qk_int32(const int8_t* qc, const int8_t* kc, int64_t n, int64_t h, int64_t d,
                     int64_t head, int64_t i0, int64_t j0, int64_t rows, int64_t cols,
                     int32_t* out) {
  int64_t np = pad128(n);
  (void)h;
  for (int64_t i = 0; i < rows; ++i)
    for (int64_t j = 0; j < cols; ++j) {
      int64_t acc = 0;
      const int8_t* a = qc + (head * np + i0 + i) * d;
      const int8_t* b = kc + (head * np + j0 + j) * d;
      for (int64_t c = 0; c < d; ++c) acc += (int64_t)a[c] * (int64_t)b[c];
      out[i * cols + j] = (int32_t)acc;
    }
}

/* ------------------------------------------------------------------------------------
 * 6-8. Same-quantisation attention for selected query rows (all heads).
 *   s_ij = S_ij * s_q[h, i/qb] * s_k[h, j/64] * sm_scale     (qb = 128 unless the Q scales
 *   are per smaller block, see oracle_quant_q_blk)
 *   p_ij = exp(s_ij - m_i);  P8_ij = E4M3(448 p_ij)  (static scale 448: p <= 1 never overflows)
 *   l_i  = sum_j 448 p_ij                (unquantised p)
 *   O_ic = (sum_j P8_ij * E4M3val(vc[h,c,j])) * s_v[h,c] / l_i
 * tile == 0 (the definition, fp64): m_i is the row's global max, all arithmetic in fp64.
 * tile  > 0: keys are visited in tiles of `tile` keys; m_i is the running max up to the
 *   current tile, P8 is formed against it, and whenever m_i rises the partial sums (O, l)
 *   are multiplied by exp(m_old - m_new) -- an exact rescale on every increase, the schedule
 *   of an online-softmax kernel that holds P in E4M3.
 *   score_f32 == 0: scores and exponents in fp64.
 *   score_f32 != 0: the discrete step (the E4M3 rounding of 448 p) is taken in the kernel's
 *   precision: in base 2, x = fma_f32(S, c_b, fl32(log2(448) - m)) with
 *   c_b = fl32(fl32(s_q * fl32(sm_scale * log2 e)) * s_k[b]), m the fp32 running max of
 *   fl32(c_b * max S over each 64-key half), and 448 p = RN_f32(2^x); sums stay in fp64.
 * The V options of oracle_quant_v_fmt:
 *   vfmt 1 (INT8 V): P is INT8 too, with the static scale 127 that p <= 1 allows:
 *     P8_ij = rint(127 p_ij) in [0, 127] (ties to even), l_i = sum_j 127 p_ij, V values are the
 *     integer codes; in the score_f32 schedule x uses log2(127) and P8 = rint(RN_f32(2^x)).
 *   vmu != NULL (V smoothed): O_ic += vmu[h][c] after the division by l (each softmax row
 *     sums to 1, so the mean taken out of V before quantisation comes back whole).
 * out[r][h][c] (fp64).
 * ---------------------------------------------------------------------------------- */
/* Value of one V code: the E4M3 number, or the INT8 integer. */
static double v_value(uint8_t code, int64_t vfmt) {
  return vfmt ? (double)(int8_t)code : oracle_e4m3_decode(code);
}

/* Value of P's code for pp = 448 p (E4M3) or 127 p (INT8, round half to even). */
static double p_code(double pp, int64_t vfmt) {
  if (!vfmt) return oracle_e4m3_decode(oracle_e4m3_encode(pp));
  return rint(g_mutation == MUT_P_I8_255 ? pp * (255.0 / 127.0) : pp);
}

/* One (query row i, head hh) of the same-quantisation attention described above, written to
 * o[0..d).  When tr_pp is not NULL, each key j < n also leaves a trace: tr_pp[j] = the 448 p
 * (127 p) whose code P takes, tr_p8[j] = the value of that code, tr_lw[j] = the running max that
 * key's p is relative to, as a base-2 exponent (so the weight key j carries in the final sums is
 * 2^(tr_lw[j] - tr_lw[n-1])).  Keys the row does not visit keep pp = p8 = 0. */
static void attn_row(const int8_t* qc, const float* qs, int64_t qb, const int8_t* kc, const float* ks,
                     const uint8_t* vc, const float* vs, const float* vmu, int64_t vfmt, int64_t n,
                     int64_t d, double sm_scale, int64_t i, int64_t hh, int64_t tile, int64_t score_f32,
                     double* o, double* tr_pp, double* tr_p8, double* tr_lw) {
  int64_t np = pad128(n), nbq = np / qb, nbk = np / 64;
  int64_t nkeys = (g_mutation == MUT_DROP_LAST_KEY) ? n - 1 : n;
  const float kLog2E = 1.4426950408889634f;
  /* log2 of P's static scale: log2(448) for E4M3 P, log2(127) for INT8 P */
  const float kLog2P = vfmt ? 6.988684686772166f : 8.807354922057604f;
  const double pscale = vfmt ? 127.0 : 448.0;
  const double log2e = 1.4426950408889634;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  int64_t* S = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
  const int8_t* a = qc + (hh * np + i) * d;
  /* the Q block of row i (the planted mistake reads the 128-row block's index instead) */
  const int64_t qbi = (g_mutation == MUT_Q_BLOCK_INDEX) ? i / 128 : i / qb;
  double sq = (double)qs[hh * nbq + qbi];
  for (int64_t c = 0; c < d; ++c) o[c] = 0.0;
  if (tr_pp)
    for (int64_t j = 0; j < n; ++j) tr_pp[j] = tr_p8[j] = tr_lw[j] = 0.0;
  for (int64_t j = 0; j < nkeys; ++j) {
    int64_t jj = (g_mutation == MUT_KEY_INDEX) ? (j ^ 1) % n : j;
    const int8_t* b = kc + (hh * np + jj) * d;
    int64_t acc = 0;
    for (int64_t c = 0; c < d; ++c) acc += (int64_t)a[c] * (int64_t)b[c];
    S[j] = acc;
    s[j] = (double)acc * sq * (double)ks[hh * nbk + j / 64] * sm_scale;
  }
  double m = -INFINITY, l = 0.0;
  float mf = -INFINITY;
  int64_t tw = tile > 0 ? tile : nkeys;
  if (tile <= 0)
    for (int64_t j = 0; j < nkeys; ++j) if (s[j] > m) m = s[j];
  const float cq = qs[hh * nbq + qbi] * ((float)sm_scale * kLog2E);
  for (int64_t j0 = 0; j0 < nkeys; j0 += tw) {
    int64_t j1 = j0 + tw < nkeys ? j0 + tw : nkeys;
    if (tile > 0 && score_f32) {
      float mt = -INFINITY;
      for (int64_t h0 = j0; h0 < j1; h0 += 64) {       /* 64-key halves, one K scale each */
        int64_t h1 = h0 + 64 < j1 ? h0 + 64 : j1;
        float mx = -INFINITY;
        for (int64_t j = h0; j < h1; ++j) if ((float)S[j] > mx) mx = (float)S[j];
        int64_t kb = h0 / 64;
        if (g_mutation == MUT_F32_HALF_SCALE && (kb ^ 1) < nbk) kb ^= 1;
        float cb = cq * ks[hh * nbk + kb];
        float v = cb * mx;
        if (v > mt) mt = v;
      }
      if (mt > mf) {
        if (mf != -INFINITY) {
          float dm = (g_mutation == MUT_RESCALE_SIGN) ? mt - mf : mf - mt;
          double alpha = exp2((double)dm);
          for (int64_t c = 0; c < d; ++c) o[c] *= alpha;
          l *= alpha;
        }
        mf = mt;
      }
      const float bias = kLog2P - mf;
      for (int64_t j = j0; j < j1; ++j) {
        int64_t kb = (g_mutation == MUT_F32_KSCALE_TILE) ? j0 / 64 : j / 64;
        float cb = cq * ks[hh * nbk + kb];
        float x = fmaf((float)S[j], cb, bias);
        /* 448 p or 127 p, rounded to fp32 (the planted mistake takes e^x for 2^x) */
        float pp = (g_mutation == MUT_F32_EXP_BASE) ? (float)exp((double)x) : (float)exp2((double)x);
        double p8 = p_code((double)pp, vfmt);
        l += (g_mutation == MUT_F32_L_CODES) ? p8 : (double)pp;
        if (tr_pp) { tr_pp[j] = (double)pp; tr_p8[j] = p8; tr_lw[j] = (double)mf; }
        if (p8 == 0.0) continue;
        for (int64_t c = 0; c < d; ++c) o[c] += p8 * v_value(vc[(hh * d + c) * np + j], vfmt);
      }
      continue;
    }
    if (tile > 0) {
      double mt = -INFINITY;
      for (int64_t j = j0; j < j1; ++j) if (s[j] > mt) mt = s[j];
      if (mt > m) {
        if (m != -INFINITY) {
          double alpha = (g_mutation == MUT_RESCALE_SIGN) ? exp(mt - m) : exp(m - mt);
          for (int64_t c = 0; c < d; ++c) o[c] *= alpha;
          l *= alpha;
        }
        m = mt;
      }
    }
    for (int64_t j = j0; j < j1; ++j) {
      double p = exp(s[j] - m);
      l += pscale * p;
      double p8 = p_code(pscale * p, vfmt);
      if (tr_pp) { tr_pp[j] = pscale * p; tr_p8[j] = p8; tr_lw[j] = m * log2e; }
      if (p8 == 0.0) continue;
      for (int64_t c = 0; c < d; ++c) o[c] += p8 * v_value(vc[(hh * d + c) * np + j], vfmt);
    }
  }
  for (int64_t c = 0; c < d; ++c) {
    double mean = 0.0;
    if (vmu) mean = (g_mutation == MUT_V_MEAN_SIGN) ? -(double)vmu[hh * d + c] : (double)vmu[hh * d + c];
    o[c] = o[c] * (double)vs[hh * d + c] / l + mean;
  }
  free(s);
  free(S);
}

void oracle_attn_sq_v(const int8_t* qc, const float* qs, int64_t qb, const int8_t* kc, const float* ks,
                      const uint8_t* vc, const float* vs, const float* vmu, int64_t vfmt, int64_t n,
                      int64_t h, int64_t d, double sm_scale, const int64_t* rows, int64_t nrows,
                      int64_t tile, int64_t score_f32, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t rh = 0; rh < nrows * h; ++rh) {
    int64_t r = rh / h, hh = rh % h;
    attn_row(qc, qs, qb, kc, ks, vc, vs, vmu, vfmt, n, d, sm_scale, rows[r], hh, tile, score_f32,
             out + (r * h + hh) * d, NULL, NULL, NULL);
  }
}

/* The same computation for query `rows` of one head, with each key's trace (see attn_row):
 * out [nrows][d], pp / p8 / lw [nrows][n]. */
void oracle_attn_sq_trace(const int8_t* qc, const float* qs, int64_t qb, const int8_t* kc, const float* ks,
                          const uint8_t* vc, const float* vs, const float* vmu, int64_t vfmt, int64_t n,
                          int64_t d, double sm_scale, int64_t head, const int64_t* rows, int64_t nrows,
                          int64_t tile, int64_t score_f32, double* out, double* pp, double* p8, double* lw) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < nrows; ++r)
    attn_row(qc, qs, qb, kc, ks, vc, vs, vmu, vfmt, n, d, sm_scale, rows[r], head, tile, score_f32,
             out + r * d, pp + r * n, p8 + r * n, lw + r * n);
}

/* E4M3 V as in oracle_quant_v (Q and K scales per qb-row / 64-row block as above). */
void oracle_attn_sq_blk(const int8_t* qc, const float* qs, int64_t qb, const int8_t* kc, const float* ks,
                        const uint8_t* vc, const float* vs, int64_t n, int64_t h, int64_t d,
                        double sm_scale, const int64_t* rows, int64_t nrows, int64_t tile,
                        int64_t score_f32, double* out) {
  oracle_attn_sq_v(qc, qs, qb, kc, ks, vc, vs, NULL, 0, n, h, d, sm_scale, rows, nrows, tile, score_f32, out);
}

/* The method's default: Q scales per 128-row block. */
void oracle_attn_sq(const int8_t* qc, const float* qs, const int8_t* kc, const float* ks,
                    const uint8_t* vc, const float* vs, int64_t n, int64_t h, int64_t d,
                    double sm_scale, const int64_t* rows, int64_t nrows, int64_t tile,
                    int64_t score_f32, double* out) {
  oracle_attn_sq_blk(qc, qs, 128, kc, ks, vc, vs, n, h, d, sm_scale, rows, nrows, tile, score_f32, out);
}

/* 9. Exact attention of the bf16 inputs in fp64: O = softmax(sm_scale * q k^T) v, no
 * smoothing, no quantisation.  out[r][h][c]. */
void oracle_attn_exact(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t n,
                       int64_t h, int64_t d, int64_t qst, int64_t qsh, int64_t kst, int64_t ksh,
                       int64_t vst, int64_t vsh, double sm_scale, const int64_t* rows,
                       int64_t nrows, double* out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t rh = 0; rh < nrows * h; ++rh) {
    int64_t r = rh / h, hh = rh % h, i = rows[r];
    double* qi = (double*)malloc(sizeof(double) * (size_t)d);
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    double* o = (double*)calloc((size_t)d, sizeof(double));
    for (int64_t c = 0; c < d; ++c) qi[c] = bf16_to_f32(q[i * qst + hh * qsh + c]);
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int64_t c = 0; c < d; ++c) acc += qi[c] * (double)bf16_to_f32(k[j * kst + hh * ksh + c]);
      s[j] = sm_scale * acc;
      if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
      double p = exp(s[j] - m);
      l += p;
      for (int64_t c = 0; c < d; ++c) o[c] += p * (double)bf16_to_f32(v[j * vst + hh * vsh + c]);
    }
    for (int64_t c = 0; c < d; ++c) out[(r * h + hh) * d + c] = o[c] / l;
    free(qi);
    free(s);
    free(o);
  }
}

/* Threads OpenMP will use (1 without OpenMP). */
/* ------------------------------------------------------------------------------------
 * 0. The qk_transform stage of the strided-NHD dataflow ("in-place ... RMSNorm and RoPE on
 * strided views", gb10-sage-strided-nhd-summary key dataflow.qk_transform; timed as rms_rope
 * in the block profile), in place on a bf16 [N, H, D] view, per (token t, head h):
 *   ms = (sum_c x_c^2) / D,   r = 1 / sqrt(ms + eps),   y_c = (x_c * r) * gamma[c]
 *   z_2i   = y_2i * cos[t][i] - y_2i+1 * sin[t][i]
 *   z_2i+1 = y_2i * sin[t][i] + y_2i+1 * cos[t][i]           (rotation of channel pairs)
 *   x_c <- bf16_RNE(z_c)
 * The pages fix neither the precision nor the order of the sum, and the bf16 rounding of z
 * turns a float into a code, so this follows the kernel's fp32 arithmetic exactly: every
 * product and sum rounded to fp32 (no fused multiply-add), IEEE sqrt and division, and
 * sum_c x_c^2 formed as D/8 partial sums of 8 consecutive channels (each in channel order)
 * folded pairwise: partial g += partial g + stride for stride = D/16, ..., 2, 1.
 * cos and sin hold [N][D/2] fp32 angles' cosines and sines (the caller's rotary table). */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40);   /* quiet NaN */
  u += 0x7FFFu + ((u >> 16) & 1u);                                            /* ties to even */
  return (uint16_t)(u >> 16);
}

void oracle_rmsnorm_rope(uint16_t* x, int64_t n, int64_t h, int64_t d, int64_t st, int64_t sh,
                         const float* gamma, const float* cosb, const float* sinb, float eps) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t t = 0; t < n; ++t)
    for (int64_t hh = 0; hh < h; ++hh) {
      uint16_t* row = x + t * st + hh * sh;
      float v[128], part[16];
      for (int64_t c = 0; c < d; ++c) v[c] = bf16_to_f32(row[c]);
      const int64_t ng = d / 8;
      for (int64_t g = 0; g < ng; ++g) {
        float acc = 0.0f;
        for (int64_t j = 0; j < 8; ++j) {
          float sq = v[8 * g + j] * v[8 * g + j];
          acc = acc + sq;
        }
        part[g] = acc;
      }
      for (int64_t stride = ng / 2; stride >= 1; stride /= 2)
        for (int64_t g = 0; g < stride; ++g) part[g] = part[g] + part[g + stride];
      float ms = (g_mutation == MUT_RMS_SUM) ? part[0] : part[0] * (1.0f / (float)d);
      float r = 1.0f / sqrtf(ms + eps);
      for (int64_t i = 0; i < d / 2; ++i) {
        float y0 = (v[2 * i] * r) * gamma[2 * i];
        float y1 = (v[2 * i + 1] * r) * gamma[2 * i + 1];
        float c = cosb[t * (d / 2) + i], s = sinb[t * (d / 2) + i];
        float a = y0 * c, b = y1 * s, e = y0 * s, f = y1 * c;
        float z0 = (g_mutation == MUT_ROPE_SIGN) ? a + b : a - b;
        float z1 = e + f;
        row[2 * i] = f32_to_bf16_rne(z0);
        row[2 * i + 1] = f32_to_bf16_rne(z1);
      }
    }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
