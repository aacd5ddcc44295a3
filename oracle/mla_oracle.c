/*
 * mla_oracle.c -- plain fp64 CPU oracle for absorbed-form MLA decode over a
 * paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg use it.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (all arithmetic in IEEE double, plain loops, no blocking):
 *
 *   For sequence b, query token i < Sq, head h < H:
 *     ctx   = seq_lens[b]
 *     n     = causal ? ctx - Sq + i + 1 : ctx       (visible keys, clamped to [0, ctx])
 *     row_j = dequant(cache[bt[b][j / ps]][j % ps][0:576])      for j < n
 *     z_j   = softmax_scale * sum_{d<576} q[b,i,h,d] * row_j[d]
 *     LSE   = max_j z_j + ln( sum_j exp(z_j - max_j z_j) )       (natural log)
 *     O[d]  = sum_j exp(z_j - LSE) * row_j[d]                    for d < 512
 *   n == 0 gives O = 0 and LSE = -inf.
 *
 * Sources for each step:
 *   - the 576-wide latent row (512 latent + 64 rope), the first 512 of which
 *     are the value: "[Perf][Kimi-K3] Cut MLA decode concat/cache epilogue
 *     latency" (vLLM PR 54896), Purpose, item 1 ("576-wide row");
 *   - the paged cache read through a block table at any page size, and the
 *     causal mask over the 1+MTP query tokens: "HK MLA: MI35x m16x8 retune,
 *     new m16x4 kernel, page_size + mask support" (aiter PR 3072), Summary,
 *     track 1 (variable page size, causal mask for nh64+mtp1, nh32+mtp3,
 *     nh16+mtp7);
 *   - the split of the key range into chunks, each storing its own slice,
 *     with empty chunks returning at once: "perf(mla): chunk the non-FP4
 *     gather_kv_b_proj over KV" (aiter PR 4776), description, third
 *     paragraph.  The merge of the chunk results is the log-sum-exp merge,
 *     which the pages imply but do not write out.
 *   - softmax, log-sum-exp and the weighted sum are the textbook definition
 *     of scaled dot-product attention; the pages give no formula of their
 *     own.
 *   - the cached-prefix expansion (mla_oracle_gather_kv_b_proj): every
 *     cached latent row of a sequence, gathered through the block table and
 *     dequantised, multiplied by each head's kv_b_proj block into that head's
 *     128 no-rope key dims and 128 value dims; the key row is completed by
 *     the row's 64 rope dims: "perf(mla): chunk the non-FP4 gather_kv_b_proj
 *     over KV" (aiter PR 4776), description, first and second paragraphs;
 *   - the decode epilogue (mla_oracle_epilogue): the q-concat of ql_nope and
 *     q_pe into the 576-wide query row and the insert of the new latent row
 *     into the paged cache through slot_mapping, bf16 or fp8: "[Perf]
 *     [Kimi-K3] Cut MLA decode concat/cache epilogue latency" (vLLM PR
 *     54896), Purpose, items 1-3.
 *
 * Numeric formats decoded here, from their published definitions:
 *   - bfloat16: the upper 16 bits of an IEEE binary32;
 *   - fp8 E4M3FN (OCP 8-bit floating point specification): 1 sign bit,
 *     4 exponent bits with bias 7, 3 mantissa bits, subnormals at exponent
 *     field 0, no infinities, S.1111.111 is NaN, largest finite 448.
 *     Encoding (mla_oracle_e4m3_encode): the nearest representable value,
 *     ties to the even code, magnitudes beyond 448 saturated to 448 (the
 *     "saturating" conversion of the same specification), found by trying
 *     every code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_D_QK 576
#define ORACLE_D_V 512

enum { ORACLE_KV_BF16 = 0, ORACLE_KV_FP8_E4M3 = 1 };

/* bfloat16 bits -> double: bf16 is the high half of a binary32. */
double mla_oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* fp8 E4M3FN code -> double, written from the OCP definition. */
double mla_oracle_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int expo = (code >> 3) & 0xF;
  int mant = code & 0x7;
  double v;
  if (expo == 0xF && mant == 0x7) return NAN; /* the only NaN encodings */
  if (expo == 0) {
    v = ldexp((double)mant / 8.0, 1 - 7); /* subnormal: 0.mmm * 2^(1-bias) */
  } else {
    v = ldexp(1.0 + (double)mant / 8.0, expo - 7);
  }
  return sign ? -v : v;
}

int mla_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Dequantised element d of logical key j of sequence b. */
static double cache_elem(const void* cache, int kv_dtype, double kv_scale,
                         const int32_t* bt, int64_t bt_stride, int b,
                         int page_size, int64_t j, int d) {
  int64_t page = bt[(int64_t)b * bt_stride + j / page_size];
  int64_t slot = j % page_size;
  int64_t idx = (page * page_size + slot) * ORACLE_D_QK + d;
  if (kv_dtype == ORACLE_KV_BF16) {
    return mla_oracle_bf16_to_double(((const uint16_t*)cache)[idx]);
  }
  return mla_oracle_e4m3_to_double(((const uint8_t*)cache)[idx]) * kv_scale;
}

/* Number of keys query token i of a sequence with ctx keys may see. */
static int64_t visible_keys(int64_t ctx, int sq, int i, int causal) {
  int64_t n = causal ? ctx - sq + i + 1 : ctx;
  if (n < 0) n = 0;
  if (n > ctx) n = ctx;
  return n;
}

/*
 * Attention of one query row over logical keys [k_begin, k_end) of its
 * visible range (the range is clipped to the visible keys).  Writes the
 * normalised output o[0:512] and the log-sum-exp of the scaled scores of
 * that range.  An empty range gives o = 0, lse = -inf.
 */
static void attend_range(const uint16_t* q_row, const void* cache, int kv_dtype,
                         double kv_scale, const int32_t* bt, int64_t bt_stride,
                         int b, int page_size, int64_t n_visible,
                         int64_t k_begin, int64_t k_end, double scale,
                         double* z, double* o, double* lse) {
  int64_t j, lo = k_begin < 0 ? 0 : k_begin;
  int64_t hi = k_end < n_visible ? k_end : n_visible;
  int d;
  double m = -INFINITY, sum = 0.0, l;
  for (d = 0; d < ORACLE_D_V; ++d) o[d] = 0.0;
  if (hi <= lo) {
    *lse = -INFINITY;
    return;
  }
  /* scores */
  for (j = lo; j < hi; ++j) {
    double acc = 0.0;
    for (d = 0; d < ORACLE_D_QK; ++d) {
      acc += mla_oracle_bf16_to_double(q_row[d]) *
             cache_elem(cache, kv_dtype, kv_scale, bt, bt_stride, b, page_size, j, d);
    }
    z[j - lo] = scale * acc;
    if (z[j - lo] > m) m = z[j - lo];
  }
  /* log-sum-exp */
  for (j = lo; j < hi; ++j) sum += exp(z[j - lo] - m);
  l = m + log(sum);
  *lse = l;
  /* weighted sum of the value part (first 512 dims) of the same rows */
  for (j = lo; j < hi; ++j) {
    double w = exp(z[j - lo] - l);
    for (d = 0; d < ORACLE_D_V; ++d) {
      o[d] += w * cache_elem(cache, kv_dtype, kv_scale, bt, bt_stride, b, page_size, j, d);
    }
  }
}

/*
 * Full decode for sequences [b_begin, b_end) of a batch, restricted to the
 * key range [k_begin, k_end) of every row (pass 0 and INT64_MAX for the
 * whole range).
 *
 *   q         [B, Sq, H, 576] bf16 bits, contiguous
 *   cache     [num_pages, page_size, 576] bf16 bits or e4m3 codes
 *   kv_scale  dequant multiplier for fp8 (ignored for bf16)
 *   bt        [B, bt_stride] int32 page ids
 *   seq_lens  [B] keys per sequence (the Sq new tokens included)
 *   out       [(b_end-b_begin), Sq, H, 512] doubles
 *   lse       [(b_end-b_begin), Sq, H] doubles
 */
void mla_oracle_decode_range(const uint16_t* q, const void* cache, int kv_dtype,
                             double kv_scale, int page_size, const int32_t* bt,
                             int64_t bt_stride, const int32_t* seq_lens, int B,
                             int Sq, int H, int causal, double softmax_scale,
                             int b_begin, int b_end, int64_t k_begin,
                             int64_t k_end, double* out, double* lse) {
  int64_t rows = (int64_t)(b_end - b_begin) * Sq * H;
  int64_t r;
  int64_t max_ctx = 0;
  int b;
  (void)B;
  for (b = b_begin; b < b_end; ++b)
    if (seq_lens[b] > max_ctx) max_ctx = seq_lens[b];
#pragma omp parallel
  {
    double* z = (double*)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
#pragma omp for schedule(dynamic, 1)
    for (r = 0; r < rows; ++r) {
      int h = (int)(r % H);
      int i = (int)((r / H) % Sq);
      int bb = b_begin + (int)(r / ((int64_t)H * Sq));
      const uint16_t* q_row = q + (((int64_t)bb * Sq + i) * H + h) * ORACLE_D_QK;
      int64_t n = visible_keys(seq_lens[bb], Sq, i, causal);
      attend_range(q_row, cache, kv_dtype, kv_scale, bt, bt_stride, bb, page_size,
                   n, k_begin, k_end, softmax_scale, z, out + r * ORACLE_D_V,
                   lse + r);
    }
    free(z);
  }
}

/*
 * One query row (b, i, h) only, over its whole visible range.  Used to
 * check sampled outputs of large problems one by one.
 */
void mla_oracle_decode_row(const uint16_t* q, const void* cache, int kv_dtype,
                           double kv_scale, int page_size, const int32_t* bt,
                           int64_t bt_stride, const int32_t* seq_lens, int Sq,
                           int H, int causal, double softmax_scale, int b, int i,
                           int h, double* out, double* lse) {
  int64_t n = visible_keys(seq_lens[b], Sq, i, causal);
  double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  const uint16_t* q_row = q + (((int64_t)b * Sq + i) * H + h) * ORACLE_D_QK;
  attend_range(q_row, cache, kv_dtype, kv_scale, bt, bt_stride, b, page_size, n, 0,
               n, softmax_scale, z, out, lse);
  free(z);
}

/*
 * Log-sum-exp merge of S partial results of the same rows.
 *   o_parts   [S, rows, 512]  each part normalised over its own keys
 *   lse_parts [S, rows]       -inf for a part with no keys
 * out = sum_s exp(lse_s - L) * o_s with L = ln sum_s exp(lse_s); a row whose
 * parts are all empty gives out = 0, L = -inf.
 */
void mla_oracle_lse_merge(const double* o_parts, const double* lse_parts, int S,
                          int64_t rows, double* out, double* lse) {
  int64_t r;
  for (r = 0; r < rows; ++r) {
    double m = -INFINITY, sum = 0.0, L;
    int s, d;
    for (s = 0; s < S; ++s)
      if (lse_parts[(int64_t)s * rows + r] > m) m = lse_parts[(int64_t)s * rows + r];
    for (d = 0; d < ORACLE_D_V; ++d) out[r * ORACLE_D_V + d] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    for (s = 0; s < S; ++s) sum += exp(lse_parts[(int64_t)s * rows + r] - m);
    L = m + log(sum);
    lse[r] = L;
    for (s = 0; s < S; ++s) {
      double ls = lse_parts[(int64_t)s * rows + r];
      double w;
      if (ls == -INFINITY) continue;
      w = exp(ls - L);
      for (d = 0; d < ORACLE_D_V; ++d)
        out[r * ORACLE_D_V + d] += w * o_parts[((int64_t)s * rows + r) * ORACLE_D_V + d];
    }
  }
}

/*
 * binary32 value -> fp8 E4M3FN code, round to nearest, ties to even,
 * saturating: every non-negative finite code is tried and the nearest kept
 * (on a tie the code whose last mantissa bit is 0); |y| > 448 gives 448;
 * NaN gives 0x7F.  The sign bit is the sign of y, so -0 and negative values
 * that round to zero give 0x80.
 */
uint8_t mla_oracle_e4m3_encode(float y) {
  double a = fabs((double)y);
  int best = 0, c;
  double best_err = INFINITY;
  uint8_t sign = signbit(y) ? 0x80 : 0x00;
  if (isnan(y)) return 0x7F;
  if (a > 448.0) return (uint8_t)(sign | 0x7E);
  for (c = 0; c <= 0x7E; ++c) {
    double err = fabs(a - mla_oracle_e4m3_to_double((uint8_t)c));
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best_err = err;
      best = c;
    }
  }
  return (uint8_t)(sign | best);
}

/*
 * The decode epilogue for T tokens of H heads:
 *   q_out[t][h][0:512] = ql_nope[t][h][:],  q_out[t][h][512:576] = q_pe[t][h][:]
 *   slot = slot_mapping[t]; if 0 <= slot < num_pages * page_size:
 *     cache[slot / page_size][slot % page_size][d] = x_d            (bf16)
 *                                                  = e4m3(x_d / s)  (fp8)
 *   with x = kv_c[t][:] || k_pe[t][:] and x_d / s the binary32 quotient
 *   (computed in double and rounded once to binary32: the correctly rounded
 *   single-precision division).  Slots < 0 are padding tokens: no write.
 */
void mla_oracle_epilogue(const uint16_t* ql_nope, const uint16_t* q_pe,
                         const uint16_t* kv_c, const uint16_t* k_pe,
                         const int64_t* slot_mapping, int T, int H, uint16_t* q_out,
                         void* cache, int64_t num_pages, int page_size, int kv_dtype,
                         float kv_scale) {
  int t, h, d;
  for (t = 0; t < T; ++t) {
    for (h = 0; h < H; ++h) {
      uint16_t* dst = q_out + ((int64_t)t * H + h) * ORACLE_D_QK;
      for (d = 0; d < 512; ++d) dst[d] = ql_nope[((int64_t)t * H + h) * 512 + d];
      for (d = 0; d < 64; ++d) dst[512 + d] = q_pe[((int64_t)t * H + h) * 64 + d];
    }
    {
      int64_t slot = slot_mapping[t];
      int64_t page, off;
      if (slot < 0 || slot >= num_pages * (int64_t)page_size) continue;
      page = slot / page_size;
      off = slot % page_size;
      for (d = 0; d < ORACLE_D_QK; ++d) {
        uint16_t x = d < 512 ? kv_c[(int64_t)t * 512 + d] : k_pe[(int64_t)t * 64 + (d - 512)];
        int64_t idx = (page * page_size + off) * ORACLE_D_QK + d;
        if (kv_dtype == ORACLE_KV_BF16) {
          ((uint16_t*)cache)[idx] = x;
        } else {
          float y = (float)(mla_oracle_bf16_to_double(x) / (double)kv_scale);
          ((uint8_t*)cache)[idx] = mla_oracle_e4m3_encode(y);
        }
      }
    }
  }
}

/*
 * Cached-prefix expansion of the paged latent into per-head keys and values:
 * for sequence b, cached token j < seq_lens[b], head h < H,
 *   c_j             = dequant(cache[bt[b][j / ps]][j % ps][0:512])
 *   r_j             = dequant(cache[bt[b][j / ps]][j % ps][512:576])
 *   k[t, h, 0:128]  = sum_d W[h][0:128][d]   * c_j[d]
 *   k[t, h, 128:192]= r_j
 *   v[t, h, 0:128]  = sum_d W[h][128:256][d] * c_j[d]
 * with output row t = cu_seqlens[b] + j (the valid tokens, packed).
 * W is [H][256][512] bf16 bits (kv_b_proj, each head's 128 key rows then
 * 128 value rows); k is [T][H][192], v [T][H][128], in double.
 */
void mla_oracle_gather_kv_b_proj(const void* cache, int kv_dtype, double kv_scale,
                                 int page_size, const int32_t* bt, int64_t bt_stride,
                                 const int32_t* seq_lens, const int32_t* cu_seqlens, int B,
                                 const uint16_t* W, int H, double* k, double* v) {
  int b;
  for (b = 0; b < B; ++b) {
    int64_t j, n = seq_lens[b];
#pragma omp parallel for schedule(dynamic, 16)
    for (j = 0; j < n; ++j) {
      double c[ORACLE_D_QK];
      int64_t t = (int64_t)cu_seqlens[b] + j;
      int h, o, d;
      for (d = 0; d < ORACLE_D_QK; ++d)
        c[d] = cache_elem(cache, kv_dtype, kv_scale, bt, bt_stride, b, page_size, j, d);
      for (h = 0; h < H; ++h) {
        for (o = 0; o < 256; ++o) {
          double acc = 0.0;
          const uint16_t* w = W + ((int64_t)h * 256 + o) * 512;
          for (d = 0; d < 512; ++d) acc += mla_oracle_bf16_to_double(w[d]) * c[d];
          if (o < 128)
            k[(t * H + h) * 192 + o] = acc;
          else
            v[(t * H + h) * 128 + (o - 128)] = acc;
        }
        for (d = 0; d < 64; ++d) k[(t * H + h) * 192 + 128 + d] = c[512 + d];
      }
    }
  }
}
