/*
 * Oracle for split-KV verify attention (EAGLE target-verify, topk = 1).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA product path
 * never links, imports or calls it, and this file shares no code, header,
 * table or constant with that path.
 *
 * What it computes (the plain definition, in fp64, with full score rows):
 *   sglang "verify_splitkv.py" (page 1), module docstring and the two stage
 *   kernels: every draft query row i of sequence b attends, under one softmax,
 *   over
 *     - every prefix key j < P_b, gathered through kv_indices[kv_indptr[b]+j],
 *       with score sm_scale * k_scale * <q, K_pool[loc, kvh]> and value
 *       v_scale * V_pool[loc, kvh]            ("_verify_prefix_stage1");
 *     - every draft key t <= i of the same sequence, with score
 *       sm_scale * <q, k_ext[s_b + t, kvh]> and value v_ext[s_b + t, kvh],
 *       no k_scale / v_scale            ("_verify_combine_stage2", part (b)),
 *   where kvh = h / (h_q / h_kv).  The split-KV partition and the log-sum-exp
 *   merges of the method only reorder this sum, so the oracle materialises the
 *   whole score row instead and never splits.
 *
 * Readings taken where the page is silent:
 *   - empty prefix (P_b = 0): the output is causal attention over the drafts
 *     alone (the page's stage-2 merge would produce NaN there);
 *   - k_scale and v_scale are dequantisation multipliers on prefix scores and
 *     prefix values only;
 *   - an fp8 pool is decoded exactly (e4m3 "fn" variant: bias 7, no infinity,
 *     S.1111.111 is NaN, largest finite 448); q is used unquantised;
 *   - L_b = qo_indptr[b+1] - qo_indptr[b] rows per sequence;
 *   - tree verify (speculative topk > 1), when a custom mask is given: the
 *     mask of sequence b is an L_b x (P_b + L_b) byte matrix stored row-major
 *     from mask_indptr[b] (row i = draft query i, column j = prefix keys then
 *     draft keys, nonzero = visible), the layout the "aiter_backend.py" page
 *     builds for target verify (seq_mask_len = draft_num * (seq_len +
 *     draft_num), mask_indptr = its running sum).  With the prefix part of
 *     the mask skipped (skip_prefix_custom_mask, the verify default), every
 *     prefix key stays visible and only the draft columns are read; draft key
 *     t is visible to row i iff mask[mask_indptr[b] + i*(P_b+L_b) + P_b + t];
 *   - a row that sees no key at all (empty prefix and no visible draft) has
 *     output 0 and lse -inf;
 *   - drafts already in a paged cache (the unified target-verify path of the
 *     "aiter_backend.py" page: block_table [B, max_blocks] of page ids over a
 *     pool of pages of page_size tokens, seqused_k = seq_lens + draft_num,
 *     causal): the keys of sequence b are cache positions 0 .. P_b + L_b - 1,
 *     position j at pool row block_table[b][j / page_size] * page_size +
 *     j % page_size; positions < P_b = seq_lens[b] are the prefix, the next
 *     L_b are the drafts (row i sees drafts t <= i); every key is a cache
 *     entry, so k_scale and v_scale apply to the drafts too.
 *
 * Writing new K/V rows into the cache (the draft K/V store that precedes
 * unified verify on the "aiter_backend.py" page, where the bf16 -> fp8 cast
 * and the paged write are one kernel, given the cache's k_scale / v_scale as
 * descales): the stored code of a bf16 value x is the cache dtype's
 * round-to-nearest-even of the binary32 quotient x / scale; an e4m3 cache
 * saturates finite quotients beyond +-448 to +-448 (the saturating fp8 cast
 * such kernels use), a NaN stays NaN.  Reading it back multiplies by the same
 * scale, so a write followed by paged verify sees the dequantised value.
 *
 * Debug outputs (optional) split the same sum into its prefix part and its
 * draft part: o_prefix / lse_prefix over the prefix keys only (lse = -inf and
 * o = 0 when P_b = 0) and o_draft / lse_draft over the causal drafts only.
 * Log-sum-exp values are natural logarithms.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_POOL_BF16 0
#define ORC_POOL_E4M3 1
#define ORC_IDX_I32 0
#define ORC_IDX_I64 1

typedef struct {
  int64_t batch;   /* B: number of sequences                              */
  int64_t h_q;     /* query heads                                         */
  int64_t h_kv;    /* key/value heads                                     */
  int64_t d;       /* query/key head size                                 */
  int64_t dv;      /* value head size                                     */
  int64_t n_rows;  /* rows of q / k_ext / v_ext / o                       */
  /* q [n_rows, h_q, d], k_ext [n_rows, h_kv, d], v_ext [n_rows, h_kv, dv]:
     bf16 bit patterns; strides in elements, last dimension contiguous.    */
  const uint16_t* q;     int64_t q_s0, q_s1;
  const uint16_t* k_ext; int64_t ke_s0, ke_s1;
  const uint16_t* v_ext; int64_t ve_s0, ve_s1;
  /* K/V pools [pool_tokens, h_kv, d|dv]: bf16 bits (uint16) or e4m3 codes
     (uint8) according to pool_dtype; strides in elements.                  */
  const void* k_pool; int64_t kp_s0, kp_s1;
  const void* v_pool; int64_t vp_s0, vp_s1;
  int32_t pool_dtype;
  int32_t idx_dtype;
  const int32_t* qo_indptr;  /* [B+1] */
  const int32_t* kv_indptr;  /* [B+1] */
  const void* kv_indices;    /* int32 or int64, per idx_dtype */
  double sm_scale, k_scale, v_scale;
  const uint8_t* custom_mask;   /* NULL: causal drafts (t <= i) */
  const int64_t* mask_indptr;   /* [B+1], used with custom_mask  */
  /* drafts in a paged cache (kv_indptr / kv_indices / k_ext / v_ext unused) */
  int32_t paged;
  const int32_t* block_table;   /* [B, bt_s0] page ids */
  int64_t bt_s0;
  int64_t page_size;
  const int32_t* seq_lens;      /* [B] cached tokens before the drafts */
} orc_problem;

/* bf16 is the upper half of an IEEE-754 binary32: widen the bit pattern. */
double orc_bf16_to_f64(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* e4m3 "fn": 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no
   infinities, S.1111.111 is NaN.  Subnormals: 2^-6 * m/8.                  */
double orc_e4m3_to_f64(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

static double e4m3_table[256];
static int e4m3_table_ready = 0;

static void build_e4m3_table(void) {
  if (e4m3_table_ready) return;
  for (int c = 0; c < 256; ++c) e4m3_table[c] = orc_e4m3_to_f64((uint8_t)c);
  e4m3_table_ready = 1;
}

static double pool_elem(const orc_problem* p, const void* pool, int64_t off) {
  if (p->pool_dtype == ORC_POOL_E4M3) return e4m3_table[((const uint8_t*)pool)[off]];
  return orc_bf16_to_f64(((const uint16_t*)pool)[off]);
}

/* Pool row of cache position j of sequence b (paged problems). */
static int64_t paged_row(const orc_problem* p, int64_t b, int64_t j) {
  return (int64_t)p->block_table[b * p->bt_s0 + j / p->page_size] * p->page_size + j % p->page_size;
}

static int64_t kv_index(const orc_problem* p, int64_t n) {
  if (p->idx_dtype == ORC_IDX_I64) return ((const int64_t*)p->kv_indices)[n];
  return (int64_t)((const int32_t*)p->kv_indices)[n];
}

/* Pool row of prefix key j of sequence b (p_b = kv_indptr[b]). */
static int64_t prefix_row(const orc_problem* p, int64_t b, int64_t p_b, int64_t j) {
  return p->paged ? paged_row(p, b, j) : kv_index(p, p_b + j);
}

/* Value element c of draft key t of sequence b (KV head kvh). */
static double draft_value(const orc_problem* p, int64_t b, int64_t s_b, int64_t P_b, int64_t t, int64_t kvh,
                          int64_t c) {
  if (p->paged)
    return p->v_scale * pool_elem(p, p->v_pool, paged_row(p, b, P_b + t) * p->vp_s0 + kvh * p->vp_s1 + c);
  return orc_bf16_to_f64(p->v_ext[(s_b + t) * p->ve_s0 + kvh * p->ve_s1 + c]);
}

/* Is draft key t visible to draft row i of sequence b? */
static int draft_visible(const orc_problem* p, int64_t b, int64_t i, int64_t t, int64_t P_b, int64_t L_b) {
  if (!p->custom_mask) return t <= i;
  return p->custom_mask[p->mask_indptr[b] + i * (P_b + L_b) + P_b + t] != 0;
}

/* One (sequence b, query head h): every draft row of b.  Scratch holds the
   decoded q row, the score row and a value accumulator.                     */
static void one_head(const orc_problem* p, int64_t b, int64_t h, double* out,
                     double* o_prefix, double* lse_prefix, double* o_draft,
                     double* lse_draft) {
  const int64_t group = p->h_q / p->h_kv;
  const int64_t kvh = h / group;
  const int64_t s_b = p->qo_indptr[b];
  const int64_t L_b = (int64_t)p->qo_indptr[b + 1] - s_b;
  const int64_t p_b = p->paged ? 0 : p->kv_indptr[b];
  const int64_t P_b = p->paged ? (int64_t)p->seq_lens[b] : (int64_t)p->kv_indptr[b + 1] - p_b;
  const int64_t D = p->d, DV = p->dv;

  double* qrow = (double*)malloc(sizeof(double) * (size_t)D);
  double* score = (double*)malloc(sizeof(double) * (size_t)(P_b + L_b + 1));
  double* acc = (double*)malloc(sizeof(double) * (size_t)DV);
  double* acc2 = (double*)malloc(sizeof(double) * (size_t)DV);

  for (int64_t i = 0; i < L_b; ++i) {
    const int64_t row = s_b + i;
    for (int64_t c = 0; c < D; ++c) qrow[c] = orc_bf16_to_f64(p->q[row * p->q_s0 + h * p->q_s1 + c]);

    /* scores: prefix keys first, then the visible drafts t <= i */
    for (int64_t j = 0; j < P_b; ++j) {
      const int64_t loc = prefix_row(p, b, p_b, j);
      double dot = 0.0;
      for (int64_t c = 0; c < D; ++c) dot += qrow[c] * pool_elem(p, p->k_pool, loc * p->kp_s0 + kvh * p->kp_s1 + c);
      score[j] = p->sm_scale * p->k_scale * dot;
    }
    for (int64_t t = 0; t < L_b; ++t) {
      double dot = 0.0;
      if (p->paged) {
        const int64_t loc = paged_row(p, b, P_b + t);
        for (int64_t c = 0; c < D; ++c) dot += qrow[c] * pool_elem(p, p->k_pool, loc * p->kp_s0 + kvh * p->kp_s1 + c);
        dot *= p->k_scale;
      } else {
        for (int64_t c = 0; c < D; ++c)
          dot += qrow[c] * orc_bf16_to_f64(p->k_ext[(s_b + t) * p->ke_s0 + kvh * p->ke_s1 + c]);
      }
      score[P_b + t] = draft_visible(p, b, i, t, P_b, L_b) ? p->sm_scale * dot : -INFINITY;
    }
    const int64_t n_keys = P_b + L_b;

    /* full softmax over the whole row */
    double mx = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) if (score[j] > mx) mx = score[j];
    double denom = 0.0;
    for (int64_t c = 0; c < DV; ++c) acc[c] = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
      const double w = (score[j] == -INFINITY) ? 0.0 : exp(score[j] - mx);
      denom += w;
      if (j < P_b) {
        const int64_t loc = prefix_row(p, b, p_b, j);
        for (int64_t c = 0; c < DV; ++c)
          acc[c] += w * p->v_scale * pool_elem(p, p->v_pool, loc * p->vp_s0 + kvh * p->vp_s1 + c);
      } else {
        const int64_t t = j - P_b;
        for (int64_t c = 0; c < DV; ++c)
          acc[c] += w * draft_value(p, b, s_b, P_b, t, kvh, c);
      }
    }
    double* o = out + (row * p->h_q + h) * DV;
    for (int64_t c = 0; c < DV; ++c) o[c] = (mx == -INFINITY) ? 0.0 : acc[c] / denom;

    if (o_prefix) {
      /* prefix keys alone */
      double* op = o_prefix + (row * p->h_q + h) * DV;
      if (P_b == 0) {
        for (int64_t c = 0; c < DV; ++c) op[c] = 0.0;
        lse_prefix[row * p->h_q + h] = -INFINITY;
      } else {
        double pm = -INFINITY;
        for (int64_t j = 0; j < P_b; ++j) if (score[j] > pm) pm = score[j];
        double pd = 0.0;
        for (int64_t c = 0; c < DV; ++c) acc2[c] = 0.0;
        for (int64_t j = 0; j < P_b; ++j) {
          const double w = exp(score[j] - pm);
          const int64_t loc = prefix_row(p, b, p_b, j);
          pd += w;
          for (int64_t c = 0; c < DV; ++c)
            acc2[c] += w * p->v_scale * pool_elem(p, p->v_pool, loc * p->vp_s0 + kvh * p->vp_s1 + c);
        }
        for (int64_t c = 0; c < DV; ++c) op[c] = acc2[c] / pd;
        lse_prefix[row * p->h_q + h] = pm + log(pd);
      }
      /* causal drafts alone */
      double* od = o_draft + (row * p->h_q + h) * DV;
      double dm = -INFINITY;
      for (int64_t t = 0; t < L_b; ++t) if (score[P_b + t] > dm) dm = score[P_b + t];
      double dd = 0.0;
      for (int64_t c = 0; c < DV; ++c) acc2[c] = 0.0;
      for (int64_t t = 0; t < L_b; ++t) {
        if (score[P_b + t] == -INFINITY) continue;
        const double w = exp(score[P_b + t] - dm);
        dd += w;
        for (int64_t c = 0; c < DV; ++c)
          acc2[c] += w * draft_value(p, b, s_b, P_b, t, kvh, c);
      }
      for (int64_t c = 0; c < DV; ++c) od[c] = (dm == -INFINITY) ? 0.0 : acc2[c] / dd;
      lse_draft[row * p->h_q + h] = (dm == -INFINITY) ? -INFINITY : dm + log(dd);
    }
  }
  free(qrow);
  free(score);
  free(acc);
  free(acc2);
}

/* Output rows for sequences [b0, b1) and query heads [h0, h1).
   out (and the optional debug arrays) are dense [n_rows, h_q, dv] / [n_rows,
   h_q]; rows and heads outside the requested ranges are left untouched.
   nthreads <= 0 uses every processor (whatever an earlier call asked for).
   Returns 0, or -1 on bad ranges.  */
int orc_verify_forward(const orc_problem* p, int64_t b0, int64_t b1, int64_t h0, int64_t h1,
                       double* out, double* o_prefix, double* lse_prefix, double* o_draft,
                       double* lse_draft, int nthreads) {
  if (b0 < 0 || b1 > p->batch || b0 > b1 || h0 < 0 || h1 > p->h_q || h0 > h1) return -1;
  if (p->h_kv <= 0 || p->h_q % p->h_kv != 0) return -1;
  build_e4m3_table();
  const int64_t nb = b1 - b0, nh = h1 - h0;
  const int64_t n_work = nb * nh;
#ifdef _OPENMP
  omp_set_num_threads(nthreads > 0 ? nthreads : omp_get_num_procs());
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int64_t w = 0; w < n_work; ++w) {
    const int64_t b = b0 + w / nh;
    const int64_t h = h0 + w % nh;
    one_head(p, b, h, out, o_prefix, lse_prefix, o_draft, lse_draft);
  }
  return 0;
}

/* Threads an OpenMP parallel region would use (1 without OpenMP). */
int orc_max_threads(int nthreads) {
#ifdef _OPENMP
  omp_set_num_threads(nthreads > 0 ? nthreads : omp_get_num_procs());
  return omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* Element-wise decoders, exported so tests can check them exhaustively. */
void orc_decode_bf16(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(in[i]);
}

void orc_decode_e4m3(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_f64(in[i]);
}

/* ---------------------------------------------------------------------------
 * Quantised store of new K/V values (see the header comment).
 * ------------------------------------------------------------------------- */

/* e4m3 "fn" code nearest to y, ties to the code with an even mantissa, finite
   values beyond the largest finite code (448) saturating to it; NaN -> the
   NaN code.  Written as a search over the 127 non-negative finite codes,
   whose values increase with the code.                                       */
static uint8_t encode_e4m3_satfinite(float y) {
  if (isnan(y)) return 0x7F;
  const uint8_t sign = signbit(y) ? 0x80 : 0x00;
  const double a = fabs((double)y);
  uint8_t best = 0;
  for (int c = 1; c <= 0x7E; ++c) {
    const double lo = orc_e4m3_to_f64((uint8_t)(c - 1)), hi = orc_e4m3_to_f64((uint8_t)c);
    if (a >= hi) {
      best = (uint8_t)c;  /* at or above this code: keep climbing */
      continue;
    }
    /* lo <= a < hi: nearer of the two, a tie goes to the even code */
    const double dl = a - lo, dh = hi - a;
    if (dh < dl || (dh == dl && (c & 1) == 0)) best = (uint8_t)c;
    else best = (uint8_t)(c - 1);
    break;
  }
  return (uint8_t)(sign | best);
}

/* bf16 nearest to y (ties to even), i.e. the binary32 values whose low 16
   bits are zero; beyond the largest finite bf16 plus half an ulp -> infinity. */
static uint16_t encode_bf16_rne(float y) {
  uint32_t w;
  memcpy(&w, &y, sizeof w);
  if (isnan(y)) return (uint16_t)((w >> 16) | 0x40);
  const uint32_t lo = w & 0xFFFF0000u;
  if (lo == w) return (uint16_t)(w >> 16);
  const uint32_t hi = lo + 0x10000u;  /* next value away from zero */
  float flo, fhi;
  memcpy(&flo, &lo, sizeof flo);
  memcpy(&fhi, &hi, sizeof fhi);
  const double vy = fabs((double)y), vlo = fabs((double)flo);
  /* past the largest finite value the next step is 2^128 (infinity) */
  const double vhi = isinf(fhi) ? ldexp(1.0, 128) : fabs((double)fhi);
  const double dl = vy - vlo, dh = vhi - vy;
  if (dh < dl || (dh == dl && ((hi >> 16) & 1u) == 0)) return (uint16_t)(hi >> 16);
  return (uint16_t)(lo >> 16);
}

/* dst[i] = code of bf16 src[i] / scale in the cache dtype (ORC_POOL_BF16:
   uint16 bits, ORC_POOL_E4M3: uint8 codes); the quotient is binary32.       */
void orc_quantize(const uint16_t* src, int64_t n, float scale, int dst_dtype, void* dst) {
  for (int64_t i = 0; i < n; ++i) {
    const float x = (float)orc_bf16_to_f64(src[i]);
    const float y = x / scale;
    if (dst_dtype == ORC_POOL_E4M3)
      ((uint8_t*)dst)[i] = encode_e4m3_satfinite(y);
    else
      ((uint16_t*)dst)[i] = encode_bf16_rne(y);
  }
}

/* Element-wise encoders alone (binary32 in), for the tests. */
void orc_encode_e4m3(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = encode_e4m3_satfinite(in[i]);
}

void orc_encode_bf16(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = encode_bf16_rne(in[i]);
}
