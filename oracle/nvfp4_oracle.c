/*
 * nvfp4_oracle.c -- plain float64 CPU oracle (TEST INFRASTRUCTURE ONLY; see
 * nvfp4_oracle.h for what may use it and for the sources of each step).
 *
 * Every function is the textbook definition written out, in float64, with
 * no blocking, fusion or reordering beyond what that definition states.
 */
#include "nvfp4_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- scalar formats --------------------------------------------------- */

/* e2m1 (OCP FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no
 * inf/NaN.  Exponent field 0 is subnormal: 0.m * 2^(1-1).  The storage type
 * named by the pages is __nv_fp4_e2m1 / float4_e2m1fn_x2. */
double orc_e2m1_value(uint8_t code) {
  int s = (code >> 3) & 1;
  int e = (code >> 1) & 3;
  int m = code & 1;
  double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -mag : mag;
}

/* E4M3 "fn": 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent
 * field 0 is subnormal (0.m * 2^-6); S.1111.111 is NaN; no infinities. */
double orc_e4m3_value(uint8_t byte) {
  int s = (byte >> 7) & 1;
  int e = (byte >> 3) & 15;
  int m = byte & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp(m / 8.0, -6);
  else
    mag = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -mag : mag;
}

double orc_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round |x| to the nearest multiple of the grid spacing of its binade,
 * ties to even (rint in the default rounding mode), for a binary format with
 * `mbits` mantissa bits whose smallest normal binade starts at 2^emin;
 * below 2^emin the spacing stays 2^(emin - mbits) (subnormals). */
static double round_binade(double a, int mbits, int emin) {
  int k;
  double spacing;
  if (a < ldexp(1.0, emin)) {
    spacing = ldexp(1.0, emin - mbits);
  } else {
    (void)frexp(a, &k); /* a = f * 2^k, f in [0.5, 1): binade 2^(k-1) */
    spacing = ldexp(1.0, (k - 1) - mbits);
  }
  return rint(a / spacing) * spacing;
}

uint8_t orc_e2m1_encode(double x) {
  uint8_t sign = signbit(x) ? 8 : 0;
  double v = round_binade(fabs(x), 1, 0);
  int k;
  uint8_t code;
  if (v > 6.0) v = 6.0; /* satfinite */
  if (v < 1.0) {
    code = (uint8_t)(v * 2.0); /* 0 or 0.5 */
  } else {
    double f = frexp(v, &k); /* v = 2^(k-1) * (2f) */
    int e = k - 1;
    int m = (int)((2.0 * f - 1.0) * 2.0);
    code = (uint8_t)(((e + 1) << 1) | m);
  }
  return (uint8_t)(sign | code);
}

uint8_t orc_e4m3_encode(double x) {
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double v = round_binade(fabs(x), 3, -6);
  int k;
  uint8_t code;
  if (v > 448.0) v = 448.0; /* satfinite */
  if (v < ldexp(1.0, -6)) {
    code = (uint8_t)(v / ldexp(1.0, -9)); /* subnormal m in 0..7 */
  } else {
    double f = frexp(v, &k);
    int e = k - 1;
    int m = (int)((2.0 * f - 1.0) * 8.0);
    code = (uint8_t)(((e + 7) << 3) | m);
  }
  return (uint8_t)(sign | code);
}

/* Block recipe.  The quotient amax / (6 g) and x / (s g) are evaluated in
 * float64: 6 g and s g are exact (at most 28 significant bits), and the one
 * rounding of the division cannot move a quotient onto or across a rounding
 * midpoint of E4M3 / e2m1, because a bf16 numerator differs from any
 * midpoint * divisor by at least 2^-36 relative, far above 2^-53.  So these
 * are the exact-real round-to-nearest-even decisions. */
void orc_quantize_block16(const double x[16], double g, uint8_t packed[8],
                          uint8_t* sf) {
  double amax = 0.0;
  double s;
  uint8_t code[16];
  int i;
  for (i = 0; i < 16; ++i) amax = fmax(amax, fabs(x[i]));
  *sf = orc_e4m3_encode(amax / (6.0 * g));
  s = orc_e4m3_value(*sf);
  for (i = 0; i < 16; ++i) {
    if (s == 0.0)
      code[i] = signbit(x[i]) ? 8 : 0;
    else
      code[i] = orc_e2m1_encode(x[i] / (s * g));
  }
  for (i = 0; i < 8; ++i)
    packed[i] = (uint8_t)(code[2 * i] | (code[2 * i + 1] << 4));
}

/* ---- paged cache ------------------------------------------------------ */

/* L_b = (npages - 1) * page_size + last_page_len[b]; 0 without pages. */
int64_t orc_kv_len(const orc_page_table* pt, int32_t b, int32_t page_size) {
  int64_t np = (int64_t)pt->kv_indptr[b + 1] - pt->kv_indptr[b];
  if (np <= 0) return 0;
  return (np - 1) * page_size + pt->last_page_len[b];
}

static uint8_t* row_ptr(const orc_cache* c, int which, int sf, int32_t page,
                        int32_t slot, int32_t head) {
  if (which == 0 && !sf)
    return c->k_data + page * c->k_stride_page + slot * c->k_stride_slot +
           head * c->k_stride_head;
  if (which == 1 && !sf)
    return c->v_data + page * c->v_stride_page + slot * c->v_stride_slot +
           head * c->v_stride_head;
  if (which == 0)
    return c->k_sf + page * c->k_sf_stride_page + slot * c->k_sf_stride_slot +
           head * c->k_sf_stride_head;
  return c->v_sf + page * c->v_sf_stride_page + slot * c->v_sf_stride_slot +
         head * c->v_sf_stride_head;
}

/* Locate token `pos` of request b: page id and slot.  Returns ORC_OK or
 * ORC_BAD_INDEX. */
static int locate(const orc_cache* c, const orc_page_table* pt, int32_t b,
                  int64_t pos, int32_t* page, int32_t* slot) {
  int64_t np, pidx;
  if (b < 0 || b >= pt->batch || pos < 0) return ORC_BAD_INDEX;
  np = (int64_t)pt->kv_indptr[b + 1] - pt->kv_indptr[b];
  pidx = pos / c->page_size;
  if (pidx >= np || pos >= orc_kv_len(pt, b, c->page_size)) return ORC_BAD_INDEX;
  *page = pt->kv_indices[pt->kv_indptr[b] + pidx];
  *slot = (int32_t)(pos % c->page_size);
  if (*page < 0 || *page >= c->num_pages) return ORC_BAD_INDEX;
  return ORC_OK;
}

static void quantize_row(const orc_cache* c, int which, const uint16_t* src,
                         int32_t page, int32_t slot, int32_t head) {
  int dim = which == 0 ? c->head_dim_qk : c->head_dim_vo;
  double g = which == 0 ? c->k_global_scale : c->v_global_scale;
  uint8_t* data = row_ptr(c, which, 0, page, slot, head);
  uint8_t* sfp = row_ptr(c, which, 1, page, slot, head);
  double blk[16];
  int j, i;
  for (j = 0; j < dim / 16; ++j) {
    for (i = 0; i < 16; ++i) blk[i] = orc_bf16_value(src[16 * j + i]);
    orc_quantize_block16(blk, g, data + 8 * j, sfp + j);
  }
}

int orc_quantize_append(const orc_cache* c, const uint16_t* k_bf16,
                        int64_t k_stride_tok, int64_t k_stride_head,
                        const uint16_t* v_bf16, int64_t v_stride_tok,
                        int64_t v_stride_head, int32_t nnz,
                        const int32_t* batch_idx, const int32_t* positions,
                        const orc_page_table* pt) {
  int32_t t, h, page, slot;
  if (c->head_dim_qk % 16 || c->head_dim_vo % 16 || c->page_size <= 0)
    return ORC_BAD_ARGUMENT;
  for (t = 0; t < nnz; ++t)
    if (locate(c, pt, batch_idx[t], positions[t], &page, &slot) != ORC_OK)
      return ORC_BAD_INDEX;
  for (t = 0; t < nnz; ++t) {
    locate(c, pt, batch_idx[t], positions[t], &page, &slot);
    for (h = 0; h < c->num_kv_heads; ++h) {
      quantize_row(c, 0, k_bf16 + t * k_stride_tok + h * k_stride_head, page,
                   slot, h);
      quantize_row(c, 1, v_bf16 + t * v_stride_tok + h * v_stride_head, page,
                   slot, h);
    }
  }
  return ORC_OK;
}

/* x_hat = value(code) * value(scale byte) * g  (nvfp4_to_float in the
 * pages' decode test). */
void orc_dequant_row(const orc_cache* c, int which, int32_t page, int32_t slot,
                     int32_t head, double* out) {
  int dim = which == 0 ? c->head_dim_qk : c->head_dim_vo;
  double g = which == 0 ? c->k_global_scale : c->v_global_scale;
  const uint8_t* data = row_ptr(c, which, 0, page, slot, head);
  const uint8_t* sfp = row_ptr(c, which, 1, page, slot, head);
  int d;
  for (d = 0; d < dim; ++d) {
    uint8_t byte = data[d / 2];
    uint8_t code = (d % 2 == 0) ? (byte & 15) : (byte >> 4);
    out[d] = orc_e2m1_value(code) * orc_e4m3_value(sfp[d / 16]) * g;
  }
}

/* ---- attention -------------------------------------------------------- */

void orc_merge_states(int32_t n, int32_t dim, const double* o_partial,
                      const double* lse_partial, double* o_out,
                      double* lse_out) {
  double M = -INFINITY, sum = 0.0, lse;
  int32_t i, d;
  for (i = 0; i < n; ++i) M = fmax(M, lse_partial[i]);
  for (d = 0; d < dim; ++d) o_out[d] = 0.0;
  if (n == 0 || M == -INFINITY) {
    *lse_out = -INFINITY;
    return;
  }
  for (i = 0; i < n; ++i) sum += exp(lse_partial[i] - M);
  lse = M + log(sum);
  for (i = 0; i < n; ++i) {
    double w = exp(lse_partial[i] - lse);
    for (d = 0; d < dim; ++d) o_out[d] += w * o_partial[(int64_t)i * dim + d];
  }
  *lse_out = lse;
}

/* Exact two-pass softmax attention of `rows` query rows over the keys
 * j in [j0, j1) of request b that each row may see.
 * qv[r*Dk + d] are the query values, limit[r] the last visible key index
 * (inclusive).  Writes o[r*Dv + d] and lse[r]. */
static int attend_range(const orc_cache* c, const orc_page_table* pt, int32_t b,
                        int32_t h_kv, int32_t rows, const double* qv,
                        const int64_t* limit, double sm_scale, int64_t j0,
                        int64_t j1, double* o, double* lse) {
  int32_t dk = c->head_dim_qk, dv = c->head_dim_vo;
  int64_t n = j1 - j0, j;
  int32_t r, d, page, slot;
  double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * rows);
  double* kr = (double*)malloc(sizeof(double) * dk);
  double* vr = (double*)malloc(sizeof(double) * dv);
  double* M = (double*)malloc(sizeof(double) * rows);
  double* Z = (double*)malloc(sizeof(double) * rows);
  int rc = ORC_OK;
  if (!s || !kr || !vr || !M || !Z) {
    rc = ORC_BAD_ARGUMENT;
    goto done;
  }
  /* pass 1: scores s_j = sm_scale * sum_d q_d k_hat_{j,d} */
  for (j = j0; j < j1; ++j) {
    if (locate(c, pt, b, j, &page, &slot) != ORC_OK) {
      rc = ORC_BAD_INDEX;
      goto done;
    }
    orc_dequant_row(c, 0, page, slot, h_kv, kr);
    for (r = 0; r < rows; ++r) {
      double acc = 0.0;
      for (d = 0; d < dk; ++d) acc += qv[(int64_t)r * dk + d] * kr[d];
      s[(j - j0) * rows + r] = sm_scale * acc;
    }
  }
  /* pass 2: M = max over visible keys, Z = sum exp(s_j - M) */
  for (r = 0; r < rows; ++r) {
    M[r] = -INFINITY;
    Z[r] = 0.0;
    for (j = j0; j < j1; ++j)
      if (j <= limit[r]) M[r] = fmax(M[r], s[(j - j0) * rows + r]);
    if (M[r] != -INFINITY)
      for (j = j0; j < j1; ++j)
        if (j <= limit[r]) Z[r] += exp(s[(j - j0) * rows + r] - M[r]);
    for (d = 0; d < dv; ++d) o[(int64_t)r * dv + d] = 0.0;
  }
  /* pass 3: o = sum_j exp(s_j - M) v_hat_j / Z */
  for (j = j0; j < j1; ++j) {
    locate(c, pt, b, j, &page, &slot);
    orc_dequant_row(c, 1, page, slot, h_kv, vr);
    for (r = 0; r < rows; ++r) {
      double w;
      if (j > limit[r] || M[r] == -INFINITY) continue;
      w = exp(s[(j - j0) * rows + r] - M[r]);
      for (d = 0; d < dv; ++d) o[(int64_t)r * dv + d] += w * vr[d];
    }
  }
  for (r = 0; r < rows; ++r) {
    if (M[r] == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    for (d = 0; d < dv; ++d) o[(int64_t)r * dv + d] /= Z[r];
    lse[r] = M[r] + log(Z[r]);
  }
done:
  free(s);
  free(kr);
  free(vr);
  free(M);
  free(Z);
  return rc;
}

int orc_attention_unit(const orc_cache* c, const orc_page_table* pt,
                       const int32_t* qo_indptr, const uint16_t* q_bf16,
                       int64_t q_stride_tok, int64_t q_stride_head,
                       int32_t num_qo_heads, int32_t causal, double sm_scale,
                       int32_t b, int32_t h_kv, int64_t chunk_tokens,
                       double* out, double* lse) {
  int32_t G, nq, rows, r, i, g, d;
  int64_t L, q0, j0;
  double *qv = NULL, *o = NULL, *l = NULL, *oc = NULL, *lc = NULL;
  int64_t* limit = NULL;
  int64_t nchunks, ci;
  int rc = ORC_OK;
  if (num_qo_heads <= 0 || c->num_kv_heads <= 0 ||
      num_qo_heads % c->num_kv_heads || b < 0 || b >= pt->batch || h_kv < 0 ||
      h_kv >= c->num_kv_heads || chunk_tokens < 0)
    return ORC_BAD_ARGUMENT;
  G = num_qo_heads / c->num_kv_heads;
  q0 = qo_indptr[b];
  nq = qo_indptr[b + 1] - qo_indptr[b];
  L = orc_kv_len(pt, b, c->page_size);
  if (nq > L) return ORC_BAD_ARGUMENT;
  rows = nq * G;
  if (rows == 0) return ORC_OK;
  qv = (double*)malloc(sizeof(double) * rows * c->head_dim_qk);
  o = (double*)malloc(sizeof(double) * rows * c->head_dim_vo);
  l = (double*)malloc(sizeof(double) * rows);
  limit = (int64_t*)malloc(sizeof(int64_t) * rows);
  if (!qv || !o || !l || !limit) {
    rc = ORC_BAD_ARGUMENT;
    goto done;
  }
  /* row r = i * G + g : query row i (absolute position L - nq + i), head
   * h_kv * G + g */
  for (i = 0; i < nq; ++i)
    for (g = 0; g < G; ++g) {
      r = i * G + g;
      for (d = 0; d < c->head_dim_qk; ++d)
        qv[(int64_t)r * c->head_dim_qk + d] = orc_bf16_value(
            q_bf16[(q0 + i) * q_stride_tok + (h_kv * G + g) * q_stride_head + d]);
      limit[r] = causal ? (L - nq + i) : (L - 1);
    }
  if (chunk_tokens == 0) {
    rc = attend_range(c, pt, b, h_kv, rows, qv, limit, sm_scale, 0, L, o, l);
  } else {
    nchunks = (L + chunk_tokens - 1) / chunk_tokens;
    oc = (double*)malloc(sizeof(double) * nchunks * rows * c->head_dim_vo);
    lc = (double*)malloc(sizeof(double) * nchunks * rows);
    if (!oc || !lc) {
      rc = ORC_BAD_ARGUMENT;
      goto done;
    }
    for (ci = 0; ci < nchunks && rc == ORC_OK; ++ci) {
      j0 = ci * chunk_tokens;
      rc = attend_range(c, pt, b, h_kv, rows, qv, limit, sm_scale, j0,
                        (j0 + chunk_tokens < L) ? j0 + chunk_tokens : L,
                        oc + ci * rows * c->head_dim_vo, lc + ci * rows);
    }
    if (rc == ORC_OK) {
      /* gather the chunk states of each row and merge them */
      double* orow = (double*)malloc(sizeof(double) * nchunks * c->head_dim_vo);
      double* lrow = (double*)malloc(sizeof(double) * nchunks);
      for (r = 0; r < rows && orow && lrow; ++r) {
        for (ci = 0; ci < nchunks; ++ci) {
          memcpy(orow + ci * c->head_dim_vo,
                 oc + (ci * rows + r) * c->head_dim_vo,
                 sizeof(double) * c->head_dim_vo);
          lrow[ci] = lc[ci * rows + r];
        }
        orc_merge_states((int32_t)nchunks, c->head_dim_vo, orow, lrow,
                         o + (int64_t)r * c->head_dim_vo, l + r);
      }
      if (!orow || !lrow) rc = ORC_BAD_ARGUMENT;
      free(orow);
      free(lrow);
    }
  }
  if (rc == ORC_OK)
    for (i = 0; i < nq; ++i)
      for (g = 0; g < G; ++g) {
        int64_t row = q0 + i, head = h_kv * G + g;
        r = i * G + g;
        for (d = 0; d < c->head_dim_vo; ++d)
          out[(row * num_qo_heads + head) * c->head_dim_vo + d] =
              o[(int64_t)r * c->head_dim_vo + d];
        lse[row * num_qo_heads + head] = l[r];
      }
done:
  free(qv);
  free(o);
  free(l);
  free(limit);
  free(oc);
  free(lc);
  return rc;
}

/* ---- attention with FP4 query and probabilities ------------------------ */

/* x -> NVFP4 (orc_quantize_block16 with global scale 1) -> value. */
static void fp4_round16(const double x[16], double y[16]) {
  uint8_t packed[8], sf;
  double s;
  int i;
  orc_quantize_block16(x, 1.0, packed, &sf);
  s = orc_e4m3_value(sf);
  for (i = 0; i < 16; ++i)
    y[i] = orc_e2m1_value((uint8_t)((packed[i / 2] >> (4 * (i & 1))) & 15)) * s;
}

int orc_attention_unit_fp4qp(const orc_cache* c, const orc_page_table* pt,
                             const int32_t* qo_indptr, const uint16_t* q_bf16,
                             int64_t q_stride_tok, int64_t q_stride_head,
                             int32_t num_qo_heads, int32_t causal,
                             double sm_scale, int32_t b, int32_t h_kv,
                             double* out, double* lse) {
  const double kPScale = 448.0 * 6.0;
  int32_t G, nq, rows, r, i, g, d, page, slot, t;
  int32_t dk = c->head_dim_qk, dv = c->head_dim_vo;
  int64_t L, q0, j, blk;
  double *qv = NULL, *s = NULL, *M = NULL, *Z = NULL, *o = NULL, *kr = NULL,
         *vb = NULL;
  int64_t* limit = NULL;
  int rc = ORC_OK;
  if (num_qo_heads <= 0 || c->num_kv_heads <= 0 ||
      num_qo_heads % c->num_kv_heads || b < 0 || b >= pt->batch || h_kv < 0 ||
      h_kv >= c->num_kv_heads || dk % 16)
    return ORC_BAD_ARGUMENT;
  G = num_qo_heads / c->num_kv_heads;
  q0 = qo_indptr[b];
  nq = qo_indptr[b + 1] - qo_indptr[b];
  L = orc_kv_len(pt, b, c->page_size);
  if (nq > L) return ORC_BAD_ARGUMENT;
  rows = nq * G;
  if (rows == 0) return ORC_OK;
  qv = (double*)malloc(sizeof(double) * rows * dk);
  s = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * rows);
  M = (double*)malloc(sizeof(double) * rows);
  Z = (double*)malloc(sizeof(double) * rows);
  o = (double*)malloc(sizeof(double) * rows * dv);
  kr = (double*)malloc(sizeof(double) * dk);
  vb = (double*)malloc(sizeof(double) * 16 * dv);
  limit = (int64_t*)malloc(sizeof(int64_t) * rows);
  if (!qv || !s || !M || !Z || !o || !kr || !vb || !limit) {
    rc = ORC_BAD_ARGUMENT;
    goto done;
  }
  /* row r = i * G + g: the query row quantised per 16 dims */
  for (i = 0; i < nq; ++i)
    for (g = 0; g < G; ++g) {
      double x[16];
      r = i * G + g;
      for (d = 0; d < dk; d += 16) {
        for (t = 0; t < 16; ++t)
          x[t] = orc_bf16_value(q_bf16[(q0 + i) * q_stride_tok +
                                       (h_kv * G + g) * q_stride_head + d + t]);
        fp4_round16(x, qv + (int64_t)r * dk + d);
      }
      limit[r] = causal ? L - nq + i : L - 1;
    }
  /* scores with the quantised query, the row maxima and sums of exp */
  for (j = 0; j < L; ++j) {
    if (locate(c, pt, b, j, &page, &slot) != ORC_OK) {
      rc = ORC_BAD_INDEX;
      goto done;
    }
    orc_dequant_row(c, 0, page, slot, h_kv, kr);
    for (r = 0; r < rows; ++r) {
      double acc = 0.0;
      for (d = 0; d < dk; ++d) acc += qv[(int64_t)r * dk + d] * kr[d];
      s[j * rows + r] = sm_scale * acc;
    }
  }
  for (r = 0; r < rows; ++r) {
    M[r] = -INFINITY;
    Z[r] = 0.0;
    for (j = 0; j <= limit[r]; ++j) M[r] = fmax(M[r], s[j * rows + r]);
    if (M[r] != -INFINITY)
      for (j = 0; j <= limit[r]; ++j) Z[r] += exp(s[j * rows + r] - M[r]);
    for (d = 0; d < dv; ++d) o[(int64_t)r * dv + d] = 0.0;
  }
  /* per block of 16 key positions: P' = 448 * 6 * p quantised, o += P_hat v */
  for (blk = 0; blk * 16 < L; ++blk) {
    for (t = 0; t < 16; ++t) {
      j = blk * 16 + t;
      if (j < L) {
        locate(c, pt, b, j, &page, &slot);
        orc_dequant_row(c, 1, page, slot, h_kv, vb + (int64_t)t * dv);
      } else {
        for (d = 0; d < dv; ++d) vb[(int64_t)t * dv + d] = 0.0;
      }
    }
    for (r = 0; r < rows; ++r) {
      double pp[16], ph[16];
      if (M[r] == -INFINITY) continue;
      for (t = 0; t < 16; ++t) {
        j = blk * 16 + t;
        pp[t] = (j < L && j <= limit[r]) ? kPScale * exp(s[j * rows + r] - M[r]) : 0.0;
      }
      fp4_round16(pp, ph);
      for (t = 0; t < 16; ++t)
        if (ph[t] != 0.0)
          for (d = 0; d < dv; ++d)
            o[(int64_t)r * dv + d] += ph[t] * vb[(int64_t)t * dv + d];
    }
  }
  for (i = 0; i < nq; ++i)
    for (g = 0; g < G; ++g) {
      int64_t row = q0 + i, head = h_kv * G + g;
      r = i * G + g;
      for (d = 0; d < dv; ++d)
        out[(row * num_qo_heads + head) * dv + d] =
            M[r] == -INFINITY ? 0.0 : o[(int64_t)r * dv + d] / (kPScale * Z[r]);
      lse[row * num_qo_heads + head] = M[r] == -INFINITY ? -INFINITY : M[r] + log(Z[r]);
    }
done:
  free(qv);
  free(s);
  free(M);
  free(Z);
  free(o);
  free(kr);
  free(vb);
  free(limit);
  return rc;
}
