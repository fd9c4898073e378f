/*
 * MSA decode oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU restatement of what the MiniMax Sparse Attention (MSA)
 * decode path computes, in FP64, written from the pages' prose. Only the tests,
 * the package's smoke check and the benchmark's CPU-baseline leg may load it;
 * the product path (libmsa) never does, and the two share no code.
 *
 * Sources, cited below by the short tag in brackets:
 *   [vLLM-zh]  "vLLM 对 MiniMax-M3.1-Flash 的 Day-0 支持：NVFP4 MSA 内核、MegaMoE 与
 *              Agentic 基准测试" (agentlenshq.com) — the vLLM day-0 blog post on
 *              MiniMax-M3.1-Flash, Chinese rewrite.
 *   [vLLM-ja]  the same vLLM blog post, Japanese translation (spke.com).
 *   [MSA-fig]  "MiniMax goes sparse: reading the M3 attention mechanism from one
 *              diagram" (atlascloud.ai, Arabic).
 *
 * Geometry fixed by the method as these pages and the workload define it:
 * 4 KV heads (= GQA groups) of head dim 128, 8 query heads per group (32 query
 * heads), one shared index-key head of dim 128, 128-token KV blocks, top-16
 * blocks per group. NVFP4 = E2M1 element codes with one E4M3 scale per 16
 * consecutive elements (no second-level scale).
 *
 * Cache layout (data plane and scale plane stored separately, element 2i in the
 * low nibble of byte i):
 *   k_data/v_data  [num_pages][4][128][64]  u8   k_scale/v_scale [num_pages][4][128][8] u8
 *   ki_data        [num_pages][128][64]     u8   ki_scale        [num_pages][128][8]    u8
 *   q              [total_rows][32][128] E4M3,   q_idx [total_rows][4][128] E4M3
 * Request b owns rows [q_indptr[b], q_indptr[b+1]); row r of R sits at position
 * N-R+r (N = context_lens[b], counting this step's rows) and sees tokens t <= N-R+r.
 *
 * Parity pins for every function here live in tests/test_oracle_*.py; output
 * values of the whole path beyond those pins are checked only against this file
 * (the pages print no worked example).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_G 4        /* KV heads = GQA groups */
#define OR_HQ 32      /* query heads */
#define OR_D 128      /* head dim */
#define OR_BLK 128    /* tokens per KV block */

enum { OR_OK = 0, OR_EINVAL = -1, OR_ENOMEM = -2 };

/* ------------------------------------------------------------------------- */
/* Formats. [vLLM-zh] "使用 CUDA 13.4 QMUL4 指令将 NVFP4 反量化为 FP8": the cache holds */
/* NVFP4 (E2M1 values scaled per 16 elements by an E4M3 factor); queries are   */
/* FP8 E4M3; the kernel turns NVFP4 into FP8 and runs FP8 MMA.                  */
/* ------------------------------------------------------------------------- */

/* E2M1: sign bit 3, exponent bits 2:1 (bias 1), mantissa bit 0. */
double oracle_e2m1_value(int code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return s ? -v : v;
}

/* E4M3 (OCP "FN" variant): sign bit 7, exponent bits 6:3 (bias 7), mantissa bits
 * 2:0; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; no infinities. */
double oracle_e4m3_value(int byte) {
  int s = (byte >> 7) & 1, e = (byte >> 3) & 15, m = byte & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  v = (e == 0) ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* Round to the nearest E4M3 value, ties to the even code, saturating to
 * +-448 (no overflow to NaN); NaN stays NaN. Done by plain search over the
 * 127 non-negative finite codes, whose values increase with the code. */
int oracle_e4m3_round(double x) {
  int sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  int c;
  if (isnan(x)) return 0x7F;
  if (a >= 448.0) return sign | 0x7E;
  c = 0;
  while (c < 0x7E && oracle_e4m3_value(c + 1) <= a) c++;
  if (oracle_e4m3_value(c) != a) {
    double lo = a - oracle_e4m3_value(c), hi = oracle_e4m3_value(c + 1) - a;
    if (hi < lo || (hi == lo && (c & 1))) c = c + 1;
  }
  return sign | c;
}

/* The FP8 value the MMA consumes for one NVFP4 element: the exact product of
 * the E2M1 element and its E4M3 group scale, re-rounded to E4M3. The re-rounding
 * is what FP8 MMA after dequantisation implies ([vLLM-zh] "NVIDIA Rubin MSA 内核":
 * the FP16 path on Rubin avoids "the E4M3 re-rounding FP8 MMA needs"). */
double oracle_dequant_value(int code, int scale_byte) {
  return oracle_e4m3_value(oracle_e4m3_round(oracle_e2m1_value(code) * oracle_e4m3_value(scale_byte)));
}

/* The exact value of one NVFP4 element: its E2M1 value times its E4M3 group scale,
 * with no re-rounding. [vLLM-zh] "Rubin MSA kernels": dequantising to FP16 keeps the
 * product exact and the scores free of the E4M3 re-rounding an FP8 MMA needs; the
 * exact-score indexer computes the index scores from these values. */
double oracle_dequant_value_exact(int code, int scale_byte) {
  return oracle_e2m1_value(code) * oracle_e4m3_value(scale_byte);
}

/* All 256 scales x 16 codes, out[scale*16 + code]. The oracle looks values up
 * here instead of re-running the search per element; the table is the same
 * definition, evaluated once. */
static double g_dq[256 * 16];
static int g_dq_ready = 0;
void oracle_dequant_table(double* out) {
  int s, c;
  if (!g_dq_ready) {
    for (s = 0; s < 256; s++)
      for (c = 0; c < 16; c++) g_dq[s * 16 + c] = oracle_dequant_value(c, s);
    g_dq_ready = 1;
  }
  if (out) memcpy(out, g_dq, sizeof(g_dq));
}

/* Exact dequantisation of one 128-element NVFP4 row (no E4M3 re-rounding). */
static void dequant_row_exact(const uint8_t* codes, const uint8_t* scales, double* out) {
  int i;
  for (i = 0; i < OR_D; i++) {
    int code = (i & 1) ? (codes[i / 2] >> 4) : (codes[i / 2] & 15);
    out[i] = oracle_dequant_value_exact(code, scales[i / 16]);
  }
}

/* Dequantise one 128-element NVFP4 row (64 code bytes, 8 scale bytes). */
static void dequant_row(const uint8_t* codes, const uint8_t* scales, double* out) {
  int j;
  for (j = 0; j < OR_D; j++) {
    int byte = codes[j / 2];
    int code = (j & 1) ? (byte >> 4) : (byte & 15);
    out[j] = g_dq[scales[j / 16] * 16 + code];
  }
}

/* ------------------------------------------------------------------------- */
/* Arguments                                                                  */
/* ------------------------------------------------------------------------- */
typedef struct {
  int32_t num_reqs, num_pages, max_pages_per_req, top_k;
  double sm_scale;
  const int32_t* context_lens;
  const int32_t* q_indptr;
  const int32_t* block_table;
  const uint8_t *q, *q_idx;
  const uint8_t *k_data, *k_scale, *v_data, *v_scale, *ki_data, *ki_scale;
  int32_t exact_index_scores; /* 1: index keys dequantised exactly (no E4M3 re-rounding) */
} oracle_args;

static int req_geometry(const oracle_args* a, int b, int* N, int* R, int* row0) {
  if (b < 0 || b >= a->num_reqs) return OR_EINVAL;
  *N = a->context_lens[b];
  *row0 = a->q_indptr[b];
  *R = a->q_indptr[b + 1] - a->q_indptr[b];
  if (*N < 0 || *R < 0 || *R > *N || *N > a->max_pages_per_req * OR_BLK) return OR_EINVAL;
  return OR_OK;
}

static int page_of(const oracle_args* a, int b, int block) {
  int p = a->block_table[(int64_t)b * a->max_pages_per_req + block];
  return (p >= 0 && p < a->num_pages) ? p : -1;
}

/* ------------------------------------------------------------------------- */
/* Step 1 — index scan. [vLLM-zh] "MiniMax 稀疏注意力的工作原理": a lightweight     */
/* indexer scores every key in the context with one index query per GQA group   */
/* against a single shared index-key head. [MSA-fig] §1 step 1: K_idx has one   */
/* head shared by all groups; score = Q_idx · K_idxᵀ. The score is the plain    */
/* dot product (the pages name no scale or activation).                        */
/* s[(r*4 + g)*N + t], -inf where t > N-R+r.                                   */
/* ------------------------------------------------------------------------- */
int oracle_token_scores(const oracle_args* a, int b, double* s) {
  int N, R, row0, t, r, g, j, rc;
  double kv[OR_D];
  double* qd;
  oracle_dequant_table(NULL);
  if ((rc = req_geometry(a, b, &N, &R, &row0)) != OR_OK) return rc;
  /* the request's index queries as values, [r][g][j] */
  qd = (double*)malloc(sizeof(double) * ((size_t)R * OR_G * OR_D + 1));
  if (!qd) return OR_ENOMEM;
  for (j = 0; j < R * OR_G * OR_D; j++) qd[j] = oracle_e4m3_value(a->q_idx[(int64_t)row0 * OR_G * OR_D + j]);
  for (t = 0; t < N; t++) {
    int page = page_of(a, b, t / OR_BLK), slot = t % OR_BLK;
    if (page < 0) { free(qd); return OR_EINVAL; }
    (a->exact_index_scores ? dequant_row_exact : dequant_row)(a->ki_data + ((int64_t)page * OR_BLK + slot) * 64,
                                                             a->ki_scale + ((int64_t)page * OR_BLK + slot) * 8, kv);
    for (r = 0; r < R; r++) {
      int pos = N - R + r;
      for (g = 0; g < OR_G; g++) {
        double acc = 0.0;
        const double* qi = qd + ((size_t)r * OR_G + g) * OR_D;
        if (t > pos) { s[((int64_t)r * OR_G + g) * N + t] = -INFINITY; continue; }
        for (j = 0; j < OR_D; j++) acc += qi[j] * kv[j];
        s[((int64_t)r * OR_G + g) * N + t] = acc;
      }
    }
  }
  free(qd);
  return OR_OK;
}

/* Step 2 — block max pool. [vLLM-zh] same section: the per-key scores are max-
 * pooled into one score per 128-token block. [MSA-fig] §1 "Block Max Pool".
 * With several query rows (speculative decode) the group's block score is also
 * the max over rows. Blocks with no visible token get -inf.
 * in: s[(r*4+g)*N + t]; out: S[g*nb + c], nb = ceil(N/128). */
int oracle_block_maxpool(int R, int N, const double* s, double* S) {
  int nb = (N + OR_BLK - 1) / OR_BLK, g, c, r, t;
  for (g = 0; g < OR_G; g++)
    for (c = 0; c < nb; c++) {
      double m = -INFINITY;
      for (r = 0; r < R; r++)
        for (t = c * OR_BLK; t < N && t < (c + 1) * OR_BLK; t++) {
          double v = s[((int64_t)r * OR_G + g) * N + t];
          if (v > m) m = v;
        }
      S[g * nb + c] = m;
    }
  return OR_OK;
}

/* Steps 1+2 for request b: S[g*nb + c]. */
int oracle_block_scores(const oracle_args* a, int b, double* S) {
  int N, R, row0, rc;
  double* s;
  if ((rc = req_geometry(a, b, &N, &R, &row0)) != OR_OK) return rc;
  s = (double*)malloc(sizeof(double) * ((size_t)R * OR_G * N + 1));
  if (!s) return OR_ENOMEM;
  rc = oracle_token_scores(a, b, s);
  if (rc == OR_OK) rc = oracle_block_maxpool(R, N, s, S);
  free(s);
  return rc;
}

/* Step 3 — top-k block selection for one group. [vLLM-zh] same section: main
 * attention runs exactly on only the top 16 blocks, the most recent block always
 * kept, so at most 2,048 keys per query. [MSA-fig] §1 "TopK ... I1, I2".
 * Reading: the 16 include the most recent block (block nb-1) plus the 15 best
 * of the others; ties go to the lower block id; with nb <= top_k every block is
 * kept. Output ids ascending, padded with -1 to top_k. */
typedef struct { double v; int id; } scored;
static int cmp_desc(const void* x, const void* y) {
  const scored* p = (const scored*)x;
  const scored* q = (const scored*)y;
  int pn = isnan(p->v), qn = isnan(q->v);
  if (pn != qn) return pn - qn;                 /* NaN last */
  if (!pn && p->v != q->v) return (p->v > q->v) ? -1 : 1;
  return (p->id < q->id) ? -1 : (p->id > q->id);
}
static int cmp_int(const void* x, const void* y) {
  int p = *(const int*)x, q = *(const int*)y;
  return (p > q) - (p < q);
}
int oracle_select(int nb, int top_k, const double* S, int32_t* ids) {
  int i, n = 0;
  int* chosen;
  if (nb < 0 || top_k < 1) return OR_EINVAL;
  chosen = (int*)malloc(sizeof(int) * (top_k + 1));
  if (!chosen) return OR_ENOMEM;
  if (nb <= top_k) {
    for (i = 0; i < nb; i++) chosen[n++] = i;
  } else {
    scored* c = (scored*)malloc(sizeof(scored) * nb);
    if (!c) { free(chosen); return OR_ENOMEM; }
    for (i = 0; i < nb - 1; i++) { c[i].v = S[i]; c[i].id = i; }
    qsort(c, nb - 1, sizeof(scored), cmp_desc);
    for (i = 0; i < top_k - 1; i++) chosen[n++] = c[i].id;
    chosen[n++] = nb - 1;
    free(c);
    qsort(chosen, n, sizeof(int), cmp_int);
  }
  for (i = 0; i < top_k; i++) ids[i] = (i < n) ? chosen[i] : -1;
  free(chosen);
  return OR_OK;
}

/* Step 4 — exact attention over the selected blocks. [vLLM-zh] same section and
 * [MSA-fig] §1 step 2: standard GQA shapes, Q in R^{n x H x d}, K,V in
 * R^{n x h x d}; the blocks picked by the group's index are gathered from the
 * real K/V and ordinary softmax attention runs on them; every query head of a
 * group shares that group's selection ([MSA-fig] §1, Q1-Q3 use I1). K and V are
 * the dequantised FP8 values the MMA consumes. logits = (q . k) * sm_scale;
 * out = softmax(logits) V; lse = log sum exp(logits) (natural log).
 * ids[g*top_k + i] (-1 = unused); out[(r*32 + h)*128 + d], lse[r*32 + h]. */
int oracle_attend(const oracle_args* a, int b, const int32_t* ids, double* out, double* lse) {
  int N, R, row0, rc, g, i, r, hh, j, t;
  int nkeys;
  double *kd, *vd, *logit;
  int* kpos;
  oracle_dequant_table(NULL);
  if ((rc = req_geometry(a, b, &N, &R, &row0)) != OR_OK) return rc;
  kd = (double*)malloc(sizeof(double) * (size_t)a->top_k * OR_BLK * OR_D);
  vd = (double*)malloc(sizeof(double) * (size_t)a->top_k * OR_BLK * OR_D);
  kpos = (int*)malloc(sizeof(int) * (size_t)a->top_k * OR_BLK);
  logit = (double*)malloc(sizeof(double) * (size_t)a->top_k * OR_BLK);
  if (!kd || !vd || !kpos || !logit) { rc = OR_ENOMEM; goto done; }
  for (g = 0; g < OR_G; g++) {
    /* gather the selected keys of this group */
    nkeys = 0;
    for (i = 0; i < a->top_k; i++) {
      int blk = ids[g * a->top_k + i], page;
      if (blk < 0) continue;
      if (blk * OR_BLK >= N) { rc = OR_EINVAL; goto done; }
      page = page_of(a, b, blk);
      if (page < 0) { rc = OR_EINVAL; goto done; }
      for (t = blk * OR_BLK; t < N && t < (blk + 1) * OR_BLK; t++) {
        int64_t row = ((int64_t)page * OR_G + g) * OR_BLK + (t % OR_BLK);
        dequant_row(a->k_data + row * 64, a->k_scale + row * 8, kd + (size_t)nkeys * OR_D);
        dequant_row(a->v_data + row * 64, a->v_scale + row * 8, vd + (size_t)nkeys * OR_D);
        kpos[nkeys++] = t;
      }
    }
    for (r = 0; r < R; r++) {
      int pos = N - R + r;
      for (hh = 0; hh < OR_HQ / OR_G; hh++) {
        int h = g * (OR_HQ / OR_G) + hh;
        const uint8_t* qb = a->q + ((int64_t)(row0 + r) * OR_HQ + h) * OR_D;
        double m = -INFINITY, l = 0.0, o[OR_D], qv[OR_D];
        int any = 0;
        for (j = 0; j < OR_D; j++) qv[j] = oracle_e4m3_value(qb[j]);
        for (i = 0; i < nkeys; i++) {
          double acc = 0.0;
          if (kpos[i] > pos) { logit[i] = -INFINITY; continue; }
          for (j = 0; j < OR_D; j++) acc += qv[j] * kd[(size_t)i * OR_D + j];
          logit[i] = acc * a->sm_scale;
          if (logit[i] > m) m = logit[i];
          any = 1;
        }
        for (j = 0; j < OR_D; j++) o[j] = 0.0;
        if (any) {
          for (i = 0; i < nkeys; i++) {
            double p;
            if (kpos[i] > pos) continue;
            p = exp(logit[i] - m);
            l += p;
            for (j = 0; j < OR_D; j++) o[j] += p * vd[(size_t)i * OR_D + j];
          }
          for (j = 0; j < OR_D; j++) o[j] /= l;
        }
        for (j = 0; j < OR_D; j++) out[((int64_t)(row0 + r) * OR_HQ + h) * OR_D + j] = o[j];
        if (lse) lse[(int64_t)(row0 + r) * OR_HQ + h] = any ? m + log(l) : -INFINITY;
      }
    }
  }
  rc = OR_OK;
done:
  free(kd); free(vd); free(kpos); free(logit);
  return rc;
}

/* The whole path for a list of requests: scores -> block max -> top-k ->
 * attention. ids[(i*4 + g)*top_k + k] for the i-th listed request; S (optional)
 * [(i*4 + g)*max_pages_per_req + c]; out/lse are full-size [total_rows][32][128]
 * / [total_rows][32] arrays of which the listed requests' rows are written.
 * Requests run in parallel (OpenMP) when the library was built with it. */
int oracle_decode(const oracle_args* a, int nreq, const int32_t* reqs, int32_t* ids, double* S, double* out, double* lse) {
  int i, err = OR_OK;
  oracle_dequant_table(NULL);
#pragma omp parallel for schedule(dynamic, 1)
  for (i = 0; i < nreq; i++) {
    int b = reqs[i], N, R, row0, g, rc, nb;
    double* Sb;
    if (req_geometry(a, b, &N, &R, &row0) != OR_OK) { err = OR_EINVAL; continue; }
    nb = (N + OR_BLK - 1) / OR_BLK;
    Sb = (double*)malloc(sizeof(double) * ((size_t)OR_G * nb + 1));
    if (!Sb) { err = OR_ENOMEM; continue; }
    rc = oracle_block_scores(a, b, Sb);
    for (g = 0; g < OR_G && rc == OR_OK; g++) {
      rc = oracle_select(nb, a->top_k, Sb + (size_t)g * nb, ids + ((int64_t)i * OR_G + g) * a->top_k);
      if (S) {
        int c;
        for (c = 0; c < a->max_pages_per_req; c++)
          S[((int64_t)i * OR_G + g) * a->max_pages_per_req + c] = (c < nb) ? Sb[(size_t)g * nb + c] : -INFINITY;
      }
    }
    if (rc == OR_OK) rc = oracle_attend(a, b, ids + (int64_t)i * OR_G * a->top_k, out, lse);
    if (rc != OR_OK) err = rc;
    free(Sb);
  }
  return err;
}

/* ------------------------------------------------------------------------- */
/* NVFP4 insertion of new keys and values. [vLLM-zh] "QKV GEMM + norm + RoPE + KV */
/* 插入融合": the fused epilogue takes the FP32 accumulators head by head and     */
/* quantises K, V and the index keys to NVFP4, writing them straight into their   */
/* caches. NVFP4 as everywhere here: per 16 consecutive elements one E4M3 scale,  */
/* amax / 6 rounded to E4M3 (nearest, ties to even, saturating; no second-level   */
/* scale), and per element the E2M1 value nearest x / scale (ties to the even     */
/* code, saturating at 6) with the sign of x. A zero scale gives zero codes.      */
/* ------------------------------------------------------------------------- */

/* E2M1 code of y: sign of y in bit 3, magnitude = the nearest of the 8 E2M1
 * magnitudes (codes 0..7 in increasing value), ties to the even code, values
 * beyond 6 saturating to 6. Plain search over the 8 magnitudes. */
int oracle_e2m1_round(double y) {
  int sign = signbit(y) ? 8 : 0, c, best = 0;
  double a = fabs(y), dbest = INFINITY;
  /* beyond the largest magnitude that magnitude is the nearest (and the distances
   * to the others can round to equal doubles for huge y) */
  if (a >= 6.0) return sign | 7;
  for (c = 0; c < 8; c++) {
    double d = fabs(oracle_e2m1_value(c) - a);
    if (d < dbest || (d == dbest && (c & 1) == 0)) { dbest = d; best = c; }
  }
  return sign | best;
}

/* One row of n elements (n a multiple of 16) to n/2 code bytes (element 2i in
 * the low nibble of byte i) and n/16 scale bytes. */
void oracle_nvfp4_quantize_row(const float* x, int n, uint8_t* codes, uint8_t* scales) {
  int g, j;
  for (g = 0; g < n / 16; g++) {
    double amax = 0.0, s;
    for (j = 0; j < 16; j++) amax = fmax(amax, fabs((double)x[g * 16 + j]));
    scales[g] = (uint8_t)oracle_e4m3_round(amax / 6.0);
    s = oracle_e4m3_value(scales[g]);
    for (j = 0; j < 16; j += 2) {
      int lo = s > 0.0 ? oracle_e2m1_round((double)x[g * 16 + j] / s) : 0;
      int hi = s > 0.0 ? oracle_e2m1_round((double)x[g * 16 + j + 1] / s) : 0;
      codes[(g * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

/* Write T new tokens into the caches (layout as in the header): token t goes to
 * page slot_mapping[t] / 128, slot slot_mapping[t] % 128, as 4 K rows, 4 V rows
 * and 1 index-key row; a negative slot skips the token, and a NULL source leaves
 * that cache untouched. Returns OR_EINVAL (after writing the valid tokens) if a
 * page is out of range. */
int oracle_kv_insert(int T, int num_pages, const int64_t* slot_mapping, const float* k, const float* v,
                     const float* ki, uint8_t* k_data, uint8_t* k_scale, uint8_t* v_data, uint8_t* v_scale,
                     uint8_t* ki_data, uint8_t* ki_scale) {
  int t, h, err = OR_OK;
  for (t = 0; t < T; t++) {
    int64_t sl = slot_mapping[t], page, slot;
    if (sl < 0) continue;
    page = sl / OR_BLK;
    slot = sl % OR_BLK;
    if (page >= num_pages) { err = OR_EINVAL; continue; }
    for (h = 0; h < OR_G; h++) {
      int64_t row = (page * OR_G + h) * OR_BLK + slot;
      if (k) oracle_nvfp4_quantize_row(k + ((int64_t)t * OR_G + h) * OR_D, OR_D, k_data + row * 64, k_scale + row * 8);
      if (v) oracle_nvfp4_quantize_row(v + ((int64_t)t * OR_G + h) * OR_D, OR_D, v_data + row * 64, v_scale + row * 8);
    }
    if (ki) {
      int64_t row = page * OR_BLK + slot;
      oracle_nvfp4_quantize_row(ki + (int64_t)t * OR_D, OR_D, ki_data + row * 64, ki_scale + row * 8);
    }
  }
  return err;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Thread count for the request loop of oracle_decode (host-side scheduling only; it
 * changes no arithmetic: each request's result is computed by one thread in a fixed
 * order). n < 1 leaves it unchanged. Returns the count now in effect. */
int oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}
