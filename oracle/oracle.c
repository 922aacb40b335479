/*
 * FP64 CPU oracle for paged grouped-query verify attention over an FP8 E4M3
 * KV cache.  TEST INFRASTRUCTURE ONLY: tests, the smoke check and the CPU
 * baseline leg of the benchmark call it; the product path never does.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (plain definitions, no blocking or fusion):
 *
 *  - E4M3 decode, OCP FP8 E4M3FN format (1 sign bit, 4 exponent bits with
 *    bias 7, 3 mantissa bits, no infinities, NaN only at S.1111.111).  The
 *    pages require an exact decode checked on every byte (1Cat-vLLM PR #566
 *    "[Kernel] Finalize the audited TP2 DFlash2 31/29 ms endpoint", Final
 *    audit and Test Result) but do not define the format; the reading taken
 *    is the OCP definition, whose largest finite value is the 448 in the
 *    per-head scale amax/448.
 *
 *  - E5M2 decode (the other FP8 KV format the pages keep available: PR #560,
 *    Purpose; PR #524, Scope and non-duplication), OCP FP8 E5M2 (1 sign bit,
 *    5 exponent bits with bias 15, 2 mantissa bits, infinities at
 *    S.11111.00, NaN at S.11111.xx otherwise), largest finite value 57344.
 *
 *  - Two cache layouts, read through one addressing rule: token j of
 *    sequence b, KV head h is the D bytes at base + phys * page_stride +
 *    (j % page) * token_stride + h * head_stride, phys = block_table[b][j /
 *    page], with separate K and V bases.  The library's pool
 *    [n_pages][2 (K,V)][Hkv][page][D] is one choice of bases and strides;
 *    the pages' token-major cache [blocks][block_size][kv_heads][D] with
 *    padded token strides (the [1,848,1,256] tensor with strides
 *    [223872,264,256,1] of PR #524 "[Kernel][SM70] Add opt-in E4M3 grouped
 *    attention with FP32 partials", AI integration review) is another.
 *
 *  - Per-KV-head dequantisation x = dec(byte) * s_h, with separate scales for
 *    K and V (PR #560 "[Bugfix] Use FP32 state and E4M3 defaults for
 *    DFlash2", Test Plan and Results).
 *
 *  - Scaled-dot-product attention per (sequence b, query i, q head hq) in
 *    FP64: q head hq reads KV head hq / (Hq/Hkv) (GQA6/D256 grouping, PR #524
 *    "[Kernel][SM70] Add opt-in E4M3 grouped attention with FP32 partials",
 *    Scope and non-duplication).  The q_len queries occupy the last q_len
 *    positions of the L cached tokens, so query i sees keys 0 .. L-q_len+i
 *    (lengths per query, same section).  Token j of sequence b lives
 *    in physical page block_table[b][j / page] at slot j % page.
 *
 *  - Two evaluation modes.  Direct: two passes (maximum, then exponentials
 *    and sums).  Split: the context [0, L) is cut into partitions of T
 *    tokens; each keeps its own FP32-style state, maximum, sum and
 *    unnormalised P.V, merged only at the end (PR #524, final status), and
 *    the partitions are combined in ascending order.  Both give
 *    the same exact result; the split mode exists so tests can pin that
 *    re-association.
 *
 * Padded query slots (i >= q_len), sequences with L == 0 and sequences with
 * q_len > L produce zeros.  The oracle returns a nonzero code when the
 * inputs are malformed (block id out of range, L beyond the block table).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double oracle_e4m3_value(uint32_t byte) {
  const int s = (byte >> 7) & 1;
  const int e = (byte >> 3) & 15;
  const int m = byte & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9);           /* subnormal: m/8 * 2^(1-7) */
  else
    mag = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7)      */
  return s ? -mag : mag;
}

void oracle_e4m3_table(double *out256) {
  for (int b = 0; b < 256; ++b) out256[b] = oracle_e4m3_value((uint32_t)b);
}

double oracle_e5m2_value(uint32_t byte) {
  const int s = (byte >> 7) & 1;
  const int e = (byte >> 2) & 31;
  const int m = byte & 3;
  double mag;
  if (e == 31) return m == 0 ? (s ? -INFINITY : INFINITY) : NAN;
  if (e == 0)
    mag = ldexp((double)m, -16);          /* subnormal: m/4 * 2^(1-15)  */
  else
    mag = ldexp(4.0 + (double)m, e - 17); /* (1 + m/4) * 2^(e-15)       */
  return s ? -mag : mag;
}

/* kv_format 0 = E4M3, 1 = E5M2 */
void oracle_fp8_table(double *out256, int kv_format) {
  for (int b = 0; b < 256; ++b)
    out256[b] = kv_format == 1 ? oracle_e5m2_value((uint32_t)b) : oracle_e4m3_value((uint32_t)b);
}

/* Error codes of the oracle (independent of the library's). */
#define ORC_OK 0
#define ORC_BAD_ARGS -1
#define ORC_BAD_BLOCK -2
#define ORC_BAD_LENGTH -3

typedef struct {
  int B, Qmax, Hq, Hkv, D, page, max_pages;
  int64_t n_pages;
} orc_shape;

/* Where the cache's bytes live: K (sel 0) and V (sel 1) bases, strides in
 * bytes of a page, a token slot and a KV head; d is contiguous. */
typedef struct {
  const uint8_t *base[2];
  int64_t page_stride, token_stride, head_stride;
} orc_cache;

static const uint8_t *kv_row(const orc_cache *c, int64_t phys, int kv_sel, int h, int slot) {
  return c->base[kv_sel] + phys * c->page_stride + (int64_t)slot * c->token_stride +
         (int64_t)h * c->head_stride;
}

/* One output row: out[d] for (b, i, hq).  z is scratch of length >= L. */
static int one_row(const double *q, const orc_cache *kv, const int32_t *bt,
                   const int32_t *seq_len, const int32_t *q_len,
                   const double *scales, const orc_shape *sh, double sm_scale,
                   int split_tokens, const double *dec, int b, int i, int hq,
                   double *z, double *acc, double *out) {
  const int D = sh->D;
  const int G = sh->Hq / sh->Hkv;
  const int h = hq / G;
  const int L = seq_len[b];
  const int ql = q_len[b];
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (L <= 0 || i >= ql || ql > L) return ORC_OK; /* zero rows by contract */
  if ((int64_t)L > (int64_t)sh->max_pages * sh->page) return ORC_BAD_LENGTH;

  const double sK = scales[2 * h + 0];
  const double sV = scales[2 * h + 1];
  const double *qv = q + (((int64_t)b * sh->Qmax + i) * sh->Hq + hq) * D;
  const int pos = L - ql + i; /* last visible key of this query */

  /* scores z_j = sm_scale * sum_d q[d] * (dec(K[j][d]) * sK), j = 0..pos */
  for (int j = 0; j <= pos; ++j) {
    const int64_t phys = bt[(int64_t)b * sh->max_pages + j / sh->page];
    if (phys < 0 || phys >= sh->n_pages) return ORC_BAD_BLOCK;
    const uint8_t *kr = kv_row(kv, phys, 0, h, j % sh->page);
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += qv[d] * (dec[kr[d]] * sK);
    z[j] = sm_scale * dot;
  }

  if (split_tokens <= 0) {
    /* direct mode */
    double zmax = -INFINITY;
    for (int j = 0; j <= pos; ++j) zmax = z[j] > zmax ? z[j] : zmax;
    double den = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int j = 0; j <= pos; ++j) {
      const double w = exp(z[j] - zmax);
      const int64_t phys = bt[(int64_t)b * sh->max_pages + j / sh->page];
      const uint8_t *vr = kv_row(kv, phys, 1, h, j % sh->page);
      den += w;
      for (int d = 0; d < D; ++d) acc[d] += w * (dec[vr[d]] * sV);
    }
    for (int d = 0; d < D; ++d) out[d] = acc[d] / den;
    return ORC_OK;
  }

  /* split mode: partitions [p*T, min((p+1)*T, L)) of the whole context,
   * each intersected with the keys this query sees, combined in ascending
   * partition order. */
  const int T = split_tokens;
  const int P = (L + T - 1) / T;
  double M = -INFINITY;
  /* first pass over partitions: the combine's maximum of partition maxima */
  for (int p = 0; p < P; ++p) {
    const int j0 = p * T;
    int j1 = (p + 1) * T - 1;
    if (j1 > pos) j1 = pos;
    if (j0 > j1) continue; /* empty for this query: skipped by the combine */
    double mp = -INFINITY;
    for (int j = j0; j <= j1; ++j) mp = z[j] > mp ? z[j] : mp;
    M = mp > M ? mp : M;
  }
  double lam = 0.0;
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  for (int p = 0; p < P; ++p) {
    const int j0 = p * T;
    int j1 = (p + 1) * T - 1;
    if (j1 > pos) j1 = pos;
    if (j0 > j1) continue;
    double mp = -INFINITY;
    for (int j = j0; j <= j1; ++j) mp = z[j] > mp ? z[j] : mp;
    double lp = 0.0;
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int j = j0; j <= j1; ++j) {
      const double w = exp(z[j] - mp);
      const int64_t phys = bt[(int64_t)b * sh->max_pages + j / sh->page];
      const uint8_t *vr = kv_row(kv, phys, 1, h, j % sh->page);
      lp += w;
      for (int d = 0; d < D; ++d) acc[d] += w * (dec[vr[d]] * sV);
    }
    const double wp = exp(mp - M);
    lam += wp * lp;
    for (int d = 0; d < D; ++d) out[d] += wp * acc[d];
  }
  for (int d = 0; d < D; ++d) out[d] /= lam;
  return ORC_OK;
}

/*
 * Attention for the requested rows.
 *   q            [B][Qmax][Hq][D]      fp64 (the fp16 queries, widened exactly)
 *   kv           [n_pages][2][Hkv][page][D] FP8 bytes (E4M3, or E5M2 when
 *                kv_format == 1)
 *   block_table  [B][max_pages]        physical page ids
 *   seq_len      [B]                   L, including the q tail
 *   q_len        [B]                   queries in the tail (<= Qmax)
 *   scales       [Hkv][2]              (s_K, s_V), the fp32 scales widened
 *   rows         NULL for every (b, i, hq) (out is [B][Qmax][Hq][D]) or
 *                n_rows triples (b, i, hq) (out is [n_rows][D])
 *   split_tokens 0 for direct mode, else the partition length T
 *   n_threads    OpenMP threads (0 = runtime default)
 * Returns ORC_OK or the first error code met.
 */
static int verify_rows(const double *q, const orc_cache *kv, const int32_t *block_table,
                       const int32_t *seq_len, const int32_t *q_len, const double *scales,
                       int B, int Qmax, int Hq, int Hkv, int D, int page, int64_t n_pages,
                       int max_pages, double sm_scale, int split_tokens, const int32_t *rows,
                       int64_t n_rows, double *out, int n_threads, int kv_format) {
  if (B < 0 || Qmax <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || page <= 0 ||
      max_pages <= 0 || Hq % Hkv != 0 || kv_format < 0 || kv_format > 1)
    return ORC_BAD_ARGS;
  for (int b = 0; b < B; ++b)
    if (q_len[b] < 0 || q_len[b] > Qmax || seq_len[b] < 0) return ORC_BAD_ARGS;
  orc_shape sh = {B, Qmax, Hq, Hkv, D, page, max_pages, n_pages};
  double dec[256];
  oracle_fp8_table(dec, kv_format);
  int Lmax = 1;
  for (int b = 0; b < B; ++b) Lmax = seq_len[b] > Lmax ? seq_len[b] : Lmax;
  const int64_t total = rows ? n_rows : (int64_t)B * Qmax * Hq;
  int status = ORC_OK;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    double *z = (double *)malloc(sizeof(double) * (size_t)Lmax);
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t r = 0; r < total; ++r) {
      int b, i, hq;
      double *o;
      if (rows) {
        b = rows[3 * r + 0];
        i = rows[3 * r + 1];
        hq = rows[3 * r + 2];
        o = out + r * D;
      } else {
        hq = (int)(r % Hq);
        i = (int)((r / Hq) % Qmax);
        b = (int)(r / ((int64_t)Hq * Qmax));
        o = out + r * D;
      }
      int rc = ORC_BAD_ARGS;
      if (b >= 0 && b < B && i >= 0 && i < Qmax && hq >= 0 && hq < Hq)
        rc = one_row(q, kv, block_table, seq_len, q_len, scales, &sh, sm_scale,
                     split_tokens, dec, b, i, hq, z, acc, o);
      if (rc != ORC_OK) {
#ifdef _OPENMP
#pragma omp critical
#endif
        if (status == ORC_OK) status = rc;
      }
    }
    free(z);
    free(acc);
  }
  return status;
}

int oracle_verify_attn_fmt(const double *q, const uint8_t *kv, const int32_t *block_table,
                           const int32_t *seq_len, const int32_t *q_len,
                           const double *scales, int B, int Qmax, int Hq, int Hkv,
                           int D, int page, int64_t n_pages, int max_pages,
                           double sm_scale, int split_tokens, const int32_t *rows,
                           int64_t n_rows, double *out, int n_threads, int kv_format) {
  /* the pool [n_pages][2 (K,V)][Hkv][page][D] */
  const int64_t slice = (int64_t)page * D;
  orc_cache c;
  c.base[0] = kv;
  c.base[1] = kv + (int64_t)Hkv * slice;
  c.page_stride = 2 * (int64_t)Hkv * slice;
  c.token_stride = D;
  c.head_stride = slice;
  return verify_rows(q, &c, block_table, seq_len, q_len, scales, B, Qmax, Hq, Hkv, D, page,
                     n_pages, max_pages, sm_scale, split_tokens, rows, n_rows, out, n_threads,
                     kv_format);
}

/*
 * The same attention over a cache given by explicit K and V bases and byte
 * strides (page, token slot, KV head; d contiguous): any layout, e.g. the
 * token-major [blocks][block_size][kv_heads][D] cache with a padded token
 * stride.  Arguments otherwise as oracle_verify_attn_fmt.
 */
int oracle_verify_attn_strided(const double *q, const uint8_t *k_base, const uint8_t *v_base,
                               int64_t page_stride, int64_t token_stride, int64_t head_stride,
                               const int32_t *block_table, const int32_t *seq_len,
                               const int32_t *q_len, const double *scales, int B, int Qmax,
                               int Hq, int Hkv, int D, int page, int64_t n_pages, int max_pages,
                               double sm_scale, int split_tokens, const int32_t *rows,
                               int64_t n_rows, double *out, int n_threads, int kv_format) {
  if (!k_base || !v_base) return ORC_BAD_ARGS;
  orc_cache c;
  c.base[0] = k_base;
  c.base[1] = v_base;
  c.page_stride = page_stride;
  c.token_stride = token_stride;
  c.head_stride = head_stride;
  return verify_rows(q, &c, block_table, seq_len, q_len, scales, B, Qmax, Hq, Hkv, D, page,
                     n_pages, max_pages, sm_scale, split_tokens, rows, n_rows, out, n_threads,
                     kv_format);
}

/* Threads the OpenMP runtime would use by default (for the CPU baseline). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* The E4M3 entry point (kv_format 0). */
int oracle_verify_attn(const double *q, const uint8_t *kv, const int32_t *block_table,
                       const int32_t *seq_len, const int32_t *q_len,
                       const double *scales, int B, int Qmax, int Hq, int Hkv,
                       int D, int page, int64_t n_pages, int max_pages,
                       double sm_scale, int split_tokens, const int32_t *rows,
                       int64_t n_rows, double *out, int n_threads) {
  return oracle_verify_attn_fmt(q, kv, block_table, seq_len, q_len, scales, B, Qmax, Hq, Hkv,
                                D, page, n_pages, max_pages, sm_scale, split_tokens, rows,
                                n_rows, out, n_threads, 0);
}

/*
 * Paged FP8 -> FP16 bridge, exact values (before the one rounding to FP16,
 * which the caller applies): for sequence b, KV head h, token t < L,
 *   k[b][h][t][d] = dec(K byte) * s_K[h],  v likewise with s_V[h]
 * (raw != 0: dec(byte) alone), computed in FP64 (exact: a 4-bit by 24-bit
 * product).  Entries for t >= L are left as they are.  Output arrays are
 * dense [B][Hkv][cap][D].  Returns ORC_BAD_BLOCK / ORC_BAD_LENGTH on
 * malformed inputs (first error met; the rest is still written).
 */
int oracle_bridge_fp16(const uint8_t *kv, const int32_t *block_table, const int32_t *seq_len,
                       const double *scales, int B, int Hkv, int D, int page, int64_t n_pages,
                       int max_pages, int cap, int kv_format, int raw, double *out_k,
                       double *out_v) {
  if (B < 0 || Hkv <= 0 || D <= 0 || page <= 0 || max_pages <= 0 || cap <= 0 ||
      kv_format < 0 || kv_format > 1)
    return ORC_BAD_ARGS;
  double dec[256];
  oracle_fp8_table(dec, kv_format);
  int status = ORC_OK;
  for (int b = 0; b < B; ++b) {
    const int L = seq_len[b];
    if (L < 0 || L > cap || (L + page - 1) / page > max_pages) {
      if (status == ORC_OK) status = ORC_BAD_LENGTH;
      continue;
    }
    for (int h = 0; h < Hkv; ++h) {
      for (int t = 0; t < L; ++t) {
        const int32_t phys = block_table[(int64_t)b * max_pages + t / page];
        double *ok = out_k + (((int64_t)b * Hkv + h) * cap + t) * D;
        double *ov = out_v + (((int64_t)b * Hkv + h) * cap + t) * D;
        if (phys < 0 || phys >= n_pages) {
          if (status == ORC_OK) status = ORC_BAD_BLOCK;
          for (int d = 0; d < D; ++d) ok[d] = ov[d] = 0.0;
          continue;
        }
        const uint8_t *kr = kv + ((((int64_t)phys * 2 + 0) * Hkv + h) * page + t % page) * D;
        const uint8_t *vr = kv + ((((int64_t)phys * 2 + 1) * Hkv + h) * page + t % page) * D;
        const double sk = raw ? 1.0 : scales[h * 2 + 0], sv = raw ? 1.0 : scales[h * 2 + 1];
        for (int d = 0; d < D; ++d) {
          ok[d] = dec[kr[d]] * sk;
          ov[d] = dec[vr[d]] * sv;
        }
      }
    }
  }
  return status;
}
