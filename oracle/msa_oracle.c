/*
 * msa_oracle.c -- plain, slow CPU oracle for two-stage GQA block-sparse
 * attention (the "MiniMax Sparse Attention" block).
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke run and the benchmark's CPU
 * baseline load this library (through oracle/msa_oracle.py). It shares no code,
 * header or constant with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes follows the Atlas Cloud guide "MiniMax goes sparse: decoding
 * M3's attention from a single diagram" (Portuguese, Spanish and French
 * editions), section 1:
 *   Step 1, the index branch: one index query per GQA group, block-level
 *     scores from keys pooled per block, and a top-k that keeps a short list
 *     of KV blocks per layer and group;
 *   Step 2, the sparse branch: ordinary softmax attention of every query head
 *     of the group over the real K/V of the blocks its group selected.
 * The readings that fill what the guide leaves open are stated at each
 * function (block size 64; the summary key is the mean of the block's keys;
 * the index query is the sum of the group's query vectors; the newest or
 * diagonal block is always kept and never scored; ties go to the lower block).
 *
 * Style: scalar C99, every sum accumulated in double in the order written, no
 * SIMD intrinsics, no reordering beyond what a definition states. OpenMP is
 * used only across independent (sequence, KV head) units in the *_units
 * functions. Inputs are read as the exact values their bits encode: float64,
 * float32, or bfloat16 (the upper 16 bits of a binary32 pattern).
 * Build with -ffp-contract=off so that no multiply-add is fused and x86 and
 * Arm give the same bits.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define ORA_BLOCK 64
#define ORA_D 128

enum { ORA_F64 = 0, ORA_F32 = 1, ORA_BF16 = 2 };

/* The exact value of element i of an array of `type`. */
static double ld(const void* p, int type, int64_t i) {
  if (type == ORA_F64) return ((const double*)p)[i];
  if (type == ORA_F32) return (double)((const float*)p)[i];
  /* bfloat16: the bits are the upper half of a binary32 pattern */
  uint32_t bits = (uint32_t)((const uint16_t*)p)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Rounding into the storage type                                           */
/* ------------------------------------------------------------------------ */

/* Round a double to the nearest bfloat16 value, ties to even, in one step
 * (no intermediate binary32 rounding). bfloat16 keeps 8 significant bits and
 * the binary32 exponent range: normal numbers down to 2^-126, subnormals in
 * steps of 2^-133, and values at or beyond 2^128 - 2^119 (halfway past the
 * largest finite value) become infinite. */
double ora_round_bf16(double x) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  int e = 0;
  (void)frexp(x, &e); /* |x| = m * 2^e, m in [0.5, 1) */
  int shift = e - 8;  /* spacing of 8-significant-bit numbers at this size */
  if (shift < -133) shift = -133;
  double scaled = ldexp(x, -shift); /* exact: a power-of-two scaling */
  double r = nearbyint(scaled);     /* default rounding mode: to nearest, ties to even */
  double y = ldexp(r, shift);
  if (fabs(y) >= ldexp(1.0, 128)) return x > 0 ? INFINITY : -INFINITY;
  return y;
}

/* Value of x once stored in `store` (ORA_F32: C's double -> float
 * conversion, which rounds to nearest even; ORA_BF16: ora_round_bf16). */
double ora_store(double x, int store) {
  if (store == ORA_F32) return (double)(float)x;
  if (store == ORA_BF16) return ora_round_bf16(x);
  return x;
}

/* ------------------------------------------------------------------------ */
/* Step 1: index branch                                                      */
/* ------------------------------------------------------------------------ */

/* Block summary keys of one (sequence, KV head) -- guide §1, Step 1 (block
 * pooling of the index branch), with the mean of the block's keys as the
 * summary. For each complete block b (64 b + 63 < seq_len):
 *   exact[b][d]  = (sum_{i<64} K[64 b + i][d]) / 64   (double)
 *   stored[b][d] = that value rounded to nearest even into `store`.
 * k: rows of the head in token order, row r at element offset r * ld_k.
 * Returns the number of complete blocks. */
int64_t ora_pool_block_keys(const void* k, int ktype, int64_t ld_k, int64_t seq_len, int store, double* stored,
                            double* exact) {
  int64_t nbf = seq_len / ORA_BLOCK;
  for (int64_t b = 0; b < nbf; ++b) {
    for (int d = 0; d < ORA_D; ++d) {
      double sum = 0.0;
      for (int i = 0; i < ORA_BLOCK; ++i) sum += ld(k, ktype, (b * ORA_BLOCK + i) * ld_k + d);
      double mean = sum / ORA_BLOCK;
      if (exact) exact[b * ORA_D + d] = mean;
      if (stored) stored[b * ORA_D + d] = ora_store(mean, store);
    }
  }
  return nbf;
}

/* The index query of one group -- guide §1, Step 1 ("Idx Q", one per GQA
 * group): the sum of the group's query vectors (for a prefill tile, of the
 * tile's tokens x the group's heads). q: n_rows rows of 128, contiguous. */
void ora_index_query(const void* q, int qtype, int64_t n_rows, double* q_idx) {
  for (int d = 0; d < ORA_D; ++d) {
    double s = 0.0;
    for (int64_t r = 0; r < n_rows; ++r) s += ld(q, qtype, r * ORA_D + d);
    q_idx[d] = s;
  }
}

/* Block scores -- guide §1, Step 1 (the index query against the block keys):
 * scores[b] = sum_d q_idx[d] * pooled[b][d] for b < n_cand, unscaled (a
 * positive scale does not change the ranking). */
void ora_score_blocks(const double* q_idx, const double* pooled, int64_t n_cand, double* scores) {
  for (int64_t b = 0; b < n_cand; ++b) {
    double s = 0.0;
    for (int d = 0; d < ORA_D; ++d) s += q_idx[d] * pooled[b * ORA_D + d];
    scores[b] = s;
  }
}

/* The guide's Step 1 as drawn (§1, Step 1: token-level scores against one
 * index-key head shared by the layer's groups, then a max pool per block):
 * scores[b] = max_{t in block b} sum_d q_idx[d] * kidx[t][d], b < n_cand
 * (every candidate block is complete). */
void ora_score_blocks_token_max(const double* q_idx, const void* kidx, int ktype, int64_t ld_k, int64_t n_cand,
                                double* scores) {
  for (int64_t b = 0; b < n_cand; ++b) {
    double best = -INFINITY;
    for (int i = 0; i < ORA_BLOCK; ++i) {
      double s = 0.0;
      for (int d = 0; d < ORA_D; ++d) s += q_idx[d] * ld(kidx, ktype, (b * ORA_BLOCK + i) * ld_k + d);
      if (s > best) best = s;
    }
    scores[b] = best;
  }
}

typedef struct {
  double score;
  int64_t block;
} ora_cand;

/* Ranking of the top-k: higher score first, equal scores to the lower block. */
static int rank_cmp(const void* a, const void* b) {
  const ora_cand* x = (const ora_cand*)a;
  const ora_cand* y = (const ora_cand*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->block > y->block) - (x->block < y->block);
}

static int int64_cmp(const void* a, const void* b) {
  int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
  return (x > y) - (x < y);
}

/* Top-k block selection -- guide §1, Step 1 (TopK keeps the k best blocks per
 * layer and group; output lists I1, I2):
 *   candidates are blocks first..n-1 (first = 1 with an attention sink, whose
 *   block 0 is kept without being scored -- the guide, §2, names a sink among
 *   the likely replacements of the dropped sliding window; else 0), ranked by
 *   score descending, ties to the lower block; the first
 *   min(k_scored, #candidates) are kept; then block 0 when keep0, then the
 *   forced block (newest / diagonal, when >= 0 and not already listed); the
 *   list is sorted ascending and padded with -1 to k_total.
 * Returns the number of listed blocks, or -1 if k_total is too small. */
int64_t ora_select_blocks(const double* scores, int64_t n, int64_t k_scored, int64_t forced, int64_t first,
                          int keep0, int64_t k_total, int64_t* sel) {
  int64_t m = n > first ? n - first : 0;
  ora_cand* c = (ora_cand*)malloc((size_t)(m > 0 ? m : 1) * sizeof(ora_cand));
  int64_t* out = (int64_t*)malloc((size_t)(m + 2 > 0 ? m + 2 : 1) * sizeof(int64_t));
  if (!c || !out) {
    free(c);
    free(out);
    return -1;
  }
  for (int64_t i = 0; i < m; ++i) {
    c[i].score = scores[first + i];
    c[i].block = first + i;
  }
  qsort(c, (size_t)m, sizeof(ora_cand), rank_cmp);
  int64_t kk = k_scored < m ? k_scored : m;
  if (kk < 0) kk = 0;
  int64_t cnt = 0;
  for (int64_t i = 0; i < kk; ++i) out[cnt++] = c[i].block;
  if (keep0) out[cnt++] = 0;
  if (forced >= 0) {
    int listed = 0;
    for (int64_t i = 0; i < cnt; ++i) listed |= out[i] == forced;
    if (!listed) out[cnt++] = forced;
  }
  free(c);
  if (cnt > k_total) {
    free(out);
    return -1;
  }
  qsort(out, (size_t)cnt, sizeof(int64_t), int64_cmp);
  for (int64_t i = 0; i < k_total; ++i) sel[i] = i < cnt ? out[i] : -1;
  free(out);
  return cnt;
}

/* ------------------------------------------------------------------------ */
/* Step 2: sparse branch                                                     */
/* ------------------------------------------------------------------------ */

/* Softmax attention of n_heads query vectors over the token set `tokens` --
 * guide §1, Step 2 (the gathered subsets of the real K/V go through ordinary
 * softmax attention; every head of a group uses its group's list):
 *   z_t = scale * sum_d q[d] K[t][d],  p_t = exp(z_t - max z) / sum_u exp(z_u - max z),
 *   o[d] = sum_t p_t V[t][d],  lse = max z + log(sum_u exp(z_u - max z)).
 * q: [n_heads][128]; k, v: rows in token order with row stride ld_kv.
 * p (nullable): [n_heads][n_tok]. An empty token set gives o = 0,
 * lse = -inf. */
void ora_attend(const void* q, int qtype, int64_t n_heads, const void* k, const void* v, int kvtype, int64_t ld_kv,
                const int64_t* tokens, int64_t n_tok, double scale, double* o, double* lse, double* p) {
  double* z = (double*)malloc((size_t)(n_tok > 0 ? n_tok : 1) * sizeof(double));
  for (int64_t h = 0; h < n_heads; ++h) {
    double* oh = o + h * ORA_D;
    for (int d = 0; d < ORA_D; ++d) oh[d] = 0.0;
    if (n_tok == 0) {
      lse[h] = -INFINITY;
      continue;
    }
    double zmax = -INFINITY;
    for (int64_t i = 0; i < n_tok; ++i) {
      double s = 0.0;
      for (int d = 0; d < ORA_D; ++d) s += ld(q, qtype, h * ORA_D + d) * ld(k, kvtype, tokens[i] * ld_kv + d);
      z[i] = s * scale;
      if (z[i] > zmax) zmax = z[i];
    }
    double denom = 0.0;
    for (int64_t i = 0; i < n_tok; ++i) {
      z[i] = exp(z[i] - zmax);
      denom += z[i];
    }
    for (int64_t i = 0; i < n_tok; ++i) {
      double w = z[i] / denom;
      if (p) p[h * n_tok + i] = w;
      for (int d = 0; d < ORA_D; ++d) oh[d] += w * ld(v, kvtype, tokens[i] * ld_kv + d);
    }
    lse[h] = zmax + log(denom);
  }
  free(z);
}

/* Dense causal GQA attention -- the full-attention comparator the guide's
 * speed-ups are quoted against (§3): every head attends to tokens
 * 0..position of its KV head. Written apart from ora_attend (no shared code),
 * with an online (running-max) softmax, so the sparse path with every block
 * selected can be checked against it. */
void ora_dense_gqa(const void* q, int qtype, int64_t n_heads, const void* k, const void* v, int kvtype, int64_t ld_kv,
                   int64_t position, double scale, double* o, double* lse) {
  double acc[ORA_D];
  for (int64_t h = 0; h < n_heads; ++h) {
    double run_max = -INFINITY, run_sum = 0.0;
    for (int d = 0; d < ORA_D; ++d) acc[d] = 0.0;
    for (int64_t t = 0; t <= position; ++t) {
      double logit = 0.0;
      for (int d = 0; d < ORA_D; ++d) logit += ld(q, qtype, h * ORA_D + d) * ld(k, kvtype, t * ld_kv + d);
      logit *= scale;
      if (logit > run_max) {
        /* rescale what was summed under the old maximum */
        double f = run_max == -INFINITY ? 0.0 : exp(run_max - logit);
        run_sum *= f;
        for (int d = 0; d < ORA_D; ++d) acc[d] *= f;
        run_max = logit;
      }
      double w = exp(logit - run_max);
      run_sum += w;
      for (int d = 0; d < ORA_D; ++d) acc[d] += w * ld(v, kvtype, t * ld_kv + d);
    }
    for (int d = 0; d < ORA_D; ++d) o[h * ORA_D + d] = position >= 0 ? acc[d] / run_sum : 0.0;
    lse[h] = position >= 0 ? run_max + log(run_sum) : -INFINITY;
  }
}

/* ------------------------------------------------------------------------ */
/* Whole decode units, OpenMP across units                                   */
/* ------------------------------------------------------------------------ */

static int64_t num_blocks(int64_t n) { return (n + ORA_BLOCK - 1) / ORA_BLOCK; }

/* Candidate count and kept block of a decode unit: candidates are the
 * complete blocks, minus the newest block nb - 1 when it is kept (bit 0 of
 * force_local). */
static void decode_candidates(int64_t len, int force_local, int64_t* n_cand, int64_t* forced) {
  int64_t nb = num_blocks(len), nbf = len / ORA_BLOCK;
  int local = force_local & 1;
  int64_t c = local ? (nbf < nb - 1 ? nbf : nb - 1) : nbf;
  *n_cand = c > 0 ? c : 0;
  *forced = (local && nb > 0) ? nb - 1 : -1;
}

/* Step 1 for n_units decode units: pool (from the keys), index query, scores
 * and selection. Unit u: q rows [u][G][128]; keys at k + u * unit_stride
 * (elements), row stride ld_k; length lens[u].
 * Outputs: sel [n_units][k_total]; scores (nullable) [n_units][max_blocks]
 * (entries past the unit's candidates are NaN); pooled (nullable)
 * [n_units][max_blocks][128] stored values (NaN past the complete blocks);
 * gap [n_units][2]: the k-th and (k+1)-th ranked candidate scores (NaN when
 * every candidate is kept). Returns 0, or -1 on a bad argument. */
int ora_decode_select_units(int64_t n_units, const void* q, int qtype, int G, const void* k, int ktype,
                            int64_t unit_stride, int64_t ld_k, const int64_t* lens, int store, int64_t k_scored,
                            int force_local, int64_t k_total, int64_t max_blocks, int64_t* sel, double* scores,
                            double* pooled, double* gap) {
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t u = 0; u < n_units; ++u) {
    int64_t len = lens[u];
    int64_t nbf = len / ORA_BLOCK;
    if (nbf > max_blocks || num_blocks(len) > max_blocks) {
      bad |= 1;
      continue;
    }
    double* kp = (double*)malloc((size_t)(nbf > 0 ? nbf : 1) * ORA_D * sizeof(double));
    double* sc = (double*)malloc((size_t)(nbf > 0 ? nbf : 1) * sizeof(double));
    double qi[ORA_D];
    const char* kb = (const char*)k + u * unit_stride * (ktype == ORA_F64 ? 8 : ktype == ORA_F32 ? 4 : 2);
    const char* qb = (const char*)q + u * (int64_t)G * ORA_D * (qtype == ORA_F64 ? 8 : qtype == ORA_F32 ? 4 : 2);
    ora_pool_block_keys(kb, ktype, ld_k, len, store, kp, NULL);
    ora_index_query(qb, qtype, G, qi);
    int64_t n_cand = 0, forced = -1;
    decode_candidates(len, force_local, &n_cand, &forced);
    int sink = (force_local & 2) != 0;
    ora_score_blocks(qi, kp, n_cand, sc);
    int64_t first = (sink && n_cand > 0) ? 1 : 0;
    int keep0 = sink && num_blocks(len) > 0 && forced != 0;
    if (ora_select_blocks(sc, n_cand, k_scored, forced, first, keep0, k_total, sel + u * k_total) < 0) bad |= 1;
    if (gap) {
      /* boundary scores of the ranking among the scored candidates */
      int64_t m = n_cand - first;
      gap[2 * u] = NAN;
      gap[2 * u + 1] = NAN;
      if (k_scored > 0 && m > k_scored) {
        ora_cand* c = (ora_cand*)malloc((size_t)m * sizeof(ora_cand));
        for (int64_t i = 0; i < m; ++i) {
          c[i].score = sc[first + i];
          c[i].block = first + i;
        }
        qsort(c, (size_t)m, sizeof(ora_cand), rank_cmp);
        gap[2 * u] = c[k_scored - 1].score;
        gap[2 * u + 1] = c[k_scored].score;
        free(c);
      }
    }
    if (scores)
      for (int64_t b = 0; b < max_blocks; ++b) scores[u * max_blocks + b] = b < n_cand ? sc[b] : NAN;
    if (pooled)
      for (int64_t b = 0; b < max_blocks; ++b)
        for (int d = 0; d < ORA_D; ++d) pooled[(u * max_blocks + b) * ORA_D + d] = b < nbf ? kp[b * ORA_D + d] : NAN;
    free(kp);
    free(sc);
  }
  return bad ? -1 : 0;
}

/* One whole decode step (Step 1 from precomputed stored summaries, then
 * Step 2) for n_units units: index query, scores, selection, and softmax
 * attention of the G heads over the tokens t < len of the selected blocks.
 * pooled: [n_units][max_blocks][128] double; k, v as in
 * ora_decode_select_units. Outputs o [n_units][G][128], lse [n_units][G].
 * The benchmark times this as the CPU baseline. */
int ora_decode_step_units(int64_t n_units, const void* q, int qtype, int G, const double* pooled, int64_t max_blocks,
                          const void* k, const void* v, int kvtype, int64_t unit_stride, int64_t ld_kv,
                          const int64_t* lens, int64_t k_scored, int force_local, int64_t k_total, double scale,
                          int64_t* sel, double* o, double* lse) {
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t u = 0; u < n_units; ++u) {
    int64_t len = lens[u];
    int esz_kv = kvtype == ORA_F64 ? 8 : kvtype == ORA_F32 ? 4 : 2;
    int esz_q = qtype == ORA_F64 ? 8 : qtype == ORA_F32 ? 4 : 2;
    const char* qb = (const char*)q + u * (int64_t)G * ORA_D * esz_q;
    const char* kb = (const char*)k + u * unit_stride * esz_kv;
    const char* vb = (const char*)v + u * unit_stride * esz_kv;
    double qi[ORA_D];
    ora_index_query(qb, qtype, G, qi);
    int64_t n_cand = 0, forced = -1;
    decode_candidates(len, force_local, &n_cand, &forced);
    double* sc = (double*)malloc((size_t)(n_cand > 0 ? n_cand : 1) * sizeof(double));
    ora_score_blocks(qi, pooled + u * max_blocks * ORA_D, n_cand, sc);
    int sink = (force_local & 2) != 0;
    int keep0 = sink && num_blocks(len) > 0 && forced != 0;
    int64_t* s = sel + u * k_total;
    if (ora_select_blocks(sc, n_cand, k_scored, forced, (sink && n_cand > 0) ? 1 : 0, keep0, k_total, s) < 0)
      bad |= 1;
    free(sc);
    int64_t* toks = (int64_t*)malloc((size_t)(k_total * ORA_BLOCK + 1) * sizeof(int64_t));
    int64_t nt = 0;
    for (int64_t i = 0; i < k_total; ++i) {
      if (s[i] < 0) continue;
      for (int64_t t = s[i] * ORA_BLOCK; t < s[i] * ORA_BLOCK + ORA_BLOCK && t < len; ++t) toks[nt++] = t;
    }
    ora_attend(qb, qtype, G, kb, vb, kvtype, ld_kv, toks, nt, scale, o + u * (int64_t)G * ORA_D, lse + u * G, NULL);
    free(toks);
  }
  return bad ? -1 : 0;
}

/* Number of OpenMP threads the *_units functions use (1 without OpenMP). */
int ora_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Chunked-prefill tiles (guide §1, Step 1 and Step 2; §3: during prefill the
 * index branch still scans the whole input): for n_units (tile, KV head)
 * units of one sequence, unit u = tile tiles[u] of KV head heads[u], whose
 * queries are chunk rows row_lo[u] .. row_hi[u] - 1 at absolute positions
 * q_start + row: the index query is the sum of those rows' G heads; the
 * candidates are the blocks before the tile's diagonal block
 * q_start / 64 + tiles[u] (always kept); selection as ora_select_blocks; each
 * row then attends, causally, over the tokens <= its position of the listed
 * blocks. q: [n_rows][Hq][128]; k, v: [Hkv][T][128] (row stride 128);
 * pooled: [Hkv][max_blocks][128] stored summaries. Outputs: sel
 * [n_units][k_total]; o [n_rows][Hq][128] and lse [n_rows][Hq] for the rows
 * and heads of the listed units (others untouched). */
int ora_prefill_tile_units(int64_t n_units, const int64_t* tiles, const int64_t* heads, const int64_t* row_lo,
                           const int64_t* row_hi, int64_t q_start, const void* q, int qtype, int Hq, int G,
                           const double* pooled, int64_t max_blocks, const void* k, const void* v, int kvtype,
                           int64_t T, int64_t k_scored, int64_t k_total, double scale, int64_t* sel, double* o,
                           double* lse) {
  int bad = 0;
  int esz_q = qtype == ORA_F64 ? 8 : qtype == ORA_F32 ? 4 : 2;
  int esz_kv = kvtype == ORA_F64 ? 8 : kvtype == ORA_F32 ? 4 : 2;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t u = 0; u < n_units; ++u) {
    int64_t h = heads[u], diag = q_start / ORA_BLOCK + tiles[u];
    if (diag > max_blocks) {
      bad |= 1;
      continue;
    }
    double qi[ORA_D];
    for (int d = 0; d < ORA_D; ++d) {
      double acc = 0.0;
      for (int64_t r = row_lo[u]; r < row_hi[u]; ++r)
        for (int g = 0; g < G; ++g) acc += ld(q, qtype, (r * Hq + h * G + g) * ORA_D + d);
      qi[d] = acc;
    }
    double* sc = (double*)malloc((size_t)(diag > 0 ? diag : 1) * sizeof(double));
    ora_score_blocks(qi, pooled + h * max_blocks * ORA_D, diag, sc);
    int64_t* s = sel + u * k_total;
    if (ora_select_blocks(sc, diag, k_scored, diag, 0, 0, k_total, s) < 0) bad |= 1;
    free(sc);
    const char* kb = (const char*)k + h * T * ORA_D * esz_kv;
    const char* vb = (const char*)v + h * T * ORA_D * esz_kv;
    int64_t* toks = (int64_t*)malloc((size_t)(k_total * ORA_BLOCK + 1) * sizeof(int64_t));
    for (int64_t r = row_lo[u]; r < row_hi[u]; ++r) {
      int64_t pos = q_start + r, nt = 0;
      for (int64_t i = 0; i < k_total; ++i) {
        if (s[i] < 0) continue;
        for (int64_t t = s[i] * ORA_BLOCK; t < s[i] * ORA_BLOCK + ORA_BLOCK && t <= pos && t < T; ++t) toks[nt++] = t;
      }
      const char* qr = (const char*)q + (r * Hq + h * G) * ORA_D * esz_q;
      ora_attend(qr, qtype, G, kb, vb, kvtype, ORA_D, toks, nt, scale, o + (r * Hq + h * G) * ORA_D, lse + r * Hq + h * G,
                 NULL);
    }
    free(toks);
  }
  return bad ? -1 : 0;
}
