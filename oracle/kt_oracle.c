/*
 * kt_oracle.c — the CPU oracle for block-sparse long-context decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load or call this code; the product path
 * never does.  It shares no source with the CUDA library.
 *
 * It is a plain, slow, single-threaded restatement of what the method
 * computes, in double precision, following the article
 *   [LC] "KTransformers 长上下文稀疏注意力实战：单张 24GB GPU 跑通 1M Token
 *         KVCache 的完整方案" (section numbers as printed in the article)
 * and the configuration keys of
 *   [HOWTO] "How to Implement Long Context Inference (Up to 139K Tokens) with
 *           KTransformers", Step 1 (YAML) and Step 3 (attention constructor).
 *
 * Steps, in the article's order:
 *   partition  [LC §4.2, §4.3]  Initial / Context / Local, 128-token blocks
 *   reps       [LC §4.3 table, §3.1]  Max, Mean, Quest (min+max), Fix, Dynamic
 *   score      [LC §3.1] Quest upper bound; dot product for the other methods
 *   select     [LC §4.5] top-k context blocks per KV head (SEPARATE) or jointly
 *                        (SHARED)
 *   attend     [LC §4.6 decode_attention: attn(query, kvcache_after_retrieval)],
 *              softmax(q k^T / sqrt(d_k)) as written in [LC §3.2]
 *   dense      the full scan that [LC §1] says the method avoids
 *
 * Readings where the article is silent:
 *   - Initial/Local are whole blocks; Local counts back from the last, possibly
 *     partial, block; with nb <= I + L every block is attended.
 *   - SHARED sums per-head block scores over all query heads; SEPARATE sums over
 *     the query heads of one KV head (GQA group).
 *   - Preselection [LC §4.4, §4.6]: the vote of a context token is its
 *     accumulated softmax probability over the unit's local query rows (the
 *     Dynamic token scores, summed over the unit's KV heads); "pool1d" is an
 *     average pool with zero padding (odd kernel, padding kernel/2, stride 1)
 *     over the context tokens; a block is preselected when its tokens come
 *     first in descending pooled vote, i.e. the top `count` blocks by their
 *     largest pooled vote.
 *   - Fix and Dynamic score a block by the max over its reps of q.rep.
 *   - Fix takes tokens 0, s, 2s, ... of the block.
 *   - Mean is the exact mean rounded once to binary32.
 *   - Max/min use the binary16 total order, so -0 < +0.
 *   - Top-k ties go to the lower block index; k > C selects all C blocks.
 *   - Selection scores are unscaled; attention uses scale 1/sqrt(d).
 *   - The decode query sees all n cached tokens (no mask).
 *   - Dynamic: accumulated probability of each token = sum over the last T
 *     positions' queries (causal: position p sees tokens <= p) and the query
 *     heads of the KV head; the num_reps best tokens of a block (ties: lower
 *     index) are its reps, kept in token order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_MAX = 0, ORC_MEAN = 1, ORC_QUEST = 2, ORC_FIX = 3, ORC_DYNAMIC = 4 };
enum { ORC_SHARED = 0, ORC_SEPARATE = 1 };

typedef struct {
  const uint16_t* k_pool;      /* [P][H_kv][bs][d] binary16 bits */
  const uint16_t* v_pool;      /* [P][H_kv][bs][d] */
  const int32_t* block_table;  /* [B][max_blocks] logical block -> page */
  const int32_t* seq_lens;     /* [B] tokens */
  int64_t B, H_kv, d, bs, max_blocks, P;
} orc_kv;

typedef struct {
  int64_t H_q;
  int64_t initial_blocks, local_blocks, top_k;
  int64_t rep, head_mode, num_reps, fix_stride;
  double softmax_scale;
} orc_params;

/* ---- binary16 ------------------------------------------------------------ */

/* Value of a binary16 bit pattern (IEEE 754-2008 §3.4: sign, 5-bit biased
 * exponent, 10-bit trailing significand; bias 15). */
double orc_f16_to_double(uint16_t h) {
  int s = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);            /* subnormal: m * 2^(1-15-10) */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return s ? -v : v;
}

/* Decoded value of every binary16 pattern (filled once from orc_f16_to_double). */
static double F16[65536];
static int f16_ready = 0;

static double dec(uint16_t h) {
  if (!f16_ready) {
    for (int i = 0; i < 65536; ++i) F16[i] = orc_f16_to_double((uint16_t)i);
    f16_ready = 1;
  }
  return F16[h];
}

/* a < b in the binary16 total order (values first; -0 below +0). */
static int h16_less(uint16_t a, uint16_t b) {
  double va = dec(a), vb = dec(b);
  if (va != vb) return va < vb;
  return (a & 0x8000u) && !(b & 0x8000u); /* -0 < +0 */
}

/* ---- partition [LC §4.2, §4.3] --------------------------------------------- */

/* nb blocks; context blocks are [*c0, *c1); Initial = [0, c0), Local = [c1, nb). */
void orc_partition(int64_t n, int64_t bs, int64_t I, int64_t L, int64_t* nb,
                   int64_t* c0, int64_t* c1) {
  int64_t nbl = (n + bs - 1) / bs;
  int64_t a = I < nbl ? I : nbl;
  int64_t z = nbl - L;
  if (z < a) z = a;
  *nb = nbl;
  *c0 = a;
  *c1 = z;
}

static uint16_t k_bits(const orc_kv* kv, int64_t b, int64_t h, int64_t t, int64_t c) {
  int64_t page = kv->block_table[b * kv->max_blocks + t / kv->bs];
  return kv->k_pool[((page * kv->H_kv + h) * kv->bs + t % kv->bs) * kv->d + c];
}

static double k_val(const orc_kv* kv, int64_t b, int64_t h, int64_t t, int64_t c) {
  return dec(k_bits(kv, b, h, t, c));
}

static double v_val(const orc_kv* kv, int64_t b, int64_t h, int64_t t, int64_t c) {
  int64_t page = kv->block_table[b * kv->max_blocks + t / kv->bs];
  return dec(kv->v_pool[((page * kv->H_kv + h) * kv->bs + t % kv->bs) * kv->d + c]);
}

int64_t orc_reps_per_block(const orc_params* p, int64_t bs) {
  switch (p->rep) {
    case ORC_MAX: case ORC_MEAN: return 1;
    case ORC_QUEST: return 2;
    case ORC_FIX: return (bs + p->fix_stride - 1) / p->fix_stride;
    default: return p->num_reps;
  }
}

/* ---- representatives [LC §4.3 table; Quest §3.1] ------------------------------
 * For a full block j of sequence b and KV head h.  Binary16 methods write R*d
 * bit patterns to out_h16; Mean writes d binary32 values to out_f32.
 * Dynamic needs the accumulated token scores (see orc_dynamic_token_scores).
 */
void orc_block_reps(const orc_kv* kv, int64_t b, int64_t j, int64_t h, const orc_params* p,
                    const double* dyn_scores /* [n] of (b, h) or NULL */,
                    uint16_t* out_h16, float* out_f32) {
  const int64_t bs = kv->bs, d = kv->d, t0 = j * bs;
  if (p->rep == ORC_MAX || p->rep == ORC_QUEST) {
    /* Max: per channel maximum; Quest: per channel minimum and maximum (rows 0, 1). */
    for (int64_t c = 0; c < d; ++c) {
      uint16_t mx = k_bits(kv, b, h, t0, c), mn = mx;
      for (int64_t t = 1; t < bs; ++t) {
        uint16_t x = k_bits(kv, b, h, t0 + t, c);
        if (h16_less(mx, x)) mx = x;
        if (h16_less(x, mn)) mn = x;
      }
      if (p->rep == ORC_MAX) {
        out_h16[c] = mx;
      } else {
        out_h16[c] = mn;
        out_h16[d + c] = mx;
      }
    }
  } else if (p->rep == ORC_MEAN) {
    /* Per channel mean.  The double sum of 128 binary16 values is exact (all are
     * multiples of 2^-24 below 2^16, so partial sums need < 47 bits); the single
     * rounding is the conversion to binary32. */
    for (int64_t c = 0; c < d; ++c) {
      double s = 0.0;
      for (int64_t t = 0; t < bs; ++t) s += k_val(kv, b, h, t0 + t, c);
      out_f32[c] = (float)(s / (double)bs);
    }
  } else if (p->rep == ORC_FIX) {
    /* Tokens at a fixed interval: offsets 0, s, 2s, ... */
    int64_t r = 0;
    for (int64_t t = 0; t < bs; t += p->fix_stride, ++r)
      for (int64_t c = 0; c < d; ++c) out_h16[r * d + c] = k_bits(kv, b, h, t0 + t, c);
  } else {
    /* Dynamic: the num_reps tokens with the highest accumulated score; ties go to
     * the lower token index; the chosen rows are emitted in token order. */
    int64_t R = p->num_reps;
    char* taken = (char*)calloc((size_t)bs, 1);
    for (int64_t r = 0; r < R && r < bs; ++r) {
      int64_t best = -1;
      for (int64_t t = 0; t < bs; ++t) {
        if (taken[t]) continue;
        if (best < 0 || dyn_scores[t0 + t] > dyn_scores[t0 + best]) best = t;
      }
      taken[best] = 1;
    }
    int64_t r = 0;
    for (int64_t t = 0; t < bs; ++t)
      if (taken[t]) {
        for (int64_t c = 0; c < d; ++c) out_h16[r * d + c] = k_bits(kv, b, h, t0 + t, c);
        ++r;
      }
    free(taken);
  }
}

/* ---- Dynamic token scores [LC §4.3 "Dynamic"; softmax as in §3.2] -------------
 * acc[t], t in [0, n): sum over the T local queries (positions n-T+i) and the G
 * query heads of KV head h of softmax_t(q . k_t * scale), where the query at
 * position pos sees tokens 0..pos.  q_local is [T][H_q][d] for sequence b.
 */
void orc_dynamic_token_scores(const orc_kv* kv, int64_t b, int64_t h, const orc_params* p,
                              const uint16_t* q_local, int64_t T, double* acc) {
  const int64_t n = kv->seq_lens[b], d = kv->d, G = p->H_q / kv->H_kv;
  double* kd = (double*)malloc(sizeof(double) * (size_t)((n > 0 ? n : 1) * d));
  double* logit = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* q = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t t = 0; t < n; ++t)
    for (int64_t c = 0; c < d; ++c) kd[t * d + c] = k_val(kv, b, h, t, c);
  for (int64_t t = 0; t < n; ++t) acc[t] = 0.0;
  for (int64_t i = 0; i < T; ++i) {
    int64_t pos = n - T + i;
    if (pos < 0) continue;
    for (int64_t g = 0; g < G; ++g) {
      int64_t hq = h * G + g;
      for (int64_t c = 0; c < d; ++c) q[c] = dec(q_local[(i * p->H_q + hq) * d + c]);
      double m = -INFINITY;
      for (int64_t t = 0; t <= pos; ++t) {
        double s = 0.0;
        for (int64_t c = 0; c < d; ++c) s += q[c] * kd[t * d + c];
        logit[t] = s * p->softmax_scale;
        if (logit[t] > m) m = logit[t];
      }
      double z = 0.0;
      for (int64_t t = 0; t <= pos; ++t) z += exp(logit[t] - m);
      for (int64_t t = 0; t <= pos; ++t) acc[t] += exp(logit[t] - m) / z;
    }
  }
  free(kd);
  free(logit);
  free(q);
}

/* ---- block score of one query head [LC §3.1, §4.3] ----------------------------
 * reps: R*d values of the block's reps for the head's KV head.
 */
double orc_head_block_score(const double* q, const double* reps, int64_t R, int64_t d, int64_t rep) {
  if (rep == ORC_QUEST) {
    /* Upper bound of q.k over the block: per channel the larger of q_c*kmax_c and
     * q_c*kmin_c, summed over channels.  Row 0 holds kmin, row 1 kmax. */
    double s = 0.0;
    for (int64_t c = 0; c < d; ++c) {
      double a = q[c] * reps[d + c], bb = q[c] * reps[c];
      s += a > bb ? a : bb;
    }
    return s;
  }
  double best = -INFINITY;
  for (int64_t r = 0; r < R; ++r) {
    double s = 0.0;
    for (int64_t c = 0; c < d; ++c) s += q[c] * reps[r * d + c];
    if (s > best) best = s;
  }
  return best;
}

/* ---- selection [LC §4.5] ----------------------------------------------------- */

typedef struct { double s; int64_t j; } scored;

static int by_score_then_block(const void* a, const void* b) {
  const scored* x = (const scored*)a;
  const scored* y = (const scored*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->j > y->j) - (x->j < y->j);
}

static int ascending_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

/* Top min(k, C) of blocks c0..c0+C-1 by (score desc, block asc), written in
 * ascending block order.  Returns the count. */
int64_t orc_select(const double* score /* [C] */, int64_t c0, int64_t C, int64_t k,
                   int32_t* sel) {
  if (C <= 0 || k <= 0) return 0;
  scored* v = (scored*)malloc(sizeof(scored) * (size_t)C);
  for (int64_t i = 0; i < C; ++i) {
    v[i].s = score[i];
    v[i].j = c0 + i;
  }
  qsort(v, (size_t)C, sizeof(scored), by_score_then_block);
  int64_t cnt = k < C ? k : C;
  for (int64_t i = 0; i < cnt; ++i) sel[i] = (int32_t)v[i].j;
  qsort(sel, (size_t)cnt, sizeof(int32_t), ascending_i32);
  free(v);
  return cnt;
}

/* ---- attention [LC §4.6; softmax(q k^T / sqrt(d_k)) of §3.2] -------------------
 * Exact softmax attention of query head hq of sequence b over the valid tokens
 * of the listed logical blocks: m = max logit, w = exp(logit - m),
 * out = sum w v / sum w.  With no tokens the output is zero.
 */
void orc_attend(const orc_kv* kv, int64_t b, int64_t hq, int64_t H_q, const uint16_t* q_bits,
                const int32_t* blocks, int64_t nblocks, double scale, double* out) {
  const int64_t d = kv->d, bs = kv->bs, n = kv->seq_lens[b];
  const int64_t h = hq / (H_q / kv->H_kv);
  double* q = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t c = 0; c < d; ++c) q[c] = dec(q_bits[c]);
  int64_t ntok = 0;
  for (int64_t i = 0; i < nblocks; ++i) {
    int64_t t1 = (blocks[i] + 1) * bs < n ? (blocks[i] + 1) * bs : n;
    ntok += t1 - blocks[i] * bs;
  }
  double* logit = (double*)malloc(sizeof(double) * (size_t)(ntok > 0 ? ntok : 1));
  int64_t* tok = (int64_t*)malloc(sizeof(int64_t) * (size_t)(ntok > 0 ? ntok : 1));
  int64_t k = 0;
  double m = -INFINITY;
  for (int64_t i = 0; i < nblocks; ++i) {
    int64_t t1 = (blocks[i] + 1) * bs < n ? (blocks[i] + 1) * bs : n;
    for (int64_t t = blocks[i] * bs; t < t1; ++t, ++k) {
      double s = 0.0;
      for (int64_t c = 0; c < d; ++c) s += q[c] * k_val(kv, b, h, t, c);
      logit[k] = s * scale;
      tok[k] = t;
      if (logit[k] > m) m = logit[k];
    }
  }
  for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
  double z = 0.0;
  for (k = 0; k < ntok; ++k) {
    double w = exp(logit[k] - m);
    z += w;
    for (int64_t c = 0; c < d; ++c) out[c] += w * v_val(kv, b, h, tok[k], c);
  }
  if (ntok > 0)
    for (int64_t c = 0; c < d; ++c) out[c] /= z;
  free(q);
  free(logit);
  free(tok);
}

/* Dense decode: every query head over all n tokens [LC §1 full scan]. */
void orc_dense(const orc_kv* kv, const uint16_t* q /* [B][H_q][d] */, int64_t H_q, double scale,
               double* out /* [B][H_q][d] */) {
  int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)(kv->max_blocks > 0 ? kv->max_blocks : 1));
  for (int64_t b = 0; b < kv->B; ++b) {
    int64_t nb = (kv->seq_lens[b] + kv->bs - 1) / kv->bs;
    for (int64_t j = 0; j < nb; ++j) all[j] = (int32_t)j;
    for (int64_t hq = 0; hq < H_q; ++hq)
      orc_attend(kv, b, hq, H_q, q + (b * H_q + hq) * kv->d, all, nb, scale,
                 out + (b * H_q + hq) * kv->d);
  }
  free(all);
}

/* ---- one decode step ---------------------------------------------------------
 * reps -> unit scores -> top-k -> attention over Initial + selected + Local.
 * Split in two so that the (amortised) representative build can be timed apart
 * from the per-step work.
 *
 *   q            [B][H_q][d]                 decode queries
 *   q_local      [B][T][H_q][d] or NULL      local-window queries (Dynamic only)
 *   rv           [B][max_blocks][H_kv][R][d] representative values as doubles
 *   reps_h16     [B][max_blocks][H_kv][R][d] or NULL   binary16 reps (not Mean)
 *   reps_f32     [B][max_blocks][H_kv][d] or NULL      Mean reps
 *   dyn_scores   [B][H_kv][max_blocks*bs] or NULL      Dynamic token scores
 *   unit_scores  [B][SEL][max_blocks] or NULL  (NaN outside the context range)
 *   sel          [B][SEL][top_k], cnt [B][SEL]     SEL = 1 (SHARED) or H_kv
 *   out          [B][H_q][d]
 *   unit_lo/hi   only selection units in [unit_lo, unit_hi) and their query heads
 *                are computed (for sampled checks); pass 0, SEL for all.
 * Each returns 0, or -1 on an unsupported argument.
 */
static int check_args(const orc_kv* kv, const orc_params* p, const uint16_t* q_local,
                      int64_t T) {
  if (p->H_q % kv->H_kv != 0 || p->local_blocks < 1 || p->top_k < 0) return -1;
  if (p->rep == ORC_DYNAMIC && (q_local == NULL || T < 1)) return -1;
  if (p->rep == ORC_FIX && p->fix_stride < 1) return -1;
  return 0;
}

int orc_build_all_reps(const orc_kv* kv, const orc_params* p, const uint16_t* q_local, int64_t T,
                       double* rv, uint16_t* reps_h16, float* reps_f32, double* dyn_scores,
                       int64_t unit_lo, int64_t unit_hi) {
  const int64_t B = kv->B, H_kv = kv->H_kv, d = kv->d, bs = kv->bs, MB = kv->max_blocks;
  const int64_t H_q = p->H_q, R = orc_reps_per_block(p, bs);
  if (check_args(kv, p, q_local, T)) return -1;
  uint16_t* hb = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(R * d));
  float* fb = (float*)malloc(sizeof(float) * (size_t)d);
  double* dyn = p->rep == ORC_DYNAMIC ? (double*)malloc(sizeof(double) * (size_t)(MB * bs)) : NULL;
  for (int64_t b = 0; b < B; ++b) {
    int64_t n = kv->seq_lens[b], nb, c0, c1;
    orc_partition(n, bs, p->initial_blocks, p->local_blocks, &nb, &c0, &c1);
    for (int64_t h = 0; h < H_kv; ++h) {
      int64_t u = p->head_mode == ORC_SHARED ? 0 : h;
      if (u < unit_lo || u >= unit_hi) continue;
      if (p->rep == ORC_DYNAMIC) {
        orc_dynamic_token_scores(kv, b, h, p, q_local + b * T * H_q * d, T, dyn);
        if (dyn_scores)
          for (int64_t t = 0; t < MB * bs; ++t)
            dyn_scores[(b * H_kv + h) * MB * bs + t] = t < n ? dyn[t] : 0.0;
      }
      for (int64_t j = 0; j < nb; ++j) {
        if ((j + 1) * bs > n) continue; /* reps exist for full blocks only */
        orc_block_reps(kv, b, j, h, p, dyn, hb, fb);
        double* dst = rv + ((b * MB + j) * H_kv + h) * R * d;
        if (p->rep == ORC_MEAN) {
          for (int64_t c = 0; c < d; ++c) dst[c] = (double)fb[c];
          if (reps_f32) memcpy(reps_f32 + ((b * MB + j) * H_kv + h) * d, fb, sizeof(float) * (size_t)d);
        } else {
          for (int64_t i = 0; i < R * d; ++i) dst[i] = dec(hb[i]);
          if (reps_h16)
            memcpy(reps_h16 + ((b * MB + j) * H_kv + h) * R * d, hb, sizeof(uint16_t) * (size_t)(R * d));
        }
      }
    }
  }
  free(hb);
  free(fb);
  free(dyn);
  return 0;
}

/* Score, select and attend; with presel (non-NULL) the selection of unit u
 * of sequence b only considers the presel_cnt[b*SEL+u] blocks listed at
 * presel[(b*SEL+u)*presel_stride ...] (the preselection of [LC §4.4]). */
int orc_score_select_attend_presel(const orc_kv* kv, const uint16_t* q, const orc_params* p,
                                   const double* rv, double* unit_scores, int32_t* sel,
                                   int32_t* cnt, double* out, int64_t unit_lo, int64_t unit_hi,
                                   const int32_t* presel, const int32_t* presel_cnt,
                                   int64_t presel_stride) {
  const int64_t B = kv->B, H_kv = kv->H_kv, d = kv->d, bs = kv->bs, MB = kv->max_blocks;
  const int64_t H_q = p->H_q, G = H_q / H_kv, R = orc_reps_per_block(p, bs);
  const int64_t SEL = p->head_mode == ORC_SHARED ? 1 : H_kv;
  if (p->H_q % kv->H_kv != 0 || p->local_blocks < 1 || p->top_k < 0) return -1;
  if (unit_lo < 0) unit_lo = 0;
  if (unit_hi > SEL) unit_hi = SEL;
  double* qd = (double*)malloc(sizeof(double) * (size_t)d);
  double* score = (double*)malloc(sizeof(double) * (size_t)(MB > 0 ? MB : 1));
  int32_t* list = (int32_t*)malloc(sizeof(int32_t) * (size_t)(MB + 1));
  for (int64_t b = 0; b < B; ++b) {
    int64_t n = kv->seq_lens[b], nb, c0, c1;
    orc_partition(n, bs, p->initial_blocks, p->local_blocks, &nb, &c0, &c1);
    for (int64_t u = unit_lo; u < unit_hi; ++u) {
      /* unit score of each context block: sum of head scores over the unit's
       * query heads, in ascending head order */
      int64_t h_first = p->head_mode == ORC_SHARED ? 0 : u * G;
      int64_t h_last = p->head_mode == ORC_SHARED ? H_q : (u + 1) * G;
      for (int64_t j = c0; j < c1; ++j) score[j - c0] = 0.0;
      for (int64_t hq = h_first; hq < h_last; ++hq) {
        int64_t h = hq / G;
        for (int64_t c = 0; c < d; ++c) qd[c] = dec(q[(b * H_q + hq) * d + c]);
        for (int64_t j = c0; j < c1; ++j)
          score[j - c0] +=
              orc_head_block_score(qd, rv + ((b * MB + j) * H_kv + h) * R * d, R, d, p->rep);
      }
      if (unit_scores)
        for (int64_t j = 0; j < MB; ++j)
          unit_scores[(b * SEL + u) * MB + j] = (j >= c0 && j < c1) ? score[j - c0] : NAN;
      int32_t* su = sel + (b * SEL + u) * p->top_k;
      int64_t cu;
      if (presel) {
        /* only the preselected context blocks compete */
        const int32_t* ps = presel + (b * SEL + u) * presel_stride;
        const int64_t np = presel_cnt[b * SEL + u];
        scored* v = (scored*)malloc(sizeof(scored) * (size_t)(np > 0 ? np : 1));
        int64_t m2 = 0;
        for (int64_t i = 0; i < np; ++i)
          if (ps[i] >= c0 && ps[i] < c1) {
            v[m2].s = score[ps[i] - c0];
            v[m2].j = ps[i];
            ++m2;
          }
        qsort(v, (size_t)m2, sizeof(scored), by_score_then_block);
        cu = p->top_k < m2 ? p->top_k : m2;
        for (int64_t i = 0; i < cu; ++i) su[i] = (int32_t)v[i].j;
        qsort(su, (size_t)cu, sizeof(int32_t), ascending_i32);
        free(v);
      } else {
        cu = orc_select(score, c0, c1 - c0, p->top_k, su);
      }
      cnt[b * SEL + u] = (int32_t)cu;
      /* token set = Initial + selected Context + Local [LC §4.2] */
      int64_t m = 0;
      for (int64_t j = 0; j < c0; ++j) list[m++] = (int32_t)j;
      for (int64_t i = 0; i < cu; ++i) list[m++] = su[i];
      for (int64_t j = c1; j < nb; ++j) list[m++] = (int32_t)j;
      for (int64_t hq = h_first; hq < h_last; ++hq)
        orc_attend(kv, b, hq, H_q, q + (b * H_q + hq) * d, list, m, p->softmax_scale,
                   out + (b * H_q + hq) * d);
    }
  }
  free(qd);
  free(score);
  free(list);
  return 0;
}

int orc_score_select_attend(const orc_kv* kv, const uint16_t* q, const orc_params* p,
                            const double* rv, double* unit_scores, int32_t* sel, int32_t* cnt,
                            double* out, int64_t unit_lo, int64_t unit_hi) {
  return orc_score_select_attend_presel(kv, q, p, rv, unit_scores, sel, cnt, out, unit_lo,
                                        unit_hi, NULL, NULL, 0);
}

/* ---- preselection [LC §4.4; §4.6 preselect_block()] ----------------------------
 * Average pooling along a vector with zero padding: out[t] = (sum of in[u] for
 * u in [t - kernel/2, t + kernel/2] inside [0, n)) / kernel, kernel odd. */
void orc_avg_pool1d(const double* in, int64_t n, int64_t kernel, double* out) {
  const int64_t half = kernel / 2;
  for (int64_t t = 0; t < n; ++t) {
    double s = 0.0;
    for (int64_t u = t - half; u <= t + half; ++u)
      if (u >= 0 && u < n) s += in[u];
    out[t] = s / (double)kernel;
  }
}

/* The vote of each context token of a unit is its accumulated softmax
 * probability over the unit's local query rows (the Dynamic token scores of
 * each of the unit's KV heads, summed over those heads); votes are
 * average-pooled along the context tokens; tokens are taken in descending
 * pooled vote and their blocks collected until `count` distinct context blocks
 * are preselected.  Taking tokens in that order reaches each block at its
 * largest pooled vote, so this equals the top `count` blocks by (largest
 * pooled vote of its tokens desc, block asc).  Writes presel[(b*SEL+u)*count ..]
 * ascending and presel_cnt[b*SEL+u] = min(count, C). */
int orc_preselect(const orc_kv* kv, const orc_params* p, const uint16_t* q_local, int64_t T,
                  int64_t kernel, int64_t count, int32_t* presel, int32_t* presel_cnt) {
  const int64_t B = kv->B, H_kv = kv->H_kv, bs = kv->bs, H_q = p->H_q, d = kv->d;
  const int64_t SEL = p->head_mode == ORC_SHARED ? 1 : H_kv;
  if (kernel < 1 || (kernel % 2) == 0 || count < 1 || T < 1 || H_q % H_kv != 0) return -1;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t n = kv->seq_lens[b];
    int64_t nb, c0, c1;
    orc_partition(n, bs, p->initial_blocks, p->local_blocks, &nb, &c0, &c1);
    const int64_t C = c1 - c0, ntok = C * bs;
    double* acc = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double* vote = (double*)calloc((size_t)(ntok > 0 ? ntok : 1), sizeof(double));
    double* pooled = (double*)malloc(sizeof(double) * (size_t)(ntok > 0 ? ntok : 1));
    double* bscore = (double*)malloc(sizeof(double) * (size_t)(C > 0 ? C : 1));
    const uint16_t* qb = q_local + b * T * H_q * d;
    for (int64_t u = 0; u < SEL; ++u) {
      for (int64_t t = 0; t < ntok; ++t) vote[t] = 0.0;
      const int64_t h0 = p->head_mode == ORC_SHARED ? 0 : u;
      const int64_t h1 = p->head_mode == ORC_SHARED ? H_kv : u + 1;
      for (int64_t h = h0; h < h1; ++h) {
        orc_dynamic_token_scores(kv, b, h, p, qb, T, acc);
        for (int64_t t = 0; t < ntok; ++t) vote[t] += acc[c0 * bs + t];
      }
      orc_avg_pool1d(vote, ntok, kernel, pooled);
      for (int64_t j = 0; j < C; ++j) {
        double m = -INFINITY;
        for (int64_t t = 0; t < bs; ++t)
          if (pooled[j * bs + t] > m) m = pooled[j * bs + t];
        bscore[j] = m;
      }
      presel_cnt[b * SEL + u] =
          (int32_t)orc_select(bscore, c0, C, count, presel + (b * SEL + u) * count);
    }
    free(acc);
    free(vote);
    free(pooled);
    free(bscore);
  }
  return 0;
}

int orc_sparse_step(const orc_kv* kv, const uint16_t* q, const orc_params* p,
                    const uint16_t* q_local, int64_t T, uint16_t* reps_h16, float* reps_f32,
                    double* dyn_scores, double* unit_scores, int32_t* sel, int32_t* cnt,
                    double* out, int64_t unit_lo, int64_t unit_hi) {
  const int64_t R = orc_reps_per_block(p, kv->bs);
  if (check_args(kv, p, q_local, T)) return -1;
  double* rv = (double*)calloc((size_t)(kv->B * kv->max_blocks * kv->H_kv * R * kv->d), sizeof(double));
  int rc = orc_build_all_reps(kv, p, q_local, T, rv, reps_h16, reps_f32, dyn_scores, unit_lo, unit_hi);
  if (rc == 0) rc = orc_score_select_attend(kv, q, p, rv, unit_scores, sel, cnt, out, unit_lo, unit_hi);
  free(rv);
  return rc;
}

/* orc_sparse_step with the selection restricted to a preselection. */
int orc_sparse_step_presel(const orc_kv* kv, const uint16_t* q, const orc_params* p,
                           const uint16_t* q_local, int64_t T, double* unit_scores, int32_t* sel,
                           int32_t* cnt, double* out, int64_t unit_lo, int64_t unit_hi,
                           const int32_t* presel, const int32_t* presel_cnt,
                           int64_t presel_stride) {
  const int64_t R = orc_reps_per_block(p, kv->bs);
  if (check_args(kv, p, q_local, T)) return -1;
  double* rv = (double*)calloc((size_t)(kv->B * kv->max_blocks * kv->H_kv * R * kv->d), sizeof(double));
  int rc = orc_build_all_reps(kv, p, q_local, T, rv, NULL, NULL, NULL, unit_lo, unit_hi);
  if (rc == 0)
    rc = orc_score_select_attend_presel(kv, q, p, rv, unit_scores, sel, cnt, out, unit_lo,
                                        unit_hi, presel, presel_cnt, presel_stride);
  free(rv);
  return rc;
}

/* Vector form of orc_f16_to_double, for the tests. */
void orc_f16_array(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_double(in[i]);
}

/* ---- quantised KV, Q8_0 (the kv_type choices FP16 / FP32 / Q4_0 / Q8_0 of
 * [HOWTO] Step 1; Q8_0 is the 8-bit block format of the llama.cpp family that
 * the key names) ---------------------------------------------------------------
 * Reading taken (the pages name the type, not its arithmetic): a row of 128
 * channels of K or V is cut into 4 groups of 32 channels; a group keeps one
 * binary16 scale and 32 signed 8-bit codes.  With amax the largest |x| of the
 * group in binary32, dd = amax / 127 and id = 1 / dd (0 when dd is 0) in
 * binary32, the code of x is round-half-away-from-zero(x * id) (binary32
 * product) and the stored scale is dd rounded to binary16; the dequantised
 * value is dec(scale) * code.  The codes are decided in binary32 so that an
 * implementation in that precision reproduces them exactly. */

/* binary32 -> binary16, round to nearest even (IEEE 754-2008 §4.3.1, §3.4). */
uint16_t orc_f32_to_f16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  if (f != f) return (uint16_t)(sign | 0x7E00u);
  const double a = fabs((double)f);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u); /* past the midpoint above 65504 */
  if (a < ldexp(1.0, -14)) {
    /* subnormal (or zero): units of 2^-24; 1024 units become the smallest normal */
    const double qq = rint(ldexp(a, 24));
    return (uint16_t)(sign | (uint16_t)qq);
  }
  int e;
  const double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
  double q = rint(ldexp(m, 11));  /* 1024 .. 2048 */
  int E = e - 1;                  /* a in [2^E, 2^(E+1)) */
  if (q >= 2048.0) {
    q = 1024.0;
    E += 1;
  }
  if (E > 15) return (uint16_t)(sign | 0x7C00u);
  return (uint16_t)(sign | (uint16_t)((E + 15) << 10) | (uint16_t)(q - 1024.0));
}

/* rows x 128 binary16 values -> codes [rows][128] and scales [rows][4]. */
void orc_quantize_q8_0(const uint16_t* x, int64_t rows, int8_t* code, uint16_t* scale) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t g = 0; g < 4; ++g) {
      const uint16_t* xs = x + r * 128 + g * 32;
      float amax = 0.0f;
      for (int j = 0; j < 32; ++j) {
        const float a = fabsf((float)dec(xs[j]));
        if (a > amax) amax = a;
      }
      const float dd = amax / 127.0f;
      const float id = dd != 0.0f ? 1.0f / dd : 0.0f;
      scale[r * 4 + g] = orc_f32_to_f16(dd);
      for (int j = 0; j < 32; ++j) {
        const float t = (float)dec(xs[j]) * id;
        code[r * 128 + g * 32 + j] = (int8_t)roundf(t);
      }
    }
}

typedef struct {
  const int8_t* k_code;      /* [P][H_kv][bs][d] */
  const uint16_t* k_scale;   /* [P][H_kv][bs][d/32] binary16 */
  const int8_t* v_code;
  const uint16_t* v_scale;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int64_t B, H_kv, d, bs, max_blocks, P;
} orc_kvq;

static double q8_val(const int8_t* code, const uint16_t* scale, const orc_kvq* kv, int64_t b,
                     int64_t h, int64_t t, int64_t c) {
  const int64_t page = kv->block_table[b * kv->max_blocks + t / kv->bs];
  const int64_t row = (page * kv->H_kv + h) * kv->bs + t % kv->bs;
  return dec(scale[row * (kv->d / 32) + c / 32]) * (double)code[row * kv->d + c];
}

/* orc_attend over the dequantised K and V of the listed blocks. */
void orc_attend_q8(const orc_kvq* kv, int64_t b, int64_t hq, int64_t H_q, const uint16_t* q_bits,
                   const int32_t* blocks, int64_t nblocks, double scale, double* out) {
  const int64_t d = kv->d, bs = kv->bs, G = H_q / kv->H_kv, h = hq / G;
  const int64_t n = kv->seq_lens[b];
  double* q = (double*)malloc(sizeof(double) * (size_t)d);
  for (int64_t c = 0; c < d; ++c) q[c] = dec(q_bits[c]);
  double m = -INFINITY;
  for (int64_t i = 0; i < nblocks; ++i)
    for (int64_t t = blocks[i] * bs; t < (blocks[i] + 1) * bs && t < n; ++t) {
      double s = 0.0;
      for (int64_t c = 0; c < d; ++c) s += q[c] * q8_val(kv->k_code, kv->k_scale, kv, b, h, t, c);
      s *= scale;
      if (s > m) m = s;
    }
  double z = 0.0;
  for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
  for (int64_t i = 0; i < nblocks; ++i)
    for (int64_t t = blocks[i] * bs; t < (blocks[i] + 1) * bs && t < n; ++t) {
      double s = 0.0;
      for (int64_t c = 0; c < d; ++c) s += q[c] * q8_val(kv->k_code, kv->k_scale, kv, b, h, t, c);
      const double w = exp(s * scale - m);
      z += w;
      for (int64_t c = 0; c < d; ++c) out[c] += w * q8_val(kv->v_code, kv->v_scale, kv, b, h, t, c);
    }
  for (int64_t c = 0; c < d; ++c) out[c] = z > 0.0 ? out[c] / z : 0.0;
  free(q);
}
