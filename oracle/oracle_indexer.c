/*
 * oracle_indexer.c -- plain, slow, fp64 reference of the sparse-attention key
 * selection (the "lightning indexer" and its top-k).  TEST INFRASTRUCTURE
 * ONLY: only the tests, the package smoke check and the benchmark's
 * CPU-baseline leg may load it.  It shares no code, header or table with the
 * CUDA library.
 *
 * What it computes, and where the pages state it:
 *
 *  "25GB RAM runs 744B GLM-5.2" page (pwwt.cn), section 3.3: every layer keeps
 *  only the top-2048 causal keys for attention; section 4.4: a light indexer
 *  first scores the earlier keys, then the top-k entries are selected, and the
 *  indexer itself still has to do the scoring and the top-k.  The pages give
 *  no scoring formula; the reading here is that of the DeepSeek-V3.2 paper the
 *  page cites for DSA:
 *
 *    I[t][s] = sum_{j < H} w[t][j] * max(0, sum_{i < d} q[t][j][i] * k[s][i])
 *
 *  with H indexer heads of dimension d, one key vector per earlier position s
 *  and per-head weights w of the query token.  Query t sits at position
 *  pos0 + t and sees the keys s <= pos0 + t (causal).  The selection keeps the
 *  topk largest scores, a tie going to the lower key index; it is reported in
 *  ascending key order, padded with -1 when fewer keys are visible.
 *
 * q and k are bf16 bit patterns (converted exactly), w is fp32; everything
 * accumulates in double in the index order written here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* scores[t][s] for s < L; keys the query does not see get -INFINITY */
int orc_indexer_scores(int T, int L, int H, int d, int pos0, const uint16_t* q, const float* w, const uint16_t* k,
                       double* scores, int nthreads) {
  if (T < 1 || L < 1 || H < 1 || d < 1) return -1;
#pragma omp parallel for schedule(static) num_threads(nthreads > 0 ? nthreads : 1)
  for (long long ts = 0; ts < (long long)T * L; ++ts) {
    const int t = (int)(ts / L), s = (int)(ts % L);
    if (s > pos0 + t) {
      scores[ts] = -INFINITY;
      continue;
    }
    double acc = 0.0;
    for (int j = 0; j < H; ++j) {
      double dot = 0.0;
      for (int i = 0; i < d; ++i)
        dot += bf16_value(q[((size_t)t * H + j) * d + i]) * bf16_value(k[(size_t)s * d + i]);
      acc += (double)w[(size_t)t * H + j] * (dot > 0.0 ? dot : 0.0);
    }
    scores[ts] = acc;
  }
  return 0;
}

typedef struct {
  double v;
  int s;
} orc_scored;

/* descending score, ties -> lower key index first */
static int by_score_desc(const void* pa, const void* pb) {
  const orc_scored* a = (const orc_scored*)pa;
  const orc_scored* b = (const orc_scored*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->s > b->s) - (a->s < b->s);
}

static int by_index(const void* pa, const void* pb) {
  const int a = *(const int*)pa, b = *(const int*)pb;
  return (a > b) - (a < b);
}

/* idx[t][0..topk): the selected keys in ascending order, -1 padded;
   gap[t] = topk-th minus (topk+1)-th largest visible score (+INFINITY when
   all visible keys are selected) */
int orc_indexer_topk(int T, int L, int topk, const double* scores, int32_t* idx, double* gap) {
  if (T < 1 || L < 1 || topk < 1) return -1;
  orc_scored* buf = (orc_scored*)malloc(sizeof(orc_scored) * (size_t)L);
  int* sel = (int*)malloc(sizeof(int) * (size_t)topk);
  if (!buf || !sel) {
    free(buf);
    free(sel);
    return -2;
  }
  for (int t = 0; t < T; ++t) {
    int n = 0;
    for (int s = 0; s < L; ++s) {
      const double v = scores[(size_t)t * L + s];
      if (v == -INFINITY) continue;  /* not visible to this query */
      buf[n].v = v;
      buf[n].s = s;
      ++n;
    }
    qsort(buf, (size_t)n, sizeof(orc_scored), by_score_desc);
    const int m = n < topk ? n : topk;
    for (int i = 0; i < m; ++i) sel[i] = buf[i].s;
    qsort(sel, (size_t)m, sizeof(int), by_index);
    for (int i = 0; i < topk; ++i) idx[(size_t)t * topk + i] = i < m ? sel[i] : -1;
    gap[t] = n > topk ? buf[topk - 1].v - buf[topk].v : INFINITY;
  }
  free(buf);
  free(sel);
  return 0;
}
