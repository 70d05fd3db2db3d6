/*
 * wfst_oracle.c — CPU reference decoder.  TEST INFRASTRUCTURE ONLY: loaded by
 * the test suite, the package smoke check and the benchmark's CPU-baseline
 * leg, never by the decoder itself.  It shares no code with the CUDA path.
 *
 * A plain, slow, single-threaded, frame-synchronous Viterbi token-passing
 * decoder that restates, one step at a time, the rules of the page
 * "GPU WFST Beam-Search Decoder" (OASR documentation, wfst_decoder_gpu):
 *
 *   §1 Purpose: every frame relaxes each emitting arc leaving a frontier
 *      token, with end = score[src] + arc_weight + log_prob[t][ilabel]; each
 *      destination state keeps its best incoming candidate; the result is
 *      backtracked to words.
 *   §3 Decoding Semantics: the dynamic-beam update (relax / widen / tighten,
 *      the last-frames min_active rule), admission end > exact_max - b with
 *      the exact per-step maximum, the final step, allow_partial, output_beam
 *      applied only by the lattice backward prune, and the online (streaming)
 *      beam semantics in which the offline-only clauses never fire.
 *   §5.3 (upper-bound paragraph): the association (s + w) + lp of every end.
 *   §5.5: epsilon closure on graphs with epsilon arcs; lattice persistence of
 *      every in-beam candidate after the closure.
 *   §7: 1-best backtrack from the final token, arcs in forward order, words =
 *      the non-zero output labels; lattice records.
 *
 * Readings where the page is open (each also listed in the design notes):
 *   - ties: exact-score ties pick the LOWEST arc id (the page leaves them to
 *     atomic scheduling); final-state ties pick the lowest state; the start
 *     token (arc -1) is the lowest of all.
 *   - "last ~5 frames": the rule applies at steps t >= T - 5, with the
 *     integer max_active / 2.
 *   - the beam update uses the current frontier size, before this step's
 *     cutoff; relax on the closed interval [min_active, max_active] or an
 *     empty frontier.  Its constants follow the page's text and are pinned to
 *     hand-derived values of that text; against k2's own implementation,
 *     which is not available here: parity unpinned.  All arithmetic is IEEE fp32, round to nearest, no
 *     fused multiply-add (compile with -ffp-contract=off).
 *   - epsilon closure: a full closure in epsilon-topological order (ties by
 *     lower state id), each relaxation admitted iff e > the emitting step's
 *     cutoff; the start frontier uses cutoff 0 - search_beam.
 *   - final weights are per-state; the final step is a virtual arc A + s.
 *     Without any final state and with allow_partial, the best frontier token
 *     (score unchanged) is the result; otherwise ok = 0.
 *   - lattice: nodes are (frame, state) tokens plus one super-final node;
 *     backward scores bwd[super] = 0, bwd[node] = max over its records of
 *     (arcscore + bwd[dst]) in reverse frame order (epsilon records of one
 *     frame in reverse epsilon-topological order); a record is kept iff
 *     end + bwd[dst] >= best - output_beam.
 *   - interval lattice prune (§7 lat_prune_interval: every N frames a loose
 *     prune over a window of recent frames, the final prune staying exact).
 *     The page does not say which records it may drop; here it drops only
 *     records the final prune can never keep.  After the step that makes
 *     frame t (a positive multiple of N) the frontier, every frontier token
 *     u gets beta(u) = -score(u); beta flows backward over the records of
 *     the groups R_r = emit(r) + eps(r + 1), r in [max(-1, t - 2N), t - 1]
 *     as bwd does (beta(src) = max over its records of arcscore +
 *     beta(dst)).  A record of the window stays iff beta(dst) > -inf and
 *     end + beta(dst) >= -((output_beam + 1) + 2^-12 |M|), M being the
 *     exact max of the step that made frame t.  Every complete path passes
 *     through one token u of frame t and its prefix score up to u is at most
 *     score(u), so end + beta(dst) is minus the least amount by which a path
 *     through the record falls behind the best path into its frontier
 *     token; the final prune keeps a record only if some path through it is
 *     within output_beam of the best complete path, which passes through
 *     the frontier too, so only records with end + beta(dst) >= -output_beam
 *     can be kept.  The margin 1 + 2^-12 |M| covers fp32 rounding of the
 *     sums (|M| grows with the utterance).
 */
#include "wfst_oracle.h"

#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* small helpers                                                       */
/* ------------------------------------------------------------------ */

static int grow(void** p, int64_t* cap, int64_t need, size_t elem) {
  if (need <= *cap) return 0;
  int64_t nc = *cap ? *cap : 1024;
  while (nc < need) nc *= 2;
  void* q = realloc(*p, (size_t)nc * elem);
  if (!q) return -1;
  *p = q;
  *cap = nc;
  return 0;
}

/* binary min-heap of state ids ordered by key[state] (key NULL: by id) */
typedef struct {
  int32_t* a;
  int64_t n, cap;
  const int32_t* key;
} heap_t;

static int32_t hkey(const heap_t* h, int32_t s) { return h->key ? h->key[s] : s; }

static int heap_push(heap_t* h, int32_t s) {
  if (grow((void**)&h->a, &h->cap, h->n + 1, sizeof(int32_t))) return -1;
  int64_t i = h->n++;
  h->a[i] = s;
  while (i > 0) {
    int64_t p = (i - 1) / 2;
    if (hkey(h, h->a[p]) <= hkey(h, h->a[i])) break;
    int32_t t = h->a[p];
    h->a[p] = h->a[i];
    h->a[i] = t;
    i = p;
  }
  return 0;
}

static int32_t heap_pop(heap_t* h) {
  int32_t top = h->a[0];
  h->a[0] = h->a[--h->n];
  int64_t i = 0;
  for (;;) {
    int64_t l = 2 * i + 1, r = l + 1, m = i;
    if (l < h->n && hkey(h, h->a[l]) < hkey(h, h->a[m])) m = l;
    if (r < h->n && hkey(h, h->a[r]) < hkey(h, h->a[m])) m = r;
    if (m == i) break;
    int32_t t = h->a[m];
    h->a[m] = h->a[i];
    h->a[i] = t;
    i = m;
  }
  return top;
}

/* ------------------------------------------------------------------ */
/* graph                                                               */
/* ------------------------------------------------------------------ */

struct or_graph {
  int32_t N, start, V;
  int64_t A;
  int64_t* rs;
  int32_t* il;
  int32_t* ol;
  float* w;
  int32_t* dst;
  float* fin;
  int32_t* eps_rank;  /* position of each state in an epsilon-topological order */
  int32_t* eps_count; /* epsilon out-arcs per state */
  int has_eps;
};

void or_graph_free(or_graph* g) {
  if (!g) return;
  free(g->rs);
  free(g->il);
  free(g->ol);
  free(g->w);
  free(g->dst);
  free(g->fin);
  free(g->eps_rank);
  free(g->eps_count);
  free(g);
}

#define FAIL(...)                                  \
  do {                                             \
    if (err && errlen > 0) snprintf(err, (size_t)errlen, __VA_ARGS__); \
    or_graph_free(g);                              \
    return NULL;                                   \
  } while (0)

or_graph* or_graph_new(const or_graph_desc* d, char* err, int32_t errlen) {
  or_graph* g = (or_graph*)calloc(1, sizeof(or_graph));
  if (!g) return NULL;
  if (!d || d->num_states <= 0) FAIL("num_states must be positive");
  const int32_t N = d->num_states;
  const int64_t A = d->num_arcs;
  if (d->start_state < 0 || d->start_state >= N) FAIL("start state out of range");
  if (d->vocab_size <= 0) FAIL("vocab_size must be positive");
  if (A < 0 || A + (int64_t)N >= 2147483647LL) FAIL("arc count out of range");
  if (d->row_splits[0] != 0 || d->row_splits[N] != A) FAIL("row_splits must run from 0 to num_arcs");
  for (int32_t s = 0; s < N; s++)
    if (d->row_splits[s + 1] < d->row_splits[s]) FAIL("row_splits not monotone at state %d", s);
  for (int64_t a = 0; a < A; a++) {
    if (d->dst[a] < 0 || d->dst[a] >= N) FAIL("arc %lld: destination out of range", (long long)a);
    if (d->ilabel[a] < -1 || d->ilabel[a] >= d->vocab_size)
      FAIL("arc %lld: ilabel out of range", (long long)a);
  }
  g->N = N;
  g->start = d->start_state;
  g->V = d->vocab_size;
  g->A = A;
  g->rs = (int64_t*)malloc(sizeof(int64_t) * (size_t)(N + 1));
  g->il = (int32_t*)malloc(sizeof(int32_t) * (size_t)(A ? A : 1));
  g->ol = (int32_t*)malloc(sizeof(int32_t) * (size_t)(A ? A : 1));
  g->w = (float*)malloc(sizeof(float) * (size_t)(A ? A : 1));
  g->dst = (int32_t*)malloc(sizeof(int32_t) * (size_t)(A ? A : 1));
  g->fin = (float*)malloc(sizeof(float) * (size_t)N);
  g->eps_rank = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  g->eps_count = (int32_t*)calloc((size_t)N, sizeof(int32_t));
  if (!g->rs || !g->il || !g->ol || !g->w || !g->dst || !g->fin || !g->eps_rank || !g->eps_count)
    FAIL("out of memory");
  memcpy(g->rs, d->row_splits, sizeof(int64_t) * (size_t)(N + 1));
  if (A) {
    memcpy(g->il, d->ilabel, sizeof(int32_t) * (size_t)A);
    memcpy(g->ol, d->olabel, sizeof(int32_t) * (size_t)A);
    memcpy(g->w, d->weight, sizeof(float) * (size_t)A);
    memcpy(g->dst, d->dst, sizeof(int32_t) * (size_t)A);
  }
  memcpy(g->fin, d->final_weight, sizeof(float) * (size_t)N);

  /* epsilon-topological order (Kahn; among ready states the lowest id first).
   * Every state gets a rank; a state left unranked lies on an epsilon cycle. */
  int32_t* indeg = (int32_t*)calloc((size_t)N, sizeof(int32_t));
  if (!indeg) FAIL("out of memory");
  for (int32_t s = 0; s < N; s++)
    for (int64_t a = g->rs[s]; a < g->rs[s + 1]; a++)
      if (g->il[a] < 0) {
        indeg[g->dst[a]]++;
        g->eps_count[s]++;
        g->has_eps = 1;
      }
  heap_t h = {0};
  for (int32_t s = 0; s < N; s++)
    if (indeg[s] == 0 && heap_push(&h, s)) {
      free(indeg);
      free(h.a);
      FAIL("out of memory");
    }
  int32_t rank = 0;
  while (h.n > 0) {
    int32_t s = heap_pop(&h);
    g->eps_rank[s] = rank++;
    for (int64_t a = g->rs[s]; a < g->rs[s + 1]; a++)
      if (g->il[a] < 0 && --indeg[g->dst[a]] == 0) heap_push(&h, g->dst[a]);
  }
  free(indeg);
  free(h.a);
  if (rank != N) FAIL("epsilon arcs form a cycle");
  return g;
}

int32_t or_graph_eps_rank(const or_graph* g, int32_t* out) {
  memcpy(out, g->eps_rank, sizeof(int32_t) * (size_t)g->N);
  return g->has_eps;
}

/* ------------------------------------------------------------------ */
/* decoder                                                             */
/* ------------------------------------------------------------------ */

typedef struct {
  int32_t state; /* graph state */
  float score;   /* forward (Viterbi) score */
  int32_t arc;   /* arc id of the winning incoming arc, -1 for the start */
  int32_t prev;  /* token the arc leaves from, -1 for the start */
} tok_t;

typedef struct {
  int32_t src_tok, arc;
  float end, arcscore;
} cand_t;

typedef struct {
  int32_t frame;     /* frame of the source node */
  int32_t src_tok;
  int32_t arc;       /* arc id; A + s for final / redirect records */
  int32_t dst_tok;   /* -1: super-final node */
  int32_t dst_state; /* -1: super-final node */
  int32_t flags;     /* OR_REC_*; REC_DROPPED: removed by an interval prune */
  float end;         /* forward value of the candidate */
  float arcscore;    /* the record's own score */
} rec_t;

#define REC_DROPPED 64

struct or_dec {
  const or_graph* g;
  or_params p;
  int32_t t_eff;
  tok_t* tok;
  int64_t ntok, cap_tok;
  int64_t fb; /* first token of the current frame */
  int64_t* fbase; /* first token of each frame 0..t */
  int64_t cap_fbase;
  int32_t t;  /* frames consumed */
  float beam;
  int finalized;
  int32_t* where;   /* state -> token of the current frame, or -1 */
  uint8_t* in_heap; /* closure queue membership */
  heap_t heap;
  cand_t* cand;
  int64_t ncand, cap_cand;
  rec_t* rec;
  int64_t nrec, cap_rec;
  uint8_t* keep;
  or_step* trace;
  int64_t ntrace, cap_trace;
  int64_t st[OR_ST_COUNT];
  int ok;
  float best_score;
};

void or_dec_free(or_dec* d) {
  if (!d) return;
  free(d->tok);
  free(d->where);
  free(d->in_heap);
  free(d->heap.a);
  free(d->cand);
  free(d->rec);
  free(d->keep);
  free(d->trace);
  free(d->fbase);
  free(d);
}

static int64_t new_tok(or_dec* d, int32_t state, float score, int32_t arc, int64_t prev) {
  if (grow((void**)&d->tok, &d->cap_tok, d->ntok + 1, sizeof(tok_t))) return -1;
  tok_t* k = &d->tok[d->ntok];
  k->state = state;
  k->score = score;
  k->arc = arc;
  k->prev = (int32_t)prev;
  d->where[state] = (int32_t)d->ntok;
  return d->ntok++;
}

static int add_rec(or_dec* d, int32_t frame, int64_t src_tok, int32_t arc, int32_t dst_tok,
                   int32_t dst_state, int32_t flags, float end, float arcscore) {
  if (!d->p.lattice) return 0;
  if (grow((void**)&d->rec, &d->cap_rec, d->nrec + 1, sizeof(rec_t))) return -1;
  rec_t* r = &d->rec[d->nrec++];
  r->frame = frame;
  r->src_tok = (int32_t)src_tok;
  r->arc = arc;
  r->dst_tok = dst_tok;
  r->dst_state = dst_state;
  r->flags = flags;
  r->end = end;
  r->arcscore = arcscore;
  return 0;
}

/* Epsilon closure of the current frame against `cutoff` (§5.5).  States are
 * visited in epsilon-topological order, so a state's score is final when its
 * epsilon arcs are relaxed. */
static int closure(or_dec* d, float cutoff) {
  const or_graph* g = d->g;
  heap_t* h = &d->heap;
  h->n = 0;
  h->key = g->eps_rank;
  for (int64_t i = d->fb; i < d->ntok; i++) {
    int32_t s = d->tok[i].state;
    if (g->eps_count[s] > 0 && !d->in_heap[s]) {
      if (heap_push(h, s)) return OR_ENOMEM;
      d->in_heap[s] = 1;
    }
  }
  while (h->n > 0) {
    int32_t u = heap_pop(h);
    d->in_heap[u] = 0;
    int64_t ui = d->where[u];
    float su = d->tok[ui].score;
    for (int64_t a = g->rs[u]; a < g->rs[u + 1]; a++) {
      if (g->il[a] >= 0) continue;
      float e = su + g->w[a];
      d->st[OR_ST_EPS_RELAXED]++;
      d->st[OR_ST_ARCS_EXPANDED]++;
      if (!(e > cutoff)) continue;
      int32_t v = g->dst[a];
      int64_t vi = d->where[v];
      if (vi < 0) {
        vi = new_tok(d, v, e, (int32_t)a, ui);
        if (vi < 0) return OR_ENOMEM;
        if (g->eps_count[v] > 0 && !d->in_heap[v]) {
          if (heap_push(h, v)) return OR_ENOMEM;
          d->in_heap[v] = 1;
        }
      } else {
        tok_t* k = &d->tok[vi];
        if (e > k->score || (e == k->score && a < k->arc)) {
          k->score = e;
          k->arc = (int32_t)a;
          k->prev = (int32_t)ui;
        }
      }
      if (add_rec(d, d->t, ui, (int32_t)a, d->where[v], v, OR_REC_EPS, e, g->w[a])) return OR_ENOMEM;
    }
  }
  return OR_OK;
}

or_dec* or_dec_new(const or_graph* g, const or_params* p, int32_t t_eff) {
  or_dec* d = (or_dec*)calloc(1, sizeof(or_dec));
  if (!d) return NULL;
  d->g = g;
  d->p = *p;
  d->t_eff = t_eff;
  d->where = (int32_t*)malloc(sizeof(int32_t) * (size_t)g->N);
  d->in_heap = (uint8_t*)calloc((size_t)g->N, 1);
  if (!d->where || !d->in_heap) {
    or_dec_free(d);
    return NULL;
  }
  for (int32_t s = 0; s < g->N; s++) d->where[s] = -1;
  d->beam = p->search_beam;
  /* the start frontier: one token, score 0, no arc */
  if (new_tok(d, g->start, 0.0f, -1, -1) < 0) {
    or_dec_free(d);
    return NULL;
  }
  d->fb = 0;
  if (grow((void**)&d->fbase, &d->cap_fbase, 1, sizeof(int64_t))) {
    or_dec_free(d);
    return NULL;
  }
  d->fbase[0] = 0;
  if (g->has_eps) {
    float cutoff0 = 0.0f - p->search_beam;
    if (closure(d, cutoff0) != OR_OK) {
      or_dec_free(d);
      return NULL;
    }
  }
  return d;
}

static int interval_prune(or_dec* d, float M);

/* One emitting step: consume the log-prob row `lp` (frame d->t). */
static int step(or_dec* d, const float* lp) {
  const or_graph* g = d->g;
  const int64_t n = d->ntok - d->fb;

  /* dynamic beam (§3) */
  int32_t min_a = d->p.min_active;
  if (d->t_eff >= 0 && d->t >= d->t_eff - 5) {
    int32_t half = d->p.max_active / 2;
    if (half > min_a) min_a = half;
  }
  const float sb = d->p.search_beam;
  float b = d->beam;
  if (n == 0 || (min_a <= n && n <= d->p.max_active)) {
    float x = 0.8f * b;
    float y = 0.2f * sb;
    b = x + y;
  } else if (n < min_a) {
    float m = b > sb ? b : sb;
    b = m * 1.25f;
  } else {
    float m = b < sb ? b : sb;
    b = m * 0.8f;
  }
  d->beam = b;

  /* every emitting out-arc of every frontier token, and their exact max */
  d->ncand = 0;
  float max_end = -INFINITY;
  for (int64_t i = d->fb; i < d->ntok; i++) {
    const int32_t s = d->tok[i].state;
    const float sc = d->tok[i].score;
    for (int64_t a = g->rs[s]; a < g->rs[s + 1]; a++) {
      const int32_t il = g->il[a];
      if (il < 0) continue;
      const float lpv = lp[il];
      const float partial = sc + g->w[a];
      const float end = partial + lpv;
      if (grow((void**)&d->cand, &d->cap_cand, d->ncand + 1, sizeof(cand_t))) return OR_ENOMEM;
      cand_t* c = &d->cand[d->ncand++];
      c->src_tok = (int32_t)i;
      c->arc = (int32_t)a;
      c->end = end;
      c->arcscore = g->w[a] + lpv;
      if (d->ncand == 1 || end > max_end) max_end = end;
    }
  }

  or_step tr;
  memset(&tr, 0, sizeof(tr));
  tr.t = d->t;
  tr.n = (int32_t)n;
  tr.num_cands = (int32_t)d->ncand;
  tr.beam = b;
  tr.max_end = max_end;

  /* the old frame's state map is no longer needed */
  for (int64_t i = d->fb; i < d->ntok; i++) d->where[d->tok[i].state] = -1;
  const int64_t nb = d->ntok;
  const int64_t rec0 = d->nrec;
  int64_t admitted = 0;
  float cutoff = -INFINITY;

  if (d->ncand > 0) {
    cutoff = max_end - b;
    for (int64_t k = 0; k < d->ncand; k++) {
      const cand_t c = d->cand[k];
      if (!(c.end > cutoff)) continue;
      admitted++;
      const int32_t v = g->dst[c.arc];
      int64_t vi = d->where[v];
      if (vi < 0) {
        if (new_tok(d, v, c.end, c.arc, c.src_tok) < 0) return OR_ENOMEM;
      } else {
        tok_t* tk = &d->tok[vi];
        if (c.end > tk->score || (c.end == tk->score && c.arc < tk->arc)) {
          tk->score = c.end;
          tk->arc = c.arc;
          tk->prev = c.src_tok;
        }
      }
      if (add_rec(d, d->t, c.src_tok, c.arc, -1, v, 0, c.end, c.arcscore)) return OR_ENOMEM;
    }
  }
  d->fb = nb;
  d->t++;
  if (grow((void**)&d->fbase, &d->cap_fbase, d->t + 1, sizeof(int64_t))) return OR_ENOMEM;
  d->fbase[d->t] = nb;
  if (d->ncand > 0 && g->has_eps) {
    int rc = closure(d, cutoff);
    if (rc != OR_OK) return rc;
  }
  /* emitting records of this step point at the destination's token in the
   * new frame (after its closure) */
  for (int64_t r = rec0; r < d->nrec; r++)
    if (!(d->rec[r].flags & OR_REC_EPS)) d->rec[r].dst_tok = d->where[d->rec[r].dst_state];

  const int64_t m = d->ntok - d->fb;
  tr.cutoff = cutoff;
  tr.num_admitted = (int32_t)admitted;
  tr.next_size = (int32_t)m;
  if (grow((void**)&d->trace, &d->cap_trace, d->ntrace + 1, sizeof(or_step))) return OR_ENOMEM;
  d->trace[d->ntrace++] = tr;

  if (d->p.lattice && d->p.lat_prune_interval > 0 && d->t % d->p.lat_prune_interval == 0) {
    int rc = interval_prune(d, max_end);
    if (rc != OR_OK) return rc;
  }

  d->st[OR_ST_FRAMES]++;
  d->st[OR_ST_ARCS_EXPANDED] += d->ncand;
  d->st[OR_ST_SUM_N] += n;
  d->st[OR_ST_SUM_D] += d->ncand;
  d->st[OR_ST_SUM_A] += admitted;
  d->st[OR_ST_SUM_M] += m;
  if (n > d->st[OR_ST_MAX_N]) d->st[OR_ST_MAX_N] = n;
  if (d->ncand > d->st[OR_ST_MAX_D]) d->st[OR_ST_MAX_D] = d->ncand;
  return OR_OK;
}

int32_t or_dec_advance(or_dec* d, const float* lp, int64_t stride_t, int32_t nframes) {
  if (!d || d->finalized || nframes < 0) return OR_EINVAL;
  for (int32_t r = 0; r < nframes; r++) {
    int rc = step(d, lp + (int64_t)r * stride_t);
    if (rc != OR_OK) return rc;
  }
  return OR_OK;
}

/* best token of the current frame by (score, then lowest arc id) */
static int64_t best_token(const or_dec* d) {
  int64_t best = -1;
  for (int64_t i = d->fb; i < d->ntok; i++) {
    const tok_t* k = &d->tok[i];
    if (best < 0 || k->score > d->tok[best].score ||
        (k->score == d->tok[best].score && k->arc < d->tok[best].arc))
      best = i;
  }
  return best;
}

/* arcs of the path ending in token `i`, forward order; returns the length */
static int64_t backtrack(const or_dec* d, int64_t i, int32_t* arcs, int64_t cap) {
  int64_t len = 0;
  for (int64_t k = i; k >= 0 && d->tok[k].arc >= 0; k = d->tok[k].prev) len++;
  int64_t pos = len;
  for (int64_t k = i; k >= 0 && d->tok[k].arc >= 0; k = d->tok[k].prev) {
    --pos;
    if (pos < cap) arcs[pos] = d->tok[k].arc;
  }
  return len;
}

static int32_t words_of(const or_dec* d, int64_t tok, int32_t* words, int32_t cap) {
  int32_t nw = 0;
  for (int64_t k = tok; k >= 0 && d->tok[k].arc >= 0; k = d->tok[k].prev)
    if (d->g->ol[d->tok[k].arc] != 0) nw++;
  int32_t pos = nw;
  for (int64_t k = tok; k >= 0 && d->tok[k].arc >= 0; k = d->tok[k].prev) {
    int32_t o = d->g->ol[d->tok[k].arc];
    if (o != 0) {
      --pos;
      if (pos < cap) words[pos] = o;
    }
  }
  return nw;
}

int32_t or_dec_partial(or_dec* d, int32_t* words, int32_t words_cap, int32_t* n_words, float* score,
                       int32_t* ok) {
  if (!d || d->finalized) return OR_EINVAL;
  int64_t best = best_token(d);
  if (best < 0) {
    *ok = 0;
    *n_words = 0;
    *score = -INFINITY;
    return OR_OK;
  }
  *ok = 1;
  *score = d->tok[best].score;
  *n_words = words_of(d, best, words, words_cap);
  return OR_OK;
}

typedef struct {
  int64_t r;
  int32_t frame, cls, rank;
} ord_t;

static int ord_cmp(const void* a, const void* b) {
  const ord_t* x = (const ord_t*)a;
  const ord_t* y = (const ord_t*)b;
  if (x->frame != y->frame) return x->frame > y->frame ? -1 : 1; /* later frames first */
  if (x->cls != y->cls) return x->cls < y->cls ? -1 : 1;         /* non-epsilon first */
  if (x->rank != y->rank) return x->rank > y->rank ? -1 : 1;     /* reverse topological */
  return x->r < y->r ? -1 : (x->r > y->r);
}

/* Interval lattice prune after the step that made frame d->t the frontier
 * (§7 lat_prune_interval; the reading in this file's header): beta over the
 * window's records backward from the frontier, in the final prune's order,
 * then the window's records that no complete path within output_beam of
 * the best can use are marked dropped.  M: the exact max of that step. */
static int interval_prune(or_dec* d, float M) {
  const or_graph* g = d->g;
  const int32_t t = d->t, N = d->p.lat_prune_interval;
  const int32_t r0 = t - 2 * N < -1 ? -1 : t - 2 * N;  /* oldest group of the window */
  const int64_t tok0 = d->fbase[r0 < 0 ? 0 : r0];      /* first token of the window's nodes */
  const int64_t nt = d->ntok - tok0;
  float* beta = (float*)malloc(sizeof(float) * (size_t)(nt ? nt : 1));
  ord_t* ord = (ord_t*)malloc(sizeof(ord_t) * (size_t)(d->nrec ? d->nrec : 1));
  if (!beta || !ord) {
    free(beta);
    free(ord);
    return OR_ENOMEM;
  }
  for (int64_t i = 0; i < nt; i++) beta[i] = -INFINITY;
  for (int64_t i = d->fb; i < d->ntok; i++) beta[i - tok0] = -d->tok[i].score;
  /* the window: emitting records of frames r0..t-1, epsilon records of
   * frames r0+1..t (group R_r holds emit(r) and eps(r + 1)) */
  int64_t nord = 0;
  for (int64_t r = 0; r < d->nrec; r++) {
    const rec_t* x = &d->rec[r];
    if (x->flags & REC_DROPPED) continue;
    const int eps = (x->flags & OR_REC_EPS) != 0;
    const int32_t grp = eps ? x->frame - 1 : x->frame;
    if (grp < r0 || grp > t - 1) continue;
    ord[nord].r = r;
    ord[nord].frame = x->frame;
    ord[nord].cls = eps;
    ord[nord].rank = eps ? g->eps_rank[d->tok[x->src_tok].state] : 0;
    nord++;
  }
  qsort(ord, (size_t)nord, sizeof(ord_t), ord_cmp);
  for (int64_t k = 0; k < nord; k++) {
    const rec_t* x = &d->rec[ord[k].r];
    const float v = x->arcscore + beta[x->dst_tok - tok0];
    if (v > beta[x->src_tok - tok0]) beta[x->src_tok - tok0] = v;
  }
  const float margin = 0x1p-12f * fabsf(M);
  const float room = d->p.output_beam + 1.0f;
  const float lim = -(room + margin);
  for (int64_t k = 0; k < nord; k++) {
    rec_t* x = &d->rec[ord[k].r];
    const float bd = beta[x->dst_tok - tok0];
    const float tot = x->end + bd;
    if (!(bd > -INFINITY && tot >= lim)) {
      x->flags |= REC_DROPPED;
      d->st[OR_ST_DROPPED]++;
    }
  }
  free(beta);
  free(ord);
  return OR_OK;
}

/* backward output_beam prune over the persisted records (§3, §7) */
static int prune_lattice(or_dec* d) {
  const or_graph* g = d->g;
  d->keep = (uint8_t*)calloc((size_t)(d->nrec ? d->nrec : 1), 1);
  float* bwd = (float*)malloc(sizeof(float) * (size_t)(d->ntok ? d->ntok : 1));
  ord_t* ord = (ord_t*)malloc(sizeof(ord_t) * (size_t)(d->nrec ? d->nrec : 1));
  if (!d->keep || !bwd || !ord) {
    free(bwd);
    free(ord);
    return OR_ENOMEM;
  }
  for (int64_t i = 0; i < d->ntok; i++) bwd[i] = -INFINITY;
  int64_t nord = 0;
  for (int64_t r = 0; r < d->nrec; r++) {
    if (d->rec[r].flags & REC_DROPPED) continue;
    ord[nord].r = r;
    ord[nord].frame = d->rec[r].frame;
    ord[nord].cls = (d->rec[r].flags & OR_REC_EPS) ? 1 : 0;
    ord[nord].rank = (d->rec[r].flags & OR_REC_EPS) ? g->eps_rank[d->tok[d->rec[r].src_tok].state] : 0;
    nord++;
  }
  qsort(ord, (size_t)nord, sizeof(ord_t), ord_cmp);
  for (int64_t k = 0; k < nord; k++) {
    const rec_t* r = &d->rec[ord[k].r];
    const float bd = r->dst_tok < 0 ? 0.0f : bwd[r->dst_tok];
    const float v = r->arcscore + bd;
    if (v > bwd[r->src_tok]) bwd[r->src_tok] = v;
  }
  const float thr = d->best_score - d->p.output_beam;
  for (int64_t r = 0; r < d->nrec; r++) {
    const rec_t* x = &d->rec[r];
    if (x->flags & REC_DROPPED) continue;
    const float bd = x->dst_tok < 0 ? 0.0f : bwd[x->dst_tok];
    const float tot = x->end + bd;
    d->keep[r] = (uint8_t)(tot >= thr);
  }
  free(bwd);
  free(ord);
  return OR_OK;
}

int32_t or_dec_finalize(or_dec* d, int32_t* words, int32_t words_cap, int32_t* n_words, int32_t* arcs,
                        int32_t arcs_cap, int32_t* n_arcs, float* score, int32_t* reached_final,
                        int32_t* ok) {
  if (!d || d->finalized) return OR_EINVAL;
  const or_graph* g = d->g;
  d->finalized = 1;
  /* final step (§3): only final weights, no acoustic term, no pruning */
  int64_t best = -1;
  float best_fe = -INFINITY;
  for (int64_t i = d->fb; i < d->ntok; i++) {
    const int32_t s = d->tok[i].state;
    const float f = g->fin[s];
    if (!(f > -INFINITY)) continue;
    const float fe = d->tok[i].score + f;
    d->st[OR_ST_FINALS]++;
    d->st[OR_ST_ARCS_EXPANDED]++;
    if (best < 0 || fe > best_fe || (fe == best_fe && s < d->tok[best].state)) {
      best = i;
      best_fe = fe;
    }
    if (add_rec(d, d->t, i, (int32_t)(g->A + s), -1, -1, OR_REC_FINAL, fe, f)) return OR_ENOMEM;
  }
  *reached_final = 0;
  if (best >= 0) {
    *reached_final = 1;
    *ok = 1;
    d->best_score = best_fe;
  } else if (d->p.allow_partial && (best = best_token(d)) >= 0) {
    *ok = 1;
    d->best_score = d->tok[best].score;
    if (add_rec(d, d->t, best, (int32_t)(g->A + d->tok[best].state), -1, -1, OR_REC_REDIRECT,
                d->best_score, 0.0f))
      return OR_ENOMEM;
  } else {
    *ok = 0;
    d->best_score = -INFINITY;
  }
  d->ok = *ok;
  *score = d->best_score;
  if (*ok) {
    *n_words = words_of(d, best, words, words_cap);
    *n_arcs = (int32_t)backtrack(d, best, arcs, arcs_cap);
  } else {
    *n_words = 0;
    *n_arcs = 0;
  }
  d->st[OR_ST_TOKENS] = d->ntok;
  d->st[OR_ST_RECORDS] = d->nrec;
  if (d->p.lattice && d->ok) return prune_lattice(d);
  return OR_OK;
}

static int lat_cmp(const void* a, const void* b) {
  const or_lat_record* x = (const or_lat_record*)a;
  const or_lat_record* y = (const or_lat_record*)b;
  if (x->t != y->t) return x->t < y->t ? -1 : 1;
  if (x->src_state != y->src_state) return x->src_state < y->src_state ? -1 : 1;
  if (x->arc_id != y->arc_id) return x->arc_id < y->arc_id ? -1 : 1;
  return 0;
}

static int64_t export_records(or_dec* d, or_lat_record* out, int64_t cap, int only_kept) {
  if (!d->finalized || !d->p.lattice) return 0;
  int64_t n = 0;
  for (int64_t r = 0; r < d->nrec; r++) {
    if (d->rec[r].flags & REC_DROPPED) continue;
    if (only_kept && !(d->ok && d->keep && d->keep[r])) continue;
    n++;
  }
  if (!out || cap < n) return n;
  int64_t k = 0;
  for (int64_t r = 0; r < d->nrec; r++) {
    if (d->rec[r].flags & REC_DROPPED) continue;
    if (only_kept && !(d->ok && d->keep && d->keep[r])) continue;
    const rec_t* x = &d->rec[r];
    or_lat_record* o = &out[k++];
    o->t = x->frame;
    o->src_state = d->tok[x->src_tok].state;
    o->dst_state = x->dst_tok < 0 ? -1 : d->tok[x->dst_tok].state;
    o->arc_id = x->arc;
    o->flags = x->flags;
    o->score = x->arcscore;
  }
  qsort(out, (size_t)n, sizeof(or_lat_record), lat_cmp);
  return n;
}

int64_t or_dec_lattice(or_dec* d, or_lat_record* out, int64_t cap) { return export_records(d, out, cap, 1); }

int64_t or_dec_lattice_all(or_dec* d, or_lat_record* out, int64_t cap) {
  return export_records(d, out, cap, 0);
}

void or_dec_stats(const or_dec* d, int64_t* out) {
  memcpy(out, d->st, sizeof(d->st));
  out[OR_ST_TOKENS] = d->ntok;
  out[OR_ST_RECORDS] = d->nrec;
}

int64_t or_dec_trace(const or_dec* d, or_step* out, int64_t cap) {
  int64_t n = d->ntrace < cap ? d->ntrace : cap;
  if (out && n > 0) memcpy(out, d->trace, sizeof(or_step) * (size_t)n);
  return d->ntrace;
}
