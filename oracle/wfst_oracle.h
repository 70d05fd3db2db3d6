/*
 * wfst_oracle.h — CPU reference decoder.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the package smoke check and the benchmark's CPU
 * baseline leg may load this library.  It shares no code with the CUDA
 * decoder.  See wfst_oracle.c for the rules it implements and where the page
 * "GPU WFST Beam-Search Decoder" states each of them.
 */
#ifndef WFST_ORACLE_H
#define WFST_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_ECORRUPT (-2)
#define OR_ENOMEM (-5)

/* record flags */
#define OR_REC_EPS 1
#define OR_REC_FINAL 2
#define OR_REC_REDIRECT 4

typedef struct {
  int32_t num_states, start_state, vocab_size, pad_;
  int64_t num_arcs;
  const int64_t* row_splits; /* [N+1] */
  const int32_t* ilabel;     /* [A] -1 epsilon, 0 blank, 1..V-1 */
  const int32_t* olabel;     /* [A] 0 = no word */
  const float* weight;       /* [A] */
  const int32_t* dst;        /* [A] */
  const float* final_weight; /* [N] -inf = not final */
} or_graph_desc;

typedef struct {
  float search_beam, output_beam;
  int32_t min_active, max_active;
  int32_t allow_partial;
  int32_t lattice;
  int32_t lat_prune_interval; /* interval lattice prune every N frames, 0 = off */
} or_params;

typedef struct {
  int32_t t, src_state, dst_state, arc_id, flags;
  float score;
} or_lat_record;

/* per-step trace entry */
typedef struct {
  int32_t t, n, num_cands, num_admitted, next_size, pad_;
  float beam, max_end, cutoff, pad2_;
} or_step;

/* counters (or_dec_stats) */
enum {
  OR_ST_FRAMES = 0, OR_ST_ARCS_EXPANDED, OR_ST_SUM_N, OR_ST_SUM_D, OR_ST_SUM_A,
  OR_ST_SUM_M, OR_ST_MAX_N, OR_ST_MAX_D, OR_ST_TOKENS, OR_ST_RECORDS,
  OR_ST_EPS_RELAXED, OR_ST_FINALS, OR_ST_DROPPED, OR_ST_COUNT
};

typedef struct or_graph or_graph;
typedef struct or_dec or_dec;

or_graph* or_graph_new(const or_graph_desc* d, char* err, int32_t errlen);
void or_graph_free(or_graph* g);
/* topological rank of each state in the epsilon subgraph (ties by lower id) */
int32_t or_graph_eps_rank(const or_graph* g, int32_t* out);

/* t_eff >= 0: offline decode of exactly t_eff frames (the last-frames
 * min_active rule applies); t_eff < 0: streaming (online) semantics. */
or_dec* or_dec_new(const or_graph* g, const or_params* p, int32_t t_eff);
void or_dec_free(or_dec* d);
/* consume nframes rows of fp32 log-probs, row r at lp + r*stride_t */
int32_t or_dec_advance(or_dec* d, const float* lp, int64_t stride_t, int32_t nframes);
/* best current token (no final weights), backtracked; stream continues */
int32_t or_dec_partial(or_dec* d, int32_t* words, int32_t words_cap, int32_t* n_words,
                       float* score, int32_t* ok);
/* final step + backtrack (+ lattice prune); ends the decode */
int32_t or_dec_finalize(or_dec* d, int32_t* words, int32_t words_cap, int32_t* n_words,
                        int32_t* arcs, int32_t arcs_cap, int32_t* n_arcs, float* score,
                        int32_t* reached_final, int32_t* ok);
/* kept lattice records after finalize, sorted by (t, src_state, arc_id) */
int64_t or_dec_lattice(or_dec* d, or_lat_record* out, int64_t cap);
/* every persisted record before pruning (same order), for invariant checks */
int64_t or_dec_lattice_all(or_dec* d, or_lat_record* out, int64_t cap);
void or_dec_stats(const or_dec* d, int64_t* out /* OR_ST_COUNT */);
int64_t or_dec_trace(const or_dec* d, or_step* out, int64_t cap);

#ifdef __cplusplus
}
#endif
#endif
