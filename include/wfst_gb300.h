/*
 * wfst_gb300.h — C ABI of the GB300 (sm_103a) WFST beam-search decoder for
 * CTC speech recognition.
 *
 * The decoder follows the page "GPU WFST Beam-Search Decoder" (OASR
 * documentation, wfst_decoder_gpu).  Section numbers below are that page's.
 * Inputs: a batch of CTC log-posterior matrices log_prob[B, T, V] and a
 * decoding graph (epsilon-free HLG style, or TLG style with epsilon arcs).
 * Outputs, per utterance: the best word sequence and its score, optionally an
 * output_beam-pruned lattice, and, in streaming mode, a partial hypothesis
 * per chunk.
 *
 * Conventions shared by every entry point
 *   - Return value: WFST_OK (0) on success, a negative WFST_ERR_* code
 *     otherwise; wfst_last_error() then holds a message (thread-local).
 *   - Device pointers are CUDA device addresses on the decoder's device; host
 *     pointers are plain (pageable or pinned) host memory.  "stream" is a
 *     cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - Calls on one decoder are serialised by an internal mutex (§10: one
 *     instance runs one call at a time); use one decoder per concurrent
 *     caller.
 *   - A lane whose capacity was exceeded is not an error: its meta[2]
 *     overflow bits are set (§7 "Overflow bits") and its result may be
 *     degraded.  Offline decodes grow the capacity and re-run such lanes
 *     themselves (see wfst_decode); streaming channels only report it.
 *   - Exact-score ties are broken by the LOWEST arc id (final-state ties by
 *     the lowest state), so results are deterministic and bit-exact with the
 *     CPU reference.  (§3 leaves ties to atomic scheduling.)
 */
#ifndef WFST_GB300_H
#define WFST_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define WFST_OK 0
#define WFST_ERR_INVALID_ARG (-1)   /* a bad pointer, size, stride, length or id   */
#define WFST_ERR_CORRUPT_GRAPH (-2) /* graph failed validation (§4 loader checks)  */
#define WFST_ERR_CUDA (-3)          /* a CUDA runtime call failed                  */
#define WFST_ERR_OOM (-4)           /* device or host allocation failed            */
#define WFST_ERR_CAPACITY (-5)      /* requested capacities exceed the int32 tables */
#define WFST_ERR_TIMEOUT (-6)       /* a bounded device-side wait gave up           */
#define WFST_ERR_STATE (-7)         /* call not valid in the object's current state */

/* ---- log-prob element types ------------------------------------------ */
#define WFST_F32 0
#define WFST_F16 1 /* widened exactly to fp32 inside (§11 "fp16") */

/* ---- per-lane overflow bits (meta[3*b + 2]; §7 "Overflow bits") ------- */
#define WFST_OVF_ARENA 4     /* winners log or lattice arena full            */
#define WFST_OVF_KEPT 16     /* surviving frontier larger than frontier_cap  */
#define WFST_OVF_PATH 32     /* best path longer than path_cap (oldest arcs lost),
                                or, with the winners-log GC, fin_cap words finalized */

/* ---- lattice record flags -------------------------------------------- */
#define WFST_REC_EPS 1
#define WFST_REC_FINAL 2
#define WFST_REC_REDIRECT 4

typedef struct wfst_graph wfst_graph;     /* opaque: device-resident graph, refcounted */
typedef struct wfst_decoder wfst_decoder; /* opaque: workspace + lanes + streaming channels */

/*
 * Graph description (host arrays, borrowed only for the duration of
 * wfst_graph_upload).  CSR by source state, arcs sorted by source; the arc
 * index a in [0, num_arcs) is the arc id used everywhere (results, ties,
 * lattice records) — the library never renumbers arcs (§4 "Identity arc
 * order").
 */
typedef struct {
  int32_t num_states;          /* N > 0 */
  int32_t start_state;         /* in [0, N) */
  int32_t vocab_size;          /* V in [1, 65535): ilabels are stored as u16 (§4) */
  int32_t reserved;
  int64_t num_arcs;            /* A >= 0, A + N < 2^31 */
  const int64_t* row_splits;   /* [N+1], row_splits[0] = 0, monotone, row_splits[N] = A */
  const int32_t* ilabel;       /* [A] -1 = epsilon (consumes no frame), 0 = blank, 1..V-1 */
  const int32_t* olabel;       /* [A] output word id, 0 = none */
  const float* weight;         /* [A] log-semiring score added on the arc (higher is better) */
  const int32_t* dst;          /* [A] in [0, N) */
  const float* final_weight;   /* [N] final score, -INFINITY = not final */
} wfst_graph_desc;

typedef struct {
  float search_beam;      /* k2 search beam (§3 "Dynamic beam") */
  float output_beam;      /* lattice backward prune only (§3) */
  int32_t min_active;     /* soft lower frontier target */
  int32_t max_active;     /* soft upper frontier target (beam decay only, never top-k) */
  int32_t allow_partial;  /* 1: without a final state, return the best frontier token */
  int32_t lattice;        /* 1: persist candidates for wfst_lattice_export */
  int32_t streaming;      /* 1: decoder serves wfst_stream_* (online beam semantics) */
  int32_t options;        /* WFST_OPT_* bits, 0 = defaults */
  int32_t gc_interval;    /* winners-log GC every gc_interval frames per lane, 0 = off (§6.3, §8.1) */
  int32_t lat_prune_interval; /* lattice = 1: interval lattice prune every N frames, 0 = off (§7) */
} wfst_params;

/*
 * Interval lattice prune (params.lat_prune_interval = N > 0, lattice = 1;
 * §7: every N frames a prune runs over a window of recent frames, the final
 * output_beam prune staying exact).  When frame t (a positive multiple of
 * N) is committed, the records of the groups R_r = emit(r) + eps(r + 1),
 * r in [max(-1, t - 2N), t - 1], are tested against frame t's frontier:
 * every frontier token u starts at beta(u) = -score(u), beta flows backward
 * over the window (beta(src) = max of arcscore + beta(dst)), and a record
 * stays iff beta(dst) > -inf and end + beta(dst) >= -((output_beam + 1) +
 * 2^-12 |M|), M the exact max of the step that made frame t.  Every complete
 * path passes one frontier token u with a prefix score of at most score(u),
 * so only records the final prune can never keep are dropped (the margin
 * covers fp32 rounding): the exported lattice is the same with or without
 * it, and the arena holds far fewer records on long audio.  Dropped records
 * are compacted out of the arena, group by group.
 */

/* Turn off the per-token upper-bound skips of the max and expand passes
 * (§5.3 "Upper-bound skip"; exact either way — for identity tests). */
#define WFST_OPT_NO_UB_SKIP 1
/* Report capacity overflows without growing (see wfst_decode). */
#define WFST_OPT_NO_GROW 4

/* Per-lane capacities; 0 in any field selects its default. */
typedef struct {
  int64_t frontier_cap;   /* tokens per lane per frame (default min(num_states, max(64Ki, 16*max_active))) */
  int64_t log_cap;        /* winners-log entries per lane (default (max_frames+2)*1.5*max_active, >= 1Mi) */
  int64_t lattice_cap;    /* lattice records per lane (default (max_frames+2)*max_active/2, >= 1Mi) */
  int64_t path_cap;       /* arcs of one best path (default 4*(max_frames+2)*(1 + epsilon depth);
                             with the GC, 4*max(max_frames+2, 1024)*(1 + epsilon depth)) */
  int64_t fin_cap;        /* GC only: finalized words per lane (default 65536) */
} wfst_capacity;

/*
 * Winners-log GC (params.gc_interval > 0; §6.3 "Winners-log GC for long-form
 * audio", §8.1 "Per-chunk GC").  Each lane's winners log becomes a ring of
 * log_cap entries (rounded down to a power of two, at most 2^29).  Every
 * gc_interval frames a round finds the lane's convergence point — the newest
 * entry that every chain from the current frontier passes through — moves
 * the words of the path up to it (the finalized prefix) into a per-lane list
 * of fin_cap words, cuts the chain there and frees the ring below it.  Words,
 * scores and flags are identical to a decode without GC; a lane only needs
 * ring space for the frames since its chains last converged, so a streaming
 * channel can run for any length.  If the chains do not converge within the
 * ring, the lane overflows (bit 4), as without GC.  Not with lattice = 1:
 * lattice records refer to winners-log entries of every frame.
 */

typedef struct {
  int32_t t;          /* frame of the source node (epsilon and final records: the frame they sit in) */
  int32_t src_state;
  int32_t dst_state;  /* -1 = super-final node */
  int32_t arc_id;     /* arc id; num_arcs + s for the final (or redirect) record of state s */
  int32_t flags;      /* WFST_REC_* */
  float score;        /* the record's own score: weight + log_prob, weight, or final weight */
} wfst_lat_record;

/*
 * Upload and validate a graph on `device` (§4 "Graph Image": every index the
 * decoder follows is checked — start state, monotone row_splits, arc
 * destinations, label ranges, acyclic epsilon subgraph, finite weights).
 * On success *out owns one reference.  Errors: INVALID_ARG (NULL pointers, a
 * negative device, or a device id at or above the visible device count; the
 * count is checked after the graph itself), CORRUPT_GRAPH (validation), CUDA
 * (no CUDA device), OOM.
 */
int wfst_graph_upload(const wfst_graph_desc* desc, int32_t device, wfst_graph** out);

/* out[0..7] = {num_states, num_arcs, vocab_size, start_state, has_epsilon,
 *              epsilon depth (longest epsilon path), device bytes, device} */
int wfst_graph_info(const wfst_graph* g, int64_t* out);

/* Drop the caller's reference; device arrays live on while a decoder holds
 * the graph (§10: a decoder co-owns its graph). */
void wfst_graph_free(wfst_graph* g);

/*
 * Create a decoder with max_lanes lanes (utterances decoded together, or
 * streaming channels) for frames up to max_frames per lane (offline: per
 * call; streaming: per channel when lattice is on).  caps may be NULL.
 * The workspace is set up here: fixed tables are allocated; the frontier,
 * winners-log and lattice tables reserve address space and commit device
 * memory for their initial capacities (§6.2 lazily committed regions).
 * Later calls commit more only when a capacity grows (an offline overflow,
 * or a streaming channel past half of its winners log or lattice arena),
 * plus a host-input staging buffer (see wfst_decode).
 * Errors: INVALID_ARG, CAPACITY (a table would exceed 2^31 entries), OOM,
 * CUDA (also when the device lacks virtual memory management).
 */
int wfst_decoder_create(wfst_graph* g, const wfst_params* params, int32_t max_lanes,
                        int32_t max_frames, const wfst_capacity* caps, wfst_decoder** out);
void wfst_decoder_free(wfst_decoder* d);

/*
 * Offline batched decode (§1, §3, §7).  log_probs: [B, T, V] elements of
 * `dtype`, element (b, t, v) at log_probs[b*stride_b + t*stride_t + v]
 * (unit stride over v, stride_t >= V).  It may be a device pointer (read in
 * place) or a host pointer (copied to device inside the call).  Entries are
 * log-posteriors: finite or -INFINITY (a label that cannot be emitted); NaN
 * and +INFINITY are outside the contract and not checked (the input is read
 * in place, once).  lens: host
 * [B], 0 <= lens[b] <= T.  Requires B <= max_lanes and a decoder created with
 * streaming = 0.  T above max_frames first grows the decoder's per-frame
 * tables to max(T, 2 * max_frames) (§6 frame-capacity doubling; the
 * best-path buffer grows with them while it has its default size), unless
 * the decoder was created with WFST_OPT_NO_GROW (then INVALID_ARG).
 * Outputs (host, caller-allocated): words [B*words_cap] (lane b's words at
 * b*words_cap, forward order), word_lens [B] (TRUE length, may exceed
 * words_cap: re-issue with a larger buffer), scores [B] (fp32 path score
 * widened), meta [B*3] = {ok, reached_final, overflow bits}.
 * Capacities grow on demand: lanes that overflow the winners log or lattice
 * arena (bit 4), the frontier capacity (bit 16) or the best-path buffer (bit
 * 32) have that capacity doubled (the workspace arrays are reallocated) and
 * are decoded again, up to 12 times per call; a lane keeps its overflow bits
 * only if the capacity is at its largest, memory runs out, or the decoder was
 * created with WFST_OPT_NO_GROW.  Decoding is idempotent, so the re-run
 * lanes give the results an unbounded decoder would give.
 * The call is stream-ordered on `stream` and returns after the results are
 * on the host.  Errors: INVALID_ARG, STATE (a streaming decoder), CAPACITY
 * (T too large for the frame tables), CUDA, TIMEOUT, OOM.
 */
int wfst_decode(wfst_decoder* d, const void* log_probs, int32_t dtype, int64_t stride_b,
                int64_t stride_t, const int32_t* lens, int32_t B, int32_t T, void* stream,
                int32_t* words, int32_t words_cap, int32_t* word_lens, double* scores,
                int32_t* meta);

/*
 * Lattice of one lane after wfst_decode or wfst_stream_finalize with
 * params.lattice = 1: every in-beam candidate (emitting, epsilon, final,
 * redirect) whose best complete path is within output_beam of the best path
 * (§3: output_beam acts only in this backward prune, never on the forward
 * search; §7).
 * Records are sorted by (t, src_state, arc_id) and each such triple occurs
 * once (an epsilon arc is one record per source token, evaluated with the
 * token's final score, however many closure passes relaxed it).
 * *n_records receives the true count; at most `cap` records are written.
 * Errors: INVALID_ARG, STATE.
 */
int wfst_lattice_export(wfst_decoder* d, int32_t lane, wfst_lat_record* out, int64_t cap,
                        int64_t* n_records);

/* ---- streaming (§8 "Streaming Lifecycle"); decoder created with streaming = 1 */

/* Claim a free channel (= lane) and open its start frontier; *channel = -1
 * (and WFST_OK) when every channel is busy.  Errors: INVALID_ARG, STATE (not
 * a streaming decoder), CUDA, TIMEOUT. */
int wfst_stream_create(wfst_decoder* d, int32_t* channel);

/*
 * Advance n channels by their next chunk: log_probs [n, chunk_T, V] (device
 * or host, strides as in wfst_decode), chunk_lens host [n] in [0, chunk_T].
 * Online beam semantics: the offline last-frames rule never fires (§3).
 * If want_partial, the outputs receive each channel's best current
 * hypothesis (§8: backtracked from the highest-scoring token of the
 * channel's current frontier), laid out as in wfst_decode (meta
 * reached_final is 0); otherwise they may be NULL.  Channels do not grow
 * their capacities mid-stream: an overflow is reported in meta (a caller can
 * restart the stream on a fresh channel, as the binding's StreamingSearch
 * does).  Errors: INVALID_ARG (channel ids out of range or repeated,
 * chunk_T > max_frames, lengths, strides, a lattice stream longer than
 * max_frames), STATE (not a streaming decoder, a channel not open), CUDA,
 * TIMEOUT.
 */
int wfst_stream_advance(wfst_decoder* d, const int32_t* channels, int32_t n,
                        const void* log_probs, int32_t dtype, int64_t stride_b, int64_t stride_t,
                        const int32_t* chunk_lens, int32_t chunk_T, int32_t want_partial,
                        void* stream, int32_t* words, int32_t words_cap, int32_t* word_lens,
                        double* scores, int32_t* meta);

/* Final step + backtrack (+ lattice prune) of n channels; outputs as in
 * wfst_decode.  The channels stay claimed until wfst_stream_release.
 * Errors: INVALID_ARG, STATE (not a streaming decoder, a channel not open),
 * CUDA, TIMEOUT. */
int wfst_stream_finalize(wfst_decoder* d, const int32_t* channels, int32_t n, void* stream,
                         int32_t* words, int32_t words_cap, int32_t* word_lens, double* scores,
                         int32_t* meta);

/* Return a channel to the pool (its lattice is discarded).  Errors:
 * INVALID_ARG (channel not in use), CUDA. */
int wfst_stream_release(wfst_decoder* d, int32_t channel);

/*
 * Counters of the last decode / stream call (host int64, n entries written,
 * at most WFST_STAT_COUNT): see WFST_STAT_* for the order.  Errors:
 * INVALID_ARG (NULL pointers, n < 0).
 */
#define WFST_STAT_FRAMES 0        /* frames consumed (sum over lanes) */
#define WFST_STAT_ARCS 1          /* arcs expanded: emitting + epsilon relaxations + final arcs */
#define WFST_STAT_SUM_N 2         /* sum over lane-steps of the frontier size */
#define WFST_STAT_SUM_D 3         /* sum of emitting arcs expanded */
#define WFST_STAT_SUM_A 4         /* sum of admitted emitting candidates */
#define WFST_STAT_SUM_M 5         /* sum of next-frontier sizes (after closure) */
#define WFST_STAT_EPS 6           /* epsilon arcs relaxed (once per closure token) */
#define WFST_STAT_STEPS 7         /* grid steps of the device loop */
#define WFST_STAT_BARRIERS 8      /* grid barriers executed */
#define WFST_STAT_KERNEL_NS 9     /* device time of the decode kernel (ns) */
#define WFST_STAT_NS_INIT 10      /* device time in lane initialisation + start closure */
#define WFST_STAT_NS_MAX 11       /* ... in the commit + exact-max phases */
#define WFST_STAT_NS_EXPAND 12    /* ... in the admission/recombination + final-step phases */
#define WFST_STAT_NS_CLOSURE 13   /* ... in epsilon-closure passes */
#define WFST_STAT_NS_PRUNE 14     /* ... in the lattice backward prune */
/* CTA 0's own timeline inside a frame step (ns): prologue, commit, clear,
 * max tiles, wait at the first barrier, expand tiles, final-step tasks, wait
 * at the second barrier */
#define WFST_STAT_NS_PROLOGUE 15
#define WFST_STAT_LAT_HELD 23     /* lattice records held in the arenas of the call's lanes at its end */
#define WFST_STAT_EPS_PASSES 24   /* epsilon-closure worklist passes (each ends at a grid barrier) */
#define WFST_STAT_LOG_HW 25       /* most winners-log entries any lane held live during the call */
#define WFST_STAT_COUNT 26
int wfst_stats(wfst_decoder* d, int64_t* out, int32_t n);

/*
 * Workspace of a decoder (host int64, n entries written, at most
 * WFST_MEM_COUNT): device bytes held, then the current per-lane capacities
 * (frontier tokens, winners-log entries, lattice records, best-path arcs) and
 * the number of capacity doublings so far, then max_frames (which offline
 * decodes of longer utterances raise), then the address space reserved for
 * the lazily committed tables and the device memory committed to them.
 * §6.2 of the page reports the decoder's memory the same way: the frontier,
 * winners-log and lattice tables reserve worst-case address ranges and
 * commit physical memory only for their current capacities.
 * Errors: INVALID_ARG (NULL pointers, n < 0).
 */
#define WFST_MEM_BYTES 0
#define WFST_MEM_FRONTIER_CAP 1
#define WFST_MEM_LOG_CAP 2
#define WFST_MEM_LATTICE_CAP 3
#define WFST_MEM_PATH_CAP 4
#define WFST_MEM_GROWS 5
#define WFST_MEM_MAX_FRAMES 6    /* frames per call the per-frame tables hold now */
#define WFST_MEM_RESERVED 7      /* address space reserved for the lazily committed tables */
#define WFST_MEM_LAZY_COMMITTED 8 /* device memory committed to them (part of WFST_MEM_BYTES) */
#define WFST_MEM_COUNT 9
int wfst_mem_stats(wfst_decoder* d, int64_t* out, int32_t n);

/*
 * Test hook for the failure path of the device-side grid barrier (§5: the
 * step loop's phases are separated by barriers; here every wait on one is
 * bounded).  Arms the decoder's NEXT call only: each grid barrier of that
 * launch waits for one arrival more than the grid makes, with a limit of
 * timeout_ns instead of 4 s.  The first wait therefore gives up, sets the
 * abort flag, and every CTA returns; the call returns WFST_ERR_TIMEOUT
 * after wiping the decoder's per-state tables and closing its streaming
 * channels, exactly as after a real timeout.  Later calls run normally.
 * Nothing faults, traps or waits without a bound.
 * Errors: INVALID_ARG (NULL decoder, timeout_ns outside [1 ms, 4 s]).
 */
int wfst_test_barrier_timeout(wfst_decoder* d, int64_t timeout_ns);

/*
 * A measurement kernel, not part of the decoder (the page has no
 * counterpart): reads random seg_bytes-long segments (16, 64 or 128 bytes,
 * segment-aligned) of the caller's device table, grid CTAs of 512 threads,
 * loads_per_thread reads per thread (a multiple of 4, issued four at a
 * time).  Timed by the caller on `stream`, it gives the device's ceiling for
 * random reads per second, the limit of the decoder's own random line
 * accesses.  table: device, 16-byte aligned, table_bytes / seg_bytes in
 * [1, 2^32); sink: a device int32 the kernel practically never writes.
 * Errors: INVALID_ARG, CUDA (launch).
 */
int wfst_probe_random_gather(const void* table, int64_t table_bytes, int32_t seg_bytes, int32_t grid,
                             int32_t loads_per_thread, int32_t seed, int32_t* sink, void* stream);

/*
 * Offline decode that allocates nothing (no device or pinned memory, no
 * decoder object).  The web page "GPU WFST Beam-Search Decoder" has no
 * counterpart for it.  This is the same decode as wfst_decode for callers
 * that may not allocate once running (their own memory pool, a real-time
 * thread): its working memory is one region of WFST_STATIC_SCRATCH_BYTES
 * that the library declares statically, one per device per process.
 * Arguments as in wfst_decode, with the decoder replaced by the graph and
 * its params: lattice and streaming must be 0; log_probs must be device
 * memory on the graph's device; B <= WFST_STATIC_MAX_LANES.  The frontier
 * holds every state; the winners log gets whatever the region has left
 * after the call's other tables (at most one entry per state and frame) and
 * cannot grow: a lane that fills it comes back with overflow bit 4 and the
 * call returns CAPACITY, its outputs written and flagged (wfst_decode would
 * grow the log and decode the lane again).
 * The first call on a device resolves the region's address and may load the
 * module there: make it before any stream capture begins.  The zero-start
 * part of the region (entries, marks, counters, barrier, results) is cleared
 * by every call.  Calls on one device are serialized by a lock held until
 * the results are on the host: calls that overlapped would race on the
 * region.
 * Errors: INVALID_ARG, CAPACITY (B or the call's tables exceed the region,
 * the message giving the bytes needed; or a lane filled the winners log),
 * CUDA, TIMEOUT.
 */
#define WFST_STATIC_SCRATCH_BYTES (16u << 20)
#define WFST_STATIC_MAX_LANES 8
int wfst_decode_static(const wfst_graph* g, const wfst_params* params, const void* log_probs,
                       int32_t dtype, int64_t stride_b, int64_t stride_t, const int32_t* lens,
                       int32_t B, int32_t T, void* stream, int32_t* words, int32_t words_cap,
                       int32_t* word_lens, double* scores, int32_t* meta);

/*
 * Blank-skip frame pre-slicing, a pre-pass outside the decoder (§3 Decoding
 * Semantics: blank-dominated frames are removed before the search, not
 * inside it, WeNet-style, threshold 0.98 by default).  Frame t < lens[b] of
 * lane b is dropped iff log_probs[b, t, blank_id] > log(threshold), with log(threshold) computed in
 * double and rounded once to fp32 and the log-prob widened exactly to fp32.
 * The kept rows are packed in order into out[b, i, v] at out + (b*T + i)*V
 * (same dtype), out_lens[b] receives the kept count and frame_map[b*T + i] the
 * source frame of kept row i (-1 past the count).  Decode the result with
 * lens = out_lens and stride_t = V, stride_b = T*V.
 * log_probs [B, T, V] with strides as in wfst_decode; lens, out, out_lens and
 * frame_map are DEVICE arrays ([B], [B*T*V], [B], [B*T]); nothing is
 * allocated and nothing is copied to the host: the two kernels are enqueued on
 * `stream` and the call returns without waiting.  Rows past out_lens[b] are
 * left as they were.  Errors: INVALID_ARG (NULL or host pointers, blank_id out
 * of [0, V), threshold <= 0, bad strides), CUDA.
 */
int wfst_blank_skip(const void* log_probs, int32_t dtype, int64_t stride_b, int64_t stride_t,
                    int32_t vocab_size, int32_t blank_id, float threshold, const int32_t* lens,
                    int32_t B, int32_t T, void* out, int32_t* out_lens, int32_t* frame_map,
                    void* stream);

const char* wfst_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* WFST_GB300_H */
