// wfst_internal.h — device data layout shared by the host API and the
// persistent decode kernel.  See the design notes for the memory plan.
#pragma once
#include <cstdint>

namespace wfst {

constexpr int kThreads = 512;     // threads per CTA of the persistent kernel
constexpr int kTile = 128;        // arc slots per work tile (one warp walks one tile)
constexpr int kTokCap = 128;      // frontier tokens a warp stages in shared memory per chunk
constexpr int kMaxLanes = 256;    // lanes per decoder
constexpr int kWarps = kThreads / 32;

// overflow bits (the page's §7 values)
constexpr int kOvfArena = 4;
constexpr int kOvfKept = 16;
constexpr int kOvfPath = 32;
constexpr int kMaxGrowRounds = 12;  // offline capacity doublings per decode call
constexpr unsigned long long kBarrierTimeoutNs = 4000000000ull;  // a grid barrier wait gives up after 4 s

// lattice record flags
constexpr int kRecEps = 1;
constexpr int kRecFinal = 2;
constexpr int kRecRedirect = 4;
constexpr int kRecDead = 8;       // epsilon relaxation evaluated with a non-final score

// lane status
constexpr int kLaneFree = 0;
constexpr int kLaneRunning = 1;
constexpr int kLaneDone = 2;

// per-call lane flags
constexpr int kCallInit = 1;      // reset the lane and open its start frontier
constexpr int kCallFinal = 2;     // run the final step + backtrack at the end of the call
constexpr int kCallPartial = 4;   // backtrack the best current token at the end of the call

// Graph, internal layout: per state, emitting arcs first then epsilon arcs
// (a stable partition of the caller's arcs; caller arc ids are kept).
struct DevGraph {
  int32_t N, start, V, has_eps;
  int64_t A;
  int32_t eps_depth;              // longest epsilon path (passes needed by a closure)
  int32_t pad;
  const int4* meta;               // [N] {row_begin, emit_end, eps_end, emit_maxw bits}
  const int4* arcs;               // [A] internal {dst, weight bits, ilabel (-1 = epsilon), caller id}
  const int32_t* c_src;           // [A] caller id -> src state | (epsilon << 31)
  const int32_t* c_dst;           // [A] caller id -> dst state
  const int32_t* c_olabel;        // [A] caller id -> olabel
  const float* final_w;           // [N]
};

struct FrameCnt {                 // per lane, per frame (ring of 4 frames)
  unsigned long long cnt;         // (tokens << 32) | emitting arcs of the frame's tokens
  unsigned int maxkey;            // ordered max end of the step that consumes the frame
  unsigned int admitted;          // admitted emitting candidates of that step
  unsigned long long final_key;   // (ordered final score, 0x7fffffff - state)
  unsigned long long best_key;    // (ordered score, 0x7fffffff - arc) of the best token
  unsigned int anc_hi;            // ancestor GC: 1 + the largest checkpoint ancestor of the frame's tokens
  unsigned int anc_lo;            // ... 0x7fffffff - the smallest (both 0 = none committed)
};

struct LaneState {                // persistent per lane (mirrored in shared memory)
  int32_t t;                      // frames consumed; the frontier is frame t
  int32_t committed;              // last frame whose tokens are in the winners log
  float beam;
  int32_t status;
  int64_t cursor;                 // next free winners-log entry
  int64_t base_cur;               // log base of frame `committed`
  int64_t base_prev;              // log base of frame `committed - 1`
  int64_t lat_cursor;             // next free lattice record
  uint32_t eps_pass;              // epsilon worklist pass id (dedupe marks)
  int32_t overflow;
  int32_t t_eff;                  // offline length (last-frames rule), -1 streaming
  int32_t bt_top;                 // frame of the last backtracked path's newest token, -1 = none
  int32_t bt_len;                 // arcs of that path (kept oldest-first in path)
  int32_t gc_t;                   // frames consumed at the lane's last winners-log GC round
  int64_t floor;                  // winners-log GC root: entries below it are free (0 without GC)
  int32_t fin_n;                  // finalized words (the GC-cut prefix of the best path)
  int32_t gc_c;                   // ancestor GC: the checkpoint frame
  int64_t gc_cbase;               // ancestor GC: winners-log index of the checkpoint frame's first token
};

struct LaneCall {                 // per lane, per call
  int32_t row;                    // row of the call's log-prob tensor, -1 = not in this call
  int32_t nframes;                // frames to consume in this call
  int32_t flags;                  // kCall*
  int32_t t_eff;                  // offline length, -1 streaming
};

struct LaneStats {                // per lane, accumulated by the kernel (zeroed per call)
  unsigned long long frames, sum_n, sum_d, sum_a, sum_m, eps, finals;
  unsigned long long steps;
  unsigned long long lat_held;    // lattice records in the lane's arena at the end of the call
  unsigned long long log_hw;      // most winners-log entries live (after the last cut) in the call
};

struct LatRec {                   // 32 bytes
  int32_t frame_flags;            // (frame << 4) | flags
  int32_t src_tok;                // winners-log index of the source token
  int32_t dst_tok;                // winners-log index of the destination (-1 super-final)
  int32_t src_state;
  int32_t dst_state;              // -1 super-final
  int32_t arc;                    // caller arc id, or A + s
  float end;                      // forward value of the candidate
  float arcscore;                 // the record's own score
};

struct Result {                   // per lane, per call
  int32_t ok, reached_final, overflow, n_words;
  float score;
  int32_t n_arcs;
  int32_t pad0, pad1;
};

struct GridBar {
  unsigned int count;             // arrivals (monotonic within a launch)
  unsigned int abort;             // set when any wait gave up
  unsigned int error;             // 1 = barrier timeout, 2 = closure did not converge
  unsigned int epochs;            // barriers executed (written at the end)
  unsigned int changed[3];        // per-pass change flags (lattice epsilon groups)
  unsigned int eps_passes;        // epsilon-closure worklist passes run (written at the end)
};

struct TokRec {                   // a frontier token (or epsilon worklist entry), 16 bytes
  int32_t state;
  uint32_t off;                   // first slot of its arcs in the frame's arc-slot space
  int32_t row;                    // first internal arc (emitting, or epsilon for worklists)
  float maxw;                     // max emitting arc weight (upper-bound skip)
};

struct DevWork {
  int32_t L, N;
  int64_t qcap;                   // frontier capacity per lane per frame
  int64_t log_cap, lat_cap, path_cap;
  // distance in entries between consecutive lanes' regions of the front /
  // score / worklist, winners-log / bwd and lattice arrays: the reserved
  // size, at least the capacity (lazily committed regions, §6.2)
  int64_t q_stride, log_stride, lat_stride;
  int64_t tiles_cap;              // tiles per lane per frame
  int32_t lattice, max_frames;
  ulonglong2* ent;                // [L][N][2] recombination entries, 16 bytes per state and frame
                                  // parity: {key, src}; 0 = empty (see the kernel)
  int2* tpos;                     // [L][N] position of a state's token in its frame, per parity
  TokRec* front;                  // [2][L][qcap] tokens of a frame (the frontier), claim order
  float* score;                   // [2][L][qcap] token scores, staged by the max pass
  int32_t* tile_first;            // [2][L][tiles_cap] token holding each tile's first slot
  TokRec* wl;                     // [2][L][qcap] epsilon worklists
  int32_t* wl_tile_first;         // [2][L][tiles_cap]
  float* maxlp;                   // [L][max_frames] max log-prob of each row of the call
  uint32_t* mark;                 // [L][N] worklist dedupe marks
  unsigned long long* wl_cnt;     // [3][L] (tokens << 32) | epsilon arcs
  int2* wlog;                     // [L][log_cap] winners log {delta, arc}: the predecessor is
                                  // entry i - delta (0 = none); a ring (index & log_mask) with GC
  unsigned long long log_mask;    // log_cap - 1 with GC (log_cap a power of two), else all ones
  int32_t* fin;                   // [L][fin_cap] finalized words (GC)
  int32_t* anc;                   // [2][L][qcap] ancestor GC (epsilon-free graphs): each token's
                                  // ancestor among the lane's checkpoint-frame tokens (its position)
  int64_t fin_cap;
  FrameCnt* fcnt;                 // [4][L]
  LaneState* lanes;               // [L]
  LaneStats* stats;               // [L]
  LatRec* lat;                    // [L][lat_cap]
  unsigned long long* lat_cnt;    // [L] records appended
  int64_t* lat_groups;            // [L][max_frames+2] B_t: first record appended after frame t's closure
  int64_t* lat_gtmp;              // [L][max_frames+2] interval prune: survivors, then write cursors, per group
  uint32_t* bwd;                  // [L][log_cap] ordered backward scores
  LatRec* lat_out;                // [L][lat_cap] kept records (compacted)
  unsigned long long* lat_out_n;  // [L]
  int32_t* path;                  // [L][path_cap] best path, oldest arc first (the tail is walk scratch)
  int2* pframe;                   // [L][max_frames+2] per frame of that path: {winners-log index, path position}
  Result* res;                    // [L]
  int32_t* words;                 // [L][words_cap] (words_cap per call)
  GridBar* bar;
  unsigned long long* prof;       // [kProfSlots] ns per phase kind (CTA 0's view)
};

// phase timers (ns, summed over a call, measured by CTA 0 thread 0)
enum ProfSlot { kProfInit = 0, kProfCommitMax, kProfExpand, kProfClosure, kProfPrune, kProfTail,
                kProfPrologue, kProfCommit, kProfClear, kProfMaxTiles, kProfBarX, kProfExpTiles,
                kProfFinal, kProfBarY, kProfSlots = 16 };

struct RunArgs {
  DevGraph g;
  DevWork w;
  const void* lp;                 // log-prob base (device)
  int64_t stride_b, stride_t;     // elements
  const LaneCall* calls;          // [L] device
  int32_t nlanes;                 // lanes scanned (max_lanes)
  int32_t words_cap;
  float search_beam, output_beam;
  int32_t min_active, max_active, allow_partial, lattice;
  int32_t nblocks;
  int32_t ub_skip;                // upper-bound skips in the max/expand passes
  int32_t gc_interval;            // winners-log GC every gc_interval frames, 0 = off
  int32_t lat_interval;           // interval lattice prune every lat_interval frames, 0 = off
  uint32_t bar_extra;             // arrivals a grid barrier waits for beyond the grid (0; 1 = test hook)
  unsigned long long timeout_ns;  // limit of one grid barrier wait
};

}  // namespace wfst
