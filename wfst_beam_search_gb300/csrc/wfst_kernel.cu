// wfst_kernel.cu — the persistent decode kernel (sm_103a).
//
// One cooperative launch runs a whole decode call on the device: lane
// initialisation, the frame-synchronous step loop, epsilon closure, the final
// step, backtrack to words and the lattice backward prune.  Phases are
// separated by a software grid barrier whose waits are bounded in time (an
// expired wait aborts the launch with an error flag instead of hanging).
//
// Method: "GPU WFST Beam-Search Decoder" (OASR docs).  Per frame and lane:
//   §3  dynamic beam update from the frontier size;
//   §5.1/§5.2 the frontier's emitting arcs form one flattened slot space over
//        all lanes, cut into fixed tiles that every CTA walks (load balance
//        with one hot lane);
//   §5.3 pass 1 (max): exact per-lane maximum of end = (score + w) + lp over
//        every slot, skipping tokens whose upper bound (score + max weight) +
//        max log-prob cannot beat an end already posted; pass 2 (expand):
//        admit end > max - beam and recombine by destination with a 128-bit
//        CAS on {(ordered score, lowest arc id), source token} — a
//        direct-indexed per-lane table replaces the page's hash;
//   §5.4 commit: each frontier token gets a winners-log entry {delta, arc}
//        (its predecessor is the entry delta places back);
//   §5.5 epsilon closure by worklist passes to a fixpoint; lattice records;
//   §7  backtrack from the final token; lattice backward output_beam prune.
// Work distribution: the arc slots of a frame form tiles of kTile slots; a
// CTA owns every (G*W)-th group of W adjacent tiles (W warps per CTA), the
// last partial round dealt out one tile per CTA, and hands them, in order,
// to whichever of its warps is free; a warp stages its tile's tokens in its
// own shared-memory area, and every lane issues the loads of its kSPT slots
// together (one chain of dependent accesses per tile).
// Three instantiations (Kind) compile only the code their decodes need.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "wfst_internal.h"

namespace wfst {

constexpr int kSPT = kTile / 32;                           // slots per lane per tile
constexpr int kCB = 5;                                     // tokens per thread per commit batch

enum Phase { kNone = 0, kEmit = 1, kFin = 2, kPart = 3 };

// Kernel instantiations.  The epsilon closure, lattices and the walking GC
// round live in the general one only; a decode of an epsilon-free graph
// without lattices runs a kernel with that code compiled out (its registers
// then serve the emitting passes), with or without the ancestor GC.
enum Kind { kKindGeneral = 0, kKindPlain = 1, kKindAnc = 2 };

struct SmLane {
  int32_t t, committed, status, phase;
  float beam, cutoff;
  int32_t n_cur, n_prev;
  uint32_t d_cur;
  int32_t row, t0, t_end, flags, t_eff;
  int32_t need_commit, done_final, done_partial, expanded;
  int64_t cursor, base_cur, base_prev;
  uint32_t eps_pass, wl_e;
  int32_t wl_n, closure;
  int64_t res_lo, res_hi;         // lattice records resolved in this step's commit phase
  unsigned long long frames, sum_n, sum_d, sum_m;
  float maxlp;                    // max log-prob of frame t
  int32_t was_emit;
  float cur_max;                  // this step's exact max end (expand pass)
  int32_t seed_next;              // the expand pass seeds the next step's max
  int32_t prev_cleared;           // the previous frame's entries were cleared by its expand pass
  int64_t floor;                  // winners-log GC root (entries below it are free)
  int32_t fin_n;                  // finalized words of the lane (GC)
  int32_t gc_t;                   // frames consumed at the last GC round
  int32_t gc_due;                 // a GC round runs at the end of this step
  int32_t gc_c;                   // ancestor GC: checkpoint frame
  int64_t gc_cbase;               // ancestor GC: winners-log index of its first token
  int64_t gc_e;                   // ancestor GC: the cut point of this step's round
  int64_t log_hw;                 // most winners-log entries live (cursor - root) in this call
};

struct WStage {                   // one warp's staged tokens of its current tile
  uint32_t off[kTokCap + 1];
  int32_t row[kTokCap];
  float score[kTokCap];
  int32_t state[kTokCap];
  float ub[kTokCap];
  int32_t tpos[kTokCap];          // epsilon worklists: the token's position in its frame
};

// Shared memory of a CTA: this struct, then the per-lane arrays it points to,
// sized by the launch's lane count (shared memory left unused is L1 cache on
// this part, and the log-prob gathers live on L1 hits).
struct Smem {
  SmLane* lane;                   // [L] lane mirrors
  int32_t* pre_a;                 // [L+1] work units per lane, exclusive prefix (tiles)
  int32_t* pre_b;                 // [L+1] commit tokens / tasks
  int32_t* pre_c;                 // [L+1] clear tokens
  int32_t* pre_d;                 // [L+1] lattice records to resolve
  int32_t* pre_e;                 // [L+1] lattice prune: records of the current group
  int64_t* glo;                   // [L] lattice prune: first record of the current group
  alignas(16) WStage ws[kWarps];
  float redf[kWarps];
  uint32_t redu[kWarps];
  int32_t scan_tmp[kWarps];
  int32_t flag, abort, any, bt_n;
  unsigned tctr[2];                // per-CTA tile counters of the max / expand passes
  unsigned long long prof[kProfSlots + 2];  // CTA 0's phase timers + two time marks
  int64_t bt_idx;
  int32_t bt_ok, bt_reached, bt_state, bt_pad;
  int32_t bt_d, bt_lo, bt_hi;
  float bt_score;
  unsigned long long gc_min;      // GC round: deepest anchor-chain depth another chain met
  int32_t gc_ok, gc_nw;
  int32_t gc_pre;                 // ancestor GC: the chain walk of the CTA's first task, run
                                  // during the expand pass (-2: not run)
  unsigned eps_passes;            // epsilon-closure worklist passes of this launch
};

// ------------------------------------------------------------------ helpers

__device__ __forceinline__ unsigned ord_f(float x) {
  unsigned u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord_f(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// (score, id): a higher score wins, then the LOWER id; id -1 (start token) is lowest.
__device__ __forceinline__ unsigned long long mk_key(float s, int32_t id) {
  return ((unsigned long long)ord_f(s) << 32) | (unsigned)(0x7fffffffu - (unsigned)id);
}
__device__ __forceinline__ int32_t key_id(unsigned long long k) {
  return (int32_t)(0x7fffffffu - (unsigned)(k & 0xffffffffull));
}
__device__ __forceinline__ float key_score(unsigned long long k) { return unord_f((unsigned)(k >> 32)); }

__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}
__device__ __forceinline__ TokRec ld_tok(const TokRec* p) {
  const int4 v = __ldcg(reinterpret_cast<const int4*>(p));
  TokRec r;
  r.state = v.x;
  r.off = (uint32_t)v.y;
  r.row = v.z;
  r.maxw = __int_as_float(v.w);
  return r;
}

// An arc record read by the expand pass or an epsilon pass: read-only, and
// read once in the pass, so it is kept out of L1 (which then holds the
// log-prob rows and token rows the same tiles reuse).
__device__ __forceinline__ int4 ld_arc(const int4* p) {
  int4 v;
  asm("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// Bring a line into L2 with evict-last priority (used for each admitted
// candidate's entry just before its CAS: the next max pass reads it again).
__device__ __forceinline__ void prefetch_l2_keep(const void* p) {
  asm volatile("prefetch.global.L2::evict_last [%0];" : : "l"(p));
}
// The max pass's read of a token's recombination entry, with an L2
// evict-last policy: a state that stays in the beam (a blank self-loop) has
// its entry's line taken by the next expand pass's CAS.
__device__ __forceinline__ ulonglong2 ld_ent_keep(const ulonglong2* p) {
  unsigned long long pol;
  asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  ulonglong2 v;
  asm volatile("ld.global.cg.L2::cache_hint.v2.u64 {%0, %1}, [%2], %3;" : "=l"(v.x), "=l"(v.y) : "l"(p), "l"(pol));
  return v;
}

template <typename T>
__device__ __forceinline__ float lp_at(const T* row, int v);
template <>
__device__ __forceinline__ float lp_at<float>(const float* row, int v) { return __ldg(row + v); }
template <>
__device__ __forceinline__ float lp_at<__half>(const __half* row, int v) {
  return __half2float(__ldg(row + v));
}

// Largest l in [0, L) with pre[l] <= x (pre: exclusive prefix, pre[L] = total).
__device__ __forceinline__ int find_lane(const int32_t* pre, int L, int32_t x) {
  int lo = 0, hi = L;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Largest i in [0, n) with off[i] <= slot.
__device__ __forceinline__ int find_tok(const uint32_t* off, int n, uint32_t slot) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (off[mid] <= slot) lo = mid; else hi = mid;
  }
  return lo;
}

// In-place exclusive prefix of pre[0..L) (pre[L] = total), computed
// redundantly by every CTA.  Callers synchronise before writing `pre`.
__device__ void lane_scan(int32_t* pre, int L) {
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int per = (L + 31) / 32;
    int32_t local = 0;
    for (int i = 0; i < per; i++) {
      const int idx = lane * per + i;
      if (idx < L) local += pre[idx];
    }
    int32_t inc = local;
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    int32_t run = inc - local;
    for (int i = 0; i < per; i++) {
      const int idx = lane * per + i;
      if (idx < L) {
        const int32_t v = pre[idx];
        pre[idx] = run;
        run += v;
      }
    }
    if (lane == 31) pre[L] = inc;
  }
  __syncthreads();
}

// lane_scan of four arrays at once (warp w scans array w), one barrier.
__device__ void lane_scan4(int32_t* p0, int32_t* p1, int32_t* p2, int32_t* p3, int L) {
  const int warp = threadIdx.x >> 5;
  if (warp < 4) {
    int32_t* pre = warp == 0 ? p0 : warp == 1 ? p1 : warp == 2 ? p2 : p3;
    const int lane = threadIdx.x & 31;
    const int per = (L + 31) / 32;
    int32_t local = 0;
    for (int i = 0; i < per; i++) {
      const int idx = lane * per + i;
      if (idx < L) local += pre[idx];
    }
    int32_t inc = local;
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    int32_t run = inc - local;
    for (int i = 0; i < per; i++) {
      const int idx = lane * per + i;
      if (idx < L) {
        const int32_t v = pre[idx];
        pre[idx] = run;
        run += v;
      }
    }
    if (lane == 31) pre[L] = inc;
  }
  __syncthreads();
}

// Phase timer: CTA 0 thread 0 charges the time since the last mark (kept in
// shared memory, slot `from`) to accumulator `slot`.
__device__ __forceinline__ void prof_mark(unsigned long long* acc, int from, int slot) {
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const unsigned long long now = gtimer();
    acc[slot] += now - acc[kProfSlots + from];
    acc[kProfSlots + from] = now;
  }
}

// Bounded software grid barrier.  Returns false when the launch aborts.  A
// wait gives up after a.timeout_ns; a.bar_extra (0 except under the test
// hook that exercises this path) raises the arrival target beyond the grid.
// The arrival is a release add at GPU scope (after the CTA barrier, it
// publishes every write of the CTA), the wait an acquire load of the count
// (it sees every write the other CTAs published); the abort flag and the
// time limit are looked at every 16 polls.
__device__ bool grid_sync(const RunArgs& a, Smem& S, unsigned& epoch) {
  __syncthreads();
  if (threadIdx.x == 0) {
    GridBar* bar = a.w.bar;
    epoch++;
    const unsigned target = epoch * (unsigned)gridDim.x + a.bar_extra;
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" : : "l"(&bar->count) : "memory");
    int ab = 0;
    const unsigned long long t0 = gtimer();
    for (unsigned it = 1;; it++) {
      const unsigned c = ld_acquire(&bar->count);
      if ((int)(c - target) >= 0) break;
      if ((it & 15u) == 0u) {
        if (ld_acquire(&bar->abort)) { ab = 1; break; }
        if (gtimer() - t0 > a.timeout_ns) {
          atomicExch(&bar->abort, 1u);
          atomicOr(&bar->error, 1u);
          ab = 1;
          break;
        }
      }
      __nanosleep(32);
    }
    S.abort = ab;
  }
  __syncthreads();
  return S.abort == 0;
}

__device__ __forceinline__ float block_max_f(float v, Smem& S) {
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) S.redf[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = S.redf[0];
  for (int i = 1; i < kWarps; i++) r = fmaxf(r, S.redf[i]);
  return r;
}
__device__ __forceinline__ uint32_t block_sum_u(uint32_t v, Smem& S) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) S.redu[threadIdx.x >> 5] = v;
  __syncthreads();
  uint32_t r = 0;
  for (int i = 0; i < kWarps; i++) r += S.redu[i];
  return r;
}

__device__ __forceinline__ void lane_ovf(const RunArgs& a, int l, int bits) {
  atomicOr(&a.w.lanes[l].overflow, bits);
}

__device__ __forceinline__ size_t pl(const DevWork& w, int par, int l) {
  return ((size_t)par * w.L + l) * (size_t)w.N;       // per-state arrays of a lane (marks)
}
__device__ __forceinline__ size_t ql(const DevWork& w, int par, int l) {
  return ((size_t)par * w.L + l) * (size_t)w.q_stride;  // front / score / worklists
}
__device__ __forceinline__ size_t tl(const DevWork& w, int par, int l) {
  return ((size_t)par * w.L + l) * (size_t)w.tiles_cap;
}
__device__ __forceinline__ FrameCnt* fc_of(const DevWork& w, int f, int l) {
  return w.fcnt + (size_t)(f & 3) * w.L + l;
}

// Recombination entry of state d, lane l, frame parity par: 16 bytes
// {key, src} where key = (ordered score, 0x7fffffff - arc id) of the best
// incoming candidate so far and src = the position of that candidate's source
// token (in the previous frame for an emitting arc; in the same frame, with
// bit 31 set, for an epsilon arc); with the ancestor GC the upper half of the
// src word carries that source token's checkpoint ancestor.  Both parities of a state share one
// 32-byte sector, so a state that stays in the frontier keeps hitting the
// same line frame after frame.  The token's own position lives in tpos.
__device__ __forceinline__ ulonglong2* ent_at(const DevWork& w, int l, int32_t d, int par) {
  return w.ent + ((((size_t)l * (size_t)w.N + (size_t)d) << 1) | (size_t)par);
}


__device__ __forceinline__ ulonglong2 cas128(ulonglong2* p, ulonglong2 cmp, ulonglong2 val) {
  ulonglong2 old;
  asm volatile(
      "{\n\t.reg .b128 c, v, o;\n\t"
      "mov.b128 c, {%2, %3};\n\t"
      "mov.b128 v, {%4, %5};\n\t"
      "atom.relaxed.gpu.global.cas.b128 o, [%6], c, v;\n\t"
      "mov.b128 {%0, %1}, o;\n\t}"
      : "=l"(old.x), "=l"(old.y)
      : "l"(cmp.x), "l"(cmp.y), "l"(val.x), "l"(val.y), "l"(p)
      : "memory");
  return old;
}

constexpr int kCasTries = 1 << 16;  // a CAS retry only follows another thread's progress

// Offer a candidate: 2 = claimed the empty entry, 1 = improved it, 0 = no change.
// The first attempt assumes an empty entry (the common case for a new
// state), so a claim costs one round trip; a failed CAS returns the current
// value and the loop continues from it.
__device__ __forceinline__ int relax_ent(const RunArgs& a, ulonglong2* e, unsigned long long key,
                                         unsigned long long srcw) {
  ulonglong2 cur = make_ulonglong2(0ull, 0ull);
  const ulonglong2 nv = make_ulonglong2(key, srcw);
  for (int it = 0; it < kCasTries; it++) {
    if (key <= cur.x) return 0;
    const ulonglong2 old = cas128(e, cur, nv);
    if (old.x == cur.x && old.y == cur.y) return cur.x == 0ull ? 2 : 1;
    cur = old;
  }
  atomicOr(&a.w.bar->error, 4u);
  return 0;
}

__device__ __forceinline__ uint32_t ent_src(const ulonglong2& e) { return (uint32_t)e.y; }

// Winners-log entry i (a logical index) of lane l: {delta, arc}, the
// predecessor being entry i - delta (delta 0: none; arc -1: the start token
// or a GC root).  delta is signed: an epsilon arc's source token sits in the
// same frame, possibly at a later position.  Without the GC, delta is the
// whole 32-bit word and the log is flat.  With the GC the log is a ring
// (i & log_mask), delta is the low 30 bits (two's complement) and a GC round
// marks entries with the two high bits; an anchor-chain entry holds its
// depth on the chain in the low bits while it is marked.
constexpr uint32_t kMarkAnchor = 0x80000000u;  // on the anchor chain of a GC round
constexpr uint32_t kMarkWalk = 0x40000000u;    // on another token's walk of a GC round
constexpr uint32_t kDeltaMask = 0x3fffffffu;
__device__ __forceinline__ int32_t sext30(uint32_t x) { return (int32_t)(x << 2) >> 2; }
__device__ __forceinline__ int32_t wlog_delta(const RunArgs& a, int32_t x) {
  return a.gc_interval > 0 ? sext30((uint32_t)x) : x;
}
__device__ __forceinline__ int2* wlog_at(const DevWork& w, int l, int64_t i) {
  return w.wlog + (size_t)l * (size_t)w.log_stride + (size_t)((unsigned long long)i & w.log_mask);
}
// The winners-log entry of a frame token: its arc and the distance back to
// the token it came from (0 for the start token).
__device__ __forceinline__ void wlog_commit(const RunArgs& a, int l, int64_t idx, int64_t floor,
                                            int32_t arc, int64_t prev) {
  const DevWork& w = a.w;
  const int64_t d = arc < 0 ? 0 : idx - prev;
  const int32_t x = a.gc_interval > 0 ? (int32_t)((uint32_t)d & kDeltaMask) : (int32_t)d;
  // a streaming store: the entry is read again only by a backtrack or a GC
  if (idx - floor < w.log_cap) __stcs(wlog_at(w, l, idx), make_int2(x, arc));
  else lane_ovf(a, l, kOvfArena);
}
// Ancestor GC (winners-log GC on epsilon-free graphs): every committed token
// of frame f records the position of its ancestor among the tokens of the
// lane's checkpoint frame C (its predecessor's position when f = C + 1, else
// its predecessor's recorded ancestor).  A frame whose tokens all share one
// ancestor has converged: every chain passes through that checkpoint token.
// The winning candidate's source ancestor rides in the entry (upper half of
// its src word), so the commit needs no read of the previous frame.
__device__ __forceinline__ int32_t anc_of(int f, int32_t arc, unsigned long long srcw, int32_t gc_c) {
  if (arc < 0) return 0;  // the start token
  return (f - 1 == gc_c) ? (int32_t)(srcw & 0x7fffffffull) : (int32_t)(srcw >> 32);
}
__device__ __forceinline__ void anc_post(const RunArgs& a, int l, int f, int32_t amin, int32_t amax) {
  for (int o = 16; o; o >>= 1) {
    amin = min(amin, __shfl_xor_sync(0xffffffffu, amin, o));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  }
  if ((threadIdx.x & 31) == 0 && amax >= 0) {
    FrameCnt* fc = fc_of(a.w, f, l);
    atomicMax(&fc->anc_hi, (unsigned)(amax + 1));
    atomicMax(&fc->anc_lo, 0x7fffffffu - (unsigned)amin);
  }
}

// Token positions per state are kept only where something looks a state's
// token up (epsilon worklists, lattice records); the final backtrack of other
// graphs finds its one token by a scan of the frame.
__device__ __forceinline__ bool tpos_kept(const RunArgs& a) { return a.g.has_eps || a.lattice; }

__device__ __forceinline__ int32_t* tpos_at(const DevWork& w, int l, int32_t d, int par) {
  return reinterpret_cast<int32_t*>(w.tpos + ((size_t)l * (size_t)w.N + (size_t)d)) + par;
}

__device__ __forceinline__ uint32_t warp_inc_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += x;
  }
  return v;
}

// Warp-cooperative append of up to K states per thread to a token list (a
// frame's frontier, EPS = false, or an epsilon worklist, EPS = true).  One
// 64-bit atomic per warp returns the positions and an exclusive prefix of the
// states' arc counts (in (k, lane) order), so each token owns a contiguous
// arc-slot range; each tile boundary inside a token's range records that
// token.  The per-state row data is re-read in the second pass (an L1 hit)
// rather than kept live across the atomic.
template <int K, bool EPS>
__device__ __forceinline__ void warp_append(const bool (&want)[K], const int32_t (&d)[K],
                                            unsigned long long* ctr, TokRec* list, int32_t* tfirst,
                                            int pos_par, int64_t cap, const RunArgs& a, int l) {
  const unsigned full = 0xffffffffu;
  uint32_t cnt_sum = 0, tot_sum = 0;
#pragma unroll
  for (int k = 0; k < K; k++) {
    cnt_sum += __popc(__ballot_sync(full, want[k]));
    uint32_t v = 0;
    if (want[k]) {
      const int4 m = __ldg(a.g.meta + d[k]);
      v = EPS ? (uint32_t)(m.z - m.y) : (uint32_t)(m.y - m.x);
    }
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(full, v, o);
    tot_sum += v;
  }
  if (!cnt_sum) return;
  const int lane = threadIdx.x & 31;
  unsigned long long base = 0;
  if (lane == 0) base = atomicAdd(ctr, ((unsigned long long)cnt_sum << 32) | tot_sum);
  base = __shfl_sync(full, base, 0);
  uint32_t pb = (uint32_t)(base >> 32), ob = (uint32_t)base;
  const unsigned lt = lanemask_lt();
#pragma unroll
  for (int k = 0; k < K; k++) {
    const unsigned m = __ballot_sync(full, want[k]);
    int4 md = make_int4(0, 0, 0, 0);
    if (want[k]) md = __ldg(a.g.meta + d[k]);
    const uint32_t dv = EPS ? (uint32_t)(md.z - md.y) : (uint32_t)(md.y - md.x);
    const uint32_t inc = warp_inc_scan(dv);
    if (want[k]) {
      const uint32_t p = pb + __popc(m & lt);
      const uint32_t off = ob + inc - dv;
      if (p < (uint64_t)cap) {
        *reinterpret_cast<int4*>(list + p) = make_int4(d[k], (int)off, EPS ? md.y : md.x, EPS ? 0 : md.w);
        if (pos_par >= 0) *tpos_at(a.w, l, d[k], pos_par) = (int32_t)p;
        if (dv > 0) {
          const uint32_t k0 = (off + kTile - 1) / kTile, k1 = (off + dv - 1) / kTile;
          for (uint32_t q = k0; q <= k1; q++) tfirst[q] = (int32_t)p;
        }
      } else {
        lane_ovf(a, l, kOvfKept);
      }
    }
    pb += __popc(m);
    ob += __shfl_sync(full, inc, 31);
  }
}

// Claim states into frame f of lane l (and seed the epsilon worklist W0 with
// the claimed states that have epsilon arcs).
template <int K, bool GEN = true>
__device__ __forceinline__ void warp_claim(const RunArgs& a, const bool (&want)[K], const int32_t (&d)[K],
                                           int l, int f, bool seed_worklist) {
  const DevWork& w = a.w;
  const int par = f & 1;
  warp_append<K, false>(want, d, &fc_of(w, f, l)->cnt, w.front + ql(w, par, l), w.tile_first + tl(w, par, l),
                        (GEN && tpos_kept(a)) ? par : -1, w.qcap, a, l);
  if (GEN && a.g.has_eps && seed_worklist) {
    bool ws[K];
#pragma unroll
    for (int k = 0; k < K; k++) {
      ws[k] = false;
      if (want[k]) {
        const int4 m = __ldg(a.g.meta + d[k]);
        ws[k] = m.z > m.y;
      }
    }
    warp_append<K, true>(ws, d, &w.wl_cnt[l], w.wl + ql(w, 0, l), w.wl_tile_first + tl(w, 0, l), -1,
                         w.qcap, a, l);
  }
}

// Warp-cooperative lattice record append: one 64-bit atomic reserves the
// records of all K slots of every thread (ballot m[k] per slot); the record
// of slot k of this thread goes to base + sum_{k' < k} popc(m[k']) +
// popc(m[k] & lanemask_lt) (lat_put).  The backward prune treats the records
// of a frame's group in any order.
template <int K>
__device__ __forceinline__ unsigned long long warp_lat_reserve(const RunArgs& a, const bool (&want)[K], int l,
                                                               unsigned (&m)[K]) {
  const unsigned full = 0xffffffffu;
  uint32_t tot = 0;
#pragma unroll
  for (int k = 0; k < K; k++) {
    m[k] = __ballot_sync(full, want[k]);
    tot += __popc(m[k]);
  }
  unsigned long long b = 0;
  if (tot && (threadIdx.x & 31) == 0) b = atomicAdd(&a.w.lat_cnt[l], (unsigned long long)tot);
  return __shfl_sync(full, b, 0);
}
__device__ __forceinline__ void lat_put(const RunArgs& a, int l, unsigned long long p, const LatRec& r) {
  const DevWork& w = a.w;
  if (p < (unsigned long long)w.lat_cap) w.lat[(size_t)l * w.lat_stride + p] = r;
  else lane_ovf(a, l, kOvfArena);
}

// ------------------------------------------------------------------ emitting tiles

// MODE 0 (max): exact per-lane max of end over the frame's emitting arcs;
//   stages every token's score for MODE 1.
// MODE 1 (expand): admission against the cutoff + recombination into the
//   next frame.
template <int MODE, typename LP, int KIND>
__device__ void emit_tiles(const RunArgs& a, Smem& S) {
  constexpr bool ANC = KIND == kKindAnc;
  constexpr bool GEN = KIND == kKindGeneral;  // epsilon arcs and lattices possible
  const DevWork& w = a.w;
  const DevGraph& g = a.g;
  const bool lat = GEN && a.lattice;
  const int L = a.nlanes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WStage& ws = S.ws[warp];
  const int total = S.pre_a[L];
  const LP* lpb = reinterpret_cast<const LP*>(a.lp);
  const int nw = gridDim.x * kWarps;
  // the CTA's tiles, handed in order to whichever of its warps is free by a
  // shared-memory counter: in each of the R full rounds of nw tiles, the W
  // adjacent tiles b*W + j + i*nw (j < W); the last, partial round is dealt
  // out one tile per CTA in turn (tiles R*nw + b + m*G), so that no CTA holds
  // a whole extra group of W tiles while others have none
  const int rounds = total / nw;
  for (;;) {
    unsigned c_ = 0;
    if (lane == 0) c_ = atomicAdd(&S.tctr[MODE], 1u);
    c_ = __shfl_sync(0xffffffffu, c_, 0);
    const int tile = ((int)c_ < rounds * kWarps)
                         ? blockIdx.x * kWarps + (int)(c_ % kWarps) + (int)(c_ / kWarps) * nw
                         : rounds * nw + (int)blockIdx.x + ((int)c_ - rounds * kWarps) * (int)gridDim.x;
    if (tile >= total) break;
    const int l = find_lane(S.pre_a, L, tile);
    const int k = tile - S.pre_a[l];
    const SmLane& s = S.lane[l];
    const int f = s.t, par = f & 1;
    const int ntiles = S.pre_a[l + 1] - S.pre_a[l];
    const uint32_t s_lo = (uint32_t)k * kTile;
    const uint32_t s_hi = min(s_lo + (uint32_t)kTile, s.d_cur);
    // tokens [p_lo, p_hi) hold this tile's slots (tile 0 also takes the
    // arc-less tokens before the first slot); the tile owns [p_lo, own_hi):
    // every token of the frame is owned by exactly one tile, which commits it
    // in the max pass; the expand pass clears every staged token's entry
    const int32_t p_lo = (k == 0) ? 0 : __ldcg(w.tile_first + tl(w, par, l) + k);
    const int32_t own_hi = (k + 1 < ntiles) ? __ldcg(w.tile_first + tl(w, par, l) + k + 1) : s.n_cur;
    int32_t p_hi = (k + 1 < ntiles) ? own_hi + 1 : s.n_cur;
    if (p_hi > s.n_cur) p_hi = s.n_cur;
    const LP* row = lpb + (int64_t)s.row * a.stride_b + (int64_t)(f - s.t0) * a.stride_t;
    const size_t q = ql(w, par, l);
    const float maxlp = s.maxlp;
    // the skip threshold: an end already achieved (max) / the cutoff (expand)
    float thr = s.cutoff;
    if (MODE == 0) {
      unsigned ek = lane == 0 ? __ldcg(&fc_of(w, f, l)->maxkey) : 0u;
      ek = __shfl_sync(0xffffffffu, ek, 0);
      thr = ek ? unord_f(ek) : -INFINITY;
    }
    float vmax = -INFINITY;
    uint32_t admitted = 0;
    int32_t amin = 0x7fffffff, amax = -1;  // ancestor GC: the tile's committed tokens' ancestors
    uint32_t eps_n = 0;                    // epsilon arcs of the tile's committed tokens (statistic)
    for (int32_t c = p_lo; c < p_hi; c += kTokCap) {
      const int ntok = min(kTokCap, p_hi - c);
      __syncwarp();
#pragma unroll
      for (int r = 0; r < kTokCap / 32; r++) {
        const int i = r * 32 + lane;
        if (i < ntok) {
          const TokRec tr = ld_tok(w.front + q + c + i);
          float sc;
          if (MODE == 0) {
            const ulonglong2 e = ld_ent_keep(ent_at(w, l, tr.state, par));
            sc = key_score(e.x);
            w.score[q + c + i] = sc;
            const int32_t p = c + i;
            // a token that no other tile stages is cleared right after its
            // read (its line is in L2 now); the first token of tile k > 0 is
            // also staged by tile k-1 and is cleared by the expand pass
            if (!lat && p < own_hi && (p > p_lo || k == 0))
              *ent_at(w, l, tr.state, par) = make_ulonglong2(0ull, 0ull);
            if (s.need_commit && p < own_hi) {
              // commit (§5.4): the winners-log entry {delta, arc} of the token
              const int32_t arc = key_id(e.x);
              const uint32_t src = ent_src(e);
              const int64_t base_new = s.cursor, base_old = s.base_cur;
              const int64_t prev = ((src >> 31) ? base_new : base_old) + (src & 0x7fffffffu);
              wlog_commit(a, l, base_new + p, s.floor, arc, prev);
              if (GEN && g.has_eps) {
                const int4 m = __ldg(g.meta + tr.state);
                eps_n += (uint32_t)(m.z - m.y);
              }
              if (ANC) {
                const int32_t an = anc_of(f, arc, e.y, s.gc_c);
                w.anc[q + p] = an;
                amin = min(amin, an);
                amax = max(amax, an);
              }
            }
          } else {
            sc = __ldcg(w.score + q + c + i);
            if (ANC) ws.tpos[i] = __ldcg(w.anc + q + c + i);  // the token's checkpoint ancestor
            // entries the max pass left (lattices, tile-boundary tokens)
            if (lat || (c + i == p_lo && k > 0))
              *ent_at(w, l, tr.state, par) = make_ulonglong2(0ull, 0ull);
          }
          ws.off[i] = tr.off;
          ws.row[i] = tr.row;
          ws.score[i] = sc;
          ws.state[i] = tr.state;
          ws.ub[i] = __fadd_rn(__fadd_rn(sc, tr.maxw), maxlp);
        }
      }
      if (lane == 0) ws.off[ntok] = (c + ntok < s.n_cur) ? ld_tok(w.front + q + c + ntok).off : s.d_cur;
      __syncwarp();
      const uint32_t c_lo = max(s_lo, ws.off[0]);
      const uint32_t c_hi = min(s_hi, ws.off[ntok]);
      int ti[kSPT];
      bool act[kSPT];
      int32_t ai[kSPT];
#pragma unroll
      for (int j = 0; j < kSPT; j++) {
        const uint32_t slot = c_lo + (uint32_t)(j * 32 + lane);
        act[j] = slot < c_hi;
        ti[j] = act[j] ? find_tok(ws.off, ntok, slot) : 0;
        if (act[j] && a.ub_skip && ws.ub[ti[j]] <= thr) act[j] = false;
        ai[j] = act[j] ? ws.row[ti[j]] + (int32_t)(slot - ws.off[ti[j]]) : 0;
      }
      // one 16-byte record per arc {dst, weight, ilabel, arc id} (one vector
      // load); the expand pass finds the max pass's lines still in L2
      int il[kSPT];
      float wt[kSPT];
      int32_t d[kSPT], id[kSPT];
#pragma unroll
      for (int j = 0; j < kSPT; j++) {
        if (MODE == 0) {
          const int4 r = act[j] ? __ldg(g.arcs + ai[j]) : make_int4(0, 0, 0, 0);
          il[j] = r.z;
          wt[j] = __int_as_float(r.y);
          d[j] = id[j] = 0;
        } else {
          const int4 r = act[j] ? ld_arc(g.arcs + ai[j]) : make_int4(0, 0, 0, 0);
          d[j] = r.x;
          wt[j] = __int_as_float(r.y);
          il[j] = r.z;
          id[j] = r.w;
        }
      }
      float end[kSPT];
#pragma unroll
      for (int j = 0; j < kSPT; j++) {
        const float lpv = act[j] ? lp_at<LP>(row, il[j]) : 0.f;
        end[j] = act[j] ? __fadd_rn(__fadd_rn(ws.score[ti[j]], wt[j]), lpv) : -INFINITY;
        if (MODE == 1 && lat) wt[j] = __fadd_rn(wt[j], lpv);  // the record's own score
      }
      if (MODE == 0) {
#pragma unroll
        for (int j = 0; j < kSPT; j++) vmax = fmaxf(vmax, end[j]);
      } else {
        bool adm[kSPT], claim[kSPT];
#pragma unroll
        for (int j = 0; j < kSPT; j++) {
          adm[j] = act[j] && (end[j] > thr);
          if (!adm[j]) d[j] = id[j] = 0;
        }
        if (s.seed_next) {
          // an arc that attains this step's max makes its destination a best
          // token of the next frame: one chunk of that state's arcs posts an
          // achieved end of the next step before its max pass (§5.3
          // upper-bound skip) begins
          const LP* nrow = row + a.stride_t;
#pragma unroll
          for (int j = 0; j < kSPT; j++) {
            unsigned m32 = __ballot_sync(0xffffffffu, adm[j] && end[j] == s.cur_max);
            while (m32) {
              const int sl = __ffs(m32) - 1;
              m32 &= m32 - 1;
              const int32_t dd = __shfl_sync(0xffffffffu, d[j], sl);
              const float e0 = __shfl_sync(0xffffffffu, end[j], sl);
              const int4 m = __ldg(g.meta + dd);
              const int32_t ai = m.x + lane;
              float mx = -INFINITY;
              if (ai < m.y) {
                const int4 r = __ldg(g.arcs + ai);
                mx = __fadd_rn(__fadd_rn(e0, __int_as_float(r.y)), lp_at<LP>(nrow, r.z));
              }
              for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
              if (lane == 0 && mx > -INFINITY) atomicMax(&fc_of(w, f + 1, l)->maxkey, ord_f(mx));
            }
          }
        }
        if (lat) {
          unsigned lm[kSPT];
          unsigned long long lb = warp_lat_reserve<kSPT>(a, adm, l, lm);
          const unsigned lt = lanemask_lt();
#pragma unroll
          for (int j = 0; j < kSPT; j++) {
            if (adm[j]) {
              LatRec r;
              r.frame_flags = f << 4;
              r.src_tok = (int32_t)(s.base_cur + (c + ti[j]));
              r.dst_tok = -1;
              r.src_state = ws.state[ti[j]];
              r.dst_state = d[j];
              r.arc = id[j];
              r.end = end[j];
              r.arcscore = wt[j];
              lat_put(a, l, lb + __popc(lm[j] & lt), r);
            }
            lb += __popc(lm[j]);
          }
        }
        // the admitted candidates' entry lines, marked evict-last in L2: the
        // next max pass reads them again (and the next expand pass's CAS, for
        // a state that stays in the beam)
#pragma unroll
        for (int j = 0; j < kSPT; j++)
          if (adm[j]) prefetch_l2_keep(ent_at(w, l, d[j], par ^ 1));
#pragma unroll
        for (int j = 0; j < kSPT; j++) {
          const unsigned long long srcw =
              (unsigned long long)(uint32_t)(c + ti[j]) |
              (ANC ? (unsigned long long)(uint32_t)ws.tpos[ti[j]] << 32 : 0ull);
          claim[j] = adm[j] && relax_ent(a, ent_at(w, l, d[j], par ^ 1), mk_key(end[j], id[j]), srcw) == 2;
          admitted += adm[j] ? 1u : 0u;
        }
        warp_claim<kSPT, GEN>(a, claim, d, l, f + 1, true);
      }
    }
    if (MODE == 0) {
      for (int o = 16; o; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
      if (lane == 0 && vmax > -INFINITY) atomicMax(&fc_of(w, f, l)->maxkey, ord_f(vmax));
      if (GEN && g.has_eps) {  // one atomic per tile, not per token
        for (int o = 16; o; o >>= 1) eps_n += __shfl_xor_sync(0xffffffffu, eps_n, o);
        if (lane == 0 && eps_n) atomicAdd(&w.stats[l].eps, (unsigned long long)eps_n);
      }
      // the frame's ancestor bounds are read only at the GC's check frames
      if (ANC && f % a.gc_interval == 0) anc_post(a, l, f, amin, amax);
    } else {
      for (int o = 16; o; o >>= 1) admitted += __shfl_xor_sync(0xffffffffu, admitted, o);
      if (lane == 0 && admitted) atomicAdd(&w.stats[l].sum_a, (unsigned long long)admitted);
    }
  }
}

// ------------------------------------------------------------------ epsilon closure

// Relax the epsilon arcs of worklist `buf` (each closure lane's frame);
// improved or new states with epsilon arcs go to worklist buf^1, count slot
// `next_slot`, deduplicated by this pass's mark.
__device__ void eps_tiles(const RunArgs& a, Smem& S, int buf, int next_slot) {
  const DevWork& w = a.w;
  const DevGraph& g = a.g;
  const int L = a.nlanes;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  WStage& ws = S.ws[warp];
  const int total = S.pre_a[L];
  const int nw = gridDim.x * kWarps;
  // tiles dealt out across the CTAs first (tile t to CTA t mod G, warp
  // t / G of each round), so that a pass smaller than the grid spreads over
  // every SM instead of filling the first CTAs' warps
  for (int tile = warp * (int)gridDim.x + (int)blockIdx.x; tile < total; tile += nw) {
    const int l = find_lane(S.pre_a, L, tile);
    const int k = tile - S.pre_a[l];
    const SmLane& s = S.lane[l];
    const int fr = s.closure - 1;  // closure frame
    const int par = fr & 1;
    const int ntiles = S.pre_a[l + 1] - S.pre_a[l];
    const uint32_t s_lo = (uint32_t)k * kTile;
    const uint32_t s_hi = min(s_lo + (uint32_t)kTile, s.wl_e);
    const int32_t p_lo = __ldcg(w.wl_tile_first + tl(w, buf, l) + k);
    int32_t p_hi = (k + 1 < ntiles) ? __ldcg(w.wl_tile_first + tl(w, buf, l) + k + 1) + 1 : s.wl_n;
    if (p_hi > s.wl_n) p_hi = s.wl_n;
    const float cutoff = s.cutoff;
    const size_t q = ql(w, buf, l);
    const uint32_t pass_id = s.eps_pass + 1;
    for (int32_t c = p_lo; c < p_hi; c += kTokCap) {
      const int ntok = min(kTokCap, p_hi - c);
      __syncwarp();
#pragma unroll
      for (int r = 0; r < kTokCap / 32; r++) {
        const int i = r * 32 + lane;
        if (i < ntok) {
          const TokRec tr = ld_tok(w.wl + q + c + i);
          ws.off[i] = tr.off;
          ws.row[i] = tr.row;  // first epsilon arc
          ws.score[i] = key_score(__ldcg(&ent_at(w, l, tr.state, par)->x));
          ws.tpos[i] = __ldcg(tpos_at(w, l, tr.state, par));
          ws.state[i] = tr.state;
        }
      }
      if (lane == 0) ws.off[ntok] = (c + ntok < s.wl_n) ? ld_tok(w.wl + q + c + ntok).off : s.wl_e;
      __syncwarp();
      const uint32_t c_lo = max(s_lo, ws.off[0]);
      const uint32_t c_hi = min(s_hi, ws.off[ntok]);
      int ti[kSPT];
      bool act[kSPT];
      int32_t ai[kSPT];
#pragma unroll
      for (int j = 0; j < kSPT; j++) {
        const uint32_t slot = c_lo + (uint32_t)(j * 32 + lane);
        act[j] = slot < c_hi;
        ti[j] = act[j] ? find_tok(ws.off, ntok, slot) : 0;
        ai[j] = act[j] ? ws.row[ti[j]] + (int32_t)(slot - ws.off[ti[j]]) : 0;
      }
      float wt[kSPT], e[kSPT];
      bool adm[kSPT];
      int32_t d[kSPT], id[kSPT];
#pragma unroll
      for (int j = 0; j < kSPT; j++) {
        const int4 r = act[j] ? ld_arc(g.arcs + ai[j]) : make_int4(0, 0, 0, 0);
        d[j] = r.x;
        wt[j] = __int_as_float(r.y);
        id[j] = r.w;
      }
#pragma unroll
      for (int j = 0; j < kSPT; j++) {
        e[j] = __fadd_rn(ws.score[ti[j]], wt[j]);
        adm[j] = act[j] && (e[j] > cutoff);
        if (!adm[j]) d[j] = id[j] = 0;
      }
      if (a.lattice) {
        unsigned lm[kSPT];
        unsigned long long lb = warp_lat_reserve<kSPT>(a, adm, l, lm);
        const unsigned lt = lanemask_lt();
#pragma unroll
        for (int j = 0; j < kSPT; j++) {
          if (adm[j]) {
            LatRec r;
            r.frame_flags = (fr << 4) | kRecEps;
            r.src_tok = __float_as_int(ws.score[ti[j]]);  // score used; checked at resolution
            r.dst_tok = -1;
            r.src_state = ws.state[ti[j]];
            r.dst_state = d[j];
            r.arc = id[j];
            r.end = e[j];
            r.arcscore = wt[j];
            lat_put(a, l, lb + __popc(lm[j] & lt), r);
          }
          lb += __popc(lm[j]);
        }
      }
      bool claim[kSPT], better[kSPT];
#pragma unroll
      for (int j = 0; j < kSPT; j++)
        if (adm[j]) prefetch_l2_keep(ent_at(w, l, d[j], par));
#pragma unroll
      for (int j = 0; j < kSPT; j++) {
        const int r = adm[j] ? relax_ent(a, ent_at(w, l, d[j], par), mk_key(e[j], id[j]),
                                         0x80000000u | (uint32_t)ws.tpos[ti[j]])
                             : 0;
        claim[j] = r == 2;
        better[j] = r >= 1;
      }
      warp_claim<kSPT>(a, claim, d, l, fr, false);
      // improved states with epsilon arcs go to the next worklist once per
      // pass (the mark); a state this warp claimed is new in the frame, so
      // it is appended without waiting for the mark's old value (a later
      // improvement by another warp that misses the store appends it again:
      // the next pass relaxes it twice with the same score)
      bool wl[kSPT];
#pragma unroll
      for (int j = 0; j < kSPT; j++) {
        wl[j] = false;
        if (better[j]) {
          const int4 m = __ldg(g.meta + d[j]);
          if (m.z > m.y) {
            uint32_t* mk = w.mark + (size_t)l * w.N + d[j];
            if (claim[j]) {
              *mk = pass_id;
              wl[j] = true;
            } else {
              wl[j] = atomicExch(mk, pass_id) != pass_id;
            }
          }
        }
      }
      warp_append<kSPT, true>(wl, d, &w.wl_cnt[(size_t)next_slot * L + l], w.wl + ql(w, buf ^ 1, l),
                              w.wl_tile_first + tl(w, buf ^ 1, l), -1, w.qcap, a, l);
    }
  }
}

// Closure, to a fixpoint, of frame (s.closure - 1) of every lane with
// s.closure > 0, against s.cutoff.  Worklist W0 is in buffer 0 / count slot 0.
__device__ bool run_closure(const RunArgs& a, Smem& S, unsigned& epoch) {
  const DevWork& w = a.w;
  const int L = a.nlanes;
  const int tid = threadIdx.x;
  for (int k = 0;; k++) {
    const int buf = k & 1, slot = k % 3, next_slot = (k + 1) % 3, zero_slot = (k + 2) % 3;
    for (int l = tid; l < L; l += kThreads) {
      SmLane& s = S.lane[l];
      S.pre_a[l] = 0;
      if (s.closure) {
        const unsigned long long c = __ldcg(w.wl_cnt + (size_t)slot * L + l);
        if ((c >> 32) > (unsigned long long)w.qcap) {
          s.wl_n = 0;  // the worklist overflowed (lane already flagged)
          s.wl_e = 0;
        } else {
          s.wl_n = (int32_t)(c >> 32);
          s.wl_e = (uint32_t)c;
        }
        S.pre_a[l] = (int32_t)((s.wl_e + kTile - 1) / kTile);
      }
    }
    __syncthreads();
    lane_scan(S.pre_a, L);
    if (S.pre_a[L] == 0) break;
    if (k > a.g.eps_depth + 2) {  // cannot happen on an acyclic epsilon subgraph
      if (tid == 0 && blockIdx.x == 0) atomicOr(&w.bar->error, 2u);
      break;
    }
    if (blockIdx.x == 0)
      for (int l = tid; l < L; l += kThreads)
        if (S.lane[l].closure) w.wl_cnt[(size_t)zero_slot * L + l] = 0ull;
    if (tid == 0) S.eps_passes++;
    eps_tiles(a, S, buf, next_slot);
    __syncthreads();
    for (int l = tid; l < L; l += kThreads)
      if (S.lane[l].closure) S.lane[l].eps_pass += 1;
    if (!grid_sync(a, S, epoch)) return false;
  }
  for (int l = tid; l < L; l += kThreads)
    if (S.lane[l].closure) S.lane[l].eps_pass += 1;
  __syncthreads();
  return true;
}

// ------------------------------------------------------------------ winners-log GC

// The chain walk of an ancestor-GC cut of lane l at entry E (one thread):
// follows the winners chain from E down to the root (one load per hop) and
// keeps its arcs newest first in the lane's path buffer.  Returns the number
// of arcs, or -1 for no cut (an overflowed lane, an E that is not above the
// root, a chain longer than the path buffer).  The entries it reads were
// committed in earlier steps and are not written again before the cut, so
// the walk may run while the step's expand pass is under way.
__device__ int gc_walk(const RunArgs& a, const SmLane& s, int l, int64_t E) {
  const DevWork& w = a.w;
  int32_t* path = w.path + (size_t)l * (size_t)w.path_cap;
  const int64_t root = s.floor, hi = s.cursor;
  if ((__ldcg(&w.lanes[l].overflow) & (kOvfArena | kOvfKept | kOvfPath)) || E <= root || E >= hi) return -1;
  int n = 0;
  int64_t i = E;
  while (i > root && i < hi) {
    const int2 e = __ldcg(wlog_at(w, l, i));
    if (e.y < 0) break;
    if (n >= w.path_cap) return -1;  // longer than the buffer: no cut
    path[n++] = e.y;
    i -= sext30((uint32_t)e.x);
  }
  return n;
}

// Cut lane l's winners log at entry E (the whole CTA): the words of the path
// from the root up to E are appended to the lane's finalized words, E becomes
// the root (arc -1, no predecessor) and the ring below it is free.  The chain
// walk (gc_walk) is either done here by thread 0 (n_pre = -2) or was done
// earlier in the step by this CTA's thread 0 (n_pre its result); the CTA
// then looks the arcs' output labels up and packs the words oldest first.
// The kept path of the lane (partial backtracks splice with it) reaches below
// E, so it is dropped.  Lanes whose log, frontier or path overflowed are left
// alone.
__device__ void gc_cut(const RunArgs& a, Smem& S, int l, int64_t E, int n_pre) {
  const DevWork& w = a.w;
  const DevGraph& g = a.g;
  const SmLane& s = S.lane[l];
  const int tid = threadIdx.x;
  int32_t* path = w.path + (size_t)l * (size_t)w.path_cap;
  if (tid == 0) {
    int n = n_pre >= -1 ? n_pre : gc_walk(a, s, l, E);
    if (__ldcg(&w.lanes[l].overflow) & (kOvfArena | kOvfKept | kOvfPath)) n = -1;
    if (n >= 0) {
      w.lanes[l].bt_top = -1;
      w.lanes[l].bt_len = 0;
    }
    S.bt_n = n;
  }
  __syncthreads();
  const int n = S.bt_n;
  if (n < 0) return;
  // words, oldest arc first: path[n-1] .. path[0]
  int32_t* fin = w.fin + (size_t)l * (size_t)w.fin_cap;
  int run = s.fin_n;
  for (int base = 0; base < n; base += kThreads) {
    const int j = base + tid;
    const int32_t o = j < n ? __ldg(g.c_olabel + __ldcg(path + (n - 1 - j))) : 0;
    const unsigned bal = __ballot_sync(0xffffffffu, o != 0);
    if ((tid & 31) == 0) S.scan_tmp[tid >> 5] = __popc(bal);
    __syncthreads();
    int wbase = 0, tot = 0;
    for (int ww = 0; ww < kWarps; ww++) {
      if (ww < (tid >> 5)) wbase += S.scan_tmp[ww];
      tot += S.scan_tmp[ww];
    }
    const int pos = run + wbase + __popc(bal & lanemask_lt());
    if (o != 0 && pos < w.fin_cap) fin[pos] = o;
    run += tot;
    __syncthreads();
  }
  if (tid == 0) {
    if ((int64_t)run > w.fin_cap) {
      lane_ovf(a, l, kOvfPath);  // no room for the finalized words: no cut
    } else {
      *wlog_at(w, l, E) = make_int2(0, -1);
      w.lanes[l].floor = E;
      w.lanes[l].fin_n = run;
    }
  }
}

// One winners-log GC round of lane l (§6.3 "Winners-log GC", §8.1 "Per-chunk
// GC"), run by one CTA at the end of a step.  Frame t's tokens are the
// entries [base_cur, cursor) and every live chain passes through one of them.
//   1. thread 0 marks the first token's chain (the anchor chain) back to the
//      root, writing each entry's depth on the chain into it and keeping its
//      delta in the lane's path buffer (free here: the next backtrack walks
//      the whole tail again);
//   2. every other token walks its own chain, marking it, until it meets a
//      marked entry; meeting the anchor chain posts that entry's depth.  The
//      deepest such entry E is on every chain: each chain joins the anchor
//      chain at or above E and follows it from there (a chain that meets
//      another walk follows that walk to its meeting point);
//   3. the marks are cleared and the anchor chain's deltas restored;
//   4. the words of the path from the root up to E are appended to the
//      lane's finalized words, E becomes the root (arc -1, no predecessor)
//      and the ring below it is free.
// Depth, not index, orders the meeting points: an epsilon arc's source token
// can sit at a later position of the same frame.  Walks are capped at H hops
// (a few GC intervals of frames): if some chain has not met the anchor chain
// within H hops the chains have not converged yet and the round cuts nothing.
// Lanes whose log, frontier or path overflowed are left alone.
__device__ void gc_round(const RunArgs& a, Smem& S, int l) {
  const DevWork& w = a.w;
  const DevGraph& g = a.g;
  const SmLane& s = S.lane[l];
  const int tid = threadIdx.x;
  const int64_t lo = s.base_cur, hi = s.cursor, root = s.floor;
  const int64_t max_hops = hi - root;
  const int64_t H = min((int64_t)w.path_cap - 1,
                        (int64_t)(4 * a.gc_interval + 64) * (1 + (int64_t)g.eps_depth));
  int32_t* keep = w.path + (size_t)l * (size_t)w.path_cap;  // anchor-chain deltas by depth
  if (tid == 0) {
    S.gc_min = 0;   // deepest meeting depth (the anchor itself: 0)
    S.gc_nw = 0;    // anchor-chain entries marked
    S.gc_ok = ((__ldcg(&w.lanes[l].overflow) & (kOvfArena | kOvfKept | kOvfPath)) == 0 && root <= lo &&
               lo < hi && hi - root <= w.log_cap) ? 1 : 0;
    if (S.gc_ok) {
      int64_t i = lo;
      for (int32_t dep = 0; dep <= H; dep++) {
        if (i < root || i >= hi || dep > max_hops) { S.gc_ok = 0; break; }
        int2* p = wlog_at(w, l, i);
        const int2 e = __ldcg(p);
        keep[dep] = e.x;
        p->x = (int32_t)(kMarkAnchor | (uint32_t)dep);
        S.gc_nw = dep + 1;
        if (e.y < 0) break;  // the root
        const int32_t dl = sext30((uint32_t)e.x);
        if (dl == 0) { S.gc_ok = 0; break; }
        i -= dl;
      }
    }
  }
  __threadfence();  // marks reach L2 before the walks read them
  __syncthreads();
  const bool run = S.gc_ok != 0;
  if (run) {
    for (int64_t x = lo + 1 + tid; x < hi; x += kThreads) {
      int64_t i = x;
      bool met = false;
      for (int64_t h = 0; h <= H && i >= root && i < hi; h++) {
        int2* p = wlog_at(w, l, i);
        const int2 e = __ldcg(p);
        const uint32_t dx = (uint32_t)e.x;
        if (dx & kMarkAnchor) {
          atomicMax(&S.gc_min, (unsigned long long)(dx & kDeltaMask));
          met = true;
          break;
        }
        if (dx & kMarkWalk) {  // another walk continues from here
          met = true;
          break;
        }
        p->x = (int32_t)(dx | kMarkWalk);
        const int32_t dl = sext30(dx);
        if (e.y < 0 || dl == 0) break;  // (an unmarked root cannot occur)
        i -= dl;
      }
      if (!met) S.gc_ok = 0;  // not converged within H hops: no cut this round
    }
  }
  __threadfence();
  __syncthreads();
  if (run) {  // clear the walks' marks (each walk ends where its own marks end)
    for (int64_t x = lo + 1 + tid; x < hi; x += kThreads) {
      int64_t i = x;
      for (int64_t h = 0; h <= H && i >= root && i < hi; h++) {
        int2* p = wlog_at(w, l, i);
        const uint32_t dx = (uint32_t)__ldcg(&p->x);
        if (!(dx & kMarkWalk)) break;
        const uint32_t cx = dx & ~kMarkWalk;
        p->x = (int32_t)cx;
        const int32_t dl = sext30(cx);
        if (dl == 0) break;
        i -= dl;
      }
    }
  }
  if (tid == 0) {  // restore the anchor chain; E = its entry at the deepest meeting depth
    int64_t i = lo, E = -1;
    for (int32_t dep = 0; dep < S.gc_nw; dep++) {
      const int32_t x = keep[dep];
      wlog_at(w, l, i)->x = x;
      if ((unsigned long long)dep == S.gc_min) E = i;
      i -= sext30((uint32_t)x);
    }
    S.bt_idx = E;
    w.lanes[l].bt_top = -1;  // the path buffer was scratch space
    w.lanes[l].bt_len = 0;
  }
  __threadfence();
  __syncthreads();
  if (run && S.gc_ok) gc_cut(a, S, l, S.bt_idx, -2);
  __syncthreads();
}

// ------------------------------------------------------------------ lane setup

__device__ void init_lane_global(const RunArgs& a, int l) {
  const DevWork& w = a.w;
  const DevGraph& g = a.g;
  FrameCnt z;
  z.cnt = 0; z.maxkey = 0; z.admitted = 0; z.final_key = 0; z.best_key = 0; z.anc_hi = 0; z.anc_lo = 0;
  for (int r = 0; r < 4; r++) w.fcnt[(size_t)r * w.L + l] = z;
  for (int r = 0; r < 3; r++) w.wl_cnt[(size_t)r * w.L + l] = 0ull;
  if (w.lattice) {
    w.lat_cnt[l] = 0ull;
    w.lat_out_n[l] = 0ull;
  }
  w.lanes[l].overflow = 0;
  w.lanes[l].bt_top = -1;  // no path to continue from
  w.lanes[l].bt_len = 0;
  w.lanes[l].floor = 0;
  w.lanes[l].fin_n = 0;
  const int32_t s0 = g.start;
  const int4 m = __ldg(g.meta + s0);
  const uint32_t deg = (uint32_t)(m.y - m.x);
  *ent_at(w, l, s0, 0) = make_ulonglong2(mk_key(0.0f, -1), 0ull);
  if (tpos_kept(a)) *tpos_at(w, l, s0, 0) = 0;
  *reinterpret_cast<int4*>(w.front + ql(w, 0, l)) = make_int4(s0, 0, m.x, m.w);
  if (deg > 0)
    for (uint32_t k = 0; k <= (deg - 1) / kTile; k++) w.tile_first[tl(w, 0, l) + k] = 0;
  w.fcnt[l].cnt = (1ull << 32) | deg;
  if (g.has_eps && m.z > m.y) {
    const uint32_t edeg = (uint32_t)(m.z - m.y);
    *reinterpret_cast<int4*>(w.wl + ql(w, 0, l)) = make_int4(s0, 0, m.y, 0);
    for (uint32_t k = 0; k <= (edeg - 1) / kTile; k++) w.wl_tile_first[tl(w, 0, l) + k] = 0;
    w.wl_cnt[l] = (1ull << 32) | edeg;
  }
}

// Row maxima of the call's log-probs (one warp per row): the acoustic half
// of the per-token upper bound.
template <typename LP>
__device__ void row_maxima(const RunArgs& a, Smem& S) {
  const DevWork& w = a.w;
  const int L = a.nlanes;
  const int total = S.pre_a[L];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const LP* lpb = reinterpret_cast<const LP*>(a.lp);
  const int V = a.g.V;
  for (int r = blockIdx.x * kWarps + warp; r < total; r += gridDim.x * kWarps) {
    const int l = find_lane(S.pre_a, L, r);
    const int j = r - S.pre_a[l];
    const LP* row = lpb + (int64_t)S.lane[l].row * a.stride_b + (int64_t)j * a.stride_t;
    float m = -INFINITY;
    for (int v = lane; v < V; v += 32) m = fmaxf(m, lp_at<LP>(row, v));
    for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) w.maxlp[(size_t)l * w.max_frames + j] = m;
  }
}

// ------------------------------------------------------------------ lattice prune

// Backward max-plus sweep over persisted records, group by group, for every
// lane with s.closure set.  Append order per lane: R_{-1} = eps(0), then for
// t = 0..T-1 R_t = emit(t) + eps(t+1), then R_T = final(T) (+ redirect);
// B_t (the start of R_t) is recorded in lat_groups during frame t's commit.
//   final sweep: group 0 = R_T, then for k = 0, 1, ...: the epsilon records
//     (k even) or the emitting records (k odd) of R_{T-1-k/2}, down to R_{-1};
//   interval sweep: the same from R_{s.t-1} down to R_{s.res_hi}.
// bwd[src] = max over the group's records of arcscore + bwd[dst] (dst -1:
// the super-final node, 0).  Epsilon groups repeat until nothing changes.
__device__ bool bwd_sweep(const RunArgs& a, Smem& S, unsigned& epoch, bool final_mode) {
  const DevWork& w = a.w;
  const DevGraph& g = a.g;
  const int L = a.nlanes;
  const int tid = threadIdx.x;
  const int64_t gstride = (int64_t)gridDim.x * kThreads;
  const int64_t gstart = (int64_t)blockIdx.x * kThreads + tid;
  if (blockIdx.x == 0 && tid < 3) w.bar->changed[tid] = 0u;
  if (!grid_sync(a, S, epoch)) return false;
  int maxg = 0;
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (s.closure) maxg = max(maxg, final_mode ? 2 * s.t + 2 : 2 * (s.t - (int)s.res_hi));
  }
  int pass_no = 0;
  for (int j = 0; j < maxg; j++) {
    const int kk = final_mode ? j - 1 : j;     // -1: the final group
    const bool eps_group = kk >= 0 && (kk & 1) == 0;
    if (eps_group && !g.has_eps) continue;
    const int npass = eps_group ? g.eps_depth + 2 : 1;
    for (int pass = 0; pass < npass; pass++, pass_no++) {
      const int fl = pass_no % 3;
      if (blockIdx.x == 0 && tid == 0) w.bar->changed[(pass_no + 1) % 3] = 0u;
      // this group's record range of every lane, flattened into one index
      // space so that all lanes' records are spread over the whole grid
      for (int l = tid; l < L; l += kThreads) {
        const SmLane& s = S.lane[l];
        int64_t lo = 0, hi = 0;
        if (s.closure) {
          const int64_t* B = w.lat_groups + (size_t)l * (w.max_frames + 2);
          if (kk < 0) {
            lo = B[s.t];
            hi = (int64_t)min(__ldcg(&w.lat_cnt[l]), (unsigned long long)w.lat_cap);
          } else {
            const int r = s.t - 1 - kk / 2;  // R_r
            const int r_bot = final_mode ? -1 : (int)s.res_hi;
            if (r >= r_bot) {
              lo = (r < 0) ? 0 : B[r];
              hi = B[r + 1];
            }
          }
        }
        S.glo[l] = lo;
        S.pre_e[l] = (int32_t)max((int64_t)0, hi - lo);
      }
      __syncthreads();
      lane_scan(S.pre_e, L);
      const int gtotal = S.pre_e[L];
      for (int gi = (int)gstart; gi < gtotal; gi += (int)gstride) {
        const int l = find_lane(S.pre_e, L, gi);
        const int64_t r = S.glo[l] + (gi - S.pre_e[l]);
        const LatRec rec = w.lat[(size_t)l * w.lat_stride + r];
        const int flags = rec.frame_flags & 15;
        if (flags & kRecDead) continue;
        if (kk >= 0 && (((flags & kRecEps) != 0) != eps_group)) continue;
        uint32_t* bw = w.bwd + (size_t)l * w.log_stride;
        const float bd = rec.dst_tok < 0 ? 0.0f : unord_f(__ldcg(bw + rec.dst_tok));
        const unsigned ov = ord_f(__fadd_rn(rec.arcscore, bd));
        const unsigned old = atomicMax(bw + rec.src_tok, ov);
        if (eps_group && ov > old) w.bar->changed[fl] = 1u;
      }
      if (!grid_sync(a, S, epoch)) return false;
      if (eps_group && ld_acquire(&w.bar->changed[fl]) == 0u) break;
    }
  }
  return true;
}

// Backward scores over the persisted records of every lane with s.closure
// set (the final sweep), then the keep test (§3: output_beam acts only
// here) and compaction of the kept records.
__device__ bool lattice_prune(const RunArgs& a, Smem& S, unsigned& epoch) {
  const DevWork& w = a.w;
  const int L = a.nlanes;
  const int tid = threadIdx.x;
  const int64_t gstride = (int64_t)gridDim.x * kThreads;
  const int64_t gstart = (int64_t)blockIdx.x * kThreads + tid;
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (!s.closure) continue;
    const int64_t n = min(s.cursor, w.log_cap);
    uint32_t* bw = w.bwd + (size_t)l * w.log_stride;
    for (int64_t i = gstart; i < n; i += gstride) bw[i] = ord_f(-INFINITY);
  }
  if (!bwd_sweep(a, S, epoch, true)) return false;
  // keep test and compaction
  const int lane = tid & 31;
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (!s.closure) continue;
    const float thr = __fsub_rn(__ldcg(&w.res[l].score), a.output_beam);
    const int64_t hi = (int64_t)min(__ldcg(&w.lat_cnt[l]), (unsigned long long)w.lat_cap);
    const LatRec* R = w.lat + (size_t)l * w.lat_stride;
    const uint32_t* bw = w.bwd + (size_t)l * w.log_stride;
    for (int64_t base = (int64_t)blockIdx.x * kThreads + (tid & ~31); base < hi; base += gstride) {
      const int64_t r = base + lane;
      bool keep = false;
      LatRec rec;
      if (r < hi) {
        rec = R[r];
        if (!(rec.frame_flags & kRecDead)) {
          const float bd = rec.dst_tok < 0 ? 0.0f : unord_f(__ldcg(bw + rec.dst_tok));
          keep = __fadd_rn(rec.end, bd) >= thr;
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, keep);
      if (m) {
        const int ld = __ffs(m) - 1;
        unsigned long long b = 0;
        if (lane == ld) b = atomicAdd(&w.lat_out_n[l], (unsigned long long)__popc(m));
        b = __shfl_sync(0xffffffffu, b, ld);
        if (keep) w.lat_out[(size_t)l * w.lat_stride + b + __popc(m & lanemask_lt())] = rec;
      }
    }
  }
  return true;
}

// Interval lattice prune (§7 lat_prune_interval) of the lanes with s.closure
// set, right after frame t = s.t was committed (its tokens are the winners-
// log entries [s.cursor, s.cursor + s.n_cur) and their entries still hold
// their final scores).  Only records the final prune can never keep are
// dropped: every frontier token u of frame t starts at beta(u) = -score(u),
// beta flows backward over the groups R_r, r in [max(-1, t - 2N), t - 1]
// (the window), and a window record stays iff beta(dst) > -inf and
// end + beta(dst) >= -((output_beam + 1) + 2^-12 |M|), M the exact max of
// the step that made frame t.  A complete path through a record passes one
// token u of frame t and its prefix up to u scores at most score(u), so
// end + beta(dst) is minus the least amount by which a path through the
// record falls behind the best path into its frontier token; the final
// prune keeps only records within output_beam of the best complete path.
// The margin covers fp32 rounding.  Survivors are compacted group by group
// through the lane's lat_out region (unused until the final prune) and the
// group bounds B_r rewritten.
__device__ bool interval_prune(const RunArgs& a, Smem& S, unsigned& epoch) {
  const DevWork& w = a.w;
  const int L = a.nlanes;
  const int tid = threadIdx.x;
  const int64_t gstride = (int64_t)gridDim.x * kThreads;
  const int64_t gstart = (int64_t)blockIdx.x * kThreads + tid;
  const int N = a.lat_interval;
  const size_t mf = (size_t)w.max_frames + 2;
  for (int l = tid; l < L; l += kThreads) {
    SmLane& s = S.lane[l];
    if (!s.closure) continue;
    s.res_hi = max(-1, s.t - 2 * N);                 // the window's oldest group
    s.res_lo = w.lat_groups[(size_t)l * mf + s.t];  // the window's end before compaction
  }
  __syncthreads();
  // (1) beta of every node a window record touches: -inf; group counters 0
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (!s.closure) continue;
    const int64_t* B = w.lat_groups + (size_t)l * mf;
    const int64_t lo = s.res_hi < 0 ? 0 : B[s.res_hi], hi = B[s.t];
    const LatRec* R = w.lat + (size_t)l * w.lat_stride;
    uint32_t* bw = w.bwd + (size_t)l * w.log_stride;
    for (int64_t r = lo + gstart; r < hi; r += gstride) {
      const LatRec rec = R[r];
      if (rec.frame_flags & kRecDead) continue;
      bw[rec.src_tok] = ord_f(-INFINITY);
      bw[rec.dst_tok] = ord_f(-INFINITY);
    }
    if (blockIdx.x == 0)
      for (int k = tid; k <= s.t - (int)s.res_hi; k += kThreads) w.lat_gtmp[(size_t)l * mf + k] = 0;
  }
  if (!grid_sync(a, S, epoch)) return false;
  // (2) the frontier: beta(u) = -score(u)
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (!s.closure) continue;
    const int par = s.t & 1;
    uint32_t* bw = w.bwd + (size_t)l * w.log_stride;
    for (int64_t p = gstart; p < s.n_cur; p += gstride) {
      const int32_t st = __ldcg(&w.front[ql(w, par, l) + p].state);
      const float sc = key_score(__ldcg(&ent_at(w, l, st, par)->x));
      bw[s.cursor + p] = ord_f(-sc);
    }
  }
  // (3) backward over the window's groups
  if (!bwd_sweep(a, S, epoch, false)) return false;
  // (4) the keep test; surviving records counted per group
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (!s.closure) continue;
    const unsigned mk = __ldcg(&fc_of(w, s.t - 1, l)->maxkey);
    const float M = mk ? unord_f(mk) : -INFINITY;
    const float lim = -__fadd_rn(__fadd_rn(a.output_beam, 1.0f), __fmul_rn(0x1p-12f, fabsf(M)));
    const int64_t* B = w.lat_groups + (size_t)l * mf;
    const int64_t lo = s.res_hi < 0 ? 0 : B[s.res_hi], hi = B[s.t];
    LatRec* R = w.lat + (size_t)l * w.lat_stride;
    const uint32_t* bw = w.bwd + (size_t)l * w.log_stride;
    for (int64_t r = lo + gstart; r < hi; r += gstride) {
      const LatRec rec = R[r];
      bool keep = false;
      if (!(rec.frame_flags & kRecDead)) {
        const float bd = unord_f(__ldcg(bw + rec.dst_tok));
        keep = bd > -INFINITY && __fadd_rn(rec.end, bd) >= lim;
      }
      if (keep) {
        const int grp = (rec.frame_flags >> 4) - ((rec.frame_flags & kRecEps) ? 1 : 0);
        atomicAdd(reinterpret_cast<unsigned long long*>(w.lat_gtmp) + (size_t)l * mf + (grp - (int)s.res_hi), 1ull);
      } else {
        R[r].frame_flags = rec.frame_flags | kRecDead;
      }
    }
  }
  if (!grid_sync(a, S, epoch)) return false;
  // (5) new group starts (one thread per lane): B_r, and each group's
  //     counter becomes its write cursor
  if (blockIdx.x == 0)
    for (int l = tid; l < L; l += kThreads) {
      const SmLane& s = S.lane[l];
      if (!s.closure) continue;
      int64_t* B = w.lat_groups + (size_t)l * mf;
      int64_t* cnt = w.lat_gtmp + (size_t)l * mf;
      const int r0 = (int)s.res_hi;
      int64_t pos = r0 < 0 ? 0 : B[r0];
      for (int r = r0; r < s.t; r++) {
        const int64_t c = cnt[r - r0];
        cnt[r - r0] = pos;
        if (r >= 0) B[r] = pos;
        pos += c;
      }
      B[s.t] = pos;
      w.lat_cnt[l] = (unsigned long long)pos;
    }
  if (!grid_sync(a, S, epoch)) return false;
  // (6) survivors into the lane's lat_out region at their new positions
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (!s.closure) continue;
    const int64_t lo = s.res_hi < 0 ? 0 : w.lat_groups[(size_t)l * mf + s.res_hi];  // unchanged by (5)
    const int64_t hi = s.res_lo;
    const LatRec* R = w.lat + (size_t)l * w.lat_stride;
    LatRec* O = w.lat_out + (size_t)l * w.lat_stride;
    unsigned long long* cur = reinterpret_cast<unsigned long long*>(w.lat_gtmp) + (size_t)l * mf;
    for (int64_t r = lo + gstart; r < hi; r += gstride) {
      const LatRec rec = R[r];
      if (rec.frame_flags & kRecDead) continue;
      const int grp = (rec.frame_flags >> 4) - ((rec.frame_flags & kRecEps) ? 1 : 0);
      const unsigned long long p = atomicAdd(cur + (grp - (int)s.res_hi), 1ull);
      O[p - lo] = rec;
    }
  }
  if (!grid_sync(a, S, epoch)) return false;
  // (7) back into the arena
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (!s.closure) continue;
    const int64_t* B = w.lat_groups + (size_t)l * mf;
    const int64_t lo = s.res_hi < 0 ? 0 : B[s.res_hi], hi = B[s.t];
    LatRec* R = w.lat + (size_t)l * w.lat_stride;
    const LatRec* O = w.lat_out + (size_t)l * w.lat_stride;
    for (int64_t r = lo + gstart; r < hi; r += gstride) R[r] = O[r - lo];
  }
  return grid_sync(a, S, epoch);
}

// ------------------------------------------------------------------ the kernel

// Dynamic shared memory of a launch over L lanes, and the carving of it.
__host__ __device__ inline size_t smem_lane_offset() { return (sizeof(Smem) + 15) & ~(size_t)15; }
__host__ __device__ inline size_t smem_size(int L) {
  size_t o = smem_lane_offset() + (size_t)L * sizeof(SmLane);
  o += 5 * (size_t)(L + 1) * sizeof(int32_t);
  o = (o + 7) & ~(size_t)7;
  return o + (size_t)L * sizeof(int64_t);
}
__device__ inline void smem_carve(Smem& S, unsigned char* raw, int L) {
  unsigned char* p = raw + smem_lane_offset();
  S.lane = reinterpret_cast<SmLane*>(p);
  p += (size_t)L * sizeof(SmLane);
  int32_t* q = reinterpret_cast<int32_t*>(p);
  S.pre_a = q; q += L + 1;
  S.pre_b = q; q += L + 1;
  S.pre_c = q; q += L + 1;
  S.pre_d = q; q += L + 1;
  S.pre_e = q; q += L + 1;
  p = reinterpret_cast<unsigned char*>(q);
  p = reinterpret_cast<unsigned char*>(((size_t)p + 7) & ~(size_t)7);
  S.glo = reinterpret_cast<int64_t*>(p);
}

// KIND (see Kind): kKindAnc runs the ancestor GC (the winners-log GC of an
// epsilon-free graph), kKindPlain an epsilon-free graph without lattices or
// GC, kKindGeneral everything else; separate instantiations, so that each
// carries only the registers its own code needs.
template <typename LP, int KIND>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(const RunArgs a) {
  constexpr bool ANC = KIND == kKindAnc;
  constexpr bool GEN = KIND == kKindGeneral;  // epsilon arcs, lattices, the walking GC round
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  if (threadIdx.x == 0) smem_carve(S, smem_raw, a.nlanes);
  __syncthreads();
  const DevWork& w = a.w;
  const DevGraph& g = a.g;
  const int L = a.nlanes;
  const int tid = threadIdx.x;
  const int G = gridDim.x;
  const int64_t gstride = (int64_t)G * kThreads;
  const int64_t gstart = (int64_t)blockIdx.x * kThreads + tid;
  const bool lat = GEN && a.lattice != 0;
  unsigned epoch = 0;
  unsigned long long steps = 0;
  unsigned long long* prof = S.prof;
  if (tid < kProfSlots) prof[tid] = 0;
  if (tid < 2) S.tctr[tid] = 0u;
  if (tid == 0) S.eps_passes = 0u;
  if (tid == 0) prof[kProfSlots] = prof[kProfSlots + 1] = gtimer();
  const int tlast = 0, tsub = 1;

  // ---- lane mirrors (every CTA holds an identical copy)
  for (int l = tid; l < L; l += kThreads) {
    SmLane& s = S.lane[l];
    const LaneState st = w.lanes[l];
    const LaneCall c = a.calls[l];
    s.t = st.t;
    s.committed = st.committed;
    s.status = st.status;
    s.beam = st.beam;
    s.cursor = st.cursor;
    s.base_cur = st.base_cur;
    s.base_prev = st.base_prev;
    s.eps_pass = st.eps_pass;
    s.t_eff = st.t_eff;
    s.floor = st.floor;
    s.fin_n = st.fin_n;
    s.gc_t = st.gc_t;
    s.gc_due = 0;
    s.gc_c = st.gc_c;
    s.gc_cbase = st.gc_cbase;
    s.gc_e = 0;
    s.log_hw = 0;
    s.row = c.row;
    s.flags = c.row >= 0 ? c.flags : 0;
    s.phase = kNone;
    s.need_commit = 0;
    s.done_final = s.done_partial = 0;
    s.frames = s.sum_n = s.sum_d = s.sum_m = 0;
    s.was_emit = 0;
    s.closure = 0;
    s.cutoff = 0.f;
    s.n_cur = s.n_prev = 0;
    s.prev_cleared = 0;  // not known at launch: the first step clears as well
    s.d_cur = 0;
    if (s.flags & kCallInit) {
      s.t = 0;
      s.committed = -1;
      s.status = kLaneRunning;
      s.beam = a.search_beam;
      s.cursor = s.base_cur = s.base_prev = 0;
      s.t_eff = c.t_eff;
      s.floor = 0;
      s.fin_n = 0;
      s.gc_t = 0;
      s.gc_c = 0;
      s.gc_cbase = 0;
    }
    s.t0 = s.t;
    s.t_end = s.t + (c.row >= 0 ? c.nframes : 0);
    S.pre_a[l] = (c.row >= 0 && s.status == kLaneRunning) ? c.nframes : 0;
  }
  __syncthreads();

  // ---- lane initialisation and the call's row maxima, then the start
  //      frontier's closure (cutoff 0 - search_beam)
  lane_scan(S.pre_a, L);
  if (tid == 0) {
    int any = 0;
    for (int l = 0; l < L; l++) any |= (S.lane[l].flags & kCallInit);
    S.any = any;
    S.flag = S.pre_a[L] > 0;
  }
  __syncthreads();
  if (S.any || S.flag) {
    if (tid == 0)
      for (int l = blockIdx.x; l < L; l += G)
        if (S.lane[l].flags & kCallInit) init_lane_global(a, l);
    row_maxima<LP>(a, S);
    if (!grid_sync(a, S, epoch)) return;
    if (S.any && (GEN && g.has_eps)) {
      for (int l = tid; l < L; l += kThreads) {
        SmLane& s = S.lane[l];
        s.closure = (s.flags & kCallInit) ? 1 : 0;  // frame 0
        s.cutoff = __fsub_rn(0.0f, a.search_beam);
      }
      __syncthreads();
      if (!run_closure(a, S, epoch)) return;
      for (int l = tid; l < L; l += kThreads) S.lane[l].closure = 0;
      __syncthreads();
    }
  }
  prof_mark(prof, tlast, kProfInit);

  // ---- the frame loop
  for (;;) {
    // prologue: each lane's phase and frame sizes (identical in every CTA;
    // the counters it reads are final since the last barrier)
    for (int l = tid; l < L; l += kThreads) {
      SmLane& s = S.lane[l];
      s.phase = kNone;
      s.need_commit = 0;
      S.pre_a[l] = S.pre_b[l] = S.pre_c[l] = S.pre_d[l] = 0;
      s.res_lo = s.res_hi = 0;
      if (s.row < 0 || s.status != kLaneRunning) continue;
      // the step's global reads, issued together
      const unsigned long long cnt = __ldcg(&fc_of(w, s.t, l)->cnt);
      const unsigned long long cp = s.t >= 1 ? __ldcg(&fc_of(w, s.t - 1, l)->cnt) : 0ull;
      const float mlp = s.t < s.t_end ? __ldcg(w.maxlp + (size_t)l * w.max_frames + (s.t - s.t0)) : 0.f;
      if (s.was_emit) s.sum_m += cnt >> 32;
      s.was_emit = 0;
      if (s.gc_due) {  // a GC round of the last step moved the root and finalized words
        s.floor = __ldcg(&w.lanes[l].floor);
        s.fin_n = __ldcg(&w.lanes[l].fin_n);
        s.gc_due = 0;
      }
      if (s.t < s.t_end) s.phase = kEmit;
      else if ((s.flags & kCallFinal) && !s.done_final) s.phase = kFin;
      else if ((s.flags & kCallPartial) && !(s.flags & kCallFinal) && !s.done_partial) s.phase = kPart;
      if (s.phase == kNone) continue;
      const unsigned long long n_raw = cnt >> 32;
      s.n_cur = (int32_t)min(n_raw, (unsigned long long)w.qcap);
      s.d_cur = (uint32_t)cnt;
      if (n_raw > (unsigned long long)w.qcap) {
        // tokens past the capacity were dropped: their slots are the tail
        const TokRec r = ld_tok(w.front + ql(w, s.t & 1, l) + s.n_cur - 1);
        const int4 m = __ldg(g.meta + r.state);
        s.d_cur = r.off + (uint32_t)(m.y - m.x);
      }
      s.n_prev = 0;
      if (s.t >= 1 && s.phase != kPart) s.n_prev = (int32_t)min(cp >> 32, (unsigned long long)w.qcap);
      s.need_commit = (s.committed < s.t) ? 1 : 0;
      if (s.phase == kEmit) {
        // dynamic beam (§3 "Dynamic beam")
        int32_t min_a = a.min_active;
        if (s.t_eff >= 0 && s.t >= s.t_eff - 5) min_a = max(min_a, a.max_active / 2);
        const int64_t n = (int64_t)n_raw;
        const float sb = a.search_beam;
        float b = s.beam;
        if (n == 0 || ((int64_t)min_a <= n && n <= (int64_t)a.max_active))
          b = __fadd_rn(__fmul_rn(0.8f, b), __fmul_rn(0.2f, sb));
        else if (n < (int64_t)min_a)
          b = __fmul_rn(fmaxf(b, sb), 1.25f);
        else
          b = __fmul_rn(fminf(b, sb), 0.8f);
        s.beam = b;
        S.pre_a[l] = (int32_t)((s.d_cur + kTile - 1) / kTile);
        s.frames += 1;
        s.sum_n += n_raw;
        s.sum_d += s.d_cur;
        s.maxlp = mlp;
      }
      // the commit loop: final / partial lanes, and frames without emitting
      // arcs (no tiles); the max pass commits every other frame
      S.pre_b[l] = (s.phase == kFin || s.phase == kPart || (s.need_commit && s.d_cur == 0)) ? s.n_cur : 0;
      // the previous frame's entries, unless its expand pass cleared them
      S.pre_c[l] = s.prev_cleared ? 0 : s.n_prev;
      if (lat && s.need_commit) {
        // records appended since frame t-1's commit: emit(t-1) and eps(t)
        // (for t = 0: the start closure's records)
        const int64_t* B = w.lat_groups + (size_t)l * (w.max_frames + 2);
        s.res_lo = (s.t >= 1) ? B[s.t - 1] : 0;
        s.res_hi = (int64_t)min(__ldcg(&w.lat_cnt[l]), (unsigned long long)w.lat_cap);
        S.pre_d[l] = (int32_t)(s.res_hi - s.res_lo);
      }
    }
    int any_active = 0;
    for (int l = tid; l < L; l += kThreads) any_active |= S.lane[l].phase;
    if (!__syncthreads_or(any_active)) break;
    steps++;
    lane_scan4(S.pre_a, S.pre_b, S.pre_c, S.pre_d, L);
    prof_mark(prof, tsub, kProfPrologue);

    // ================= phase X: commit frame t, clear frame t-1, exact max
    if (tid == 0) S.tctr[1] = 0u;
    if (blockIdx.x == 0) {
      for (int l = tid; l < L; l += kThreads) {
        const SmLane& s = S.lane[l];
        if (s.phase == kEmit) {
          FrameCnt z;
          z.cnt = 0; z.maxkey = 0; z.admitted = 0; z.final_key = 0; z.best_key = 0; z.anc_hi = 0; z.anc_lo = 0;
          *fc_of(w, s.t + 1, l) = z;
          if (GEN && g.has_eps) w.wl_cnt[l] = 0ull;
        }
        if (lat && s.phase != kNone && s.need_commit)
          w.lat_groups[(size_t)l * (w.max_frames + 2) + s.t] = s.res_hi;
      }
    }
    {  // commit (§5.4) of final / partial lanes and of frames without
       // emitting arcs: winners-log entry {delta, arc} per token; final-step
       // keys and the best token
      const int total = S.pre_b[L];
      const int wlane = tid & 31;
      // every CTA takes an equal contiguous share (one batch per thread when
      // the frame fits G * kThreads * kCB tokens)
      const int per = (total + G - 1) / G;
      const int c0 = min(total, blockIdx.x * per), c1 = min(total, c0 + per);
      for (int wb = c0 + (tid & ~31); wb < c1; wb += kThreads * kCB) {
        const int g0 = wb + wlane;
        int lk[kCB];
        int32_t pk[kCB], st[kCB];
        bool v[kCB];
        unsigned long long key[kCB];
#pragma unroll
        for (int k = 0; k < kCB; k++) {
          const int gi = g0 + k * kThreads;
          v[k] = gi < c1;
          lk[k] = v[k] ? find_lane(S.pre_b, L, gi) : 0;
          pk[k] = v[k] ? gi - S.pre_b[lk[k]] : 0;
          st[k] = v[k] ? __ldcg(&w.front[ql(w, S.lane[lk[k]].t & 1, lk[k]) + pk[k]].state) : 0;
        }
        unsigned long long src[kCB], fkey[kCB], bkey[kCB];
#pragma unroll
        for (int k = 0; k < kCB; k++) {
          const ulonglong2 e = v[k] ? __ldcg(ent_at(w, lk[k], st[k], S.lane[lk[k]].t & 1)) : make_ulonglong2(0, 0);
          key[k] = e.x;
          src[k] = e.y;
          fkey[k] = bkey[k] = 0ull;
        }
#pragma unroll
        for (int k = 0; k < kCB; k++) {
          if (!v[k]) continue;
          const int l = lk[k];
          const SmLane& s = S.lane[l];
          const int f = s.t;
          const int32_t arc = key_id(key[k]);
          const float score = key_score(key[k]);
          if (s.need_commit) {
            const int64_t base_new = s.cursor;   // frame f
            const int64_t base_old = s.base_cur; // frame f-1
            // the winner's source token: same frame for an epsilon arc, else the previous one
            const int64_t prev = ((src[k] >> 31) & 1ull ? base_new : base_old) + (int64_t)(src[k] & 0x7fffffffull);
            wlog_commit(a, l, base_new + pk[k], s.floor, arc, prev);
            if (GEN && g.has_eps) {
              const int4 m = __ldg(g.meta + st[k]);
              if (m.z > m.y) atomicAdd(&w.stats[l].eps, (unsigned long long)(m.z - m.y));
            }
            if (ANC) {
              const int32_t an = anc_of(f, arc, src[k], s.gc_c);
              w.anc[ql(w, f & 1, l) + pk[k]] = an;
              if (f % a.gc_interval == 0) {  // bounds read at the GC's check frames only
                FrameCnt* fc = fc_of(w, f, l);
                atomicMax(&fc->anc_hi, (unsigned)(an + 1));
                atomicMax(&fc->anc_lo, 0x7fffffffu - (unsigned)an);
              }
            }
          }
          if (s.phase == kFin) {
            const float fw = __ldg(g.final_w + st[k]);
            if (fw > -INFINITY) fkey[k] = mk_key(__fadd_rn(score, fw), st[k]);
          }
          if (s.phase == kFin || s.phase == kPart) bkey[k] = key[k];
        }
        // final-step keys, finals count and best key: reduced over the warp
        // first when its tokens of a slot all belong to one lane (the usual
        // case), so that a lane's address takes one atomic per warp, not per
        // token
#pragma unroll
        for (int k = 0; k < kCB; k++) {
          const int l = lk[k];
          const int l0 = __shfl_sync(0xffffffffu, l, 0);
          unsigned long long fk = fkey[k], bk = bkey[k];
          if (__all_sync(0xffffffffu, !v[k] || l == l0)) {
            uint32_t nf = fk ? 1u : 0u;
            for (int o = 16; o; o >>= 1) {
              fk = max(fk, __shfl_xor_sync(0xffffffffu, fk, o));
              bk = max(bk, __shfl_xor_sync(0xffffffffu, bk, o));
              nf += __shfl_xor_sync(0xffffffffu, nf, o);
            }
            if ((tid & 31) == 0) {
              const int f0 = S.lane[l0].t;
              if (fk) atomicMax(&fc_of(w, f0, l0)->final_key, fk);
              if (nf) atomicAdd(&w.stats[l0].finals, (unsigned long long)nf);
              if (bk) atomicMax(&fc_of(w, f0, l0)->best_key, bk);
            }
          } else if (v[k]) {
            const int f = S.lane[l].t;
            if (fk) {
              atomicMax(&fc_of(w, f, l)->final_key, fk);
              atomicAdd(&w.stats[l].finals, 1ull);
            }
            if (bk) atomicMax(&fc_of(w, f, l)->best_key, bk);
          }
        }
      }
    }
    prof_mark(prof, tsub, kProfCommit);
    {  // clear frame t-1's recombination entries
      const int total = S.pre_c[L];
      const int per = (total + G - 1) / G;
      const int c0 = min(total, blockIdx.x * per), c1 = min(total, c0 + per);
      for (int g0 = c0 + tid; g0 < c1; g0 += kThreads * kCB) {
        int32_t st[kCB];
        int lk[kCB];
        bool v[kCB];
#pragma unroll
        for (int k = 0; k < kCB; k++) {
          const int gi = g0 + k * kThreads;
          v[k] = gi < c1;
          lk[k] = v[k] ? find_lane(S.pre_c, L, gi) : 0;
          st[k] = v[k] ? __ldcg(&w.front[ql(w, (S.lane[lk[k]].t - 1) & 1, lk[k]) + gi - S.pre_c[lk[k]]].state)
                       : 0;
        }
#pragma unroll
        for (int k = 0; k < kCB; k++)
          if (v[k]) *ent_at(w, lk[k], st[k], (S.lane[lk[k]].t - 1) & 1) = make_ulonglong2(0ull, 0ull);
      }
    }
    if (lat) {  // lattice records of the last step: resolve their frame-t tokens
      // (two records per thread at a time, so that their dependent reads
      // overlap)
      const int total = S.pre_d[L];
      for (int g0 = (int)gstart; g0 < total; g0 += (int)gstride * 2) {
        const int g1 = g0 + (int)gstride;
        const int l0 = find_lane(S.pre_d, L, g0);
        const int l1 = g1 < total ? find_lane(S.pre_d, L, g1) : l0;
        LatRec* r0 = w.lat + (size_t)l0 * w.lat_stride + (S.lane[l0].res_lo + (g0 - S.pre_d[l0]));
        LatRec* r1 = w.lat + (size_t)l1 * w.lat_stride + (S.lane[l1].res_lo + (g1 - S.pre_d[l1]));
        int4 h0 = __ldcg(reinterpret_cast<const int4*>(r0));
        const int32_t d0 = __ldcg(&r0->dst_state);
        int4 h1 = make_int4(0, 0, 0, 0);
        int32_t d1 = 0;
        if (g1 < total) {
          h1 = __ldcg(reinterpret_cast<const int4*>(r1));
          d1 = __ldcg(&r1->dst_state);
        }
        const int p0 = S.lane[l0].t & 1, p1 = S.lane[l1].t & 1;
        const int32_t t0 = __ldcg(tpos_at(w, l0, d0, p0));
        const int32_t t1 = g1 < total ? __ldcg(tpos_at(w, l1, d1, p1)) : 0;
        h0.z = (int32_t)(S.lane[l0].cursor + t0);
        h1.z = (int32_t)(S.lane[l1].cursor + t1);
        if (h0.x & kRecEps) {
          // keep only the relaxation evaluated with the source's final score
          const unsigned used = (unsigned)h0.y;
          const float fin = key_score(__ldcg(&ent_at(w, l0, h0.w, p0)->x));
          h0.y = (int32_t)(S.lane[l0].cursor + __ldcg(tpos_at(w, l0, h0.w, p0)));
          if (ord_f(__uint_as_float(used)) != ord_f(fin)) h0.x |= kRecDead;
        }
        if (g1 < total && (h1.x & kRecEps)) {
          const unsigned used = (unsigned)h1.y;
          const float fin = key_score(__ldcg(&ent_at(w, l1, h1.w, p1)->x));
          h1.y = (int32_t)(S.lane[l1].cursor + __ldcg(tpos_at(w, l1, h1.w, p1)));
          if (ord_f(__uint_as_float(used)) != ord_f(fin)) h1.x |= kRecDead;
        }
        *reinterpret_cast<int4*>(r0) = h0;
        if (g1 < total) *reinterpret_cast<int4*>(r1) = h1;
      }
    }
    prof_mark(prof, tsub, kProfClear);
    emit_tiles<0, LP, KIND>(a, S);
    prof_mark(prof, tsub, kProfMaxTiles);
    if (!grid_sync(a, S, epoch)) return;
    prof_mark(prof, tsub, kProfBarX);
    prof_mark(prof, tlast, kProfCommitMax);

    // ================= interval lattice prune of the lanes whose frame t
    // (committed above) is a positive multiple of the interval
    if (lat && a.lat_interval > 0) {
      int due = 0;
      for (int l = tid; l < L; l += kThreads) {
        SmLane& s = S.lane[l];
        const int ovf = __ldcg(&w.lanes[l].overflow);
        s.closure = (s.phase != kNone && s.need_commit && s.t > 0 && s.t % a.lat_interval == 0 &&
                     !(ovf & (kOvfArena | kOvfKept)))
                        ? 1 : 0;
        due |= s.closure;
      }
      if (__syncthreads_or(due) && !interval_prune(a, S, epoch)) return;
      for (int l = tid; l < L; l += kThreads) S.lane[l].closure = 0;
      __syncthreads();
      prof_mark(prof, tlast, kProfPrune);
      if (blockIdx.x == 0 && tid == 0) prof[kProfSlots + tsub] = prof[kProfSlots + tlast];
    }

    // ================= phase Y: expand (admit + recombine); final / partial
    if (tid == 0) S.tctr[0] = 0u;
    for (int l = tid; l < L; l += kThreads) {
      SmLane& s = S.lane[l];
      S.pre_a[l] = 0;
      if (s.phase == kNone) continue;
      if (s.need_commit) {
        s.base_prev = s.base_cur;
        s.base_cur = s.cursor;
        s.cursor += s.n_cur;
        s.committed = s.t;
        s.log_hw = max(s.log_hw, s.cursor - s.floor);
      }
      s.expanded = 0;
      // winners-log GC of frame t (committed above) at the end of this step
      if (ANC) {
        // at frames that are multiples of gc_interval (the same steps in
        // every lane, so that the lanes' cuts run side by side), a frame
        // whose tokens share one checkpoint ancestor is cut there; frame t
        // is then the next checkpoint
        s.gc_due = 0;
        if (s.phase == kEmit && s.n_cur > 0 && s.t % a.gc_interval == 0 && s.t - s.gc_c >= a.gc_interval) {
          const FrameCnt* fc = fc_of(w, s.t, l);
          const unsigned hi = __ldcg(&fc->anc_hi), lo = __ldcg(&fc->anc_lo);
          if (hi > 0u && hi - 1u == 0x7fffffffu - lo) {
            s.gc_due = 1;
            s.gc_e = s.gc_cbase + (int64_t)(hi - 1u);
            s.gc_c = s.t;
            s.gc_cbase = s.base_cur;
          }
        }
      } else {
        s.gc_due = (GEN && a.gc_interval > 0 && s.phase == kEmit && s.n_cur > 0 &&
                    s.t + 1 - s.gc_t >= a.gc_interval)
                       ? 1 : 0;
        if (s.gc_due) s.gc_t = s.t + 1;
      }
      if (s.phase == kEmit) {
        const unsigned mk = __ldcg(&fc_of(w, s.t, l)->maxkey);
        s.expanded = mk != 0u;
        s.cutoff = mk ? __fsub_rn(unord_f(mk), s.beam) : INFINITY;
        s.cur_max = mk ? unord_f(mk) : -INFINITY;
        s.seed_next = (a.ub_skip && mk && s.t + 1 < s.t_end) ? 1 : 0;
        if (s.expanded) S.pre_a[l] = (int32_t)((s.d_cur + kTile - 1) / kTile);
      }
    }
    // the step's end-of-step tasks (final step, partial, GC round), one per
    // lane with a task, the task-th going to CTA task mod G
    for (int l = tid; l < L; l += kThreads)
      S.pre_b[l] = (S.lane[l].phase == kFin || S.lane[l].phase == kPart || S.lane[l].gc_due) ? 1 : 0;
    __syncthreads();
    lane_scan(S.pre_a, L);
    lane_scan(S.pre_b, L);
    if (blockIdx.x == 0 && (GEN && g.has_eps))
      for (int l = tid; l < L; l += kThreads)
        if (S.lane[l].phase == kEmit) w.wl_cnt[(size_t)1 * L + l] = 0ull;
    if (ANC) {
      // the chain walk of this CTA's first task, when that is a GC cut, runs
      // now in thread 0 while the CTA's other warps start on the expand
      // tiles (warp 0 joins them after the walk): its serial loads overlap
      // the pass instead of holding the step's end
      if (tid == 0) {
        S.gc_pre = -2;
        if ((int)blockIdx.x < S.pre_b[L]) {
          const int l = find_lane(S.pre_b, L, (int)blockIdx.x);
          if (S.lane[l].gc_due) S.gc_pre = gc_walk(a, S.lane[l], l, S.lane[l].gc_e);
        }
      }
      __syncwarp();
    }
    emit_tiles<1, LP, KIND>(a, S);
    prof_mark(prof, tsub, kProfExpTiles);

    // final-arc lattice records (read the entries; cleared only after the loop)
    if (lat) {
      for (int l = tid; l < L; l += kThreads)
        S.pre_c[l] = (S.lane[l].phase == kFin) ? S.lane[l].n_cur : 0;
      __syncthreads();
      lane_scan(S.pre_c, L);
      const int total = S.pre_c[L];
      for (int gi = (int)gstart; gi < total; gi += (int)gstride) {
        const int l = find_lane(S.pre_c, L, gi);
        const int32_t p = gi - S.pre_c[l];
        const SmLane& s = S.lane[l];
        const int par = s.t & 1;
        const int32_t d = __ldcg(&w.front[ql(w, par, l) + p].state);
        const float fw = __ldg(g.final_w + d);
        if (fw > -INFINITY) {
          const float score = key_score(__ldcg(&ent_at(w, l, d, par)->x));
          LatRec r;
          r.frame_flags = (s.t << 4) | kRecFinal;
          r.src_tok = (int32_t)(s.base_cur + p);
          r.dst_tok = -1;
          r.src_state = d;
          r.dst_state = -1;
          r.arc = (int32_t)(g.A + d);
          r.end = __fadd_rn(score, fw);
          r.arcscore = fw;
          const unsigned long long pos = atomicAdd(&w.lat_cnt[l], 1ull);
          if (pos < (unsigned long long)w.lat_cap) w.lat[(size_t)l * w.lat_stride + pos] = r;
          else lane_ovf(a, l, kOvfArena);
        }
      }
    }

    {  // final step (§3) / partial (§8): one CTA per lane walks the winners log
      __syncthreads();
      const int ntask = S.pre_b[L];
      for (int task = blockIdx.x; task < ntask; task += G) {
        const int l = find_lane(S.pre_b, L, task);
        const SmLane& s = S.lane[l];
        const int f = s.t, par = f & 1;
        if (s.gc_due) {
          if (ANC) {
            gc_cut(a, S, l, s.gc_e, task == (int)blockIdx.x ? S.gc_pre : -2);
            __syncthreads();  // the CTA's next task reuses the path scan space
          } else if (GEN) {
            gc_round(a, S, l);
          }
          continue;
        }
        if (tid == 0) {
          const FrameCnt* fc = fc_of(w, f, l);
          const unsigned long long fk = __ldcg(&fc->final_key);
          const unsigned long long bk = __ldcg(&fc->best_key);
          int ok = 0, reached = 0, state = -1;
          float score = -INFINITY;
          if (s.phase == kFin && fk) {
            ok = 1; reached = 1; state = key_id(fk); score = key_score(fk);
          } else if ((s.phase == kPart || a.allow_partial) && bk) {
            ok = 1;
            const int32_t arc = key_id(bk);
            state = arc < 0 ? g.start : __ldg(g.c_dst + arc);
            score = key_score(bk);
          }
          if (__ldcg(&w.lanes[l].overflow) & kOvfArena) ok = 0;
          S.bt_ok = ok;
          S.bt_reached = reached;
          S.bt_state = state;
          S.bt_score = score;
          S.bt_n = -1;   // the token's position in frame f, when kept
          S.bt_pad = -1; // ... else found by the scan below
          if (ok && GEN && tpos_kept(a)) S.bt_n = __ldcg(tpos_at(w, l, state, par));
        }
        __syncthreads();
        if (S.bt_ok && S.bt_n < 0) {
          // positions are not kept for this graph: find the state in the frame
          for (int i = tid; i < s.n_cur; i += kThreads)
            if (__ldcg(&w.front[ql(w, par, l) + i].state) == S.bt_state) S.bt_pad = i;
          __syncthreads();
        }
        if (tid == 0) {
          int ok = S.bt_ok;
          const int reached = S.bt_reached, state = S.bt_state;
          const float score = S.bt_score;
          const int32_t pos = S.bt_n >= 0 ? S.bt_n : S.bt_pad;
          if (pos < 0) ok = 0;
          int64_t idx = -1;
          if (ok) idx = s.base_cur + pos;
          // Walk the winners chain from the newest arc back, writing the arcs
          // newest-first into the tail of the path buffer.  The previous
          // backtrack of this lane (an earlier partial, §8) left its path
          // oldest-first at the head, with each frame's first entry in pframe:
          // once this walk meets that entry the two paths are the same from
          // there back to the start, and the walk stops.
          int64_t n = 0;
          int32_t* path = w.path + (size_t)l * w.path_cap;
          int2* pf = w.pframe + (size_t)l * (w.max_frames + 2);
          const int prev_top = __ldcg(&w.lanes[l].bt_top);
          int32_t d = -1;  // path position of the meeting entry (-1: the walk reached the start)
          int32_t fr = f, fr_seen = f + 1;
          int64_t i = idx;
          // entries [floor, cursor) are live (floor: the GC root, else 0)
          const int64_t lo_i = s.floor, hi_i = s.cursor;
          while (ok && i >= lo_i && i < hi_i && i - lo_i < w.log_cap && n <= hi_i - lo_i) {
            // (frames past the table, possible on a long stream, are simply
            // not recorded: the walk meets the earlier path at a later check)
            if (fr != fr_seen) {  // the first entry of frame fr on this walk
              const bool in_table = fr >= 0 && fr <= w.max_frames + 1;
              if (in_table && fr <= prev_top) {
                const int2 pe = __ldcg(pf + fr);
                if (pe.x == (int32_t)i) { d = pe.y; break; }
              }
              if (in_table) pf[fr] = make_int2((int32_t)i, (int32_t)n);
              fr_seen = fr;
            }
            const int2 e = __ldcg(wlog_at(w, l, i));
            if (e.y < 0) break;
            if (n < w.path_cap) path[w.path_cap - 1 - n] = e.y;
            n++;
            if (!(__ldg(g.c_src + e.y) >> 31)) fr--;  // an emitting arc ends one frame later
            const int32_t dl = wlog_delta(a, e.x);
            if (dl == 0) break;
            i -= dl;
          }
          const int64_t len = (int64_t)d + 1 + n;
          if (n > w.path_cap || len + n > w.path_cap) {
            lane_ovf(a, l, kOvfPath);
            ok = 0;
          }
          S.bt_n = (int32_t)n;
          S.bt_d = d;
          S.bt_lo = fr_seen;  // frames [fr_seen, f] were recorded by this walk
          S.bt_hi = f;
          S.bt_ok = ok;
          S.bt_reached = reached;
          S.bt_score = ok ? score : -INFINITY;
          if (lat && s.phase == kFin && ok && !reached) {
            LatRec r;
            r.frame_flags = (f << 4) | kRecRedirect;
            r.src_tok = (int32_t)idx;
            r.dst_tok = -1;
            r.src_state = state;
            r.dst_state = -1;
            r.arc = (int32_t)(g.A + state);
            r.end = score;
            r.arcscore = 0.f;
            const unsigned long long pos = atomicAdd(&w.lat_cnt[l], 1ull);
            if (pos < (unsigned long long)w.lat_cap) w.lat[(size_t)l * w.lat_stride + pos] = r;
            else lane_ovf(a, l, kOvfArena);
          }
        }
        __syncthreads();
        {  // splice: the walk's arcs go after the shared prefix, oldest first;
           // the recorded frames get their final path positions
          const int nw = S.bt_n, dd = S.bt_d;
          int32_t* path = w.path + (size_t)l * w.path_cap;
          int2* pf = w.pframe + (size_t)l * (w.max_frames + 2);
          if (S.bt_ok) {
            for (int k = tid; k < nw; k += kThreads) path[dd + nw - k] = path[w.path_cap - 1 - k];
            const int fr_hi = min(S.bt_hi, w.max_frames + 1);
            for (int fr = max(S.bt_lo, 0) + tid; fr <= fr_hi; fr += kThreads) {
              int2 e = pf[fr];
              e.y = dd + nw - e.y;
              pf[fr] = e;
            }
          }
          __syncthreads();
          if (tid == 0) {
            w.lanes[l].bt_top = S.bt_ok ? S.bt_hi : -1;
            w.lanes[l].bt_len = S.bt_ok ? dd + 1 + nw : 0;
            S.bt_n = S.bt_ok ? dd + 1 + nw : 0;
          }
          __syncthreads();
        }
        // words = the finalized words (GC), then the path's non-zero output
        // labels, forward order
        const int n = S.bt_n;
        const int32_t* path = w.path + (size_t)l * w.path_cap;
        int32_t* out = w.words + (size_t)l * a.words_cap;
        const int nfin = S.bt_ok ? s.fin_n : 0;
        for (int j = tid; j < min(nfin, a.words_cap); j += kThreads)
          out[j] = __ldcg(w.fin + (size_t)l * (size_t)w.fin_cap + j);
        int run = nfin;
        for (int base = 0; base < n; base += kThreads) {
          const int j = base + tid;
          int32_t o = 0;
          if (j < n) o = __ldg(g.c_olabel + __ldcg(path + j));
          const unsigned bal = __ballot_sync(0xffffffffu, o != 0);
          if ((tid & 31) == 0) S.scan_tmp[tid >> 5] = __popc(bal);
          __syncthreads();
          int wbase = 0, tot = 0;
          for (int ww = 0; ww < kWarps; ww++) {
            if (ww < (tid >> 5)) wbase += S.scan_tmp[ww];
            tot += S.scan_tmp[ww];
          }
          const int pos = run + wbase + __popc(bal & lanemask_lt());
          if (o != 0 && pos < a.words_cap) out[pos] = o;
          run += tot;
          __syncthreads();
        }
        if (tid == 0) {
          Result r;
          r.ok = S.bt_ok;
          r.reached_final = S.bt_reached;
          r.overflow = 0;
          r.n_words = run;
          r.score = S.bt_score;
          r.n_arcs = n;
          r.pad0 = r.pad1 = 0;
          w.res[l] = r;
        }
        __syncthreads();
      }
    }
    prof_mark(prof, tsub, kProfFinal);
    if (!grid_sync(a, S, epoch)) return;
    prof_mark(prof, tsub, kProfBarY);
    prof_mark(prof, tlast, kProfExpand);

    // ================= epsilon closure of the new frames (§5.5)
    if (GEN && g.has_eps) {
      for (int l = tid; l < L; l += kThreads) {
        SmLane& s = S.lane[l];
        s.closure = (s.phase == kEmit && s.expanded) ? s.t + 2 : 0;  // frame t+1
      }
      __syncthreads();
      if (tid == 0) {
        int anyc = 0;
        for (int l = 0; l < L; l++) anyc |= S.lane[l].closure;
        S.flag = anyc;
      }
      __syncthreads();
      if (S.flag && !run_closure(a, S, epoch)) return;
      for (int l = tid; l < L; l += kThreads) S.lane[l].closure = 0;
      prof_mark(prof, tlast, kProfClosure);
      if (blockIdx.x == 0 && tid == 0) prof[kProfSlots + tsub] = prof[kProfSlots + tlast];
    }

    // ================= lane bookkeeping (identical in every CTA)
    for (int l = tid; l < L; l += kThreads) {
      SmLane& s = S.lane[l];
      s.was_emit = 0;
      s.prev_cleared = 0;
      if (s.phase == kEmit) {
        s.t += 1;
        s.was_emit = 1;
        s.prev_cleared = s.expanded;  // the expand pass staged, and cleared, every token
      } else if (s.phase == kFin) {
        s.done_final = 1;
        s.status = kLaneDone;
      } else if (s.phase == kPart) {
        s.done_partial = 1;
      }
    }
    __syncthreads();
  }

  // ---- lattice backward prune of the lanes finished in this call
  if (lat) {
    for (int l = tid; l < L; l += kThreads) {
      SmLane& s = S.lane[l];
      const int ovf = __ldcg(&w.lanes[l].overflow);
      s.closure = (s.done_final && __ldcg(&w.res[l].ok) && !(ovf & (kOvfArena | kOvfKept))) ? 1 : 0;
    }
    __syncthreads();
    if (tid == 0) {
      int any = 0;
      for (int l = 0; l < L; l++) any |= S.lane[l].closure;
      S.any = any;
    }
    __syncthreads();
    if (S.any && !lattice_prune(a, S, epoch)) return;
  }
  prof_mark(prof, tlast, kProfPrune);

  // ---- finished lanes: clear the last frame's recombination entries
  for (int l = 0; l < L; l++) {
    const SmLane& s = S.lane[l];
    if (!s.done_final) continue;
    const int par = s.t & 1;
    for (int64_t p = gstart; p < s.n_cur; p += gstride) {
      const int32_t d = __ldcg(&w.front[ql(w, par, l) + p].state);
      *ent_at(w, l, d, par) = make_ulonglong2(0ull, 0ull);
    }
  }

  // ---- write the lane mirrors back
  if (blockIdx.x == 0) {
    for (int l = tid; l < L; l += kThreads) {
      const SmLane& s = S.lane[l];
      if (s.row < 0) continue;
      LaneState& st = w.lanes[l];
      st.t = s.t;
      st.committed = s.committed;
      st.beam = s.beam;
      st.status = s.status;
      st.cursor = s.cursor;
      st.base_cur = s.base_cur;
      st.base_prev = s.base_prev;
      st.eps_pass = s.eps_pass;
      st.t_eff = s.t_eff;
      st.gc_t = s.gc_t;
      st.gc_c = s.gc_c;
      st.gc_cbase = s.gc_cbase;
      LaneStats& ls = w.stats[l];
      ls.frames += s.frames;
      ls.sum_n += s.sum_n;
      ls.sum_d += s.sum_d;
      ls.sum_m += s.sum_m;
      ls.steps = steps;
      if (lat) ls.lat_held = __ldcg(&w.lat_cnt[l]);
      ls.log_hw = (unsigned long long)s.log_hw;
    }
    if (tid == 0) {
      w.bar->epochs = epoch;
      w.bar->eps_passes = S.eps_passes;
      prof_mark(prof, tlast, kProfTail);
      for (int i = 0; i < kProfSlots; i++) w.prof[i] = prof[i];
    }
  }
}

// ------------------------------------------------------------------ launcher

size_t smem_bytes(int L) { return smem_size(L); }

template <typename LP, int KIND>
static cudaError_t prepare_t() {
  return cudaFuncSetAttribute(decode_kernel<LP, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_size(kMaxLanes));
}

template <typename LP, int KIND>
static cudaError_t launch_t(const RunArgs& a, int grid, cudaStream_t st) {
  void* args[] = {(void*)&a};
  cudaError_t e = prepare_t<LP, KIND>();
  if (e != cudaSuccess) return e;
  return cudaLaunchCooperativeKernel((const void*)decode_kernel<LP, KIND>, dim3(grid), dim3(kThreads), args,
                                     smem_size(a.nlanes), st);
}

// The instantiation a call runs: the ancestor GC (an epsilon-free graph with
// its ancestor table), the plain kernel (epsilon-free, no lattice, no GC) or
// the general one.
template <typename LP>
static cudaError_t launch_kind(const RunArgs& a, int grid, cudaStream_t st) {
  if (a.gc_interval > 0 && a.w.anc != nullptr) return launch_t<LP, kKindAnc>(a, grid, st);
  if (!a.g.has_eps && !a.lattice && a.gc_interval == 0) return launch_t<LP, kKindPlain>(a, grid, st);
  return launch_t<LP, kKindGeneral>(a, grid, st);
}

cudaError_t launch_decode(const RunArgs& a, int dtype, int grid, cudaStream_t st) {
  return dtype == 1 ? launch_kind<__half>(a, grid, st) : launch_kind<float>(a, grid, st);
}

template <typename LP, int KIND>
static cudaError_t occupancy_t(size_t sm, int* per) {
  cudaError_t e = prepare_t<LP, KIND>();
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per, decode_kernel<LP, KIND>, kThreads, sm);
  return e;
}

// Cooperative grid for a launch over L lanes: resident CTAs per SM x SMs
// (the smallest over the instantiations, so that each fits the grid).
cudaError_t max_grid(int dtype, int L, int* grid) {
  int dev = 0, sms = 0, p0 = 0, p1 = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const size_t sm = smem_size(L);
  int p2 = 0;
  if (dtype == 1) {
    e = occupancy_t<__half, kKindGeneral>(sm, &p0);
    if (e == cudaSuccess) e = occupancy_t<__half, kKindAnc>(sm, &p1);
    if (e == cudaSuccess) e = occupancy_t<__half, kKindPlain>(sm, &p2);
  } else {
    e = occupancy_t<float, kKindGeneral>(sm, &p0);
    if (e == cudaSuccess) e = occupancy_t<float, kKindAnc>(sm, &p1);
    if (e == cudaSuccess) e = occupancy_t<float, kKindPlain>(sm, &p2);
  }
  if (e != cudaSuccess) return e;
  *grid = std::min(p0, std::min(p1, p2)) * sms;
  return cudaSuccess;
}

}  // namespace wfst
