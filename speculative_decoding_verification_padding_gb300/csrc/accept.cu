// accept.cu — sv_accept: per-row vocabulary softmax statistics and the
// lossless accept / reject rule (or greedy longest matching prefix).
//
// Sources: [DSpark] glossary ("사전검증 디코딩": the longest matching prefix is
// accepted and the target distribution is preserved); [FASER] mechanism 1
// (per-request number of drafts) and mechanism 2 (a request stops at its
// first rejection; chunks of rows).  The accept / reject formula itself is
// the standard lossless speculative-sampling rule (not printed on the pages).
//
// Kernels, in stream order (a call works on every request, skipping those
// with nothing to decide; in a chunk of a chunked step, on the list of
// requests with a non-empty window that the attention planner wrote):
//   stats  (warps, grid-stride over request x window row x {target, draft} x
//                    vocabulary slice)
//                    one pass over the slice, eight 128-bit loads in flight
//                    per lane: online max / sum of exp(x - max) of
//                    x = logit / T (T > 0), or max and lowest-index argmax of
//                    the raw logits (T = 0); one 8-byte partial per slice.
//                    The first chunk of a chunked step also clears every
//                    request's sampling job.
//   decide (one warp per request)
//                    merges the slice partials of the window rows, then the
//                    chain scan (or the tree descent) with Philox uniforms;
//                    writes the path and, for T > 0, a sampling job for the
//                    emitted token (a draft tree at T > 0: a walk job).  The
//                    fused commit moves the path's K/V and releases the rest.
//   tree   (T > 0 and requests of more than two rows; one thread-block
//                    cluster of sixteen 256-thread CTAs per tree when a
//                    request may hold more than 16 rows, else one 1024-thread
//                    CTA; every CTA without a walk job leaves at once)
//                    the children of each node tried in index order against
//                    the parent's residual, one vocabulary pass per rejected
//                    sibling spread over the cluster; leaves a residual or
//                    bonus job.  In one-pass fused calls its KV commit is
//                    left to the race kernel's extra CTA.
//   race   (warps, grid-stride over request x vocabulary slice)
//                    the residual / bonus token, w = max(0, p - q) after a
//                    rejection or p for the bonus token: an exponential race
//                    among groups of four entries, then the entry inside the
//                    winning group; each warp streams its slice of target
//                    logits through a shared-memory ring (bulk copies) and
//                    prunes groups that cannot win, and draws the entry
//                    inside its own best group; the warp that brings a
//                    request's last slice (release-acquire ticket) reduces
//                    the slice winners and writes the winner's entry.  A
//                    chunked step runs it once, after its last chunk.  One
//                    extra CTA runs the KV commits tree walks left to it.

#include <math.h>

#include <mutex>

#include "sv_accept_internal.h"
#include "sv_internal.cuh"

namespace sv {
namespace acc {

struct StatPart {
  float m;      // T > 0: max of x; T == 0: max raw logit
  float lv;     // T > 0: sum exp(x - m); T == 0: bits of the lowest index of the max
};

struct Job {
  int mode;     // 0 none, 1 residual max(0, p - c q), 2 bonus (p), 3 tree walk pending;
                // | 4: the walk's KV commit is pending (the race kernel runs it)
  int row;      // packed row of the target (and draft) logits
  int pos;      // position of the emitted token
  float c;      // residual coefficient (1 after one rejection)
  float mp, lp, mq, lq;
};

struct RacePart {
  float key;
  int idx;   // the slice's best group
  int tok;   // the entry drawn inside that group
};

constexpr int kStatThreads = 256;
constexpr int kDepth = 8;  // 128-bit loads in flight per lane in the statistics pass
constexpr int kRaceThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

// Slices per row (stats) and per request (race): about 32 warps per SM in
// flight, slices of at least 2 KB.
constexpr int kMaxSlices = 64;  // vocabulary slices per row at most
constexpr long kKeepL2Bytes = 48L << 20;  // logits of a call the statistics keep in L2

inline int stats_chunks(int rows_bound, int V, int nsm) {
  const int maxc = max(1, min(kMaxSlices, V / 512));
  const int want = (nsm * 32 + 2 * rows_bound - 1) / max(1, 2 * rows_bound);
  return max(1, min(want, maxc));
}
inline int race_chunks(int R, int V, int nsm) {
  const int maxc = max(1, min(1024, V / 512));
  const int want = (nsm * 32 + R - 1) / max(1, R);
  return max(1, min(want, maxc));
}
inline __host__ __device__ int chunk_len(int V, int nch) { return ((V + nch - 1) / nch + 3) & ~3; }

Layout layout(int R, int total_rows, int V, int maxw, bool commit) {
  Layout L;
  L.nsm = sizing_sms();
  L.maxw = max(1, min(maxw, kMaxRows));
  const long bound = min((long)total_rows, (long)R * L.maxw);
  L.nch = stats_chunks((int)max(1L, bound), V, L.nsm);
  L.nch_cap = max(L.nch, min(min(kMaxSlices, V / 2048), 16384 / max(1, total_rows)));
  L.nch_r = race_chunks(R, V, L.nsm);
  L.nch_r_cap = max(L.nch_r, min(min(256, V / 512), 16384 / max(1, R)));
  size_t off = 0;
  L.parts = off; off += align256(sizeof(StatPart) * (size_t)total_rows * 2 * L.nch_cap);
  L.jobs = off; off += align256(sizeof(Job) * (size_t)R);
  L.race = off; off += align256(sizeof(RacePart) * (size_t)R * L.nch_r_cap);
  // per request: the race ticket, then the best key any warp has found (bits)
  L.race_tickets = off; off += align256(sizeof(int) * 2 * (size_t)R);
  L.act = off; off += align256(sizeof(int) * (size_t)(R + 1));  // act[R] = count
  L.ctick = L.cspan = 0;
  if (commit) {
    L.ctick = off; off += align256(sizeof(int));
    L.cspan = off; off += align256(sizeof(int2) * (size_t)R);
  }
  L.total = off;
  return L;
}

// Slices actually used (the same value in every kernel of a call).  With an
// active list the items are (listed request, window row, type, slice): about
// two per warp of a 32-warps-per-SM grid.  Without a list they are (packed
// row, type, slice): about four per warp.
__device__ __forceinline__ int stats_slices(const Layout& L, int count, int ntypes, bool listed,
                                            int total_rows) {
  const long slots = listed ? (long)max(1, count) * L.maxw * ntypes
                            : (long)max(1, total_rows) * ntypes;
  const long per_warp = listed ? 2 : 4;
  const long want = (per_warp * L.nsm * 32 + slots - 1) / slots;
  return (int)max((long)L.nch, min(want, (long)L.nch_cap));
}
// Race slices: at most one per warp of the race grid (24 warps per SM), so
// that no warp takes two slices one after the other; slices of >= 2 KB.
constexpr int kRaceWarpsPerSM = 24;
__device__ __forceinline__ int race_slices(const Layout& L, int count, int V) {
  const long want = (long)L.nsm * kRaceWarpsPerSM / max(1, count);
  const long cap = min((long)L.nch_r_cap, max(1L, (long)V / 512));
  return (int)max(1L, min(want, cap));
}

// The paged cache and block pool a fused accept + commit updates.
struct CommitArgs {
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  int num_blocks, Hkv, D, max_blocks;
  int32_t* tables;
  int32_t* cache_lens;
  int32_t* free_list;
  int32_t* free_count;
  int capacity;
};

struct Args {
  sv_batch bt;
  const float* target;
  const float* draft;
  int V;
  float T;
  uint64_t seed;
  int32_t* accepted_len;
  int32_t* accepted_nodes;
  int32_t* next_token;
  uint8_t* ambiguous;
  int32_t* done;
  float* row_stats;
  uint8_t* ws;
  Layout L;
  int32_t* dev_status;
  int race_all;   // race kernel: every request 0..R-1 instead of the active list
  int clear_jobs; // stats kernel: first clear every request's sampling job and race ticket
  int use_list;   // the requests come from the active list (chunked steps)
  const int4* act4;  // with the list: (request, first row, rows, draft rows) per entry
  int commit;     // fused KV commit (sv_accept_commit)
  int keep_l2;    // the statistics load the logits to stay in L2 (small
                  // calls: the decision and the race read them again)
  int tree_commit_race;  // one-pass fused commit at T > 0: a tree walk leaves its
                         // request's commit to the race kernel (job mode bit 2),
                         // whose last CTA runs it beside the race
  CommitArgs kv;
};

__device__ __forceinline__ void merge_ml(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  l = l * ex2((m - M) * kLog2e) + l2 * ex2((m2 - M) * kLog2e);
  m = M;
}
__device__ __forceinline__ void merge_am(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}

// ------------------------------------------------------------- requests --
// The requests a call works on: in a chunk of a chunked step, the list the
// attention planner wrote (requests with a non-empty window, count at
// act[R]); otherwise every request, each kernel skipping those with nothing
// to decide (invalid or empty window, or a continuation window already
// decided).
__device__ __forceinline__ int n_slots(const Args& a, const int* act) {
  return a.use_list ? act[a.bt.n_req] : a.bt.n_req;
}
__device__ __forceinline__ int req_of(const Args& a, const int* act, int k) {
  return a.use_list ? act[k] : k;
}
__device__ __forceinline__ bool live(const Args& a, const Window& w, int i) {
  return w.ok && w.b < w.e && !(w.b > 0 && a.next_token[i] >= 0);
}

// ---------------------------------------------------------------- decide --
struct DecideSmem {
  float mp[kMaxRows], lp[kMaxRows], mq[kMaxRows], lq[kMaxRows];
  int am[kMaxRows], len[kMaxRows], child[kMaxRows], par[kMaxRows], tok[kMaxRows];
  int dep[kMaxRows];          // greedy tree: depth of each node
  unsigned key[kMaxRows];     // greedy tree: best (1 + descent) << 8 | (255 - child)
};

// Merge the slice partials of n0 target rows r0.. (type 0) and n1 draft rows
// r0.. (type 1) into m*/lv* (shared memory, index from 0).  The pairs are
// spread over the warp: up to 32 at a time, each on a group of G lanes (the
// largest power of two that fits), every lane merging slices sub, sub + G, ...
// of its pair, then log2(G) shuffle rounds inside the group.
// kLoads: partial loads in flight per lane (fewer where registers are scarce).
template <int kLoads = 32>
__device__ __forceinline__ void merge_pairs(const Args& a, int nch, int r0, int n0, int n1,
                                            float* m0, float* lv0, float* m1, float* lv1) {
  const int lane = threadIdx.x & 31;
  const float T = a.T;
  const StatPart* parts = reinterpret_cast<const StatPart*>(a.ws + a.L.parts);
  const int np = n0 + n1;
  for (int base = 0; base < np; base += 32) {
    const int cnt = min(32, np - base);
    int G = 32;
    while (G > 1 && G * cnt > 32) G >>= 1;
    const int p = base + lane / G, sub = lane % G;
    const bool live = lane / G < cnt;
    const int type = p < n0 ? 0 : 1;
    const int row = r0 + (p < n0 ? p : p - n0);
    float m = -INFINITY, lv = 0.f;
    int am = 0x7fffffff;
    if (live) {
      // kLoads loads in flight per lane, then the merges
      const StatPart* pr = parts + ((size_t)row * 2 + type) * nch;
      const float2 ident = make_float2(-INFINITY, T > 0.f ? 0.f : __int_as_float(0x7fffffff));
      for (int c0 = sub; c0 < nch; c0 += kLoads * G) {
        float2 v[kLoads];
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
          const int c = c0 + k * G;
          v[k] = c < nch ? __ldcg(reinterpret_cast<const float2*>(pr + c)) : ident;
        }
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
          if (T > 0.f) merge_ml(m, lv, v[k].x, v[k].y);
          else merge_am(m, am, v[k].x, __float_as_int(v[k].y));
        }
      }
    }
    for (int o = G >> 1; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, lv, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, am, o);
      if (T > 0.f) merge_ml(m, lv, m2, l2); else merge_am(m, am, m2, i2);
    }
    if (live && sub == 0) {
      const float out_lv = T > 0.f ? lv : __int_as_float(am);
      if (type == 0) { m0[p] = m; lv0[p] = out_lv; }
      else { m1[p - n0] = m; lv1[p - n0] = out_lv; }
    }
  }
}

// a + b as s + e exactly (Knuth's two-sum; IEEE operations, no contraction).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// The acceptance ratio min(1, p / q) of a drafted token with x = logit / T
// (xp target, xq draft) and row statistics (m, l): p = exp(xp - mp) / lp,
// q = exp(xq - mq) / lq, so p / q = exp((xp - mp) - (xq - mq)) * lq / lp.
// The exponent is formed exactly (two-sums) and one expf is taken, so the
// ratio carries a few 1e-7 of relative error besides that of the fp32
// normalisers -- inside the 1e-6 band where a decision counts as ambiguous.
// Everything stays in fp32: double precision runs at a small fraction of the
// fp32 rate on this GPU, and the dependent fp64 chain of the former form
// cost microseconds per decision.  q that would vanish in double (q below
// the smallest denormal) gives ratio 1, as the definition's q > 0 test does.
// p and q themselves (row statistics output) are formed in fp32.
// p / q itself (unclamped), by the same exact exponent: +inf stands for a q
// that vanishes in double, 0 for p = 0.
__device__ __forceinline__ float pq_ratio(float xp, float xq, float mp, float lp, float mq,
                                          float lq) {
  float s1, e1, s2, e2, h, l;
  two_sum(xq, -mq, s2, e2);
  if (s2 - logf(lq) < -745.13f) return INFINITY;  // also xq = -inf
  two_sum(xp, -mp, s1, e1);
  if (s1 == -INFINITY) return 0.f;                // p = 0
  two_sum(s1, -s2, h, l);
  l = __fadd_rn(l, __fsub_rn(e1, e2));
  return __fdiv_rn(__fmul_rn(expf(h) * (1.f + l), lq), lp);
}
__device__ __forceinline__ float accept_ratio(float xp, float xq, float mp, float lp, float mq,
                                              float lq, float* p_out, float* q_out) {
  if (p_out) {
    *p_out = __fdiv_rn(expf(__fsub_rn(xp, mp)), lp);
    *q_out = __fdiv_rn(expf(__fsub_rn(xq, mq)), lq);
  }
  return fminf(1.f, pq_ratio(xp, xq, mp, lp, mq, lq));
}

// The decision for request i, by one warp, once all its row partials exist.
// Returns kFinal when the request's path is decided, kToTree when the tree
// kernel takes it over, kSkipped when nothing was decided.
constexpr int kFinal = 0, kToTree = 1, kSkipped = 2;

// What a fused commit of a decided chain of at most 32 rows takes from the
// decision instead of reading it again: the rows, the accepted drafts, the
// cache length and, per lane k < rows, the block id of slot ctx + k (loaded
// with the parents and tokens).
struct CommitHint {
  int rows, al, ctx, blk;
  bool chain;
};

__device__ int decide_request(const Args& a, int nch, int i, DecideSmem& sm, CommitHint& h) {
  const int lane = threadIdx.x & 31;
  Job* job = reinterpret_cast<Job*>(a.ws + a.L.jobs) + i;
  if (a.T > 0.f && lane == 0) {
    // Only jobs created by this call may reach the race kernel.
    job->mode = 0;
    reinterpret_cast<int*>(a.ws + a.L.race_tickets)[i] = 0;
    reinterpret_cast<int*>(a.ws + a.L.race_tickets)[a.bt.n_req + i] = 0;
  }
  const Window w = window_of(a.bt, i);
  // loaded with the window: the accepted drafts of the earlier windows, and
  // for a fused commit the cache length
  const int prev_len = a.accepted_len[i];
  const int ctx_c = a.commit ? a.kv.cache_lens[i] : 0;
  h.chain = false;
  if (!a.use_list && !live(a, w, i)) {
    if (!w.ok && lane == 0) flag(a.dev_status, SV_DEV_BAD_WINDOW);
    return kSkipped;
  }
  const int cu = w.cu;  // loaded with the window (a reload would follow the job store)
  const int V = a.V;
  bool chain = true, badp = false, badt = false;
  h.blk = -1;
  if (a.commit && w.rows <= 32 && lane < w.rows && ctx_c >= 0 &&
      (long)ctx_c + lane < (long)a.kv.max_blocks * kBlockSize)
    h.blk = a.kv.tables[(size_t)i * a.kv.max_blocks + (ctx_c + lane) / kBlockSize];
  for (int j = lane; j < w.rows; j += 32) {
    const int p = a.bt.parent[cu + j];
    const int t = a.bt.tokens[cu + j];
    sm.par[j] = p;
    sm.tok[j] = t;
    if (j == 0) {
      if (p != -1) badp = true;
    } else {
      if (p < 0 || p >= j) badp = true;
      if (p != j - 1) chain = false;
      if (t < 0 || t >= V) badt = true;
    }
  }
  __syncwarp();
  badp = __any_sync(0xffffffffu, badp);
  badt = __any_sync(0xffffffffu, badt);
  chain = __all_sync(0xffffffffu, chain);
  if (badp || badt || (!chain && (w.b != 0 || w.e != w.rows))) {
    if (lane == 0)
      flag(a.dev_status, badp ? SV_DEV_BAD_PARENT : badt ? SV_DEV_BAD_TOKEN : SV_DEV_BAD_WINDOW);
    return kSkipped;
  }
  h.rows = w.rows;
  h.ctx = ctx_c;
  h.chain = chain && w.rows <= 32;
  const int max_rows = a.bt.max_rows_per_req;
  int32_t* nodes = a.accepted_nodes + (size_t)i * max_rows;
  if (w.b == 0) {
    for (int k = lane; k < max_rows; k += 32) nodes[k] = k == 0 ? 0 : -1;
  } else if (prev_len != w.b) {
    if (lane == 0) flag(a.dev_status, SV_DEV_BAD_WINDOW);
    return kSkipped;
  }
  if (!chain && a.T > 0.f) {
    // Tree sampling: the walk needs vocabulary passes, one CTA per tree
    // (tree_kernel) takes it over from here.
    if (lane == 0) {
      Job jb{};
      jb.mode = 3;
      jb.row = cu;
      *job = jb;
      a.accepted_len[i] = 0;
      a.next_token[i] = -1;
      a.ambiguous[i] = 0;
      if (a.done) a.done[i] = 0;
    }
    return kToTree;
  }
  int len = w.b;   // accepted drafts so far
  int next = -1;
  bool amb = false;
  float* rs = a.row_stats;

  if (a.T == 0.f) {
    merge_pairs(a, nch, cu + w.b, w.e - w.b, 0, sm.mp + w.b, sm.lp + w.b, nullptr, nullptr);
    __syncwarp();
    for (int r = w.b + lane; r < w.e; r += 32) {
      const int idx = __float_as_int(sm.lp[r]);
      sm.am[r] = idx;
      if (rs) {
        rs[(size_t)(cu + r) * 4 + 0] = sm.mp[r];
        rs[(size_t)(cu + r) * 4 + 1] = (float)idx;
      }
    }
    __syncwarp();
    if (chain) {
      if (lane == 0) {
        const int jmax = min(w.e, w.lim - 1);
        for (int j = w.b + 1; j <= jmax; ++j) {
          const int am = sm.am[j - 1];
          if (sm.tok[j] == am) {
            len = j;
            nodes[j] = j;
          } else {
            next = am;
            break;
          }
        }
        if (next < 0 && w.e == w.lim && len == w.lim - 1) next = sm.am[w.lim - 1];
      }
    } else {
      // tree: longest valid path, lower node index on ties.  Every node n
      // gets len[n] = max over children c whose token is the argmax of row n
      // of 1 + len[c] (0 without one) and child[n] = the lowest such c of
      // that length, computed level by level from the deepest: a child
      // offers (1 + len[c]) << 8 | (255 - c) to its parent by an atomic max
      // (rows <= 128, so the low byte orders the indices).  Depths by
      // pointer jumping: 7 rounds cover 128 levels.
      const int rows = w.rows;
      int jmp[4], dd[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int c = lane + 32 * t;
        jmp[t] = c < rows && c > 0 ? sm.par[c] : 0;
        dd[t] = c < rows && c > 0 ? 1 : 0;
        if (c < rows) {
          sm.dep[c] = dd[t];
          sm.child[c] = jmp[t];  // jump pointers, replaced below
          sm.key[c] = 0u;
        }
      }
      __syncwarp();
      for (int round = 0; round < 7; ++round) {
        int nj[4], nd[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          nj[t] = jmp[t] ? sm.child[jmp[t]] : 0;
          nd[t] = dd[t] + (jmp[t] ? sm.dep[jmp[t]] : 0);
        }
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int c = lane + 32 * t;
          jmp[t] = nj[t];
          dd[t] = nd[t];
          if (c < rows) {
            sm.child[c] = nj[t];
            sm.dep[c] = nd[t];
          }
        }
        __syncwarp();
      }
      int maxd = 0;
#pragma unroll
      for (int t = 0; t < 4; ++t) maxd = max(maxd, dd[t]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) maxd = max(maxd, __shfl_xor_sync(0xffffffffu, maxd, o));
      for (int level = maxd; level >= 1; --level) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int c = lane + 32 * t;
          if (c < rows && dd[t] == level) {
            const int p = sm.par[c];
            if (sm.tok[c] == sm.am[p])
              atomicMax(&sm.key[p], ((1u + (sm.key[c] >> 8)) << 8) | (unsigned)(255 - c));
          }
        }
        __syncwarp();
      }
      for (int n = lane; n < rows; n += 32) {
        const unsigned k = sm.key[n];
        sm.len[n] = (int)(k >> 8);
        sm.child[n] = k ? 255 - (int)(k & 255u) : -1;
      }
      __syncwarp();
      if (lane == 0) {
        int n = 0, k = 0;
        while (sm.child[n] >= 0) {
          n = sm.child[n];
          nodes[++k] = n;
        }
        len = k;
        next = sm.am[n];
      }
    }
    if (lane == 0) {
      a.accepted_len[i] = len;
      a.next_token[i] = next;
      if (w.b == 0) a.ambiguous[i] = 0;
      if (a.done) a.done[i] = next >= 0 ? 1 : 0;
    }
    h.al = __shfl_sync(0xffffffffu, len, 0);
    return kFinal;
  }

  // ---- T > 0: speculative sampling on a chain ----
  const int jmax = min(w.e, w.lim - 1);
  const int nq = max(0, min(w.e, w.lim - 1) - w.b);  // draft rows with a tested child
  const int nd = jmax - w.b;  // drafts decided by this window
  // The logits at the drafted tokens do not depend on the partials: their
  // loads go out before the merge.
  float xp_raw = 0.f, xq_raw = 0.f;
  if (lane < nd) {
    const int j = w.b + 1 + lane;
    const size_t off = (size_t)(cu + j - 1) * V + sm.tok[j];
    xp_raw = a.target[off];
    xq_raw = a.draft[off];
  }
  merge_pairs(a, nch, cu + w.b, w.e - w.b, nq, sm.mp + w.b, sm.lp + w.b, sm.mq + w.b,
              sm.lq + w.b);
  __syncwarp();
  if (rs)
    for (int r = w.b + lane; r < w.e; r += 32) {
      rs[(size_t)(cu + r) * 4 + 0] = sm.mp[r] + logf(sm.lp[r]);
      if (r - w.b < nq) rs[(size_t)(cu + r) * 4 + 1] = sm.mq[r] + logf(sm.lq[r]);
    }
  // Lane j - b - 1 evaluates draft j's ratio and draws its uniform; the scan
  // then reads them by shuffle.
  const float T = a.T;
  float ratio = 1.f;
  float u_lane = 0.f;
  {
    const int j = w.b + 1 + lane;
    if (lane < nd) {
      u_lane = accept_u(a.seed, i, j);
      float p, q;
      ratio = accept_ratio(xp_raw / T, xq_raw / T, sm.mp[j - 1], sm.lp[j - 1], sm.mq[j - 1],
                           sm.lq[j - 1], rs ? &p : nullptr, &q);
      if (rs) {
        rs[(size_t)(cu + j) * 4 + 2] = p;
        rs[(size_t)(cu + j) * 4 + 3] = q;
      }
    }
  }
  __syncwarp();
  Job jb;
  jb.mode = 0;
  jb.c = 1.f;
  for (int k = 0; k < nd; ++k) {
    const int j = w.b + 1 + k;
    const float rk = __shfl_sync(0xffffffffu, ratio, k & 31);
    const float uk = __shfl_sync(0xffffffffu, u_lane, k & 31);
    if (k >= 32) {  // windows longer than a warp: evaluate the rest serially
      const int x = sm.tok[j];
      const size_t off = (size_t)(cu + j - 1) * V + x;
      float p, q;
      ratio = accept_ratio(a.target[off] / T, a.draft[off] / T, sm.mp[j - 1], sm.lp[j - 1],
                           sm.mq[j - 1], sm.lq[j - 1], rs ? &p : nullptr, &q);
      if (rs && lane == 0) {
        rs[(size_t)(cu + j) * 4 + 2] = p;
        rs[(size_t)(cu + j) * 4 + 3] = q;
      }
    }
    const float r_j = k >= 32 ? ratio : rk;
    const float u = k >= 32 ? accept_u(a.seed, i, j) : uk;
    // u and r_j lie in [0, 1]: their difference is exact when it is small
    if (fabsf(u - r_j) < 1e-6f) amb = true;
    if (u < r_j) {
      len = j;
      if (lane == 0) nodes[j] = j;
    } else {
      jb.mode = 1;
      jb.row = cu + j - 1;
      jb.pos = j;
      jb.mp = sm.mp[j - 1];
      jb.lp = sm.lp[j - 1];
      jb.mq = sm.mq[j - 1];
      jb.lq = sm.lq[j - 1];
      break;
    }
  }
  h.al = len;
  if (lane != 0) return kFinal;
  if (jb.mode == 0 && w.e == w.lim && len == w.lim - 1) {
    jb.mode = 2;
    jb.row = cu + w.lim - 1;
    jb.pos = w.lim;
    jb.mp = sm.mp[w.lim - 1];
    jb.lp = sm.lp[w.lim - 1];
    jb.mq = 0.f;
    jb.lq = 1.f;
  }
  *job = jb;
  a.accepted_len[i] = len;
  a.next_token[i] = -1;
  if (w.b == 0) a.ambiguous[i] = 0;
  if (amb) a.ambiguous[i] = 1;
  if (a.done) a.done[i] = jb.mode != 0 ? 1 : 0;
  return kFinal;
}

// ----------------------------------------------------------------- stats --
// Warp-granular: every warp owns one slice of one row at a time and reduces
// it with shuffles into one partial (no warp waits for another); the
// decision kernel merges the partials.
// KEEP: the logits are loaded to stay in L2 (small calls), else streamed.
template <bool VEC, bool KEEP>
__global__ void __launch_bounds__(kStatThreads, 4) stats_kernel(Args a) {
  griddep_entry();
  const int* act = reinterpret_cast<const int*>(a.ws + a.L.act);
  const int R = a.bt.n_req;
  const int count = n_slots(a, act);
  const float T = a.T;
  const int ntypes = T > 0.f ? 2 : 1;
  const int maxw = a.L.maxw;
  // Requests finished so far (fused commit): none in a one-pass call; in the
  // first chunk of a chunked step, the ones the planner did not list (their
  // window is invalid: no chunk ever runs them).
  const bool commit_start = a.use_list ? a.clear_jobs != 0 : true;
  if (a.commit && commit_start && blockIdx.x == 0 && threadIdx.x == 0)
    *reinterpret_cast<int*>(a.ws + a.L.ctick) = a.use_list ? R - count : 0;
  if (a.clear_jobs) {
    // First chunk of a chunked step: the step's single race pass reads every
    // request's job, so none may be left over from an earlier call (the
    // decision kernel, which runs after this one, writes this step's).
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < R; i += gridDim.x * blockDim.x) {
      reinterpret_cast<Job*>(a.ws + a.L.jobs)[i].mode = 0;
      reinterpret_cast<int*>(a.ws + a.L.race_tickets)[i] = 0;
      reinterpret_cast<int*>(a.ws + a.L.race_tickets)[R + i] = 0;
      // fused commit: a request no chunk lists (invalid window) never writes
      // its released span, which the release still reads
      if (a.commit) reinterpret_cast<int2*>(a.ws + a.L.cspan)[i] = make_int2(0, 0);
    }
  }
  const bool listed = a.use_list != 0;
  const int nch = stats_slices(a.L, count, ntypes, listed, a.bt.total_rows);
  const int chl = chunk_len(a.V, nch);
  const long total = listed ? (long)count * maxw * ntypes * nch
                            : (long)a.bt.total_rows * ntypes * nch;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long stride = (long)gridDim.x * (kStatThreads / 32);
  const bool unit = T == 1.f;
  const float rT = T > 0.f ? 1.f / T : 1.f;
  for (long item = (long)blockIdx.x * (kStatThreads / 32) + wid; item < total; item += stride) {
    const int c = (int)(item % nch);
    const long rest = item / nch;
    const int type = (int)(rest % ntypes);
    const long ro = rest / ntypes;
    int i, j, off, r, ndraft;
    Window w;
    if (listed && a.act4) {
      // the planner's row range of the listed request: one load
      off = (int)(ro % maxw);
      const int4 e4 = a.act4[ro / maxw];
      if (off >= e4.z) continue;
      i = e4.x;
      r = e4.y + off;
      ndraft = T > 0.f ? e4.w : 0;
    } else if (listed) {
      off = (int)(ro % maxw);
      i = act[ro / maxw];
      w = window_of(a.bt, i);
      j = w.b + off;
      if (j >= w.e) continue;
      ndraft = T > 0.f ? max(0, min(w.e, w.lim - 1) - w.b) : 0;
      r = a.bt.cu_rows[i] + j;
    } else {
      // packed row ro of request i
      i = find_segment(a.bt.cu_rows, R, (int)ro);
      w = window_of(a.bt, i);
      if (!live(a, w, i)) continue;
      j = (int)ro - a.bt.cu_rows[i];
      if (j < w.b || j >= w.e) continue;
      off = j - w.b;
      ndraft = T > 0.f ? max(0, min(w.e, w.lim - 1) - w.b) : 0;
      r = (int)ro;
    }
    if (type == 1 && off >= ndraft) continue;
    const float* row = (type ? a.draft : a.target) + (size_t)r * a.V;
    const int lo = c * chl;
    const int hi = min(a.V, lo + chl);
    float m = -INFINITY, l = 0.f;
    int am = 0x7fffffff;
    if (T > 0.f) {
      // x = logit / T; exp(x - m) as 2^((x - m) log2 e).  These only build
      // the normaliser: the decision recomputes its own x with an exact
      // division and its ratio from an exactly formed exponent.
      if (VEC) {
        // kDepth 128-entry groups per round: all loads first (entries past
        // the slice read as -inf), then one max and at most one rescale.
        const float4* p4 = reinterpret_cast<const float4*>(row);
        for (int v0 = lo + 4 * lane; v0 < hi + 4 * lane; v0 += 128 * kDepth) {
          float4 x[kDepth];
#pragma unroll
          for (int k = 0; k < kDepth; ++k) {
            const int v = v0 + 128 * k;
            x[k] = v < hi ? (KEEP ? __ldg(p4 + (v >> 2)) : __ldcs(p4 + (v >> 2)))
                           : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          }
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < kDepth; ++k) {
            if (!unit && v0 + 128 * k < hi) {  // the -inf padding stays as it is
              x[k].x = div_by(x[k].x, T, rT);
              x[k].y = div_by(x[k].y, T, rT);
              x[k].z = div_by(x[k].z, T, rT);
              x[k].w = div_by(x[k].w, T, rT);
            }
            mx = fmaxf(mx, fmaxf(fmaxf(x[k].x, x[k].y), fmaxf(x[k].z, x[k].w)));
          }
          if (mx > m) {
            l *= ex2((m - mx) * kLog2e);
            m = mx;
          }
          if (m != -INFINITY) {  // nothing but -inf so far adds nothing
            const float mb = m * kLog2e;
#pragma unroll
            for (int k = 0; k < kDepth; ++k)
              l += (ex2(fmaf(x[k].x, kLog2e, -mb)) + ex2(fmaf(x[k].y, kLog2e, -mb))) +
                   (ex2(fmaf(x[k].z, kLog2e, -mb)) + ex2(fmaf(x[k].w, kLog2e, -mb)));
          }
        }
      } else {
        for (int v = lo + lane; v < hi; v += 32) {
          const float x = unit ? row[v] : div_by(row[v], T, rT);
          if (x > m) {
            l *= ex2((m - x) * kLog2e);
            m = x;
          }
          l += ex2((x - m) * kLog2e);
        }
      }
    } else {
      if (VEC) {
        const float4* p4 = reinterpret_cast<const float4*>(row);
        for (int v0 = lo + 4 * lane; v0 < hi + 4 * lane; v0 += 128 * kDepth) {
          float4 x[kDepth];
#pragma unroll
          for (int k = 0; k < kDepth; ++k) {
            const int v = v0 + 128 * k;
            x[k] = v < hi ? (KEEP ? __ldg(p4 + (v >> 2)) : __ldcs(p4 + (v >> 2)))
                           : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
          }
#pragma unroll
          for (int k = 0; k < kDepth; ++k) {
            const int v = v0 + 128 * k;
            if (x[k].x > m) { m = x[k].x; am = v; }
            if (x[k].y > m) { m = x[k].y; am = v + 1; }
            if (x[k].z > m) { m = x[k].z; am = v + 2; }
            if (x[k].w > m) { m = x[k].w; am = v + 3; }
          }
        }
      } else {
        for (int v = lo + lane; v < hi; v += 32) {
          const float x = row[v];
          if (x > m) { m = x; am = v; }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, am, o);
      if (T > 0.f) merge_ml(m, l, m2, l2); else merge_am(m, am, m2, i2);
    }
    if (lane == 0) {
      StatPart sp;
      sp.m = m;
      sp.lv = T > 0.f ? l : __int_as_float(am);
      reinterpret_cast<StatPart*>(a.ws + a.L.parts)[((size_t)r * 2 + type) * nch + c] = sp;
    }
  }
}

// ---------------------------------------------------------- fused commit --
// sv_accept_commit: the warp that finalises a request's path also commits it
// ([SwiftSpec] mechanism 3: verification result and KV update fused;
// mechanism 2: the accepted path's KV kept, the rest released), with the
// same rule and order as sv_commit_kv:
//   - the K/V of staged slot ctx + path[k] moves to slot ctx + k, for k =
//     1 .. a in ascending order (a slot written at step k is never the
//     source of a later step, since path[k'] >= k' > k), every head, by the
//     warp's lanes;
//   - the new cache length is ctx + 1 + a; table entries past it are the
//     blocks to release.
// Every request of the call counts itself done on a ticket; the warp that
// brings it to n_req appends all released blocks to the pool in (request,
// table index) order and clears their table entries.

// Same validity rule as sv_commit_kv, checked by the whole warp (every
// lane holds the same rows, ctx, al): 0 when the commit is valid, else the
// SV_DEV_* bit of the first rule broken, in the order path / window, cache
// length, block ids.  A request failing it is left as it was.
__device__ __forceinline__ int commit_check(const Args& a, int rows, int ctx, int al, const int32_t* path,
                            const int32_t* table) {
  const int lane = threadIdx.x & 31;
  const CommitArgs& c = a.kv;
  if (rows < 1 || rows > a.bt.max_rows_per_req || al < 0 || al > rows - 1)
    return SV_DEV_BAD_WINDOW;
  bool bad = false;
  for (int k = lane; k <= al; k += 32) {
    const int pk = path[k];
    bad |= k == 0 ? pk != 0 : (pk <= path[k - 1] || pk >= rows);
  }
  if (__any_sync(0xffffffffu, bad)) return SV_DEV_BAD_WINDOW;
  if (ctx < 0 || (long)ctx + rows > (long)c.max_blocks * kBlockSize) return SV_DEV_BAD_LENGTH;
  // path[k] in [0, rows) now, so both table indexes are below max_blocks
  for (int k = lane; k <= al; k += 32) {
    const int b1 = table[(ctx + path[k]) / kBlockSize];
    const int b2 = table[(ctx + k) / kBlockSize];
    bad |= b1 < 0 || b1 >= c.num_blocks || b2 < 0 || b2 >= c.num_blocks;
  }
  if (__any_sync(0xffffffffu, bad)) return SV_DEV_BAD_BLOCK_ID;
  return 0;
}

// One warp: move the path's K/V, set the new length, record the table span
// [keep, used) whose blocks the release frees.  final = false: nothing was
// decided for the request, which is only counted.  The lanes look up the
// moves of 32 path positions at once (chains move nothing); the moves
// themselves run in ascending k, every lane copying part of the slot.
// pairs: two moves at a time (more registers; the decision kernel has them).
// lean: a single move's loads and stores under guards (fewest registers: the
// 1024-thread walk has 64 a thread).
__device__ __forceinline__ void commit_request(const Args& a, int i, bool final,
                                               const CommitHint* hint, bool pairs = false,
                                               bool lean = false) {
  const int lane = threadIdx.x & 31;
  const CommitArgs& c = a.kv;
  // A call with one request needs no ticket: its warp releases at once (the
  // free count's load goes out first).
  const bool alone = a.bt.n_req == 1;
  const int fc_alone = alone ? *c.free_count : 0;
  const bool chain_hint = final && hint && hint->chain;
  int2 span = make_int2(0, 0);
  int ctx_span = 0;  // cache length the span was computed from
  if (chain_hint) {
    // A chain the decision just decided: its path is 0..al (nothing moves);
    // the same rules as commit_check, on the values the decision holds.
    const int rows = hint->rows, ctx = hint->ctx, al = hint->al;
    ctx_span = ctx;
    int bad = 0;
    if (rows < 1 || rows > a.bt.max_rows_per_req || al < 0 || al > rows - 1) {
      bad = SV_DEV_BAD_WINDOW;
    } else if (ctx < 0 || (long)ctx + rows > (long)c.max_blocks * kBlockSize) {
      bad = SV_DEV_BAD_LENGTH;
    } else if (__any_sync(0xffffffffu,
                          lane <= al && (hint->blk < 0 || hint->blk >= c.num_blocks))) {
      bad = SV_DEV_BAD_BLOCK_ID;
    }
    if (bad) {
      if (lane == 0) flag(a.dev_status, bad);
    } else {
      span = make_int2((ctx + 1 + al + kBlockSize - 1) / kBlockSize,
                       (ctx + rows + kBlockSize - 1) / kBlockSize);
      if (lane == 0) c.cache_lens[i] = ctx + 1 + al;
    }
  } else if (final) {
    const int rows = a.bt.cu_rows[i + 1] - a.bt.cu_rows[i];
    const int ctx = c.cache_lens[i];
    const int al = a.accepted_len[i];
    ctx_span = ctx;
    const int32_t* path = a.accepted_nodes + (size_t)i * a.bt.max_rows_per_req;
    const int32_t* table = c.tables + (size_t)i * c.max_blocks;
    const int bad = commit_check(a, rows, ctx, al, path, table);
    if (bad) {
      if (lane == 0) flag(a.dev_status, bad);
    } else {
      const int cpr = c.D / 8;  // int4 per token row of one head
      const int per_slot = 2 * c.Hkv * cpr;
      for (int k0 = 1; k0 <= al; k0 += 32) {
        const int k = k0 + lane;
        unsigned long long srow = 0, drow = 0;
        bool mv = false;
        if (k <= al) {
          const int src = path[k];
          mv = src != k;
          if (mv) {
            const int ss = ctx + src, ds = ctx + k;
            srow = ((unsigned long long)table[ss / kBlockSize] * c.Hkv) * kBlockSize +
                   ss % kBlockSize;
            drow = ((unsigned long long)table[ds / kBlockSize] * c.Hkv) * kBlockSize +
                   ds % kBlockSize;
          }
        }
        // A slot written at step k is never the source of a later step
        // (path[k'] >= k' > k), so ascending k reads every source first.  Two
        // moves go at once (both sources read, then both destinations
        // written): the second move's destination can only be the first's
        // source, which is read before it is written.
        unsigned m = __ballot_sync(0xffffffffu, mv);
        auto slot_int4 = [&](unsigned long long row, int x) {
          const int tensor = x / (c.Hkv * cpr), rem = x % (c.Hkv * cpr);
          const int g = rem / cpr, q = rem % cpr;
          return reinterpret_cast<int4*>((tensor ? c.v : c.k) + (row + (size_t)g * kBlockSize) * c.D) + q;
        };
        while (m) {
          const int j = __ffs(m) - 1;
          m &= m - 1;
          const int j2 = (pairs && m && per_slot <= 32 * 8) ? __ffs(m) - 1 : -1;
          if (j2 >= 0) m &= m - 1;
          const unsigned long long sr = __shfl_sync(0xffffffffu, srow, j);
          const unsigned long long dr = __shfl_sync(0xffffffffu, drow, j);
          const unsigned long long sr2 = __shfl_sync(0xffffffffu, srow, j2 >= 0 ? j2 : j);
          const unsigned long long dr2 = __shfl_sync(0xffffffffu, drow, j2 >= 0 ? j2 : j);
          // eight 16-byte loads of each slot in flight per lane, then the
          // stores, branch-free: a lane past the slot repeats its last entry,
          // and without a second move sr2 / dr2 repeat sr / dr (the same
          // value to the same place) -- guarded loads and stores went out one
          // after another, 6 us more per draft-tree step, measured.  (pairs
          // and lean are constants at every call.)
          for (int x0 = 0; x0 < per_slot; x0 += 32 * 8) {
            int4 val[8], val2[8];
            if (pairs) {
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                const int x = min(x0 + 32 * t + lane, per_slot - 1);
                val[t] = *slot_int4(sr, x);
                val2[t] = *slot_int4(sr2, x);
              }
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                const int x = min(x0 + 32 * t + lane, per_slot - 1);
                *slot_int4(dr, x) = val[t];
                *slot_int4(dr2, x) = val2[t];
              }
            } else if (!lean) {
#pragma unroll
              for (int t = 0; t < 8; ++t) val[t] = *slot_int4(sr, min(x0 + 32 * t + lane, per_slot - 1));
#pragma unroll
              for (int t = 0; t < 8; ++t) *slot_int4(dr, min(x0 + 32 * t + lane, per_slot - 1)) = val[t];
            } else {
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                const int x = x0 + 32 * t + lane;
                if (x < per_slot) val[t] = *slot_int4(sr, x);
              }
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                const int x = x0 + 32 * t + lane;
                if (x < per_slot) *slot_int4(dr, x) = val[t];
              }
            }
          }
          __syncwarp();
        }
      }
      span = make_int2((ctx + 1 + al + kBlockSize - 1) / kBlockSize,
                       (ctx + rows + kBlockSize - 1) / kBlockSize);
      if (lane == 0) c.cache_lens[i] = ctx + 1 + al;
    }
  }
  if (alone) {
    // The span (at most nine blocks: rows <= 128) with its block ids in
    // registers: a decided chain's from the decision's own loads (lane k
    // holds the block of slot ctx + k), else one load per lane.
    const int n = span.y - span.x;
    int32_t* table = c.tables + (size_t)i * c.max_blocks;
    int blk = -1;
    if (chain_hint) {
      const int kt = max(0, (span.x + lane) * kBlockSize - ctx_span);
      const int b = __shfl_sync(0xffffffffu, hint->blk, min(kt, 31));
      if (lane < n) blk = b;
    } else if (lane < n) {
      blk = table[span.x + lane];
    }
    const bool has = lane < n && blk >= 0;
    const unsigned m = __ballot_sync(0xffffffffu, has);
    const int nfree = __popc(m);
    if (nfree == 0) return;
    if ((long)fc_alone + nfree <= c.capacity) {
      if (has) {
        c.free_list[fc_alone + __popc(m & ((1u << lane) - 1u))] = blk;
        table[span.x + lane] = -1;
      }
      if (lane == 0) *c.free_count = fc_alone + nfree;
    } else if (lane == 0) {
      flag(a.dev_status, SV_DEV_POOL_OVERFLOW);
    }
    return;
  }
  int last = 0;
  if (lane == 0) {
    reinterpret_cast<int2*>(a.ws + a.L.cspan)[i] = span;
    last = ticket_add(reinterpret_cast<int*>(a.ws + a.L.ctick), 1) == a.bt.n_req - 1;
  }
  last = __shfl_sync(0xffffffffu, last, 0);
  if (!last) return;
  // Every request is done: release in (request, table index) order.
  __syncwarp();
  const int R = a.bt.n_req;
  const int2* spans = reinterpret_cast<const int2*>(a.ws + a.L.cspan);
  const int fc0 = *c.free_count;
  int carry = 0, pushed = 0;
  // 64 requests per round, lane l taking requests l and l + 32: both halves'
  // spans, then both halves' table entries, are loaded together before the
  // blocks go to the list in (request, table index) order
  for (int base = 0; base < R; base += 64) {
    int nfree[2] = {0, 0};
    int2 sp[2];
    const int32_t* table[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = base + 32 * h + lane;
      sp[h] = r < R ? __ldcg(spans + r) : make_int2(0, 0);
      table[h] = c.tables + (size_t)min(r, R - 1) * c.max_blocks;
    }
    const int len = max(sp[0].y - sp[0].x, sp[1].y - sp[1].x);
    for (int t = 0; t < len; ++t) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (sp[h].x + t < sp[h].y) nfree[h] += __ldcg(table[h] + sp[h].x + t) >= 0;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int x = nfree[h];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      const int total = __shfl_sync(0xffffffffu, x, 31);
      if (nfree[h]) {
        const long start = (long)fc0 + carry + x - nfree[h];
        if (start + nfree[h] <= c.capacity) {
          int32_t* tb = const_cast<int32_t*>(table[h]);
          int n = 0;
          for (int t = sp[h].x; t < sp[h].y; ++t) {
            const int blk = tb[t];
            if (blk < 0) continue;
            c.free_list[start + n++] = blk;
            tb[t] = -1;
          }
          pushed = max(pushed, (int)(start + nfree[h] - fc0));
        } else {
          flag(a.dev_status, SV_DEV_POOL_OVERFLOW);
        }
      }
      carry += total;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pushed = max(pushed, __shfl_xor_sync(0xffffffffu, pushed, o));
  if (lane == 0) {
    *c.free_count = fc0 + pushed;
    *reinterpret_cast<int*>(a.ws + a.L.ctick) = 0;
  }
}

// ---------------------------------------------------------------- decide --
// One warp per active request, once every row partial exists.
constexpr int kDecideWarps = 4;

__global__ void __launch_bounds__(kDecideWarps * 32, 1) decide_kernel(Args a) {
  griddep_entry();
  __shared__ DecideSmem s_dec[kDecideWarps];
  const int* act = reinterpret_cast<const int*>(a.ws + a.L.act);
  const int count = n_slots(a, act);
  const int nch = stats_slices(a.L, count, a.T > 0.f ? 2 : 1, a.use_list != 0, a.bt.total_rows);
  const int wid = threadIdx.x >> 5;
  for (int ai = blockIdx.x * kDecideWarps + wid; ai < count; ai += gridDim.x * kDecideWarps) {
    const int i = req_of(a, act, ai);
    CommitHint hint;
    const int outcome = decide_request(a, nch, i, s_dec[wid], hint);
    if (a.commit && outcome != kToTree) {
      __syncwarp();  // the path and state lane 0 wrote are visible to the warp
      bool now = true;
      if (a.use_list) {
        // Chunked step: a request is committed in the chunk that stops it; one
        // whose input is invalid stops here and is only counted.
        if (outcome == kSkipped) {
          if ((threadIdx.x & 31) == 0) a.done[i] = 1;
        } else {
          now = a.done[i] != 0;
        }
      }
      if (now) commit_request(a, i, outcome == kFinal, outcome == kFinal ? &hint : nullptr, true);
    }
  }
}

// ------------------------------------------------------------- tree walk --
// Sampling on a draft tree (T > 0; siblings drawn independently from the
// parent's q), one CTA per tree, after the decision kernel marked it.  From
// the root, the children of node n are tried in index order: child c (token
// x) is accepted iff u(i, c) < min(1, p'(x) / q_n(x)) with p' the target
// distribution left by the siblings rejected before it.  After j rejections
// p' = max(0, p - c_j q) / S(c_j), S(c) = sum_v max(0, p_v - c q_v),
// c_0 = 0, S(c_0) = 1, c_{j+1} = c_j + S(c_j): one vocabulary pass per
// rejection (all threads; per-thread Kahan sums, then fp64).  If S vanishes,
// the remaining siblings are not tried and the token comes from p_n.  The
// walk ends at a leaf (bonus from p_leaf) or when every child is rejected
// (a residual job with coefficient c); the race draws the token.
//
// NT threads per CTA, CL CTAs per tree: with CL > 1 the tree's CTAs form one
// thread-block cluster that shares each vocabulary pass (thread t of CTA r
// takes the entries of global thread r * NT + t), adds the CTAs' sums in rank
// order over distributed shared memory, and takes every decision in each CTA
// alike (the same inputs and operations: the same walk everywhere); rank 0
// writes the results.
constexpr int kTreeThreads = 1024;         // one CTA per tree
constexpr int kTreeClusterThreads = 256;   // CTAs of a tree's cluster
constexpr int kTreeCluster = 16;
// The cluster walk when a request may hold more rows than this (a deep tree;
// chains of draft length <= 16 and small trees keep the single-CTA walk: a
// cluster launch behind the decision kernel costs a few microseconds even
// when no request walks, measured in stream order with a cold L2).
constexpr int kTreeClusterMinRows = 17;

template <int NT, int CL>
__global__ void __launch_bounds__(NT) tree_kernel(Args a) {
  griddep_entry();
  const int i = blockIdx.x / CL;
  const int rank = CL > 1 ? (int)cluster_rank() : 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Job* job = reinterpret_cast<Job*>(a.ws + a.L.jobs) + i;
  __shared__ int s_mode, s_nk, s_dec;
  __shared__ int s_kids[kMaxRows];
  __shared__ float s_st[4];  // merged max / normaliser of p and of q at the current node
  __shared__ double s_red[NT / 32];
  __shared__ double s_S;
  __shared__ double s_part[2];  // this CTA's sum of the current pass (pass parity)
  if (tid == 0) s_mode = job->mode;
  __syncthreads();
  if (s_mode != 3) return;  // the same for every CTA of the tree
  const int* act = reinterpret_cast<const int*>(a.ws + a.L.act);
  const int nch = stats_slices(a.L, n_slots(a, act), 2, a.use_list != 0, a.bt.total_rows);
  const float T = a.T, rT = 1.f / T;
  const int V = a.V;
  const bool vec =
      (V & 3) == 0 && ((((uintptr_t)a.target) | ((uintptr_t)a.draft)) & 15) == 0;
  const int cu = a.bt.cu_rows[i];
  const int rows = a.bt.cu_rows[i + 1] - cu;  // checked by the decision kernel
  int32_t* nodes = a.accepted_nodes + (size_t)i * a.bt.max_rows_per_req;
  int n = 0, k = 0;
  bool amb = false;
  Job out{};
  int npass = 0;  // vocabulary passes so far (parity of the cluster's sum slot)
  // 128-bit loads of each row in flight per thread in a pass (a cluster's
  // 4096 threads cover a 128256-entry row in one round)
  constexpr int kPassDepth = CL > 1 ? 8 : 4;
  // Before the first step, every load a step needs, all at once: the merged
  // statistics of every node (draft ones of the nodes that can be parents,
  // rows - 1 at most) and, for every non-root node, its parent's link and its
  // token's target and draft logits at the parent.  A step then only reads
  // shared memory.  (The decision kernel checked the parents, in [0, r), and
  // the tokens, in [0, V).)
  __shared__ float s_mp[kMaxRows], s_lp[kMaxRows], s_mq[kMaxRows], s_lq[kMaxRows];
  __shared__ float s_xp[kMaxRows], s_xq[kMaxRows];
  __shared__ int s_par[kMaxRows];
  {
    constexpr int kRowsPerWarp = 8;
    for (int base = warp * kRowsPerWarp; base < rows; base += (NT / 32) * kRowsPerWarp) {
      const int cnt = min(kRowsPerWarp, rows - base);
      merge_pairs<16>(a, nch, cu + base, cnt, max(0, min(cnt, rows - 1 - base)), s_mp + base,
                      s_lp + base, s_mq + base, s_lq + base);
    }
    for (int r = tid; r < rows; r += NT) {
      const int p = r == 0 ? -1 : a.bt.parent[cu + r];
      s_par[r] = p;
      if (r > 0) {
        const int x = a.bt.tokens[cu + r];
        s_xp[r] = a.target[(size_t)(cu + p) * V + x];
        s_xq[r] = a.draft[(size_t)(cu + p) * V + x];
      }
    }
  }
  __syncthreads();
  for (int step = 0; step < kMaxRows; ++step) {  // every move goes to a larger node
    if (warp == 0) {
      // children of n in index order, and the node's statistics
      int cnt = 0;
      for (int base = n + 1; base < rows; base += 32) {
        const int c = base + lane;
        const bool is = c < rows && s_par[c] == n;
        const unsigned m = __ballot_sync(0xffffffffu, is);
        if (is) s_kids[cnt + __popc(m & ((1u << lane) - 1u))] = c;
        cnt += __popc(m);
      }
      if (lane == 0) {
        s_nk = cnt;
        s_st[0] = s_mp[n];
        s_st[1] = s_lp[n];
        if (cnt > 0) {
          s_st[2] = s_mq[n];
          s_st[3] = s_lq[n];
        }
      }
    }
    __syncthreads();
    const int nk = s_nk;
    if (nk == 0) {  // leaf: bonus token from p_n
      out.mode = 2;
      break;
    }
    const float* lp = a.target + (size_t)(cu + n) * V;
    const float* lq = a.draft + (size_t)(cu + n) * V;
    double c = 0.0, S = 1.0, inv_S = 1.0;
    bool moved = false, vanished = false;
    for (int t = 0; t < nk; ++t) {
      const int ch = s_kids[t];
      if (tid == 0) {  // (in every CTA of a cluster: the same decision)
        // pres / q = max(0, p - c q) / (S q) = max(0, p/q - c) / S, with p/q
        // from the exact exponent in fp32 (as on chains; fp64 runs at a
        // small fraction of the fp32 rate on this GPU) and 1 / S taken once
        // per pass.  q that vanishes gives ratio 1, as the definition's
        // q > 0 test does; p = 0 gives 0.
        const float r_pq = pq_ratio(s_xp[ch] / T, s_xq[ch] / T, s_st[0], s_st[1], s_st[2], s_st[3]);
        const double ratio =
            r_pq == INFINITY ? 1.0 : fmin(1.0, fmax(0.0, (double)r_pq - c) * inv_S);
        const double u = (double)accept_u(a.seed, i, ch);
        if (fabs(u - ratio) < 1e-6) amb = true;
        s_dec = u < ratio ? 1 : 0;
      }
      __syncthreads();
      const int dec = s_dec;
      __syncthreads();  // s_dec is rewritten by the next test
      if (dec) {
        if (tid == 0 && rank == 0) nodes[k + 1] = ch;
        ++k;
        n = ch;
        moved = true;
        break;
      }
      c += S;
      // S(c) over the whole vocabulary
      const float mpb = s_st[0] * kLog2e, mqb = s_st[2] * kLog2e;
      const float inv_lp = 1.f / s_st[1], cq = (float)c / s_st[3];
      float sum = 0.f, comp = 0.f;
      auto add = [&](float xp, float xq) {  // Kahan step of max(0, p_v - c q_v)
        const float pv = ex2(fmaf(div_by(xp, T, rT), kLog2e, -mpb)) * inv_lp;
        const float qv = ex2(fmaf(div_by(xq, T, rT), kLog2e, -mqb)) * cq;
        const float y = fmaxf(pv - qv, 0.f) - comp;
        const float tsum = sum + y;
        comp = (tsum - sum) - y;
        sum = tsum;
      };
      if (vec) {
        // 128-bit loads, kPassDepth of each row in flight per thread (entries past
        // the row read as -inf logits: p = 0 adds nothing)
        const float4* p4 = reinterpret_cast<const float4*>(lp);
        const float4* q4 = reinterpret_cast<const float4*>(lq);
        const int n4 = V >> 2;
        const float4 none = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        for (int v0 = rank * NT + tid; v0 < n4; v0 += kPassDepth * NT * CL) {
          float4 xp[kPassDepth], xq[kPassDepth];
#pragma unroll
          for (int k = 0; k < kPassDepth; ++k) {
            const int v = v0 + k * NT * CL;
            xp[k] = v < n4 ? __ldg(p4 + v) : none;
            xq[k] = v < n4 ? __ldg(q4 + v) : none;
          }
#pragma unroll
          for (int k = 0; k < kPassDepth; ++k) {
            add(xp[k].x, xq[k].x);
            add(xp[k].y, xq[k].y);
            add(xp[k].z, xq[k].z);
            add(xp[k].w, xq[k].w);
          }
        }
      } else {
        for (int v = rank * NT + tid; v < V; v += NT * CL) add(lp[v], lq[v]);
      }
      double d = (double)sum - (double)comp;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      if (lane == 0) s_red[warp] = d;
      __syncthreads();
      if (warp == 0) {
        double e = lane < NT / 32 ? s_red[lane] : 0.0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
        if (lane == 0) {
          if (CL > 1) s_part[npass & 1] = e;
          else s_S = e;
        }
      }
      if constexpr (CL > 1) {
        // every CTA's sum of this pass is in place; each CTA adds them in
        // rank order (the slot of this parity is next written two passes on,
        // after every CTA has passed the next pass's barrier)
        cluster_sync();
        if (tid == 0) {
          // all the CTAs' sums in flight at once, then added in rank order
          const uint32_t slot = smem_u32(&s_part[npass & 1]);
          double v[CL];
#pragma unroll
          for (int q = 0; q < CL; ++q) v[q] = dsmem_ld_f64(dsmem_addr(slot, (uint32_t)q));
          double t = 0.0;
#pragma unroll
          for (int q = 0; q < CL; ++q) t += v[q];
          s_S = t;
        }
      }
      __syncthreads();
      ++npass;
      S = s_S;
      if (!(S > 0.0)) {
        vanished = true;
        break;
      }
      inv_S = 1.0 / S;
    }
    if (moved) continue;
    out.mode = vanished ? 2 : 1;
    out.c = (float)c;
    break;
  }
  if (tid == 0 && rank == 0) {
    out.row = cu + n;
    out.pos = k + 1;
    out.mp = s_st[0];
    out.lp = s_st[1];
    out.mq = s_st[2];
    out.lq = s_st[3];
    if (out.mode == 2) {
      out.mq = 0.f;
      out.lq = 1.f;
    }
    if (a.commit && a.tree_commit_race) out.mode |= 4;
    *job = out;
    a.accepted_len[i] = k;
    a.next_token[i] = -1;
    if (amb) a.ambiguous[i] = 1;
    if (a.done) a.done[i] = 1;
  }
  if (a.commit && !a.tree_commit_race && warp == 0 && rank == 0) {
    __syncwarp();  // the path thread 0 wrote is visible to the warp
    commit_request(a, i, true, nullptr, false, CL == 1);
  }
  // no CTA leaves while its peers may still read its last pass's sum
  if constexpr (CL > 1) cluster_sync();
}

// ------------------------------------------------------------------ race --
// The residual / bonus token in two steps, both exact ([DSpark] glossary: the
// target distribution is preserved):
//   1. a race among groups of four entries: group g has weight W_g, the sum
//      of its entries' w = max(0, p - c q) (residual) or p (bonus), and key
//      W_g / E_g with E_g = -log(U_g); the largest key wins, lowest g on
//      ties, so P(g) = W_g / sum W;
//   2. inside the winning group, with u from pick_u: the first entry whose
//      running sum of w (index order) exceeds u W_g, so P(v | g) = w_v / W_g.
// One uniform per group (one generator call per lane per 16 entries) instead
// of one per entry.
__device__ __forceinline__ void race_take(float& best, int& bi, float key, int v) {
  if (key > best || (key == best && v < bi)) { best = key; bi = v; }
}
// The same, carrying the entry drawn inside the group along.
__device__ __forceinline__ void race_take(float& best, int& bi, int& tok, float key, int v, int t) {
  if (key > best || (key == best && v < bi)) { best = key; bi = v; tok = t; }
}

constexpr int kRaceBlock = 512;  // entries of 128 groups: one counter per lane

// Constants of one race job for its weights w = p (bonus) or max(0, p - c q).
struct RaceW {
  float T, rT, mpb, inv_lp, mqb, cq;
  bool unit, resid;
};
__device__ __forceinline__ float race_p(const RaceW& r, float l) {
  const float x = r.unit ? l : div_by(l, r.T, r.rT);
  return ex2(fmaf(x, kLog2e, -r.mpb)) * r.inv_lp;
}
__device__ __forceinline__ float race_q(const RaceW& r, float l) {
  const float x = r.unit ? l : div_by(l, r.T, r.rT);
  return ex2(fmaf(x, kLog2e, -r.mqb)) * r.cq;
}
// p of the n valid entries of a group (the rest 0), and the weights w.
__device__ __forceinline__ float4 group_p(const RaceW& r, float4 x, int n) {
  return make_float4(n > 0 ? race_p(r, x.x) : 0.f, n > 1 ? race_p(r, x.y) : 0.f,
                     n > 2 ? race_p(r, x.z) : 0.f, n > 3 ? race_p(r, x.w) : 0.f);
}
__device__ __forceinline__ float4 group_w(const RaceW& r, float4 p, float4 xq, int n) {
  if (!r.resid) return p;
  return make_float4(n > 0 ? fmaxf(p.x - race_q(r, xq.x), 0.f) : 0.f,
                     n > 1 ? fmaxf(p.y - race_q(r, xq.y), 0.f) : 0.f,
                     n > 2 ? fmaxf(p.z - race_q(r, xq.z), 0.f) : 0.f,
                     n > 3 ? fmaxf(p.w - race_q(r, xq.w), 0.f) : 0.f);
}
__device__ __forceinline__ float sum4(float4 w) { return ((w.x + w.y) + w.z) + w.w; }

// Running best (W, E) of a lane: group g beats it iff W_g E_b > W_b E_g,
// lower index on ties.
__device__ __forceinline__ bool race_keep(float wg, float E, int g, float& bw, float& bE, int& bi) {
  const float lhs = wg * bE, rhs = bw * E;
  if (lhs > rhs || (lhs == rhs && g < bi)) {
    bw = wg;
    bE = E;
    bi = g;
    return true;
  }
  return false;
}

// Step 2 of the draw: the entry of group g (weights w, invalid entries 0)
// whose running sum first exceeds t = u W, with u from pick_u; at the very
// top of the range, the last positive entry.
__device__ __forceinline__ int pick_in_group(uint64_t seed, int i, int pos, int g, float4 w) {
  const float s1 = w.x, s2 = s1 + w.y, s3 = s2 + w.z, W = s3 + w.w;
  const float t = pick_u(seed, i, pos, g) * W;
  int k = t < s1 ? 0 : t < s2 ? 1 : t < s3 ? 2 : t < W ? 3 : -1;
  if (k < 0) k = w.w > 0.f ? 3 : w.z > 0.f ? 2 : w.y > 0.f ? 1 : 0;
  return 4 * g + k;
}

// Shared-memory ring of the vectorised race: per warp kRaceStages blocks in
// flight, each the block's target logits then (residual jobs) its draft
// logits, 2 KB apiece, filled by bulk copies.
constexpr int kRaceStages = 2;
constexpr int kRaceWarps = kRaceThreads / 32;
constexpr int kRaceStageFloats = 2 * kRaceBlock;
constexpr size_t kRaceSmem =
    (size_t)kRaceWarps * kRaceStages * (kRaceStageFloats * sizeof(float) + sizeof(uint64_t));

// The race kernel's last CTA: the commits tree walks left to it, one warp
// per request (kept out of line: the race's own code stays as small as it was)
__device__ __noinline__ void commit_deferred(const Args& a) {
  const Job* jobs = reinterpret_cast<const Job*>(a.ws + a.L.jobs);
  for (int i = (int)(threadIdx.x >> 5); i < a.bt.n_req; i += kRaceWarps)
    if (jobs[i].mode & 4) commit_request(a, i, true, nullptr);
}

// Warp-granular like the statistics: a warp scans one slice (whole blocks of
// 128 groups) of a request's row(s) and arrives on the request's ticket; the
// last one reduces and picks the entry.  With VEC the warp's logits stream
// through its ring, kRaceStages - 1 blocks ahead of their use, so that no
// step waits on a global load; else they are plain loads.
template <bool VEC>
__global__ void __launch_bounds__(kRaceThreads, 3) race_kernel(Args a) {
  griddep_entry();
  extern __shared__ __align__(128) uint8_t s_race[];
  const int* act = reinterpret_cast<const int*>(a.ws + a.L.act);
  const int R = a.bt.n_req;
  // the last CTA commits the requests whose tree walk left its commit here
  // (one warp per request), beside the race of the other CTAs
  const int ncta = (int)gridDim.x - (a.tree_commit_race ? 1 : 0);
  if ((int)blockIdx.x >= ncta) {
    commit_deferred(a);
    return;
  }
  const int count = a.race_all ? R : n_slots(a, act);
  const int V = a.V;
  int nch = race_slices(a.L, count, V);
  const int chl = (V + nch - 1) / nch + kRaceBlock - 1 - ((V + nch - 1) / nch + kRaceBlock - 1) % kRaceBlock;
  nch = (V + chl - 1) / chl;
  const long total = (long)count * nch;
  const float T = a.T;
  const float rT = 1.f / T;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // this warp's ring: stage buffers, then their barriers
  float* ring = reinterpret_cast<float*>(s_race) + (size_t)wid * kRaceStages * kRaceStageFloats;
  const uint32_t bar0 =
      smem_u32(s_race + (size_t)kRaceWarps * kRaceStages * kRaceStageFloats * 4) +
      (uint32_t)(wid * kRaceStages * 8);
  if (VEC) {
    if (lane == 0)
      for (int st = 0; st < kRaceStages; ++st) mbar_init(bar0 + 8 * st, 1);
    fence_mbar_init();
    __syncwarp();
  }
  uint32_t issued = 0, used = 0;  // blocks this warp has requested / consumed
  bool timed_out = false;
  const long stride = (long)ncta * kRaceWarps;
  for (long item = (long)blockIdx.x * kRaceWarps + wid; item < total && !timed_out;
       item += stride) {
    const int c = (int)(item % nch);
    const int i = a.race_all ? (int)(item / nch) : req_of(a, act, (int)(item / nch));
    // decide_request cleared every request's job before it could
    // return early (and, for a whole chunked step, the first chunk's list
    // pass cleared every request's), so a non-zero mode here was written by
    // this call.
    const Job jb = reinterpret_cast<const Job*>(a.ws + a.L.jobs)[i];
    const int md = jb.mode & 3;
    if (md != 1 && md != 2) continue;
    const bool resid = md == 1;
    const float* lp = a.target + (size_t)jb.row * V;
    const float* lq = a.draft + (size_t)jb.row * V;
    const float inv_lq = 1.f / jb.lq;
    const RaceW rw{T, rT, jb.mp * kLog2e, 1.f / jb.lp, jb.mq * kLog2e, jb.c * inv_lq, T == 1.f,
                   resid};
    const int lo = c * chl;
    const int hi = min(V, lo + chl);
    const int nb = (hi - lo + kRaceBlock - 1) / kRaceBlock;
    // Request block b of the slice into the ring (lane 0).
    auto request = [&](int b) {
      const int st = (int)(issued % kRaceStages);
      const int base = lo + b * kRaceBlock;
      const uint32_t bytes = (uint32_t)(min(hi, base + kRaceBlock) - base) * 4u;
      float* dst = ring + st * kRaceStageFloats;
      mbar_arrive_expect_tx(bar0 + 8 * st, resid ? 2u * bytes : bytes);
      bulk_load(smem_u32(dst), lp + base, bytes, bar0 + 8 * st);
      if (resid) bulk_load(smem_u32(dst + kRaceBlock), lq + base, bytes, bar0 + 8 * st);
    };
    if (VEC) {
      if (lane == 0)
        for (int b = 0; b < min(nb, kRaceStages); ++b, ++issued) request(b);
      __syncwarp();
      issued = __shfl_sync(0xffffffffu, issued, 0);
    }
    // valid entries of group k of the block at `base` (with VEC the vocabulary
    // is a multiple of 4: a group is whole or absent)
    auto nof = [&](int base, int k) {
      const int v = base + 128 * k + 4 * lane;
      return VEC ? (v < hi ? 4 : 0) : max(0, min(4, hi - v));
    };
    // Running best of this lane as (W, E).  K bounds the winner's key from
    // below: the best key this warp has seen, or any other warp of the
    // request (published in kbest, an atomic max on the bits of a
    // non-negative float, read one block ahead of its use), taken with a fast
    // division whose error the 2^-20 margin below covers.  W_g <= P_g (the
    // group's target mass) <= B_g = 4 p(max logit of the group) (p is
    // monotone in the logit; the factor 1 + 2^-16 covers the rounding of p
    // and of the sum), and E_g >= 1 - u_g, so a group with B_g < K (1 - u_g)
    // (less a 2^-20 margin) cannot win: its exact mass, draft probabilities
    // and logarithm are never computed.  While K is 0 (the first block) each
    // lane first keys its group with the largest B_g / (1 - u_g) exactly, and
    // the best of those keys bounds the rest.  The trip count is uniform
    // across the warp so that the lanes can share K.
    int* kbest = reinterpret_cast<int*>(a.ws + a.L.race_tickets) + R + i;
    float bw = -1.f, bE = 1.f, K = 0.f;
    int bi = 0x7fffffff;
    float4 bwv = make_float4(0.f, 0.f, 0.f, 0.f);  // weights of this lane's best group
    int kg_bits = 0;
    for (int b = 0; b < nb; ++b) {
      const int base = lo + b * kRaceBlock;
      const int st = (int)(used % kRaceStages);
      const float4* r4 = reinterpret_cast<const float4*>(ring + st * kRaceStageFloats);
      float4 xp[4];
      if (VEC) {
        if (!mbar_wait_sleep_bounded(bar0 + 8 * st, (used / kRaceStages) & 1u)) timed_out = true;
        timed_out = __any_sync(0xffffffffu, timed_out);
        if (timed_out) break;  // the block stays counted as in flight
#pragma unroll
        for (int k = 0; k < 4; ++k) xp[k] = r4[32 * k + lane];
      } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int v = base + 128 * k + 4 * lane;
          const int nk = nof(base, k);
          xp[k] = make_float4(nk > 0 ? lp[v] : -INFINITY, nk > 1 ? lp[v + 1] : -INFINITY,
                              nk > 2 ? lp[v + 2] : -INFINITY, nk > 3 ? lp[v + 3] : -INFINITY);
        }
      }
      if (b > 0) {
        // (one value for the whole warp: K decides warp-wide branches below)
        const float kg = __shfl_sync(0xffffffffu, __int_as_float(kg_bits), 0);
        const float mine = warp_max(bi == 0x7fffffff ? 0.f : __fdividef(bw, bE));
        if (lane == 0 && mine > kg) atomicMax(kbest, __float_as_int(mine));
        K = fmaxf(K, fmaxf(kg, mine));
        if (lane == 0) kg_bits = __ldcg(kbest);
      }
      const U4 bits = race_bits(a.seed, i, jb.pos, (base / kRaceBlock) * 32 + lane);
      const uint32_t wd[4] = {bits.a, bits.b, bits.c, bits.d};
      float Bk[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float mx = fmaxf(fmaxf(xp[k].x, xp[k].y), fmaxf(xp[k].z, xp[k].w));
        Bk[k] = nof(base, k) > 0 ? race_p(rw, mx) * (4.f * (1.f + 0x1p-16f)) : 0.f;
      }
      // Exact key of group k of this lane (all lanes at once).
      auto key_exact = [&](int k) {
        const int nk = nof(base, k);
        float4 xk, xq = make_float4(0.f, 0.f, 0.f, 0.f);
        uint32_t wk = wd[0];
#pragma unroll
        for (int t = 1; t < 4; ++t)
          if (k == t) wk = wd[t];
        if (VEC) {
          xk = r4[32 * k + lane];
          if (resid) xq = r4[kRaceBlock / 4 + 32 * k + lane];
        } else {
          const int v = base + 128 * k + 4 * lane;
          xk = make_float4(lp[v], nk > 1 ? lp[v + 1] : 0.f, nk > 2 ? lp[v + 2] : 0.f,
                           nk > 3 ? lp[v + 3] : 0.f);
          if (resid)
            xq = make_float4(lq[v], nk > 1 ? lq[v + 1] : 0.f, nk > 2 ? lq[v + 2] : 0.f,
                             nk > 3 ? lq[v + 3] : 0.f);
        }
        const float4 w4 = group_w(rw, group_p(rw, xk, nk), xq, nk);
        if (race_keep(sum4(w4), -logf(race_u(wk)), base / 4 + 32 * k + lane, bw, bE, bi))
          bwv = w4;
      };
      unsigned todo = 0;  // groups of this lane still to key exactly
      if (K == 0.f) {
        // Start (the first block): each lane keys its group with the largest
        // bound B_g / (1 - u_g); the best of those keys bounds the rest.
        float ub = -1.f;
        int kk = -1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float c = nof(base, k) > 0 ? __fdividef(Bk[k], 1.f - race_u(wd[k])) : -1.f;
          if (c > ub) { ub = c; kk = k; }
        }
        if (kk >= 0) key_exact(kk);
        K = warp_max(bi == 0x7fffffff ? 0.f : __fdividef(bw, bE));
        const float Km = K * (1.f - 0x1p-20f);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k != kk && nof(base, k) > 0 && !(Bk[k] < Km * (1.f - race_u(wd[k]))))
            todo |= 1u << k;
      } else {
        const float Km = K * (1.f - 0x1p-20f);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (nof(base, k) > 0 && !(Bk[k] < Km * (1.f - race_u(wd[k])))) todo |= 1u << k;
      }
      // Usually no group of the warp is left: a warp-wide test, so that the
      // exact path is not issued at all then; else the lanes key their
      // remaining groups side by side.
      while (__any_sync(0xffffffffu, todo != 0)) {
        if (todo) {
          const int k = __ffs(todo) - 1;
          todo &= todo - 1;
          key_exact(k);
        }
      }
      if (VEC) {
        // the stage is read: refill it with block b + kRaceStages
        ++used;
        __syncwarp();
        if (b + kRaceStages < nb) {
          if (lane == 0) {
            fence_proxy_async_smem();
            request(b + kRaceStages);
          }
          ++issued;
        }
      }
    }
    if (timed_out) break;
    // The warp's best group, and its entry drawn by the lane that holds it
    // (the same weights the last warp would compute from the logits).
    float best = bi == 0x7fffffff ? -1.f : bw / bE;
    const int own = bi;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      race_take(best, bi, b2, i2);
    }
    const bool holder = bi != 0x7fffffff && own == bi;
    const int tok_own = holder ? pick_in_group(a.seed, i, jb.pos, bi, bwv) : -1;
    const unsigned hm = __ballot_sync(0xffffffffu, holder);
    const int tok = __shfl_sync(0xffffffffu, tok_own, hm ? __ffs(hm) - 1 : 0);
    RacePart* parts = reinterpret_cast<RacePart*>(a.ws + a.L.race) + (size_t)i * nch;
    int* ticket = reinterpret_cast<int*>(a.ws + a.L.race_tickets) + i;
    int last = 0;
    if (lane == 0) {
      parts[c].key = best;
      parts[c].idx = bi;
      parts[c].tok = tok;
      last = ticket_add(ticket, 1) == nch - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      // last slice of request i: the winning group (its entry drawn already),
      // eight slices' loads in flight per lane
      __syncwarp();
      float bk = -1.f;
      int g = 0x7fffffff, tk = -1;
      for (int k0 = lane; k0 < nch; k0 += 32 * 8) {
        float kk[8];
        int gg[8], tt[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int k = k0 + 32 * j;
          kk[j] = k < nch ? __ldcg(&parts[k].key) : -1.f;
          gg[j] = k < nch ? __ldcg(&parts[k].idx) : 0x7fffffff;
          tt[j] = k < nch ? __ldcg(&parts[k].tok) : -1;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) race_take(bk, g, tk, kk[j], gg[j], tt[j]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float b2 = __shfl_xor_sync(0xffffffffu, bk, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, g, o);
        const int t2 = __shfl_xor_sync(0xffffffffu, tk, o);
        race_take(bk, g, tk, b2, i2, t2);
      }
      if (lane == 0) {
        // every non-empty slice finds a group; none: an empty vocabulary set
        a.next_token[i] = (g >= 0 && g < (V + 3) / 4) ? tk : -1;
        *ticket = 0;
      }
    }
  }
  if (timed_out && lane == 0) {
    // a copy that never completed: report, and wait (bounded) for every copy
    // still in flight so that none lands after the warp has gone
    flag(a.dev_status, SV_DEV_TIMEOUT);
    for (; used < issued; ++used)
      mbar_wait_sleep_bounded(bar0 + 8 * (int)(used % kRaceStages), (used / kRaceStages) & 1u);
  }
}

// ------------------------------------------------------------------ host --

static sv_status check_accept_args(const sv_batch* bt, const float* target_logits,
                                   const float* draft_logits, int32_t vocab, float temperature,
                                   const int32_t* accepted_len, const int32_t* accepted_nodes,
                                   const int32_t* next_token, const uint8_t* ambiguous,
                                   const void* ws) {
  if (!bt || bt->n_req < 0 || bt->total_rows < 0 || vocab < 1) return SV_ERR_INVALID_ARGUMENT;
  if (!(temperature >= 0.f) || isinf(temperature)) return SV_ERR_INVALID_ARGUMENT;
  if (bt->max_rows_per_req < 1) return SV_ERR_INVALID_ARGUMENT;
  if (bt->max_rows_per_req > kMaxRows) return SV_ERR_UNSUPPORTED_SHAPE;
  if (bt->n_req == 0 || bt->total_rows == 0) return SV_OK;
  if (!bt->cu_rows || !bt->parent || !bt->tokens || !target_logits || !accepted_len ||
      !accepted_nodes || !next_token || !ambiguous || !ws)
    return SV_ERR_INVALID_ARGUMENT;
  if (temperature > 0.f && !draft_logits) return SV_ERR_INVALID_ARGUMENT;
  if ((uintptr_t)ws & 255) return SV_ERR_INVALID_ARGUMENT;
  return SV_OK;
}

static sv_status launch_race(const Args& a, bool vec, cudaStream_t s) {
  const long ritems = (long)a.bt.n_req * a.L.nch_r_cap;
  const long rwarps = kRaceThreads / 32;
  const unsigned gr = (unsigned)max(
      1L, min((ritems + rwarps - 1) / rwarps, (long)a.L.nsm * kRaceWarpsPerSM / rwarps));
  if (vec) {
    static PerDevice smem_set;  // the ring is above the 48 KB default
    if (smem_limit_once(smem_set, race_kernel<true>, kRaceSmem) != cudaSuccess) return SV_ERR_CUDA;
  }
  if (sv::launch(vec ? race_kernel<true> : race_kernel<false>, gr + (a.tree_commit_race ? 1u : 0u),
                 kRaceThreads, vec ? kRaceSmem : 0, s, a) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

static bool vec_ok(int32_t vocab, const float* target_logits, const float* draft_logits) {
  return (vocab % 4 == 0) &&
         ((((uintptr_t)target_logits) | ((uintptr_t)(draft_logits ? draft_logits : target_logits))) &
          15) == 0;
}

// Enqueue the statistics, the decision and the race; in a chunked step
// (chunk_index >= 0) the kernels take the attention planner's list and the
// race is left to race_all after the last chunk.
sv_status run(const sv_batch* bt, const float* target_logits, const float* draft_logits,
              int32_t vocab, float temperature, uint64_t seed, int32_t* accepted_len,
              int32_t* accepted_nodes, int32_t* next_token, uint8_t* ambiguous, int32_t* done,
              float* row_stats, void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t s,
              int maxw, int chunk_index, const sv_paged_kv* commit_kv,
              const sv_block_pool* commit_pool, const int4* act4) {
  const bool chunk_step = chunk_index >= 0;
  sv_status st = check_accept_args(bt, target_logits, draft_logits, vocab, temperature,
                                   accepted_len, accepted_nodes, next_token, ambiguous, ws);
  if (st != SV_OK || bt->n_req == 0 || bt->total_rows == 0) return st;
  Args a;
  a.bt = *bt;
  a.target = target_logits;
  a.draft = draft_logits;
  a.V = vocab;
  a.T = temperature;
  a.seed = seed;
  a.accepted_len = accepted_len;
  a.accepted_nodes = accepted_nodes;
  a.next_token = next_token;
  a.ambiguous = ambiguous;
  a.done = done;
  a.row_stats = row_stats;
  a.ws = static_cast<uint8_t*>(ws);
  const bool commit = commit_kv != nullptr;
  if (commit && (!commit_pool || (chunk_step && !done))) return SV_ERR_INVALID_ARGUMENT;
  a.L = layout(bt->n_req, bt->total_rows, vocab, maxw, commit);
  a.dev_status = dev_status;
  a.race_all = 0;
  a.clear_jobs = chunk_index == 0 ? 1 : 0;
  a.commit = commit ? 1 : 0;
  // one-pass calls at T > 0 run the race after the tree walk: it takes the
  // walks' commits
  a.tree_commit_race = commit && !chunk_step && temperature > 0.f ? 1 : 0;
  a.kv = CommitArgs{};
  if (commit) {
    a.kv.k = static_cast<__nv_bfloat16*>(commit_kv->k_cache);
    a.kv.v = static_cast<__nv_bfloat16*>(commit_kv->v_cache);
    a.kv.num_blocks = commit_kv->num_blocks;
    a.kv.Hkv = commit_kv->n_kv_heads;
    a.kv.D = commit_kv->head_dim;
    a.kv.max_blocks = commit_kv->max_blocks_per_req;
    a.kv.tables = commit_kv->block_tables;
    a.kv.cache_lens = commit_kv->cache_lens;
    a.kv.free_list = commit_pool->free_list;
    a.kv.free_count = commit_pool->free_count;
    a.kv.capacity = commit_pool->capacity;
  }
  if (ws_bytes < a.L.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  // Logits of a small call (up to kKeepL2Bytes) are loaded so that they stay
  // in L2 for the decision and the race; larger ones stream past it.
  const long stat_rows = min((long)bt->total_rows, (long)bt->n_req * a.L.maxw);
  a.keep_l2 = stat_rows * vocab * 4L * (temperature > 0.f ? 2 : 1) <= kKeepL2Bytes ? 1 : 0;
  const bool vec = vec_ok(vocab, target_logits, draft_logits);
  a.use_list = chunk_step ? 1 : 0;
  a.act4 = chunk_step ? act4 : nullptr;
  const long items = (long)bt->n_req * a.L.maxw * (temperature > 0.f ? 2 : 1) * a.L.nch_cap;
  const long warps = kStatThreads / 32;
  const unsigned gs = (unsigned)max(1L, min((items + warps - 1) / warps, (long)a.L.nsm * 4));
  auto stats = a.keep_l2 ? (vec ? stats_kernel<true, true> : stats_kernel<false, true>)
                         : (vec ? stats_kernel<true, false> : stats_kernel<false, false>);
  if (sv::launch(stats, gs, kStatThreads, 0, s, a) != cudaSuccess) return SV_ERR_CUDA;
  const unsigned gd = (unsigned)max(1, min((bt->n_req + kDecideWarps - 1) / kDecideWarps, a.L.nsm * 8));
  if (sv::launch(decide_kernel, gd, kDecideWarps * 32, 0, s, a) != cudaSuccess) return SV_ERR_CUDA;
  if (temperature > 0.f && bt->max_rows_per_req > 2 &&
      (!chunk_step || (chunk_index == 0 && a.L.maxw > 2))) {
    // draft trees at T > 0 (requests the decision marked); the other CTAs
    // exit at once.  A tree is verified in one window: in a chunked step only
    // the first chunk, and only when a chunk holds more than a chain's two
    // rows, can take one whole.
    static ClusterFit tree_fit;
    const bool clu =
        bt->max_rows_per_req >= kTreeClusterMinRows &&
        tree_fit.get(tree_kernel<kTreeClusterThreads, kTreeCluster>, kTreeCluster,
                     kTreeClusterThreads, 0) > 0;
    const cudaError_t e =
        clu ? sv::launch_cluster(tree_kernel<kTreeClusterThreads, kTreeCluster>,
                                 (unsigned)bt->n_req * kTreeCluster, kTreeClusterThreads, 0, s,
                                 kTreeCluster, a)
            : sv::launch(tree_kernel<kTreeThreads, 1>, (unsigned)bt->n_req, kTreeThreads, 0, s, a);
    if (e != cudaSuccess) return SV_ERR_CUDA;
  }
  if (temperature > 0.f && !chunk_step) return launch_race(a, vec, s);
  return SV_OK;
}

sv_status race_all(const sv_batch* bt, const float* target_logits, const float* draft_logits,
                   int32_t vocab, float temperature, uint64_t seed, int32_t* next_token, void* ws,
                   int maxw, int32_t* dev_status, cudaStream_t s) {
  if (!(temperature > 0.f) || bt->n_req == 0 || bt->total_rows == 0) return SV_OK;
  Args a{};
  a.bt = *bt;
  a.target = target_logits;
  a.draft = draft_logits;
  a.V = vocab;
  a.T = temperature;
  a.seed = seed;
  a.next_token = next_token;
  a.ws = static_cast<uint8_t*>(ws);
  a.L = layout(bt->n_req, bt->total_rows, vocab, maxw, false);
  a.dev_status = dev_status;
  a.race_all = 1;
  a.clear_jobs = 0;
  a.use_list = 0;
  a.commit = 0;
  return launch_race(a, vec_ok(vocab, target_logits, draft_logits), s);
}

}  // namespace acc
}  // namespace sv

using namespace sv;

extern "C" size_t sv_accept_workspace(const sv_batch* bt, int32_t vocab) {
  if (!bt || bt->n_req < 0 || bt->total_rows < 0 || vocab < 1) return 0;
  return acc::layout(bt->n_req, bt->total_rows, vocab, bt->max_rows_per_req, false).total;
}

extern "C" sv_status sv_accept(const sv_batch* bt, const float* target_logits,
                               const float* draft_logits, int32_t vocab, float temperature,
                               uint64_t seed, int32_t* accepted_len, int32_t* accepted_nodes,
                               int32_t* next_token, uint8_t* ambiguous, int32_t* done,
                               float* row_stats, void* ws, size_t ws_bytes, int32_t* dev_status,
                               void* stream) {
  SV_TRACE("sv_accept");
  if (!bt) return SV_ERR_INVALID_ARGUMENT;
  return acc::run(bt, target_logits, draft_logits, vocab, temperature, seed, accepted_len,
                  accepted_nodes, next_token, ambiguous, done, row_stats, ws, ws_bytes, dev_status,
                  static_cast<cudaStream_t>(stream), bt->max_rows_per_req, -1);
}

// ------------------------------------------------- accept + commit fused --
extern "C" size_t sv_accept_commit_workspace(const sv_batch* bt, int32_t vocab) {
  if (!bt || bt->n_req < 0 || bt->total_rows < 0 || vocab < 1) return 0;
  return acc::layout(bt->n_req, bt->total_rows, vocab, bt->max_rows_per_req, true).total;
}

extern "C" sv_status sv_accept_commit(const sv_batch* bt, const float* target_logits,
                                      const float* draft_logits, int32_t vocab, float temperature,
                                      uint64_t seed, int32_t* accepted_len,
                                      int32_t* accepted_nodes, int32_t* next_token,
                                      uint8_t* ambiguous, int32_t* done, float* row_stats,
                                      const sv_paged_kv* kv, const sv_block_pool* pool, void* ws,
                                      size_t ws_bytes, int32_t* dev_status, void* stream) {
  SV_TRACE("sv_accept_commit");
  if (!bt || !kv || !pool) return SV_ERR_INVALID_ARGUMENT;
  if (kv->block_size != kBlockSize) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->head_dim != 64 && kv->head_dim != 128) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->n_kv_heads < 1 || kv->num_blocks < 0 || kv->max_blocks_per_req < 0 ||
      pool->capacity < 0)
    return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req > 0 && (!kv->k_cache || !kv->v_cache || !kv->block_tables || !kv->cache_lens ||
                        !pool->free_list || !pool->free_count))
    return SV_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)kv->k_cache | (uintptr_t)kv->v_cache) & 15) return SV_ERR_INVALID_ARGUMENT;
  return acc::run(bt, target_logits, draft_logits, vocab, temperature, seed, accepted_len,
                  accepted_nodes, next_token, ambiguous, done, row_stats, ws, ws_bytes, dev_status,
                  static_cast<cudaStream_t>(stream), bt->max_rows_per_req, -1, kv, pool);
}

// ------------------------------------------------ no-allocation variant ----
// sv_accept_static: sv_accept without a caller workspace.  Its scratch is the
// file-scope device array below, which every GPU that loads the library keeps
// until the process exits.  The address of that array on the current device
// is looked up once per device (cudaGetSymbolAddress) on the first call made
// with that device current; make that first call before any stream capture.
// The cached address belongs to the device's context as it was then: after a
// device reset it is stale, so the header tells callers not to use this entry
// point on a device they have reset.  All calls share the array: two calls whose work overlaps on the GPU (for
// example on two streams) race on it.  Nothing in it has to start at zero:
// the accept kernels write every scratch word before they read it (the
// decision clears every request's sampling job and race ticket before
// anything reads them, and the statistics write every partial the decision
// merges).


namespace {

static __device__ __align__(256) uint8_t g_accept_scratch[SV_ACCEPT_STATIC_SCRATCH_BYTES];

std::mutex g_accept_scratch_mu;
constexpr int kMaxDevices = 64;
void* g_accept_scratch_addr[kMaxDevices] = {};

sv_status accept_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_accept_scratch_mu);
  if (!g_accept_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess || !p) return SV_ERR_CUDA;
    g_accept_scratch_addr[dev] = p;
  }
  *out = g_accept_scratch_addr[dev];
  return SV_OK;
}

}  // namespace

extern "C" sv_status sv_accept_static(const sv_batch* bt, const float* target_logits,
                                      const float* draft_logits, int32_t vocab, float temperature,
                                      uint64_t seed, int32_t* accepted_len,
                                      int32_t* accepted_nodes, int32_t* next_token,
                                      uint8_t* ambiguous, int32_t* done, float* row_stats,
                                      int32_t* dev_status, void* stream) {
  SV_TRACE("sv_accept_static");
  if (!bt || bt->n_req < 0 || bt->total_rows < 0 || vocab < 1) return SV_ERR_INVALID_ARGUMENT;
  const size_t need = sv_accept_workspace(bt, vocab);
  if (need > (size_t)SV_ACCEPT_STATIC_SCRATCH_BYTES) return SV_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const sv_status st = accept_scratch_address(&scratch);
  if (st != SV_OK) return st;
  return sv_accept(bt, target_logits, draft_logits, vocab, temperature, seed, accepted_len,
                   accepted_nodes, next_token, ambiguous, done, row_stats, scratch,
                   (size_t)SV_ACCEPT_STATIC_SCRATCH_BYTES, dev_status, stream);
}
