// accept.cu — sv_accept: per-row vocabulary softmax statistics and the
// lossless accept / reject rule (or greedy longest matching prefix).
//
// Sources: [DSpark] glossary ("사전검증 디코딩": the longest matching prefix is
// accepted and the target distribution is preserved); [FASER] mechanism 1
// (per-request number of drafts) and mechanism 2 (a request stops at its
// first rejection; chunks of rows).  The accept / reject formula itself is
// the standard lossless speculative-sampling rule (not printed on the pages).
//
// Kernels, in stream order:
//   stats  (grid: row x vocab chunk x {target, draft})
//          one pass over the row with 128-bit loads: online max / sum of
//          exp(x - max) of x = logit / T (T > 0), or max and lowest-index
//          argmax of the raw logits (T = 0); one partial per chunk.
//   decide (one warp per request)
//          merges the partials of the rows it needs, then scans the chain
//          (or runs the tree descent) with Philox uniforms; writes the path
//          and, for T > 0, a sampling job for the emitted token.
//   race   (grid: request x vocab chunk)
//          the exponential race argmax_v w_v / E_v over the job's row(s),
//          w = max(0, p - q) after a rejection or p for the bonus token; the
//          last CTA of a request (atomic ticket) reduces the chunk winners.

#include <math.h>

#include "sv_internal.cuh"

namespace sv {
namespace acc {

struct StatPart {
  float m;      // T > 0: max of x; T == 0: max raw logit
  float l;      // T > 0: sum exp(x - m)
  int amax;     // T == 0: lowest index of the max
  int pad;
};

struct Job {
  int mode;     // 0 none, 1 residual, 2 bonus
  int row;      // packed row of the target (and draft) logits
  int pos;      // position of the emitted token
  int pad;
  float mp, lp, mq, lq;
};

struct RacePart {
  float key;
  int idx;
};

constexpr int kStatThreads = 256;
constexpr int kRaceThreads = 256;
constexpr int kDecideWarps = 4;

inline int stats_chunks(int total_rows, int V) {
  const int maxc = max(1, min(64, V / 1024));
  const int want = (kNumSMs * 32 + 2 * total_rows - 1) / max(1, 2 * total_rows);
  return max(1, min(want, maxc));
}
inline int race_chunks(int R, int V) {
  const int maxc = max(1, min(256, V / 1024));
  const int want = (kNumSMs * 16 + R - 1) / max(1, R);
  return max(1, min(want, maxc));
}
inline int chunk_len(int V, int nch) { return ((V + nch - 1) / nch + 3) & ~3; }

struct Layout {
  size_t parts, jobs, race, tickets, total;
  int nch, nch_r, ch, ch_r;
};

inline Layout layout(int R, int total_rows, int V) {
  Layout L;
  L.nch = stats_chunks(total_rows, V);
  L.nch_r = race_chunks(R, V);
  L.ch = chunk_len(V, L.nch);
  L.ch_r = chunk_len(V, L.nch_r);
  size_t off = 0;
  L.parts = off; off += align256(sizeof(StatPart) * (size_t)total_rows * 2 * L.nch);
  L.jobs = off; off += align256(sizeof(Job) * (size_t)R);
  L.race = off; off += align256(sizeof(RacePart) * (size_t)R * L.nch_r);
  L.tickets = off; off += align256(sizeof(int) * (size_t)R);
  L.total = off;
  return L;
}

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
};

__device__ __forceinline__ void merge_ml(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  l = l * expf(m - M) + l2 * expf(m2 - M);
  m = M;
}
__device__ __forceinline__ void merge_am(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}

// ----------------------------------------------------------------- stats --
template <bool VEC>
__global__ void __launch_bounds__(kStatThreads) stats_kernel(Args a) {
  const int nch = a.L.nch;
  const int c = blockIdx.x % nch;
  const int r = blockIdx.x / nch;
  const int type = blockIdx.y;
  if (r >= a.bt.total_rows) return;
  const int R = a.bt.n_req;
  const int i = find_segment(a.bt.cu_rows, R, r);
  const Window w = window_of(a.bt, i);
  const int j = r - a.bt.cu_rows[i];
  if (!w.ok || j < w.b || j >= w.e) return;
  if (w.b > 0 && a.next_token[i] >= 0) return;      // decided in an earlier window
  if (type == 1 && (a.T == 0.f || j + 1 > w.lim - 1)) return;
  const float* row = (type ? a.draft : a.target) + (size_t)r * a.V;
  const int lo = c * a.L.ch;
  const int hi = min(a.V, lo + a.L.ch);
  const float T = a.T;
  float m = -INFINITY, l = 0.f;
  int am = 0x7fffffff;
  if (T > 0.f) {
    if (VEC) {
      const float4* p4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
      for (int v = lo + 4 * threadIdx.x; v < hi; v += 4 * kStatThreads) {
        const float4 x4 = __ldcs(p4 + (v >> 2));
        const float x0 = x4.x / T, x1 = x4.y / T, x2 = x4.z / T, x3 = x4.w / T;
        const float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
        if (mx > m) {
          l *= expf(m - mx);
          m = mx;
        }
        l += expf(x0 - m) + expf(x1 - m) + expf(x2 - m) + expf(x3 - m);
      }
    } else {
      for (int v = lo + threadIdx.x; v < hi; v += kStatThreads) {
        const float x = row[v] / T;
        if (x > m) {
          l *= expf(m - x);
          m = x;
        }
        l += expf(x - m);
      }
    }
  } else {
    if (VEC) {
      const float4* p4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
      for (int v = lo + 4 * threadIdx.x; v < hi; v += 4 * kStatThreads) {
        const float4 x4 = __ldcs(p4 + (v >> 2));
        if (x4.x > m) { m = x4.x; am = v; }
        if (x4.y > m) { m = x4.y; am = v + 1; }
        if (x4.z > m) { m = x4.z; am = v + 2; }
        if (x4.w > m) { m = x4.w; am = v + 3; }
      }
    } else {
      for (int v = lo + threadIdx.x; v < hi; v += kStatThreads) {
        const float x = row[v];
        if (x > m) { m = x; am = v; }
      }
    }
  }
  // block reduction
  __shared__ float s_m[kStatThreads / 32], s_l[kStatThreads / 32];
  __shared__ int s_i[kStatThreads / 32];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, am, o);
    if (T > 0.f) merge_ml(m, l, m2, l2); else merge_am(m, am, m2, i2);
  }
  if (lane == 0) { s_m[wid] = m; s_l[wid] = l; s_i[wid] = am; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < kStatThreads / 32; ++k) {
      if (T > 0.f) merge_ml(m, l, s_m[k], s_l[k]); else merge_am(m, am, s_m[k], s_i[k]);
    }
    StatPart sp;
    sp.m = m;
    sp.l = l;
    sp.amax = am;
    sp.pad = 0;
    reinterpret_cast<StatPart*>(a.ws + a.L.parts)[((size_t)r * 2 + type) * nch + c] = sp;
  }
}

// ---------------------------------------------------------------- decide --
__device__ __forceinline__ void row_ml(const Args& a, int r, int type, float& m, float& l) {
  const StatPart* parts = reinterpret_cast<const StatPart*>(a.ws + a.L.parts) +
                          ((size_t)r * 2 + type) * a.L.nch;
  const int lane = threadIdx.x & 31;
  m = -INFINITY;
  l = 0.f;
  for (int c = lane; c < a.L.nch; c += 32) merge_ml(m, l, parts[c].m, parts[c].l);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    merge_ml(m, l, m2, l2);
  }
}

__device__ __forceinline__ void row_argmax(const Args& a, int r, float& v, int& idx) {
  const StatPart* parts = reinterpret_cast<const StatPart*>(a.ws + a.L.parts) +
                          ((size_t)r * 2) * a.L.nch;
  const int lane = threadIdx.x & 31;
  v = -INFINITY;
  idx = 0x7fffffff;
  for (int c = lane; c < a.L.nch; c += 32) merge_am(v, idx, parts[c].m, parts[c].amax);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    merge_am(v, idx, v2, i2);
  }
}

__global__ void __launch_bounds__(kDecideWarps * 32) decide_kernel(Args a) {
  __shared__ float s_mp[kDecideWarps][kMaxRows], s_lp[kDecideWarps][kMaxRows];
  __shared__ float s_mq[kDecideWarps][kMaxRows], s_lq[kDecideWarps][kMaxRows];
  __shared__ int s_am[kDecideWarps][kMaxRows];
  __shared__ int s_len[kDecideWarps][kMaxRows], s_child[kDecideWarps][kMaxRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x * kDecideWarps + warp;
  if (i >= a.bt.n_req) return;
  Job* job = reinterpret_cast<Job*>(a.ws + a.L.jobs) + i;
  if (a.T > 0.f && lane == 0) {
    // Only jobs created by this call may reach the race kernel.
    job->mode = 0;
    reinterpret_cast<int*>(a.ws + a.L.tickets)[i] = 0;
  }
  const Window w = window_of(a.bt, i);
  if (!w.ok) {
    if (lane == 0) flag(a.dev_status, SV_DEV_BAD_WINDOW);
    return;
  }
  if (w.b >= w.e) return;
  const int cu = a.bt.cu_rows[i];
  const int V = a.V;
  bool chain = true, badp = false, badt = false;
  for (int j = lane; j < w.rows; j += 32) {
    const int p = a.bt.parent[cu + j];
    if (j == 0) {
      if (p != -1) badp = true;
    } else {
      if (p < 0 || p >= j) badp = true;
      if (p != j - 1) chain = false;
      const int t = a.bt.tokens[cu + j];
      if (t < 0 || t >= V) badt = true;
    }
  }
  badp = __any_sync(0xffffffffu, badp);
  badt = __any_sync(0xffffffffu, badt);
  chain = __all_sync(0xffffffffu, chain);
  if (badp || badt || (!chain && (w.b != 0 || w.e != w.rows)) || (!chain && a.T > 0.f)) {
    if (lane == 0)
      flag(a.dev_status, badp ? SV_DEV_BAD_PARENT
                              : badt ? SV_DEV_BAD_TOKEN
                                     : (!chain && a.T > 0.f && w.b == 0 && w.e == w.rows)
                                           ? SV_DEV_UNSUPPORTED
                                           : SV_DEV_BAD_WINDOW);
    return;
  }
  const int max_rows = a.bt.max_rows_per_req;
  int32_t* nodes = a.accepted_nodes + (size_t)i * max_rows;
  if (w.b == 0) {
    for (int k = lane; k < max_rows; k += 32) nodes[k] = k == 0 ? 0 : -1;
  } else {
    const int nt = a.next_token[i], al = a.accepted_len[i];
    if (nt >= 0) return;  // decided in an earlier window
    if (al != w.b) {
      if (lane == 0) flag(a.dev_status, SV_DEV_BAD_WINDOW);
      return;
    }
  }
  int len = w.b;   // accepted drafts so far
  int next = -1;
  bool amb = false;
  float* rs = a.row_stats;

  if (a.T == 0.f) {
    for (int r = w.b; r < w.e; ++r) {
      float v;
      int idx;
      row_argmax(a, cu + r, v, idx);
      if (lane == 0) {
        s_am[warp][r] = idx;
        if (rs) {
          rs[(size_t)(cu + r) * 4 + 0] = v;
          rs[(size_t)(cu + r) * 4 + 1] = (float)idx;
        }
      }
    }
    __syncwarp();
    if (chain) {
      if (lane == 0) {
        const int jmax = min(w.e, w.lim - 1);
        for (int j = w.b + 1; j <= jmax; ++j) {
          const int am = s_am[warp][j - 1];
          if (a.bt.tokens[cu + j] == am) {
            len = j;
            nodes[j] = j;
          } else {
            next = am;
            break;
          }
        }
        if (next < 0 && w.e == w.lim && len == w.lim - 1) next = s_am[warp][w.lim - 1];
      }
    } else {
      // tree: longest valid path, lower node index on ties (bottom-up)
      for (int n = w.rows - 1; n >= 0; --n) {
        int best = 0, bc = -1;
        for (int c = n + 1 + lane; c < w.rows; c += 32) {
          if (a.bt.parent[cu + c] == n && a.bt.tokens[cu + c] == s_am[warp][n]) {
            const int cand = 1 + s_len[warp][c];
            if (cand > best || (cand == best && bc >= 0 && c < bc)) { best = cand; bc = c; }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const int b2 = __shfl_xor_sync(0xffffffffu, best, o);
          const int c2 = __shfl_xor_sync(0xffffffffu, bc, o);
          if (b2 > best || (b2 == best && c2 >= 0 && (bc < 0 || c2 < bc))) { best = b2; bc = c2; }
        }
        if (lane == 0) {
          s_len[warp][n] = best;
          s_child[warp][n] = bc;
        }
        __syncwarp();
      }
      if (lane == 0) {
        int n = 0, k = 0;
        while (s_child[warp][n] >= 0) {
          n = s_child[warp][n];
          nodes[++k] = n;
        }
        len = k;
        next = s_am[warp][n];
      }
    }
    if (lane == 0) {
      a.accepted_len[i] = len;
      a.next_token[i] = next;
      if (w.b == 0) a.ambiguous[i] = 0;
      if (a.done) a.done[i] = next >= 0 ? 1 : 0;
    }
    return;
  }

  // ---- T > 0: speculative sampling on a chain ----
  const int jmax = min(w.e, w.lim - 1);
  for (int r = w.b; r < w.e; ++r) {
    float m, l;
    row_ml(a, cu + r, 0, m, l);
    if (lane == 0) {
      s_mp[warp][r] = m;
      s_lp[warp][r] = l;
      if (rs) rs[(size_t)(cu + r) * 4 + 0] = m + logf(l);
    }
    if (r + 1 <= w.lim - 1) {
      row_ml(a, cu + r, 1, m, l);
      if (lane == 0) {
        s_mq[warp][r] = m;
        s_lq[warp][r] = l;
        if (rs) rs[(size_t)(cu + r) * 4 + 1] = m + logf(l);
      }
    }
  }
  __syncwarp();
  if (lane != 0) return;
  const float T = a.T;
  Job jb;
  jb.mode = 0;
  jb.pad = 0;
  for (int j = w.b + 1; j <= jmax; ++j) {
    const int x = a.bt.tokens[cu + j];
    const size_t off = (size_t)(cu + j - 1) * V + x;
    const float xp = a.target[off] / T;
    const float xq = a.draft[off] / T;
    const double p = exp((double)xp - (double)s_mp[warp][j - 1]) / (double)s_lp[warp][j - 1];
    const double q = exp((double)xq - (double)s_mq[warp][j - 1]) / (double)s_lq[warp][j - 1];
    if (rs) {
      rs[(size_t)(cu + j) * 4 + 2] = (float)p;
      rs[(size_t)(cu + j) * 4 + 3] = (float)q;
    }
    const double ratio = q > 0.0 ? fmin(1.0, p / q) : 1.0;
    const double u = (double)accept_u(a.seed, i, j);
    if (fabs(u - ratio) < 1e-6) amb = true;
    if (u < ratio) {
      len = j;
      nodes[j] = j;
    } else {
      jb.mode = 1;
      jb.row = cu + j - 1;
      jb.pos = j;
      jb.mp = s_mp[warp][j - 1];
      jb.lp = s_lp[warp][j - 1];
      jb.mq = s_mq[warp][j - 1];
      jb.lq = s_lq[warp][j - 1];
      break;
    }
  }
  if (jb.mode == 0 && w.e == w.lim && len == w.lim - 1) {
    jb.mode = 2;
    jb.row = cu + w.lim - 1;
    jb.pos = w.lim;
    jb.mp = s_mp[warp][w.lim - 1];
    jb.lp = s_lp[warp][w.lim - 1];
    jb.mq = 0.f;
    jb.lq = 1.f;
  }
  *job = jb;
  reinterpret_cast<int*>(a.ws + a.L.tickets)[i] = 0;
  a.accepted_len[i] = len;
  a.next_token[i] = -1;
  if (w.b == 0) a.ambiguous[i] = 0;
  if (amb) a.ambiguous[i] = 1;
  if (a.done) a.done[i] = jb.mode != 0 ? 1 : 0;
}

// ------------------------------------------------------------------ race --
__device__ __forceinline__ void race_take(float& best, int& bi, float key, int v) {
  if (key > best || (key == best && v < bi)) { best = key; bi = v; }
}

template <bool VEC>
__global__ void __launch_bounds__(kRaceThreads) race_kernel(Args a) {
  const int nch = a.L.nch_r;
  const int c = blockIdx.x % nch;
  const int i = blockIdx.x / nch;
  // decide_kernel clears every request's job before it can return early,
  // so a non-zero mode here was written by this call.
  const Job jb = reinterpret_cast<const Job*>(a.ws + a.L.jobs)[i];
  if (jb.mode == 0) return;
  const float T = a.T;
  const bool resid = jb.mode == 1;
  const float* lp = a.target + (size_t)jb.row * a.V;
  const float* lq = a.draft + (size_t)jb.row * a.V;
  const float inv_lp = 1.f / jb.lp, inv_lq = 1.f / jb.lq;
  const int lo = c * a.L.ch_r;
  const int hi = min(a.V, lo + a.L.ch_r);
  float best = -1.f;
  int bi = 0x7fffffff;
  if (VEC) {
    for (int v = lo + 4 * threadIdx.x; v < hi; v += 4 * kRaceThreads) {
      const U4 bits = race_bits(a.seed, i, jb.pos, v >> 2);
      const float4 xp = __ldcs(reinterpret_cast<const float4*>(lp) + (v >> 2));
      float4 xq = make_float4(0.f, 0.f, 0.f, 0.f);
      if (resid) xq = __ldcs(reinterpret_cast<const float4*>(lq) + (v >> 2));
      const float pv[4] = {xp.x, xp.y, xp.z, xp.w};
      const float qv[4] = {xq.x, xq.y, xq.z, xq.w};
      const uint32_t bv[4] = {bits.a, bits.b, bits.c, bits.d};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = expf(pv[e] / T - jb.mp) * inv_lp;
        float wv = p;
        if (resid) wv = fmaxf(p - expf(qv[e] / T - jb.mq) * inv_lq, 0.f);
        const float E = -logf(race_u(bv[e]));
        race_take(best, bi, wv / E, v + e);
      }
    }
  } else {
    for (int v = lo + threadIdx.x; v < hi; v += kRaceThreads) {
      const U4 bits = race_bits(a.seed, i, jb.pos, v >> 2);
      const uint32_t bw = (v & 3) == 0 ? bits.a : (v & 3) == 1 ? bits.b : (v & 3) == 2 ? bits.c : bits.d;
      const float p = expf(lp[v] / T - jb.mp) * inv_lp;
      float wv = p;
      if (resid) wv = fmaxf(p - expf(lq[v] / T - jb.mq) * inv_lq, 0.f);
      const float E = -logf(race_u(bw));
      race_take(best, bi, wv / E, v);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    race_take(best, bi, b2, i2);
  }
  __shared__ float s_b[kRaceThreads / 32];
  __shared__ int s_i[kRaceThreads / 32];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  if (lane == 0) { s_b[wid] = best; s_i[wid] = bi; }
  __syncthreads();
  RacePart* parts = reinterpret_cast<RacePart*>(a.ws + a.L.race) + (size_t)i * nch;
  int* ticket = reinterpret_cast<int*>(a.ws + a.L.tickets) + i;
  if (threadIdx.x == 0) {
    for (int k = 1; k < kRaceThreads / 32; ++k) race_take(best, bi, s_b[k], s_i[k]);
    parts[c].key = best;
    parts[c].idx = bi;
    __threadfence();
    s_last = atomicAdd(ticket, 1) == nch - 1;
  }
  __syncthreads();
  if (!s_last) return;
  // last CTA of request i: reduce the chunk winners
  if (threadIdx.x < 32) {
    float b = -1.f;
    int x = 0x7fffffff;
    for (int k = lane; k < nch; k += 32) race_take(b, x, __ldcg(&parts[k].key), __ldcg(&parts[k].idx));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float b2 = __shfl_xor_sync(0xffffffffu, b, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, x, o);
      race_take(b, x, b2, i2);
    }
    if (lane == 0) {
      a.next_token[i] = x;
      *ticket = 0;
    }
  }
}

}  // namespace acc
}  // namespace sv

using namespace sv;

extern "C" size_t sv_accept_workspace(const sv_batch* bt, int32_t vocab) {
  if (!bt || bt->n_req < 0 || bt->total_rows < 0 || vocab < 1) return 0;
  return acc::layout(bt->n_req, bt->total_rows, vocab).total;
}

extern "C" sv_status sv_accept(const sv_batch* bt, const float* target_logits,
                               const float* draft_logits, int32_t vocab, float temperature,
                               uint64_t seed, int32_t* accepted_len, int32_t* accepted_nodes,
                               int32_t* next_token, uint8_t* ambiguous, int32_t* done,
                               float* row_stats, void* ws, size_t ws_bytes, int32_t* dev_status,
                               void* stream) {
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
  acc::Args a;
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
  a.L = acc::layout(bt->n_req, bt->total_rows, vocab);
  a.dev_status = dev_status;
  if (ws_bytes < a.L.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  const bool vec = (vocab % 4 == 0) && ((((uintptr_t)target_logits) |
                                         ((uintptr_t)(draft_logits ? draft_logits : target_logits))) & 15) == 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 gs((unsigned)((long)bt->total_rows * a.L.nch), temperature > 0.f ? 2 : 1);
  if (vec) acc::stats_kernel<true><<<gs, acc::kStatThreads, 0, s>>>(a);
  else acc::stats_kernel<false><<<gs, acc::kStatThreads, 0, s>>>(a);
  SV_LAUNCH_CHECK();
  acc::decide_kernel<<<(bt->n_req + acc::kDecideWarps - 1) / acc::kDecideWarps,
                       acc::kDecideWarps * 32, 0, s>>>(a);
  SV_LAUNCH_CHECK();
  if (temperature > 0.f) {
    const unsigned gr = (unsigned)((long)bt->n_req * a.L.nch_r);
    if (vec) acc::race_kernel<true><<<gr, acc::kRaceThreads, 0, s>>>(a);
    else acc::race_kernel<false><<<gr, acc::kRaceThreads, 0, s>>>(a);
    SV_LAUNCH_CHECK();
  }
  return SV_OK;
}

// ------------------------------------------------ no-allocation variant ----
// sv_accept_static: sv_accept without a caller workspace.  Its scratch is the
// file-scope device array below, which every GPU that loads the library keeps
// until the process exits.  The address of that array on the current device
// is looked up once per device (cudaGetSymbolAddress) on the first call made
// with that device current; make that first call before any stream capture.
// All calls share the array: two calls whose work overlaps on the GPU (for
// example on two streams) race on it.  Nothing in it has to start at zero:
// the accept kernels write every scratch word before they read it (the
// decide kernel clears each request's sampling job and ticket itself).

#include <mutex>

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
