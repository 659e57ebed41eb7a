// attend.cu — sv_tree_attend: padding-free verification attention of draft
// chains / trees against a paged bf16 GQA KV cache.
//
// Sources: [SwiftSpec] core design, mechanism 2 (every tree node has its own
// KV prefix) and mechanism 3 (one padding-free attention call verifies all
// draft tokens of a request); [FASER] operations notes (the attention kernel
// must accept a chunk of the rows); [SSD] section details (PagedAttention).
//
// Launches, on one stream:
//   plan   (1 CTA, one thread per request; one warp for one-pass calls of
//                    at most four requests) validates parents / windows /
//                    lengths and builds length-weighted split-KV work lists:
//                    the keys of each (request, KV head, query tile) are cut
//                    into splits of P pages so that about kUnitsPerSM units
//                    per SM exist (P at least 32 pages, 64 when the work still
//                    fills every SM; small batches aim for one wave and go
//                    down to 8 pages); every unit gets a self-contained 48-byte
//                    work item; clears the per-group merge tickets.  Requests
//                    with at least 128 virtual rows per KV head go to the
//                    tcgen05 list, the others to the mma.sync list.  An empty
//                    call (no keys anywhere) only publishes zero counts.
//   attend_tc (the tcgen05 list, when a request can reach 128 virtual rows;
//                    described with its kernel below).
//   attend (mma.sync list; 1 CTA per unit, 4 warps, 2 CTAs per SM)
//                    the query rows of the whole GQA group (row x head packed
//                    as "virtual rows") share every KV page.  Pages stream
//                    through a 3-stage ring of 64-token stages: lane 0 of
//                    warp p issues page p of each stage as 2-D tiled TMA loads
//                    (cp.async.bulk.tensor, 128-byte swizzle, one 64-element x
//                    16-row box per half page) that complete on an mbarrier
//                    per slot (thread 0 arms it with the stage's bytes); the
//                    warps wait on it with a bounded spin, and one block
//                    barrier per stage frees the slot.  A warp owns a 16-row
//                    m-tile and a slice of each stage's tokens: with one m-tile
//                    the four warps take 16 tokens each, with two they take
//                    32, with three or four every warp sees the whole stage.
//                    QK^T and PV run on mma.sync m16n8k16 bf16 -> fp32 with an
//                    online softmax in the log2 domain; the ancestor mask
//                    (built per CTA from the parent links held in shared
//                    memory) is applied only where staged draft slots lie.
//                    Warps that shared an m-tile merge through shared memory.
//                    A unit that covers all keys of its rows writes bf16
//                    output directly; otherwise it writes (m, l, O) partials
//                    and the last CTA of the group (atomic ticket) merges all
//                    splits -- or, in small batches, the merge launch does.
//                    One-pass calls of at most four requests with no window
//                    on the tcgen05 list, whose split groups all fit on the
//                    GPU at once as 16-CTA clusters, launch the same kernel as
//                    thread-block clusters (attend_kernel<D, true>): each
//                    group's 16 splits are one cluster, and its CTAs merge
//                    their partials over distributed shared memory.
//   merge (when the tcgen05 kernel ran or the batch is small and not
//                    clustered) the units of each split group merge its
//                    partials together.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "sv_attend_internal.h"
#include "sv_internal.cuh"
#include "sv_tcgen05.cuh"

namespace sv {
namespace attn {

constexpr int kTB = 64;          // tokens per pipeline stage (four pages)
constexpr int kStages = 3;       // TMA ring depth
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileRows = 64;    // virtual rows per unit
// About this many units per SM are aimed for (two resident CTAs, four waves).
constexpr int kUnitsPerSM = 8;
// Splits never go below kMinPagesPerSplit pages (each unit pays a start-up
// of a few microseconds and a merge share), nor below twice that when the
// work still gives every SM such a unit.
constexpr int kMinPagesPerSplit = 32;
// Calls with at most this many requests are latency-bound: splits go down to
// kSmallPagesPerSplit pages and a separate kernel merges them, every unit of
// a split group taking a slice of its rows (in-kernel, the group's last CTA
// would merge every split alone) -- unless the split groups run as clusters
// (one-pass calls, below).
constexpr int kSmallBatch = 4;
constexpr int kSmallPagesPerSplit = 8;
// One-pass calls of at most kSmallBatch requests run the splits of each
// (row tile, KV head) group of the mma.sync list as one thread-block cluster
// of kClusterSplits CTAs (on one GPC, two CTAs per SM fit), which merge their
// partials through distributed shared memory at the end: no partials in
// global memory and no merge launch (a one-request 4096-token chain step:
// 53.3 -> 49.8 us, measured).
constexpr int kClusterSplits = 16;
constexpr int kMaxPagesPerSplit = 1024;  // block ids of a unit staged in shared memory

struct ReqInfo {
  int ubase, nsplit, nrt, b, e, ctx, nblk, valid;
  int act;     // chunk mode: the window is not empty (the accept list)
  int cu, rows;
  int tc;      // units of 128 virtual rows on the tcgen05 kernel
};

// Requests whose window holds at least this many virtual rows (query rows x
// GQA group) per KV head form dense 128-row tiles: they run on the tcgen05
// kernel (tensor memory accumulators), the others on the mma.sync kernel.
constexpr int kTcRows = 128;       // virtual rows per tcgen05 unit (one M = 128 tile)
constexpr int kTcMinRows = 128;
constexpr int kTcMinPages = 16;    // pages per split at least (four stages)
constexpr int kTcMaxPages = 256;   // pages per split at most (block ids in shared memory)
// The planner keeps the per-request records in shared memory up to this many
// requests (about 45 KB), in its workspace beyond.
constexpr int kPlanSmemRequests = 1024;

// One unit of the work list: everything its CTA needs to start (a single
// 48-byte load, issued together with the header's unit count).
struct __align__(16) WorkItem {
  int i;       // request
  int local;   // unit within the request: (row tile * Hkv + KV head) * nsplit + split
  int nsplit, nblk, ctx, b, e;
  int ubase;   // the request's first unit
  int cu;      // the request's first packed row
  int rows;    // the request's packed rows
  int P;       // pages per split
  int pad;
};

struct Header {
  int U;     // units in the work list (mma.sync kernel)
  int P;     // pages per split
  int Utc;   // units in the tcgen05 work list
  int Ptc;   // pages per split there
  int pad[60];
};

struct Layout {
  size_t header, info, work, tickets, ml, o;
  size_t work_tc, ml_tc, o_tc, total;
  int ucap, ucap_tc;
  int ucap_cl;      // units of a small one-pass call whose split groups are clusters
  int nsm;          // SMs of the device the call runs on
  int unit_target;  // units the planner aims for: kUnitsPerSM per SM
  int small;        // at most kSmallBatch requests: small splits, merge kernel
};

// Units are at most W / P + Hkv * (row tiles): P >= W / unit_target unless it
// is capped at kMaxPagesPerSplit, and W <= Hkv * (row tiles) * max_blocks.
inline int unit_cap(int R, int total_rows, int group, int Hkv, int max_blocks, int unit_target) {
  long nrt = (long)group * total_rows / kTileRows + R + 1;
  long rt_units = (long)Hkv * nrt;
  return (int)(rt_units + unit_target + (rt_units * max_blocks + kMaxPagesPerSplit - 1) / kMaxPagesPerSplit);
}

// tcgen05 units: the planner picks Ptc >= W_tc / (2 SMs - row-tile units),
// so they number at most two per SM unless Ptc is capped at kTcMaxPages.
inline int unit_cap_tc(int R, int total_rows, int group, int Hkv, int D, int max_rows,
                       int max_blocks, int nsm) {
  if (D != 128 || group * max_rows < kTcMinRows) return 0;
  const long rt = (long)Hkv * ((long)group * total_rows / kTcRows + R + 1);
  return (int)(2L * nsm + rt + (rt * max_blocks + kTcMaxPages - 1) / kTcMaxPages);
}

inline Layout layout(int R, int total_rows, int group, int Hkv, int D, int max_blocks,
                     int max_rows) {
  Layout L;
  size_t off = 0;
  L.nsm = sizing_sms();
  L.small = R <= kSmallBatch ? 1 : 0;
  // small batches aim for one wave (two units per SM), the rest for four
  L.unit_target = L.nsm * (L.small ? 2 : kUnitsPerSM);
  L.ucap = unit_cap(R, total_rows, group, Hkv, max_blocks, L.unit_target);
  L.ucap_tc = unit_cap_tc(R, total_rows, group, Hkv, D, max_rows, max_blocks, L.nsm);
  L.ucap_cl = 0;
  if (L.small) {
    // kClusterSplits units per (row tile, KV head): at most
    // floor(group * total_rows / 64) + R row tiles (clusters only when no
    // window can reach the tcgen05 list; the work list holds either plan)
    const long tiles = (long)group * total_rows / kTileRows + R;
    L.ucap_cl = L.ucap_tc > 0 ? 0 : (int)((long)Hkv * tiles * kClusterSplits);
    L.ucap = std::max(L.ucap, L.ucap_cl);
  }
  L.header = off; off += align256(sizeof(Header));
  L.info = off; off += align256(sizeof(ReqInfo) * (size_t)R);
  L.work = off; off += align256(sizeof(WorkItem) * (size_t)L.ucap);
  L.tickets = off; off += align256(sizeof(int) * (size_t)L.ucap);
  L.ml = off; off += align256((size_t)L.ucap * kTileRows * 2 * sizeof(float));
  L.o = off; off += align256((size_t)L.ucap * kTileRows * (size_t)D * sizeof(float));
  L.work_tc = off; off += align256(sizeof(WorkItem) * (size_t)L.ucap_tc);
  L.ml_tc = off; off += align256((size_t)L.ucap_tc * kTcRows * 2 * sizeof(float));
  L.o_tc = off; off += align256((size_t)L.ucap_tc * kTcRows * (size_t)D * sizeof(float));
  L.total = off;
  return L;
}

struct Args {
  sv_batch bt;
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int num_blocks, Hkv, max_blocks;
  const int32_t* tables;
  const int32_t* cache_lens;
  const __nv_bfloat16* q;
  __nv_bfloat16* out;
  int Hq, group;
  float scale_log2;
  uint8_t* ws;
  Layout L;
  int32_t* dev_status;
  ChunkPlan chunk;  // chunk.index < 0: windows come from the batch
  int cl;           // > 0: each split group of the mma.sync list is a cluster of cl CTAs
};

// ------------------------------------------------------------------ plan --

__device__ __forceinline__ void block_excl_scan(int* s_warp, int v, int& excl, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;  // inclusive per warp
  }
  __syncthreads();
  int warp_off = warp ? s_warp[warp - 1] : 0;
  excl = warp_off + x - v;
  total = s_warp[(blockDim.x >> 5) - 1];
  __syncthreads();
}

__global__ void __launch_bounds__(1024) plan_kernel(Args a) {
  griddep_entry();
  const int R = a.bt.n_req;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Header* hdr = reinterpret_cast<Header*>(a.ws + a.L.header);
  extern __shared__ ReqInfo s_info[];
  ReqInfo* info = R <= kPlanSmemRequests ? s_info : reinterpret_cast<ReqInfo*>(a.ws + a.L.info);
  int* tickets = reinterpret_cast<int*>(a.ws + a.L.tickets);
  __shared__ unsigned long long s_W, s_Wtc;
  __shared__ int s_warp[32];
  __shared__ int s_carry, s_acarry, s_carry_tc, s_Rtc;

  __shared__ int s_none;
  const bool chunked = a.chunk.index >= 0;
  // One thread per request: its window (and in a chunked step its done flag)
  // and its cache length are loaded before the header check below, so both
  // round trips overlap.
  auto window_at = [&](int i, bool& badw) {
    badw = false;
    return chunked ? chunk_window(a.bt, i, a.chunk.index, a.chunk.size, a.chunk.done, &badw)
                   : window_of(a.bt, i);
  };
  bool badw0 = false;
  Window w0{};
  int ctx0 = 0;
  if (tid < R) {
    w0 = window_at(tid, badw0);
    ctx0 = a.cache_lens[tid];
  }
  if (tid == 0) {
    // Each request's rows are checked against the packed total by its window;
    // a prefix that does not start at 0 or end at the total is reported too.
    if (a.bt.cu_rows[0] != 0 || a.bt.cu_rows[R] != a.bt.total_rows)
      flag(a.dev_status, SV_DEV_BAD_WINDOW);
    s_W = 0ull;
    s_Wtc = 0ull;
    s_carry = 0;
    s_acarry = 0;
    s_carry_tc = 0;
    s_Rtc = 0;
    // A chunk after one that listed no request is empty too (requests only
    // ever stop): nothing to plan.
    s_none = (a.chunk.index > 0 && a.chunk.act[R] == 0) ? 1 : 0;
    if (s_none) {
      hdr->U = 0;
      hdr->Utc = 0;
    }
  }
  __syncthreads();
  if (s_none) return;
  // Per request: window, parents (all loads of a thread issued together),
  // length, work.
  unsigned long long myW = 0, myWtc = 0;
  int myRtc = 0;
  for (int i = tid; i < R; i += blockDim.x) {
    bool badw = badw0;
    Window w = w0;
    int ctx = ctx0;
    if (i != tid) {
      w = window_at(i, badw);
      ctx = a.cache_lens[i];
    }
    if (chunked) {
      a.chunk.row_begin[i] = w.b;
      a.chunk.row_end[i] = w.e;
      if (badw && a.chunk.index == 0) flag(a.dev_status, SV_DEV_BAD_WINDOW);
    }
    if (badw) w.ok = false;  // reported above (once); the window is empty anyway
    const int cu = a.bt.cu_rows[i];
    bool badp = false;
    // parents are checked once per call: a later chunk of a chunked step runs
    // only requests the first chunk found valid (one with bad parents stops
    // there)
    if (w.ok && !(chunked && a.chunk.index > 0)) {
      for (int j0 = 0; j0 < w.rows; j0 += 8) {  // eight loads in flight, then the checks
        int pp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pp[k] = j0 + k < w.rows ? a.bt.parent[cu + j0 + k] : 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int j = j0 + k;
          if (j < w.rows) badp |= (j == 0) ? (pp[k] != -1) : (pp[k] < 0 || pp[k] >= j);
        }
      }
    }
    bool valid = w.ok && !badp;
    if (!w.ok && !chunked) flag(a.dev_status, SV_DEV_BAD_WINDOW);
    if (badp) flag(a.dev_status, SV_DEV_BAD_PARENT);
    // A request that stopped in an earlier chunk may have been committed
    // already (its cache length moved on): nothing of it is read now.
    const bool stopped = chunked && a.chunk.index > 0 && w.b >= w.e;
    if (valid && !stopped && (ctx < 0 || (long)ctx + w.rows > (long)a.max_blocks * kBlockSize)) {
      valid = false;
      flag(a.dev_status, SV_DEV_BAD_LENGTH);
    }
    const int nw = valid ? max(0, w.e - w.b) : 0;
    const bool tc = a.L.ucap_tc > 0 && a.group * nw >= kTcMinRows;
    const int nrt = tc ? (a.group * nw + kTcRows - 1) / kTcRows
                       : (a.group * nw + kTileRows - 1) / kTileRows;
    const int nblk = nw ? (ctx + w.e + kBlockSize - 1) / kBlockSize : 0;
    if (tc) {
      myWtc += (unsigned long long)nrt * a.Hkv * nblk;
      myRtc += nrt * a.Hkv;
    } else {
      myW += (unsigned long long)nrt * a.Hkv * nblk;
    }
    ReqInfo ri;
    ri.valid = valid && nw > 0;
    ri.b = w.b;
    ri.e = w.e;
    ri.ctx = ctx;
    ri.nrt = nrt;
    ri.nblk = nblk;
    ri.nsplit = 0;
    ri.ubase = 0;
    // listed: 1 + the window's rows with a tested child (draft rows)
    ri.act = (!badw && w.b < w.e) ? 1 + max(0, min(w.e, w.lim - 1) - w.b) : 0;
    ri.cu = cu;
    ri.rows = w.rows;
    ri.tc = tc ? 1 : 0;
    info[i] = ri;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    myW += __shfl_xor_sync(0xffffffffu, myW, o);
    myWtc += __shfl_xor_sync(0xffffffffu, myWtc, o);
    myRtc += __shfl_xor_sync(0xffffffffu, myRtc, o);
  }
  if (lane == 0 && myW) atomicAdd(&s_W, myW);
  if (lane == 0 && myWtc) {
    atomicAdd(&s_Wtc, myWtc);
    atomicAdd(&s_Rtc, myRtc);
  }
  __syncthreads();
  const unsigned long long W = s_W;
  // tcgen05 units: about two per SM (two resident CTAs): splits of
  // W_tc / (2 SMs - row-tile units) pages, within [kTcMinPages, kTcMaxPages].
  int Ptc = 0;
  if (s_Wtc) {
    const long avail = max(1L, 2L * a.L.nsm - s_Rtc);
    Ptc = (int)min((unsigned long long)kTcMaxPages, (s_Wtc + avail - 1) / avail);
    Ptc = max(Ptc, kTcMinPages);
  }
  const unsigned long long target = (unsigned long long)a.L.unit_target;
  int P = (int)min((unsigned long long)kMaxPagesPerSplit, (W + target - 1) / target);
  const int Pmin = a.L.small ? kSmallPagesPerSplit
                 : W >= (unsigned long long)a.L.nsm * 2 * kMinPagesPerSplit ? 2 * kMinPagesPerSplit
                                                                         : kMinPagesPerSplit;
  if (P < Pmin) P = Pmin;
  // Work list offsets (exclusive scan of units per request); in chunk mode
  // also the accept's list of requests with a non-empty window, in request
  // order, with its count at act[R].
  for (int base = 0; base < R; base += blockDim.x) {
    const int i = base + tid;
    int units = 0, units_tc = 0, act = 0;
    if (i < R) {
      const ReqInfo ri = info[i];
      const int Pi = ri.tc ? Ptc : P;
      const int nsplit = ri.valid ? (ri.nblk + Pi - 1) / Pi : 0;
      (ri.tc ? units_tc : units) = ri.nrt * a.Hkv * nsplit;
      act = ri.act != 0;
      info[i].nsplit = nsplit;
    }
    int excl, total, excl_tc = 0, total_tc = 0;
    block_excl_scan(s_warp, units, excl, total);
    if (a.L.ucap_tc > 0) block_excl_scan(s_warp, units_tc, excl_tc, total_tc);
    if (i < R) info[i].ubase = info[i].tc ? s_carry_tc + excl_tc : s_carry + excl;
    if (chunked) {
      int aexcl, atotal;
      block_excl_scan(s_warp, act, aexcl, atotal);
      if (act) {
        const ReqInfo ri = info[i];
        a.chunk.act[s_acarry + aexcl] = i;
        a.chunk.act4[s_acarry + aexcl] = make_int4(i, ri.cu + ri.b, ri.e - ri.b, ri.act - 1);
      }
      __syncthreads();
      if (tid == 0) s_acarry += atotal;
    }
    __syncthreads();
    if (tid == 0) {
      s_carry += total;
      s_carry_tc += total_tc;
    }
    __syncthreads();
  }
  if (chunked && tid == 0) a.chunk.act[R] = s_acarry;
  int U = s_carry, Utc = s_carry_tc;
  if (U > a.L.ucap || Utc > a.L.ucap_tc) {  // cannot happen with the workspace's bounds
    U = Utc = 0;
    if (tid == 0) flag(a.dev_status, SV_DEV_BAD_LENGTH);
  }
  for (int u = tid; u < U; u += blockDim.x) tickets[u] = 0;
  WorkItem* work = reinterpret_cast<WorkItem*>(a.ws + a.L.work);
  WorkItem* work_tc = reinterpret_cast<WorkItem*>(a.ws + a.L.work_tc);
  if (U > 0 || Utc > 0)
    for (int i = warp; i < R; i += (int)(blockDim.x >> 5)) {
      const ReqInfo ri = info[i];
      const int n = ri.nrt * a.Hkv * ri.nsplit;
      if (n == 0 || (ri.tc ? Utc : U) == 0) continue;
      WorkItem* list = ri.tc ? work_tc : work;
      const int Pi = ri.tc ? Ptc : P;
      const int cu = ri.cu;
      const int rows = ri.rows;
      for (int x = lane; x < n; x += 32) {
        WorkItem it;
        it.i = i;
        it.local = x;
        it.nsplit = ri.nsplit;
        it.nblk = ri.nblk;
        it.ctx = ri.ctx;
        it.b = ri.b;
        it.e = ri.e;
        it.ubase = ri.ubase;
        it.cu = cu;
        it.rows = rows;
        it.P = Pi;
        it.pad = 0;
        list[ri.ubase + x] = it;
      }
    }
  if (tid == 0) {
    hdr->U = U;
    hdr->P = P;
    hdr->Utc = Utc;
    hdr->Ptc = Ptc;
  }
}

// ------------------------------------------------------------ small plan --
// One-pass calls with at most kSmallBatch requests are planned by a single
// warp (the rules of plan_kernel, without its block-wide scans and barriers):
// lane r loads request r's window and cache length while lane 0 checks the
// packed total, then the warp checks every request's parents with all loads
// in flight, and shuffles give the work, the split sizes and the list
// offsets.  Two dependent round trips in all.
struct SmallPlan {
  int U, P, Utc, Ptc;
  int ubase[kSmallBatch], nsplit[kSmallBatch], nrt[kSmallBatch], tc[kSmallBatch];
  int b[kSmallBatch], e[kSmallBatch], ctx[kSmallBatch], nblk[kSmallBatch];
  int cu[kSmallBatch], rows[kSmallBatch], Pr[kSmallBatch];
};

__device__ __forceinline__ void small_plan_warp(const Args& a, SmallPlan& sp, bool report) {
  const unsigned kAll = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int R = a.bt.n_req;  // 1 .. kSmallBatch
  Window w{};
  int ctx = 0;
  if (lane < R) {
    w = window_of(a.bt, lane);
    ctx = a.cache_lens[lane];
  }
  if (report && lane == 0 && (a.bt.cu_rows[0] != 0 || a.bt.cu_rows[R] != a.bt.total_rows))
    flag(a.dev_status, SV_DEV_BAD_WINDOW);
  // parents of every request with a valid window, all loads in flight at once
  // (a valid window has at most kMaxRows = 128 rows: four per lane)
  int pv[kSmallBatch][4];
  int wrows[kSmallBatch];
  bool wok[kSmallBatch];
#pragma unroll
  for (int r = 0; r < kSmallBatch; ++r) {
    wrows[r] = __shfl_sync(kAll, w.rows, r);
    const int okr = __shfl_sync(kAll, (int)w.ok, r);
    wok[r] = r < R && okr != 0;
    const int cu = __shfl_sync(kAll, w.cu, r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = lane + 32 * k;
      pv[r][k] = (wok[r] && j < wrows[r]) ? a.bt.parent[cu + j] : 0;
    }
  }
  int badp_mask = 0;
#pragma unroll
  for (int r = 0; r < kSmallBatch; ++r) {
    bool bad = false;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int j = lane + 32 * k;
      if (wok[r] && j < wrows[r]) bad |= (j == 0) ? (pv[r][k] != -1) : (pv[r][k] < 0 || pv[r][k] >= j);
    }
    if (__any_sync(kAll, bad)) badp_mask |= 1 << r;
  }
  // lane r: request r's rule checks, row tiles and pages
  bool valid = false, tc = false;
  int nrt = 0, nblk = 0;
  if (lane < R) {
    const bool badp = (badp_mask >> lane) & 1;
    bool v = w.ok && !badp;
    if (report && !w.ok) flag(a.dev_status, SV_DEV_BAD_WINDOW);
    if (report && badp) flag(a.dev_status, SV_DEV_BAD_PARENT);
    if (v && (ctx < 0 || (long)ctx + w.rows > (long)a.max_blocks * kBlockSize)) {
      v = false;
      if (report) flag(a.dev_status, SV_DEV_BAD_LENGTH);
    }
    const int nw = v ? max(0, w.e - w.b) : 0;
    tc = a.L.ucap_tc > 0 && a.group * nw >= kTcMinRows;
    nrt = tc ? (a.group * nw + kTcRows - 1) / kTcRows : (a.group * nw + kTileRows - 1) / kTileRows;
    nblk = nw ? (ctx + w.e + kBlockSize - 1) / kBlockSize : 0;
    valid = v && nw > 0;
  }
  unsigned long long W = (!tc) ? (unsigned long long)nrt * a.Hkv * nblk : 0ull;
  unsigned long long Wtc = tc ? (unsigned long long)nrt * a.Hkv * nblk : 0ull;
  int Rtc = tc ? nrt * a.Hkv : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    W += __shfl_xor_sync(kAll, W, o);
    Wtc += __shfl_xor_sync(kAll, Wtc, o);
    Rtc += __shfl_xor_sync(kAll, Rtc, o);
  }
  int Ptc = 0;
  if (Wtc) {
    const long avail = max(1L, 2L * a.L.nsm - Rtc);
    Ptc = (int)min((unsigned long long)kTcMaxPages, (Wtc + avail - 1) / avail);
    Ptc = max(Ptc, kTcMinPages);
  }
  const unsigned long long target = (unsigned long long)a.L.unit_target;
  int P = (int)min((unsigned long long)kMaxPagesPerSplit, (W + target - 1) / target);
  if (P < kSmallPagesPerSplit) P = kSmallPagesPerSplit;
  // clusters: exactly cl splits of ceil(nblk / cl) pages (the last ones may
  // hold no page)
  const bool clu = a.cl > 0 && !tc;
  const int Pi = tc ? Ptc : clu ? max(1, (nblk + a.cl - 1) / a.cl) : P;
  const int nsplit = valid ? (clu ? a.cl : (nblk + Pi - 1) / Pi) : 0;
  const int units = nrt * a.Hkv * nsplit;
  // exclusive prefix of the units within each list (lanes 0 .. R-1)
  int x = tc ? 0 : units, xt = tc ? units : 0;
#pragma unroll
  for (int o = 1; o < kSmallBatch; o <<= 1) {
    const int y = __shfl_up_sync(kAll, x, o), yt = __shfl_up_sync(kAll, xt, o);
    if (lane >= o) { x += y; xt += yt; }
  }
  int U = __shfl_sync(kAll, x, R - 1), Utc = __shfl_sync(kAll, xt, R - 1);
  if (U > (a.cl > 0 ? a.L.ucap_cl : a.L.ucap) || Utc > a.L.ucap_tc) {  // cannot happen with the workspace's bounds
    U = Utc = 0;
    if (report && lane == 0) flag(a.dev_status, SV_DEV_BAD_LENGTH);
  }
  if (lane < R) {
    sp.ubase[lane] = tc ? xt - units : x - units;
    sp.nsplit[lane] = nsplit;
    sp.nrt[lane] = nrt;
    sp.tc[lane] = tc ? 1 : 0;
    sp.b[lane] = w.b;
    sp.e[lane] = w.e;
    sp.ctx[lane] = ctx;
    sp.nblk[lane] = nblk;
    sp.cu[lane] = w.cu;
    sp.rows[lane] = w.rows;
    sp.Pr[lane] = Pi;
  }
  if (lane == 0) {
    sp.U = U;
    sp.P = P;
    sp.Utc = Utc;
    sp.Ptc = Ptc;
  }
}

__global__ void __launch_bounds__(32) plan_small_kernel(Args a) {
  griddep_entry();
  __shared__ SmallPlan sp;
  small_plan_warp(a, sp, true);
  __syncwarp();
  const int lane = threadIdx.x;
  Header* hdr = reinterpret_cast<Header*>(a.ws + a.L.header);
  WorkItem* work = reinterpret_cast<WorkItem*>(a.ws + a.L.work);
  WorkItem* work_tc = reinterpret_cast<WorkItem*>(a.ws + a.L.work_tc);
  for (int r = 0; r < a.bt.n_req; ++r) {
    const int n = sp.nrt[r] * a.Hkv * sp.nsplit[r];
    if (n == 0 || (sp.tc[r] ? sp.Utc : sp.U) == 0) continue;
    WorkItem* list = sp.tc[r] ? work_tc : work;
    for (int x = lane; x < n; x += 32) {
      WorkItem it;
      it.i = r;
      it.local = x;
      it.nsplit = sp.nsplit[r];
      it.nblk = sp.nblk[r];
      it.ctx = sp.ctx[r];
      it.b = sp.b[r];
      it.e = sp.e[r];
      it.ubase = sp.ubase[r];
      it.cu = sp.cu[r];
      it.rows = sp.rows[r];
      it.P = sp.Pr[r];
      it.pad = 0;
      list[sp.ubase[r] + x] = it;
    }
  }
  if (lane == 0) {
    hdr->U = sp.U;
    hdr->P = sp.P;
    hdr->Utc = sp.Utc;
    hdr->Ptc = sp.Ptc;
  }
}

// ---------------------------------------------------------------- attend --

// The last CTA of a (request, row tile, KV head) group merges the (m, l, O)
// partials of all the group's splits -- m in the log2 domain, O unnormalised
// -- in one online pass per (virtual row, 4 columns) and writes bf16 rows.
// ml_all / op_all: partials of TILE rows per unit; gidx: the group's split-0
// unit; row0: packed row of the window's first row; kLoads: the splits' loads
// a lane issues before merging any.
template <int D, int TILE, int kLoads = 8>
__device__ __forceinline__ void merge_splits(const Args& a, const float* ml_all,
                                             const float* op_all, int gidx, int nsplit, int r0,
                                             int r1, int vr0, int row0, int g, int tid,
                                             int nthreads) {
  constexpr int kQuads = D / 4;
  const int group = a.group;
  // SL adjacent lanes share one output quad, lane s of them merging splits
  // s, s + SL, ...: with SL * kLoads >= nsplit every split of the quad is in
  // flight at once; the SL partial states then merge by shuffles.  The trip
  // count is the same for every thread (nthreads is a multiple of 32 and
  // every thread of the block calls this), so whole warps shuffle.
  int SL = 1;
  while (SL < 32 && SL * kLoads < nsplit) SL <<= 1;
  const int items = (r1 - r0) * kQuads * SL;
  for (int x0 = 0; x0 < items; x0 += nthreads) {
    const int x = x0 + tid;
    const bool live = x < items;
    const int sl = x % SL, q = x / SL;
    const int vr = r0 + q / kQuads, c4 = q % kQuads;
    // one online pass (running max, rescaled sums) over this lane's splits
    float Mx = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) {
      for (int sp0 = sl; sp0 < nsplit; sp0 += kLoads * SL) {
        float2 ml2[kLoads];
        float4 o4[kLoads];
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
          const size_t row = (size_t)(gidx + min(sp0 + k * SL, nsplit - 1)) * TILE + vr;
          ml2[k] = __ldcg(reinterpret_cast<const float2*>(ml_all + row * 2));
          o4[k] = __ldcg(reinterpret_cast<const float4*>(op_all + row * D) + c4);
        }
#pragma unroll
        for (int k = 0; k < kLoads; ++k) {
          const float nm = fmaxf(Mx, ml2[k].x);
          if (sp0 + k * SL >= nsplit || nm == -INFINITY) continue;
          const float s_old = exp2f(Mx - nm), s_new = exp2f(ml2[k].x - nm);
          L = L * s_old + ml2[k].y * s_new;
          acc.x = acc.x * s_old + o4[k].x * s_new;
          acc.y = acc.y * s_old + o4[k].y * s_new;
          acc.z = acc.z * s_old + o4[k].z * s_new;
          acc.w = acc.w * s_old + o4[k].w * s_new;
          Mx = nm;
        }
      }
    }
    for (int o = SL >> 1; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, Mx, o);
      const float l2 = __shfl_xor_sync(0xffffffffu, L, o);
      float4 a2;
      a2.x = __shfl_xor_sync(0xffffffffu, acc.x, o);
      a2.y = __shfl_xor_sync(0xffffffffu, acc.y, o);
      a2.z = __shfl_xor_sync(0xffffffffu, acc.z, o);
      a2.w = __shfl_xor_sync(0xffffffffu, acc.w, o);
      const float nm = fmaxf(Mx, m2);
      if (nm != -INFINITY) {
        const float s_old = exp2f(Mx - nm), s_new = exp2f(m2 - nm);
        L = L * s_old + l2 * s_new;
        acc.x = acc.x * s_old + a2.x * s_new;
        acc.y = acc.y * s_old + a2.y * s_new;
        acc.z = acc.z * s_old + a2.z * s_new;
        acc.w = acc.w * s_old + a2.w * s_new;
        Mx = nm;
      }
    }
    if (!live || sl != 0) continue;
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int vgl = vr0 + vr;
    const int prow = row0 + vgl / group;
    const int head = g * group + vgl % group;
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + ((size_t)prow * a.Hq + head) * D + c4 * 4);
    dst[0] = pack_bf16(acc.x * inv, acc.y * inv);
    dst[1] = pack_bf16(acc.z * inv, acc.w * inv);
  }
}

// Shared-memory image of one stage: for K then V, 4 pages x (D / 64) boxes of
// 16 rows x 128 bytes, as TMA writes them with the 128-byte swizzle (16-byte
// chunk c of row r of a box stored at chunk c ^ (r % 8)).
template <int D>
struct StageLayout {
  static constexpr int kHalves = D / 64;                 // boxes per page
  static constexpr int kBoxBytes = 16 * 128;
  static constexpr int kTensorBytes = 4 * kHalves * kBoxBytes;  // 64 tokens
  static constexpr int kStageBytes = 2 * kTensorBytes;
  // byte offset of (token t of the stage, 16-byte chunk c of the head dim)
  __device__ static __forceinline__ uint32_t off(int t, int c) {
    const int r = t & 15;
    return (uint32_t)((((t >> 4) * kHalves + (c >> 3)) * kBoxBytes) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
  }
};

template <int D>
struct Frag {
  float o[D / 8][4];
  float m_a, m_b, l_a, l_b;
};

// NT * 8 tokens starting at stage row `s0` for this warp's two rows.
template <int D, int NT>
__device__ __forceinline__ void slice_compute(Frag<D>& f, const uint32_t (&qf)[D / 16][4],
                                              uint32_t kbase, uint32_t vbase, int tfirst, int s0,
                                              int ctx, int tok_end, float scale_log2,
                                              unsigned long long mk_a0, unsigned long long mk_a1,
                                              unsigned long long mk_b0, unsigned long long mk_b1,
                                              int lane) {
  using SL = StageLayout<D>;
  const int tq = lane & 3;
  float sc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ks += 2) {
      const int trow = s0 + nt * 8 + (lane & 7);
      const int chunk = 2 * ks + (lane >> 3);
      uint32_t r[4];
      ldsm_x4(r, kbase + SL::off(trow, chunk));
      mma16816(sc[nt], qf[ks], r[0], r[1]);
      mma16816(sc[nt], qf[ks + 1], r[2], r[3]);
    }
  }
  const int tbeg = tfirst + s0;
  const bool need_mask = (tbeg + NT * 8 > ctx) || (tbeg + NT * 8 > tok_end);
  float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = sc[nt][e] * scale_log2;
      if (need_mask) {
        const int tok = tbeg + nt * 8 + 2 * tq + (e & 1);
        bool ok = tok < tok_end;
        if (ok && tok >= ctx) {
          const int m = tok - ctx;
          const unsigned long long w0 = (e < 2) ? mk_a0 : mk_b0;
          const unsigned long long w1 = (e < 2) ? mk_a1 : mk_b1;
          ok = ((m < 64 ? (w0 >> m) : (w1 >> (m - 64))) & 1ull) != 0ull;
        }
        if (!ok) v = -INFINITY;
      }
      sc[nt][e] = v;
      if (e < 2) mx_a = fmaxf(mx_a, v); else mx_b = fmaxf(mx_b, v);
    }
  }
  mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
  mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
  mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
  mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
  const float nm_a = fmaxf(f.m_a, mx_a), nm_b = fmaxf(f.m_b, mx_b);
  const float base_a = nm_a == -INFINITY ? 0.f : nm_a;
  const float base_b = nm_b == -INFINITY ? 0.f : nm_b;
  const float al_a = ex2(f.m_a - base_a), al_b = ex2(f.m_b - base_b);
  f.m_a = nm_a;
  f.m_b = nm_b;
  float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    sc[nt][0] = ex2(sc[nt][0] - base_a);
    sc[nt][1] = ex2(sc[nt][1] - base_a);
    sc[nt][2] = ex2(sc[nt][2] - base_b);
    sc[nt][3] = ex2(sc[nt][3] - base_b);
    ps_a += sc[nt][0] + sc[nt][1];
    ps_b += sc[nt][2] + sc[nt][3];
  }
  f.l_a = f.l_a * al_a + ps_a;
  f.l_b = f.l_b * al_b + ps_b;
  // Once the running maxima settle, most slices leave every row's max in
  // the warp unchanged: the factor is then exactly 1 and O is left alone.
  if (__any_sync(0xffffffffu, al_a != 1.f || al_b != 1.f)) {
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      f.o[dn][0] *= al_a;
      f.o[dn][1] *= al_a;
      f.o[dn][2] *= al_b;
      f.o[dn][3] *= al_b;
    }
  }
#pragma unroll
  for (int kk = 0; kk < NT / 2; ++kk) {
    uint32_t pa[4];
    pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
    pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
    pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
    pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
    for (int dn = 0; dn < D / 8; dn += 2) {
      const int trow = s0 + 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
      const int chunk = dn + (lane >> 4);
      uint32_t r[4];
      ldsm_x4_t(r, vbase + SL::off(trow, chunk));
      mma16816(f.o[dn], pa, r[0], r[1]);
      mma16816(f.o[dn + 1], pa, r[2], r[3]);
    }
  }
}

// The kClusterSplits CTAs of a split group form one cluster: each leaves its
// (m, l, O) partial of the tile's rows in its own shared memory (the stage
// ring, idle by now) and, after a cluster barrier, CTA rank r merges rows
// r, r + kClusterSplits, ... reading every peer's partial of the row through
// distributed shared memory (all sixteen loads in flight), then writes bf16
// rows.  A second barrier keeps each CTA resident until its peers have read
// it.  Every thread of every CTA of the cluster calls this.
template <int D>
__device__ __forceinline__ void cluster_merge(const Args& a, const Frag<D>& f, bool owner,
                                              bool real_a, bool real_b, int vl_a, int vl_b, int tq,
                                              uint8_t* ring_ptr, int Mu, int vr0, int row0, int g) {
  constexpr int kStride = D + 4;  // floats per partial row (spreads the stores over banks)
  constexpr int kQuads = D / 4;
  static_assert(kTileRows * kStride * 4 + kTileRows * 8 <= kStages * StageLayout<D>::kStageBytes,
                "partials fit in the ring");
  float* po = reinterpret_cast<float*>(ring_ptr);
  float2* pml = reinterpret_cast<float2*>(ring_ptr + (size_t)kTileRows * kStride * sizeof(float));
  __syncthreads();  // the ring's exchange area has been read
  if (owner) {
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      if (real_a)
        *reinterpret_cast<float2*>(po + vl_a * kStride + dn * 8 + 2 * tq) = make_float2(f.o[dn][0], f.o[dn][1]);
      if (real_b)
        *reinterpret_cast<float2*>(po + vl_b * kStride + dn * 8 + 2 * tq) = make_float2(f.o[dn][2], f.o[dn][3]);
    }
    if (tq == 0) {
      if (real_a) pml[vl_a] = make_float2(f.m_a, f.l_a);
      if (real_b) pml[vl_b] = make_float2(f.m_b, f.l_b);
    }
  }
  cluster_sync();
  const int rank = (int)cluster_rank();
  const int nrow = rank < Mu ? (Mu - rank + kClusterSplits - 1) / kClusterSplits : 0;
  const uint32_t po_s = smem_u32(po), pml_s = smem_u32(pml);
  for (int x = threadIdx.x; x < nrow * kQuads; x += blockDim.x) {
    const int vr = rank + (x / kQuads) * kClusterSplits, c4 = x % kQuads;
    float2 ml[kClusterSplits];
    float4 o4[kClusterSplits];
#pragma unroll
    for (int q = 0; q < kClusterSplits; ++q) {
      ml[q] = dsmem_ld2(dsmem_addr(pml_s + (uint32_t)vr * 8u, (uint32_t)q));
      o4[q] = dsmem_ld4(dsmem_addr(po_s + (uint32_t)(vr * kStride + c4 * 4) * 4u, (uint32_t)q));
    }
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < kClusterSplits; ++q) mx = fmaxf(mx, ml[q].x);
    const float base = mx == -INFINITY ? 0.f : mx;  // m in the log2 domain
    float L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < kClusterSplits; ++q) {
      const float w = exp2f(ml[q].x - base);  // 0 for a split that saw no key of the row
      L += w * ml[q].y;
      acc.x += w * o4[q].x;
      acc.y += w * o4[q].y;
      acc.z += w * o4[q].z;
      acc.w += w * o4[q].w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int vgl = vr0 + vr;
    const int prow = row0 + vgl / a.group;
    const int head = g * a.group + vgl % a.group;
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.out + ((size_t)prow * a.Hq + head) * D + c4 * 4);
    dst[0] = pack_bf16(acc.x * inv, acc.y * inv);
    dst[1] = pack_bf16(acc.z * inv, acc.w * inv);
  }
  cluster_sync();
}

// CL: the launch groups each split group's kClusterSplits units into one
// thread-block cluster (small one-pass calls), which merges at the end.
template <int D, bool CL>
__global__ void __launch_bounds__(kThreads, 2)
    attend_kernel(Args a, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV) {
  griddep_entry();
  using SL = StageLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int s_par[kMaxRows];
  __shared__ int s_tbl[kMaxPagesPerSplit];
  __shared__ unsigned long long s_mask[kTileRows][2];
  __shared__ __align__(8) unsigned long long s_full[kStages];
  __shared__ int s_last;
  __shared__ int s_abort;
  const Header* hdr = reinterpret_cast<const Header*>(a.ws + a.L.header);
  const int u = blockIdx.x;
  // Both loads at once: the item of a CTA past the unit count is never used
  // (it lies inside the workspace: the grid is the workspace's unit bound).
  const int U = hdr->U;
  const WorkItem ri = reinterpret_cast<const WorkItem*>(a.ws + a.L.work)[u];
  // a cluster leaves as a whole (its CTAs meet at cluster barriers later);
  // U is a multiple of the cluster size, so this only drops idle clusters
  if (CL ? (u / kClusterSplits + 1) * kClusterSplits > U : u >= U) return;
  const int P = ri.P;
  const int i = ri.i;
  const int local = ri.local;
  const int s = local % ri.nsplit;
  const int rest = local / ri.nsplit;
  const int g = rest % a.Hkv;
  const int rt = rest / a.Hkv;
  const int group = a.group;
  const int M = group * (ri.e - ri.b);
  const int vr0 = rt * kTileRows;
  const int Mu = min(kTileRows, M - vr0);
  const int blk0 = s * P;
  // (a cluster's last splits may be empty)
  const int blk1 = CL ? max(blk0, min(blk0 + P, ri.nblk)) : min(blk0 + P, ri.nblk);
  const int ctx = ri.ctx;
  const int tok_end = min(ctx + ri.e, blk1 * kBlockSize);
  const int cu = ri.cu;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  // Warp roles: m-tile mt, token slice ts of TS per stage.
  const int MT = (Mu + 15) >> 4;
  const int TS = MT == 1 ? 4 : MT == 2 ? 2 : 1;
  const int mt = MT == 3 ? warp : warp % MT;
  const int ts = MT == 3 ? 0 : warp / MT;
  const bool active = mt < MT;

  const int n_stage = (blk1 - blk0 + 3) / 4;
  const int32_t* table = a.tables + (size_t)i * a.max_blocks;
  // 1024-byte aligned ring for the 128-byte swizzle atoms.
  const uint32_t ring = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* ring_ptr = smem_raw + (ring - smem_u32(smem_raw));

  // Block ids of this unit's pages (and the parent links, if the unit reaches
  // staged slots) into shared memory with one round trip.
  const int r_first = vr0 / group;
  const int r_count = (vr0 + Mu - 1) / group - r_first + 1;
  const bool unit_masked = blk1 * kBlockSize > ctx;
  for (int p = tid; p < blk1 - blk0; p += kThreads) s_tbl[p] = __ldg(table + blk0 + p);
  if (unit_masked)
    for (int j = tid; j < ri.rows; j += kThreads) s_par[j] = a.bt.parent[cu + j];
  if (tid == 0) {
    s_abort = 0;
    for (int k = 0; k < kStages; ++k) mbar_init(smem_u32(&s_full[k]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  // One stage: lane 0 of warp p issues page p's boxes (K and V); thread 0
  // also arms the slot's barrier with the stage's total bytes (the barrier's
  // transaction count may dip below zero until it does).
  static_assert(kWarps == 4, "one page of a stage per warp");
  auto issue = [&](int st) {
    if (lane != 0 || st >= n_stage) return;
    const int slot = st % kStages;
    const uint32_t bar = smem_u32(&s_full[slot]);
    const uint32_t kdst = ring + slot * SL::kStageBytes;
    auto bid_of = [&](int p) {
      const int page = blk0 + 4 * st + p;
      if (page >= blk1) return -1;
      const int bid = s_tbl[page - blk0];
      return (bid < 0 || bid >= a.num_blocks) ? -2 : bid;
    };
    if (warp == 0) {
      uint32_t bytes = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p)
        if (bid_of(p) >= 0) bytes += 2 * SL::kHalves * SL::kBoxBytes;
      mbar_arrive_expect_tx(bar, bytes);
    }
    const int bid = bid_of(warp);
    if (bid == -2) flag(a.dev_status, SV_DEV_BAD_BLOCK_ID);
    if (bid < 0) return;
    const int y = (bid * a.Hkv + g) * kBlockSize;
#pragma unroll
    for (int h = 0; h < SL::kHalves; ++h) {
      const uint32_t o = (uint32_t)((warp * SL::kHalves + h) * SL::kBoxBytes);
      tma_load_2d(kdst + o, &tmK, 64 * h, y, bar);
      tma_load_2d(kdst + SL::kTensorBytes + o, &tmV, 64 * h, y, bar);
    }
  };

#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) issue(st);

  // Ancestor-or-self masks of the unit's rows, only if it reaches staged slots.
  if (unit_masked) {
    for (int t = tid; t < r_count; t += kThreads) {
      unsigned long long lo = 0ull, hi = 0ull;
      int m = ri.b + r_first + t;
      for (int steps = 0; m >= 0 && steps <= kMaxRows; ++steps) {  // parents validated by plan
        if (m < 64) lo |= 1ull << m; else hi |= 1ull << (m - 64);
        m = s_par[m];
      }
      s_mask[t][0] = lo;
      s_mask[t][1] = hi;
    }
    __syncthreads();
  }

  // This thread's two virtual rows of m-tile mt.
  const int vl_a = mt * 16 + gq, vl_b = vl_a + 8;
  const bool real_a = active && vl_a < Mu, real_b = active && vl_b < Mu;
  const int va = vr0 + vl_a, vb = vr0 + vl_b;
  const int prow_a = cu + ri.b + (real_a ? va / group : 0);
  const int prow_b = cu + ri.b + (real_b ? vb / group : 0);
  const int head_a = g * group + va % group;
  const int head_b = g * group + vb % group;
  unsigned long long mk_a0 = 0, mk_a1 = 0, mk_b0 = 0, mk_b1 = 0;
  if (unit_masked) {
    if (real_a) { mk_a0 = s_mask[va / group - r_first][0]; mk_a1 = s_mask[va / group - r_first][1]; }
    if (real_b) { mk_b0 = s_mask[vb / group - r_first][0]; mk_b1 = s_mask[vb / group - r_first][1]; }
  }
  uint32_t qf[D / 16][4];
  {
    const uint32_t* qa = reinterpret_cast<const uint32_t*>(a.q + ((size_t)prow_a * a.Hq + head_a) * D);
    const uint32_t* qb = reinterpret_cast<const uint32_t*>(a.q + ((size_t)prow_b * a.Hq + head_b) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qf[ks][0] = real_a ? __ldg(qa + ks * 8 + tq) : 0u;
      qf[ks][1] = real_b ? __ldg(qb + ks * 8 + tq) : 0u;
      qf[ks][2] = real_a ? __ldg(qa + ks * 8 + 4 + tq) : 0u;
      qf[ks][3] = real_b ? __ldg(qb + ks * 8 + 4 + tq) : 0u;
    }
  }

  Frag<D> f;
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) f.o[dn][0] = f.o[dn][1] = f.o[dn][2] = f.o[dn][3] = 0.f;
  f.m_a = f.m_b = -INFINITY;
  f.l_a = f.l_b = 0.f;

  int issued_hi = min(kStages - 1, n_stage);  // stages issued so far
  int abort_at = -1;                           // stage whose wait gave up
  for (int st = 0; st < n_stage; ++st) {
    issue(st + kStages - 1);
    if (st + kStages - 1 < n_stage) issued_hi = st + kStages;
    const int slot = st % kStages;
    // A wait that gives up marks the CTA; the decision to stop is taken by
    // all threads together after this stage's barrier.
    if (!mbar_wait_bounded(smem_u32(&s_full[slot]), (uint32_t)((st / kStages) & 1))) s_abort = 1;
    const uint32_t kbase = ring + slot * SL::kStageBytes;
    const uint32_t vbase = kbase + SL::kTensorBytes;
    const int t0 = (blk0 + 4 * st) * kBlockSize;
    if (t0 + kTB > tok_end) {
      // Slots past the last key may hold anything (unwritten cache slots, or
      // pages not loaded): zero their V rows so that P = 0 meets V = 0.
      const int first = max(0, tok_end - t0);
      for (int x = tid; x < (kTB - first) * (D / 8); x += kThreads) {
        const int t = first + x / (D / 8), c = x % (D / 8);
        *reinterpret_cast<int4*>(ring_ptr + (vbase - ring) + SL::off(t, c)) = make_int4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();  // before later TMA writes to the same slot
      __syncthreads();
    }
    if (active) {
      if (TS == 4) {
        slice_compute<D, 2>(f, qf, kbase, vbase, t0, ts * 16, ctx, tok_end, a.scale_log2, mk_a0,
                            mk_a1, mk_b0, mk_b1, lane);
      } else if (TS == 2) {
        slice_compute<D, 4>(f, qf, kbase, vbase, t0, ts * 32, ctx, tok_end, a.scale_log2, mk_a0,
                            mk_a1, mk_b0, mk_b1, lane);
      } else {
        slice_compute<D, 4>(f, qf, kbase, vbase, t0, 0, ctx, tok_end, a.scale_log2, mk_a0,
                            mk_a1, mk_b0, mk_b1, lane);
        slice_compute<D, 4>(f, qf, kbase, vbase, t0, 32, ctx, tok_end, a.scale_log2, mk_a0,
                            mk_a1, mk_b0, mk_b1, lane);
      }
    }
    __syncthreads();  // the slot is free: the next issue may overwrite it
    if (s_abort) {
      abort_at = st;
      if (tid == 0) flag(a.dev_status, SV_DEV_TIMEOUT);
      break;
    }
  }
  if (abort_at >= 0) {
    // Let copies still in flight (stages abort_at .. issued_hi - 1) land
    // before the CTA leaves; every wait is bounded.
    if (tid == 0)
      for (int st = abort_at; st < issued_hi; ++st)
        mbar_wait_bounded(smem_u32(&s_full[st % kStages]), (uint32_t)((st / kStages) & 1));
    __syncthreads();
    if constexpr (!CL) {
      return;
    } else {
      // in a cluster the CTA still meets its peers: it contributes nothing
      // (the call's status already reports the timeout)
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) f.o[dn][0] = f.o[dn][1] = f.o[dn][2] = f.o[dn][3] = 0.f;
      f.m_a = f.m_b = -INFINITY;
      f.l_a = f.l_b = 0.f;
    }
  }

  // Warps that split the tokens of one m-tile merge through shared memory
  // (the stage ring is free now): every thread hands its fragment to the
  // same lane of the ts = 0 warp.
  float* xch = reinterpret_cast<float*>(ring_ptr);
  constexpr int kFragFloats = D / 2 + 4;  // o (D/8 * 4) + m_a, m_b, l_a, l_b
  if (TS > 1) {
    if (active && ts > 0) {
      float* dst = xch + ((size_t)warp * kFragFloats) * 32 + lane;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn)
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[(dn * 4 + e) * 32] = f.o[dn][e];
      dst[(D / 2 + 0) * 32] = f.m_a;
      dst[(D / 2 + 1) * 32] = f.m_b;
      dst[(D / 2 + 2) * 32] = f.l_a;
      dst[(D / 2 + 3) * 32] = f.l_b;
    }
    __syncthreads();
    if (active && ts == 0) {
      for (int t = 1; t < TS; ++t) {
        const float* src = xch + ((size_t)(warp + t * MT) * kFragFloats) * 32 + lane;
        const float m2a = src[(D / 2 + 0) * 32], m2b = src[(D / 2 + 1) * 32];
        const float l2a = src[(D / 2 + 2) * 32], l2b = src[(D / 2 + 3) * 32];
        const float na = fmaxf(f.m_a, m2a), nb = fmaxf(f.m_b, m2b);
        const float ba = na == -INFINITY ? 0.f : na, bb = nb == -INFINITY ? 0.f : nb;
        const float s1a = exp2f(f.m_a - ba), s2a = exp2f(m2a - ba);
        const float s1b = exp2f(f.m_b - bb), s2b = exp2f(m2b - bb);
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          f.o[dn][0] = f.o[dn][0] * s1a + src[(dn * 4 + 0) * 32] * s2a;
          f.o[dn][1] = f.o[dn][1] * s1a + src[(dn * 4 + 1) * 32] * s2a;
          f.o[dn][2] = f.o[dn][2] * s1b + src[(dn * 4 + 2) * 32] * s2b;
          f.o[dn][3] = f.o[dn][3] * s1b + src[(dn * 4 + 3) * 32] * s2b;
        }
        f.l_a = f.l_a * s1a + l2a * s2a;
        f.l_b = f.l_b * s1b + l2b * s2b;
        f.m_a = na;
        f.m_b = nb;
      }
    }
  }
  const bool owner = active && ts == 0;
  if (owner) {
    f.l_a += __shfl_xor_sync(0xffffffffu, f.l_a, 1);
    f.l_a += __shfl_xor_sync(0xffffffffu, f.l_a, 2);
    f.l_b += __shfl_xor_sync(0xffffffffu, f.l_b, 1);
    f.l_b += __shfl_xor_sync(0xffffffffu, f.l_b, 2);
  }
  if constexpr (CL) {
    cluster_merge<D>(a, f, owner, real_a, real_b, vl_a, vl_b, tq, ring_ptr, Mu, vr0, cu + ri.b, g);
    return;
  }

  if (ri.nsplit == 1) {
    if (!owner) return;
    const float inv_a = f.l_a > 0.f ? 1.f / f.l_a : 0.f;
    const float inv_b = f.l_b > 0.f ? 1.f / f.l_b : 0.f;
    uint32_t* oa = reinterpret_cast<uint32_t*>(a.out + ((size_t)prow_a * a.Hq + head_a) * D);
    uint32_t* ob = reinterpret_cast<uint32_t*>(a.out + ((size_t)prow_b * a.Hq + head_b) * D);
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      if (real_a) oa[dn * 4 + tq] = pack_bf16(f.o[dn][0] * inv_a, f.o[dn][1] * inv_a);
      if (real_b) ob[dn * 4 + tq] = pack_bf16(f.o[dn][2] * inv_b, f.o[dn][3] * inv_b);
    }
    return;
  }

  // Several splits: write this split's partials, then the group's last CTA merges.
  float* ml_all = reinterpret_cast<float*>(a.ws + a.L.ml);
  float* op_all = reinterpret_cast<float*>(a.ws + a.L.o);
  if (owner) {
    float* ml = ml_all + (size_t)u * kTileRows * 2;
    float* op = op_all + (size_t)u * kTileRows * D;
    if (tq == 0) {
      if (real_a) { ml[2 * vl_a] = f.m_a; ml[2 * vl_a + 1] = f.l_a; }
      if (real_b) { ml[2 * vl_b] = f.m_b; ml[2 * vl_b + 1] = f.l_b; }
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      if (real_a)
        *reinterpret_cast<float2*>(op + (size_t)vl_a * D + dn * 8 + 2 * tq) = make_float2(f.o[dn][0], f.o[dn][1]);
      if (real_b)
        *reinterpret_cast<float2*>(op + (size_t)vl_b * D + dn * 8 + 2 * tq) = make_float2(f.o[dn][2], f.o[dn][3]);
    }
  }
  if (a.L.small) return;  // merge_kernel combines the splits
  __threadfence();
  __syncthreads();
  const int gidx = ri.ubase + (rt * a.Hkv + g) * ri.nsplit;  // unit of split 0
  if (tid == 0) {
    int* tickets = reinterpret_cast<int*>(a.ws + a.L.tickets);
    const int prev = atomicAdd(tickets + gidx, 1);
    s_last = prev == ri.nsplit - 1;
    if (s_last) tickets[gidx] = 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // the group's last CTA merges alone: sixteen splits' loads in flight per
  // lane halve its rounds (the main loop's registers are free by now)
  merge_splits<D, kTileRows, 16>(a, ml_all, op_all, gidx, ri.nsplit, 0, Mu, vr0, cu + ri.b, g, tid,
                             kThreads);
}

// ------------------------------------------------------------ tcgen05 --
// Units of 128 virtual rows (the dense tiles of draft trees and long chains:
// query rows x GQA group >= 128 per KV head) run on the fifth-generation
// tensor cores with the accumulators in tensor memory:
//   S = Q K^T (M 128 x N 64 tokens x K 128, Q and K from shared memory) and
//   O += P V (M 128 x N 128 x K 64 tokens, P from tensor memory, V from
//   shared memory as an MN-major operand) per 64-token stage, tcgen05.mma
//   issued by one thread;
//   warps 0-3: thread t owns virtual row t (TMEM lane t): it loads S from
//     tensor memory, masks, keeps the running max and sum, and writes P
//     (bf16, two per column) back over the first half of S's columns; it
//     rescales the O accumulator in tensor memory only when its max grows
//     by more than 2^8 (P stays below 256: exact in fp32, within bf16's
//     range);
//   warps 4 and 6: the TMA loads of K (warp 4, which also allocates the
//     tensor memory) and of V (warp 6) pages into a 2-slot ring (each slot K
//     16 KB then V 16 KB, 64-element halves of d as 8-row swizzle atoms, the
//     layout both MMAs read).  K and V of a slot are refilled on their own
//     schedules: K of stage s + 2 as soon as QK^T of stage s has run, V once
//     PV of stage s has;
//   warp 5: the MMA thread (QK^T of stage s + 1 is issued before PV of stage
//     s, so the tensor cores work while the softmax warps do).
// Two CTAs per SM (97 KB of shared memory and 256 TMEM columns each).
// Every wait is bounded; a CTA that gives up flags SV_DEV_TIMEOUT, lets its
// copies and MMAs land and frees its tensor memory before it returns.
namespace tcu {
constexpr int kTok = 64;                      // tokens per stage
constexpr int kThreads = 224;
constexpr int kQBytes = kTcRows * 256;        // Q: two halves of d, 128 rows x 128 B each
constexpr int kHalf = kTok * 128;             // one 64-element half of d for 64 tokens
constexpr int kSlotBytes = 4 * kHalf;         // K (two halves), then V (two halves)
constexpr int kSmem = kQBytes + 2 * kSlotBytes + 1024;  // + 1024-byte alignment
constexpr uint32_t kTmemCols = 256;           // S of two stages (64 columns each), O (128)
constexpr uint32_t kColO = 128;
}  // namespace tcu

// Keys t0 .. t0 + 63 that a row sees, bit j for key t0 + j: every key below
// ctx, key ctx + m for m an ancestor-or-self of the row (bit m of the 128-bit
// mask mk1:mk0), none at or past tok_end.
__device__ __forceinline__ unsigned long long stage_visible(int t0, int ctx, int tok_end,
                                                            unsigned long long mk0,
                                                            unsigned long long mk1) {
  auto low_bits = [](int n) {  // bits 0 .. n - 1, n clamped to [0, 64]
    return n <= 0 ? 0ull : n >= 64 ? ~0ull : (1ull << n) - 1ull;
  };
  unsigned long long staged;  // bit j = ancestor bit (t0 + j - ctx)
  const int sh = t0 - ctx;
  if (sh >= 128 || sh <= -64) {
    staged = 0ull;
  } else if (sh >= 64) {
    staged = mk1 >> (sh - 64);
  } else if (sh > 0) {
    staged = (mk0 >> sh) | (mk1 << (64 - sh));
  } else if (sh == 0) {
    staged = mk0;
  } else {
    staged = mk0 << (-sh);
  }
  return (low_bits(ctx - t0) | (staged & ~low_bits(ctx - t0))) & low_bits(tok_end - t0);
}

template <int D>
__global__ void __launch_bounds__(tcu::kThreads, 2)
    attend_tc_kernel(const __grid_constant__ Args a, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV) {
  static_assert(D == 128, "tcgen05 units: head_dim 128");
  griddep_entry();
  using tcu::kTok;
  using tcu::kQBytes;
  using tcu::kHalf;
  using tcu::kSlotBytes;
  using tcu::kTmemCols;
  using tcu::kColO;
  constexpr int kThreads = tcu::kThreads;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ int s_tbl[kTcMaxPages];
  __shared__ int s_par[kMaxRows];
  // per slot: K landed / K free (QK^T done), V landed / V free (PV done);
  // per S buffer: S ready, P written; PV done; drain of the MMA thread
  __shared__ __align__(8) unsigned long long s_kfull[2], s_kfree[2], s_vfull[2], s_vfree[2],
      s_sfull[2], s_pfull[2], s_odone, s_drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_issued[4];  // last stage issued into K slot 0, 1, V slot 0, 1 (-1: none)
  const Header* hdr = reinterpret_cast<const Header*>(a.ws + a.L.header);
  const int u = blockIdx.x;
  const int U = hdr->Utc;
  const WorkItem ri = reinterpret_cast<const WorkItem*>(a.ws + a.L.work_tc)[u];
  if (u >= U) return;
  const int P = ri.P;
  const int s = ri.local % ri.nsplit;
  const int rest = ri.local / ri.nsplit;
  const int g = rest % a.Hkv;
  const int rt = rest / a.Hkv;
  const int group = a.group;
  const int M = group * (ri.e - ri.b);
  const int vr0 = rt * kTcRows;
  const int Mu = min(kTcRows, M - vr0);
  const int blk0 = s * P;
  const int blk1 = min(blk0 + P, ri.nblk);
  const int ctx = ri.ctx;
  const int tok_end = min(ctx + ri.e, blk1 * kBlockSize);
  const int cu = ri.cu;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_stage = (blk1 - blk0 + 3) / 4;
  const int32_t* table = a.tables + (size_t)ri.i * a.max_blocks;
  const bool unit_masked = blk1 * kBlockSize > ctx;
  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - smem_u32(smem_raw));
  const uint32_t qs = base, ring = base + kQBytes;

  for (int p = tid; p < blk1 - blk0; p += kThreads) s_tbl[p] = __ldg(table + blk0 + p);
  if (unit_masked)
    for (int j = tid; j < ri.rows; j += kThreads) s_par[j] = a.bt.parent[cu + j];
  if (tid == 0) {
    s_abort = 0;
    for (int k = 0; k < 4; ++k) s_issued[k] = -1;
    for (int k = 0; k < 2; ++k) {
      mbar_init(smem_u32(&s_kfull[k]), 1);
      mbar_init(smem_u32(&s_kfree[k]), 1);
      mbar_init(smem_u32(&s_vfull[k]), 1);
      mbar_init(smem_u32(&s_vfree[k]), 1);
      mbar_init(smem_u32(&s_sfull[k]), 1);
      mbar_init(smem_u32(&s_pfull[k]), 128);
    }
    mbar_init(smem_u32(&s_odone), 1);
    mbar_init(smem_u32(&s_drain), 1);
    fence_mbar_init();
  }
  if (warp == 4) {
    tc5::tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tc5::tmem_relinquish();
  }
  // Q tile: thread t < 128 copies virtual row vr0 + t (zeros past the tile's
  // rows) into the K-major swizzled layout (half h of d at h * 16 KB).
  const bool real = tid < 128 && tid < Mu;
  const int va = vr0 + tid;
  const int lrow = real ? va / group : 0;  // row within the window
  if (tid < 128) {
    const int4* src = reinterpret_cast<const int4*>(
        a.q + ((size_t)(cu + ri.b + lrow) * a.Hq + g * group + (real ? va % group : 0)) * D);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int4 v = real ? __ldg(src + c) : make_int4(0, 0, 0, 0);
      const uint32_t off = (uint32_t)((c >> 3) * (kTcRows * 128) + tid * 128 + (((c & 7) ^ (tid & 7)) << 4));
      *reinterpret_cast<int4*>(base_ptr + off) = v;
    }
    fence_proxy_async_smem();
  }
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == 4 || warp == 6) {
    // --------------------------------------------------------- producers --
    // Warp 4 loads K, warp 6 V: K of stage st once QK^T of stage st - 2 has
    // run, V once its PV has, each on its own schedule.
    if (lane == 0) {
      const int half = warp == 6 ? 1 : 0;  // 0: K, 1: V
      for (int st = 0; st < n_stage; ++st) {
        const int slot = st & 1;
        int bids[4];
        uint32_t bytes = 0;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int page = blk0 + 4 * st + p;
          int bid = page < blk1 ? s_tbl[page - blk0] : -1;
          if (page < blk1 && (bid < 0 || bid >= a.num_blocks)) {
            flag(a.dev_status, SV_DEV_BAD_BLOCK_ID);
            bid = -1;
          }
          bids[p] = bid;
          if (bid >= 0) bytes += 2u * 2048u;
        }
        const uint32_t kdst = ring + slot * kSlotBytes;
        {
          unsigned long long* freeb = half ? s_vfree : s_kfree;
          unsigned long long* fullb = half ? s_vfull : s_kfull;
          if (st >= 2 &&
              !mbar_wait_bounded(smem_u32(&freeb[slot]), (uint32_t)(((st - 2) >> 1) & 1))) {
            s_abort = 1;
            break;
          }
          if (*reinterpret_cast<volatile int*>(&s_abort)) break;
          const uint32_t bar = smem_u32(&fullb[slot]);
          mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            if (bids[p] < 0) continue;
            const int y = (bids[p] * a.Hkv + g) * kBlockSize;
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_2d(kdst + half * 2 * kHalf + h * kHalf + p * 2048, half ? &tmV : &tmK,
                          64 * h, y, bar);
          }
          s_issued[2 * half + slot] = st;
        }
        if (*reinterpret_cast<volatile int*>(&s_abort)) break;
      }
    }
  } else if (warp == 5) {
    // --------------------------------------------------------- MMA issue --
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc5::idesc_bf16_f32(kTcRows, kTok, false);
      constexpr uint32_t idesc_pv = tc5::idesc_bf16_f32(kTcRows, D, true);
      // O += P V of stage j: P (bf16) over the first 32 columns of S buffer
      // j & 1 in tensor memory, V MN-major in shared memory
      auto pv = [&](int j) -> bool {
        const int slot = j & 1;
        if (!mbar_wait_bounded(smem_u32(&s_pfull[slot]), (uint32_t)((j >> 1) & 1)) ||
            !mbar_wait_bounded(smem_u32(&s_vfull[slot]), (uint32_t)((j >> 1) & 1)))
          return false;
        tc5::fence_after_sync();
        const uint32_t sb = ring + slot * kSlotBytes;
        const uint32_t ptm = tmem + (uint32_t)(slot * kTok);
#pragma unroll
        for (int ks = 0; ks < kTok / 16; ++ks) {
          const uint64_t bd = tc5::sw128_desc(sb + 2 * kHalf + ks * 2048, kHalf, 1024);
          tc5::mma_bf16_ts(tmem + kColO, ptm + ks * 8, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc5::commit(smem_u32(&s_vfree[slot]));
        tc5::commit(smem_u32(&s_odone));
        return true;
      };
      bool ok = true;
      for (int st = 0; st < n_stage && ok; ++st) {
        const int slot = st & 1;
        // K of stage st has landed, and PV of stage st - 2 -- which read its
        // P from the S buffer this QK^T overwrites -- has completed
        if (!mbar_wait_bounded(smem_u32(&s_kfull[slot]), (uint32_t)((st >> 1) & 1)) ||
            (st >= 2 &&
             !mbar_wait_bounded(smem_u32(&s_vfree[slot]), (uint32_t)(((st - 2) >> 1) & 1))) ||
            *reinterpret_cast<volatile int*>(&s_abort)) {
          ok = false;
          break;
        }
        tc5::fence_after_sync();
        const uint32_t sb = ring + slot * kSlotBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t ad = tc5::sw128_desc(qs + (ks >> 2) * (kTcRows * 128) + (ks & 3) * 32, 16, 1024);
          const uint64_t bd = tc5::sw128_desc(sb + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024);
          tc5::mma_bf16(tmem + (uint32_t)(slot * kTok), ad, bd, idesc_qk, ks > 0 ? 1u : 0u);
        }
        tc5::commit(smem_u32(&s_sfull[slot]));
        tc5::commit(smem_u32(&s_kfree[slot]));
        if (st >= 1) ok = pv(st - 1);
      }
      if (ok && n_stage > 0) ok = pv(n_stage - 1);
      if (!ok) s_abort = 1;
      // every MMA this thread issued has completed before the CTA moves on
      tc5::commit(smem_u32(&s_drain));
      mbar_wait_bounded(smem_u32(&s_drain), 0);
    }
  } else {
    // ----------------------------------------------------- softmax, rows --
    // ancestor-or-self mask of this thread's row (only where staged slots lie)
    unsigned long long mk0 = 0ull, mk1 = 0ull;
    if (unit_masked && real) {
      int m = ri.b + lrow;
      for (int steps = 0; m >= 0 && steps <= kMaxRows; ++steps) {  // parents validated by plan
        if (m < 64) mk0 |= 1ull << m; else mk1 |= 1ull << (m - 64);
        m = s_par[m];
      }
    }
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int st = 0; st < n_stage; ++st) {
      const int slot = st & 1;
      const bool got = mbar_wait_bounded(smem_u32(&s_sfull[slot]), (uint32_t)((st >> 1) & 1));
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc5::fence_after_sync();
      // S of this row (64 keys), scaled to the log2 domain in place
      uint32_t sv[kTok];
      tc5::tmem_ld_x64(tmem + lane_base + (uint32_t)(slot * kTok), sv);
      const int t0 = (blk0 + 4 * st) * kBlockSize;
      // S stays unscaled: its max scales after (the scale is positive) and the
      // scale enters each exponent through one fma
      const float sc = a.scale_log2;
      if (t0 + kTok > ctx || t0 + kTok > tok_end) {
        // Keys of this stage the row sees, as one 64-bit word: the context,
        // then the staged slots of its ancestors-or-self, none past tok_end.
        const unsigned long long vis = stage_visible(t0, ctx, tok_end, mk0, mk1);
#pragma unroll
        for (int j = 0; j < kTok; ++j)
          if (!((vis >> j) & 1ull)) sv[j] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTok; ++j) mx = fmaxf(mx, __uint_as_float(sv[j]));
      mx *= sc;
      // a new reference max only when the row max passes it by 2^8
      const bool grow = mx > m_ref + 8.f;
      if (__any_sync(0xffffffffu, grow)) {
        const float m_new = grow ? mx : m_ref;
        const float alpha = grow ? ex2(m_ref - m_new) : 1.f;  // 0 while m_ref is -inf
        if (st > 0) {
          // O holds PV of the earlier stages: wait for the last one to land
          const bool g2 = mbar_wait_bounded(smem_u32(&s_odone), (uint32_t)((st - 1) & 1));
          if (!__all_sync(0xffffffffu, g2)) {
            ok = false;
            break;
          }
          tc5::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            tc5::tmem_ld_x32(tmem + lane_base + kColO + c, ov);
#pragma unroll
            for (int k = 0; k < 32; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
            tc5::tmem_st_x32(tmem + lane_base + kColO + c, ov);
          }
        }
        l *= alpha;
        m_ref = m_new;
      }
      const float mb = m_ref == -INFINITY ? 0.f : m_ref;
      float rs0 = 0.f, rs1 = 0.f;  // two running sums: half the dependent adds
      uint32_t pk[kTok / 2];
#pragma unroll
      for (int j = 0; j < kTok; j += 2) {
        const float p0 = ex2(fmaf(__uint_as_float(sv[j]), sc, -mb));
        const float p1 = ex2(fmaf(__uint_as_float(sv[j + 1]), sc, -mb));
        rs0 += p0;
        rs1 += p1;
        pk[j / 2] = pack_bf16(p0, p1);
      }
      l += rs0 + rs1;
      // Slots past the last key may hold anything (unwritten cache slots, or
      // pages not loaded): zero their V rows so that P = 0 meets V = 0.
      const uint32_t sb = ring + slot * kSlotBytes;
      if (t0 + kTok > tok_end) {
        // V of this stage must have landed before its tail is overwritten
        const bool gv = mbar_wait_bounded(smem_u32(&s_vfull[slot]), (uint32_t)((st >> 1) & 1));
        if (!__all_sync(0xffffffffu, gv)) {
          ok = false;
          break;
        }
        const int first = max(0, tok_end - t0);
        for (int xx = tid; xx < (kTok - first) * 16; xx += 128) {
          const int t = first + (xx >> 4), c = xx & 15;
          const uint32_t off = 2 * kHalf + (c >> 3) * kHalf + t * 128 + (((c & 7) ^ (t & 7)) << 4);
          *reinterpret_cast<int4*>(base_ptr + (sb - base) + off) = make_int4(0, 0, 0, 0);
        }
      }
      // P of row t (64 tokens, two bf16 per 32-bit column) over the first 32
      // columns of the S buffer just read
      tc5::tmem_st_x32(tmem + lane_base + (uint32_t)(slot * kTok), pk);
      fence_proxy_async_smem();  // the zeroed V rows, for the tensor cores
      tc5::fence_before_sync();
      mbar_arrive(smem_u32(&s_pfull[slot]));
    }
    // The last PV has landed: O row t, normalised, to the output or to the
    // split partials.
    // Every MMA has completed once the MMA thread's drain barrier completes
    // its only phase.  (The PV barrier would not do: a parity wait names one
    // phase only while the barrier is at most one phase from it, and here
    // the last PV may or may not have landed already.)
    if (ok && n_stage > 0) {
      const bool g3 = mbar_wait_bounded(smem_u32(&s_drain), 0u);
      if (!__all_sync(0xffffffffu, g3)) ok = false;
    }
    if (!ok) {
      s_abort = 1;
    } else {
      tc5::fence_after_sync();
      const int prow = cu + ri.b + lrow;
      const int head = g * group + (real ? va % group : 0);
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t ov[32];
        tc5::tmem_ld_x32(tmem + lane_base + kColO + c, ov);
        if (!real) continue;
        if (ri.nsplit == 1) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + ((size_t)prow * a.Hq + head) * D + c);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dst[k] = make_uint4(pack_bf16(__uint_as_float(ov[8 * k]) * inv, __uint_as_float(ov[8 * k + 1]) * inv),
                                pack_bf16(__uint_as_float(ov[8 * k + 2]) * inv, __uint_as_float(ov[8 * k + 3]) * inv),
                                pack_bf16(__uint_as_float(ov[8 * k + 4]) * inv, __uint_as_float(ov[8 * k + 5]) * inv),
                                pack_bf16(__uint_as_float(ov[8 * k + 6]) * inv, __uint_as_float(ov[8 * k + 7]) * inv));
        } else {
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(a.ws + a.L.o_tc) +
                                                  ((size_t)u * kTcRows + tid) * D + c);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(__uint_as_float(ov[4 * k]), __uint_as_float(ov[4 * k + 1]),
                                 __uint_as_float(ov[4 * k + 2]), __uint_as_float(ov[4 * k + 3]));
        }
      }
      if (real && ri.nsplit > 1)
        reinterpret_cast<float2*>(a.ws + a.L.ml_tc)[(size_t)u * kTcRows + tid] = make_float2(m_ref, l);
    }
  }

  // Every role is done with tensor memory and the ring.
  tc5::fence_before_sync();
  __syncthreads();
  tc5::fence_after_sync();
  if (s_abort) {
    // copies still in flight land before the CTA leaves (bounded waits)
    if (tid == 0) {
      flag(a.dev_status, SV_DEV_TIMEOUT);
      for (int k = 0; k < 4; ++k)
        if (s_issued[k] >= 0)
          mbar_wait_bounded(smem_u32(k < 2 ? &s_kfull[k] : &s_vfull[k - 2]),
                            (uint32_t)((s_issued[k] >> 1) & 1));
    }
    __syncthreads();
  }
  if (warp == 4) tc5::tmem_dealloc(tmem, kTmemCols);
}

// After an attention kernel whose splits only wrote partials (the tcgen05
// kernel always, the mma.sync kernel for small batches): the units of a split
// group merge the group's partials together, unit s of the group taking rows
// [s, s + 1) x ceil(rows / nsplit) -- all splits' loads in flight at once on
// many SMs, instead of one CTA reading every split of the tile.
// One launch serves both lists: CTAs [0, n_small) take the mma.sync list
// (64-row tiles; n_small = 0 unless small batches), the rest the tcgen05 list
// (128-row tiles).
constexpr int kMergeThreads = 256;
template <int D, bool TC>
__device__ __forceinline__ void merge_unit(const Args& a, int u) {
  constexpr int TILE = TC ? kTcRows : kTileRows;
  const Header* hdr = reinterpret_cast<const Header*>(a.ws + a.L.header);
  const int U = TC ? hdr->Utc : hdr->U;
  const WorkItem ri = reinterpret_cast<const WorkItem*>(a.ws + (TC ? a.L.work_tc : a.L.work))[u];
  if (u >= U || ri.nsplit == 1) return;
  const int s = ri.local % ri.nsplit;
  const int rest = ri.local / ri.nsplit;
  const int g = rest % a.Hkv;
  const int rt = rest / a.Hkv;
  const int vr0 = rt * TILE;
  const int Mu = min(TILE, a.group * (ri.e - ri.b) - vr0);
  const int per = (Mu + ri.nsplit - 1) / ri.nsplit;
  const int r0 = min(Mu, s * per), r1 = min(Mu, r0 + per);
  if (r0 >= r1) return;
  const int gidx = ri.ubase + (rt * a.Hkv + g) * ri.nsplit;  // unit of split 0
  merge_splits<D, TILE>(a, reinterpret_cast<const float*>(a.ws + (TC ? a.L.ml_tc : a.L.ml)),
                        reinterpret_cast<const float*>(a.ws + (TC ? a.L.o_tc : a.L.o)), gidx,
                        ri.nsplit, r0, r1, vr0, ri.cu + ri.b, g, threadIdx.x, kMergeThreads);
}
template <int D>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ Args a,
                                                              int n_small) {
  griddep_entry();
  const int u = blockIdx.x;
  if (u < n_small) {
    merge_unit<D, false>(a, u);
  } else if constexpr (D == 128) {
    merge_unit<D, true>(a, u - n_small);
  }
}

// cuTensorMapEncodeTiled from the driver, fetched through the runtime (no
// link against the driver library).
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// A cache viewed as rows of D bf16 (num_blocks * Hkv * 16 rows), boxes of
// 64 elements x 16 rows, 128-byte swizzle.
static bool make_map(CUtensorMap* map, const void* base, int num_blocks, int Hkv, int D) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)num_blocks * Hkv * kBlockSize};
  const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  const cuuint32_t box[2] = {64, 16};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
sv_status launch(const Args& a_in, cudaStream_t stream) {
  Args a = a_in;
  const size_t smem = (size_t)kStages * StageLayout<D>::kStageBytes + 1024;
  static PerDevice smem_set;  // the ring is above the 48 KB default
  if (smem_limit_once(smem_set, attend_kernel<D, false>, smem) != cudaSuccess) return SV_ERR_CUDA;
  static ClusterFit cluster_fit;  // sets the cluster kernel's shared-memory limit too
  CUtensorMap tmK, tmV;
  if (!make_map(&tmK, a.k, a.num_blocks, a.Hkv, D) || !make_map(&tmV, a.v, a.num_blocks, a.Hkv, D))
    return SV_ERR_CUDA;
  const size_t plan_smem =
      a.bt.n_req <= kPlanSmemRequests ? sizeof(ReqInfo) * (size_t)a.bt.n_req : 0;
  // one thread per request (its block-wide scans and barriers cost less with
  // fewer warps), at least four warps to write the work items, at most 1024
  const int plan_threads = min(1024, max(128, (a.bt.n_req + 31) / 32 * 32));
  // small one-pass calls: the one-warp planner, and split groups that merge
  // within a cluster -- when no window can reach the tcgen05 list (a cluster
  // launch behind the tcgen05 kernel waits for whole GPCs to drain: measured
  // 4-5 us slower on the draft tree), a split's block ids fit in shared
  // memory and every group's cluster can be resident at once (the device's
  // count of active 16-CTA clusters, 14 on this GPU: a second wave of
  // clusters would cost a whole split's time)
  const bool warp_plan = a.L.small && a.chunk.index < 0;
  a.cl = warp_plan && a.L.ucap_tc == 0 &&
                 (a.max_blocks + kClusterSplits - 1) / kClusterSplits <= kMaxPagesPerSplit &&
                 cluster_fit.get(attend_kernel<D, true>, kClusterSplits, kThreads, smem) >=
                     a.L.ucap_cl / kClusterSplits
             ? kClusterSplits
             : 0;
  if ((warp_plan ? sv::launch(plan_small_kernel, 1, 32, 0, stream, a)
                 : sv::launch(plan_kernel, 1, plan_threads, plan_smem, stream, a)) != cudaSuccess)
    return SV_ERR_CUDA;
  // the tensor-core units first (the long ones when there are any), then the
  // mma.sync units, then one merge launch for every split group
  int ucap_tc = 0;
  if constexpr (D == 128) {
    ucap_tc = a.L.ucap_tc;
    if (ucap_tc > 0) {
      static PerDevice smem_set_tc;
      if (smem_limit_once(smem_set_tc, attend_tc_kernel<D>, tcu::kSmem) != cudaSuccess)
        return SV_ERR_CUDA;
      if (sv::launch(attend_tc_kernel<D>, ucap_tc, tcu::kThreads, tcu::kSmem, stream, a, tmK,
                     tmV) != cudaSuccess)
        return SV_ERR_CUDA;
    }
  }
  const cudaError_t e =
      a.cl > 0 ? sv::launch_cluster(attend_kernel<D, true>, a.L.ucap_cl, kThreads, smem, stream,
                                    a.cl, a, tmK, tmV)
               : sv::launch(attend_kernel<D, false>, a.L.ucap, kThreads, smem, stream, a, tmK, tmV);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  const int n_small = a.L.small && a.cl == 0 ? a.L.ucap : 0;
  if (n_small + ucap_tc > 0 &&
      sv::launch(merge_kernel<D>, n_small + ucap_tc, kMergeThreads, 0, stream, a, n_small) !=
          cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

}  // namespace attn
}  // namespace sv

using namespace sv;

static sv_status check_attend_args(const sv_batch* bt, const sv_paged_kv* kv, int32_t Hq) {
  if (!bt || !kv) return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req < 0 || bt->total_rows < 0 || bt->max_rows_per_req < 1) return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req > 0 && (!bt->cu_rows || !bt->parent)) return SV_ERR_INVALID_ARGUMENT;
  if (bt->max_rows_per_req > kMaxRows) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->block_size != kBlockSize) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->head_dim != 64 && kv->head_dim != 128) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->n_kv_heads < 1 || Hq < 1 || Hq % kv->n_kv_heads != 0) return SV_ERR_INVALID_ARGUMENT;
  if (Hq / kv->n_kv_heads > 16) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->num_blocks < 0 || kv->max_blocks_per_req < 0) return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req > 0 && (!kv->k_cache || !kv->v_cache || !kv->block_tables || !kv->cache_lens))
    return SV_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)kv->k_cache | (uintptr_t)kv->v_cache) & 15) return SV_ERR_INVALID_ARGUMENT;
  return SV_OK;
}

extern "C" size_t sv_tree_attend_workspace(const sv_batch* bt, const sv_paged_kv* kv,
                                           int32_t n_q_heads) {
  if (check_attend_args(bt, kv, n_q_heads) != SV_OK) return 0;
  const int group = n_q_heads / kv->n_kv_heads;
  return attn::layout(bt->n_req, bt->total_rows, group, kv->n_kv_heads, kv->head_dim,
                      kv->max_blocks_per_req, bt->max_rows_per_req).total;
}

namespace sv {
namespace attn {

sv_status tree_attend(const sv_paged_kv* kv, const sv_batch* bt, const void* q, int32_t n_q_heads,
                      float softmax_scale, void* out, void* ws, size_t ws_bytes,
                      int32_t* dev_status, cudaStream_t stream, const ChunkPlan& chunk) {
  sv_status st = check_attend_args(bt, kv, n_q_heads);
  if (st != SV_OK) return st;
  if (bt->n_req == 0 || bt->total_rows == 0) return SV_OK;
  if (!q || !out || !ws) return SV_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)q | (uintptr_t)out) & 3) return SV_ERR_INVALID_ARGUMENT;
  if ((uintptr_t)ws & 255) return SV_ERR_INVALID_ARGUMENT;
  if (!(softmax_scale > 0.f)) return SV_ERR_INVALID_ARGUMENT;
  if (chunk.index >= 0 &&
      (chunk.size < 1 || !chunk.row_begin || !chunk.row_end || !chunk.act ||
       (chunk.index > 0 && !chunk.done)))
    return SV_ERR_INVALID_ARGUMENT;
  const int group = n_q_heads / kv->n_kv_heads;
  Args a;
  a.bt = *bt;
  a.k = static_cast<const __nv_bfloat16*>(kv->k_cache);
  a.v = static_cast<const __nv_bfloat16*>(kv->v_cache);
  a.num_blocks = kv->num_blocks;
  a.Hkv = kv->n_kv_heads;
  a.max_blocks = kv->max_blocks_per_req;
  a.tables = kv->block_tables;
  a.cache_lens = kv->cache_lens;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.out = static_cast<__nv_bfloat16*>(out);
  a.Hq = n_q_heads;
  a.group = group;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.ws = static_cast<uint8_t*>(ws);
  a.L = layout(bt->n_req, bt->total_rows, group, kv->n_kv_heads, kv->head_dim,
               kv->max_blocks_per_req, bt->max_rows_per_req);
  a.dev_status = dev_status;
  a.chunk = chunk;
  a.cl = 0;
  if (ws_bytes < a.L.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  return kv->head_dim == 128 ? launch<128>(a, stream) : launch<64>(a, stream);
}

}  // namespace attn
}  // namespace sv

extern "C" sv_status sv_tree_attend(const sv_paged_kv* kv, const sv_batch* bt, const void* q,
                                    int32_t n_q_heads, float softmax_scale, void* out, void* ws,
                                    size_t ws_bytes, int32_t* dev_status, void* stream) {
  SV_TRACE("sv_tree_attend");
  const attn::ChunkPlan none{-1, 0, nullptr, nullptr, nullptr, nullptr, nullptr};
  return attn::tree_attend(kv, bt, q, n_q_heads, softmax_scale, out, ws, ws_bytes, dev_status,
                           static_cast<cudaStream_t>(stream), none);
}
