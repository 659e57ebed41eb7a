// chunk.cu — chunked verification with early pruning (with the KV commit
// fused in), the chunk-size rule, the bounded-wait self test and the status
// strings.
//
// Source: [FASER] "FASER의 세 가지 메커니즘", mechanism 2 (early token
// pruning: verification is cut into chunks and, at every chunk boundary, the
// tokens behind an already rejected prefix are dropped, so no cycles are
// spent on them) and the operations notes (the verification attention kernel
// has to run on a part of the rows).
//
// The whole step is enqueued on one stream with no host synchronisation: per
// chunk, the attention planner turns `done` into the chunk's windows
// (requests that are done get an empty window, which every later kernel
// skips) and the accept list, the attention runs on those windows, then the
// accept statistics and decisions; one race pass after the last chunk draws
// every request's emitted token.  With the fused commit, the decision that
// stops a request also commits it, and the last request to stop releases the
// freed blocks.  sv_chunk_windows exposes the window rule on its own;
// sv_select_chunk prices each chunk size for the next step (the FASER remark
// that the chunk size follows the load).

#include <stdio.h>

#include "sv_accept_internal.h"
#include "sv_attend_internal.h"
#include "sv_internal.cuh"

namespace sv {
namespace chk {

__global__ void __launch_bounds__(256) windows_kernel(sv_batch bt, int c, int cs,
                                                      const int32_t* done, int32_t* rb,
                                                      int32_t* re, int32_t* dev_status) {
  griddep_entry();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= bt.n_req) return;
  bool bad = false;
  const Window w = chunk_window(bt, i, c, cs, done, &bad);
  if (bad && c == 0) flag(dev_status, SV_DEV_BAD_WINDOW);
  rb[i] = w.b;
  re[i] = w.e;
}

// The chunk driver's own part of the workspace: row_begin and row_end [R],
// then the accept list's row ranges [R] (int4 per listed request).
inline size_t windows_bytes(int R) {
  return align256(sizeof(int32_t) * (size_t)R) * 2 + align256(sizeof(int4) * (size_t)R);
}

}  // namespace chk
}  // namespace sv

using namespace sv;

extern "C" const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARGUMENT: return "invalid argument";
    case SV_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case SV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case SV_ERR_CUDA: return "CUDA launch failed";
  }
  return "unknown status";
}

extern "C" const char* sv_version(void) { return "libspecverify 0.1 (sm_103a)"; }

// ------------------------------------------------- bounded-wait self test --
// One thread arms an mbarrier for two arrivals, arrives once and waits on
// the phase with the bounded wait every kernel of the library uses: the wait
// cannot complete, gives up after `limit` rounds and the kernel reports
// SV_DEV_TIMEOUT; the second arrival then completes the phase, so nothing is
// left pending when the CTA exits.
namespace sv {
namespace chk {
__global__ void __launch_bounds__(32) selftest_wait_kernel(int limit, int32_t* dev_status) {
  griddep_entry();
  __shared__ __align__(8) unsigned long long bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 2);
  fence_mbar_init();
  mbar_arrive(b);
  if (!mbar_wait_bounded(b, 0, limit)) flag(dev_status, SV_DEV_TIMEOUT);
  mbar_arrive(b);
  if (!mbar_wait_bounded(b, 0, limit)) flag(dev_status, SV_DEV_UNSUPPORTED);  // never expected
}
}  // namespace chk
}  // namespace sv

// Chunk size of least expected cost ([FASER] mechanism 2, the chunk size
// following the load; the rule is the one in the header).  One CTA per
// candidate size c: its threads take the requests, each term in fp64 with
// every operation rounded on its own (__dmul_rn / __dadd_rn), truncated to
// whole bytes and summed as u64 (any order gives the same integer); then one
// warp picks the least cost, the larger size on ties.
namespace sv {
namespace chk {
constexpr int kChunkThreads = 256;

__global__ void __launch_bounds__(kChunkThreads) chunk_cost_kernel(
    int n_req, const int32_t* rows, const int32_t* ctx, const double* state, double kv_bytes,
    double row_bytes, unsigned long long chunk_bytes, unsigned long long* costs,
    int32_t* dev_status) {
  griddep_entry();
  const int c = blockIdx.x + 1;
  __shared__ int s_max[kChunkThreads / 32];
  __shared__ unsigned long long s_total;
  // the largest valid rows_i (every CTA computes it)
  int mr = 0;
  for (int i = threadIdx.x; i < n_req; i += kChunkThreads) {
    const int r = rows[i], x = ctx[i];
    const double S = state[2 * i], N = state[2 * i + 1];
    const bool ok = r >= 1 && r <= kMaxRows && x >= 0 && isfinite(S) && isfinite(N) &&
                    S >= 0.0 && N >= 0.0;
    if (ok) mr = max(mr, r);
    else if (c == 1) flag(dev_status, SV_DEV_BAD_LENGTH);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mr = max(mr, __shfl_xor_sync(0xffffffffu, mr, o));
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = mr;
  if (threadIdx.x == 0) s_total = 0ull;
  __syncthreads();
  int max_rows = 0;
  for (int w = 0; w < kChunkThreads / 32; ++w) max_rows = max(max_rows, s_max[w]);
  if (c > max_rows) {
    if (threadIdx.x == 0) costs[c - 1] = ~0ull;
    return;
  }
  unsigned long long part = 0ull;
  for (int i = threadIdx.x; i < n_req; i += kChunkThreads) {
    const int r = rows[i], x = ctx[i];
    const double S = state[2 * i], N = state[2 * i + 1];
    if (!(r >= 1 && r <= kMaxRows && x >= 0 && isfinite(S) && isfinite(N) && S >= 0.0 &&
          N >= 0.0))
      continue;
    const double alpha = fmin(1.0, __ddiv_rn(__dadd_rn(S, 1.0), __dadd_rn(N, 2.0)));
    double ac = 1.0;
    for (int t = 0; t < c; ++t) ac = __dmul_rn(ac, alpha);
    double P = 1.0;
    for (int b = 0; b < r; b += c) {
      const int e = min(b + c, r);
      const double bytes = __dadd_rn(__dmul_rn((double)(x + e), kv_bytes),
                                     __dmul_rn((double)(e - b), row_bytes));
      part += __double2ull_rz(__dmul_rn(P, bytes));
      P = __dmul_rn(P, ac);
    }
  }
  atomicAdd(&s_total, part);
  __syncthreads();
  if (threadIdx.x == 0)
    costs[c - 1] = (unsigned long long)((max_rows + c - 1) / c) * chunk_bytes + s_total;
}

__global__ void __launch_bounds__(32) chunk_pick_kernel(const unsigned long long* costs,
                                                        int32_t* chunk,
                                                        unsigned long long* cost) {
  griddep_entry();
  if (threadIdx.x != 0) return;
  int best = 1;
  unsigned long long bc = 0ull;
  bool any = false;
  for (int c = 1; c <= kMaxRows; ++c) {
    const unsigned long long v = costs[c - 1];
    if (v == ~0ull) continue;
    if (!any || v <= bc) {
      best = c;
      bc = v;
      any = true;
    }
  }
  *chunk = best;
  *cost = any ? bc : 0ull;
}
}  // namespace chk
}  // namespace sv

extern "C" sv_status sv_select_chunk(int32_t n_req, const int32_t* rows, const int32_t* ctx,
                                     const double* state, double kv_bytes, double row_bytes,
                                     uint64_t chunk_bytes, int32_t* chunk, uint64_t* cost,
                                     uint64_t* costs, int32_t* dev_status, void* stream) {
  SV_TRACE("sv_select_chunk");
  if (n_req < 0 || !(kv_bytes >= 0.0) || !(row_bytes >= 0.0) || isinf(kv_bytes) ||
      isinf(row_bytes))
    return SV_ERR_INVALID_ARGUMENT;
  if (!chunk || !cost || !costs || (n_req > 0 && (!rows || !ctx || !state)))
    return SV_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long* c64 = reinterpret_cast<unsigned long long*>(costs);
  if (sv::launch(chk::chunk_cost_kernel, kMaxRows, chk::kChunkThreads, 0, s, (int)n_req, rows,
                 ctx, state, kv_bytes, row_bytes, (unsigned long long)chunk_bytes, c64,
                 dev_status) != cudaSuccess)
    return SV_ERR_CUDA;
  if (sv::launch(chk::chunk_pick_kernel, 1, 32, 0, s, (const unsigned long long*)c64, chunk,
                 reinterpret_cast<unsigned long long*>(cost)) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

extern "C" sv_status sv_selftest_bounded_wait(int32_t limit, int32_t* dev_status, void* stream) {
  SV_TRACE("sv_selftest_bounded_wait");
  if (limit < 1 || limit > kWaitLimit || !dev_status) return SV_ERR_INVALID_ARGUMENT;
  if (sv::launch(chk::selftest_wait_kernel, 1, 32, 0, static_cast<cudaStream_t>(stream),
                 (int)limit, dev_status) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

extern "C" sv_status sv_chunk_windows(const sv_batch* bt, int32_t chunk_index, int32_t chunk_size,
                                      const int32_t* done, int32_t* row_begin, int32_t* row_end,
                                      void* stream) {
  SV_TRACE("sv_chunk_windows");
  if (!bt || chunk_index < 0 || chunk_size < 1 || !row_begin || !row_end || bt->n_req < 0)
    return SV_ERR_INVALID_ARGUMENT;
  if (chunk_index > 0 && !done) return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req == 0) return SV_OK;
  if (!bt->cu_rows) return SV_ERR_INVALID_ARGUMENT;
  if (sv::launch(chk::windows_kernel, (bt->n_req + 255) / 256, 256, 0,
                 static_cast<cudaStream_t>(stream), *bt, chunk_index, chunk_size, done, row_begin,
                 row_end, (int32_t*)nullptr) != cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}

extern "C" size_t sv_verify_chunked_workspace(const sv_batch* bt, const sv_paged_kv* kv,
                                              int32_t n_q_heads, int32_t vocab) {
  if (!bt || !kv || vocab < 1) return 0;
  const size_t wa = sv_tree_attend_workspace(bt, kv, n_q_heads);
  if (!wa) return 0;
  // The chunk size is not an argument here: the accept part is sized for
  // one-row windows, the largest of its layouts (fewer rows per window give
  // more vocabulary slices per row), so it fits every chunk size; it also
  // holds the fused commit's ticket and spans.
  const size_t wb = acc::layout(bt->n_req, bt->total_rows, vocab, 1, true).total;
  return chk::windows_bytes(bt->n_req) + align256(wb) + wa;
}

namespace {

// The chunked step; with `pool` the accept kernels also commit every request
// in the chunk where it stops (the same cache `kv` the attention reads: a
// stopped request is never attended again, and its released blocks go back
// to the pool only after the last request has stopped).
sv_status verify_chunked(const sv_paged_kv* kv, const sv_batch* bt, const void* q,
                         int32_t n_q_heads, float softmax_scale, void* out,
                         const float* target_logits, const float* draft_logits, int32_t vocab,
                         float temperature, uint64_t seed, int32_t chunk_size,
                         int32_t* accepted_len, int32_t* accepted_nodes, int32_t* next_token,
                         uint8_t* ambiguous, int32_t* done, const sv_block_pool* pool, void* ws,
                         size_t ws_bytes, int32_t* dev_status, void* stream) {
  if (!kv || !bt || chunk_size < 1 || !done) return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req < 0 || bt->max_rows_per_req < 1) return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req == 0 || bt->total_rows == 0) return SV_OK;
  const size_t wa = sv_tree_attend_workspace(bt, kv, n_q_heads);
  if (!wa || vocab < 1) return SV_ERR_INVALID_ARGUMENT;
  const bool commit = pool != nullptr;
  const acc::Layout AL = acc::layout(bt->n_req, bt->total_rows, vocab, chunk_size, commit);
  const size_t need = chk::windows_bytes(bt->n_req) + align256(AL.total) + wa;
  if (!ws || ((uintptr_t)ws & 255)) return SV_ERR_INVALID_ARGUMENT;
  if (ws_bytes < need) return SV_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = static_cast<uint8_t*>(ws);
  int32_t* rb = reinterpret_cast<int32_t*>(w);
  int32_t* re = reinterpret_cast<int32_t*>(w + align256(sizeof(int32_t) * (size_t)bt->n_req));
  int4* act4 = reinterpret_cast<int4*>(w + 2 * align256(sizeof(int32_t) * (size_t)bt->n_req));
  uint8_t* acc_ws = w + chk::windows_bytes(bt->n_req);
  uint8_t* att_ws = acc_ws + align256(AL.total);
  sv_batch b2 = *bt;
  b2.row_begin = rb;
  b2.row_end = re;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int n_chunks = (bt->max_rows_per_req + chunk_size - 1) / chunk_size;
  for (int c = 0; c < n_chunks; ++c) {
    char name[32];
    snprintf(name, sizeof(name), "chunk %d", c);
    TraceRange chunk_range(name);
    // The planner turns `done` into this chunk's windows and the accept list.
    const attn::ChunkPlan cp{c, chunk_size, done, rb, re,
                             reinterpret_cast<int32_t*>(acc_ws + AL.act), act4};
    sv_status st = attn::tree_attend(kv, bt, q, n_q_heads, softmax_scale, out, att_ws, wa,
                                     dev_status, s, cp);
    if (st != SV_OK) return st;
    st = acc::run(&b2, target_logits, draft_logits, vocab, temperature, seed, accepted_len,
                  accepted_nodes, next_token, ambiguous, done, nullptr, acc_ws, AL.total,
                  dev_status, s, chunk_size, c, commit ? kv : nullptr, pool, act4);
    if (st != SV_OK) return st;
  }
  // Nothing in a later chunk depends on the drawn tokens: one race pass
  // after the last chunk serves every request at once.
  return acc::race_all(bt, target_logits, draft_logits, vocab, temperature, seed, next_token,
                       acc_ws, chunk_size, dev_status, s);
}

}  // namespace

extern "C" sv_status sv_verify_chunked(const sv_paged_kv* kv, const sv_batch* bt, const void* q,
                                       int32_t n_q_heads, float softmax_scale, void* out,
                                       const float* target_logits, const float* draft_logits,
                                       int32_t vocab, float temperature, uint64_t seed,
                                       int32_t chunk_size, int32_t* accepted_len,
                                       int32_t* accepted_nodes, int32_t* next_token,
                                       uint8_t* ambiguous, int32_t* done, void* ws,
                                       size_t ws_bytes, int32_t* dev_status, void* stream) {
  SV_TRACE("sv_verify_chunked");
  return verify_chunked(kv, bt, q, n_q_heads, softmax_scale, out, target_logits, draft_logits,
                        vocab, temperature, seed, chunk_size, accepted_len, accepted_nodes,
                        next_token, ambiguous, done, nullptr, ws, ws_bytes, dev_status, stream);
}

extern "C" sv_status sv_verify_chunked_commit(
    const sv_paged_kv* kv, const sv_batch* bt, const void* q, int32_t n_q_heads,
    float softmax_scale, void* out, const float* target_logits, const float* draft_logits,
    int32_t vocab, float temperature, uint64_t seed, int32_t chunk_size, int32_t* accepted_len,
    int32_t* accepted_nodes, int32_t* next_token, uint8_t* ambiguous, int32_t* done,
    const sv_block_pool* pool, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream) {
  SV_TRACE("sv_verify_chunked_commit");
  if (!kv || !bt || !pool) return SV_ERR_INVALID_ARGUMENT;
  if (kv->block_size != kBlockSize) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->head_dim != 64 && kv->head_dim != 128) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->n_kv_heads < 1 || kv->num_blocks < 0 || kv->max_blocks_per_req < 0 ||
      pool->capacity < 0)
    return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req > 0 && (!kv->k_cache || !kv->v_cache || !kv->block_tables || !kv->cache_lens ||
                        !pool->free_list || !pool->free_count))
    return SV_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)kv->k_cache | (uintptr_t)kv->v_cache) & 15) return SV_ERR_INVALID_ARGUMENT;
  return verify_chunked(kv, bt, q, n_q_heads, softmax_scale, out, target_logits, draft_logits,
                        vocab, temperature, seed, chunk_size, accepted_len, accepted_nodes,
                        next_token, ambiguous, done, pool, ws, ws_bytes, dev_status, stream);
}
