/*
 * libspecverify — target-side speculative-decoding verification on one GPU
 * (sm_103a).  C ABI: plain pointers and sizes, no framework types.
 *
 * A verification step takes, for every request, a chain or tree of draft
 * tokens and decides which of them the target model accepts:
 *   sv_tree_attend    padding-free attention of the draft rows against a
 *                     paged bf16 GQA KV cache, each row seeing only its own
 *                     root-to-node prefix;
 *   sv_accept         per-row vocabulary softmax and the lossless accept /
 *                     reject rule (or greedy longest matching prefix);
 *   sv_commit_kv      the accepted path's K/V kept, rejected blocks freed;
 *   sv_accept_commit  sv_accept and sv_commit_kv fused in the same kernels;
 *   sv_select_budget  how many drafts of each request to verify, by sorting
 *                     every (request, position) by prefix survival and
 *                     maximising tau * SPS(B);
 *   sv_chunk_windows, sv_verify_chunked, sv_verify_chunked_commit
 *                     verification in chunks of rows with early pruning of
 *                     requests whose prefix was rejected;
 *   sv_adapt_gamma    each request's next draft length from its own
 *                     acceptance history;
 *   sv_select_chunk   the chunk size of least expected cost for the next
 *                     chunked step.
 *
 * Sources (pages by title; section names glossed):
 *   [SwiftSpec] "SwiftSpec: 드래프터와 타깃을 서로 다른 GPU에 분리하고 비동기로
 *               겹쳐 실행해 LLM 저지연 추론을 실현하는 방법 (ASPLOS 2026)",
 *               core design, mechanism 2 (tree-aware KV cache management:
 *               every node has its own KV prefix; only the accepted path's
 *               KV is kept, rejected paths are freed at once) and mechanism 3
 *               (a padding-free attention kernel verifying all draft tokens
 *               at once; verification result and KV update fused).
 *   [DSpark]    "DSpark 하드웨어 인식 검증 스케줄러와 반자동회귀 병렬 드래프터를
 *               통한 LLM 추론 가속화", hardware-aware prefix scheduler,
 *               method, technical detail, glossary (speculative decoding:
 *               the longest matching prefix is accepted and the target
 *               distribution is preserved; prefix survival).
 *   [FASER]     "FASER: 연속 배치 내 투기 디코딩의 단계 직렬화를 공간 분할 중첩으로
 *               해결하는 방법", three mechanisms: 1 per-request speculation
 *               length, 2 early token pruning (chunked verification);
 *               operations notes (the attention kernel must run on a chunk).
 *   [SSD]       "SSD: 병렬 하드웨어를 활용한 초고속 추론 알고리즘 Speculative
 *               Speculative Decoding", section details (PagedAttention).
 *
 * Conventions for every call:
 *   - Every pointer inside the structs and every array argument is a DEVICE
 *     pointer owned by the caller; the library allocates nothing, keeps no
 *     state between calls and frees nothing.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  Errors that the host can see (null pointers, bad
 *     sizes, small workspace) are returned before anything is enqueued.
 *   - A workspace (`ws`) is scratch owned by the caller: its contents need no
 *     initialisation and are not kept between calls (every word a call reads
 *     it has written first).  Two calls whose work overlaps on the GPU need
 *     separate workspaces.
 *   - Errors that depend on device data (a block id out of range, a parent
 *     that is not an earlier row, an invalid window, a full free list) are
 *     OR-ed as SV_DEV_* bits into *dev_status (a caller-owned device int32
 *     that the caller zeroes) and the affected request is skipped; no kernel
 *     traps or asserts.  dev_status may be NULL, in which case such findings
 *     are dropped (the affected request is still skipped).
 *   - SV_ERR_CUDA means a launch failed; the call may have been partly
 *     enqueued.
 */
#ifndef LIBSPECVERIFY_H
#define LIBSPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARGUMENT = 1,
  SV_ERR_UNSUPPORTED_SHAPE = 2,
  SV_ERR_WORKSPACE_TOO_SMALL = 3,
  SV_ERR_CUDA = 4
} sv_status;

/* Device-side findings OR-ed into *dev_status. */
#define SV_DEV_BAD_BLOCK_ID 1    /* block table entry outside [0, num_blocks) */
#define SV_DEV_BAD_PARENT 2      /* parent[0] != -1, or parent[j] not in [0, j) */
#define SV_DEV_POOL_OVERFLOW 4   /* free list has no room for released blocks */
#define SV_DEV_BAD_WINDOW 8      /* window outside [0, rows], tree not verified whole,
                                    continuation that does not match the state,
                                    invalid accepted path given to commit */
#define SV_DEV_TIMEOUT 16        /* reserved: a bounded device wait gave up */
#define SV_DEV_BAD_TOKEN 32      /* draft token outside [0, vocab) */
#define SV_DEV_UNSUPPORTED 64    /* reserved (no longer raised: trees at temperature > 0 are sampled) */
#define SV_DEV_BAD_LENGTH 128    /* ctx + rows does not fit the block table */

/* Paged KV cache ([SSD] PagedAttention; [SwiftSpec] mechanism 2).
 * k_cache, v_cache: bf16 [num_blocks][n_kv_heads][block_size][head_dim];
 *   one (block, head) page is block_size * head_dim contiguous bf16.
 * block_tables: int32 [n_req][max_blocks_per_req]; entry t holds the pool
 *   block of cache slots [t*block_size, (t+1)*block_size); -1 = unused.
 * cache_lens: int32 [n_req], ctx_i = committed tokens of request i.  The
 *   draft rows' K/V of this step are STAGED at slots ctx_i + j (j = local
 *   row, row 0 = the root) before sv_tree_attend; blocks holding staged
 *   slots must not be shared with another request.
 * Supported: block_size 16, head_dim 64 or 128, n_q_heads / n_kv_heads <= 16. */
typedef struct {
  void* k_cache;
  void* v_cache;
  int32_t num_blocks;
  int32_t block_size;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t* block_tables;
  int32_t max_blocks_per_req;
  int32_t* cache_lens;
} sv_paged_kv;

/* A batch of draft chains / trees, packed without padding ([SwiftSpec]
 * mechanism 3; [FASER] mechanism 1: every request has its own number of
 * drafts).
 * cu_rows: int32 [n_req + 1], exclusive prefix of rows_i (rows_i >= 1:
 *   row 0 is the root, the last committed token; rows 1.. are draft nodes).
 * parent: int32 [total_rows], LOCAL parent index; -1 at row 0, else in
 *   [0, j) (topological order).  A chain has parent[j] = j - 1.
 * tokens: int32 [total_rows], the token of every node.
 * max_rows_per_req: an upper bound of rows_i, at most 128.
 * verify_len (nullable) [n_req]: verify only drafts 1..verify_len[i]; the
 *   chain ends at row lim_i = min(rows_i, verify_len[i] + 1).  NULL: lim_i =
 *   rows_i.  ([DSpark] hardware-aware prefix scheduler: only the selected
 *   prefix is verified.)
 * row_begin, row_end (nullable) [n_req]: the window of rows handled by this
 *   call, 0 <= row_begin <= row_end <= rows_i, clipped to lim_i; NULL =
 *   [0, lim_i).  An empty window leaves the request untouched.  ([FASER]
 *   mechanism 2: verification in chunks.)  Trees are verified whole. */
typedef struct {
  int32_t n_req;
  int32_t total_rows;
  int32_t max_rows_per_req;
  const int32_t* cu_rows;
  const int32_t* parent;
  const int32_t* tokens;
  const int32_t* row_begin;
  const int32_t* row_end;
  const int32_t* verify_len;
} sv_batch;

/* Free-block pool: free_list int32 [capacity], *free_count (device int32) =
 * number of valid entries at the front. */
typedef struct {
  int32_t* free_list;
  int32_t* free_count;
  int32_t capacity;
} sv_block_pool;

const char* sv_status_string(sv_status s);
const char* sv_version(void);

/* ---------------------------------------------------------------- attend --
 * For every row r of every request inside its window and every query head h,
 *   out[r][h] = sum_k softmax_k(softmax_scale * q[r][h] . K_k) V_k
 * with K, V of KV head h / (n_q_heads / n_kv_heads), over the keys
 *   {cache slots 0 .. ctx_i - 1}  U  {staged slot ctx_i + m : m is an
 *   ancestor of r or r itself}.
 * ([SwiftSpec] mechanism 2: each node's unique prefix; mechanism 3: all
 * draft rows of a request in one padding-free call; [FASER] operations
 * notes: the kernel runs on a chunk of rows.)
 * q: bf16 [total_rows][n_q_heads][head_dim]; out: bf16, same shape.  Rows
 * outside the windows are not written.  Accumulation in fp32.
 * ws: device workspace of at least sv_tree_attend_workspace() bytes,
 * 256-byte aligned, contents need not be initialised. */
size_t sv_tree_attend_workspace(const sv_batch* batch, const sv_paged_kv* kv, int32_t n_q_heads);
sv_status sv_tree_attend(const sv_paged_kv* kv, const sv_batch* batch, const void* q,
                         int32_t n_q_heads, float softmax_scale, void* out, void* ws,
                         size_t ws_bytes, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- accept --
 * Lossless verification ([DSpark] glossary: the longest matching prefix is
 * accepted and the target distribution is preserved).  A logits row r
 * belongs to node r: target row r is p(. | path to r), draft row r the q that
 * proposed r's children.  x = logits / temperature, divided in fp32.
 *   temperature > 0 (chains): for drafts j = 1, 2, ... whose parent row lies
 *     in the window, accept x_j iff u(i, j) < min(1, p_{j-1}(x_j) /
 *     q_{j-1}(x_j)); at the first rejection emit a token drawn from
 *     normalize(max(0, p_{j-1} - q_{j-1})); if every draft up to lim_i - 1
 *     is accepted emit a token drawn from p_{lim_i - 1}.
 *   temperature > 0 (trees, one window over all rows; siblings drawn
 *     independently from the parent's q): from the root, children are tried
 *     in index order; child c (token x) is accepted iff u(i, c) <
 *     min(1, p'(x) / q_n(x)), p' the target distribution left by the
 *     siblings rejected before it: after j rejections p' = max(0, p_n -
 *     c_j q_n) / S(c_j), S(c) = sum_v max(0, p_n,v - c q_n,v), c_0 = 0,
 *     c_{j+1} = c_j + S(c_j).  On acceptance the walk moves to c; when every
 *     child is rejected the emitted token is drawn from p' (from p_n if S
 *     vanished); at a leaf it is drawn from p_leaf.  (Tree verification is
 *     on the pages; this multi-candidate rejection rule is the plainest
 *     lossless reading.)
 *   temperature == 0 (chains and trees): keep the longest root-to-node path
 *     along which each node's token is the target argmax (lowest index on
 *     ties) of its parent row; among equally long paths the one whose first
 *     differing node has the lower index; emit the argmax of the last node.
 * Randomness: Philox4x32-10 keyed by seed (key = low, high 32 bits).
 *   u(i, j): counter (j, i, 0, 0), word 0, top 24 bits * 2^-24.
 *   Residual / bonus draws are exponential races: the token is
 *   argmax_v w_v / E_v, E_v = -log U_v, U_v from counter (v/4, i, 1, pos)
 *   word v%4, ((bits >> 9) + 0.5) * 2^-23; pos = position of the emitted
 *   token, accepted drafts + 1 (j after rejecting draft j, lim_i after the
 *   last draft of a chain).
 * Outputs (state kept across the windows of one step):
 *   accepted_len [n_req]: accepted drafts a_i;
 *   accepted_nodes [n_req][max_rows_per_req]: path, [0] = 0 (root), then the
 *     accepted nodes; -1 past the end;
 *   next_token [n_req]: emitted token, -1 while undecided;
 *   ambiguous u8 [n_req]: set when some |u - min(1, p/q)| < 1e-6;
 *   done (nullable) [n_req]: 1 once next_token is decided;
 *   row_stats (nullable) fp32 [total_rows][4]: temperature > 0: [0] log-sum-
 *     exp of target row x, [1] of the draft row, [2] p and [3] q of the
 *     row's own token under its parent's rows; temperature == 0: [0] max
 *     target logit, [1] argmax.
 * A window starting at row 0 resets the request's state; a later window
 * continues it (requests already decided are skipped).
 * target_logits, draft_logits: fp32 [total_rows][vocab]; draft_logits may be
 * NULL when temperature == 0.
 * ws: at least sv_accept_workspace() bytes, 256-byte aligned. */
size_t sv_accept_workspace(const sv_batch* batch, int32_t vocab);
sv_status sv_accept(const sv_batch* batch, const float* target_logits, const float* draft_logits,
                    int32_t vocab, float temperature, uint64_t seed, int32_t* accepted_len,
                    int32_t* accepted_nodes, int32_t* next_token, uint8_t* ambiguous,
                    int32_t* done, float* row_stats, void* ws, size_t ws_bytes,
                    int32_t* dev_status, void* stream);

/* ------------------------------------------------- accept + commit fused --
 * [SwiftSpec] mechanism 3 (the verification result and the KV update fused
 * into one operation).  sv_accept_commit computes exactly what sv_accept
 * followed by sv_commit_kv computes (same arguments as each, same results,
 * same free-list order), but the warp that decides a request's path also
 * moves its K/V and sets its new length, and the last request to finish
 * appends every released block to the pool: no separate commit launches,
 * no second read of accepted_len / accepted_nodes.  One-pass calls only
 * (windows covering whole requests, as for sv_commit_kv).
 * ws: at least sv_accept_commit_workspace() bytes, 256-byte aligned. */
size_t sv_accept_commit_workspace(const sv_batch* batch, int32_t vocab);
sv_status sv_accept_commit(const sv_batch* batch, const float* target_logits,
                           const float* draft_logits, int32_t vocab, float temperature,
                           uint64_t seed, int32_t* accepted_len, int32_t* accepted_nodes,
                           int32_t* next_token, uint8_t* ambiguous, int32_t* done,
                           float* row_stats, const sv_paged_kv* kv, const sv_block_pool* pool,
                           void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------ accept without workspace --
 * No counterpart in the paper: a convenience for callers that cannot
 * allocate device memory -- for example a plugin inside another runtime that
 * is handed only its input and output buffers, or a serving engine that has
 * already reserved nearly all HBM for its KV-cache pool, or a latency-critical
 * loop that cannot afford cudaMalloc's implicit device synchronisation.
 * sv_accept_static computes exactly what sv_accept computes (same arguments,
 * same outputs) but takes its scratch from a device array of
 * SV_ACCEPT_STATIC_SCRATCH_BYTES inside the library instead of a caller
 * workspace; it calls no allocator.  That array exists once per GPU that
 * loads the library and is held until the process exits.
 * Limits and behaviour:
 *   - Problems whose sv_accept_workspace() exceeds
 *     SV_ACCEPT_STATIC_SCRATCH_BYTES (4 MiB; any batch of up to 40,000
 *     packed rows fits) are refused with SV_ERR_WORKSPACE_TOO_SMALL before
 *     anything is enqueued; use sv_accept with a workspace beyond that.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address once; make that first call before any stream
 *     capture begins.  The address is kept for the life of the process: a
 *     device reset (cudaDeviceReset) ends the context it belongs to, so do
 *     not call sv_accept_static on a device after resetting it.
 *   - Every call shares the one array: calls whose work overlaps on the GPU
 *     (for instance on two streams) race on it and must be ordered by the
 *     caller. */
#define SV_ACCEPT_STATIC_SCRATCH_BYTES (4u << 20)
sv_status sv_accept_static(const sv_batch* batch, const float* target_logits,
                           const float* draft_logits, int32_t vocab, float temperature,
                           uint64_t seed, int32_t* accepted_len, int32_t* accepted_nodes,
                           int32_t* next_token, uint8_t* ambiguous, int32_t* done,
                           float* row_stats, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- commit --
 * [SwiftSpec] mechanism 2: keep only the accepted path's KV, free rejected
 * paths.  For request i with a = accepted_len[i], path = accepted_nodes[i]:
 * slot ctx_i + k <- staged slot ctx_i + path[k] for k = 0..a (all KV heads;
 * every source is read before any destination is written); cache_lens[i] =
 * ctx_i + 1 + a; blocks at table index ceil(new_len / 16) ..
 * ceil((ctx_i + rows_i) / 16) - 1 are appended to the free list in (request,
 * table index) order and their table entries set to -1.  Invalid paths
 * (path[0] != 0, not increasing, a > rows_i - 1) set SV_DEV_BAD_WINDOW and
 * the request is left as it was.  Row windows and verify_len are ignored. */
sv_status sv_commit_kv(const sv_paged_kv* kv, const sv_batch* batch, const int32_t* accepted_len,
                       const int32_t* accepted_nodes, const sv_block_pool* pool,
                       int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------- budget --
 * [DSpark] hardware-aware prefix scheduler: S_{i,k} = c_{i,1} ... c_{i,k}
 * (fp32, left to right) for k = 1..gamma_i; all candidates sorted by key
 * (~bits(S)) << 32 | (i * gamma_max + k - 1) ascending (S descending, then
 * lower request, then lower position); with m admitted, B = n_req + m and
 * tau_fx = n_req * 2^40 + sum trunc(S * 2^40) over the admitted (u64);
 * Theta(m) = double(tau_fx) * 2^-40 * double(sps[B]); the smallest m
 * maximising Theta over 0 <= m <= min(sum gamma_i, b_max - n_req) is chosen.
 * cond_survival: fp32 [n_req][gamma_max] in [0, 1]; gamma (nullable) int32
 * [n_req] in [0, gamma_max] (NULL = gamma_max for all); sps fp32 [b_max+1].
 * Outputs: verify_len [n_req] (drafts admitted per request, ready for
 * sv_batch.verify_len), *best_B (int32), *best_theta (double).
 * Supported: n_req * gamma_max <= 8192, b_max >= n_req.  One CTA, all in
 * shared memory;
 * ws: at least sv_select_budget_workspace() bytes. */
size_t sv_select_budget_workspace(int32_t n_req, int32_t gamma_max);
sv_status sv_select_budget(int32_t n_req, int32_t gamma_max, const float* cond_survival,
                           const int32_t* gamma, const float* sps, int32_t b_max,
                           int32_t* verify_len, int32_t* best_B, double* best_theta, void* ws,
                           size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------- chunked pruning --
 * [FASER] mechanism 2 (early token pruning).  sv_chunk_windows writes the
 * window of chunk `chunk_index` for every request:
 *   [c * chunk_size, min((c + 1) * chunk_size, lim_i)) if done[i] == 0 (or
 *   c == 0), else an empty window; done may be NULL only for c == 0.
 * sv_verify_chunked runs the whole chunked step on `stream` with no host
 * synchronisation: for c = 0 .. ceil(max_rows_per_req / chunk_size) - 1,
 * windows -> sv_tree_attend -> sv_accept on the window rows; requests that
 * met a rejection or emitted their bonus token stop being attended and
 * tested.  batch->row_begin / row_end are ignored (the call uses its own);
 * done [n_req] is required.  Results equal one-pass verification: the
 * uniforms are keyed by position.  A draft tree is verified whole in the
 * first chunk, so it needs chunk_size >= its rows (a tree cut by a chunk
 * boundary sets SV_DEV_BAD_WINDOW and gets no result).
 * ws: sv_verify_chunked_workspace() (the same size serves
 * sv_verify_chunked_commit).
 * sv_verify_chunked_commit: the same step with [SwiftSpec] mechanisms 2-3
 * fused in -- it computes exactly what sv_verify_chunked followed by
 * sv_commit_kv(kv, batch, accepted_len, accepted_nodes, pool) computes
 * (same K/V moves, cache lengths, free list and its order), but each request
 * is committed by the decision that stops it, in that chunk's kernels, and
 * the last request to stop appends every released block to the pool.  A
 * stopped request is never attended again, so moving its K/V mid-step
 * changes nothing the later chunks read.  Requests whose window is invalid
 * are left as they were; one whose parents or tokens are invalid is flagged,
 * stops (done = 1) and is left as it was.  pool is required and kv must meet
 * the commit's rules (16-token blocks, head_dim 64 or 128, K and V caches
 * 16-byte aligned): else SV_ERR_INVALID_ARGUMENT / SV_ERR_UNSUPPORTED_SHAPE
 * before anything is enqueued. */
sv_status sv_chunk_windows(const sv_batch* batch, int32_t chunk_index, int32_t chunk_size,
                           const int32_t* done, int32_t* row_begin, int32_t* row_end,
                           void* stream);
size_t sv_verify_chunked_workspace(const sv_batch* batch, const sv_paged_kv* kv,
                                   int32_t n_q_heads, int32_t vocab);
sv_status sv_verify_chunked(const sv_paged_kv* kv, const sv_batch* batch, const void* q,
                            int32_t n_q_heads, float softmax_scale, void* out,
                            const float* target_logits, const float* draft_logits,
                            int32_t vocab, float temperature, uint64_t seed, int32_t chunk_size,
                            int32_t* accepted_len, int32_t* accepted_nodes, int32_t* next_token,
                            uint8_t* ambiguous, int32_t* done, void* ws, size_t ws_bytes,
                            int32_t* dev_status, void* stream);
sv_status sv_verify_chunked_commit(const sv_paged_kv* kv, const sv_batch* batch, const void* q,
                                   int32_t n_q_heads, float softmax_scale, void* out,
                                   const float* target_logits, const float* draft_logits,
                                   int32_t vocab, float temperature, uint64_t seed,
                                   int32_t chunk_size, int32_t* accepted_len,
                                   int32_t* accepted_nodes, int32_t* next_token,
                                   uint8_t* ambiguous, int32_t* done, const sv_block_pool* pool,
                                   void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* ------------------------------------------------------ chunk size --
 * [FASER] mechanism 2 (verification in chunks; requests leave at their
 * first rejection) and its remark that the chunk size follows the load.  The
 * pages give no rule; this one is fixed here exactly.  For request i with
 * rows_i verified rows (1 + drafts, at most 128), ctx_i cached tokens and the
 * draft-length controller's state (S_i, N_i) (sv_adapt_gamma):
 *   a_i = min(1, (S_i + 1) / (N_i + 2))  (acceptance estimate);
 *   for a chunk size c = 1 .. max_rows (max_rows = max_i rows_i), chunk k
 *   covers rows [b, e) = [k c, min((k+1) c, rows_i)), which request i reaches
 *   when drafts 1 .. k c were all accepted: P_ik = a_i^(k c), computed as
 *   P_i0 = 1, P_i,k+1 = P_ik * a_i^c with a_i^c by c multiplications;
 *   bytes_ik = (ctx_i + e) * kv_bytes + (e - b) * row_bytes (context KV is
 *   read again by every chunk, logits once per row);
 *   cost(c) = ceil(max_rows / c) * chunk_bytes
 *             + sum over i and k of trunc(P_ik * bytes_ik)   (u64),
 *   chunk_bytes being one chunk's fixed cost (its launches and latency
 *   chains) in bytes of HBM time.  Every fp64 operation is rounded on its
 *   own (no fused multiply-add).
 * Outputs: *chunk = the size of least cost (the larger on ties), *cost its
 * cost, costs [128]: cost(c) at c - 1 (UINT64_MAX past max_rows).  A chunk of
 * max_rows is one-pass verification.  Requests with rows outside [1, 128],
 * ctx < 0 or a state that is not finite and non-negative set
 * SV_DEV_BAD_LENGTH and are left out; with no valid request *chunk = 1 and
 * *cost = 0.  All pointers are device memory.  n_req < 0, negative or
 * infinite byte sizes, or a missing output: SV_ERR_INVALID_ARGUMENT before
 * anything is enqueued. */
sv_status sv_select_chunk(int32_t n_req, const int32_t* rows, const int32_t* ctx,
                          const double* state, double kv_bytes, double row_bytes,
                          uint64_t chunk_bytes, int32_t* chunk, uint64_t* cost, uint64_t* costs,
                          int32_t* dev_status, void* stream);

/* ------------------------------------------ per-request draft length --
 * [FASER] mechanism 1 (per-request speculation length): every request's
 * previous acceptance feeds back into its own gamma -- raised where drafts
 * are accepted, lowered where they are rejected.  The pages give no
 * formula; this controller is one choice, fixed here exactly:
 *   state [n_req][2] fp64 (S, N): decayed counts of accepted drafts and of
 *     trials (zero-initialised by the caller for a new request);
 *   after a step with a_i accepted drafts out of verified_i:
 *     S <- decay * S + a_i;  N <- decay * N + a_i + (a_i < verified_i);
 *   alpha = (S + 1) / (N + 2)   (acceptance estimate, Beta(1, 1) prior);
 *   gamma_next_i = the g in [gamma_min, gamma_max] that maximises
 *     E(g) / (g + 1 + overhead),  E(g) = sum_{k=0..g} alpha^k
 *   (expected tokens emitted per step over the rows it verifies plus a
 *   fixed per-step cost in row units), smallest g on ties.
 * All of it in IEEE fp64 add / multiply / divide in the order written (no
 * contraction), so that any implementation gives the same gamma.
 * verified [n_req]: drafts the step verified for the request (its gamma or
 * verify_len); a request with verified_i < 0 is left untouched.
 * Invalid arguments: 0 <= gamma_min <= gamma_max <= 127, 0 < decay <= 1,
 * overhead >= 0. */
sv_status sv_adapt_gamma(int32_t n_req, const int32_t* accepted_len, const int32_t* verified,
                         double* state, int32_t* gamma_next, double decay, double overhead,
                         int32_t gamma_min, int32_t gamma_max, int32_t* dev_status,
                         void* stream);

/* ------------------------------------------------------------ self test --
 * Every wait inside the library's kernels (on an mbarrier a TMA copy or a
 * thread completes) gives up after a bounded number of rounds, sets
 * SV_DEV_TIMEOUT and lets the kernel return, so that a lost copy can never
 * hang the device.  sv_selftest_bounded_wait runs that wait on a barrier
 * nothing will complete (limit rounds, 1 .. 2^20), so the timeout path can be
 * checked on a live GPU: *dev_status gets SV_DEV_TIMEOUT and the context
 * stays usable.  No other effect. */
sv_status sv_selftest_bounded_wait(int32_t limit, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* LIBSPECVERIFY_H */
