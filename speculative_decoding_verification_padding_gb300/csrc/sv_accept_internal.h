// sv_accept_internal.h — accept entry points shared by accept.cu and the
// chunk driver (host-side; not part of the public C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "libspecverify.h"

namespace sv {
namespace acc {

// Workspace of the accept kernels for a batch whose windows hold at most
// `maxw` rows per request.
// nch / nch_r: vocabulary slices per row (statistics) and per request
// (race) when every listed request is active; the kernels use more slices,
// up to nch_cap / nch_r_cap, when fewer requests are active.
struct Layout {
  size_t parts, jobs, race, race_tickets, act, ctick, cspan, total;
  int nch, nch_cap, nch_r, nch_r_cap, maxw;
  int nsm;  // SMs of the device the call runs on
};
Layout layout(int R, int total_rows, int V, int maxw, bool commit = false);

// The accept kernels.  chunk_index < 0: statistics, decision and race over
// every request.  chunk_index >= 0 (chunk of a chunked step): the active
// list in `ws` (at Layout::act) was written by the attention planner for this
// batch's windows; statistics (the first chunk also clears every sampling
// job) and decision only, the draws are left to race_all.
sv_status run(const sv_batch* bt, const float* target_logits, const float* draft_logits,
              int32_t vocab, float temperature, uint64_t seed, int32_t* accepted_len,
              int32_t* accepted_nodes, int32_t* next_token, uint8_t* ambiguous, int32_t* done,
              float* row_stats, void* ws, size_t ws_bytes, int32_t* dev_status, cudaStream_t s,
              int maxw, int chunk_index, const sv_paged_kv* commit_kv = nullptr,
              const sv_block_pool* commit_pool = nullptr, const int4* act4 = nullptr);

// After the last chunk of a chunked step (T > 0): the residual or bonus draw
// of every request whose decision set one, in a single pass.
sv_status race_all(const sv_batch* bt, const float* target_logits, const float* draft_logits,
                   int32_t vocab, float temperature, uint64_t seed, int32_t* next_token, void* ws,
                   int maxw, int32_t* dev_status, cudaStream_t s);

}  // namespace acc
}  // namespace sv
