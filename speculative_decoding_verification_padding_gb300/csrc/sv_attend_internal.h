// sv_attend_internal.h — the attention call as the chunk driver uses it
// (host-side; not part of the public C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "libspecverify.h"

namespace sv {
namespace attn {

// Chunk mode: the planner derives chunk `index`'s windows from the batch
// (given without windows) and `done`, writes them to row_begin / row_end for
// the accept kernels, and lists the requests whose window is not empty (in
// request order, count at act[n_req]) with their row ranges in act4.
struct ChunkPlan {
  int index;            // < 0: not chunked, the batch's own windows are used
  int size;             // rows per chunk
  const int32_t* done;  // [R] requests already decided (read for index > 0)
  int32_t* row_begin;   // [R] out
  int32_t* row_end;     // [R] out
  int32_t* act;         // [R + 1] out
  int4* act4;           // [R] out: per listed request (request, first window row
                        //   in the packed rows, window rows, rows with a tested child)
};

sv_status tree_attend(const sv_paged_kv* kv, const sv_batch* bt, const void* q, int32_t n_q_heads,
                      float softmax_scale, void* out, void* ws, size_t ws_bytes,
                      int32_t* dev_status, cudaStream_t stream, const ChunkPlan& chunk);

}  // namespace attn
}  // namespace sv
