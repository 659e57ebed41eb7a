// commit.cu — sv_commit_kv: keep the accepted path's K/V, free the rest.
//
// Source: [SwiftSpec] core design, mechanism 2 (tree-aware KV cache
// management: only the KV of the accepted path is kept and rejected paths
// are released at once) and mechanism 3 (verification result and KV update
// as one fused step).
//
// Two kernels:
//   copy    (1 CTA per request) moves staged slot ctx + path[k] to slot
//           ctx + k, head by head, reading every source of the head into
//           shared memory before writing any destination (sources and
//           destinations of one request can overlap).  Slots with
//           path[k] == k (every chain) are not moved.
//   release (1 CTA) counts the blocks past the new length of every request,
//           scans the counts and appends them to the free list in (request,
//           table index) order, clears their table entries and sets the new
//           cache length.

#include <mutex>

#include "sv_internal.cuh"

namespace sv {
namespace cmt {

struct Args {
  sv_batch bt;
  __nv_bfloat16* k;
  __nv_bfloat16* v;
  int num_blocks, Hkv, D, max_blocks;
  int32_t* tables;
  int32_t* cache_lens;
  const int32_t* accepted_len;
  const int32_t* accepted_nodes;
  int32_t* free_list;
  int32_t* free_count;
  int capacity;
  int32_t* dev_status;
};

// Same validity rule in both kernels: a request failing it is left as it was.
__device__ bool request_ok(const Args& a, int i, int& rows, int& ctx, int& al, bool report) {
  rows = a.bt.cu_rows[i + 1] - a.bt.cu_rows[i];
  ctx = a.cache_lens[i];
  al = a.accepted_len[i];
  const int32_t* path = a.accepted_nodes + (size_t)i * a.bt.max_rows_per_req;
  if (rows < 1 || rows > a.bt.max_rows_per_req || al < 0 || al > rows - 1 || path[0] != 0) {
    if (report) flag(a.dev_status, SV_DEV_BAD_WINDOW);
    return false;
  }
  for (int k = 1; k <= al; ++k) {
    if (path[k] <= path[k - 1] || path[k] >= rows) {
      if (report) flag(a.dev_status, SV_DEV_BAD_WINDOW);
      return false;
    }
  }
  if (ctx < 0 || (long)ctx + rows > (long)a.max_blocks * kBlockSize) {
    if (report) flag(a.dev_status, SV_DEV_BAD_LENGTH);
    return false;
  }
  const int32_t* table = a.tables + (size_t)i * a.max_blocks;
  for (int k = 0; k <= al; ++k) {
    const int b1 = table[(ctx + path[k]) / kBlockSize];
    const int b2 = table[(ctx + k) / kBlockSize];
    if (b1 < 0 || b1 >= a.num_blocks || b2 < 0 || b2 >= a.num_blocks) {
      if (report) flag(a.dev_status, SV_DEV_BAD_BLOCK_ID);
      return false;
    }
  }
  return true;
}

__global__ void __launch_bounds__(256) copy_kernel(Args a) {
  griddep_entry();
  extern __shared__ __align__(16) uint8_t smem_raw[];
  int4* buf = reinterpret_cast<int4*>(smem_raw);
  __shared__ int s_ok, s_moves;
  __shared__ long long s_src[kMaxRows], s_dst[kMaxRows];
  const int i = blockIdx.x;
  if (threadIdx.x == 0) {
    int rows, ctx, al;
    s_ok = request_ok(a, i, rows, ctx, al, true);
    s_moves = 0;
    if (s_ok) {
      const int32_t* path = a.accepted_nodes + (size_t)i * a.bt.max_rows_per_req;
      const int32_t* table = a.tables + (size_t)i * a.max_blocks;
      for (int k = 1; k <= al; ++k) {
        if (path[k] == k) continue;
        const int ss = ctx + path[k], ds = ctx + k;
        // slot addresses as (block * Hkv) * 16 + offset, head added below
        s_src[s_moves] = (long long)table[ss / kBlockSize] * kBlockSize * a.Hkv + (ss % kBlockSize);
        s_dst[s_moves] = (long long)table[ds / kBlockSize] * kBlockSize * a.Hkv + (ds % kBlockSize);
        ++s_moves;
      }
    }
  }
  __syncthreads();
  if (!s_ok || s_moves == 0) return;
  const int n = s_moves;
  const int cpr = a.D / 8;  // int4 per token row of one head
  for (int g = 0; g < a.Hkv; ++g) {
    for (int x = threadIdx.x; x < 2 * n * cpr; x += blockDim.x) {
      const int tensor = x / (n * cpr), rem = x % (n * cpr);
      const int k = rem / cpr, c = rem % cpr;
      const size_t row = (size_t)s_src[k] + (size_t)g * kBlockSize;
      const int4* src = reinterpret_cast<const int4*>((tensor ? a.v : a.k) + row * a.D) + c;
      buf[x] = *src;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < 2 * n * cpr; x += blockDim.x) {
      const int tensor = x / (n * cpr), rem = x % (n * cpr);
      const int k = rem / cpr, c = rem % cpr;
      const size_t row = (size_t)s_dst[k] + (size_t)g * kBlockSize;
      int4* dst = reinterpret_cast<int4*>((tensor ? a.v : a.k) + row * a.D) + c;
      *dst = buf[x];
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(1024) release_kernel(Args a) {
  griddep_entry();
  const int R = a.bt.n_req;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ int s_warp[32];
  __shared__ int s_carry, s_pushed, s_fc0;
  if (tid == 0) {
    s_carry = 0;
    s_pushed = 0;
    s_fc0 = *a.free_count;
  }
  __syncthreads();
  const int fc0 = s_fc0;
  for (int base = 0; base < R; base += blockDim.x) {
    const int i = base + tid;
    int rows = 0, ctx = 0, al = 0, nfree = 0, keep = 0, used = 0;
    bool ok = false;
    int32_t* table = nullptr;
    if (i < R) {
      ok = request_ok(a, i, rows, ctx, al, false);
      if (ok) {
        table = a.tables + (size_t)i * a.max_blocks;
        const int new_len = ctx + 1 + al;
        keep = (new_len + kBlockSize - 1) / kBlockSize;
        used = (ctx + rows + kBlockSize - 1) / kBlockSize;
        for (int t = keep; t < used; ++t) nfree += table[t] >= 0;
      }
    }
    // exclusive scan of nfree over the block
    int x = nfree;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int wv = s_warp[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, wv, o);
        if (lane >= o) wv += y;
      }
      s_warp[lane] = wv;
    }
    __syncthreads();
    const int excl = (warp ? s_warp[warp - 1] : 0) + x - nfree;
    const int total = s_warp[31];
    if (ok) {
      const long start = (long)fc0 + s_carry + excl;
      if (start + nfree <= a.capacity) {
        int n = 0;
        for (int t = keep; t < used; ++t) {
          const int blk = table[t];
          if (blk < 0) continue;
          a.free_list[start + n++] = blk;
          table[t] = -1;
        }
        if (nfree) atomicMax(&s_pushed, (int)(start + nfree - fc0));
      } else {
        flag(a.dev_status, SV_DEV_POOL_OVERFLOW);
      }
      a.cache_lens[i] = ctx + 1 + al;
    }
    __syncthreads();
    if (tid == 0) s_carry += total;
    __syncthreads();
  }
  if (tid == 0) *a.free_count = fc0 + s_pushed;
}

}  // namespace cmt
}  // namespace sv

using namespace sv;

extern "C" sv_status sv_commit_kv(const sv_paged_kv* kv, const sv_batch* bt,
                                  const int32_t* accepted_len, const int32_t* accepted_nodes,
                                  const sv_block_pool* pool, int32_t* dev_status, void* stream) {
  SV_TRACE("sv_commit_kv");
  if (!kv || !bt || !pool) return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req < 0 || bt->max_rows_per_req < 1) return SV_ERR_INVALID_ARGUMENT;
  if (bt->max_rows_per_req > kMaxRows) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->block_size != kBlockSize) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->head_dim != 64 && kv->head_dim != 128) return SV_ERR_UNSUPPORTED_SHAPE;
  if (kv->n_kv_heads < 1 || kv->num_blocks < 0 || kv->max_blocks_per_req < 0)
    return SV_ERR_INVALID_ARGUMENT;
  if (bt->n_req == 0) return SV_OK;
  if (!bt->cu_rows || !accepted_len || !accepted_nodes || !kv->k_cache || !kv->v_cache ||
      !kv->block_tables || !kv->cache_lens || !pool->free_list || !pool->free_count ||
      pool->capacity < 0)
    return SV_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)kv->k_cache | (uintptr_t)kv->v_cache) & 15) return SV_ERR_INVALID_ARGUMENT;
  cmt::Args a;
  a.bt = *bt;
  a.k = static_cast<__nv_bfloat16*>(kv->k_cache);
  a.v = static_cast<__nv_bfloat16*>(kv->v_cache);
  a.num_blocks = kv->num_blocks;
  a.Hkv = kv->n_kv_heads;
  a.D = kv->head_dim;
  a.max_blocks = kv->max_blocks_per_req;
  a.tables = kv->block_tables;
  a.cache_lens = kv->cache_lens;
  a.accepted_len = accepted_len;
  a.accepted_nodes = accepted_nodes;
  a.free_list = pool->free_list;
  a.free_count = pool->free_count;
  a.capacity = pool->capacity;
  a.dev_status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // one head of every moved slot, K and V: 2 * 127 * 128 * 2 B = 65 KB at most
  const size_t smem = (size_t)2 * (bt->max_rows_per_req - 1 > 0 ? bt->max_rows_per_req - 1 : 1) *
                      kv->head_dim * 2;
  if (smem > 48 * 1024) {
    static PerDevice smem_set;
    if (smem_limit_once(smem_set, cmt::copy_kernel, 96 * 1024) != cudaSuccess) return SV_ERR_CUDA;
  }
  if (sv::launch(cmt::copy_kernel, bt->n_req, 256, smem, s, a) != cudaSuccess) return SV_ERR_CUDA;
  if (sv::launch(cmt::release_kernel, 1, 1024, 0, s, a) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}
