// sv_internal.cuh — device helpers shared by the libspecverify kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "libspecverify.h"

namespace sv {

constexpr int kBlockSize = 16;   // tokens per KV page
constexpr int kMaxRows = 128;    // rows per request (ancestor masks are 128 bits)

// Device findings are OR-ed into the caller's status word; a null word drops
// them (the affected request is still skipped).
__device__ __forceinline__ void flag(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

// Index of the request owning packed position x, given an exclusive prefix
// `cu` of length n + 1 (cu[0] = 0): the largest i with cu[i] <= x.
__device__ __forceinline__ int find_segment(const int32_t* cu, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(cu + mid) <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Rows of request i handled by this call: [b, e) inside the chain end lim.
struct Window {
  int rows, lim, b, e;
  int cu;  // first packed row of the request
  bool ok;
};

__device__ __forceinline__ Window window_of(const sv_batch& bt, int i) {
  Window w;
  const int c0 = bt.cu_rows[i], c1 = bt.cu_rows[i + 1];
  w.cu = c0;
  w.rows = c1 - c0;
  w.ok = w.rows >= 1 && w.rows <= bt.max_rows_per_req && w.rows <= kMaxRows && c0 >= 0 &&
         c1 <= bt.total_rows;
  w.lim = w.rows;
  if (bt.verify_len) {
    int L = bt.verify_len[i];
    if (L < 0) w.ok = false;
    if (L + 1 < w.lim) w.lim = L + 1;
  }
  w.b = bt.row_begin ? bt.row_begin[i] : 0;
  w.e = bt.row_end ? bt.row_end[i] : w.lim;
  if (w.b < 0 || w.b > w.e || w.e > w.rows) w.ok = false;
  if (w.e > w.lim) w.e = w.lim;
  return w;
}

// Rows [b, e) of chunk c (chunk size cs) of request i, from a batch given
// without windows: rows c*cs .. c*cs + cs - 1 of the verified range, empty
// once the request is done (done[i] != 0, read only for c > 0) or past its
// rows.  A request whose own window is invalid gets an empty window and
// *bad = true (the caller reports it once, on chunk 0).
__device__ __forceinline__ Window chunk_window(sv_batch bt, int i, int c, int cs,
                                               const int32_t* done, bool* bad) {
  bt.row_begin = nullptr;
  bt.row_end = nullptr;
  Window w = window_of(bt, i);
  int b = c * cs, e = min(b + cs, w.lim);
  const bool running = c == 0 || (done && done[i] == 0);
  *bad = !w.ok;
  if (!w.ok) {
    b = e = 0;
  } else if (!running || b >= e) {
    b = e = min(b, w.rows);
  }
  w.b = b;
  w.e = e;
  w.ok = true;
  return w;
}

// ------------------------------------------------------------- Philox ----
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of
// (c0, c1, c2, c3) -> (hi(B*c2) ^ c1 ^ k0, lo(B*c2), hi(A*c0) ^ c3 ^ k1,
// lo(A*c0)) with A = 0xD2511F53, B = 0xCD9E8D57 and the key advanced by the
// Weyl increments 0x9E3779B9, 0xBB67AE85 between rounds.
struct U4 {
  uint32_t a, b, c, d;
};

__device__ __forceinline__ U4 philox10(U4 x, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t A = 0xD2511F53u, B = 0xCD9E8D57u;
    uint32_t pa_lo = A * x.a, pa_hi = __umulhi(A, x.a);
    uint32_t pb_lo = B * x.c, pb_hi = __umulhi(B, x.c);
    U4 y;
    y.a = pb_hi ^ x.b ^ k0;
    y.b = pb_lo;
    y.c = pa_hi ^ x.d ^ k1;
    y.d = pa_lo;
    x = y;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return x;
}

// Accept uniform of draft j of request i: counter (j, i, 0, 0), word 0,
// top 24 bits.
__device__ __forceinline__ float accept_u(uint64_t seed, int i, int j) {
  U4 c{(uint32_t)j, (uint32_t)i, 0u, 0u};
  U4 o = philox10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
  return (float)(o.a >> 8) * 5.9604644775390625e-08f;  // 2^-24
}

// Race uniforms of the draw at position pos.  The race is among groups of
// four vocabulary entries (group g = entries 4g .. 4g+3); groups are numbered
// in blocks of 128, and group 128 b + 32 k + l takes word k of counter
// (32 b + l, i, 1, pos): race_bits(..., 32 b + l) serves the four groups
// 128 b + l, + 32, + 64, + 96.  ((bits >> 9) + 0.5) * 2^-23 is in (0, 1).
__device__ __forceinline__ U4 race_bits(uint64_t seed, int i, int pos, int ctr) {
  U4 c{(uint32_t)ctr, (uint32_t)i, 1u, (uint32_t)pos};
  return philox10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
}
__device__ __forceinline__ float race_u(uint32_t bits) {
  return ((float)(bits >> 9) + 0.5f) * 1.1920928955078125e-07f;  // 2^-23
}
// The uniform that picks the entry inside the winning group g: word 0 of
// counter (g, i, 2, pos), same conversion.
__device__ __forceinline__ float pick_u(uint64_t seed, int i, int pos, int g) {
  U4 c{(uint32_t)g, (uint32_t)i, 2u, (uint32_t)pos};
  return race_u(philox10(c, (uint32_t)seed, (uint32_t)(seed >> 32)).a);
}

// ------------------------------------------------------ fast arithmetic ----
// x / d for a divisor d shared by many x, with r = 1 / d: the product x * r
// corrected once by the exact residual x - q * d (an fma), after Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor" (IBM J. Res. Dev. 34(1), 1990).  Equal to the correctly rounded
// quotient except in rare cases where it is one ulp away; used only where the
// result feeds a normaliser, never a decision.
__device__ __forceinline__ float div_by(float x, float d, float r) {
  const float q = x * r;
  const float e = fmaf(-q, d, x);
  return fmaf(e, r, q);
}

// 2^x by the hardware approximation (relative error below 2^-22; results
// below 2^-126 flush to zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------- warp utils ----
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// --------------------------------------------------- tensor-core / copies --
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// 16-byte asynchronous global -> shared copy; src_bytes = 0 zero-fills.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------- thread-block clusters --
// Rank of this CTA within its cluster.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster: this thread's earlier memory
// accesses (shared memory included) are visible to the cluster's threads
// after the barrier.  All threads of all the cluster's CTAs must call it.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
// Address in CTA `rank`'s shared memory of this CTA's shared address `a`.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ float2 dsmem_ld2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ double dsmem_ld_f64(uint32_t a) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];\n" : "=d"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ float4 dsmem_ld4(uint32_t a) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(a)
               : "memory");
  return v;
}

// ------------------------------------------------------- TMA / mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
// Order this thread's earlier generic-proxy shared-memory accesses before
// later asynchronous-proxy (TMA) accesses to the same addresses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Make barrier initialisation visible to the asynchronous (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Spin on a phase with an iteration limit; false means the limit was hit.
constexpr int kWaitLimit = 1 << 20;  // try_wait rounds before a wait gives up
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  int limit = kWaitLimit) {
  for (int it = 0; it < limit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// The same wait for a thread with nothing else to do: each try may suspend it
// for up to 50 us while the phase is incomplete, instead of spinning; at
// most 40000 tries (2 s) before it gives up.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint32_t bar, uint32_t parity) {
  for (int it = 0; it < 40000; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(50000u)
        : "memory");
    if (ok) return true;
  }
  return false;
}
// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 1-D bulk copy of `bytes` (a multiple of 16, both addresses 16-byte
// aligned) from global to shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
      ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// --------------------------------------------- programmatic dependent launch --
// Every kernel of the library starts with griddep_entry(): it waits until the
// previous grid in the stream has completed and its writes are visible
// (nothing is read or written before that), then lets the next grid begin
// launching, so that launch latency overlaps the tail of this grid.
__device__ __forceinline__ void griddep_entry() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// ---------------------------------------------------------------- tickets --
// The warp that finishes its part of a shared job publishes its results and
// takes a ticket with a release-acquire add at device scope: the writes it
// made before are visible to whoever takes a later ticket, and the writes
// published before earlier tickets are visible to it.  The taker's lanes then
// order their reads after the ticket with __syncwarp() (lane 0 took it).
__device__ __forceinline__ int ticket_add(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;\n"
               : "=r"(old)
               : "l"(p), "r"(v)
               : "memory");
  return old;
}

// ------------------------------------------------------------ host side --
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Per-device state set up once per device and kept for the process (calls may
// come from several host threads): run(fn) calls fn() for the current device
// the first time it is asked to, under a lock, and remembers success.
class PerDevice {
 public:
  template <class F>
  cudaError_t run(F&& fn) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if ((size_t)dev >= done_.size()) done_.resize((size_t)dev + 1, 0);
    if (done_[(size_t)dev]) return cudaSuccess;
    e = fn(dev);
    if (e == cudaSuccess) done_[(size_t)dev] = 1;
    return e;
  }

 private:
  std::mutex mu_;
  std::vector<char> done_;
};

// Raise a kernel's dynamic shared-memory limit on the current device, once
// per device (`once` is the kernel's own record).
template <typename K>
inline cudaError_t smem_limit_once(PerDevice& once, K kernel, size_t bytes) {
  return once.run([&](int) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  });
}

// Streaming multiprocessors of the current device, queried once per device;
// grids and work splits are sized from it.  0 if the query fails.
inline int num_sms() {
  static std::mutex mu;
  static std::vector<int> sms;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if ((size_t)dev >= sms.size()) sms.resize((size_t)dev + 1, 0);
  if (!sms[(size_t)dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      return 0;
    sms[(size_t)dev] = n;
  }
  return sms[(size_t)dev];
}

// The SM count that sizes workspaces and work splits: the current device's,
// or, for a size query made where no device is visible (nothing can be
// launched then), the count of the GB300 this library is built for.
constexpr int kSmsWithoutDevice = 152;
inline int sizing_sms() {
  const int n = num_sms();
  return n > 0 ? n : kSmsWithoutDevice;
}

// Launch with programmatic stream serialization allowed (see griddep_entry).
template <typename... KArgs, typename... Args>
inline cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with thread-block clusters of `cluster` CTAs along x (grid.x a
// multiple of it): the CTAs of a cluster run at once on one GPC and reach
// one another's shared memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t stream, int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// How many clusters of `cluster` CTAs (1 .. 16) of a kernel (`threads` per
// CTA, `smem` bytes of dynamic shared memory) can be resident at once on the
// current device, asked once per device and cluster size; 0 if none fits or
// the query is refused.  Sizes above the portable eight are opted into first.
class ClusterFit {
 public:
  template <class K>
  int get(K kernel, int cluster, int threads, size_t smem) {
    int dev = -1;
    if (cluster < 1 || cluster > 16) return 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    std::lock_guard<std::mutex> lock(mu_);
    const size_t key = (size_t)dev * 17 + (size_t)cluster;
    if (key >= cap_.size()) cap_.resize(key + 1, -1);
    if (cap_[key] < 0) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)cluster);
      cfg.blockDim = dim3((unsigned)threads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at;
      at.id = cudaLaunchAttributeClusterDimension;
      at.val.clusterDim.x = (unsigned)cluster;
      at.val.clusterDim.y = 1;
      at.val.clusterDim.z = 1;
      cfg.attrs = &at;
      cfg.numAttrs = 1;
      int n = 0;
      bool ok = true;
      if (smem > 48 * 1024)
        ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem) == cudaSuccess;
      if (ok && cluster > 8)
        ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
             cudaSuccess;
      ok = ok && cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess;
      if (!ok) {
        (void)cudaGetLastError();  // a refused query is an answer, not an error
        n = 0;
      }
      cap_[key] = n;
    }
    return cap_[key];
  }

 private:
  std::mutex mu_;
  std::vector<int> cap_;  // per (device, cluster size): -1 not asked
};

// A named NVTX range around the host part of a call (what it enqueues), so
// that profilers group the call's kernels under the call's name.
class TraceRange {
 public:
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace sv

#define SV_TRACE(name) ::sv::TraceRange sv_trace_range_(name)

#define SV_LAUNCH_CHECK()                                  \
  do {                                                     \
    if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA; \
  } while (0)
