// budget.cu — sv_select_budget: confidence-sorted verification budget.
//
// Source: [DSpark] "하드웨어 인식 Prefix 스케줄러" (hardware-aware prefix
// scheduler: verification length chosen as a global throughput maximisation
// of expected accepted tokens times the profiled engine throughput SPS(B)),
// "방법론" (all (request, position) candidates sorted by cumulative survival,
// descending; the batch grows one candidate at a time and Theta = tau * SPS(B)
// is maximised), "기술 상세" (SPS(B) stored as a cost table) and the glossary
// (prefix survival = product of the per-position conditional survivals).
//
// One CTA of 1024 threads:
//   1. S_{i,k} = c_{i,1} * ... * c_{i,k} (fp32, left to right); sort key
//      ~bits(S) (S is non-negative, so the bits order like the values; -0 is
//      keyed as +0).
//   2. Stable LSD radix sort of the 32-bit keys, 8-bit digits, 4 passes,
//      in shared memory; candidates enter in (request, position) order, so
//      equal S keep the lower request, then the lower position.  Ranking
//      inside a pass: per-warp digit groups from __match_any_sync, per-digit
//      warp offsets by a scan over warps, tile by tile.
//   3. tau in fixed point (2^-40 units, each S truncated) by a block scan,
//      Theta(m) = double(tau) * 2^-40 * double(SPS(R + m)), block argmax with
//      the smallest m on ties; verify_len counted from the admitted prefix.

#include <math.h>

#include "sv_internal.cuh"

namespace sv {
namespace bud {

constexpr int kMaxCand = 8192;
constexpr int kThreads = 1024;

struct Args {
  int R, gmax, b_max;
  const float* c;
  const int32_t* gamma;
  const float* sps;
  int32_t* verify_len;
  int32_t* best_B;
  double* best_theta;
  int32_t* dev_status;
};

inline size_t smem_bytes() { return (size_t)4 * kMaxCand * 4 + (size_t)32 * 256 * 4; }

__device__ __forceinline__ int block_scan_excl(int* s_warp, int v, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int excl = (warp ? s_warp[warp - 1] : 0) + x - v;
  total = s_warp[31];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(kThreads) budget_kernel(Args a) {
  griddep_entry();
  extern __shared__ __align__(16) uint32_t sm[];
  uint32_t* kA = sm;
  uint32_t* vA = kA + kMaxCand;
  uint32_t* kB = vA + kMaxCand;
  uint32_t* vB = kB + kMaxCand;
  int* wcount = reinterpret_cast<int*>(vB + kMaxCand);  // [32 warps][256 digits]
  __shared__ int hist[256], ttot[256];
  __shared__ int s_warp[32];
  __shared__ int s_carry, s_bad;
  __shared__ unsigned long long s_warp64[32];
  __shared__ double s_th[32];
  __shared__ int s_m[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = a.R, gmax = a.gmax;
  if (tid == 0) {
    s_carry = 0;
    s_bad = 0;
  }
  __syncthreads();

  // 1. survival products and keys, in (request, position) order
  for (int base = 0; base < R; base += kThreads) {
    const int i = base + tid;
    int gi = 0;
    if (i < R) {
      gi = a.gamma ? a.gamma[i] : gmax;
      if (gi < 0 || gi > gmax) {
        s_bad = 1;
        gi = 0;
      }
    }
    int total;
    const int excl = block_scan_excl(s_warp, gi, total);
    if (i < R) {
      float s = 1.0f;
      for (int k = 1; k <= gi; ++k) {
        const float ck = a.c[(size_t)i * gmax + k - 1];
        if (!(ck >= 0.0f && ck <= 1.0f)) s_bad = 1;
        s = s * ck;
        const int idx = s_carry + excl + k - 1;
        if (idx < kMaxCand) {
          // a survival of -0 (a factor c = -0) is the value 0: its key is +0's
          const uint32_t sb = __float_as_uint(s);
          kA[idx] = ~(sb == 0x80000000u ? 0u : sb);
          vA[idx] = (uint32_t)(i * gmax + k - 1);
        }
      }
    }
    __syncthreads();
    if (tid == 0) s_carry += total;
    __syncthreads();
  }
  const int n = s_carry;
  if (s_bad || n > kMaxCand) {
    for (int i = tid; i < R; i += kThreads) a.verify_len[i] = 0;
    if (tid == 0) {
      flag(a.dev_status, SV_DEV_BAD_WINDOW);
      *a.best_B = R;
      *a.best_theta = nan("");
    }
    return;
  }

  // 2. stable LSD radix sort, 4 x 8 bits
  uint32_t *kin = kA, *vin = vA, *kout = kB, *vout = vB;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 8 * pass;
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    for (int e = tid; e < n; e += kThreads) atomicAdd(&hist[(kin[e] >> shift) & 255u], 1);
    __syncthreads();
    if (warp == 0) {
      // exclusive scan of the 256 digit counts: eight per lane, then the warp
      int v[8], sum = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = hist[lane * 8 + j];
        sum += v[j];
      }
      int x = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      int run = x - sum;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        hist[lane * 8 + j] = run;
        run += v[j];
      }
    }
    __syncthreads();
    for (int t0 = 0; t0 < n; t0 += kThreads) {
      const int e = t0 + tid;
      const bool valid = e < n;
      const int d = valid ? (int)((kin[e] >> shift) & 255u) : 256;
      for (int x = tid; x < 32 * 256; x += kThreads) wcount[x] = 0;
      __syncthreads();
      const unsigned peers = __match_any_sync(0xffffffffu, d);
      const int rank = __popc(peers & ((1u << lane) - 1u));
      if (valid && rank == 0) wcount[warp * 256 + d] = __popc(peers);
      __syncthreads();
      if (tid < 256) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
          const int cnt = wcount[w * 256 + tid];
          wcount[w * 256 + tid] = run;
          run += cnt;
        }
        ttot[tid] = run;
      }
      __syncthreads();
      if (valid) {
        const int pos = hist[d] + wcount[warp * 256 + d] + rank;
        kout[pos] = kin[e];
        vout[pos] = vin[e];
      }
      __syncthreads();
      if (tid < 256) hist[tid] += ttot[tid];
      __syncthreads();
    }
    uint32_t* t = kin; kin = kout; kout = t;
    t = vin; vin = vout; vout = t;
  }

  // 3. fixed-point tau, Theta(m), argmax
  const int m_hi = min(n, a.b_max - R);
  const int per = (n + kThreads - 1) / kThreads;
  const int e0 = min(n, tid * per), e1 = min(n, e0 + per);
  unsigned long long local = 0ull;
  for (int e = e0; e < e1; ++e) {
    const float S = __uint_as_float(~kin[e]);
    local += __float2ull_rz(S * 0x1p40f);  // trunc(S * 2^40): the product is exact in fp32
  }
  unsigned long long x = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp64[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long w = s_warp64[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    s_warp64[lane] = w;
  }
  __syncthreads();
  unsigned long long run = (warp ? s_warp64[warp - 1] : 0ull) + x - local;
  const unsigned long long tau0 = (unsigned long long)R << 40;
  double best = -INFINITY;
  int bm = 0x7fffffff;
  if (tid == 0) {
    best = (double)tau0 * 0x1p-40 * (double)a.sps[R];
    bm = 0;
  }
  for (int e = e0; e < e1; ++e) {
    const float S = __uint_as_float(~kin[e]);
    run += __float2ull_rz(S * 0x1p40f);
    const int m = e + 1;
    if (m > m_hi) break;
    const double th = (double)(tau0 + run) * 0x1p-40 * (double)a.sps[R + m];
    if (th > best) {
      best = th;
      bm = m;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const double b2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int m2 = __shfl_xor_sync(0xffffffffu, bm, o);
    if (b2 > best || (b2 == best && m2 < bm)) { best = b2; bm = m2; }
  }
  if (lane == 0) { s_th[warp] = best; s_m[warp] = bm; }
  for (int i = tid; i < R; i += kThreads) a.verify_len[i] = 0;
  __syncthreads();
  if (warp == 0) {
    best = s_th[lane];
    bm = s_m[lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const double b2 = __shfl_xor_sync(0xffffffffu, best, o);
      const int m2 = __shfl_xor_sync(0xffffffffu, bm, o);
      if (b2 > best || (b2 == best && m2 < bm)) { best = b2; bm = m2; }
    }
    if (lane == 0) { s_th[0] = best; s_m[0] = bm; }
  }
  __syncthreads();
  const int mstar = s_m[0];
  for (int t = tid; t < mstar; t += kThreads) atomicAdd(&a.verify_len[vin[t] / (uint32_t)gmax], 1);
  if (tid == 0) {
    *a.best_B = R + mstar;
    *a.best_theta = s_th[0];
  }
}

}  // namespace bud
}  // namespace sv

using namespace sv;

extern "C" size_t sv_select_budget_workspace(int32_t n_req, int32_t gamma_max) {
  (void)n_req;
  (void)gamma_max;
  return 0;  // everything lives in shared memory
}

extern "C" sv_status sv_select_budget(int32_t n_req, int32_t gamma_max, const float* cond_survival,
                                      const int32_t* gamma, const float* sps, int32_t b_max,
                                      int32_t* verify_len, int32_t* best_B, double* best_theta,
                                      void* ws, size_t ws_bytes, int32_t* dev_status,
                                      void* stream) {
  SV_TRACE("sv_select_budget");
  (void)ws;
  (void)ws_bytes;
  if (n_req < 1 || gamma_max < 0 || b_max < n_req) return SV_ERR_INVALID_ARGUMENT;
  if ((long)n_req * (gamma_max > 0 ? gamma_max : 1) > bud::kMaxCand) return SV_ERR_UNSUPPORTED_SHAPE;
  if ((gamma_max > 0 && !cond_survival) || !sps || !verify_len || !best_B || !best_theta)
    return SV_ERR_INVALID_ARGUMENT;
  bud::Args a{n_req, gamma_max, b_max, cond_survival, gamma, sps, verify_len, best_B, best_theta,
              dev_status};
  const size_t smem = bud::smem_bytes();
  static PerDevice smem_set;  // the keys live in 160 KB of shared memory
  if (smem_limit_once(smem_set, bud::budget_kernel, smem) != cudaSuccess) return SV_ERR_CUDA;
  if (sv::launch(bud::budget_kernel, 1, bud::kThreads, smem, static_cast<cudaStream_t>(stream), a) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}
