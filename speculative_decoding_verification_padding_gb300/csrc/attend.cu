// attend.cu — sv_tree_attend: padding-free verification attention of draft
// chains / trees against a paged bf16 GQA KV cache.
//
// Sources: [SwiftSpec] core design, mechanism 2 (every tree node has its own
// KV prefix) and mechanism 3 (one padding-free attention call verifies all
// draft tokens of a request); [FASER] operations notes (the attention kernel
// must accept a chunk of the rows); [SSD] section details (PagedAttention).
//
// Three kernels on one stream:
//   plan   (1 CTA)   ancestor-or-self bit mask of every row (walk of the
//                    parent links), parent / window / length validation, and
//                    a length-weighted split-KV work list: the keys of each
//                    (request, KV head, 64-row query tile) are cut into
//                    splits of P pages so that about kUnitTarget units exist.
//   attend (1 CTA per unit, 4 warps)
//                    the query rows of the whole GQA group (row x head
//                    packed as "virtual rows", 16 per warp) share every KV
//                    page; pages are streamed through a 4-stage cp.async ring
//                    (16-byte copies, XOR-swizzled rows); QK^T and PV run on
//                    mma.sync m16n8k16 bf16 -> fp32; online softmax in the
//                    log2 domain; the ancestor mask is applied only on the
//                    stages that hold staged draft slots.
//   merge  (1 warp per row x head)
//                    log-sum-exp merge of the splits; requests that needed a
//                    single split were already written by the attend kernel.

#include "sv_internal.cuh"

namespace sv {
namespace attn {

constexpr int kTB = 32;          // tokens per pipeline stage (two pages)
constexpr int kStages = 4;       // cp.async ring depth
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileRows = 64;    // virtual rows per unit (16 per warp)
constexpr int kUnitTarget = kNumSMs * 16;
constexpr int kMinPagesPerSplit = 4;

struct ReqInfo {
  int ubase, nsplit, nrt, b, e, ctx, nblk, valid;
};

struct Header {
  int U;     // units in the work list
  int P;     // pages per split
  int pad[62];
};

struct Layout {
  size_t header, info, ubase, masks, ml, o, total;
  int ucap;
};

inline int unit_cap(int R, int total_rows, int group, int Hkv) {
  long nrt = (long)group * total_rows / kTileRows + R + 1;
  return (int)((long)Hkv * nrt + kUnitTarget);
}

inline Layout layout(int R, int total_rows, int group, int Hkv, int D) {
  Layout L;
  size_t off = 0;
  L.ucap = unit_cap(R, total_rows, group, Hkv);
  L.header = off; off += align256(sizeof(Header));
  L.info = off; off += align256(sizeof(ReqInfo) * (size_t)R);
  L.ubase = off; off += align256(sizeof(int) * (size_t)(R + 1));
  L.masks = off; off += align256(16 * (size_t)total_rows);
  L.ml = off; off += align256((size_t)L.ucap * kTileRows * 2 * sizeof(float));
  L.o = off; off += align256((size_t)L.ucap * kTileRows * (size_t)D * sizeof(float));
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
  const int R = a.bt.n_req;
  const int tid = threadIdx.x;
  Header* hdr = reinterpret_cast<Header*>(a.ws + a.L.header);
  ReqInfo* info = reinterpret_cast<ReqInfo*>(a.ws + a.L.info);
  int* ubase = reinterpret_cast<int*>(a.ws + a.L.ubase);
  unsigned long long* masks = reinterpret_cast<unsigned long long*>(a.ws + a.L.masks);
  __shared__ int s_bad;
  __shared__ unsigned long long s_W;
  __shared__ int s_warp[32];
  __shared__ int s_carry;

  if (tid == 0) {
    s_bad = (a.bt.cu_rows[0] != 0 || a.bt.cu_rows[R] != a.bt.total_rows) ? 1 : 0;
    s_W = 0ull;
    s_carry = 0;
  }
  for (int i = tid; i < R; i += blockDim.x) info[i].valid = 1;
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      flag(a.dev_status, SV_DEV_BAD_WINDOW);
      hdr->U = 0;
      hdr->P = 1;
    }
    return;
  }
  // Rows: ancestor-or-self masks and parent validation.
  for (int r = tid; r < a.bt.total_rows; r += blockDim.x) {
    const int i = find_segment(a.bt.cu_rows, R, r);
    const int cu = a.bt.cu_rows[i];
    const int j = r - cu;
    unsigned long long lo = 0ull, hi = 0ull;
    bool ok = j < kMaxRows;
    int m = j;
    for (int steps = 0; ok && steps <= kMaxRows; ++steps) {
      if (m < 64) lo |= 1ull << m; else hi |= 1ull << (m - 64);
      const int p = a.bt.parent[cu + m];
      if (m == 0) {
        if (p != -1) ok = false;
        break;
      }
      if (p < 0 || p >= m) { ok = false; break; }
      m = p;
    }
    masks[2 * (size_t)r] = lo;
    masks[2 * (size_t)r + 1] = hi;
    if (!ok) {
      info[i].valid = 0;
      if (j < kMaxRows) flag(a.dev_status, SV_DEV_BAD_PARENT);
    }
  }
  __syncthreads();
  // Requests: windows, lengths, total work.
  unsigned long long myW = 0;
  for (int i = tid; i < R; i += blockDim.x) {
    Window w = window_of(a.bt, i);
    bool valid = info[i].valid && w.ok;
    if (!w.ok) flag(a.dev_status, SV_DEV_BAD_WINDOW);
    const int ctx = a.cache_lens[i];
    if (valid && (ctx < 0 || (long)ctx + w.rows > (long)a.max_blocks * kBlockSize)) {
      valid = false;
      flag(a.dev_status, SV_DEV_BAD_LENGTH);
    }
    const int nw = valid ? max(0, w.e - w.b) : 0;
    const int nrt = (a.group * nw + kTileRows - 1) / kTileRows;
    const int nblk = nw ? (ctx + w.e + kBlockSize - 1) / kBlockSize : 0;
    myW += (unsigned long long)nrt * a.Hkv * nblk;
    ReqInfo ri;
    ri.valid = valid && nw > 0;
    ri.b = w.b;
    ri.e = w.e;
    ri.ctx = ctx;
    ri.nrt = nrt;
    ri.nblk = nblk;
    ri.nsplit = 0;
    ri.ubase = 0;
    info[i] = ri;
  }
  atomicAdd(&s_W, myW);
  __syncthreads();
  const unsigned long long W = s_W;
  int P = (int)((W + kUnitTarget - 1) / kUnitTarget);
  if (P < kMinPagesPerSplit) P = kMinPagesPerSplit;
  // Work list offsets (exclusive scan of units per request).
  for (int base = 0; base < R; base += blockDim.x) {
    const int i = base + tid;
    int units = 0;
    if (i < R) {
      ReqInfo ri = info[i];
      if (ri.valid) {
        ri.nsplit = (ri.nblk + P - 1) / P;
        units = ri.nrt * a.Hkv * ri.nsplit;
      }
      info[i].nsplit = ri.valid ? ri.nsplit : 0;
    }
    int excl, total;
    block_excl_scan(s_warp, units, excl, total);
    if (i < R) {
      ubase[i] = s_carry + excl;
      info[i].ubase = s_carry + excl;
    }
    __syncthreads();
    if (tid == 0) s_carry += total;
    __syncthreads();
  }
  if (tid == 0) {
    int U = s_carry;
    if (U > a.L.ucap) {  // cannot happen with the bound used for the workspace
      U = 0;
      flag(a.dev_status, SV_DEV_BAD_LENGTH);
    }
    ubase[R] = U;
    hdr->U = U;
    hdr->P = P;
  }
}

// ---------------------------------------------------------------- attend --

template <int D>
__global__ void __launch_bounds__(kThreads, 3) attend_kernel(Args a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __nv_bfloat16* smem = reinterpret_cast<__nv_bfloat16*>(smem_raw);
  const Header* hdr = reinterpret_cast<const Header*>(a.ws + a.L.header);
  const int U = hdr->U;
  const int u = blockIdx.x;
  if (u >= U) return;
  const int P = hdr->P;
  const int R = a.bt.n_req;
  const ReqInfo* infos = reinterpret_cast<const ReqInfo*>(a.ws + a.L.info);
  const int* ubase = reinterpret_cast<const int*>(a.ws + a.L.ubase);
  const unsigned long long* masks =
      reinterpret_cast<const unsigned long long*>(a.ws + a.L.masks);

  const int i = find_segment(ubase, R, u);
  const ReqInfo ri = infos[i];
  const int local = u - ri.ubase;
  const int s = local % ri.nsplit;
  const int rest = local / ri.nsplit;
  const int g = rest % a.Hkv;
  const int rt = rest / a.Hkv;
  const int M = a.group * (ri.e - ri.b);
  const int vr0 = rt * kTileRows;
  const int Mu = min(kTileRows, M - vr0);
  const int blk0 = s * P;
  const int blk1 = min(blk0 + P, ri.nblk);
  const int ctx = ri.ctx;
  const int tok_end = min(ctx + ri.e, blk1 * kBlockSize);
  const int cu = a.bt.cu_rows[i];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const bool active = warp * 16 < Mu;

  // The two virtual rows of this thread: (query row, head in group).
  const int vl_a = warp * 16 + gq, vl_b = vl_a + 8;
  const bool real_a = vl_a < Mu, real_b = vl_b < Mu;
  const int va = vr0 + vl_a, vb = vr0 + vl_b;
  const int prow_a = cu + ri.b + (real_a ? va / a.group : 0);
  const int prow_b = cu + ri.b + (real_b ? vb / a.group : 0);
  const int head_a = g * a.group + va % a.group;
  const int head_b = g * a.group + vb % a.group;

  // Q fragments (A operand), zero for padding rows.
  uint32_t qf[D / 16][4];
  {
    const uint32_t* qa = reinterpret_cast<const uint32_t*>(
        a.q + ((size_t)prow_a * a.Hq + head_a) * D);
    const uint32_t* qb = reinterpret_cast<const uint32_t*>(
        a.q + ((size_t)prow_b * a.Hq + head_b) * D);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qf[ks][0] = (active && real_a) ? __ldg(qa + ks * 8 + tq) : 0u;
      qf[ks][1] = (active && real_b) ? __ldg(qb + ks * 8 + tq) : 0u;
      qf[ks][2] = (active && real_a) ? __ldg(qa + ks * 8 + 4 + tq) : 0u;
      qf[ks][3] = (active && real_b) ? __ldg(qb + ks * 8 + 4 + tq) : 0u;
    }
  }
  unsigned long long mk_a0 = 0, mk_a1 = 0, mk_b0 = 0, mk_b1 = 0;
  if (real_a) { mk_a0 = masks[2 * (size_t)prow_a]; mk_a1 = masks[2 * (size_t)prow_a + 1]; }
  if (real_b) { mk_b0 = masks[2 * (size_t)prow_b]; mk_b1 = masks[2 * (size_t)prow_b + 1]; }

  const int n_stage = (blk1 - blk0 + 1) / 2;
  const int32_t* table = a.tables + (size_t)i * a.max_blocks;
  constexpr int kChunksPerRow = D / 8;                 // 16-byte chunks per token row
  constexpr int kChunksPerTensor = kTB * kChunksPerRow;
  constexpr int kCopiesPerThread = 2 * kChunksPerTensor / kThreads;

  auto issue = [&](int st) {
    if (st < n_stage) {
      __nv_bfloat16* buf = smem + (size_t)(st % kStages) * 2 * kTB * D;
#pragma unroll
      for (int k = 0; k < kCopiesPerThread; ++k) {
        const int c = threadIdx.x + k * kThreads;
        const int tensor = c / kChunksPerTensor;
        const int rem = c % kChunksPerTensor;
        const int row = rem / kChunksPerRow;
        const int col = rem % kChunksPerRow;
        const int page = blk0 + 2 * st + (row >> 4);
        const int tok = page * kBlockSize + (row & 15);
        const __nv_bfloat16* base = tensor ? a.v : a.k;
        const void* src = base;
        int bytes = 0;
        if (page < blk1 && tok < tok_end) {
          const int bid = __ldg(table + page);
          if (bid >= 0 && bid < a.num_blocks) {
            src = base + (((size_t)bid * a.Hkv + g) * kBlockSize + (row & 15)) * D + col * 8;
            bytes = 16;
          } else if (tensor == 0 && (row & 15) == 0 && col == 0) {
            flag(a.dev_status, SV_DEV_BAD_BLOCK_ID);
          }
        }
        __nv_bfloat16* dst = buf + (size_t)tensor * kTB * D + row * D + ((col ^ (row & 7)) << 3);
        cp_async16(smem_u32(dst), src, bytes);
      }
    }
    cp_async_commit();
  };

  float o[D / 8][4];
#pragma unroll
  for (int dn = 0; dn < D / 8; ++dn) o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

#pragma unroll
  for (int st = 0; st < kStages - 1; ++st) issue(st);

  for (int st = 0; st < n_stage; ++st) {
    issue(st + kStages - 1);
    cp_async_wait<kStages - 1>();
    __syncthreads();
    if (active) {
      const __nv_bfloat16* Ks = smem + (size_t)(st % kStages) * 2 * kTB * D;
      const uint32_t kbase = smem_u32(Ks);
      const uint32_t vbase = kbase + kTB * D * 2;
      const int t0 = (blk0 + 2 * st) * kBlockSize;
      float sc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < D / 16; ks += 2) {
          const int trow = nt * 8 + (lane & 7);
          const int chunk = 2 * ks + (lane >> 3);
          uint32_t r[4];
          ldsm_x4(r, kbase + (uint32_t)(trow * D + ((chunk ^ (trow & 7)) << 3)) * 2u);
          mma16816(sc[nt], qf[ks], r[0], r[1]);
          mma16816(sc[nt], qf[ks + 1], r[2], r[3]);
        }
      }
      // scale, mask, running max
      const bool need_mask = (t0 + kTB > ctx) || (t0 + kTB > tok_end);
      float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = sc[nt][e] * a.scale_log2;
          if (need_mask) {
            const int tok = t0 + nt * 8 + 2 * tq + (e & 1);
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
      const float nm_a = fmaxf(m_a, mx_a), nm_b = fmaxf(m_b, mx_b);
      const float base_a = nm_a == -INFINITY ? 0.f : nm_a;
      const float base_b = nm_b == -INFINITY ? 0.f : nm_b;
      const float al_a = exp2f(m_a - base_a), al_b = exp2f(m_b - base_b);
      m_a = nm_a;
      m_b = nm_b;
      float ps_a = 0.f, ps_b = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sc[nt][0] = exp2f(sc[nt][0] - base_a);
        sc[nt][1] = exp2f(sc[nt][1] - base_a);
        sc[nt][2] = exp2f(sc[nt][2] - base_b);
        sc[nt][3] = exp2f(sc[nt][3] - base_b);
        ps_a += sc[nt][0] + sc[nt][1];
        ps_b += sc[nt][2] + sc[nt][3];
      }
      l_a = l_a * al_a + ps_a;
      l_b = l_b * al_b + ps_b;
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        o[dn][0] *= al_a;
        o[dn][1] *= al_a;
        o[dn][2] *= al_b;
        o[dn][3] *= al_b;
      }
      // O += P V
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t pa[4];
        pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
        pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
        pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
        pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
        for (int dn = 0; dn < D / 8; dn += 2) {
          const int trow = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
          const int chunk = dn + (lane >> 4);
          uint32_t r[4];
          ldsm_x4_t(r, vbase + (uint32_t)(trow * D + ((chunk ^ (trow & 7)) << 3)) * 2u);
          mma16816(o[dn], pa, r[0], r[1]);
          mma16816(o[dn + 1], pa, r[2], r[3]);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  if (!active) return;
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
  l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
  l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);

  if (ri.nsplit == 1) {
    const float inv_a = l_a > 0.f ? 1.f / l_a : 0.f;
    const float inv_b = l_b > 0.f ? 1.f / l_b : 0.f;
    uint32_t* oa = reinterpret_cast<uint32_t*>(a.out + ((size_t)prow_a * a.Hq + head_a) * D);
    uint32_t* ob = reinterpret_cast<uint32_t*>(a.out + ((size_t)prow_b * a.Hq + head_b) * D);
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      if (real_a) oa[dn * 4 + tq] = pack_bf16(o[dn][0] * inv_a, o[dn][1] * inv_a);
      if (real_b) ob[dn * 4 + tq] = pack_bf16(o[dn][2] * inv_b, o[dn][3] * inv_b);
    }
  } else {
    float* ml = reinterpret_cast<float*>(a.ws + a.L.ml) + (size_t)u * kTileRows * 2;
    float* op = reinterpret_cast<float*>(a.ws + a.L.o) + (size_t)u * kTileRows * D;
    if (tq == 0) {
      if (real_a) { ml[2 * vl_a] = m_a; ml[2 * vl_a + 1] = l_a; }
      if (real_b) { ml[2 * vl_b] = m_b; ml[2 * vl_b + 1] = l_b; }
    }
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      if (real_a)
        *reinterpret_cast<float2*>(op + (size_t)vl_a * D + dn * 8 + 2 * tq) =
            make_float2(o[dn][0], o[dn][1]);
      if (real_b)
        *reinterpret_cast<float2*>(op + (size_t)vl_b * D + dn * 8 + 2 * tq) =
            make_float2(o[dn][2], o[dn][3]);
    }
  }
}

// ----------------------------------------------------------------- merge --

template <int D>
__global__ void __launch_bounds__(256) merge_kernel(Args a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long pair = (long)blockIdx.x * 8 + warp;
  if (pair >= (long)a.bt.total_rows * a.Hq) return;
  const int prow = (int)(pair / a.Hq), head = (int)(pair % a.Hq);
  const int R = a.bt.n_req;
  const int i = find_segment(a.bt.cu_rows, R, prow);
  const ReqInfo ri = reinterpret_cast<const ReqInfo*>(a.ws + a.L.info)[i];
  const int r = prow - a.bt.cu_rows[i];
  if (!ri.valid || ri.nsplit <= 1 || r < ri.b || r >= ri.e) return;
  const int g = head / a.group, hg = head % a.group;
  const int vr = (r - ri.b) * a.group + hg;
  const int rt = vr / kTileRows, vi = vr % kTileRows;
  const int ub = ri.ubase + (rt * a.Hkv + g) * ri.nsplit;
  const float* ml = reinterpret_cast<const float*>(a.ws + a.L.ml);
  const float* op = reinterpret_cast<const float*>(a.ws + a.L.o);
  float Mx = -INFINITY;
  for (int s = lane; s < ri.nsplit; s += 32)
    Mx = fmaxf(Mx, ml[((size_t)(ub + s) * kTileRows + vi) * 2]);
  Mx = warp_max(Mx);
  float L = 0.f;
  for (int s = lane; s < ri.nsplit; s += 32) {
    const size_t k = ((size_t)(ub + s) * kTileRows + vi) * 2;
    L += ml[k + 1] * exp2f(ml[k] - Mx);
  }
  L = warp_sum(L);
  constexpr int kPer = D / 32;
  float acc[kPer];
#pragma unroll
  for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
  for (int s = 0; s < ri.nsplit; ++s) {
    const size_t row = (size_t)(ub + s) * kTileRows + vi;
    const float w = exp2f(ml[row * 2] - Mx);
    const float* src = op + row * D + lane * kPer;
    if (kPer == 4) {
      const float4 x = *reinterpret_cast<const float4*>(src);
      acc[0] += w * x.x;
      acc[1 % kPer] += w * x.y;
      acc[2 % kPer] += w * x.z;
      acc[3 % kPer] += w * x.w;
    } else {
#pragma unroll
      for (int c = 0; c < kPer; ++c) acc[c] += w * src[c];
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* dst = a.out + ((size_t)prow * a.Hq + head) * D + lane * kPer;
#pragma unroll
  for (int c = 0; c < kPer; c += 2)
    *reinterpret_cast<uint32_t*>(dst + c) = pack_bf16(acc[c] * inv, acc[c + 1] * inv);
}

template <int D>
sv_status launch(const Args& a, cudaStream_t stream) {
  const size_t smem = (size_t)kStages * 2 * kTB * D * sizeof(__nv_bfloat16);
  static int attr_dev_mask = 0;  // devices whose kernel attribute is set
  int dev = 0;
  cudaGetDevice(&dev);
  if (!(attr_dev_mask & (1 << (dev & 31)))) {
    if (cudaFuncSetAttribute(attend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return SV_ERR_CUDA;
    attr_dev_mask |= 1 << (dev & 31);
  }
  plan_kernel<<<1, 1024, 0, stream>>>(a);
  SV_LAUNCH_CHECK();
  attend_kernel<D><<<a.L.ucap, kThreads, smem, stream>>>(a);
  SV_LAUNCH_CHECK();
  const long pairs = (long)a.bt.total_rows * a.Hq;
  merge_kernel<D><<<(unsigned)((pairs + 7) / 8), 256, 0, stream>>>(a);
  SV_LAUNCH_CHECK();
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
  return attn::layout(bt->n_req, bt->total_rows, group, kv->n_kv_heads, kv->head_dim).total;
}

extern "C" sv_status sv_tree_attend(const sv_paged_kv* kv, const sv_batch* bt, const void* q,
                                    int32_t n_q_heads, float softmax_scale, void* out, void* ws,
                                    size_t ws_bytes, int32_t* dev_status, void* stream) {
  sv_status st = check_attend_args(bt, kv, n_q_heads);
  if (st != SV_OK) return st;
  if (bt->n_req == 0 || bt->total_rows == 0) return SV_OK;
  if (!q || !out || !ws) return SV_ERR_INVALID_ARGUMENT;
  if (((uintptr_t)q | (uintptr_t)out) & 3) return SV_ERR_INVALID_ARGUMENT;
  if ((uintptr_t)ws & 255) return SV_ERR_INVALID_ARGUMENT;
  if (!(softmax_scale > 0.f)) return SV_ERR_INVALID_ARGUMENT;
  const int group = n_q_heads / kv->n_kv_heads;
  attn::Args a;
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
  a.L = attn::layout(bt->n_req, bt->total_rows, group, kv->n_kv_heads, kv->head_dim);
  a.dev_status = dev_status;
  if (ws_bytes < a.L.total) return SV_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return kv->head_dim == 128 ? attn::launch<128>(a, s) : attn::launch<64>(a, s);
}
