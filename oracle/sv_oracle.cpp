// sv_oracle.cpp — CPU oracle for the target-side speculative-decoding
// verification step.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
// calls this file; only the tests, the package's smoke() check and the CPU
// baseline leg of bench.py do.  It shares no source, header, table or helper
// with the CUDA path: the seeded input generator is the only thing the two
// sides have in common.
//
// It is written to be read against the pages, not to be fast: plain loops,
// fp64 wherever the device works in fp32, no blocking and no fusion.  Every
// function says which passage it follows.  Page short names used below:
//   [SwiftSpec]  "SwiftSpec: 드래프터와 타깃을 서로 다른 GPU에 분리하고 비동기로
//                겹쳐 실행해 LLM 저지연 추론을 실현하는 방법 (ASPLOS 2026)",
//                section "SwiftSpec의 핵심 설계" (core design), mechanisms 2
//                (Tree-Aware KV Cache Management) and 3 (Fused
//                Latency-Optimized Kernels).
//   [DSpark]     "DSpark 하드웨어 인식 검증 스케줄러와 반자동회귀 병렬 드래프터를
//                통한 LLM 추론 가속화", sections "하드웨어 인식 Prefix 스케줄러",
//                "방법론", "기술 상세" and the glossary "용어 해설".
//   [FASER]      "FASER: 연속 배치 내 투기 디코딩의 단계 직렬화를 공간 분할 중첩으로
//                해결하는 방법", section "FASER의 세 가지 메커니즘", mechanisms
//                1 (per-request length) and 2 (early token pruning).
//   [SSD]        "SSD: 병렬 하드웨어를 활용한 초고속 추론 알고리즘 Speculative
//                Speculative Decoding", section "섹션별 상세" (PagedAttention).
//
// The pages never print the accept/reject rule.  Its definition used here is
// the standard lossless speculative-sampling rule: accept draft x with
// probability min(1, p(x)/q(x)); on rejection sample from
// normalize(max(0, p - q)); when every draft is accepted sample one more token
// from p.  Greedy mode accepts the longest prefix that matches the target
// argmax ([DSpark] glossary, "사전검증 디코딩": longest matching prefix,
// target distribution preserved).
//
// Parity status of each function (what pins it) is listed in the tests; the
// Philox generator reproduces the published Random123 known-answer vectors
// (tests/golden/philox4x32_10_kat.txt) and is pinned statistically as well.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// Error bits returned by the oracle (its own numbering).
enum : int {
  ORC_OK = 0,
  ORC_BAD_BLOCK = 1,
  ORC_BAD_PARENT = 2,
  ORC_POOL_OVERFLOW = 4,
  ORC_BAD_WINDOW = 8,
  ORC_BAD_TOKEN = 32,
  ORC_UNSUPPORTED = 64,
  ORC_BAD_LENGTH = 128,
  ORC_BAD_ARG = 256,
};

// ---------------------------------------------------------------- bf16 ----

double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Round to bf16, nearest-even, via fp32 (the fp64 -> fp32 step can round
// twice; the attention tolerance is four orders of magnitude wider).
uint16_t double_to_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return 0x7fc0;  // NaN
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

// -------------------------------------------------------------- Philox ----
// Philox4x32-10, written from its definition in Salmon, Moraes, Dror, Shaw,
// "Parallel random numbers: as easy as 1, 2, 3" (SC'11): a 4-word counter,
// a 2-word key, ten rounds of two 32x32->64 multiplies with the key bumped by
// the Weyl constants between rounds.

void philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
  const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += W0;
      k1 += W1;
    }
    uint64_t p0 = (uint64_t)M0 * (uint64_t)c0;
    uint64_t p1 = (uint64_t)M1 * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// Uniform for the accept test of draft at position j of request i:
// counter (j, i, 0, 0), word 0, top 24 bits -> [0, 1).
double accept_uniform(uint64_t seed, int i, int j) {
  uint32_t ctr[4] = {(uint32_t)j, (uint32_t)i, 0u, 0u};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

// Uniform in (0, 1) for group g (vocabulary entries 4g .. 4g+3) of the
// sampling race that emits the token at position pos of request i.  Groups
// are numbered in blocks of 128: group g = 128 b + 32 k + l takes word k of
// counter (32 b + l, i, 1, pos).  Top 23 bits plus one half -> (0, 1), exact
// in fp32 as well as fp64.
double race_uniform(uint64_t seed, int i, int pos, int g) {
  const uint32_t b = (uint32_t)g >> 7, k = ((uint32_t)g >> 5) & 3u, l = (uint32_t)g & 31u;
  uint32_t ctr[4] = {32u * b + l, (uint32_t)i, 1u, (uint32_t)pos};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return ((double)(out[k] >> 9) + 0.5) * (1.0 / 8388608.0);
}

// Uniform in (0, 1) that picks the entry inside the race's winning group g:
// word 0 of counter (g, i, 2, pos), same conversion.
double pick_uniform(uint64_t seed, int i, int pos, int g) {
  uint32_t ctr[4] = {(uint32_t)g, (uint32_t)i, 2u, (uint32_t)pos};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t out[4];
  philox4x32_10(ctr, key, out);
  return ((double)(out[0] >> 9) + 0.5) * (1.0 / 8388608.0);
}

// ------------------------------------------------------------ windows ----
// Which rows of request i this call handles.  rows = 1 + drafts (row 0 is
// the root, the last committed token).  verify_len (if given) truncates the
// chain to rows 0..verify_len ([DSpark] "하드웨어 인식 Prefix 스케줄러": only
// the selected prefix is verified).  [row_begin, row_end) is the chunk window
// ([FASER] mechanism 2: verification split into chunks).

struct Window {
  int rows, lim, b, e;  // e already clipped to lim
  bool ok;
};

Window window_of(int i, const int32_t* cu_rows, const int32_t* row_begin, const int32_t* row_end,
                 const int32_t* verify_len) {
  Window w;
  w.rows = cu_rows[i + 1] - cu_rows[i];
  w.ok = w.rows >= 1;
  w.lim = w.rows;
  if (verify_len) {
    int L = verify_len[i];
    if (L < 0) w.ok = false;
    if (L + 1 < w.lim) w.lim = L + 1;
  }
  w.b = row_begin ? row_begin[i] : 0;
  w.e = row_end ? row_end[i] : w.lim;
  if (w.b < 0 || w.b > w.e || w.e > w.rows) w.ok = false;
  if (w.e > w.lim) w.e = w.lim;
  return w;
}

template <class F>
void parallel_for(long n, int n_threads, F f) {
  if (n_threads <= 1 || n < 2) {
    for (long u = 0; u < n; ++u) f(u);
    return;
  }
  std::vector<std::thread> pool;
  long per = (n + n_threads - 1) / n_threads;
  for (int t = 0; t < n_threads; ++t) {
    long lo = t * per, hi = std::min(n, lo + per);
    if (lo >= hi) break;
    pool.emplace_back([=]() {
      for (long u = lo; u < hi; ++u) f(u);
    });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// Exposed for the tests: one Philox4x32-10 block.
void orc_philox4x32_10(const uint32_t* ctr, const uint32_t* key, uint32_t* out) {
  philox4x32_10(ctr, key, out);
}
double orc_accept_uniform(uint64_t seed, int i, int j) { return accept_uniform(seed, i, j); }
double orc_race_uniform(uint64_t seed, int i, int pos, int g) { return race_uniform(seed, i, pos, g); }
double orc_pick_uniform(uint64_t seed, int i, int pos, int g) { return pick_uniform(seed, i, pos, g); }

// -------------------------------------------------------- attention (a2) --
// For every row r of every request inside its window and every query head h:
//   out[r][h] = sum_k softmax_k(scale * q[r][h] . K[k][g]) V[k][g],
// g = h / (n_q_heads / n_kv), over the keys
//   {cache slots 0 .. ctx-1}  U  {staged slot ctx+m : m ancestor-or-self of r}.
// The draft rows' K/V are staged in the cache at slots ctx + node before the
// call; each tree node sees only its own root-to-node prefix
// ([SwiftSpec] mechanism 2: every node has a unique KV prefix; mechanism 3:
// all draft rows of a request verified in one padding-free call).  The cache
// is paged through block tables ([SSD] "섹션별 상세": PagedAttention).
// Output in fp64 (out_f64, optional) and rounded to bf16 (out_bf16).
int orc_tree_attend(int n_req, const int32_t* cu_rows, const int32_t* parent,
                    const int32_t* row_begin, const int32_t* row_end, const int32_t* verify_len,
                    const uint16_t* k_cache, const uint16_t* v_cache, int num_blocks,
                    int block_size, int n_kv, int d, const int32_t* block_tables, int max_blocks,
                    const int32_t* cache_lens, const uint16_t* q, int n_q_heads,
                    float softmax_scale, double* out_f64, uint16_t* out_bf16, int n_threads) {
  if (n_req < 0 || block_size <= 0 || n_kv <= 0 || d <= 0 || n_q_heads % n_kv != 0)
    return ORC_BAD_ARG;
  const int group = n_q_heads / n_kv;
  int err = 0;
  // Per-request validation first; invalid requests are skipped.
  std::vector<char> skip(n_req, 0);
  for (int i = 0; i < n_req; ++i) {
    Window w = window_of(i, cu_rows, row_begin, row_end, verify_len);
    if (!w.ok) { err |= ORC_BAD_WINDOW; skip[i] = 1; continue; }
    const int cu = cu_rows[i];
    if (parent[cu] != -1) { err |= ORC_BAD_PARENT; skip[i] = 1; continue; }
    for (int j = 1; j < w.rows; ++j)
      if (parent[cu + j] < 0 || parent[cu + j] >= j) { err |= ORC_BAD_PARENT; skip[i] = 1; }
    const long need = (long)cache_lens[i] + w.rows;
    if (cache_lens[i] < 0 || need > (long)max_blocks * block_size) {
      err |= ORC_BAD_LENGTH; skip[i] = 1; continue;
    }
    const long nblk = (need + block_size - 1) / block_size;
    for (long t = 0; t < nblk; ++t) {
      int blk = block_tables[(long)i * max_blocks + t];
      if (blk < 0 || blk >= num_blocks) { err |= ORC_BAD_BLOCK; skip[i] = 1; }
    }
  }
  // Flatten (request, row, head) into independent units.
  std::vector<long> unit_row;  // packed row index
  std::vector<int> unit_req;
  for (int i = 0; i < n_req; ++i) {
    if (skip[i]) continue;
    Window w = window_of(i, cu_rows, row_begin, row_end, verify_len);
    for (int r = w.b; r < w.e; ++r) {
      unit_row.push_back(cu_rows[i] + r);
      unit_req.push_back(i);
    }
  }
  const long n_units = (long)unit_row.size() * n_q_heads;
  parallel_for(n_units, n_threads, [&](long u) {
    const long prow = unit_row[u / n_q_heads];
    const int i = unit_req[u / n_q_heads];
    const int h = (int)(u % n_q_heads);
    const int g = h / group;
    const int cu = cu_rows[i];
    const int r = (int)(prow - cu);
    const int ctx = cache_lens[i];
    // Ancestors-or-self of r, by walking the parent links.
    std::vector<char> anc(r + 1, 0);
    for (int m = r; m >= 0; m = parent[cu + m]) anc[m] = 1;
    std::vector<long> slots;
    for (int t = 0; t < ctx; ++t) slots.push_back(t);
    for (int m = 0; m <= r; ++m)
      if (anc[m]) slots.push_back((long)ctx + m);
    const uint16_t* qv = q + (prow * n_q_heads + h) * (long)d;
    std::vector<double> s(slots.size());
    double mx = -INFINITY;
    for (size_t k = 0; k < slots.size(); ++k) {
      long slot = slots[k];
      long blk = block_tables[(long)i * max_blocks + slot / block_size];
      long off = slot % block_size;
      const uint16_t* kv = k_cache + ((blk * n_kv + g) * block_size + off) * (long)d;
      double dot = 0.0;
      for (int c = 0; c < d; ++c) dot += bf16_to_double(qv[c]) * bf16_to_double(kv[c]);
      s[k] = (double)softmax_scale * dot;
      if (s[k] > mx) mx = s[k];
    }
    double denom = 0.0;
    for (size_t k = 0; k < slots.size(); ++k) {
      s[k] = std::exp(s[k] - mx);
      denom += s[k];
    }
    std::vector<double> acc(d, 0.0);
    for (size_t k = 0; k < slots.size(); ++k) {
      long slot = slots[k];
      long blk = block_tables[(long)i * max_blocks + slot / block_size];
      long off = slot % block_size;
      const uint16_t* vv = v_cache + ((blk * n_kv + g) * block_size + off) * (long)d;
      for (int c = 0; c < d; ++c) acc[c] += s[k] * bf16_to_double(vv[c]);
    }
    for (int c = 0; c < d; ++c) {
      double o = acc[c] / denom;
      long idx = (prow * n_q_heads + h) * (long)d + c;
      if (out_f64) out_f64[idx] = o;
      if (out_bf16) out_bf16[idx] = double_to_bf16(o);
    }
  });
  return err;
}

}  // extern "C"

namespace {

// --------------------------------------------------- row statistics (a3) --
// Softmax of one logits row at temperature T:  x_v = l_v / T, divided in fp32
// (the precision the logits arrive in), then p_v = exp(x_v - lse) in fp64.
struct RowSoftmax {
  double m = -INFINITY;  // max of x
  double lse = 0.0;      // log sum exp x
};

RowSoftmax row_softmax(const float* l, int V, float T) {
  RowSoftmax s;
  for (int v = 0; v < V; ++v) {
    double x = (double)(l[v] / T);
    if (x > s.m) s.m = x;
  }
  double sum = 0.0;
  for (int v = 0; v < V; ++v) sum += std::exp((double)(l[v] / T) - s.m);
  s.lse = s.m + std::log(sum);
  return s;
}

double prob(const float* l, int v, float T, const RowSoftmax& s) {
  return std::exp((double)(l[v] / T) - s.lse);
}

// Greedy: index of the largest raw logit, lowest index among equal maxima.
int row_argmax(const float* l, int V) {
  int best = 0;
  for (int v = 1; v < V; ++v)
    if (l[v] > l[best]) best = v;
  return best;
}

// ------------------------------------------------ residual / bonus (a5) --
// Draw one token from normalize(w) with w_v = max(0, p_v - c q_v) (residual:
// c = 1 after one rejection, larger after several rejections among tree
// siblings) or w_v = p_v (bonus, all drafts accepted), in two steps:
//   1. a race among groups of four entries: group g (entries 4g .. 4g+3, the
//      last one possibly shorter) has weight W_g = sum of its w_v and key
//      W_g / E_g with E_g = -log(U_g), U_g ~ U(0,1) independent; the group
//      with the largest key wins (lowest g on ties).  P(g wins) = W_g / sum W
//      (the race form of the Gumbel-max trick, over groups);
//   2. inside the winning group, with u ~ U(0,1): the first entry whose
//      running sum of w (in index order) exceeds u W_g.
// P(v) = W_g / sum W * w_v / W_g = w_v / sum w: an exact sample of
// normalize(w).
//
// Both steps are also checked for closeness: if a device computing p and q in
// fp32 (relative error at most RACE_EPS per term) could pick another group,
// or land on the other side of a running-sum boundary, the decision is
// flagged ambiguous.
const double RACE_EPS = 2e-6;

int race_sample(const float* lp, const float* lq, int V, float T, const RowSoftmax& sp,
                const RowSoftmax* sq, uint64_t seed, int i, int pos, bool* ambiguous,
                double c = 1.0) {
  std::vector<double> w(V), err(V);
  double W = 0.0;
  for (int v = 0; v < V; ++v) {
    double p = prob(lp, v, T, sp);
    double q = sq ? c * prob(lq, v, T, *sq) : 0.0;
    w[v] = sq ? std::max(0.0, p - q) : p;
    err[v] = RACE_EPS * (p + q);
    W += w[v];
  }
  if (W <= 0.0) {  // p == q everywhere: normalize(max(0, p-q)) is undefined; use p
    for (int v = 0; v < V; ++v) {
      double p = prob(lp, v, T, sp);
      w[v] = p;
      err[v] = RACE_EPS * p;
    }
  }
  // 1. the race among groups
  const int G = (V + 3) / 4;
  std::vector<double> Wg(G, 0.0), Eg(G), eg(G, 0.0);
  for (int g = 0; g < G; ++g) {
    for (int v = 4 * g; v < std::min(V, 4 * g + 4); ++v) {
      Wg[g] += w[v];
      eg[g] += err[v];
    }
    Eg[g] = -std::log(race_uniform(seed, i, pos, g));
  }
  int best = -1;
  double best_key = -1.0;
  for (int g = 0; g < G; ++g) {
    double key = Wg[g] / Eg[g];
    if (key > best_key) { best_key = key; best = g; }
  }
  const double win_lo = std::max(0.0, Wg[best] - eg[best]) / Eg[best] * (1.0 - RACE_EPS);
  for (int g = 0; g < G; ++g) {
    if (g == best) continue;
    if ((Wg[g] + eg[g]) / Eg[g] * (1.0 + RACE_EPS) >= win_lo) { *ambiguous = true; break; }
  }
  // 2. the entry inside the winning group
  const int v0 = 4 * best, v1 = std::min(V, v0 + 4);
  const double t = pick_uniform(seed, i, pos, best) * Wg[best];
  int pick = -1;
  double S = 0.0;
  for (int v = v0; v < v1; ++v) {
    S += w[v];
    if (t < S) { pick = v; break; }
  }
  if (pick < 0)  // t at the very top of the group's range: its last positive entry
    for (int v = v0; v < v1; ++v)
      if (w[v] > 0.0) pick = v;
  const double tol = 2.0 * (eg[best] + RACE_EPS * Wg[best]);
  S = 0.0;
  for (int v = v0; v + 1 < v1; ++v) {
    S += w[v];
    if (std::fabs(t - S) <= tol) *ambiguous = true;
  }
  return pick;
}

struct AcceptArgs {
  const int32_t *cu_rows, *parent, *tokens, *row_begin, *row_end, *verify_len;
  const float *target, *draft;
  int V;
  float T;
  uint64_t seed;
  int32_t *accepted_len, *accepted_nodes;
  int max_rows;
  int32_t* next_token;
  uint8_t* ambiguous;
  int32_t* done;
  double* row_stats;
};

// ------------------------------------------------ tree sampling (NEXT-1) --
// T > 0 on a draft tree whose siblings were drawn independently from the
// parent's draft distribution q_n (with replacement).  From the root, the
// children of the current node n are tried in index order: child c (token x)
// is accepted with probability min(1, p'(x) / q_n(x)), where p' is the
// target distribution left after the siblings rejected before it; on
// acceptance the walk moves to c, otherwise p' <- normalize(max(0, p' - q_n)).
// When every child is rejected the emitted token is drawn from p'; at a leaf
// it is drawn from p_leaf (the bonus).  Tree verification is on the pages
// ([SwiftSpec] mechanism 2, [SSD]); this rejection rule is the plainest
// lossless reading for several candidates (each rejection removes exactly
// the mass the next candidate could have taken).
//
// After j rejections p' = max(0, p - c_j q_n) / S(c_j), S(c) = sum_v
// max(0, p_v - c q_v), with c_0 = 0 (S(0) = 1) and c_{j+1} = c_j + S(c_j):
// max(0, max(0, p - c q) / S - q) = max(0, p - (c + S) q) / S.  If S reaches
// 0 (p <= c q everywhere) the residual is undefined: the remaining siblings
// are not tested and the token is drawn from p_n.  Uniforms: child c uses
// accept_uniform(seed, i, c); the emitted token uses the race stream at
// position (accepted nodes + 1), as for a chain.
double residual_mass(const float* lp, const float* lq, int V, float T, const RowSoftmax& sp,
                     const RowSoftmax& sq, double c) {
  double s = 0.0;
  for (int v = 0; v < V; ++v) s += std::max(0.0, prob(lp, v, T, sp) - c * prob(lq, v, T, sq));
  return s;
}

void tree_sample(const AcceptArgs& a, int i, const Window& w, int cu, int32_t* nodes) {
  const long V = a.V;
  int n = 0, k = 0, next = -1;
  bool amb = false;
  for (;;) {
    const float* lp = a.target + (cu + n) * V;
    const float* lq = a.draft + (cu + n) * V;
    const RowSoftmax sp = row_softmax(lp, a.V, a.T);
    std::vector<int> kids;
    for (int c = n + 1; c < w.rows; ++c)
      if (a.parent[cu + c] == n) kids.push_back(c);
    if (kids.empty()) {  // leaf: bonus token from p_n
      next = race_sample(lp, nullptr, a.V, a.T, sp, nullptr, a.seed, i, k + 1, &amb);
      break;
    }
    const RowSoftmax sq = row_softmax(lq, a.V, a.T);
    double c = 0.0, S = 1.0;
    bool moved = false, vanished = false;
    for (int ch : kids) {
      const int x = a.tokens[cu + ch];
      const double p = prob(lp, x, a.T, sp), q = prob(lq, x, a.T, sq);
      const double pres = std::max(0.0, p - c * q) / S;
      const double ratio = q > 0.0 ? std::min(1.0, pres / q) : 1.0;
      const double u = accept_uniform(a.seed, i, ch);
      if (std::fabs(u - ratio) < 1e-6) amb = true;
      if (u < ratio) {
        nodes[++k] = ch;
        n = ch;
        moved = true;
        break;
      }
      c += S;
      S = residual_mass(lp, lq, a.V, a.T, sp, sq, c);
      if (!(S > 0.0)) {
        vanished = true;
        break;
      }
    }
    if (moved) continue;
    next = vanished ? race_sample(lp, nullptr, a.V, a.T, sp, nullptr, a.seed, i, k + 1, &amb)
                    : race_sample(lp, lq, a.V, a.T, sp, &sq, a.seed, i, k + 1, &amb, c);
    break;
  }
  a.accepted_len[i] = k;
  a.next_token[i] = next;
  if (amb) a.ambiguous[i] = 1;
}

// Accept/reject of one request ([DSpark] glossary: the longest accepted prefix
// is kept and the target distribution is preserved; [FASER] mechanism 1:
// every request has its own number of drafts; mechanism 2: a request stops at
// its first rejection and its later rows are never examined).
int accept_one(const AcceptArgs& a, int i) {
  Window w = window_of(i, a.cu_rows, a.row_begin, a.row_end, a.verify_len);
  if (!w.ok) return ORC_BAD_WINDOW;
  if (w.b >= w.e) return ORC_OK;  // empty window: request untouched
  const int cu = a.cu_rows[i];
  const long V = a.V;
  if (a.parent[cu] != -1) return ORC_BAD_PARENT;
  bool chain = true;
  for (int j = 1; j < w.rows; ++j) {
    int p = a.parent[cu + j];
    if (p < 0 || p >= j) return ORC_BAD_PARENT;
    if (p != j - 1) chain = false;
  }
  for (int j = 1; j < w.rows; ++j)
    if (a.tokens[cu + j] < 0 || a.tokens[cu + j] >= a.V) return ORC_BAD_TOKEN;
  int32_t* nodes = a.accepted_nodes + (long)i * a.max_rows;
  if (!chain) {
    // A tree is verified in one call over all its rows.
    if (w.b != 0 || w.e != w.rows) return ORC_BAD_WINDOW;
  }
  if (w.b == 0) {  // first window of this step: reset the request's state
    a.accepted_len[i] = 0;
    nodes[0] = 0;
    for (int k = 1; k < a.max_rows; ++k) nodes[k] = -1;
    a.next_token[i] = -1;
    a.ambiguous[i] = 0;
    if (a.done) a.done[i] = 0;
  } else {
    if (a.next_token[i] >= 0) return ORC_OK;  // already decided earlier
    if (a.accepted_len[i] != w.b) return ORC_BAD_WINDOW;
  }
  const float* target = a.target;
  double* rs = a.row_stats;

  if (a.T == 0.0f) {
    // ---- greedy (a4, T = 0) ----
    if (rs)
      for (int r = w.b; r < w.e; ++r) {
        const float* l = target + (cu + r) * V;
        int am = row_argmax(l, a.V);
        rs[(cu + r) * 4 + 0] = (double)l[am];
        rs[(cu + r) * 4 + 1] = (double)am;
      }
    if (chain) {
      const int jmax = std::min(w.e, w.lim - 1);
      for (int j = w.b + 1; j <= jmax; ++j) {
        int am = row_argmax(target + (cu + j - 1) * V, a.V);
        if (a.tokens[cu + j] == am) {
          a.accepted_len[i] = j;
          nodes[j] = j;
        } else {
          a.next_token[i] = am;
          break;
        }
      }
      if (a.next_token[i] < 0 && w.e == w.lim && a.accepted_len[i] == w.lim - 1)
        a.next_token[i] = row_argmax(target + (cu + w.lim - 1) * V, a.V);
    } else {
      // Tree: keep the longest root-to-node path along which every node's
      // token is the target argmax of its parent; among equally long paths
      // the one whose first differing node has the lower index
      // ([SwiftSpec] mechanism 2: accepted path kept, the rest released).
      std::vector<int> am(w.rows), best_len(w.rows, 0), best_child(w.rows, -1);
      for (int n = 0; n < w.rows; ++n) am[n] = row_argmax(target + (cu + n) * V, a.V);
      for (int n = w.rows - 1; n >= 0; --n) {
        for (int c = n + 1; c < w.rows; ++c) {
          if (a.parent[cu + c] != n || a.tokens[cu + c] != am[n]) continue;
          if (1 + best_len[c] > best_len[n]) {
            best_len[n] = 1 + best_len[c];
            best_child[n] = c;
          }
        }
      }
      int n = 0, k = 0;
      while (best_child[n] >= 0) {
        n = best_child[n];
        nodes[++k] = n;
      }
      a.accepted_len[i] = k;
      a.next_token[i] = am[n];
    }
  } else if (!chain) {
    tree_sample(a, i, w, cu, nodes);
  } else {
    // ---- speculative sampling (a4 + a5, T > 0, chains) ----
    const float* draft = a.draft;
    std::vector<RowSoftmax> sp(w.rows), sq(w.rows);
    for (int r = w.b; r < w.e; ++r) {
      sp[r] = row_softmax(target + (cu + r) * V, a.V, a.T);
      if (rs) rs[(cu + r) * 4 + 0] = sp[r].lse;
      if (r + 1 <= w.lim - 1) {
        sq[r] = row_softmax(draft + (cu + r) * V, a.V, a.T);
        if (rs) rs[(cu + r) * 4 + 1] = sq[r].lse;
      }
    }
    bool amb = false;
    const int jmax = std::min(w.e, w.lim - 1);
    for (int j = w.b + 1; j <= jmax; ++j) {
      const float* lp = target + (cu + j - 1) * V;
      const float* lq = draft + (cu + j - 1) * V;
      const int x = a.tokens[cu + j];
      double p = prob(lp, x, a.T, sp[j - 1]);
      double q = prob(lq, x, a.T, sq[j - 1]);
      if (rs) {
        rs[(cu + j) * 4 + 2] = p;
        rs[(cu + j) * 4 + 3] = q;
      }
      double ratio = q > 0.0 ? std::min(1.0, p / q) : 1.0;
      double u = accept_uniform(a.seed, i, j);
      if (std::fabs(u - ratio) < 1e-6) amb = true;
      if (u < ratio) {
        a.accepted_len[i] = j;
        nodes[j] = j;
      } else {
        a.next_token[i] =
            race_sample(lp, lq, a.V, a.T, sp[j - 1], &sq[j - 1], a.seed, i, j, &amb);
        break;
      }
    }
    if (a.next_token[i] < 0 && w.e == w.lim && a.accepted_len[i] == w.lim - 1) {
      const int r = w.lim - 1;
      a.next_token[i] = race_sample(target + (cu + r) * V, nullptr, a.V, a.T, sp[r], nullptr,
                                    a.seed, i, w.lim, &amb);
    }
    if (amb) a.ambiguous[i] = 1;
  }
  if (a.done) a.done[i] = a.next_token[i] >= 0 ? 1 : 0;
  return ORC_OK;
}

}  // namespace

extern "C" {

// ------------------------------------------------- accept / reject (a3-a5) --
// State across windows: accepted_len, accepted_nodes[i][0..], next_token
// (-1 until decided), ambiguous, done.  A window starting at row 0 resets the
// request; a later window continues it.  row_stats (optional, [rows][4]):
// T > 0: [0] lse of the target row, [1] lse of the draft row, [2] p and [3] q
// of the row's own token under its parent's rows; T = 0: [0] max raw target
// logit, [1] its argmax.
int orc_accept(int n_req, const int32_t* cu_rows, const int32_t* parent, const int32_t* tokens,
               const int32_t* row_begin, const int32_t* row_end, const int32_t* verify_len,
               const float* target_logits, const float* draft_logits, int V, float T,
               uint64_t seed, int32_t* accepted_len, int32_t* accepted_nodes, int max_rows,
               int32_t* next_token, uint8_t* ambiguous, int32_t* done, double* row_stats,
               int n_threads) {
  if (V <= 0 || !(T >= 0.0f) || (T > 0.0f && !draft_logits)) return ORC_BAD_ARG;
  AcceptArgs a{cu_rows, parent, tokens, row_begin, row_end, verify_len, target_logits,
               draft_logits, V, T, seed, accepted_len, accepted_nodes, max_rows,
               next_token, ambiguous, done, row_stats};
  std::vector<int> errs(n_req, 0);
  parallel_for(n_req, n_threads, [&](long i) { errs[i] = accept_one(a, (int)i); });
  int err = 0;
  for (int e : errs) err |= e;
  return err;
}

// ----------------------------------------------------------- commit (a6) --
// Keep the accepted path's K/V and release the rest ([SwiftSpec] mechanism 2:
// only the accepted path's KV stays, rejected paths are freed at once).
// For request i with a = accepted_len[i] and path = accepted_nodes[i][0..a]
// (path[0] = root = 0): slot ctx+k <- staged slot ctx+path[k], all heads,
// every source read before any destination is written.  New length
// ctx + 1 + a.  Blocks at table index ceil(new_len/bs) .. ceil((ctx+rows)/bs)-1
// are pushed onto the free list in (request, table index) order and their
// table entries set to -1.
int orc_commit_kv(int n_req, const int32_t* cu_rows, uint16_t* k_cache, uint16_t* v_cache,
                  int num_blocks, int block_size, int n_kv, int d, int32_t* block_tables,
                  int max_blocks, int32_t* cache_lens, const int32_t* accepted_len,
                  const int32_t* accepted_nodes, int max_rows, int32_t* free_list,
                  int32_t* free_count, int capacity) {
  int err = 0;
  const long slot_elems = (long)n_kv * d;  // one token, all heads
  for (int i = 0; i < n_req; ++i) {
    const int rows = cu_rows[i + 1] - cu_rows[i];
    const int ctx = cache_lens[i];
    const int a = accepted_len[i];
    const int32_t* path = accepted_nodes + (long)i * max_rows;
    if (a < 0 || a > rows - 1 || path[0] != 0) { err |= ORC_BAD_WINDOW; continue; }
    bool ok = true;
    for (int k = 1; k <= a; ++k)
      if (path[k] <= path[k - 1] || path[k] >= rows) ok = false;
    if (!ok) { err |= ORC_BAD_WINDOW; continue; }
    if ((long)ctx + rows > (long)max_blocks * block_size) { err |= ORC_BAD_LENGTH; continue; }
    int32_t* table = block_tables + (long)i * max_blocks;
    auto addr = [&](long slot, int g, int c) -> long {
      long blk = table[slot / block_size];
      return ((blk * n_kv + g) * block_size + slot % block_size) * (long)d + c;
    };
    for (int k = 0; k <= a; ++k) {
      long s = (long)ctx + path[k];
      int blk = table[s / block_size];
      long t2 = ((long)ctx + k) / block_size;
      if (blk < 0 || blk >= num_blocks || table[t2] < 0 || table[t2] >= num_blocks) ok = false;
    }
    if (!ok) { err |= ORC_BAD_BLOCK; continue; }
    // Gather, then scatter.
    std::vector<uint16_t> kbuf((a + 1) * slot_elems), vbuf((a + 1) * slot_elems);
    for (int k = 0; k <= a; ++k)
      for (int g = 0; g < n_kv; ++g)
        for (int c = 0; c < d; ++c) {
          long src = addr((long)ctx + path[k], g, c);
          kbuf[k * slot_elems + (long)g * d + c] = k_cache[src];
          vbuf[k * slot_elems + (long)g * d + c] = v_cache[src];
        }
    for (int k = 0; k <= a; ++k)
      for (int g = 0; g < n_kv; ++g)
        for (int c = 0; c < d; ++c) {
          long dst = addr((long)ctx + k, g, c);
          k_cache[dst] = kbuf[k * slot_elems + (long)g * d + c];
          v_cache[dst] = vbuf[k * slot_elems + (long)g * d + c];
        }
    const long new_len = (long)ctx + 1 + a;
    const long keep = (new_len + block_size - 1) / block_size;
    const long used = ((long)ctx + rows + block_size - 1) / block_size;
    long n_free = 0;
    for (long t = keep; t < used; ++t)
      if (table[t] >= 0) ++n_free;
    if (*free_count + n_free > capacity) {
      err |= ORC_POOL_OVERFLOW;
    } else {
      for (long t = keep; t < used; ++t) {
        if (table[t] < 0) continue;
        free_list[(*free_count)++] = table[t];
        table[t] = -1;
      }
    }
    cache_lens[i] = (int32_t)new_len;
  }
  return err;
}

// ------------------------------------------------- budget selection (a8) --
// [DSpark] "하드웨어 인식 Prefix 스케줄러" / "방법론" / "기술 상세":
// prefix survival S_{i,k} = c_{i,1} * ... * c_{i,k} (product of per-position
// conditional survival probabilities, glossary "접두사 생존확률"); every
// (request, position) candidate sorted by survival, descending; candidates
// admitted one at a time; with m admitted the batch is B = R + m rows and the
// expected accepted tokens tau = R + sum of the admitted S; the budget is the
// m maximising Theta = tau * SPS(B).
// Exactness choices (not on the pages): S is an fp32 left-to-right product;
// the sort key is (~bits(S)) << 32 | (i * gamma_max + k - 1), ascending, so
// equal S go to the lower request then the lower position; tau is summed in
// fixed point (2^-40 units, each S truncated) so that the sum does not depend
// on the order of additions; Theta = double(tau_fx) * 2^-40 * double(SPS(B));
// ties go to the smaller B.
int orc_select_budget(int n_req, int gamma_max, const float* cond_survival, const int32_t* gamma,
                      const float* sps, int b_max, int32_t* verify_len, int32_t* best_B,
                      double* best_theta) {
  if (n_req <= 0 || gamma_max < 0 || b_max < n_req) return ORC_BAD_ARG;
  std::vector<uint64_t> keys;
  std::vector<float> S((size_t)n_req * (gamma_max > 0 ? gamma_max : 1), 0.0f);
  for (int i = 0; i < n_req; ++i) {
    int gi = gamma ? gamma[i] : gamma_max;
    if (gi < 0 || gi > gamma_max) return ORC_BAD_ARG;
    float s = 1.0f;
    for (int k = 1; k <= gi; ++k) {
      float c = cond_survival[(long)i * gamma_max + k - 1];
      if (!(c >= 0.0f && c <= 1.0f)) return ORC_BAD_ARG;
      s = s * c;
      S[(long)i * gamma_max + k - 1] = s;
      // The sort is by the value of S: -0 (from a factor c = -0) is the same
      // survival as +0 and takes +0's key.
      const float key_s = (s == 0.0f) ? 0.0f : s;
      uint32_t bits;
      std::memcpy(&bits, &key_s, 4);
      keys.push_back(((uint64_t)(~bits) << 32) | (uint64_t)(i * gamma_max + k - 1));
    }
  }
  std::sort(keys.begin(), keys.end());
  const long M = (long)keys.size();
  const long m_hi = std::min<long>(M, (long)b_max - n_req);
  const double two40 = 1099511627776.0;  // 2^40
  uint64_t tau_fx = (uint64_t)n_req << 40;
  long best_m = 0;
  double best = (double)tau_fx / two40 * (double)sps[n_req];
  for (long m = 1; m <= m_hi; ++m) {
    uint32_t idx = (uint32_t)(keys[m - 1] & 0xffffffffu);
    float s = S[idx];
    tau_fx += (uint64_t)std::trunc((double)s * two40);
    double theta = (double)tau_fx / two40 * (double)sps[n_req + m];
    if (theta > best) { best = theta; best_m = m; }
  }
  for (int i = 0; i < n_req; ++i) verify_len[i] = 0;
  for (long m = 0; m < best_m; ++m) {
    uint32_t idx = (uint32_t)(keys[m] & 0xffffffffu);
    verify_len[idx / gamma_max] += 1;
  }
  *best_B = (int32_t)(n_req + best_m);
  *best_theta = best;
  return ORC_OK;
}

// ------------------------------------------- chunked verification (a7) --
// [FASER] mechanism 2 (early token pruning): the verification of every
// request is split into chunks of `chunk` rows; after each chunk, requests
// that met a rejection (or emitted their bonus token) leave, so rows behind a
// rejected prefix are never attended or tested.  Chunk c covers rows
// [c*chunk, min((c+1)*chunk, lim)) of each request still running.
int orc_verify_chunked(int n_req, const int32_t* cu_rows, const int32_t* parent,
                       const int32_t* tokens, const int32_t* verify_len, int max_rows,
                       int chunk, const uint16_t* k_cache, const uint16_t* v_cache,
                       int num_blocks, int block_size, int n_kv, int d,
                       const int32_t* block_tables, int max_blocks, const int32_t* cache_lens,
                       const uint16_t* q, int n_q_heads, float softmax_scale, double* out_f64,
                       uint16_t* out_bf16, const float* target_logits, const float* draft_logits,
                       int V, float T, uint64_t seed, int32_t* accepted_len,
                       int32_t* accepted_nodes, int32_t* next_token, uint8_t* ambiguous,
                       int32_t* done, int32_t* rows_attended, int n_threads) {
  if (chunk <= 0) return ORC_BAD_ARG;
  std::vector<int32_t> rb(n_req), re(n_req);
  for (int i = 0; i < n_req; ++i) done[i] = 0;
  int err = 0;
  long attended = 0;
  for (int c = 0; c * chunk < max_rows; ++c) {
    for (int i = 0; i < n_req; ++i) {
      Window w = window_of(i, cu_rows, nullptr, nullptr, verify_len);
      int b = c * chunk, e = std::min(b + chunk, w.lim);
      if (done[i] || b >= e) b = e = std::min(b, w.rows);  // empty window
      rb[i] = b;
      re[i] = e;
      attended += e - b;
    }
    err |= orc_tree_attend(n_req, cu_rows, parent, rb.data(), re.data(), verify_len, k_cache,
                           v_cache, num_blocks, block_size, n_kv, d, block_tables, max_blocks,
                           cache_lens, q, n_q_heads, softmax_scale, out_f64, out_bf16, n_threads);
    err |= orc_accept(n_req, cu_rows, parent, tokens, rb.data(), re.data(), verify_len,
                      target_logits, draft_logits, V, T, seed, accepted_len, accepted_nodes,
                      max_rows, next_token, ambiguous, done, nullptr, n_threads);
  }
  if (rows_attended) *rows_attended = (int32_t)attended;
  return err;
}

// -------------------------------------------- draft length (NEXT-4) --
// Per-request gamma from the request's own acceptance ([FASER] mechanism 1:
// the previous acceptance rate feeds back, accepting requests get a longer
// gamma, rejecting ones a shorter).  The pages give no formula; the one
// written here (and in the library's header) is:
//   S <- decay * S + a;  N <- decay * N + a + (a < verified);
//   alpha = (S + 1) / (N + 2);
//   gamma = argmax_{g in [gmin, gmax]} E(g) / (g + 1 + overhead),
//   E(g) = sum_{k=0..g} alpha^k, smallest g on ties,
// in IEEE double, each operation rounded on its own (this file is compiled
// with -ffp-contract=off).  verified < 0 leaves the request untouched;
// a < 0 or a > verified is reported.
int orc_adapt_gamma(int n_req, const int32_t* accepted_len, const int32_t* verified,
                    double* state, int32_t* gamma_next, double decay, double overhead,
                    int gmin, int gmax) {
  if (n_req < 0 || gmin < 0 || gmax < gmin || !(decay > 0.0 && decay <= 1.0) ||
      !(overhead >= 0.0))
    return ORC_BAD_ARG;
  int err = 0;
  for (int i = 0; i < n_req; ++i) {
    const int used = verified[i];
    if (used < 0) continue;
    const int a = accepted_len[i];
    if (a < 0 || a > used) { err |= ORC_BAD_LENGTH; continue; }
    double S = decay * state[2 * i] + (double)a;
    double N = decay * state[2 * i + 1] + (double)(a + (a < used ? 1 : 0));
    state[2 * i] = S;
    state[2 * i + 1] = N;
    const double alpha = (S + 1.0) / (N + 2.0);
    double pw = 1.0, E = 0.0;
    int best = gmin;
    double best_score = -1.0;
    for (int g = 0; g <= gmax; ++g) {
      E = E + pw;
      pw = pw * alpha;
      if (g < gmin) continue;
      const double score = E / ((double)(g + 1) + overhead);
      if (score > best_score) { best_score = score; best = g; }
    }
    gamma_next[i] = best;
  }
  return err;
}

// -------------------------------------------- chunk size (NEXT-4) --
// [FASER] "FASER의 세 가지 메커니즘", mechanism 2 (verification in chunks,
// requests leave at their first rejection) with the remark that the chunk
// size follows the load.  The pages give no rule; the one written here (and
// in the library's header) is the expected cost of a chunked step:
//   a_i = min(1, (S_i + 1) / (N_i + 2))   (acceptance estimate from the
//         draft-length controller's state);
//   for a chunk size c in 1..max_rows (max_rows = max_i rows_i), chunk k
//   covers rows [b, e) = [k c, min((k+1) c, rows_i)) of request i, which
//   reaches it when drafts 1..k c were all accepted: P_ik = a_i^(k c)
//   (P_i0 = 1, P_i,k+1 = P_ik * a_i^c, a_i^c by c multiplications);
//   then it reads bytes_ik = (ctx_i + e) kv_bytes + (e - b) row_bytes;
//   cost(c) = K(c) chunk_bytes + sum over i, k of trunc(P_ik bytes_ik)
//   (u64), K(c) = ceil(max_rows / c);
//   chunk = the c of least cost, the largest c on ties.
// fp64, each operation rounded on its own (this file is compiled with
// -ffp-contract=off).  Requests with rows outside [1, 128], a negative
// context or a state that is not finite and non-negative are reported and
// left out.  costs[c - 1] for c > max_rows is UINT64_MAX.
int orc_select_chunk(int n_req, const int32_t* rows, const int32_t* ctx, const double* state,
                     double kv_bytes, double row_bytes, uint64_t chunk_bytes, int32_t* chunk,
                     uint64_t* cost, uint64_t* costs) {
  if (n_req < 0 || !(kv_bytes >= 0.0) || !(row_bytes >= 0.0)) return ORC_BAD_ARG;
  int err = 0;
  int max_rows = 0;
  std::vector<char> ok(n_req, 0);
  std::vector<double> alpha(n_req, 0.0);
  for (int i = 0; i < n_req; ++i) {
    const double S = state[2 * i], N = state[2 * i + 1];
    if (rows[i] < 1 || rows[i] > 128 || ctx[i] < 0 || !std::isfinite(S) || !std::isfinite(N) ||
        S < 0.0 || N < 0.0) {
      err |= ORC_BAD_LENGTH;
      continue;
    }
    ok[i] = 1;
    alpha[i] = std::min(1.0, (S + 1.0) / (N + 2.0));
    max_rows = std::max(max_rows, (int)rows[i]);
  }
  for (int c = 1; c <= 128; ++c) costs[c - 1] = UINT64_MAX;
  int best = 1;
  uint64_t best_cost = 0;
  for (int c = 1; c <= max_rows; ++c) {
    const uint64_t K = (uint64_t)((max_rows + c - 1) / c);
    uint64_t total = K * chunk_bytes;
    for (int i = 0; i < n_req; ++i) {
      if (!ok[i]) continue;
      double ac = 1.0;
      for (int t = 0; t < c; ++t) ac = ac * alpha[i];
      double P = 1.0;
      for (int b = 0; b < rows[i]; b += c) {
        const int e = std::min(b + c, (int)rows[i]);
        const double bytes = (double)(ctx[i] + e) * kv_bytes + (double)(e - b) * row_bytes;
        total += (uint64_t)(P * bytes);
        P = P * ac;
      }
    }
    costs[c - 1] = total;
    if (c == 1 || total <= best_cost) {
      best = c;
      best_cost = total;
    }
  }
  *chunk = best;
  *cost = best_cost;
  return err;
}

}  // extern "C"
