// adapt.cu — sv_adapt_gamma: per-request draft length from the request's own
// acceptance history.
//
// Source: [FASER] "FASER의 세 가지 메커니즘", mechanism 1 (per-request
// speculation length: each request's previous acceptance rate is fed back,
// requests that accept more get a longer gamma, requests that reject get a
// shorter one to avoid re-verifying rejected tokens).  The pages give no
// formula; the controller (decayed counts, Beta(1, 1) estimate, expected
// tokens per verified row) is specified in the header and computed here with
// IEEE fp64 add / multiply / divide in that order (__dadd_rn / __dmul_rn /
// __ddiv_rn keep the compiler from contracting them into fused operations).

#include "sv_internal.cuh"

namespace sv {
namespace adp {

__global__ void __launch_bounds__(256) adapt_kernel(int n_req, const int32_t* accepted_len,
                                                    const int32_t* verified, double* state,
                                                    int32_t* gamma_next, double decay,
                                                    double overhead, int gmin, int gmax,
                                                    int32_t* dev_status) {
  griddep_entry();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_req) return;
  const int g_used = verified[i];
  if (g_used < 0) return;
  const int a = accepted_len[i];
  if (a < 0 || a > g_used) {
    flag(dev_status, SV_DEV_BAD_LENGTH);
    return;
  }
  double S = state[2 * i], N = state[2 * i + 1];
  S = __dadd_rn(__dmul_rn(decay, S), (double)a);
  N = __dadd_rn(__dmul_rn(decay, N), (double)(a + (a < g_used ? 1 : 0)));
  state[2 * i] = S;
  state[2 * i + 1] = N;
  const double alpha = __ddiv_rn(__dadd_rn(S, 1.0), __dadd_rn(N, 2.0));
  // E(g) = sum_{k <= g} alpha^k by running products; score = E / (g + 1 + overhead)
  double pw = 1.0, E = 0.0;
  for (int g = 0; g < gmin; ++g) {
    E = __dadd_rn(E, pw);
    pw = __dmul_rn(pw, alpha);
  }
  int best = gmin;
  double best_score = -1.0;
  for (int g = gmin; g <= gmax; ++g) {
    E = __dadd_rn(E, pw);
    pw = __dmul_rn(pw, alpha);
    const double score = __ddiv_rn(E, __dadd_rn((double)(g + 1), overhead));
    if (score > best_score) {
      best_score = score;
      best = g;
    }
  }
  gamma_next[i] = best;
}

}  // namespace adp
}  // namespace sv

using namespace sv;

extern "C" sv_status sv_adapt_gamma(int32_t n_req, const int32_t* accepted_len,
                                    const int32_t* verified, double* state, int32_t* gamma_next,
                                    double decay, double overhead, int32_t gamma_min,
                                    int32_t gamma_max, int32_t* dev_status, void* stream) {
  SV_TRACE("sv_adapt_gamma");
  if (n_req < 0 || gamma_min < 0 || gamma_max < gamma_min || gamma_max > kMaxRows - 1)
    return SV_ERR_INVALID_ARGUMENT;
  if (!(decay > 0.0 && decay <= 1.0) || !(overhead >= 0.0)) return SV_ERR_INVALID_ARGUMENT;
  if (n_req == 0) return SV_OK;
  if (!accepted_len || !verified || !state || !gamma_next) return SV_ERR_INVALID_ARGUMENT;
  if (sv::launch(adp::adapt_kernel, (unsigned)((n_req + 255) / 256), 256, 0,
                 static_cast<cudaStream_t>(stream), (int)n_req, accepted_len, verified, state,
                 gamma_next, decay, overhead, (int)gamma_min, (int)gamma_max, dev_status) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  return SV_OK;
}
