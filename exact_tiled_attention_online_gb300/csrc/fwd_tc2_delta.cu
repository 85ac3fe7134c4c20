// fwd_tc2_delta.cu -- the backward's per-row term D_i = dO_i . O_i for
// callers that did not keep the forward's fp32 output: the prefill forward
// (kernel template in fwd_tc2.cuh) runs again over the same inputs, mask,
// window and biases, and its epilogue dots each row's fp32 output (before
// any rounding, normalised by the rounded-probability sum so that it is an
// exact convex combination of V rows) with the row of dO instead of storing
// O.  With O rounded to bf16, a common offset of the value rows does not
// cancel in dO . (v_j - O_i), and the rounding error of O reaches every
// gradient through D ("attention-algorithm-error-and-complexity-tests",
// fourth paragraph: a missing or wrong denominator term in the backward).
#include "fwd_tc2.cuh"

namespace attn {
namespace {

template <int D>
cudaError_t launch_delta_d(const Tc2Args &a, const CUtensorMap (&m)[5], unsigned ctas,
                           cudaStream_t st) {
  const bool pos = a.p.scale_log2 > 0.f;
  if (a.p.btab) {  // a bias tensor comes here only with a positive scale, no slopes
    if constexpr (D == 128)
      if (a.staged) return launch2<D, true, true, false, 2, true>(a, m, ctas, st);
    return launch2<D, true, true, false, 1, true>(a, m, ctas, st);
  }
  if (a.p.slopes) return launch2<D, false, true, true, 0, true>(a, m, ctas, st);
  if (pos) return launch2<D, true, true, false, 0, true>(a, m, ctas, st);
  return launch2<D, false, true, false, 0, true>(a, m, ctas, st);
}

}  // namespace

// p.delta [n_heads_q, total_q] <- dO_i . O_i for every query row (0 for
// empty rows); p.dout, p.sdo: the upstream gradient and its layout.
cudaError_t launch_fwd_tc2_delta(const FwdParams &p, cudaStream_t st) {
  Tc2Args a;
  CUtensorMap m[5];
  long long ctas = 0;
  int rows_per_cta = 0;
  if (!p.delta || !p.dout) return cudaErrorInvalidValue;
  if (!setup_tc2(p, &a, m, &ctas, &rows_per_cta)) return cudaErrorInvalidValue;
  if (ctas == 0) return cudaSuccess;
  if (p.d == 64) return launch_delta_d<64>(a, m, (unsigned)ctas, st);
  return launch_delta_d<128>(a, m, (unsigned)ctas, st);
}

}  // namespace attn
