// fwd_tc2.cu -- launcher of the tensor-core prefill forward (the kernel
// template is in fwd_tc2.cuh): the instances that write O, lse and, when
// asked, the fp32 output.
#include "fwd_tc2.cuh"

namespace attn {
namespace {

template <int D>
cudaError_t launch2_d(const Tc2Args &a, const CUtensorMap (&m)[5], unsigned ctas, cudaStream_t st) {
  const bool pos = a.p.scale_log2 > 0.f, rs = a.p.o_f32 != nullptr;
  if (a.p.btab) {  // the caller routes a bias tensor here only with a positive scale, no slopes
    if constexpr (D == 128)
      if (a.staged)
        return rs ? launch2<D, true, true, false, 2>(a, m, ctas, st)
                  : launch2<D, true, false, false, 2>(a, m, ctas, st);
    return rs ? launch2<D, true, true, false, 1>(a, m, ctas, st)
              : launch2<D, true, false, false, 1>(a, m, ctas, st);
  }
  if (a.p.slopes) return rs ? launch2<D, false, true, true>(a, m, ctas, st)
                            : launch2<D, false, false, true>(a, m, ctas, st);
  if (pos) return rs ? launch2<D, true, true, false>(a, m, ctas, st)
                     : launch2<D, true, false, false>(a, m, ctas, st);
  return rs ? launch2<D, false, true, false>(a, m, ctas, st)
            : launch2<D, false, false, false>(a, m, ctas, st);
}

}  // namespace

// Prefill plan (one head per tile, no key splits) with two query tiles per CTA.
cudaError_t launch_fwd_tc2(const FwdParams &p, cudaStream_t st, char *desc, size_t desc_len) {
  snprintf(desc, desc_len, "fwd_tc2_d%d (tensor map or grid size rejected)", p.d);
  Tc2Args a;
  CUtensorMap m[5];
  long long ctas = 0;
  int rows_per_cta = 0;
  if (!setup_tc2(p, &a, m, &ctas, &rows_per_cta)) return cudaErrorInvalidValue;
  snprintf(desc, desc_len, "fwd_tc2_d%d%s ctas=%lld rows_per_cta=%d heads_per_cta=%d", p.d,
           p.btab ? (a.staged ? "_btab_smem" : "_btab") : "", ctas, rows_per_cta,
           a.heads2 ? 2 : 1);
  if (ctas == 0) return cudaSuccess;
  if (p.d == 64) return launch2_d<64>(a, m, (unsigned)ctas, st);
  return launch2_d<128>(a, m, (unsigned)ctas, st);
}

}  // namespace attn
