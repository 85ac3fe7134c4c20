// combine.cu -- merges the per-split partial results of the split-KV forward.
// Each split s of a row holds O_s (already divided by its own denominator)
// and lse_s (log2 units, -inf when the split saw no allowed key).  With
// M = max_s lse_s and w_s = 2^(lse_s - M): O = sum_s w_s O_s / sum_s w_s and
// lse = M + log2(sum_s w_s); a row no split saw gets O = 0, lse = -inf
// ("causal-mask-and-ragged-sequence-layouts", fourth paragraph).
#include "common.cuh"
#include "plan.h"

namespace attn {

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(FwdParams p) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 8 + warp;  // t * hq + h
  const long long rows = (long long)p.total_q * p.hq;
  if (row >= rows) return;
  const int t = (int)(row / p.hq), h = (int)(row % p.hq);
  float M = -INFINITY;
  for (int s = 0; s < p.n_splits; s++)
    M = fmaxf(M, p.lse_part[((size_t)s * p.hq + h) * p.total_q + t]);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; e++) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < p.n_splits; s++) {
      const float ls = p.lse_part[((size_t)s * p.hq + h) * p.total_q + t];
      if (ls == -INFINITY) continue;
      const float w = fast_exp2(ls - M);
      wsum += w;
      const float4 *src = reinterpret_cast<const float4 *>(
          p.o_part + ((size_t)s * rows + row) * D + lane * E);
#pragma unroll
      for (int e4 = 0; e4 < E / 4; e4++) {
        float4 x = src[e4];
        acc[4 * e4 + 0] += w * x.x;
        acc[4 * e4 + 1] += w * x.y;
        acc[4 * e4 + 2] += w * x.z;
        acc[4 * e4 + 3] += w * x.w;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(p.o) + toff(p.so, t, h) + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<__nv_bfloat162 *>(op + e) =
        __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
  if (p.o_f32) {
    float *of = p.o_f32 + (size_t)row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e++) of[e] = acc[e] * inv;
  }
  if (p.lse && lane == 0)
    p.lse[(size_t)h * p.total_q + t] = wsum > 0.f ? (M + log2f(wsum)) * kLn2 : -INFINITY;
}

cudaError_t launch_combine(const FwdParams &p, const TcPlan &plan, cudaStream_t st) {
  (void)plan;
  const long long rows = (long long)p.total_q * p.hq;
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  if (p.d == 64) combine_kernel<64><<<blocks, 256, 0, st>>>(p);
  else combine_kernel<128><<<blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
