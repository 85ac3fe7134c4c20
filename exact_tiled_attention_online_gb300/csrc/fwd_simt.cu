// fwd_simt.cu -- CUDA-core forward: one warp per (query row, head), the keys
// of the row's allowed interval streamed in order through the online-softmax
// recurrence ("formal-correctness", "The FlashAttention Proof": running max,
// rescale of denominator and accumulator when the max moves, final divide).
//
// This is the fp32 path (fp32 inputs have no tensor-core kind that keeps fp32
// operands exact) and the small-problem path; each lane owns head_dim/32
// consecutive features, so every key row is read with one coalesced access
// and the score is a warp-wide reduction of lane-partial products.
#include "common.cuh"

namespace attn {

template <typename T, int D>
__global__ void __launch_bounds__(128) fwd_simt_kernel(FwdParams p) {
  constexpr int E = D / 32;  // features per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, h = blockIdx.y;
  const int i = blockIdx.x * 4 + warp;  // in-sequence query row
  SeqGeom g = load_seq(p.cu_q, p.cu_k, s, p.total_q, p.total_k, p.max_q, p.max_k, p.mask, p.window);
  if (!g.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
      raise_error(p.err, ATTN_ERR_DEVICE_BOUNDS);
    return;
  }
  if (i >= g.nq) return;
  const int hk = h / (p.hq / p.hkv);
  const int t = g.q0 + i;
  const T *qp = reinterpret_cast<const T *>(p.q) + toff(p.sq, t, h) + lane * E;
  float qf[E], acc[E];
#pragma unroll
  for (int e = 0; e < E; e++) {
    qf[e] = Elem<T>::to_f(qp[e]) * p.scale_log2;
    acc[e] = 0.f;
  }
  const int kbeg = key_begin(g.mask, g.window, i, g.nq, g.nk);
  const int kend = key_end(g.mask, i, g.nq, g.nk);
  // positional bias: key j is |bound - j| away from the row's causal bound
  const float slope2 = p.slopes ? __ldg(p.slopes + h) * kLog2e : 0.f;
  const float bound = (float)(i + causal_offset(g.mask, g.nq, g.nk));
  // explicit bias tensor row (natural-log units), or NULL
  const float *brow = btab_row(p.btab, p.bss, p.bhs, p.brs, s, h, i);
  float m = -INFINITY, l = 0.f;
  const T *kb = reinterpret_cast<const T *>(p.k) + toff(p.sk, g.k0, hk) + lane * E;
  const T *vb = reinterpret_cast<const T *>(p.v) + toff(p.sv, g.k0, hk) + lane * E;
  const size_t kstride = (size_t)p.sk.ts, vstride = (size_t)p.sv.ts;  // one key to the next
  for (int j = kbeg; j < kend; j++) {
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < E; e++) part += qf[e] * Elem<T>::to_f(kb[j * kstride + e]);
    float sc = warp_sum(part) + pos_bias2(slope2, bound, j);  // logit in log2 units
    if (brow) {
      sc += __ldg(brow + j) * kLog2e;
      if (sc == -INFINITY) continue;  // masked by the tensor: P = 0, state unchanged
    }
    const float m_new = fmaxf(m, sc);
    const float alpha = fast_exp2(m - m_new);
    const float pj = fast_exp2(sc - m_new);
    l = l * alpha + pj;
#pragma unroll
    for (int e = 0; e < E; e++) acc[e] = acc[e] * alpha + pj * Elem<T>::to_f(vb[j * vstride + e]);
    m = m_new;
  }
  T *op = reinterpret_cast<T *>(p.o) + toff(p.so, t, h) + lane * E;
  // l > 0 iff some key had a finite logit (the largest contributes 1)
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int e = 0; e < E; e++) op[e] = Elem<T>::from_f(acc[e] * inv);
  if (p.o_f32) {
    float *of = p.o_f32 + ((size_t)t * p.hq + h) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e++) of[e] = acc[e] * inv;
  }
  if (p.lse && lane == 0)
    p.lse[(size_t)h * p.total_q + t] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

cudaError_t launch_fwd_simt(const FwdParams &p, attn_dtype dtype, cudaStream_t st) {
  dim3 grid((p.max_q + 3) / 4, p.hq, p.batch), block(128);
  if (grid.x == 0 || p.batch == 0) return cudaSuccess;
  if (dtype == ATTN_DTYPE_FP32) {
    if (p.d == 64) fwd_simt_kernel<float, 64><<<grid, block, 0, st>>>(p);
    else fwd_simt_kernel<float, 128><<<grid, block, 0, st>>>(p);
  } else {
    if (p.d == 64) fwd_simt_kernel<__nv_bfloat16, 64><<<grid, block, 0, st>>>(p);
    else fwd_simt_kernel<__nv_bfloat16, 128><<<grid, block, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace attn
