// bwd_simt.cu -- CUDA-core backward (recompute form).
//
//   pre:  D_i = dO_i . O_i and lse in log2 units per (row, head);
//   dq:   one warp per (query row, head) walks the row's allowed keys,
//         recomputes P_ij = 2^(c s_ij - lse2_i), dS_ij = P_ij (dO_i.v_j - D_i)
//         and sums dQ_i = scale sum_j dS_ij k_j;
//   dkdv: one warp per (key, KV head) walks every query head of its group
//         and every row allowed to see the key, summing
//         dK_j = scale sum dS_ij q_i and dV_j = sum P_ij dO_i, so the GQA sum
//         over shared heads happens in registers.
// The same per-row key bound as the forward decides every pair
// ("causal-mask-and-ragged-sequence-layouts", sixth paragraph: backward
// recomputation rebuilds the same mask).  No atomics: each output row has one
// owner warp, so the result is deterministic.
#include <cuda_fp16.h>

#include "common.cuh"

namespace attn {

template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_pre_kernel(BwdParams p) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + warp;  // t * hq + h
  if (row >= (long long)p.total_q * p.hq) return;
  const int t = (int)(row / p.hq), h = (int)(row % p.hq);
  const T *op = reinterpret_cast<const T *>(p.o) + toff(p.so, t, h) + lane * E;
  const T *dp = reinterpret_cast<const T *>(p.dout) + toff(p.sdo, t, h) + lane * E;
  float part = 0.f;
  if (p.delta_ready) {
    // D comes from the recomputing forward
  } else if (p.o_f32) {
    const float *of = p.o_f32 + (size_t)row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e++) part += of[e] * Elem<T>::to_f(dp[e]);
  } else {
#pragma unroll
    for (int e = 0; e < E; e++) part += Elem<T>::to_f(op[e]) * Elem<T>::to_f(dp[e]);
  }
  const float D_i = warp_sum(part);
  if (p.q16) {
    // scaled fp16 copies for the tensor-core backward (exact: a power of two)
    const float fq = exp2_int(f16_copy_exponent(p.amax[kAmaxQ]));
    const float fdo = exp2_int(f16_copy_exponent(p.amax[kAmaxDO]));
    const T *qp = reinterpret_cast<const T *>(p.q) + toff(p.sq, t, h) + lane * E;
    __half *q16 = reinterpret_cast<__half *>(p.q16) + (size_t)row * D + lane * E;
    __half *d16 = reinterpret_cast<__half *>(p.do16) + (size_t)row * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e++) {
      q16[e] = __float2half_rn(Elem<T>::to_f(qp[e]) * fq);
      d16[e] = __float2half_rn(Elem<T>::to_f(dp[e]) * fdo);
    }
  }
  if (lane == 0) {
    const float l = p.lse[(size_t)h * p.total_q + t];
    if (!p.delta_ready) p.delta[(size_t)h * p.total_q + t] = D_i;
    // An empty row (lse = -inf) gets +inf so that 2^(s - lse2) = 0.
    p.lse2[(size_t)h * p.total_q + t] = l == -INFINITY ? INFINITY : l * kLog2e;
  }
}

// The same for bf16 inputs with 8- or 16-byte aligned rows: every lane moves
// its D / 32 consecutive elements with one vector access per tensor.
template <int D>
__global__ void __launch_bounds__(128) bwd_pre_vec_kernel(BwdParams p) {
  constexpr int E = D / 32;  // 4 (one 8-byte bf16 vector) or 2 (4 bytes)
  static_assert(E == 2 || E == 4, "d = 64 or 128");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * 4 + warp;  // t * hq + h
  if (row >= (long long)p.total_q * p.hq) return;
  const int t = (int)(row / p.hq), h = (int)(row % p.hq);
  const __nv_bfloat16 *base_do = reinterpret_cast<const __nv_bfloat16 *>(p.dout);
  const __nv_bfloat16 *base_q = reinterpret_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *base_o = reinterpret_cast<const __nv_bfloat16 *>(p.o);
  uint32_t dw[E / 2], qw[E / 2], ow[E / 2];  // bf16 pairs
  auto load_pairs = [&](const __nv_bfloat16 *src, uint32_t *w) {
    if constexpr (E == 4) {
      const uint2 v = *reinterpret_cast<const uint2 *>(src);
      w[0] = v.x;
      w[1] = v.y;
    } else {
      w[0] = *reinterpret_cast<const uint32_t *>(src);
    }
  };
  load_pairs(base_do + toff(p.sdo, t, h) + lane * E, dw);
  float dof[E];
#pragma unroll
  for (int k = 0; k < E / 2; k++) {
    dof[2 * k] = __uint_as_float(dw[k] << 16);
    dof[2 * k + 1] = __uint_as_float(dw[k] & 0xFFFF0000u);
  }
  float part = 0.f;
  if (p.delta_ready) {
    // D comes from the recomputing forward
  } else if (p.o_f32) {
    const float *of = p.o_f32 + (size_t)row * D + lane * E;
    float o[E];
    if constexpr (E == 4) {
      const float4 v = *reinterpret_cast<const float4 *>(of);
      o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2 *>(of);
      o[0] = v.x; o[1] = v.y;
    }
#pragma unroll
    for (int e = 0; e < E; e++) part += o[e] * dof[e];
  } else {
    load_pairs(base_o + toff(p.so, t, h) + lane * E, ow);
#pragma unroll
    for (int k = 0; k < E / 2; k++) {
      part += __uint_as_float(ow[k] << 16) * dof[2 * k];
      part += __uint_as_float(ow[k] & 0xFFFF0000u) * dof[2 * k + 1];
    }
  }
  const float D_i = warp_sum(part);
  // scaled fp16 copies of q and dout (exact: a power of two, see
  // f16_copy_exponent)
  const float fq = exp2_int(f16_copy_exponent(p.amax[kAmaxQ]));
  const float fdo = exp2_int(f16_copy_exponent(p.amax[kAmaxDO]));
  load_pairs(base_q + toff(p.sq, t, h) + lane * E, qw);
  uint32_t q16[E / 2], d16[E / 2];
#pragma unroll
  for (int k = 0; k < E / 2; k++) {
    const float a0 = __uint_as_float(qw[k] << 16) * fq, a1 = __uint_as_float(qw[k] & 0xFFFF0000u) * fq;
    const __half2 qa = __floats2half2_rn(a0, a1),
                  da = __floats2half2_rn(dof[2 * k] * fdo, dof[2 * k + 1] * fdo);
    q16[k] = *reinterpret_cast<const uint32_t *>(&qa);
    d16[k] = *reinterpret_cast<const uint32_t *>(&da);
  }
  __half *q16p = reinterpret_cast<__half *>(p.q16) + (size_t)row * D + lane * E;
  __half *d16p = reinterpret_cast<__half *>(p.do16) + (size_t)row * D + lane * E;
  if constexpr (E == 4) {
    *reinterpret_cast<uint2 *>(q16p) = make_uint2(q16[0], q16[1]);
    *reinterpret_cast<uint2 *>(d16p) = make_uint2(d16[0], d16[1]);
  } else {
    *reinterpret_cast<uint32_t *>(q16p) = q16[0];
    *reinterpret_cast<uint32_t *>(d16p) = d16[0];
  }
  if (lane == 0) {
    const float l = p.lse[(size_t)h * p.total_q + t];
    if (!p.delta_ready) p.delta[(size_t)h * p.total_q + t] = D_i;
    p.lse2[(size_t)h * p.total_q + t] = l == -INFINITY ? INFINITY : l * kLog2e;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_dq_simt_kernel(BwdParams p) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, h = blockIdx.y;
  const int i = blockIdx.x * 4 + warp;
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
  const T *dop = reinterpret_cast<const T *>(p.dout) + toff(p.sdo, t, h) + lane * E;
  float qf[E], dof[E], dq[E];
#pragma unroll
  for (int e = 0; e < E; e++) {
    qf[e] = Elem<T>::to_f(qp[e]) * p.scale_log2;
    dof[e] = Elem<T>::to_f(dop[e]);
    dq[e] = 0.f;
  }
  const float lse2 = p.lse2[(size_t)h * p.total_q + t];
  const float D_i = p.delta[(size_t)h * p.total_q + t];
  const int kbeg = key_begin(g.mask, g.window, i, g.nq, g.nk);
  const int kend = key_end(g.mask, i, g.nq, g.nk);
  const float slope2 = p.slopes ? __ldg(p.slopes + h) * kLog2e : 0.f;
  const float bound = (float)(i + causal_offset(g.mask, g.nq, g.nk));
  const float *brow = btab_row(p.btab, p.bss, p.bhs, p.brs, s, h, i);  // explicit bias row
  const T *kb = reinterpret_cast<const T *>(p.k) + toff(p.sk, g.k0, hk) + lane * E;
  const T *vb = reinterpret_cast<const T *>(p.v) + toff(p.sv, g.k0, hk) + lane * E;
  const size_t kstride = (size_t)p.sk.ts, vstride = (size_t)p.sv.ts;  // one key to the next
  for (int j = kbeg; j < kend; j++) {
    float kf[E], ps = 0.f, pd = 0.f;
#pragma unroll
    for (int e = 0; e < E; e++) {
      kf[e] = Elem<T>::to_f(kb[j * kstride + e]);
      ps += qf[e] * kf[e];
      pd += dof[e] * Elem<T>::to_f(vb[j * vstride + e]);
    }
    const float sc = warp_sum(ps) + pos_bias2(slope2, bound, j) +
                     (brow ? __ldg(brow + j) * kLog2e : 0.f),
                dpij = warp_sum(pd);
    const float pij = fast_exp2(sc - lse2);
    const float ds = pij * (dpij - D_i);
#pragma unroll
    for (int e = 0; e < E; e++) dq[e] += ds * kf[e];
  }
  T *out = reinterpret_cast<T *>(p.dq) + toff(p.sdq, t, h) + lane * E;
#pragma unroll
  for (int e = 0; e < E; e++) out[e] = Elem<T>::from_f(dq[e] * p.scale);
}

template <typename T, int D>
__global__ void __launch_bounds__(128) bwd_dkdv_simt_kernel(BwdParams p) {
  constexpr int E = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.z, hk = blockIdx.y;
  const int j = blockIdx.x * 4 + warp;  // in-sequence key
  SeqGeom g = load_seq(p.cu_q, p.cu_k, s, p.total_q, p.total_k, p.max_q, p.max_k, p.mask, p.window);
  if (!g.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
      raise_error(p.err, ATTN_ERR_DEVICE_BOUNDS);
    return;
  }
  if (j >= g.nk) return;
  const int grp = p.hq / p.hkv;
  const T *kp = reinterpret_cast<const T *>(p.k) + toff(p.sk, g.k0 + j, hk) + lane * E;
  const T *vp = reinterpret_cast<const T *>(p.v) + toff(p.sv, g.k0 + j, hk) + lane * E;
  float kf[E], vf[E], dk[E], dv[E];
#pragma unroll
  for (int e = 0; e < E; e++) {
    kf[e] = Elem<T>::to_f(kp[e]) * p.scale_log2;
    vf[e] = Elem<T>::to_f(vp[e]);
    dk[e] = 0.f;
    dv[e] = 0.f;
  }
  const int i_begin = row_begin(g.mask, j, g.nq, g.nk);
  const int i_end = row_end(g.mask, g.window, j, g.nq, g.nk);
  const int off = causal_offset(g.mask, g.nq, g.nk);
  for (int h = hk * grp; h < hk * grp + grp; h++) {
    const float slope2 = p.slopes ? __ldg(p.slopes + h) * kLog2e : 0.f;
    for (int i = i_begin; i < i_end; i++) {
      const int t = g.q0 + i;
      const T *qp = reinterpret_cast<const T *>(p.q) + toff(p.sq, t, h) + lane * E;
      const T *dop = reinterpret_cast<const T *>(p.dout) + toff(p.sdo, t, h) + lane * E;
      float qf[E], dof[E], ps = 0.f, pd = 0.f;
#pragma unroll
      for (int e = 0; e < E; e++) {
        qf[e] = Elem<T>::to_f(qp[e]);
        dof[e] = Elem<T>::to_f(dop[e]);
        ps += qf[e] * kf[e];
        pd += dof[e] * vf[e];
      }
      const float *brow = btab_row(p.btab, p.bss, p.bhs, p.brs, s, h, i);
      const float sc = warp_sum(ps) + pos_bias2(slope2, (float)(i + off), j) +
                       (brow ? __ldg(brow + j) * kLog2e : 0.f),
                  dpij = warp_sum(pd);
      const float lse2 = p.lse2[(size_t)h * p.total_q + t];
      const float D_i = p.delta[(size_t)h * p.total_q + t];
      const float pij = fast_exp2(sc - lse2);
      const float ds = pij * (dpij - D_i);
#pragma unroll
      for (int e = 0; e < E; e++) {
        dk[e] += ds * qf[e];
        dv[e] += pij * dof[e];
      }
    }
  }
  T *dkp = reinterpret_cast<T *>(p.dk) + toff(p.sdk, g.k0 + j, hk) + lane * E;
  T *dvp = reinterpret_cast<T *>(p.dv) + toff(p.sdv, g.k0 + j, hk) + lane * E;
#pragma unroll
  for (int e = 0; e < E; e++) {
    dkp[e] = Elem<T>::from_f(dk[e] * p.scale);
    dvp[e] = Elem<T>::from_f(dv[e]);
  }
}

template <typename T, int D>
static void launch_all(const BwdParams &p, cudaStream_t st) {
  const long long rows = (long long)p.total_q * p.hq;
  if (rows > 0) bwd_pre_kernel<T, D><<<(unsigned)((rows + 3) / 4), 128, 0, st>>>(p);
  if (p.max_q > 0)
    bwd_dq_simt_kernel<T, D><<<dim3((p.max_q + 3) / 4, p.hq, p.batch), 128, 0, st>>>(p);
  if (p.max_k > 0)
    bwd_dkdv_simt_kernel<T, D><<<dim3((p.max_k + 3) / 4, p.hkv, p.batch), 128, 0, st>>>(p);
}

// K and V (any token / head strides) -> contiguous scaled fp16 copies for the
// tensor-core backward (see f16_copy_exponent), 8 elements a thread.
__global__ void __launch_bounds__(256) kv_to_f16_kernel(const __nv_bfloat16 *__restrict__ k,
                                                        const __nv_bfloat16 *__restrict__ v,
                                                        __half *__restrict__ k16,
                                                        __half *__restrict__ v16, size_t n8,
                                                        int hkv, int d, Strides sk, Strides sv,
                                                        const unsigned int *__restrict__ amax) {
  const float fk = exp2_int(f16_copy_exponent(amax[kAmaxK]));
  const float fv = exp2_int(f16_copy_exponent(amax[kAmaxV]));
  const int per_row = d / 8;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < 2 * n8;
       i += (size_t)gridDim.x * blockDim.x) {
    const bool is_v = i >= n8;
    const size_t j = is_v ? i - n8 : i;              // 8-element unit of the copy
    const size_t row = j / per_row, c8 = j % per_row;  // row = token * hkv + head
    const long long t = (long long)(row / hkv), hk = (long long)(row % hkv);
    const __nv_bfloat16 *src = (is_v ? v + toff(sv, t, hk) : k + toff(sk, t, hk)) + c8 * 8;
    const uint4 in = *reinterpret_cast<const uint4 *>(src);
    const __nv_bfloat16 *x = reinterpret_cast<const __nv_bfloat16 *>(&in);
    uint4 out;
    __half *y = reinterpret_cast<__half *>(&out);
    const float f = is_v ? fv : fk;
#pragma unroll
    for (int e = 0; e < 8; e++) y[e] = __float2half_rn(__bfloat162float(x[e]) * f);
    reinterpret_cast<uint4 *>(is_v ? v16 : k16)[j] = out;
  }
}

// Largest |x| of one [T, H, d] bf16 tensor as a bit pattern (sign cleared),
// 8 elements (16 bytes) per step; contiguous tensors take a flat walk.
struct AmaxJob {
  const __nv_bfloat16 *base;
  long long n8;  // 16-byte units
  int heads, per_row;  // per_row = d / 8
  Strides s;
  bool flat;
};
struct AmaxArgs {
  AmaxJob job[4];  // q, k, v, dout
  unsigned int *amax;
  int *err;
};

__device__ __forceinline__ unsigned int max_bits8(const uint4 w) {
  const unsigned int a = max(w.x & 0x7fffu, (w.x >> 16) & 0x7fffu);
  const unsigned int b = max(w.y & 0x7fffu, (w.y >> 16) & 0x7fffu);
  const unsigned int c = max(w.z & 0x7fffu, (w.z >> 16) & 0x7fffu);
  const unsigned int e = max(w.w & 0x7fffu, (w.w >> 16) & 0x7fffu);
  return max(max(a, b), max(c, e));
}

// amax[t] = max over tensor t of |x| (bf16 bits, sign cleared; the caller
// zeroes amax first); an infinity or NaN anywhere sets ATTN_ERR_DEVICE_RANGE.
// Four independent 16-byte loads per thread and step keep enough bytes in
// flight; one atomic per block and tensor (a per-warp atomic on one address
// serialised tens of thousands of them).
__global__ void __launch_bounds__(256) bwd_amax_kernel(const AmaxArgs a) {
  __shared__ unsigned int part[4][8];
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t first = blockIdx.x * (size_t)blockDim.x + threadIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 1
  for (int t = 0; t < 4; t++) {
    const AmaxJob &j = a.job[t];
    const size_t n = (size_t)j.n8;
    unsigned int m = 0;
    if (j.flat) {
      const uint4 *src = reinterpret_cast<const uint4 *>(j.base);
      size_t i = first;
      for (; i + 3 * stride < n; i += 4 * stride) {
        const uint4 w0 = __ldg(src + i), w1 = __ldg(src + i + stride);
        const uint4 w2 = __ldg(src + i + 2 * stride), w3 = __ldg(src + i + 3 * stride);
        m = max(m, max(max(max_bits8(w0), max_bits8(w1)), max(max_bits8(w2), max_bits8(w3))));
      }
      for (; i < n; i += stride) m = max(m, max_bits8(__ldg(src + i)));
    } else {
      for (size_t i = first; i < n; i += stride) {
        const size_t row = i / j.per_row, c8 = i % j.per_row;
        const long long tok = (long long)(row / j.heads), h = (long long)(row % j.heads);
        m = max(m, max_bits8(__ldg(reinterpret_cast<const uint4 *>(j.base + toff(j.s, tok, h)) + c8)));
      }
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) part[t][warp] = m;
  }
  __syncthreads();
  if (threadIdx.x < 4) {
    const int t = threadIdx.x;
    unsigned int m = 0;
    for (int w = 0; w < 8; w++) m = max(m, part[t][w]);
    if (m != 0) {
      if (bf16_bits_nonfinite(m)) raise_error(a.err, ATTN_ERR_DEVICE_RANGE);
      atomicMax(a.amax + t, m);
    }
  }
}

cudaError_t launch_bwd_amax(const BwdParams &p, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(p.amax, 0, 4 * sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  AmaxArgs a;
  const void *base[4] = {p.q, p.k, p.v, p.dout};
  const Strides *str[4] = {&p.sq, &p.sk, &p.sv, &p.sdo};
  const int heads[4] = {p.hq, p.hkv, p.hkv, p.hq};
  const int tok[4] = {p.total_q, p.total_k, p.total_k, p.total_q};
  long long most = 0;
  for (int t = 0; t < 4; t++) {
    AmaxJob &j = a.job[t];
    j.base = static_cast<const __nv_bfloat16 *>(base[t]);
    j.heads = heads[t];
    j.per_row = p.d / 8;
    j.s = *str[t];
    j.n8 = (long long)tok[t] * heads[t] * p.d / 8;
    j.flat = j.s.hs == p.d && j.s.ts == (long long)heads[t] * p.d;
    if (j.n8 > most) most = j.n8;
  }
  a.amax = p.amax;
  a.err = p.err;
  if (most == 0) return cudaSuccess;
  long long blocks = (most + 4 * 256 - 1) / (4 * 256);  // four 16-byte loads per thread
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long cap = 8LL * (sms > 0 ? sms : 152);  // 8 blocks of 256 per SM: one full wave
  if (blocks > cap) blocks = cap;
  bwd_amax_kernel<<<(unsigned)blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_kv_to_f16(const BwdParams &p, cudaStream_t st) {
  const size_t n8 = (size_t)p.total_k * p.hkv * p.d / 8;
  if (n8 == 0) return cudaSuccess;
  size_t blocks = (2 * n8 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  kv_to_f16_kernel<<<(unsigned)blocks, 256, 0, st>>>(
      reinterpret_cast<const __nv_bfloat16 *>(p.k), reinterpret_cast<const __nv_bfloat16 *>(p.v),
      reinterpret_cast<__half *>(p.k16), reinterpret_cast<__half *>(p.v16), n8, p.hkv, p.d, p.sk,
      p.sv, p.amax);
  return cudaGetLastError();
}

// Zero every (token, head) row of a [T, H, d] tensor with any strides, 16
// bytes a thread (d * element size is a multiple of 16 for d = 64 or 128).
__global__ void __launch_bounds__(256) zero_rows_kernel(char *base, size_t n16, int h, int row_bytes,
                                                        Strides s, int elem) {
  const int per_row = row_bytes / 16;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
       i += (size_t)gridDim.x * blockDim.x) {
    const size_t row = i / per_row, c16 = i % per_row;
    const long long t = (long long)(row / h), hh = (long long)(row % h);
    *reinterpret_cast<uint4 *>(base + toff(s, t, hh) * elem + c16 * 16) = make_uint4(0, 0, 0, 0);
  }
}

cudaError_t launch_zero_rows(void *base, int T, int H, int d, Strides s, int elem,
                             cudaStream_t st) {
  const size_t n16 = (size_t)T * H * d * elem / 16;
  if (n16 == 0) return cudaSuccess;
  size_t blocks = (n16 + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  zero_rows_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<char *>(base), n16, H, d * elem,
                                                      s, elem);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(const BwdParams &p, attn_dtype dtype, cudaStream_t st) {
  const long long rows = (long long)p.total_q * p.hq;
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)((rows + 3) / 4);
  if (dtype == ATTN_DTYPE_FP32) {
    if (p.d == 64) bwd_pre_kernel<float, 64><<<blocks, 128, 0, st>>>(p);
    else bwd_pre_kernel<float, 128><<<blocks, 128, 0, st>>>(p);
  } else {
    // vector accesses need q, dout, o (or o_f32) aligned to a whole lane's
    // share of a row: 8 bytes (bf16) and 16 bytes (fp32) at d = 128
    const uintptr_t a = reinterpret_cast<uintptr_t>(p.q) | reinterpret_cast<uintptr_t>(p.dout) |
                        (p.o_f32 ? 0 : reinterpret_cast<uintptr_t>(p.o));
    const uintptr_t af = reinterpret_cast<uintptr_t>(p.o_f32);
    const bool vec = p.q16 && (a & (p.d / 16 - 1)) == 0 && (af & (p.d / 8 - 1)) == 0;
    if (vec) {
      if (p.d == 64) bwd_pre_vec_kernel<64><<<blocks, 128, 0, st>>>(p);
      else bwd_pre_vec_kernel<128><<<blocks, 128, 0, st>>>(p);
    } else {
      if (p.d == 64) bwd_pre_kernel<__nv_bfloat16, 64><<<blocks, 128, 0, st>>>(p);
      else bwd_pre_kernel<__nv_bfloat16, 128><<<blocks, 128, 0, st>>>(p);
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(const BwdParams &p, attn_dtype dtype, cudaStream_t st) {
  if (p.batch == 0) return cudaSuccess;
  if (dtype == ATTN_DTYPE_FP32) {
    if (p.d == 64) launch_all<float, 64>(p, st);
    else launch_all<float, 128>(p, st);
  } else {
    if (p.d == 64) launch_all<__nv_bfloat16, 64>(p, st);
    else launch_all<__nv_bfloat16, 128>(p, st);
  }
  return cudaGetLastError();
}

}  // namespace attn
