// common.cuh -- device helpers shared by every attention kernel: sequence
// lookup from cumulative lengths, the alignment rule as a per-row key bound,
// the device error flag, bf16 conversions and bounded mbarrier waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/attn.h"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Sequence geometry ("causal-mask-and-ragged-sequence-layouts", first and
// third paragraphs).  Every alignment rule allows, for query row i of a
// sequence, one interval of that sequence's keys: key_begin(i) <= j <
// key_end(i), a prefix (key_begin = 0) unless a bounded window keeps only
// the last `window` positions up to the causal bound ("attention-algorithm-
// error-and-complexity-tests", fifth paragraph).  Both ends are
// non-decreasing in i.  Tiles take in-sequence coordinates (row i, key j)
// before any comparison, so a packed global offset never becomes a position.
// ---------------------------------------------------------------------------
struct SeqGeom {
  int q0, nq;  // first packed query token, number of queries
  int k0, nk;  // first packed key token, number of keys
  int mask;    // attn_mask_kind
  int window;  // > 0: bounded window of that many keys (causal kinds only)
  bool ok;     // cu_seqlens consistent with the sizes passed
};

__device__ __forceinline__ SeqGeom load_seq(const int32_t *__restrict__ cu_q,
                                            const int32_t *__restrict__ cu_k,
                                            int s, int total_q, int total_k,
                                            int max_q, int max_k, int mask, int window) {
  SeqGeom g;
  g.q0 = __ldg(cu_q + s);
  int q1 = __ldg(cu_q + s + 1);
  g.k0 = __ldg(cu_k + s);
  int k1 = __ldg(cu_k + s + 1);
  g.nq = q1 - g.q0;
  g.nk = k1 - g.k0;
  g.mask = mask;
  g.window = window;
  g.ok = g.q0 >= 0 && g.k0 >= 0 && g.nq >= 0 && g.nk >= 0 && q1 <= total_q &&
         k1 <= total_k && g.nq <= max_q && g.nk <= max_k;
  if (!g.ok) {
    g.nq = 0;
    g.nk = 0;
  }
  return g;
}

// Shift of the causal diagonal: key j is allowed for row i iff j <= i + off.
__host__ __device__ __forceinline__ int causal_offset(int mask, int nq, int nk) {
  return mask == ATTN_CAUSAL_BOTTOM_RIGHT ? nk - nq : 0;
}

// Exclusive end of the allowed key prefix of in-sequence row i (0 = empty).
__host__ __device__ __forceinline__ int key_end(int mask, int i, int nq, int nk) {
  if (mask == ATTN_MASK_NONE) return nk;
  int e = i + causal_offset(mask, nq, nk) + 1;
  return e < 0 ? 0 : (e > nk ? nk : e);
}

// First allowed key of in-sequence row i: 0 without a window, else the
// first of the `window` positions that end at the causal bound i + off.
__host__ __device__ __forceinline__ int key_begin(int mask, int window, int i, int nq, int nk) {
  if (mask == ATTN_MASK_NONE || window <= 0) return 0;
  int b = i + causal_offset(mask, nq, nk) + 1 - window;
  return b < 0 ? 0 : (b > nk ? nk : b);
}

// First in-sequence query row that is allowed to see key j (rows below it do
// not); rows >= nq are out of range.
__host__ __device__ __forceinline__ int row_begin(int mask, int j, int nq, int nk) {
  if (mask == ATTN_MASK_NONE) return 0;
  int b = j - causal_offset(mask, nq, nk);
  return b < 0 ? 0 : b;
}

// Exclusive end of the query rows that see key j: a window drops every row
// whose causal bound lies `window` or more positions past j.
__host__ __device__ __forceinline__ int row_end(int mask, int window, int j, int nq, int nk) {
  if (mask == ATTN_MASK_NONE || window <= 0) return nq;
  int e = j - causal_offset(mask, nq, nk) + window;
  return e < 0 ? 0 : (e > nq ? nq : e);
}

// ---------------------------------------------------------------------------
// Tile planner.  A tile holds in-sequence query rows [i0, i0 + rows) (rows
// past nq are out-of-range lanes) against key tiles of bn keys.  Because both
// ends of a row's key interval are non-decreasing in i, the tile needs key
// tiles [n_begin, n_end): n_begin from its first row's start and n_end from
// its last in-range row's end.  Key tiles in [n_full_begin, n_full_end) lie
// inside every in-range row's interval, so they need no per-element mask.
// ---------------------------------------------------------------------------
struct KvRange {
  int n_begin, n_end;            // key tiles holding every allowed key of the tile
  int n_full_begin, n_full_end;  // key tiles allowed for every in-range row
  __host__ __device__ bool full(int n) const { return n >= n_full_begin && n < n_full_end; }
};

__host__ __device__ __forceinline__ KvRange plan_kv_tiles(int mask, int window, int nq, int nk,
                                                           int i0, int rows, int bn) {
  KvRange r{0, 0, 0, 0};
  int i_last = (i0 + rows < nq ? i0 + rows : nq) - 1;
  if (i_last < i0) return r;
  const int kb_first = key_begin(mask, window, i0, nq, nk);
  const int kb_last = key_begin(mask, window, i_last, nq, nk);
  const int ke_first = key_end(mask, i0, nq, nk);
  const int ke_last = key_end(mask, i_last, nq, nk);
  r.n_begin = kb_first / bn;
  r.n_end = (ke_last + bn - 1) / bn;
  if (r.n_end < r.n_begin) r.n_end = r.n_begin;
  r.n_full_begin = (kb_last + bn - 1) / bn;
  r.n_full_end = ke_first / bn;
  return r;
}

// Key tiles [*a, *b) of split `split` out of n_splits over [n_begin, n_end).
__host__ __device__ __forceinline__ void split_tiles(int n_begin, int n_end, int split,
                                                     int n_splits, int *a, int *b) {
  const int n = n_end - n_begin;
  int per = (n + n_splits - 1) / n_splits;
  int lo = split * per;
  *a = n_begin + (lo < n ? lo : n);
  *b = n_begin + (lo + per < n ? lo + per : n);
}

// Per-lane predicate on a boundary tile, hoisted per row: lane (row i, key j)
// is allowed iff row_key_first(i) <= j < row_key_limit(i).  Out-of-range rows
// get a limit of 0, so none of their lanes are allowed; keys past the
// sequence end are never allowed because key_end() <= nk.
__host__ __device__ __forceinline__ int row_key_limit(int mask, int i, int nq, int nk) {
  return i < nq ? key_end(mask, i, nq, nk) : 0;
}

__host__ __device__ __forceinline__ int row_key_first(int mask, int window, int i, int nq,
                                                      int nk) {
  return i < nq ? key_begin(mask, window, i, nq, nk) : 0;
}

__host__ __device__ __forceinline__ bool lane_allowed(int mask, int window, int i, int j, int nq,
                                                      int nk) {
  return j >= row_key_first(mask, window, i, nq, nk) && j < row_key_limit(mask, i, nq, nk);
}

// The same predicate hoisted per key (the backward's transposed tiles): lane
// (row i, key j) is allowed iff key_row_begin(j) <= i < key_row_end(j).  For
// j >= nk no row is allowed.
__host__ __device__ __forceinline__ int key_row_begin(int mask, int j, int nq, int nk) {
  return j < nk ? row_begin(mask, j, nq, nk) : nq;
}

__host__ __device__ __forceinline__ int key_row_end(int mask, int window, int j, int nq, int nk) {
  return j < nk ? row_end(mask, window, j, nq, nk) : 0;
}

// Linear positional bias in log2 units for in-sequence row i and key j:
// -slope2 * |i + off - j|, the distance from the row's causal bound (0 for the
// key at the bound), with slope2 = slope * log2(e).  `dist0` is i + off minus
// the tile's first key, so key e of the tile is dist0 - e away.
__device__ __forceinline__ float pos_bias2(float slope2, float dist0, int e) {
  return -slope2 * fabsf(dist0 - (float)e);
}

// Row pointer into an explicit bias tensor for (sequence s, query head h,
// in-sequence row i): entry j of the row is the bias of key j, in natural-log
// units of the scaled logit.  NULL without a tensor.
__device__ __forceinline__ const float *btab_row(const float *btab, long long bss, long long bhs,
                                                 long long brs, int s, int h, int i) {
  return btab ? btab + (long long)s * bss + (long long)h * bhs + (long long)i * brs : nullptr;
}

// ---------------------------------------------------------------------------
// Device error flag: the first error code sticks until the host clears it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_error(int *flag, int code) {
  if (flag) atomicCAS(flag, 0, code);
}

// ---------------------------------------------------------------------------
// Element access for the two supported element types.
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
  static __device__ __forceinline__ float to_f(float x) { return x; }
  static __device__ __forceinline__ float from_f(float x) { return x; }
};
template <> struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Element strides of one [tokens, heads, d] tensor: (token t, head h) starts
// t * ts + h * hs elements from the base; the d features are contiguous.
struct Strides {
  long long ts, hs;
};
__host__ __device__ __forceinline__ size_t toff(const Strides &s, long long t, long long h) {
  return (size_t)(t * s.ts + h * s.hs);
}

// Kernel launch parameters common to the forward kernels.
struct FwdParams {
  const void *q, *k, *v;
  void *o;
  float *lse;
  float *o_f32;  // optional fp32 copy of the output before rounding
  const int32_t *cu_q, *cu_k;
  int batch, max_q, max_k, total_q, total_k, hq, hkv, d;
  float scale, scale_log2;  // scale and scale * log2(e)
  int mask;
  int window;             // > 0: bounded window (causal kinds only)
  const float *slopes;    // [hq] linear positional bias slopes, or NULL
  const float *btab;      // explicit bias tensor, or NULL
  long long bss, bhs, brs;  // its sequence, head and row strides (elements)
  Strides sq, sk, sv, so;  // layouts of q, k, v, o
  int *err;
  // split-KV partial outputs (NULL when the plan writes o/lse directly)
  float *o_part, *lse_part;
  int n_splits;
  // the backward's D term (fwd_tc2_delta.cu only): upstream gradient, its
  // layout, and the [hq, total_q] output
  const void *dout;
  Strides sdo;
  float *delta;
  unsigned long long wait_ns;  // bound of every device wait (0: the 2 s default)
};

struct BwdParams {
  const void *q, *k, *v, *o, *dout;
  const float *lse;
  const float *o_f32;  // optional fp32 output of the forward (NULL: use o)
  void *dq, *dk, *dv;
  const int32_t *cu_q, *cu_k;
  int batch, max_q, max_k, total_q, total_k, hq, hkv, d;
  float scale, scale_log2;
  int mask;
  int window;             // > 0: bounded window (causal kinds only)
  const float *slopes;    // [hq] linear positional bias slopes, or NULL
  const float *btab;      // explicit bias tensor, or NULL
  long long bss, bhs, brs;  // its sequence, head and row strides (elements)
  Strides sq, sk, sv, so, sdo, sdq, sdk, sdv;  // layouts of the eight [T, H, d] tensors
  int *err;
  float *delta;    // [hq, total_q]  D_i = dO_i . O_i
  float *lse2;     // [hq, total_q]  lse in log2 units (+inf for empty rows)
  int delta_ready; // D is written by the recomputing forward: the preprocess skips it
  // fp16 copies of the inputs for the tensor-core backward (NULL otherwise),
  // each scaled by a power of two (see f16_copy_exponent)
  void *q16, *do16, *k16, *v16;
  // [4] largest bf16 magnitude (bit pattern) of q, k, v, dout: the copies'
  // scale exponents follow from it
  unsigned int *amax;
  unsigned long long wait_ns;  // bound of every device wait (0: the 2 s default)
  // [total_q, hq, d] fp32 dQ accumulator of the fused backward (NULL: the
  // two-kernel backward)
  float *dqacc;
};

// ---------------------------------------------------------------------------
// Scaled fp16 copies for the tensor-core backward.  Each of q, k, v and dout
// is copied to fp16 multiplied by 2^s, with s chosen from the tensor's
// largest magnitude so that it lands in [2^(kF16Top - 1), 2^kF16Top) = [4, 8).
// A power of two changes no significand, so every bf16 element within 2^19
// of the largest keeps its exact value (bf16 has 8 significant bits, fp16
// 11 down to 2^-14 and subnormals to 2^-24), whatever the tensor's overall
// magnitude.  The kernels undo the factors exactly: scores by 2^-(s_q + s_k),
// dP by 2^-(s_v + s_do), and so on.  With every copy below 8 in magnitude,
// |dS| = P |dP - D| <= 2 d 8 8 = 16384 (d = 128), inside fp16's 65504.
// ---------------------------------------------------------------------------
constexpr int kF16Top = 3;
constexpr int kF16ExpLimit = 60;  // |s| bound: factors and their products stay normal fp32
enum { kAmaxQ = 0, kAmaxK = 1, kAmaxV = 2, kAmaxDO = 3 };

// s for a tensor whose largest |x| has the bf16 bit pattern `bits` (sign
// cleared); 0 for an all-zero tensor.  amax lies in [2^(e-1), 2^e).
__host__ __device__ __forceinline__ int f16_copy_exponent(unsigned int bits) {
  if (bits == 0) return 0;
  const int biased = (int)((bits >> 7) & 0xffu);
  int e;
  if (biased != 0) {
    e = biased - 126;  // 1.m 2^(biased - 127)
  } else {             // subnormal: m 2^-133, m in [2^(k-1), 2^k)
    int m = (int)(bits & 0x7fu), k = 0;
    while (m >> k) k++;
    e = k - 133;
  }
  int s = kF16Top - e;
  return s < -kF16ExpLimit ? -kF16ExpLimit : (s > kF16ExpLimit ? kF16ExpLimit : s);
}

// 2^s as an fp32 for |s| <= 126.
__host__ __device__ __forceinline__ float exp2_int(int s) {
  union {
    unsigned int u;
    float f;
  } c;
  c.u = (unsigned int)(127 + s) << 23;
  return c.f;
}

// true when `bits` (bf16 pattern, sign cleared) is an infinity or NaN
__host__ __device__ __forceinline__ bool bf16_bits_nonfinite(unsigned int bits) {
  return (bits & 0x7f80u) == 0x7f80u;
}

}  // namespace attn
