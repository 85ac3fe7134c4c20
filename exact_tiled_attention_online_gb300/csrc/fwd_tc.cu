// fwd_tc.cu -- tensor-core forward for bf16: TMA-staged Q/K/V tiles in shared
// memory, tcgen05 MMAs accumulating S = Q K^T and O += P V in tensor memory,
// and the online-softmax recurrence in registers between them
// ("formal-correctness", "The FlashAttention Proof": running max, rescale of
// the denominator and the accumulator when the max moves, new exponentiated
// terms, final divide).
//
// One CTA owns one tile of 128 query rows (one head and 128 tokens, or the
// `group` query heads of one KV head times 128/group tokens) against a range
// of 128-key tiles:
//   warp 0      TMA producer: Q once, then K and V tiles through a 2-stage ring;
//   warp 1      TMEM allocation and the single MMA-issuing thread;
//   warps 2..5  softmax: thread r owns tile row r (TMEM lane r), turns S into
//               bf16 probabilities P in shared memory, keeps m and l, rescales
//               O in TMEM when the reference max moves, and writes the output.
// The MMA of the next S tile overlaps the softmax of the current one, and the
// softmax's exponentials overlap the previous P V product.
//
// Lazy rescale: the reference max m only moves when a tile's max exceeds it
// by more than kRescaleLog2 (base-2 units); O and l always share the same
// reference, so O / l and lse = m + log2(l) are exact either way, and P stays
// below 2^kRescaleLog2.
//
// Masking follows the tile planner of common.cuh: key tiles in the planner's
// full range are allowed for every in-range row and skip the per-lane test;
// boundary tiles set the scores of disallowed lanes (other sequence, past the
// key range, past the causal bound, before a bounded window's start,
// out-of-range rows) to -inf before the row max ("causal-mask-and-ragged-
// sequence-layouts", second paragraph).
#include <cudaTypedefs.h>
#include <stdio.h>

#include "common.cuh"
#include "plan.h"
#include "sm100.cuh"
#include "tma_map.h"

namespace attn {
using namespace sm100;

namespace {

constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 256;  // S buffers at columns 0 and 128, O at 256

template <int D>
struct Layout {
  static constexpr int kChunk = 128 * 128;  // one [128 rows x 64 bf16] swizzled chunk
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTile;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kP = kV + kStages * kTile;
  static constexpr int kBar = kP + 2 * kChunk;  // P: [128 rows x 128 keys]
  static constexpr int kUsed = kBar + 256;
  // Ask for enough shared memory that two CTAs never share an SM: each
  // allocates all 512 TMEM columns.
  static constexpr int kAlloc = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
};

struct TcArgs {
  FwdParams p;
  int pack, group, tile_tokens, n_m_tiles, n_splits;
};

struct Bars {
  uint64_t q_full, k_full[2], v_full[2], k_empty[2], v_empty[2], s_full[2], p_full, o_done;
  uint64_t drain;     // the MMA thread's products have all completed
  uint64_t limit_ns;  // bound of every wait of this call
  uint32_t tmem_base;
  int abort;
  // for a drain after an early exit: Q fills, K / V ring fills (stage =
  // fill % 2) the producer issued, and whether the MMA thread issued any
  int filled_q, filled_k, filled_v, mma_issued;
};

static_assert(sizeof(Bars) <= 256, "barrier block fits its shared-memory slot");

__device__ __forceinline__ bool aborted(Bars *b) {
  return *reinterpret_cast<volatile int *>(&b->abort) != 0;
}

__device__ __forceinline__ bool wait_or_abort(Bars *b, uint64_t *bar, uint32_t parity, int *err) {
  if (mbar_test_wait(bar, parity)) return true;  // already complete: the cheap path
  if (aborted(b)) return false;
  if (mbar_wait(bar, parity, b->limit_ns)) return true;
  *reinterpret_cast<volatile int *>(&b->abort) = 1;
  raise_error(err, ATTN_ERR_DEVICE_TIMEOUT);
  return false;
}

// Tile row r -> (in-sequence query row i, query head h).
__device__ __forceinline__ void row_map(const TcArgs &a, int head_idx, int i0, int r, int *i,
                                        int *h) {
  if (a.pack) {
    *i = i0 + r / a.group;
    *h = head_idx * a.group + r % a.group;
  } else {
    *i = i0 + r;
    *h = head_idx;
  }
}

// kPosScale: scale > 0, so the max of the raw scores gives the max of the
// logits (the common case); otherwise the scores are scaled before the max.
template <int D, bool kPosScale, bool kBias>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const TcArgs a) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  Bars *b = reinterpret_cast<Bars *>(smem + L::kBar);
  const FwdParams &p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // One-dimensional grid, the query-tile rank slowest: every (head, split,
  // sequence) gets its last query tile (the longest causal rows) before any
  // gets a shorter one, so the block scheduler hands out the heaviest tiles
  // first.
  const int n_heads = a.pack ? p.hkv : p.hq;
  const int per_rank = n_heads * p.batch * a.n_splits;
  const int rank = (int)blockIdx.x / per_rank;
  const int rem = (int)blockIdx.x % per_rank;
  const int head_idx = rem % n_heads;
  const int split = (rem / n_heads) % a.n_splits;
  const int seq = rem / (n_heads * a.n_splits);
  const int m_tile = a.n_m_tiles - 1 - rank;
  const SeqGeom g = load_seq(p.cu_q, p.cu_k, seq, p.total_q, p.total_k, p.max_q, p.max_k, p.mask, p.window);
  if (!g.ok) {
    if (threadIdx.x == 0 && rank == 0 && head_idx == 0 && split == 0)
      raise_error(p.err, ATTN_ERR_DEVICE_BOUNDS);
    return;
  }
  const int i0 = m_tile * a.tile_tokens;
  if (i0 >= g.nq) return;  // the whole CTA leaves together
  const KvRange kr = plan_kv_tiles(g.mask, g.window, g.nq, g.nk, i0, a.tile_tokens, kTileKeys);
  int n_begin = kr.n_begin, n_stop = kr.n_end;
  if (a.n_splits > 1) split_tiles(kr.n_begin, kr.n_end, split, a.n_splits, &n_begin, &n_stop);
  const int n_tiles = n_stop - n_begin;
  const int kvh = a.pack ? head_idx : head_idx / a.group;

  if (threadIdx.x == 0) {
    mbar_init(&b->q_full, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(&b->k_full[s], 1);
      mbar_init(&b->v_full[s], 1);
      mbar_init(&b->k_empty[s], 1);
      mbar_init(&b->v_empty[s], 1);
      mbar_init(&b->s_full[s], 1);
    }
    mbar_init(&b->p_full, 128);
    mbar_init(&b->o_done, 1);
    mbar_init(&b->drain, 1);
    b->limit_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    b->abort = 0;
    b->filled_q = b->filled_k = b->filled_v = b->mma_issued = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&b->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b->tmem_base;

  const uint32_t sQ = smem_u32(smem + L::kQ);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);
  const uint32_t sP = smem_u32(smem + L::kP);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int qh = a.pack ? kvh * a.group : head_idx;
      int filled_k = 0, filled_v = 0;
      mbar_arrive_expect_tx(&b->q_full, L::kTile);
      for (int c = 0; c < L::kChunks; c++)
        tma_load_3d(smem + L::kQ + c * L::kChunk, &tm_q, &b->q_full, c * 64, qh, g.q0 + i0);
      for (int jj = 0; jj < n_tiles; jj++) {
        const int st = jj & 1, u = jj >> 1;
        const int key_row = g.k0 + (n_begin + jj) * kTileKeys;
        if (jj >= 2 && !wait_or_abort(b, &b->k_empty[st], (u - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&b->k_full[st], L::kTile);
        filled_k++;
        for (int c = 0; c < L::kChunks; c++)
          tma_load_3d(smem + L::kK + st * L::kTile + c * L::kChunk, &tm_k, &b->k_full[st], c * 64,
                      kvh, key_row);
        if (jj >= 2 && !wait_or_abort(b, &b->v_empty[st], (u - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&b->v_full[st], L::kTile);
        filled_v++;
        for (int c = 0; c < L::kChunks; c++)
          tma_load_3d(smem + L::kV + st * L::kTile + c * L::kChunk, &tm_v, &b->v_full[st], c * 64,
                      kvh, key_row);
      }
      b->filled_q = 1;  // for a drain after an early exit
      b->filled_k = filled_k;
      b->filled_v = filled_v;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0 && n_tiles > 0) {
      b->mma_issued = 1;
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kTileKeys, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
      auto issue_qk = [&](int st) {
        const uint32_t d_tmem = tmem + (uint32_t)(st * kTileKeys);
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint32_t off = (kk >> 2) * L::kChunk + (kk & 3) * 32;
          const uint64_t ad = smem_desc_sw128(sQ + off, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sK + st * L::kTile + off, 16, 1024);
          mma_bf16_ss(d_tmem, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int st, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kTileKeys / 16; kk++) {
          const uint32_t aoff = (kk >> 2) * L::kChunk + (kk & 3) * 32;
          const uint64_t ad = smem_desc_sw128(sP + aoff, 16, 1024);
          const uint64_t bd = smem_desc_sw128(sV + st * L::kTile + kk * 16 * 128, L::kChunk, 1024);
          mma_bf16_ss(tmem + kTmemO, ad, bd, idesc_pv, (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = wait_or_abort(b, &b->q_full, 0, p.err) && wait_or_abort(b, &b->k_full[0], 0, p.err);
      if (ok) {
        tc_fence_after();
        issue_qk(0);
        mma_commit(&b->s_full[0]);
        mma_commit(&b->k_empty[0]);
      }
      for (int jj = 0; ok && jj < n_tiles; jj++) {
        const int st = jj & 1;
        if (jj + 1 < n_tiles) {
          const int st1 = (jj + 1) & 1;
          if (!wait_or_abort(b, &b->k_full[st1], ((jj + 1) >> 1) & 1, p.err)) break;
          tc_fence_after();
          issue_qk(st1);
          mma_commit(&b->s_full[st1]);
          mma_commit(&b->k_empty[st1]);
        }
        if (!wait_or_abort(b, &b->p_full, jj & 1, p.err)) break;
        if (!wait_or_abort(b, &b->v_full[st], (jj >> 1) & 1, p.err)) break;
        tc_fence_after();
        issue_pv(st, jj > 0);
        mma_commit(&b->o_done);
        mma_commit(&b->v_empty[st]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;  // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;
    int i, h;
    row_map(a, head_idx, i0, r, &i, &h);
    const bool row_in = i < g.nq;
    const int t = g.q0 + i;
    const int row_limit = row_key_limit(g.mask, i, g.nq, g.nk);
    const int row_first = row_key_first(g.mask, g.window, i, g.nq, g.nk);
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const float c2 = p.scale_log2;
    static_assert(!(kBias && kPosScale), "the bias needs the logits before the max");
    const float slope2 = kBias ? __ldg(p.slopes + h) * kLog2e : 0.f;
    const float bound = (float)(i + causal_offset(g.mask, g.nq, g.nk));  // the row's causal bound
    float m_ref = -INFINITY, l = 0.f, lr = 0.f;
    bool ok = true;
    for (int jj = 0; jj < n_tiles; jj++) {
      const int n = n_begin + jj, sb = jj & 1;
      ok = wait_or_abort(b, &b->s_full[sb], (jj >> 1) & 1, p.err);
      if (!__all_sync(0xffffffffu, ok)) {  // leave together: tcgen05.ld is warp-wide
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t raw[kTileKeys];
#pragma unroll
      for (int c = 0; c < kTileKeys / 32; c++) {
        uint32_t u32[32];
        tmem_ld32(t_lane + sb * kTileKeys + c * 32, u32);
#pragma unroll
        for (int e = 0; e < 32; e++) raw[c * 32 + e] = u32[e];
      }
      tmem_wait_ld();
      if (!kr.full(n)) {  // boundary tile: keys outside this row's interval
        const int limit = row_limit - n * kTileKeys;
        const int first = row_first - n * kTileKeys;
#pragma unroll
        for (int c = 0; c < kTileKeys; c++)
          if (c >= limit || c < first) raw[c] = 0xff800000u;  // -inf
      }
      float mt;
      if constexpr (kPosScale) {  // the max of the raw scores scales to the max of the logits
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < kTileKeys; c++) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(raw[c]));
        mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * c2;
      } else {  // scale <= 0 or a bias: logits first, keep masked lanes at -inf
        mt = -INFINITY;
        const float dist0 = bound - (float)(n * kTileKeys);
#pragma unroll
        for (int c = 0; c < kTileKeys; c++) {
          const float x = __uint_as_float(raw[c]);
          float z = x * c2;
          if constexpr (kBias) z += pos_bias2(slope2, dist0, c);
          const float y = x == -INFINITY ? -INFINITY : z;
          raw[c] = __float_as_uint(y);
          mt = fmaxf(mt, y);
        }
      }
      const float cm = kPosScale ? c2 : 1.f;  // multiplier still to apply to raw
      const float m_new = mt > m_ref + kRescaleLog2 ? mt : m_ref;
      const float alpha = m_new == m_ref ? 1.f : fast_exp2(m_ref - m_new);
      const float base = m_new == -INFINITY ? 0.f : m_new;
      // P = 2^(raw * c - base) two lanes per instruction; two denominators:
      // l sums the fp32 probabilities and gives lse; lr sums the bf16-rounded
      // probabilities that the P V product uses, so O / lr is an exact convex
      // combination of V rows and a common offset in V cancels instead of
      // carrying P's rounding error.
      const uint64_t cx2 = f2(cm, cm), nb2 = f2(-base, -base);
      uint64_t s2[4] = {0, 0, 0, 0}, r2[4] = {0, 0, 0, 0};
      uint32_t pk[kTileKeys / 2];
#pragma unroll
      for (int c = 0; c < kTileKeys / 2; c++) {
        const uint64_t x = ffma2(f2(__uint_as_float(raw[2 * c]), __uint_as_float(raw[2 * c + 1])),
                                 cx2, nb2);
        float x0, x1;
        f2_split(x, x0, x1);
        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
        s2[c & 3] = fadd2(s2[c & 3], f2(p0, p1));
        pk[c] = pack_bf16x2(p0, p1);
        r2[c & 3] = fadd2(r2[c & 3], f2(__uint_as_float(pk[c] << 16),
                                        __uint_as_float(pk[c] & 0xffff0000u)));
      }
      float rs, rr;
      {
        float a0, a1, b0, b1;
        f2_split(fadd2(fadd2(s2[0], s2[1]), fadd2(s2[2], s2[3])), a0, a1);
        f2_split(fadd2(fadd2(r2[0], r2[1]), fadd2(r2[2], r2[3])), b0, b1);
        rs = a0 + a1;
        rr = b0 + b1;
      }
      l = l * alpha + rs;
      lr = lr * alpha + rr;
      m_ref = m_new;
      if (jj > 0) {
        // P V of the previous tile must be done: it reads the P buffer and
        // writes O, both of which are about to change.
        ok = wait_or_abort(b, &b->o_done, (jj - 1) & 1, p.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; c++) {
            uint32_t o32[32];
            tmem_ld32(t_lane + kTmemO + c * 32, o32);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e++) o32[e] = __float_as_uint(__uint_as_float(o32[e]) * alpha);
            tmem_st32(t_lane + kTmemO + c * 32, o32);
          }
          tmem_wait_st();
        }
      }
      // P row r in the 128-byte-swizzled K-major layout of the MMA's A operand
#pragma unroll
      for (int v = 0; v < kTileKeys / 8; v++) {
        const uint32_t addr = sP + (v >> 3) * L::kChunk + r * 128 + (((v & 7) ^ (r & 7)) << 4);
        st_shared_v4(addr, pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&b->p_full);
    }
    if (ok && n_tiles > 0) {
      if (wait_or_abort(b, &b->o_done, (n_tiles - 1) & 1, p.err)) {
        tc_fence_after();
      } else {
        ok = false;
      }
    }
    // ------------------------------------------------------------ epilogue
    const bool have = __all_sync(0xffffffffu, ok) && n_tiles > 0;
    const float inv = lr > 0.f ? 1.f / lr : 0.f;
    const float lse2 = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
    if (a.n_splits > 1) {
      float *dst = p.o_part + (((size_t)split * p.total_q + t) * p.hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; c++) {
        uint32_t o32[32];
        if (have) {
          tmem_ld32(t_lane + kTmemO + c * 32, o32);
          tmem_wait_ld();
        }
        if (row_in) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float4 f;
            f.x = have ? __uint_as_float(o32[e]) * inv : 0.f;
            f.y = have ? __uint_as_float(o32[e + 1]) * inv : 0.f;
            f.z = have ? __uint_as_float(o32[e + 2]) * inv : 0.f;
            f.w = have ? __uint_as_float(o32[e + 3]) * inv : 0.f;
            *reinterpret_cast<float4 *>(dst + c * 32 + e) = f;
          }
        }
      }
      if (row_in) p.lse_part[((size_t)split * p.hq + h) * p.total_q + t] = have ? lse2 : -INFINITY;
    } else {
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.o) + toff(p.so, t, h);
#pragma unroll
      for (int c = 0; c < D / 32; c++) {
        uint32_t o32[32];
        if (have) {
          tmem_ld32(t_lane + kTmemO + c * 32, o32);
          tmem_wait_ld();
        }
        if (row_in) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = have ? pack_bf16x2(__uint_as_float(o32[e]) * inv, __uint_as_float(o32[e + 1]) * inv) : 0u;
            w.y = have ? pack_bf16x2(__uint_as_float(o32[e + 2]) * inv, __uint_as_float(o32[e + 3]) * inv) : 0u;
            w.z = have ? pack_bf16x2(__uint_as_float(o32[e + 4]) * inv, __uint_as_float(o32[e + 5]) * inv) : 0u;
            w.w = have ? pack_bf16x2(__uint_as_float(o32[e + 6]) * inv, __uint_as_float(o32[e + 7]) * inv) : 0u;
            *reinterpret_cast<uint4 *>(dst + c * 32 + e) = w;
          }
          if (p.o_f32) {
            float *df = p.o_f32 + ((size_t)t * p.hq + h) * D + c * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              float4 f;
              f.x = have ? __uint_as_float(o32[e]) * inv : 0.f;
              f.y = have ? __uint_as_float(o32[e + 1]) * inv : 0.f;
              f.z = have ? __uint_as_float(o32[e + 2]) * inv : 0.f;
              f.w = have ? __uint_as_float(o32[e + 3]) * inv : 0.f;
              *reinterpret_cast<float4 *>(df + e) = f;
            }
          }
        }
      }
      if (row_in && p.lse) p.lse[(size_t)h * p.total_q + t] = have ? lse2 * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  // A block in which a wait gave up may still have copies and products in
  // flight: drain them before the tensor memory is freed (the flag is only
  // set before the barrier above).
  if (aborted(b)) {
    if (threadIdx.x == 0) {
      bool drained = drain_phase(&b->q_full, b->filled_q);
      for (int st = 0; st < 2; st++)
        drained = drain_phase(&b->k_full[st], ring_armed(b->filled_k, st, 2)) &&
                  drain_phase(&b->v_full[st], ring_armed(b->filled_v, st, 2)) && drained;
      if (!drained) raise_error(p.err, ATTN_ERR_DEVICE_TIMEOUT);
    }
    if (threadIdx.x == 32 && b->mma_issued && !drain_mma(&b->drain))
      raise_error(p.err, ATTN_ERR_DEVICE_TIMEOUT);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kPos, bool kBias>
cudaError_t launch_d(const TcArgs &a, const CUtensorMap &mq, const CUtensorMap &mk,
                     const CUtensorMap &mv, dim3 grid, cudaStream_t st) {
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D, kPos, kBias>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout<D>::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  fwd_tc_kernel<D, kPos, kBias><<<grid, kThreads, Layout<D>::kAlloc, st>>>(mq, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdParams &p, const TcPlan &plan, cudaStream_t st, char *desc,
                          size_t desc_len) {
  snprintf(desc, desc_len, "fwd_tc_d%d (tensor map or grid size rejected)", p.d);
  TcArgs a;
  a.p = p;
  a.pack = plan.pack;
  a.group = plan.group;
  a.tile_tokens = plan.tile_tokens;
  a.n_m_tiles = plan.n_m_tiles;
  a.n_splits = plan.n_splits;
  CUtensorMap mq, mk, mv;
  const int box_h = plan.pack ? plan.group : 1;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(&mq, p.q, p.d, p.hq, p.total_q, box_h, plan.tile_tokens, bf, p.sq.hs, p.sq.ts) ||
      !make_map(&mk, p.k, p.d, p.hkv, p.total_k, 1, kTileKeys, bf, p.sk.hs, p.sk.ts) ||
      !make_map(&mv, p.v, p.d, p.hkv, p.total_k, 1, kTileKeys, bf, p.sv.hs, p.sv.ts))
    return cudaErrorInvalidValue;
  const long long ctas = (long long)plan.n_m_tiles * (plan.pack ? p.hkv : p.hq) * p.batch *
                         plan.n_splits;
  if (ctas >= (1LL << 31)) return cudaErrorInvalidValue;
  dim3 grid((unsigned)ctas);
  snprintf(desc, desc_len, "fwd_tc_d%d%s ctas=%lld tile_tokens=%d splits=%d%s", p.d,
           plan.pack ? "_packgqa" : "", ctas, plan.tile_tokens, plan.n_splits,
           plan.n_splits > 1 ? " +combine" : "");
  const bool pos = p.scale_log2 > 0.f;
  if (p.slopes)  // the bias goes into the logits before the max
    return p.d == 64 ? launch_d<64, false, true>(a, mq, mk, mv, grid, st)
                     : launch_d<128, false, true>(a, mq, mk, mv, grid, st);
  if (p.d == 64) return pos ? launch_d<64, true, false>(a, mq, mk, mv, grid, st)
                            : launch_d<64, false, false>(a, mq, mk, mv, grid, st);
  return pos ? launch_d<128, true, false>(a, mq, mk, mv, grid, st)
             : launch_d<128, false, false>(a, mq, mk, mv, grid, st);
}

}  // namespace attn
