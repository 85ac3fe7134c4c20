// bwd_tc.cu -- tensor-core backward for bf16 inputs (recompute form), two kernels
// that share nothing but their inputs, so no atomics and a deterministic
// result:
//
//   dkdv: one CTA per (sequence, KV head, 128-key tile).  It walks every
//         query head of the KV head's group and every 64-row query tile that
//         can see its keys, and per tile computes on tcgen05
//           S^T = K Q^T, dP^T = V dO^T        (M = 128 keys, N = 64 rows),
//         turns them into P^T = 2^(c S^T - lse2) and dS^T = P^T (dP^T - D)
//         in registers (thread = key), and accumulates
//           dV += P^T dO, dK += dS^T Q        (M = 128 keys, N = d)
//         in TMEM, so the GQA sum over shared heads never leaves the SM
//         ("attention-algorithm-error-and-complexity-tests", third paragraph).
//   dq:   one CTA per (sequence, query head, 128-row query tile).  It walks
//         the row tile's key tiles and computes S = Q K^T, dP = dO V^T,
//         dS = P (dP - D) (thread = row) and dQ += dS K in TMEM.
//
// The products run in fp16 on fp16 copies of q, k, v and dout, each scaled by
// a power of two that brings its largest magnitude into [4, 8) (exact for
// every element within 2^19 of that largest one, whatever the tensor's
// overall magnitude; the factors are undone exactly in the softmax constant,
// D and the epilogues), so the P and dS operands keep 11 significant bits:
// with bf16 P, dV of a key that thousands of rows attend misses the 1e-2
// contract.  Accumulation is fp32 in TMEM.
//
// Both rebuild the forward's mask with the same planner and lane predicate
// ("causal-mask-and-ragged-sequence-layouts", sixth paragraph); masked and
// out-of-range lanes get P = dS = 0.  D and lse2 (lse in log2 units, +inf for
// empty rows) come from the preprocess kernel.  Waits are bounded like the
// forward's.
//
// Scheduling: the streamed operand rings (Q / dO four stages deep in dkdv, K
// three in dq) cover a stage's release, which waits for the products that
// read it, plus the refill's TMA latency; dq releases its single dP buffer as
// soon as the math warps have copied dP out, so the next dP product overlaps
// the exponentials.  Biases rebuild the forward's: the linear positional bias
// in the math (kBias); an explicit bias tensor (kTab) added in registers by
// the dK/dV math, stored into the score buffer before the score product
// accumulates onto it by the dQ math (its threads hold a 64-key row segment,
// too many registers to keep a prefetched copy).
#include <stdio.h>

#include <type_traits>

#include "common.cuh"
#include "plan.h"
#include "sm100.cuh"
#include "tma_map.h"
#include "bwd_tc.cuh"

namespace attn {
using namespace sm100;

namespace {

// warp 0 TMA, warp 1 MMA + TMEM, warps 2..9 math: two warps per TMEM lane
// quarter, each taking half of a row's columns
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr int kChunk128 = 128 * 128;  // [128 rows x 64 bf16] swizzled chunk
constexpr int kChunk64 = 64 * 128;    // [64 rows x 64 bf16] swizzled chunk

// ===========================================================================
// dK, dV
// ===========================================================================
template <int D>
struct LayoutA {
  static constexpr int kChunks = D / 64;
  static constexpr int kKV = kChunks * kChunk128;  // K or V tile
  static constexpr int kQT = kChunks * kChunk64;   // Q or dO tile (64 rows)
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKV;
  static constexpr int kQ = kV + kKV;                // [kStagesA] stages
  static constexpr int kDO = kQ + kStagesA * kQT;    // [kStagesA]
  static constexpr int kRow = kDO + kStagesA * kQT;  // [2] x {-lse2[64], -D[64]}
  static constexpr int kBar = kRow + 2 * 2 * kRowsA * 4;
  static constexpr int kUsed = kBar + 512;
  static constexpr int kAlloc = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
};

struct BarsA {
  // qdo_full / qdo_empty: one barrier for a step's Q and dO tiles; st_full:
  // both of a step's score products (S^T and dP^T) done; mm_done: the last
  // gradient products done.  Few barriers keep the MMA thread's commits and
  // waits, which the tensor pipe's short issue queue does not hide, few.
  uint64_t kv_full, qdo_full[kStagesA], qdo_empty[kStagesA], st_full[2], ps_full[2], mm_done;
  uint64_t drain;  // the MMA thread's products have all completed
  uint32_t tmem_base;
  Sync sync;
};

static_assert(sizeof(BarsA) <= 512, "barrier block fits its shared-memory slot");

// kBias: add the linear positional bias to the recomputed logits.  kTab: an
// explicit bias tensor; the math warps add each step's entries (log2 units,
// loaded a step ahead) to the exponent argument in registers, so the score
// products and their buffers are those of the plain kernel.
template <int D, bool kBias, bool kTab>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdTcArgs a) {
  using L = LayoutA<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  BarsA *b = reinterpret_cast<BarsA *>(smem + L::kBar);
  const BwdParams &p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // One-dimensional grid, key-tile index slowest: early keys (seen by the
  // most causal rows) of every (KV head, sequence) are scheduled first.
  const int per_rank = p.hkv * p.batch;
  const int n = (int)blockIdx.x / per_rank;
  const int hk = (int)blockIdx.x % p.hkv;
  const int seq = ((int)blockIdx.x % per_rank) / p.hkv;
  const SeqGeom g = load_seq(p.cu_q, p.cu_k, seq, p.total_q, p.total_k, p.max_q, p.max_k, p.mask, p.window);
  if (!g.ok) {
    if (threadIdx.x == 0 && n == 0 && hk == 0)
      raise_error(p.err, ATTN_ERR_DEVICE_BOUNDS);
    return;
  }
  const int j0 = n * kKeysA;
  if (j0 >= g.nk) return;
  // 64-row query tiles with at least one row that sees a key of this tile
  // (rows [row_begin(j), row_end(j)) see key j; both ends grow with j)
  const int j_last = (j0 + kKeysA < g.nk ? j0 + kKeysA : g.nk) - 1;
  const int m_begin = row_begin(g.mask, j0, g.nq, g.nk) / kRowsA;
  const int m_end = (row_end(g.mask, g.window, j_last, g.nq, g.nk) + kRowsA - 1) / kRowsA;
  const int n_m = m_end > m_begin ? m_end - m_begin : 0;
  const int n_it = n_m * a.group;

  if (threadIdx.x == 0) {
    mbar_init(&b->kv_full, 1);
    for (int s = 0; s < kStagesA; s++) {
      mbar_init(&b->qdo_full[s], 1);
      mbar_init(&b->qdo_empty[s], 1);
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(&b->st_full[s], 1);
      mbar_init(&b->ps_full[s], 256);
    }
    mbar_init(&b->mm_done, 1);
    mbar_init(&b->drain, 1);
    b->sync.limit_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    b->sync.abort = 0;
    b->sync.filled_one = b->sync.filled_a = b->sync.filled_b = b->sync.mma_issued = 0;
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
  // TMEM columns: S^T[2] at 0 / 64, dP^T[2] at 128 / 192, dV at 256, dK at 256 + D.
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;

  const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
  const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
  float *sRow = reinterpret_cast<float *>(smem + L::kRow);

  // Steps walk the group's heads one after another over the row tiles; with a
  // bias tensor the heads of one row tile come back to back instead, so a
  // tensor shared by the heads is read from cache after the first head.
  auto it_head = [&](int it) { return hk * a.group + (kTab ? it % a.group : it / n_m); };
  auto it_row0 = [&](int it) { return (m_begin + (kTab ? it / a.group : it % n_m)) * kRowsA; };

  if (warp == 0) {
    if (lane == 0 && n_it > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      int filled = 0;  // Q / dO ring fills (stage = fill % kStagesA)
      mbar_arrive_expect_tx(&b->kv_full, 2 * L::kKV);
      for (int c = 0; c < L::kChunks; c++) {
        tma_load_3d(smem + L::kK + c * kChunk128, &tm_k, &b->kv_full, c * 64, hk, g.k0 + j0);
        tma_load_3d(smem + L::kV + c * kChunk128, &tm_v, &b->kv_full, c * 64, hk, g.k0 + j0);
      }
      for (int it = 0; it < n_it; it++) {
        const int st = it % kStagesA, u = it / kStagesA;
        const int h = it_head(it), tok = g.q0 + it_row0(it);
        if (it >= kStagesA && !wait_bar(&b->sync, &b->qdo_empty[st], (u - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&b->qdo_full[st], 2 * L::kQT);
        filled++;
        for (int c = 0; c < L::kChunks; c++) {
          tma_load_3d(smem + L::kQ + st * L::kQT + c * kChunk64, &tm_q, &b->qdo_full[st], c * 64, h,
                      tok);
          tma_load_3d(smem + L::kDO + st * L::kQT + c * kChunk64, &tm_do, &b->qdo_full[st], c * 64,
                      h, tok);
        }
      }
      b->sync.filled_one = 1;
      b->sync.filled_a = filled;
    }
  } else if (warp == 1) {
    if (lane == 0 && n_it > 0) {
      b->sync.mma_issued = 1;
      constexpr uint32_t idesc_s = idesc_f16_f32(128, kRowsA, 0, 0);
      constexpr uint32_t idesc_g = idesc_f16_f32(128, D, 0, 1);
      // Descriptors built once; byte offsets below 256 KB add to the
      // start-address field (16-byte units).
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024), dV0 = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dQk = smem_desc_sw128(sQ, 16, 1024), dDOk = smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dQm = smem_desc_sw128(sQ, kChunk64, 1024);
      const uint64_t dDOm = smem_desc_sw128(sDO, kChunk64, 1024);
      // S^T (or dP^T) = A_tile [128 keys x d] * B_tile [64 rows x d]^T
      // acc0: accumulate from the first K step on (onto a stored bias)
      auto issue_st = [&](uint64_t da, uint64_t db, uint32_t col, bool acc0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint64_t oa = (uint64_t)((((kk >> 2) * kChunk128) + (kk & 3) * 32) >> 4);
          const uint64_t ob = (uint64_t)((((kk >> 2) * kChunk64) + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + col, da + oa, db + ob, idesc_s, (acc0 || kk > 0) ? 1u : 0u);
        }
      };
      // acc [128 keys x d] += A [128 keys x 64 rows] * B [64 rows x d], A in
      // tensor memory: rows [32 h, 32 h + 32) as 16 packed columns at 32 h
      auto issue_grad = [&](uint32_t a_col, uint64_t db, uint32_t col, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kRowsA / 16; kk++)
          mma_bf16_ts(tmem + col, tmem + a_col + 32 * (kk >> 1) + 8 * (kk & 1),
                      db + (uint64_t)((kk * 16 * 128) >> 4), idesc_g, (acc || kk > 0) ? 1u : 0u);
      };
      auto qoff = [&](int s1) { return (uint64_t)((s1 * L::kQT) >> 4); };
      bool ok = wait_bar(&b->sync, &b->kv_full, 0, p.err) &&
                wait_bar(&b->sync, &b->qdo_full[0], 0, p.err);
      if (ok) {
        tc_fence_after();
        issue_st(dK0, dQk, kColS, false);
        issue_st(dV0, dDOk, kColDP, false);
        mma_commit(&b->st_full[0]);
      }
      // tb: the step's TMEM buffer (two), qs: its Q / dO stage (kStagesA)
      for (int it = 0; ok && it < n_it; it++) {
        const int tb = it & 1, qs = it % kStagesA;
        if (it + 1 < n_it) {
          const int t1 = (it + 1) & 1, q1 = (it + 1) % kStagesA, u1 = (it + 1) / kStagesA;
          if (!wait_bar(&b->sync, &b->qdo_full[q1], u1 & 1, p.err)) break;
          tc_fence_after();
          issue_st(dK0, dQk + qoff(q1), kColS + t1 * kRowsA, false);
          issue_st(dV0, dDOk + qoff(q1), kColDP + t1 * kRowsA, false);
          mma_commit(&b->st_full[t1]);
        }
        if (!wait_bar(&b->sync, &b->ps_full[tb], (it >> 1) & 1, p.err)) break;
        tc_fence_after();
        issue_grad(kColS + tb * kRowsA, dDOm + qoff(qs), kColDV, it > 0);
        issue_grad(kColDP + tb * kRowsA, dQm + qoff(qs), kColDK, it > 0);
        if (it + 1 == n_it) mma_commit(&b->mm_done);
        if (it + kStagesA < n_it) mma_commit(&b->qdo_empty[qs]);  // a later step refills it
      }
    }
  } else {
    const int wq = warp & 3;
    const int half = (warp - 2) >> 2;  // query rows [32 half, 32 half + 32) of each step
    const int r = wq * 32 + lane;      // key lane
    const int tid = threadIdx.x - 64;  // 0 .. 255; threads below 128 fetch row terms
    const int j = j0 + r;          // in-sequence key
    const int rb = key_row_begin(g.mask, j, g.nq, g.nk);  // rows [rb, re) see key j
    const int re = key_row_end(g.mask, g.window, j, g.nq, g.nk);
    // Both ends of a key's row range grow with the key, so a step's 64 rows
    // see all 128 keys of the tile iff the last key's range starts at or
    // before the step and the first key's range ends at or after it: then no
    // lane is masked and the step takes the unmasked code (a uniform branch).
    const bool tile_in = j0 + kKeysA <= g.nk;
    const int rb_last = key_row_begin(g.mask, j0 + kKeysA - 1, g.nq, g.nk);
    const int re_first = key_row_end(g.mask, g.window, j0, g.nq, g.nk);
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const CopyScales cs = copy_scales(p);
    const float c2 = cs.c2;
    bool ok = true;
    // lse2 (threads 0..63) or D (64..127, in dP' units) of one row of a step's query tile;
    // the next step's value is fetched while the current step computes.
    auto row_value = [&](int it) {
      const int c = tid & (kRowsA - 1);
      const int i = it_row0(it) + c;
      const size_t at = (size_t)it_head(it) * p.total_q + g.q0 + i;
      // stored negated: the math below adds them
      if (tid < kRowsA) return i < g.nq ? -p.lse2[at] : -INFINITY;
      return i < g.nq ? -p.delta[at] * cs.dsc : 0.f;
    };
    const bool fetcher = tid < 2 * kRowsA;
    float next_val = (n_it > 0 && fetcher) ? row_value(0) : 0.f;
    // kTab: bias entries of step u for this key and the warp's 32 rows, in
    // log2 units (rows or keys out of range: 0), added to the exponent
    // argument in registers; step u + 1's loads fly during step u
    // Raw entries (natural-log units; the use folds in log2(e)); a step wholly
    // inside the sequence loads without per-entry bounds tests.
    auto load_bias = [&](int u, float (&bv)[32]) {
      const int ib = it_row0(u) + half * 32;
      const long long rs = p.brs;
      const float *ptr = btab_row(p.btab, p.bss, p.bhs, p.brs, seq, it_head(u), ib) + j;
      if (ib + 32 <= g.nq && j < g.nk) {
#pragma unroll
        for (int c = 0; c < 32; c++, ptr += rs) bv[c] = __ldg(ptr);
      } else {
#pragma unroll
        for (int c = 0; c < 32; c++, ptr += rs) bv[c] = ib + c < g.nq && j < g.nk ? __ldg(ptr) : 0.f;
      }
    };
    // One step; kTab: the step's entries in bcur, the next step's loads issued
    // into bnext (the caller alternates the two buffers).
    auto step = [&](int it, float (&bcur)[kTab ? 32 : 1], float (&bnext)[kTab ? 32 : 1]) {
      const int st = it & 1;
      const int i0 = it_row0(it);
      if (fetcher) sRow[st * 2 * kRowsA + tid] = next_val;
      math_group_sync();  // every math thread reaches it once per step, even after an abort
      if (fetcher && it + 1 < n_it) next_val = row_value(it + 1);
      const float *nlse2 = sRow + st * 2 * kRowsA;  // -lse2 of the 64 rows
      const float *nd = nlse2 + kRowsA;              // -D of the 64 rows
      if constexpr (kTab) {
        if (it + 1 < n_it) load_bias(it + 1, bnext);
      }
      if (ok)
        ok = wait_bar(&b->sync, &b->st_full[st], (it >> 1) & 1, p.err);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return;
      tc_fence_after();
      const bool step_full = tile_in && rb_last <= i0 && re_first >= i0 + kRowsA;
      // rows i0 + c with c_lo <= c < c_lo + span see key j
      const int c_lo = rb - i0, span = re > rb ? re - rb : 0;
      const uint64_t c2x2 = f2(c2, c2);
      // positional bias of row i0 + c: -slope2 |i0 + c + off - j|
      const float slope2 = kBias ? __ldg(p.slopes + it_head(it)) * kLog2e : 0.f;
      const float bdist0 = (float)(j - i0 - causal_offset(g.mask, g.nq, g.nk));
      uint32_t pp[16], dd[16];
      uint32_t sv[32], dv[32];  // this warp's 32 rows of the step
      tmem_ld32(t_lane + kColS + st * kRowsA + half * 32, sv);
      tmem_ld32(t_lane + kColDP + st * kRowsA + half * 32, dv);
      tmem_wait_ld();
      auto body = [&](auto masked) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int c0 = half * 32 + e;
          // two lanes per instruction: x = c S - lse2, P = 2^x, dS = P (dP - D)
          float2 nl = *reinterpret_cast<const float2 *>(nlse2 + c0);
          const float2 ndd = *reinterpret_cast<const float2 *>(nd + c0);
          if constexpr (kBias) {
            nl.x += pos_bias2(slope2, bdist0, c0);
            nl.y += pos_bias2(slope2, bdist0, c0 + 1);
          }
          if constexpr (kTab) {  // a -inf entry gives P = 0
            nl.x = fmaf(bcur[e], kLog2e, nl.x);
            nl.y = fmaf(bcur[e + 1], kLog2e, nl.y);
          }
          float x0, x1;
          f2_split(ffma2(f2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2x2, f2(nl.x, nl.y)),
                   x0, x1);
          float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          if constexpr (decltype(masked)::value) {
            if ((unsigned)(c0 - c_lo) >= (unsigned)span) p0 = 0.f;
            if ((unsigned)(c0 + 1 - c_lo) >= (unsigned)span) p1 = 0.f;
          }
          const uint64_t pv = f2(p0, p1);
          float d0, d1;
          f2_split(fmul2(pv, fadd2(f2(__uint_as_float(dv[e]), __uint_as_float(dv[e + 1])),
                                   f2(ndd.x, ndd.y))),
                   d0, d1);
          pp[e / 2] = pack_f16x2(p0, p1);
          dd[e / 2] = pack_f16x2(d0, d1);
        }
      };
      if (step_full)
        body(std::false_type{});
      else
        body(std::true_type{});
      // P^T over the first 16 of the 32 S^T columns this warp just read, dS^T
      // likewise over dP^T: the A operands of the two gradient products,
      // straight from tensor memory.
      tmem_st16(t_lane + kColS + st * kRowsA + half * 32, pp);
      tmem_st16(t_lane + kColDP + st * kRowsA + half * 32, dd);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&b->ps_full[st]);
    };
    float b0[kTab ? 32 : 1], b1[kTab ? 32 : 1];
    if constexpr (kTab) {
      if (n_it > 0) load_bias(0, b0);
      for (int it = 0; it < n_it; it += 2) {  // the two buffers alternate without copies
        step(it, b0, b1);
        if (it + 1 < n_it) step(it + 1, b1, b0);
      }
    } else {
      for (int it = 0; it < n_it; it++) step(it, b0, b1);
    }
    if (ok && n_it > 0) {
      if (wait_bar(&b->sync, &b->mm_done, 0, p.err))
        tc_fence_after();
      else
        ok = false;
    }
    const bool have = __all_sync(0xffffffffu, ok) && n_it > 0;
    // this warp writes output columns [half D / 2, half D / 2 + D / 2)
    const int jt = g.k0 + (j < g.nk ? j : 0);
    __nv_bfloat16 *dkp = reinterpret_cast<__nv_bfloat16 *>(p.dk) + toff(p.sdk, jt, hk) + half * (D / 2);
    __nv_bfloat16 *dvp = reinterpret_cast<__nv_bfloat16 *>(p.dv) + toff(p.sdv, jt, hk) + half * (D / 2);
#pragma unroll
    for (int c = 0; c < D / 64; c++) {
      uint32_t kv32[32], vv32[32];
      if (have) {  // warp-uniform: every lane of the warp loads
        tmem_ld32(t_lane + kColDK + half * (D / 2) + c * 32, kv32);
        tmem_ld32(t_lane + kColDV + half * (D / 2) + c * 32, vv32);
        tmem_wait_ld();
      }
      if (j < g.nk) {  // keys past the sequence end own no storage
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 wk, wv;
          // dK = (dK' 2^-(s_v + s_do)) scale 2^-s_q, dV = dV' 2^-s_do
          auto kf = [&](int c1) { return __uint_as_float(kv32[c1]) * cs.g * cs.gk; };
          auto vf = [&](int c1) { return __uint_as_float(vv32[c1]) * cs.gv; };
          wk.x = have ? pack_bf16x2(kf(e), kf(e + 1)) : 0u;
          wk.y = have ? pack_bf16x2(kf(e + 2), kf(e + 3)) : 0u;
          wk.z = have ? pack_bf16x2(kf(e + 4), kf(e + 5)) : 0u;
          wk.w = have ? pack_bf16x2(kf(e + 6), kf(e + 7)) : 0u;
          wv.x = have ? pack_bf16x2(vf(e), vf(e + 1)) : 0u;
          wv.y = have ? pack_bf16x2(vf(e + 2), vf(e + 3)) : 0u;
          wv.z = have ? pack_bf16x2(vf(e + 4), vf(e + 5)) : 0u;
          wv.w = have ? pack_bf16x2(vf(e + 6), vf(e + 7)) : 0u;
          *reinterpret_cast<uint4 *>(dkp + c * 32 + e) = wk;
          *reinterpret_cast<uint4 *>(dvp + c * 32 + e) = wv;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // A block in which a wait gave up may still have copies and products in
  // flight: drain them before the tensor memory is freed (the flag is only
  // set before the barrier above).
  if (*reinterpret_cast<volatile int *>(&b->sync.abort)) {
    if (threadIdx.x == 0) {
      bool drained = drain_phase(&b->kv_full, b->sync.filled_one);
      for (int st = 0; st < kStagesA; st++)
        drained = drain_phase(&b->qdo_full[st], ring_armed(b->sync.filled_a, st, kStagesA)) && drained;
      if (!drained) raise_error(p.err, ATTN_ERR_DEVICE_TIMEOUT);
    }
    if (threadIdx.x == 32 && b->sync.mma_issued && !drain_mma(&b->drain))
      raise_error(p.err, ATTN_ERR_DEVICE_TIMEOUT);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// N consecutive bias-tensor entries of one row from key j0 on, divided by the
// positive scale (raw-score units: the score product accumulates onto them);
// keys at or past nk, or no row, give 0.
template <int N>
__device__ __forceinline__ void load_bias_row(const float *brow, int j0, int nk, float inv_scale,
                                              uint32_t (&bv)[N]) {
  if (brow && j0 + N <= nk && (reinterpret_cast<uintptr_t>(brow + j0) & 15) == 0) {
#pragma unroll
    for (int e = 0; e < N; e += 4) {
      const float4 f = __ldg(reinterpret_cast<const float4 *>(brow + j0 + e));
      bv[e] = __float_as_uint(f.x * inv_scale);
      bv[e + 1] = __float_as_uint(f.y * inv_scale);
      bv[e + 2] = __float_as_uint(f.z * inv_scale);
      bv[e + 3] = __float_as_uint(f.w * inv_scale);
    }
  } else {
#pragma unroll
    for (int e = 0; e < N; e++)
      bv[e] = __float_as_uint(brow && j0 + e < nk ? __ldg(brow + j0 + e) * inv_scale : 0.f);
  }
}

// ===========================================================================
// dQ
// ===========================================================================
// K ring depth: a K stage is refilled only after the dQ product of its tile
// completes (V is free as soon as dP is), and the refill's TMA latency is
// longer than the one dP product queued behind that dQ.
constexpr int kStagesK = 3;

template <int D>
struct LayoutB {
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk128;
  static constexpr int kQ = 0;
  static constexpr int kDO = kQ + kTile;
  static constexpr int kK = kDO + kTile;            // [kStagesK]
  static constexpr int kV = kK + kStagesK * kTile;  // [2]
  static constexpr int kBar = kV + 2 * kTile;
  static constexpr int kUsed = kBar + 256;
  static constexpr int kAlloc = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
};

struct BarsB {
  uint64_t qdo_full, k_full[kStagesK], v_full[2], k_empty[kStagesK], v_empty[2], s_full[2],
      dp_full, dp_free, ds_full, dq_done;
  uint64_t b_full[2], s_free[2];  // kTab: bias stored in S buffer t / buffer t read by dQ
  uint64_t drain;  // the MMA thread's products have all completed
  uint32_t tmem_base;
  Sync sync;
};

static_assert(sizeof(BarsB) <= 256, "barrier block fits its shared-memory slot");

// kTab: an explicit bias tensor; the math warps store a tile's entries (over
// the positive scale) into its S buffer and S = Q K^T accumulates onto them.
template <int D, bool kBias, bool kTab>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                     const BwdTcArgs a) {
  using L = LayoutB<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  BarsB *b = reinterpret_cast<BarsB *>(smem + L::kBar);
  const BwdParams &p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // One-dimensional grid, row-tile rank slowest: the last row tiles (most
  // causal keys) of every (head, sequence) first.
  const int per_rank = p.hq * p.batch;
  const int rank = (int)blockIdx.x / per_rank;
  const int h = (int)blockIdx.x % p.hq;
  const int seq = ((int)blockIdx.x % per_rank) / p.hq;
  const int m_tile = a.n_row_tiles - 1 - rank;
  const SeqGeom g = load_seq(p.cu_q, p.cu_k, seq, p.total_q, p.total_k, p.max_q, p.max_k, p.mask, p.window);
  if (!g.ok) {
    if (threadIdx.x == 0 && rank == 0 && h == 0)
      raise_error(p.err, ATTN_ERR_DEVICE_BOUNDS);
    return;
  }
  const int i0 = m_tile * kTileRows;
  if (i0 >= g.nq) return;
  const KvRange kr = plan_kv_tiles(g.mask, g.window, g.nq, g.nk, i0, kTileRows, kTileKeys);
  const int n_first = kr.n_begin;              // key tiles [n_first, n_first + n_tiles)
  const int n_tiles = kr.n_end - kr.n_begin;
  const int hk = h / a.group;

  if (threadIdx.x == 0) {
    mbar_init(&b->qdo_full, 1);
    for (int s = 0; s < kStagesK; s++) {
      mbar_init(&b->k_full[s], 1);
      mbar_init(&b->k_empty[s], 1);
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(&b->v_full[s], 1);
      mbar_init(&b->v_empty[s], 1);
      mbar_init(&b->s_full[s], 1);
    }
    mbar_init(&b->dp_full, 1);
    mbar_init(&b->dp_free, 256);
    for (int s = 0; s < 2; s++) {
      mbar_init(&b->b_full[s], 256);
      mbar_init(&b->s_free[s], 1);
    }
    mbar_init(&b->ds_full, 256);
    mbar_init(&b->dq_done, 1);
    mbar_init(&b->drain, 1);
    b->sync.limit_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    b->sync.abort = 0;
    b->sync.filled_one = b->sync.filled_a = b->sync.filled_b = b->sync.mma_issued = 0;
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
  // TMEM columns: S[2] at 0 / 128, dP at 256, dQ at 384.
  constexpr uint32_t kColS = 0, kColDP = 256, kColDQ = 384;

  const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
  const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);

  if (warp == 0) {
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int filled_k = 0, filled_v = 0;  // K ring fills (fill % kStagesK), V ring fills (fill % 2)
      mbar_arrive_expect_tx(&b->qdo_full, 2 * L::kTile);
      for (int c = 0; c < L::kChunks; c++) {
        tma_load_3d(smem + L::kQ + c * kChunk128, &tm_q, &b->qdo_full, c * 64, h, g.q0 + i0);
        tma_load_3d(smem + L::kDO + c * kChunk128, &tm_do, &b->qdo_full, c * 64, h, g.q0 + i0);
      }
      for (int jj = 0; jj < n_tiles; jj++) {
        const int st = jj & 1, u = jj >> 1;
        const int ks = jj % kStagesK, ku = jj / kStagesK;
        const int key_row = g.k0 + (n_first + jj) * kTileKeys;
        if (jj >= kStagesK && !wait_bar(&b->sync, &b->k_empty[ks], (ku - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&b->k_full[ks], L::kTile);
        filled_k++;
        for (int c = 0; c < L::kChunks; c++)
          tma_load_3d(smem + L::kK + ks * L::kTile + c * kChunk128, &tm_k, &b->k_full[ks], c * 64,
                      hk, key_row);
        if (jj >= 2 && !wait_bar(&b->sync, &b->v_empty[st], (u - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&b->v_full[st], L::kTile);
        filled_v++;
        for (int c = 0; c < L::kChunks; c++)
          tma_load_3d(smem + L::kV + st * L::kTile + c * kChunk128, &tm_v, &b->v_full[st], c * 64,
                      hk, key_row);
      }
      b->sync.filled_one = 1;
      b->sync.filled_a = filled_k;
      b->sync.filled_b = filled_v;
    }
  } else if (warp == 1) {
    if (lane == 0 && n_tiles > 0) {
      b->sync.mma_issued = 1;
      constexpr uint32_t idesc_s = idesc_f16_f32(128, kTileKeys, 0, 0);
      constexpr uint32_t idesc_q = idesc_f16_f32(128, D, 0, 1);
      const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024), dDO0 = smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024), dV0 = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dKm = smem_desc_sw128(sK, kChunk128, 1024);
      auto toff = [&](int s1) { return (uint64_t)((s1 * L::kTile) >> 4); };
      // acc0: accumulate from the first K step on (onto a stored bias)
      auto issue_s = [&](uint64_t da, uint64_t db, uint32_t col, bool acc0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint64_t off = (uint64_t)((((kk >> 2) * kChunk128) + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + col, da + off, db + off, idesc_s, (acc0 || kk > 0) ? 1u : 0u);
        }
      };
      // dQ += dS K, dS in tensor memory: keys [64 h, 64 h + 64) as 32 packed
      // columns at 64 h of this tile's S buffer
      auto issue_dq = [&](int st, int ks, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kTileKeys / 16; kk++)
          mma_bf16_ts(tmem + kColDQ, tmem + kColS + st * kTileKeys + 64 * (kk >> 2) + 8 * (kk & 3),
                      dKm + toff(ks) + (uint64_t)((kk * 16 * 128) >> 4), idesc_q,
                      (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_bar(&b->sync, &b->qdo_full, 0, p.err) &&
                wait_bar(&b->sync, &b->k_full[0], 0, p.err) &&
                (!kTab || wait_bar(&b->sync, &b->b_full[0], 0, p.err));
      if (ok) {
        tc_fence_after();
        issue_s(dQ0, dK0, kColS, kTab);
        mma_commit(&b->s_full[0]);
        ok = wait_bar(&b->sync, &b->v_full[0], 0, p.err);
      }
      if (ok) {
        tc_fence_after();
        issue_s(dDO0, dV0, kColDP, false);
        mma_commit(&b->dp_full);
        if (2 < n_tiles) mma_commit(&b->v_empty[0]);
      }
      // st: the tile's S buffer and V stage (two), ks: its K stage (kStagesK)
      for (int jj = 0; ok && jj < n_tiles; jj++) {
        const int st = jj & 1, ks = jj % kStagesK;
        const int s1 = (jj + 1) & 1, u1 = (jj + 1) >> 1;
        if (jj + 1 < n_tiles) {
          const int k1 = (jj + 1) % kStagesK;
          if (!wait_bar(&b->sync, &b->k_full[k1], ((jj + 1) / kStagesK) & 1, p.err)) break;
          if (kTab && !wait_bar(&b->sync, &b->b_full[s1], u1 & 1, p.err)) break;
          tc_fence_after();
          issue_s(dQ0, dK0 + toff(k1), kColS + s1 * kTileKeys, kTab);
          mma_commit(&b->s_full[s1]);
          // dP's single buffer is free as soon as the math warps have read
          // this tile's dP out, well before they finish dS: the next dP
          // product overlaps this tile's math.
          if (!wait_bar(&b->sync, &b->dp_free, jj & 1, p.err) ||
              !wait_bar(&b->sync, &b->v_full[s1], u1 & 1, p.err))
            break;
          tc_fence_after();
          issue_s(dDO0, dV0 + toff(s1), kColDP, false);
          mma_commit(&b->dp_full);
          if (jj + 3 < n_tiles) mma_commit(&b->v_empty[s1]);  // tile jj + 3 refills it
        }
        if (!wait_bar(&b->sync, &b->ds_full, jj & 1, p.err)) break;
        tc_fence_after();
        issue_dq(st, ks, jj > 0);
        if (kTab && jj + 2 < n_tiles) mma_commit(&b->s_free[st]);  // tile jj + 2's bias may go in
        if (jj + 1 == n_tiles) mma_commit(&b->dq_done);
        if (jj + kStagesK < n_tiles) mma_commit(&b->k_empty[ks]);  // a later tile refills it
      }
    }
  } else {
    const int wq = warp & 3;
    const int half = (warp - 2) >> 2;  // keys [64 half, 64 half + 64) of each tile
    const int r = wq * 32 + lane;
    const int i = i0 + r;
    const bool row_in = i < g.nq;
    const int t = g.q0 + i;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const CopyScales cs = copy_scales(p);
    const float c2 = cs.c2;
    const int row_limit = row_key_limit(g.mask, i, g.nq, g.nk);
    const int row_first = row_key_first(g.mask, g.window, i, g.nq, g.nk);
    const float lse2 = row_in ? p.lse2[(size_t)h * p.total_q + t] : INFINITY;
    const float D_i = row_in ? p.delta[(size_t)h * p.total_q + t] * cs.dsc : 0.f;  // dP' units
    const uint64_t c2x2 = f2(c2, c2), nl2 = f2(-lse2, -lse2), nd2 = f2(-D_i, -D_i);
    const float slope2 = kBias ? __ldg(p.slopes + h) * kLog2e : 0.f;
    const float bound = (float)(i + causal_offset(g.mask, g.nq, g.nk));  // the row's causal bound
    bool ok = true;
    // kTab: this warp's 64 keys of tile u's bias row into S buffer u & 1
    const float *brow = kTab && row_in ? btab_row(p.btab, p.bss, p.bhs, p.brs, seq, h, i) : nullptr;
    const float inv_scale = kTab ? cs.bias : 0.f;  // entry -> S' units
    auto store_bias = [&](int u, const uint32_t (&bv)[64]) {
      const uint32_t col = t_lane + kColS + (u & 1) * kTileKeys + half * 64;
      tmem_st32(col, *reinterpret_cast<const uint32_t(*)[32]>(bv));
      tmem_st32(col + 32, *reinterpret_cast<const uint32_t(*)[32]>(bv + 32));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&b->b_full[u & 1]);
    };
    if (kTab)
      for (int u = 0; u < 2 && u < n_tiles; u++) {
        uint32_t bv[64];
        load_bias_row<64>(brow, (n_first + u) * kTileKeys + half * 64, g.nk, inv_scale, bv);
        store_bias(u, bv);
      }
    for (int jj = 0; jj < n_tiles; jj++) {
      const int st = jj & 1;
      // S is issued before dP, so both are in once dP is
      ok = wait_bar(&b->sync, &b->dp_full, jj & 1, p.err) &&
           wait_bar(&b->sync, &b->s_full[st], (jj >> 1) & 1, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // this warp's 64 dP columns and its first 32 S columns under one wait;
      // then the dP buffer is released
      uint32_t dv[64], sv[32];
      tmem_ld64(t_lane + kColDP + half * 64, dv);
      tmem_ld32(t_lane + kColS + st * kTileKeys + half * 64, sv);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&b->dp_free);
      const bool boundary = !kr.full(n_first + jj);
      const int jb = (n_first + jj) * kTileKeys;
      // dS (fp16 pairs) of this warp's 64 keys goes over the first 32 of the
      // S columns it read.
      uint32_t dd[32];
      // 32 keys from sv: masked lanes (boundary tiles only, a uniform
      // branch) get P = dS = 0
      auto chunk = [&](int q, auto masked) {
        const int cc = 2 * half + q;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int c = cc * 32 + e;
          uint64_t add2 = nl2;
          if constexpr (kBias)
            add2 = f2(pos_bias2(slope2, bound - (float)jb, c) - lse2,
                      pos_bias2(slope2, bound - (float)jb, c + 1) - lse2);
          float x0, x1;
          f2_split(ffma2(f2(__uint_as_float(sv[e]), __uint_as_float(sv[e + 1])), c2x2, add2), x0, x1);
          float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          if constexpr (decltype(masked)::value) {
            if (jb + c >= row_limit || jb + c < row_first) p0 = 0.f;
            if (jb + c + 1 >= row_limit || jb + c + 1 < row_first) p1 = 0.f;
          }
          float d0, d1;
          f2_split(fmul2(f2(p0, p1), fadd2(f2(__uint_as_float(dv[32 * q + e]),
                                              __uint_as_float(dv[32 * q + e + 1])), nd2)),
                   d0, d1);
          dd[q * 16 + e / 2] = pack_f16x2(d0, d1);
        }
      };
      if (boundary) chunk(0, std::true_type{}); else chunk(0, std::false_type{});
      tmem_ld32(t_lane + kColS + st * kTileKeys + half * 64 + 32, sv);
      tmem_wait_ld();
      if (boundary) chunk(1, std::true_type{}); else chunk(1, std::false_type{});
      tmem_st32(t_lane + kColS + st * kTileKeys + half * 64, dd);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&b->ds_full);
      if (kTab && jj + 2 < n_tiles) {
        // tile jj + 2 reuses this S buffer once dQ has read this tile's dS
        uint32_t bv[64];
        load_bias_row<64>(brow, (n_first + jj + 2) * kTileKeys + half * 64, g.nk, inv_scale, bv);
        ok = wait_bar(&b->sync, &b->s_free[st], (jj >> 1) & 1, p.err);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        store_bias(jj + 2, bv);
      }
    }
    if (ok && n_tiles > 0) {
      if (wait_bar(&b->sync, &b->dq_done, 0, p.err))
        tc_fence_after();
      else
        ok = false;
    }
    const bool have = __all_sync(0xffffffffu, ok) && n_tiles > 0;
    // this warp writes dQ columns [half D / 2, half D / 2 + D / 2)
    __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.dq) + toff(p.sdq, t, h) + half * (D / 2);
#pragma unroll
    for (int c = 0; c < D / 64; c++) {
      uint32_t q32[32];
      if (have) {
        tmem_ld32(t_lane + kColDQ + half * (D / 2) + c * 32, q32);
        tmem_wait_ld();
      }
      if (row_in) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 w;
          // dQ = (dQ' 2^-(s_v + s_do)) scale 2^-s_k
          auto qf = [&](int c1) { return __uint_as_float(q32[c1]) * cs.g * cs.gq; };
          w.x = have ? pack_bf16x2(qf(e), qf(e + 1)) : 0u;
          w.y = have ? pack_bf16x2(qf(e + 2), qf(e + 3)) : 0u;
          w.z = have ? pack_bf16x2(qf(e + 4), qf(e + 5)) : 0u;
          w.w = have ? pack_bf16x2(qf(e + 6), qf(e + 7)) : 0u;
          *reinterpret_cast<uint4 *>(dst + c * 32 + e) = w;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // A block in which a wait gave up may still have copies and products in
  // flight: drain them before the tensor memory is freed (the flag is only
  // set before the barrier above).
  if (*reinterpret_cast<volatile int *>(&b->sync.abort)) {
    if (threadIdx.x == 0) {
      bool drained = drain_phase(&b->qdo_full, b->sync.filled_one);
      for (int ks = 0; ks < kStagesK; ks++)
        drained = drain_phase(&b->k_full[ks], ring_armed(b->sync.filled_a, ks, kStagesK)) && drained;
      for (int st = 0; st < 2; st++)
        drained = drain_phase(&b->v_full[st], ring_armed(b->sync.filled_b, st, 2)) && drained;
      if (!drained) raise_error(p.err, ATTN_ERR_DEVICE_TIMEOUT);
    }
    if (threadIdx.x == 32 && b->sync.mma_issued && !drain_mma(&b->drain))
      raise_error(p.err, ATTN_ERR_DEVICE_TIMEOUT);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kBias, bool kTab>
cudaError_t launch_d(const BwdTcArgs &a, cudaStream_t st) {
  const BwdParams &p = a.p;
  // Every tensor-core product of the backward runs on the fp16 copies.
  const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap q64, do64, q128, do128, mk, mv;
  if (!make_map(&q64, p.q16, D, p.hq, p.total_q, 1, kRowsA, f16) ||
      !make_map(&do64, p.do16, D, p.hq, p.total_q, 1, kRowsA, f16) ||
      !make_map(&q128, p.q16, D, p.hq, p.total_q, 1, kTileRows, f16) ||
      !make_map(&do128, p.do16, D, p.hq, p.total_q, 1, kTileRows, f16) ||
      !make_map(&mk, p.k16, D, p.hkv, p.total_k, 1, kTileKeys, f16) ||
      !make_map(&mv, p.v16, D, p.hkv, p.total_k, 1, kTileKeys, f16))
    return cudaErrorInvalidValue;
  static bool conf_a[64] = {false}, conf_b[64] = {false};
  cudaError_t e = set_smem(bwd_dkdv_tc_kernel<D, kBias, kTab>, LayoutA<D>::kAlloc, conf_a);
  if (e != cudaSuccess) return e;
  e = set_smem(bwd_dq_tc_kernel<D, kBias, kTab>, LayoutB<D>::kAlloc, conf_b);
  if (e != cudaSuccess) return e;
  const long long ga = (long long)a.n_key_tiles * p.hkv * p.batch;
  const long long gb = (long long)a.n_row_tiles * p.hq * p.batch;
  if (ga >= (1LL << 31) || gb >= (1LL << 31)) return cudaErrorInvalidValue;
  bwd_dkdv_tc_kernel<D, kBias, kTab><<<(unsigned)ga, kThreads, LayoutA<D>::kAlloc, st>>>(q64, do64, mk, mv, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_dq_tc_kernel<D, kBias, kTab><<<(unsigned)gb, kThreads, LayoutB<D>::kAlloc, st>>>(q128, do128, mk, mv, a);
  return cudaGetLastError();
}

}  // namespace

// The tensor-core backward after the preprocess kernel (D and lse2 ready).
cudaError_t launch_bwd_tc(const BwdParams &p, cudaStream_t st, char *desc, size_t desc_len) {
  BwdTcArgs a;
  a.p = p;
  a.group = p.hq / p.hkv;
  a.n_key_tiles = (p.max_k + kKeysA - 1) / kKeysA;
  a.n_row_tiles = (p.max_q + kTileRows - 1) / kTileRows;
  snprintf(desc, desc_len,
           "zero_rows+zero_rows+bwd_amax+bwd_pre+kv_to_f16%s+bwd_dkdv_tc_d%d+bwd_dq_tc_d%d%s "
           "ctas_dkdv=%lld ctas_dq=%lld",
           p.delta_ready ? "+fwd_tc2_delta" : "", p.d, p.d, p.btab ? "_btab" : "",
           (long long)a.n_key_tiles * p.hkv * p.batch, (long long)a.n_row_tiles * p.hq * p.batch);
  if (a.n_key_tiles == 0 || a.n_row_tiles == 0) return cudaSuccess;
  // a bias tensor comes here only with a positive scale and no slopes
  if (p.btab) return p.d == 64 ? launch_d<64, false, true>(a, st) : launch_d<128, false, true>(a, st);
  if (p.slopes) return p.d == 64 ? launch_d<64, true, false>(a, st) : launch_d<128, true, false>(a, st);
  return p.d == 64 ? launch_d<64, false, false>(a, st) : launch_d<128, false, false>(a, st);
}

}  // namespace attn
