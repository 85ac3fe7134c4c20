// fwd_tc2.cuh -- tensor-core prefill forward with two query tiles per CTA:
// the kernel template and its launch helpers, instantiated by fwd_tc2.cu
// (the forward's outputs) and fwd_tc2_delta.cu (the backward's D term).
//
// Same arithmetic as fwd_tc.cu (the online-softmax recurrence of the
// "formal-correctness" page, "The FlashAttention Proof"; masks from the tile
// planner of common.cuh), scheduled so the tensor core never waits on one
// softmax: a CTA owns 256 query rows of one head as two 128-row tiles A and B
// that share every K/V tile, and the MMA thread interleaves their products
//
//   QK_A(n), QK_B(n), PV_A(n), QK_A(n+1), PV_B(n), QK_B(n+1), PV_A(n+1), ...
//
// so that while one softmax warpgroup turns its S into P, the tensor core is
// busy with the other tile.  Warpgroups: the first holds warp 0 (TMA
// producer), warp 1 (TMEM allocation and MMA issue) and warp 2 (without a
// bias, a watcher that folds the K / V arrivals into the P barriers; with a
// staged bias tensor, the copies of its entries) and gives most of its
// registers to the other two, which run the softmax of tile A (warps 4..7)
// and tile B (warps 8..11), thread = row = TMEM lane.  TMEM: S_A, S_B, O_A,
// O_B; each tile's bf16 P overwrites the second half of its S and feeds P V
// from tensor memory, so P never passes through shared memory.  Shared
// memory: Q_A, Q_B (which also stage full O tiles for their TMA stores) and
// a 2-stage K/V ring.
//
// With the extra registers a softmax thread loads its whole 128-score row
// from TMEM with one wait, takes the max, and writes the 64 packed
// probabilities back.  Instances add the linear positional bias in the softmax (kBias)
// or an explicit bias tensor, in one of two ways (kTab): 1, the softmax warps
// load their rows' entries and store them into S before Q K^T accumulates
// onto it (then tile A's next Q K^T follows tile B's P V, since A's bias
// waits for A's P V to finish reading P); 2, for a tensor the two heads of a
// CTA share, warp 2 streams each key tile's entries into shared memory with
// TMA and the softmax adds them to the scores it loads (the schedule stays
// the plain one; with D = 128 the V ring then has one stage, for room).
#pragma once

#include <stdio.h>
#include <string.h>

#include <type_traits>

#include "common.cuh"
#include "plan.h"
#include "sm100.cuh"
#include "tma_map.h"

namespace attn {

int internal_sm_count();
using namespace sm100;

namespace {

constexpr int kThreads2 = 384;
// Registers per thread: the launch gives every thread kRegsLaunch (the most
// 384 threads can have); the control warpgroup drops to kRegsCtl and the two
// softmax warpgroups rise to kRegsSoftmax.
constexpr uint32_t kRegsLaunch = 168, kRegsCtl = 80, kRegsSoftmax = 208;
static_assert(128 * kRegsCtl + 256 * kRegsSoftmax <= kThreads2 * kRegsLaunch,
              "the increases must not exceed what the decreases free");
static_assert(kThreads2 * kRegsLaunch <= 65536, "register file");
constexpr float kRescale2 = 8.0f;
constexpr uint32_t kCols2 = 512;

// kStaged: room for one key tile of fp32 bias entries (128 rows x 128 keys
// as four 128-byte-swizzled boxes of 32 keys), the V ring shrinking to one
// stage when two do not fit beside it.
template <int D, bool kStaged = false>
struct Layout2 {
  static constexpr int kChunk = 128 * 128;
  static constexpr int kChunks = D / 64;
  static constexpr int kTile = kChunks * kChunk;
  static constexpr int kTabBox = 128 * 32 * 4;
  static constexpr int kTabBytes = kStaged ? 4 * kTabBox : 0;
  static constexpr int kMaxSmem = 227 * 1024;
  static constexpr int kVStages = 6 * kTile + kTabBytes + 256 + 1024 <= kMaxSmem ? 2 : 1;
  static constexpr int kQA = 0;
  static constexpr int kK = 2 * kTile;      // [2] stages
  static constexpr int kV = kK + 2 * kTile;  // [kVStages] stages
  static constexpr int kT = kV + kVStages * kTile;
  static constexpr int kBar = kT + kTabBytes;
  static constexpr int kUsed = kBar + 256;
  static constexpr int kAlloc = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
  static_assert(kUsed + 1024 <= kMaxSmem, "shared memory");
};

struct Tc2Args {
  FwdParams p;
  int group;
  int n_pairs;    // CTAs per (sequence, head), or per (sequence, head pair) with heads2
  int heads2;     // 1: tiles A and B are the same 128 rows of two heads of one KV head
  int compact;    // 1: the grid is the compact work list of compact_item()
  int ahead;      // > 0: near its end a CTA prefetches into L2 the Q tiles of the
                  // CTA this many blocks later (the one likely to start next)
  int staged;     // 1: the bias tensor goes through shared memory (kTab 2; heads2 set)
  int tma_o;      // 1: tm_o maps O; full tiles leave through shared memory and TMA
};

// Compact work list for packed batches of at most 32 sequences.  Work item c
// enumerates row blocks b = n_blocks - 1 .. 0 of `rows` rows (the heaviest
// causal rows first, as in the rank-major grid), within a block the
// sequences that have it, within a sequence its `units` head units, so no
// CTA is launched for a block past a sequence's end.  Every warp computes
// the same answer from one coalesced read of cu_seqlens.  false when c lies
// past the last item.
__device__ __forceinline__ bool compact_item(const int32_t *cu_q, int batch, int max_q, int rows,
                                             int n_blocks, int units, int c, int *seq, int *blk,
                                             int *unit) {
  const int lane = threadIdx.x & 31;
  int nq = 0;
  if (lane < batch) {
    nq = __ldg(cu_q + lane + 1) - __ldg(cu_q + lane);
    nq = nq < 0 ? 0 : (nq > max_q ? max_q : nq);  // inconsistent lengths are caught later
  }
  const int tiles = (nq + rows - 1) / rows;
  for (int b = n_blocks - 1; b >= 0; b--) {
    const unsigned m = __ballot_sync(0xffffffffu, tiles > b);
    const int cnt = __popc(m) * units;
    if (c < cnt) {
      *seq = (int)__fns(m, 0, c / units + 1);  // the (c / units)-th sequence with block b
      *unit = c % units;
      *blk = b;
      return true;
    }
    c -= cnt;
  }
  return false;
}

struct Bars2 {
  uint64_t q_full, k_full[2], v_full[2], k_empty[2], v_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];  // [tile A, tile B]
  uint64_t b_full[2];  // kTab 1: the next tile's bias is in the tile's S columns
  uint64_t t_full[4];  // kTab 2: box c of the key tile's entries has landed
  uint64_t t_empty;    // kTab 2: both tiles have added the entries
  uint64_t drain;      // the MMA thread's products have all completed
  uint64_t limit_ns;   // bound of every wait of this call
  uint32_t tmem_base;
  int abort;
  // for a drain after an early exit: Q fills, K / V ring fills (stage =
  // fill % 2) the producer issued, and whether the MMA thread issued any
  int filled_q, filled_k, filled_v, filled_t, mma_issued;
};

static_assert(sizeof(Bars2) <= 256, "barrier block fits its shared-memory slot");

__device__ __forceinline__ bool wait2(Bars2 *b, uint64_t *bar, uint32_t parity, int *err) {
  if (mbar_test_wait(bar, parity)) return true;  // already complete: the cheap path
  if (*reinterpret_cast<volatile int *>(&b->abort)) return false;
  if (mbar_wait(bar, parity, b->limit_ns)) return true;
  *reinterpret_cast<volatile int *>(&b->abort) = 1;
  raise_error(err, ATTN_ERR_DEVICE_TIMEOUT);
  return false;
}

// kPosScale: scale > 0 (the row max of the raw scores gives the max of the
// logits).  kRoundedSum: also sum the bf16-rounded probabilities so the fp32
// output is an exact convex combination of V rows (wanted when the caller
// keeps that output for the backward); without it O is normalised by the
// fp32 sum.  kBias: add the linear positional bias (with kPosScale false:
// the bias must be in the logits before the max).  kTab: add an explicit
// bias tensor, divided by the positive scale so that c2 times the biased
// raw score is the logit in log2 units.  kTab 1: the softmax warps write
// the entries into the tile's S columns before Q K^T accumulates onto them,
// so the scores arrive biased.  kTab 2 (heads2, a tensor shared by the two
// heads, tm_t its map): the entries of each key tile arrive in shared memory
// and each softmax thread adds its row's to the scores it loads.
// tm_o (a.tma_o): O's map; a tile whose 128 rows all lie in its sequence
// writes its bf16 rows into its Q buffer (the 128-byte swizzle of the Q
// load) and one thread stores the tile with TMA: full 128-byte lines instead
// of 16-byte pieces of 32 rows 8 KB apart per warp store.
// kDelta: the backward's per-row term instead of the outputs: the epilogue
// forms D_i = dO_i . O_i from the fp32 output (with kRoundedSum, an exact
// convex combination of V rows) and the row of dO, writes D_i to p.delta
// and stores neither O nor lse.
template <int D, bool kPosScale, bool kRoundedSum, bool kBias, int kTab, bool kDelta>
__global__ void __launch_bounds__(kThreads2, 1)
    fwd_tc2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_t,
                   const __grid_constant__ CUtensorMap tm_o, const Tc2Args a) {
  constexpr bool kTabReg = kTab == 1, kTabSmem = kTab == 2;
  using L = Layout2<D, kTabSmem>;
  // V ring: fill n uses barriers v_full / v_empty[n & 1] (phase (n >> 1) & 1)
  // and shared-memory slot n % kVSt; with one slot, fill n also waits for
  // fill n - 1 to be released (a one-stage ring behind the two-stage
  // barrier pattern, which keeps the MMA thread's code as it is)
  constexpr int kVSt = L::kVStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_base = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw_base + 1023u) & ~1023u) - raw_base);
  Bars2 *b = reinterpret_cast<Bars2 *>(smem + L::kBar);
  const FwdParams &p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // One-dimensional grid, the tile rank slowest (longest causal rows of every
  // (head, sequence) first).  Tiles A and B are rows [i0, i0 + 256) of head h,
  // or with heads2 rows [i0, i0 + 128) of heads h and h + 1 (same KV head),
  // which gives both tiles the same key range.
  const int units = a.heads2 ? p.hq / 2 : p.hq;  // CTAs per (sequence, rank)
  const int rows_b = a.heads2 ? 0 : kTileRows;   // tile B's row offset
  int rank, unit, seq;
  if (a.compact) {
    int blk;
    if (!compact_item(p.cu_q, p.batch, p.max_q, kTileRows + rows_b, a.n_pairs, units,
                      (int)blockIdx.x, &seq, &blk, &unit))
      return;
    rank = a.n_pairs - 1 - blk;
  } else {
    const int per_rank = units * p.batch;
    rank = (int)blockIdx.x / per_rank;
    unit = (int)blockIdx.x % units;
    seq = ((int)blockIdx.x % per_rank) / units;
  }
  const int h = unit * (a.heads2 ? 2 : 1);  // tile A's head
  const int h_b = a.heads2 ? h + 1 : h;     // tile B's head
  const SeqGeom g = load_seq(p.cu_q, p.cu_k, seq, p.total_q, p.total_k, p.max_q, p.max_k, p.mask, p.window);
  if (!g.ok) {
    if (threadIdx.x == 0 && (a.compact || (rank == 0 && h == 0)))
      raise_error(p.err, ATTN_ERR_DEVICE_BOUNDS);
    return;
  }
  const int i0 = (a.n_pairs - 1 - rank) * (kTileRows + rows_b);  // first row of tile A
  if (i0 >= g.nq) return;
  const KvRange kra = plan_kv_tiles(g.mask, g.window, g.nq, g.nk, i0, kTileRows, kTileKeys);
  const KvRange krb =
      plan_kv_tiles(g.mask, g.window, g.nq, g.nk, i0 + rows_b, kTileRows, kTileKeys);
  // Key tiles run n = n0 + u for u in [0, N).  Tile X is active on the u in
  // [lo_X, hi_X) (an empty range when none of its rows sees a key); the two
  // ranges overlap or touch, because tile B's first row starts its keys no
  // later than tile A's last row ends them, so [0, N) has no unused tile.
  const bool act_a = kra.n_end > kra.n_begin, act_b = krb.n_end > krb.n_begin;
  const int n0 = act_a ? kra.n_begin : krb.n_begin;
  const int lo_a = act_a ? kra.n_begin - n0 : 0, hi_a = act_a ? kra.n_end - n0 : 0;
  const int lo_b = act_b ? krb.n_begin - n0 : 0, hi_b = act_b ? krb.n_end - n0 : 0;
  const int N = hi_a > hi_b ? hi_a : hi_b;
  const int hk = h / a.group;
  // Plain scores (no bias in the softmax): a watcher warp certifies the K / V
  // tiles through the P barriers (measured 1.6% faster for the prefill; with
  // a bias the softmax is the longer leg and P(n) then waits for K(n + 1),
  // 9% slower, so the biased instances test the tiles in the MMA thread).
  constexpr bool kWatch = !kTab && !kBias;

  // Copies of Q and of key tile n's K and V (ring stage n % 2, V slot
  // n % kVSt).  Q is read by this CTA alone, each K / V tile by every row
  // block of the KV group: with the policies below Q may leave L2 first so
  // that K / V stay for the others.
  auto load_q = [&](uint64_t pol) {
    mbar_arrive_expect_tx(&b->q_full, 2 * L::kTile);
    for (int t2 = 0; t2 < 2; t2++)
      for (int c = 0; c < L::kChunks; c++)
        tma_load_3d_hint(smem + L::kQA + t2 * L::kTile + c * L::kChunk, &tm_q, &b->q_full, c * 64,
                         t2 ? h_b : h, g.q0 + i0 + t2 * rows_b, pol);
  };
  auto load_k = [&](int n, uint64_t pol) {
    const int st = n & 1;
    mbar_arrive_expect_tx(&b->k_full[st], L::kTile);
    for (int c = 0; c < L::kChunks; c++)
      tma_load_3d_hint(smem + L::kK + st * L::kTile + c * L::kChunk, &tm_k, &b->k_full[st], c * 64,
                       hk, g.k0 + (n0 + n) * kTileKeys, pol);
  };
  auto load_v = [&](int n, uint64_t pol) {
    const int st = n & 1;
    mbar_arrive_expect_tx(&b->v_full[st], L::kTile);
    for (int c = 0; c < L::kChunks; c++)
      tma_load_3d_hint(smem + L::kV + (n % kVSt) * L::kTile + c * L::kChunk, &tm_v,
                       &b->v_full[st], c * 64, hk, g.k0 + (n0 + n) * kTileKeys, pol);
  };

  if (threadIdx.x == 0) {
    mbar_init(&b->q_full, 1);
    for (int s = 0; s < 2; s++) {
      mbar_init(&b->k_full[s], 1);
      mbar_init(&b->v_full[s], 1);
      mbar_init(&b->k_empty[s], 1);
      mbar_init(&b->v_empty[s], 1);
      mbar_init(&b->s_full[s], 1);
      // kWatch: warp 2 adds one arrival per product (see below)
      mbar_init(&b->p_full[s], kWatch ? 129 : 128);
      // kTab 1 with heads2: each tile's threads store half of every row's
      // bias into both tiles' S columns, so both tiles arrive on both
      mbar_init(&b->b_full[s], kTabReg && a.heads2 ? 256 : 128);
      mbar_init(&b->pv_done[s], 1);
    }
    for (int c = 0; c < 4; c++) mbar_init(&b->t_full[c], 1);
    mbar_init(&b->t_empty, 256);  // every softmax thread of both tiles
    mbar_init(&b->drain, 1);
    b->limit_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    b->abort = 0;
    b->filled_q = b->filled_k = b->filled_v = b->filled_t = b->mma_issued = 0;
    fence_mbar_init();
    // Thread 0 is the producer: Q and key tile 0 leave before the block-wide
    // sync, so their latency overlaps the allocation of tensor memory
    if (N > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_kv = l2_policy_evict_last();
      load_q(l2_policy_evict_first());
      load_k(0, pol_kv);
      load_v(0, pol_kv);
    }
  }
  if (warp == 1) {
    tmem_alloc(&b->tmem_base, kCols2);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b->tmem_base;
  // TMEM columns: S_A 0, S_B 128, O_A 256, O_B 256 + D.
  const uint32_t sQ = smem_u32(smem + L::kQA);
  const uint32_t sK = smem_u32(smem + L::kK);
  const uint32_t sV = smem_u32(smem + L::kV);

  if (warp < 4) {
    reg_dealloc<kRegsCtl>();
    if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && N > 0) {
      int filled_k = 1, filled_v = 1;  // Q and key tile 0: issued before the sync
      const uint64_t pol_kv = l2_policy_evict_last();
      for (int n = 1; n < N; n++) {
        const int st = n & 1, u = n >> 1;
        if (n >= 2 && !wait2(b, &b->k_empty[st], (u - 1) & 1, p.err)) break;
        filled_k++;
        load_k(n, pol_kv);
        if (n >= kVSt &&
            !wait2(b, &b->v_empty[(n - kVSt) & 1], ((n - kVSt) >> 1) & 1, p.err))
          break;
        filled_v++;
        load_v(n, pol_kv);
      }
      // The grid runs one CTA per SM at a time, so a CTA's start waits on its
      // Q tiles; warm L2 with those of the CTA `ahead` blocks later (about
      // one wave on), which starts when some SM frees up.
      if (!a.compact && a.ahead > 0) {
        const long long nb = (long long)blockIdx.x + a.ahead;
        if (nb < (long long)gridDim.x) {
          const int per_rank = units * p.batch;
          const int rank2 = (int)(nb / per_rank), unit2 = (int)(nb % units);
          const int seq2 = (int)((nb % per_rank) / units);
          const int q0_2 = __ldg(p.cu_q + seq2), nq2 = __ldg(p.cu_q + seq2 + 1) - q0_2;
          const int i0_2 = (a.n_pairs - 1 - rank2) * (kTileRows + rows_b);
          const int h2 = unit2 * (a.heads2 ? 2 : 1), hb2 = a.heads2 ? h2 + 1 : h2;
          if (i0_2 < nq2)
            for (int t2 = 0; t2 < 2; t2++)
              for (int c = 0; c < L::kChunks; c++)
                tma_prefetch_3d(&tm_q, c * 64, t2 ? hb2 : h2, q0_2 + i0_2 + t2 * rows_b);
        }
      }
      b->filled_q = 1;  // for a drain after an early exit
      b->filled_k = filled_k;
      b->filled_v = filled_v;
    }
    } else if (warp == 2) {
    // --------------------------------------------------------- TMA watcher
    // kWatch: for each key tile n, once V(n) and K(n + 1) have landed,
    // one more arrival on p_full of each tile with a product n (after that
    // tile's previous phase has completed, so the arrival counts toward the
    // phase of product n).
    if (kWatch && lane == 0 && N > 0) {
      bool ok = true;
      for (int n = 0; ok && n < N; n++) {
        ok = wait2(b, &b->v_full[n & 1], (n >> 1) & 1, p.err);
        if (ok && n + 1 < N) ok = wait2(b, &b->k_full[(n + 1) & 1], ((n + 1) >> 1) & 1, p.err);
        for (int x2 = 0; ok && x2 < 2; x2++) {
          const int lo = x2 ? lo_b : lo_a, hi = x2 ? hi_b : hi_a;
          if (n < lo || n >= hi) continue;
          if (n > lo) ok = wait2(b, &b->p_full[x2], (n - 1 - lo) & 1, p.err);
          if (ok) mbar_arrive(&b->p_full[x2]);
        }
      }
    }
    // ------------------------------------------------- bias entries (kTab 2)
    // Key tile n0 + u's entries for the CTA's 128 rows (both tiles' heads
    // share them), as four boxes of 32 keys, once both tiles have added the
    // previous tile's.  Rows and keys past the tensor's extent read as 0
    // (their scores are masked or never stored).
    if (kTabSmem && lane == 0 && N > 0) {
      tma_prefetch_desc(&tm_t);
      const int tz = p.bss ? seq : 0;
      int filled_t = 0;
      for (int u = 0; u < N; u++) {
        if (u > 0 && !wait2(b, &b->t_empty, (u - 1) & 1, p.err)) break;
        const int j0 = (n0 + u) * kTileKeys;
        filled_t++;
        for (int c = 0; c < 4; c++) {
          mbar_arrive_expect_tx(&b->t_full[c], L::kTabBox);
          tma_load_3d(smem + L::kT + c * L::kTabBox, &tm_t, &b->t_full[c], j0 + 32 * c, i0, tz);
        }
      }
      b->filled_t = filled_t;
    }
    } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0 && N > 0) {
      b->mma_issued = 1;
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kTileKeys, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 0, 1);
      // Descriptors are built once; a byte offset below 256 KB adds to the
      // start-address field (16-byte units) without carrying out of it.
      const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024);
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024);
      const uint64_t dV0 = smem_desc_sw128(sV, L::kChunk, 1024);
      auto issue_qk = [&](int x, int st) {  // S_x = Q_x K^T
        const uint64_t dq = dQ0 + (uint64_t)((x * L::kTile) >> 4);
        const uint64_t dk = dK0 + (uint64_t)((st * L::kTile) >> 4);
        const uint32_t d_tmem = tmem + (uint32_t)(x * kTileKeys);
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint64_t off = (uint64_t)((((kk >> 2) * L::kChunk) + (kk & 3) * 32) >> 4);
          mma_bf16_ss(d_tmem, dq + off, dk + off, idesc_qk, (kTabReg || kk > 0) ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int x, int st, bool acc) {  // O_x += P V, P in tensor memory
        uint64_t dv = dV0 + (uint64_t)(((kVSt == 2 ? st : 0) * L::kTile) >> 4);
        // one V slot: the descriptors would be loop-invariant, and holding
        // them between products costs the control warps more registers than
        // they have; an opaque copy keeps them computed per product
        if constexpr (kVSt == 1) asm volatile("" : "+l"(dv));
        const uint32_t d_tmem = tmem + 256u + (uint32_t)(x * D);
        const uint32_t a_tmem = tmem + (uint32_t)(x * kTileKeys + 64);  // P: S columns [64, 128)
#pragma unroll
        for (int kk = 0; kk < kTileKeys / 16; kk++)
          mma_bf16_ts(d_tmem, a_tmem + kk * 8, dv + (uint64_t)((kk * 16 * 128) >> 4), idesc_pv,
                      (acc || kk > 0) ? 1u : 0u);
      };
      // Tile X's c-th product (c = n - lo_X) completes phase c of its
      // s_full / p_full / pv_done barriers.
      auto in_a = [&](int n) { return n >= lo_a && n < hi_a; };
      auto in_b = [&](int n) { return n >= lo_b && n < hi_b; };
      // kTab 1: Q K^T of tile X's c-th product accumulates onto the bias its
      // softmax warps stored, announced by phase c of b_full[X]
      bool ok = wait2(b, &b->q_full, 0, p.err) && wait2(b, &b->k_full[0], 0, p.err);
      if (ok && in_a(0) && (!kTabReg || (ok = wait2(b, &b->b_full[0], 0, p.err)))) {
        tc_fence_after();
        issue_qk(0, 0);
        mma_commit(&b->s_full[0]);
      }
      if (ok && in_b(0) && (!kTabReg || (ok = wait2(b, &b->b_full[1], 0, p.err)))) {
        tc_fence_after();
        issue_qk(1, 0);
        mma_commit(&b->s_full[1]);
      }
      if (ok) mma_commit(&b->k_empty[0]);
      // kWatch: phase c of p_full[X] (tile X's product n = lo_X + c)
      // also certifies that V(n) and K(n + 1) have landed (warp 2 arrives on
      // it only then), so the MMA thread tests those barriers only where no
      // such phase covers them: a barrier test stalls the issuing thread long
      // enough for the tensor pipe's short queue to run dry.
      for (int n = 0; ok && n < N; n++) {
        const int st = n & 1, n1 = n + 1, st1 = n1 & 1;
        bool v_ready = false, k1_ready = false;
        if (in_a(n)) {
          if (!(ok = wait2(b, &b->p_full[0], (n - lo_a) & 1, p.err))) break;
          if (!kWatch && !(ok = wait2(b, &b->v_full[st], (n >> 1) & 1, p.err))) break;
          v_ready = true;
          k1_ready = kWatch;
          tc_fence_after();
          issue_pv(0, st, n > lo_a);
          mma_commit(&b->pv_done[0]);
        }
        // kTab 1: tile A's next Q K^T waits for its bias, which waits for
        // P_A V: tile B's P V goes first
        if (!kTabReg && in_a(n1)) {
          if (!k1_ready && !(ok = wait2(b, &b->k_full[st1], (n1 >> 1) & 1, p.err))) break;
          k1_ready = true;
          tc_fence_after();
          issue_qk(0, st1);
          mma_commit(&b->s_full[0]);
        }
        if (in_b(n)) {
          if (!(ok = wait2(b, &b->p_full[1], (n - lo_b) & 1, p.err))) break;
          if (!kWatch && !v_ready && !(ok = wait2(b, &b->v_full[st], (n >> 1) & 1, p.err))) break;
          if (kWatch) k1_ready = true;
          tc_fence_after();
          issue_pv(1, st, n > lo_b);
          mma_commit(&b->pv_done[1]);
        }
        mma_commit(&b->v_empty[st]);
        if (kTabReg && in_a(n1)) {
          if (!(ok = wait2(b, &b->k_full[st1], (n1 >> 1) & 1, p.err))) break;
          k1_ready = true;
          if (!(ok = wait2(b, &b->b_full[0], (n1 - lo_a) & 1, p.err))) break;
          tc_fence_after();
          issue_qk(0, st1);
          mma_commit(&b->s_full[0]);
        }
        if (in_b(n1)) {
          if (!k1_ready && !(ok = wait2(b, &b->k_full[st1], (n1 >> 1) & 1, p.err))) break;
          if (kTabReg && !(ok = wait2(b, &b->b_full[1], (n1 - lo_b) & 1, p.err))) break;
          tc_fence_after();
          issue_qk(1, st1);
          mma_commit(&b->s_full[1]);
        }
        if (n1 < N) mma_commit(&b->k_empty[st1]);
      }
    }
    }
  } else {
    reg_alloc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int x = warp >= 8 ? 1 : 0;  // tile A (0) or B (1)
    const int wq = warp & 3;          // TMEM lane quarter this warp may access
    const int r = wq * 32 + lane;
    const int hx = x ? h_b : h;         // this tile's head
    const int i = i0 + x * rows_b + r;  // this thread's row
    const bool row_in = i < g.nq;
    const int t = g.q0 + i;
    const int row_limit = row_key_limit(g.mask, i, g.nq, g.nk);
    const int row_first = row_key_first(g.mask, g.window, i, g.nq, g.nk);
    const KvRange &kr = x ? krb : kra;
    const int n_mine = kr.n_end - kr.n_begin;  // products of this tile
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    const uint32_t s_col = t_lane + (uint32_t)(x * kTileKeys);
    const uint32_t o_col = t_lane + 256u + (uint32_t)(x * D);
    const float c2 = p.scale_log2;
    const float cm = kPosScale ? c2 : 1.f;  // multiplier still to apply to raw scores
    static_assert(!(kBias && kPosScale), "the bias needs the logits before the max");
    static_assert(!kTab || (kPosScale && !kBias), "the tensor bias rides on the raw scores");
    const float slope2 = kBias ? __ldg(p.slopes + hx) * kLog2e : 0.f;
    // causal mask and positive scale: the bias is linear over every allowed key
    const bool bias_linear = g.mask != ATTN_MASK_NONE && c2 > 0.f;
    const float bound = (float)(i + causal_offset(g.mask, g.nq, g.nk));  // the row's causal bound
    float m_ref = -INFINITY, l = 0.f, lr = 0.f;
    bool ok = true;
    // kTab 1: this row's bias entries for key tile n, divided by the positive
    // scale (so that c2 times the accumulated score is the biased logit in
    // log2 units), into the tile's S columns; keys past the sequence and rows
    // past it get 0 (their lanes are masked or never stored).
    const float *brow = kTabReg && row_in ? btab_row(p.btab, p.bss, p.bhs, p.brs, seq, hx, i) : nullptr;
    const float inv_scale = kTab ? 1.f / p.scale : 0.f;
    // the loads are issued before the wait that gates the store, so their
    // latency overlaps it
    auto load_bias = [&](int n, uint32_t (&bv)[kTileKeys]) {
      const int j0 = n * kTileKeys;
      const bool vec = brow && j0 + kTileKeys <= g.nk &&
                       ((reinterpret_cast<uintptr_t>(brow + j0) & 15) == 0);
      if (vec) {
#pragma unroll
        for (int e = 0; e < kTileKeys; e += 4) {
          const float4 f = __ldg(reinterpret_cast<const float4 *>(brow + j0 + e));
          bv[e] = __float_as_uint(f.x * inv_scale);
          bv[e + 1] = __float_as_uint(f.y * inv_scale);
          bv[e + 2] = __float_as_uint(f.z * inv_scale);
          bv[e + 3] = __float_as_uint(f.w * inv_scale);
        }
      } else {
#pragma unroll
        for (int e = 0; e < kTileKeys; e++) {
          const int j = j0 + e;
          bv[e] = __float_as_uint(brow && j < g.nk ? __ldg(brow + j) * inv_scale : 0.f);
        }
      }
    };
    auto store_bias = [&](const uint32_t (&bv)[kTileKeys]) {
#pragma unroll
      for (int c = 0; c < kTileKeys / 32; c++)
        tmem_st32(s_col + c * 32, *reinterpret_cast<const uint32_t(*)[32]>(bv + 32 * c));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&b->b_full[x]);
    };
    // With heads2 the tiles hold the same rows of two heads, and a bias
    // shared by the heads is the same for both: tile X's threads load keys
    // [64 X, 64 X + 64) of their row and store them into both tiles' S
    // columns, so every row's entries cross L2 once per CTA, not twice.
    const bool share = kTabReg && a.heads2;
    auto load_bias_half = [&](int n, uint32_t (&bv)[kTileKeys / 2]) {
      const int j0 = n * kTileKeys + x * (kTileKeys / 2);
      const bool vec = brow && j0 + kTileKeys / 2 <= g.nk &&
                       ((reinterpret_cast<uintptr_t>(brow + j0) & 15) == 0);
      if (vec) {
#pragma unroll
        for (int e = 0; e < kTileKeys / 2; e += 4) {
          const float4 f = __ldg(reinterpret_cast<const float4 *>(brow + j0 + e));
          bv[e] = __float_as_uint(f.x * inv_scale);
          bv[e + 1] = __float_as_uint(f.y * inv_scale);
          bv[e + 2] = __float_as_uint(f.z * inv_scale);
          bv[e + 3] = __float_as_uint(f.w * inv_scale);
        }
      } else {
#pragma unroll
        for (int e = 0; e < kTileKeys / 2; e++) {
          const int j = j0 + e;
          bv[e] = __float_as_uint(brow && j < g.nk ? __ldg(brow + j) * inv_scale : 0.f);
        }
      }
    };
    auto store_bias_shared = [&](const uint32_t (&bv)[kTileKeys / 2]) {
      const uint32_t half_col = t_lane + (uint32_t)(x * (kTileKeys / 2));
#pragma unroll
      for (int y = 0; y < 2; y++)
#pragma unroll
        for (int c = 0; c < kTileKeys / 64; c++)
          tmem_st32(half_col + (uint32_t)(y * kTileKeys) + c * 32,
                    *reinterpret_cast<const uint32_t(*)[32]>(bv + 32 * c));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&b->b_full[0]);
      mbar_arrive(&b->b_full[1]);
    };
    if (kTabReg && n_mine > 0) {
      if (share) {
        uint32_t bv[kTileKeys / 2];
        load_bias_half(kr.n_begin, bv);
        store_bias_shared(bv);
      } else {
        uint32_t bv[kTileKeys];
        load_bias(kr.n_begin, bv);
        store_bias(bv);
      }
    }
    for (int it = 0; it < n_mine; it++) {
      const int n = kr.n_begin + it;  // key tile in the sequence
      ok = wait2(b, &b->s_full[x], it & 1, p.err);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the whole row of 128 scores in one TMEM load instruction (measured 1%
      // faster than four of 32 columns; one store of 64 columns for P was not)
      uint32_t v[kTileKeys];
      static_assert(kTileKeys == 128, "one 128-column load");
      tmem_ld128(s_col, v);
      tmem_wait_ld();
      if constexpr (kTabSmem) {
        // fill `it` of the entries (both tiles run the same key tiles): box c
        // holds keys [32 c, 32 c + 32) for the 128 rows, row r's 16-byte
        // chunk k at 128 r + 16 (k ^ (r & 7)) (the 128-byte swizzle), so a
        // warp's 32 rows read distinct banks.  Added before the mask below,
        // which overwrites masked lanes whatever they hold.
        const uint64_t is2 = f2(inv_scale, inv_scale);
        const uint8_t *t_row = smem + L::kT + r * 128;
#pragma unroll
        for (int c = 0; c < 4; c++) {
          if (!wait2(b, &b->t_full[c], it & 1, p.err)) ok = false;
#pragma unroll
          for (int k = 0; k < 8; k++) {
            const float4 f =
                *reinterpret_cast<const float4 *>(t_row + c * L::kTabBox + ((k ^ (r & 7)) << 4));
            const int e = 32 * c + 4 * k;
            float y0, y1, y2, y3;
            f2_split(ffma2(f2(f.x, f.y), is2, f2(__uint_as_float(v[e]), __uint_as_float(v[e + 1]))), y0, y1);
            f2_split(ffma2(f2(f.z, f.w), is2, f2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]))), y2, y3);
            v[e] = __float_as_uint(y0);
            v[e + 1] = __float_as_uint(y1);
            v[e + 2] = __float_as_uint(y2);
            v[e + 3] = __float_as_uint(y3);
          }
        }
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        mbar_arrive(&b->t_empty);
      }
      if (!kr.full(n)) {
        // lanes outside [first, limit) of this row: first <= limit, so one
        // unsigned compare tests both ends
        const int first = row_first - n * kTileKeys;
        const unsigned span = (unsigned)(row_limit - row_first);
#pragma unroll
        for (int e = 0; e < kTileKeys; e++)
          if ((unsigned)(e - first) >= span) v[e] = 0xff800000u;
      }
      if constexpr (!kPosScale) {
        const float dist0 = bound - (float)(n * kTileKeys);
        if (kBias && bias_linear) {
          // Every allowed key sits at or before the causal bound, so the bias
          // is -slope2 (dist0 - e) with dist0 - e >= 0 exact in fp32, and a
          // masked lane's -inf stays -inf (c2 > 0): z = y c2 - slope2 (dist0 - e),
          // two lanes per instruction.
          const uint64_t c2x2 = f2(c2, c2), ns2 = f2(-slope2, -slope2), d2 = f2(dist0, dist0);
#pragma unroll
          for (int e = 0; e < kTileKeys; e += 2) {
            const uint64_t t2 = fadd2(d2, f2(-(float)e, -(float)(e + 1)));
            const uint64_t z2 = ffma2(ns2, t2, fmul2(f2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), c2x2));
            float z0, z1;
            f2_split(z2, z0, z1);
            v[e] = __float_as_uint(z0);
            v[e + 1] = __float_as_uint(z1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < kTileKeys; e++) {
            const float y = __uint_as_float(v[e]);
            float z = y * c2;
            if constexpr (kBias) z += pos_bias2(slope2, dist0, e);
            v[e] = __float_as_uint(y == -INFINITY ? -INFINITY : z);
          }
        }
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int e = 0; e < kTileKeys; e += 2)
        m4[(e >> 1) & 3] = fmax3(m4[(e >> 1) & 3], __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
      float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      if (kPosScale) mt *= c2;
      const float m_new = mt > m_ref + kRescale2 ? mt : m_ref;
      const float alpha = m_new == m_ref ? 1.f : fast_exp2(m_ref - m_new);
      const float base = m_new == -INFINITY ? 0.f : m_new;
      // P = 2^(raw * c - base), two lanes per instruction; l sums fp32 P (for
      // lse), lr the bf16-rounded P that P V uses (so O / lr is an exact
      // convex combination of V rows).  Each half of 64 scores becomes 32
      // packed bf16 pairs over S columns [64, 128): keys [0, 64) at 64, keys
      // [64, 128) at 96.
      const uint64_t cx2 = f2(cm, cm), nb2 = f2(-base, -base);
      uint64_t s2[2] = {0, 0}, r2[2] = {0, 0};
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          float x0, x1;
          f2_split(ffma2(f2(__uint_as_float(v[64 * hh + e]), __uint_as_float(v[64 * hh + e + 1])),
                         cx2, nb2),
                   x0, x1);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          const int k = e / 2;
          s2[k & 1] = fadd2(s2[k & 1], f2(p0, p1));
          pk[k] = pack_bf16x2(p0, p1);
          if constexpr (kRoundedSum)
            r2[k & 1] = fadd2(r2[k & 1], f2(__uint_as_float(pk[k] << 16),
                                            __uint_as_float(pk[k] & 0xffff0000u)));
        }
        tmem_st32(s_col + 64 + 32 * hh, pk);
      }
      {
        float a0, a1, b0, b1;
        f2_split(fadd2(s2[0], s2[1]), a0, a1);
        f2_split(fadd2(r2[0], r2[1]), b0, b1);
        l = l * alpha + (a0 + a1);
        lr = kRoundedSum ? lr * alpha + (b0 + b1) : l;
      }
      m_ref = m_new;
      // S_x(n) landed after every earlier product of this thread, so the
      // previous P V into O_x is complete: O_x may be rescaled now.
      if (it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < D / 32; c++) {
          uint32_t o32[32];
          tmem_ld32(o_col + c * 32, o32);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e++) o32[e] = __float_as_uint(__uint_as_float(o32[e]) * alpha);
          tmem_st32(o_col + c * 32, o32);
        }
      }
      tmem_wait_st();  // P (S columns [64, 128)) and any rescaled O are in place
      tc_fence_before();
      mbar_arrive(&b->p_full[x]);
      if (kTabReg && it + 1 < n_mine) {
        // the next tile's bias may overwrite S once P V has read P (with
        // share, both tiles' P: both tiles' S columns are written)
        if (share) {
          uint32_t bv[kTileKeys / 2];
          load_bias_half(n + 1, bv);
          ok = wait2(b, &b->pv_done[0], it & 1, p.err) && wait2(b, &b->pv_done[1], it & 1, p.err);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          store_bias_shared(bv);
        } else {
          uint32_t bv[kTileKeys];
          load_bias(n + 1, bv);
          ok = wait2(b, &b->pv_done[x], it & 1, p.err);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          store_bias(bv);
        }
      }
    }
    if (ok && n_mine > 0) {
      ok = wait2(b, &b->pv_done[x], (n_mine - 1) & 1, p.err);
      if (ok) tc_fence_after();
    }
    // ------------------------------------------------------------ epilogue
    const bool have = __all_sync(0xffffffffu, ok) && n_mine > 0;
    const float inv = lr > 0.f ? 1.f / lr : 0.f;
    const float lse2 = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
    if constexpr (kDelta) {
      // D_i = dO_i . O_i, O_i = acc / lr before any rounding
      const __nv_bfloat16 *dsrc =
          reinterpret_cast<const __nv_bfloat16 *>(p.dout) + toff(p.sdo, t, hx);
      float dsum = 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; c++) {
        uint32_t o32[32];
        if (have) {  // warp-uniform
          tmem_ld32(o_col + c * 32, o32);
          tmem_wait_ld();
          if (row_in) {
#pragma unroll
            for (int e = 0; e < 32; e += 8) {
              const uint4 w = *reinterpret_cast<const uint4 *>(dsrc + c * 32 + e);
              const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int k2 = 0; k2 < 4; k2++) {
                dsum = fmaf(__uint_as_float(o32[e + 2 * k2]), __uint_as_float(wv[k2] << 16), dsum);
                dsum = fmaf(__uint_as_float(o32[e + 2 * k2 + 1]),
                            __uint_as_float(wv[k2] & 0xffff0000u), dsum);
              }
            }
          }
        }
      }
      if (row_in) p.delta[(size_t)hx * p.total_q + t] = have ? dsum * inv : 0.f;
    } else {
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.o) + toff(p.so, t, hx);
      // the same for the tile's 128 threads: rows all in the sequence, and
      // products run (so the Q load into the buffer has landed and every
      // product that read it has completed)
      // (not in the bias-tensor instances, whose softmax warps it would push
      // past their registers)
      const bool via_tma =
          !kTab && a.tma_o && n_mine > 0 && i0 + x * rows_b + kTileRows <= g.nq;
      uint8_t *so = smem + L::kQA + x * L::kTile;
  #pragma unroll
      for (int c = 0; c < D / 32; c++) {
        uint32_t o32[32];
        if (have) {
          tmem_ld32(o_col + c * 32, o32);
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
            if (via_tma) {  // feature f = 32 c + e: chunk f / 64, 16-byte unit (f % 64) / 8
              const int f = c * 32 + e, k = (f % 64) / 8;
              st_shared_v4(smem_u32(so + (f / 64) * L::kChunk + r * 128 + ((k ^ (r & 7)) << 4)),
                           w.x, w.y, w.z, w.w);
            } else {
              __stcs(reinterpret_cast<uint4 *>(dst + c * 32 + e), w);  // written once: streaming
            }
          }
          if (p.o_f32) {
            float *df = p.o_f32 + ((size_t)t * p.hq + hx) * D + c * 32;
  #pragma unroll
            for (int e = 0; e < 32; e += 4) {
              float4 f;
              f.x = have ? __uint_as_float(o32[e]) * inv : 0.f;
              f.y = have ? __uint_as_float(o32[e + 1]) * inv : 0.f;
              f.z = have ? __uint_as_float(o32[e + 2]) * inv : 0.f;
              f.w = have ? __uint_as_float(o32[e + 3]) * inv : 0.f;
              __stcs(reinterpret_cast<float4 *>(df + e), f);
            }
          }
        }
      }
      if (via_tma) {
        fence_proxy_async_smem();    // the rows are visible to the TMA unit
        named_bar_sync(1 + x, 128);  // once the tile's 128 rows are written
        if (wq == 0 && lane == 0) {
          const uint64_t pol = l2_policy_evict_first();  // written once
          for (int ch = 0; ch < L::kChunks; ch++)
            tma_store_3d_hint(&tm_o, so + ch * L::kChunk, ch * 64, hx, g.q0 + i0 + x * rows_b, pol);
          bulk_commit();
          bulk_wait_read();  // the buffer stays allocated until the copies have read it
        }
      }
      if (row_in && p.lse) p.lse[(size_t)hx * p.total_q + t] = have ? lse2 * kLn2 : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  // A block in which a wait gave up may still have copies and products in
  // flight; they must land before its tensor memory is freed and it exits
  // (the flag is only set before the barrier above, so every thread reads
  // the same value).  On the normal path every copy and product has been
  // waited for already.
  if (*reinterpret_cast<volatile int *>(&b->abort)) {
    if (threadIdx.x == 0) {
      bool drained = drain_phase(&b->q_full, b->filled_q);
      for (int st = 0; st < 2; st++)
        drained = drain_phase(&b->k_full[st], ring_armed(b->filled_k, st, 2)) &&
                  drain_phase(&b->v_full[st], ring_armed(b->filled_v, st, 2)) && drained;
      for (int c = 0; c < 4; c++)  // every fill arms each box's barrier once
        drained = drain_phase(&b->t_full[c], b->filled_t) && drained;
      if (!drained) raise_error(p.err, ATTN_ERR_DEVICE_TIMEOUT);
    }
    if (threadIdx.x == 32 && b->mma_issued && !drain_mma(&b->drain))
      raise_error(p.err, ATTN_ERR_DEVICE_TIMEOUT);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kCols2);
  }
}

// Maps: q, k, v, the bias tensor (m[3], kTab 2 only) and O (m[4], with a.tma_o).
template <int D, bool kPos, bool kRs, bool kBias, int kTab = 0, bool kDelta = false>
cudaError_t launch2(const Tc2Args &a, const CUtensorMap (&m)[5], unsigned ctas, cudaStream_t st) {
  constexpr int smem = Layout2<D, kTab == 2>::kAlloc;
  static bool configured[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(fwd_tc2_kernel<D, kPos, kRs, kBias, kTab, kDelta>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  fwd_tc2_kernel<D, kPos, kRs, kBias, kTab, kDelta><<<ctas, kThreads2, smem, st>>>(m[0], m[1], m[2],
                                                                                  m[3], m[4], a);
  return cudaGetLastError();
}


// Shared set-up of the launchers: the CTA arrangement (two heads of one KV
// head per CTA when the group pairs up: both tiles then have the same key
// range, no idle diagonal tile (windowed prefill 2%, linear bias 1.5%
// faster, causal unchanged); with a bias tensor it measured 7% slower, so
// those keep two row blocks of one head) and the tensor maps m: q, k, v,
// the bias tensor when it goes through shared memory (zeroed otherwise) and
// O when there is one and TMA can address it (zeroed otherwise).  false
// when a map of q, k or v is rejected or the grid is too large.
inline bool setup_tc2(const FwdParams &p, Tc2Args *a, CUtensorMap (&m)[5], long long *ctas,
                      int *rows_per_cta) {
  CUtensorMap *mq = &m[0], *mk = &m[1], *mv = &m[2], *mt = &m[3], *mo = &m[4];
  a->p = p;
  a->group = p.hq / p.hkv;
  // a bias tensor pairs heads only when the heads share it (then the two
  // tiles share its entries too)
  a->heads2 = a->group % 2 == 0 && (!p.btab || p.bhs == 0) ? 1 : 0;
  // Shared entries of d = 128 heads stream through shared memory when TMA
  // can address them (16-byte aligned base and strides); otherwise the
  // softmax warps load them (kTab 1).
  memset(mt, 0, sizeof(*mt));
  a->staged = a->heads2 && p.btab && p.d == 128 &&
                      make_bias_map(mt, p.btab, p.max_k, p.max_q, p.batch, p.brs, p.bss)
                  ? 1
                  : 0;
  *rows_per_cta = a->heads2 ? kTileRows : 2 * kTileRows;
  a->n_pairs = (p.max_q + *rows_per_cta - 1) / *rows_per_cta;
  const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!make_map(mq, p.q, p.d, p.hq, p.total_q, 1, kTileRows, bf, p.sq.hs, p.sq.ts) ||
      !make_map(mk, p.k, p.d, p.hkv, p.total_k, 1, kTileKeys, bf, p.sk.hs, p.sk.ts) ||
      !make_map(mv, p.v, p.d, p.hkv, p.total_k, 1, kTileKeys, bf, p.sv.hs, p.sv.ts))
    return false;
  memset(mo, 0, sizeof(*mo));
  a->tma_o = p.o && make_map(mo, p.o, p.d, p.hq, p.total_q, 1, kTileRows, bf, p.so.hs, p.so.ts)
                 ? 1
                 : 0;
  const int units = a->heads2 ? p.hq / 2 : p.hq;
  *ctas = (long long)a->n_pairs * units * p.batch;
  // A packed batch of at most 32 sequences takes the compact work list when
  // it is shorter: sum_s ceil(nq_s / R) <= (total_q + batch (R - 1)) / R
  // items per head unit, against n_pairs per sequence and unit otherwise.
  a->compact = 0;
  a->ahead = internal_sm_count();
  if (p.batch <= 32) {
    const long long R = *rows_per_cta;
    const long long items = ((long long)p.total_q + p.batch * (R - 1)) / R * units;
    if (items < *ctas) {
      a->compact = 1;
      *ctas = items;
    }
  }
  return *ctas < (1LL << 31);
}

}  // namespace
}  // namespace attn
