// bwd_fused.cu -- tensor-core backward in one kernel per key tile (head_dim
// 128): the dK/dV kernel's walk over the query rows that see a 128-key tile
// also produces those rows' dQ contributions, so S and dP are computed once
// per (row, key) pair instead of once in each of two kernels.  Per 64-row
// step of every query head of the KV group, on tcgen05:
//   S^T = K Q^T, dP^T = V dO^T                (M = 128 keys, N = 64 rows)
//   P^T = 2^(c S^T - lse2), dS^T = P^T (dP^T - D)   (registers, thread = key)
//   dV += P^T dO, dK += dS^T Q                (M = 128 keys, N = d, in TMEM)
//   dQ^T = K^T dS^T                           (M = d, N = 64 rows)
// ("attention-algorithm-error-and-complexity-tests", third and fourth
// paragraphs: the gradients of every input, GQA sums over shared heads).
// dQ^T takes K from the same shared-memory tile as S^T (read d-major) and
// dS^T from a shared-memory copy the math warps write beside the tensor-memory
// one; a readout warpgroup moves each step's dQ^T from tensor memory through
// shared memory into an fp32 accumulator in global memory with TMA
// reduce-adds, since the rows' other key tiles belong to other CTAs.  A last
// kernel scales the accumulator back
// (the fp16 copies' power-of-two factors and the softmax scale) and writes
// dQ in bf16.  The summation order of dQ then depends on the CTAs' timing:
// the two-kernel backward stays available for bit-reproducible gradients.
//
// Tensor memory (512 columns): buffer b in {0, 1} holds a step's S^T at
// 64 b and dP^T at 128 + 64 b; the math warps write P^T and dS^T (fp16,
// packed two per column) over the S^T columns, so the dP^T columns are free
// for that step's dQ^T; dV at 256, dK at 384.  The MMA thread issues a
// step's dQ^T first, then dV and dK, and the score products of the step two
// ahead into the same buffer, dP^T only after the readout warps have copied
// dQ^T out; the readout overlaps dV, dK and S^T on the tensor pipe.
#include <stdio.h>

#include <type_traits>

#include "bwd_tc.cuh"
#include "common.cuh"
#include "plan.h"
#include "sm100.cuh"
#include "tma_map.h"

namespace attn {
using namespace sm100;

int internal_sm_count();

namespace {

// warps 0 TMA, 1 MMA + TMEM, 2 tile watcher (unbiased instances), 3 idle
// (warpgroup 0); 4-11 math, two per TMEM
// lane quarter (warpgroups 1-2); 12-15 dQ readout, one per lane quarter
constexpr int kThreadsF = 512;
constexpr uint32_t kTmemColsF = 512;
constexpr int kDF = 128;
constexpr int kChunkKV = 128 * 128;  // [128 keys x 64 fp16] swizzled chunk
constexpr int kChunkQ = 64 * 128;    // [64 rows x 64 fp16] swizzled chunk
// register split: 128 x 88 + 256 x 176 + 128 x 72 = 512 x 128 (the launch's)
constexpr uint32_t kRegCtl = 88, kRegMath = 176, kRegOut = 72;
static_assert(128 * kRegCtl + 256 * kRegMath + 128 * kRegOut <= 512 * 128,
              "register split fits the launch's allocation");

struct LayoutF {
  static constexpr int kChunks = kDF / 64;
  static constexpr int kKV = kChunks * kChunkKV;  // K or V tile
  static constexpr int kQT = kChunks * kChunkQ;   // Q or dO tile (64 rows)
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKV;
  static constexpr int kQ = kV + kKV;                // [kStagesA] stages
  static constexpr int kDO = kQ + kStagesA * kQT;    // [kStagesA]
  static constexpr int kDS = kDO + kStagesA * kQT;   // dS^T [128 keys][64 rows] fp16, swizzled
  static constexpr int kRow = kDS + kKeysA * kRowsA * 2;  // [2] x {-lse2[64], -D[64]}
  static constexpr int kBar = kRow + 2 * 2 * kRowsA * 4;
  // dQ^T readout: per readout warp two [16 rows x 32 fp32] tiles for the
  // TMA reduce-adds into the accumulator
  static constexpr int kDQ = (kBar + 512 + 1023) / 1024 * 1024;
  static constexpr int kDQWarp = 2 * 16 * 32 * 4;
  static constexpr int kUsed = kDQ + 4 * kDQWarp;
  static constexpr int kAlloc = kUsed + 1024;
};
static_assert(LayoutF::kAlloc <= 227 * 1024, "shared memory of one CTA");

struct BarsF {
  // as the dK/dV kernel's, plus dq_full (a step's dQ^T product done: the
  // readout may start and the dS^T copy may be overwritten) and dq_free (the
  // readout warps have copied dQ^T out of the buffer)
  uint64_t kv_full, qdo_full[kStagesA], qdo_empty[kStagesA], st_full[2], ps_full[2];
  uint64_t dq_full[2], dq_free[2], mm_done;
  uint64_t drain;
  uint32_t tmem_base;
  Sync sync;
};
static_assert(sizeof(BarsF) <= 512, "barrier block fits its shared-memory slot");


// kBias: linear positional bias; kTab: explicit bias tensor (entries added
// to the exponent argument in registers, loaded a step ahead), as in the
// dK/dV kernel.
template <bool kBias, bool kTab>
__global__ void __launch_bounds__(kThreadsF, 1)
    bwd_fused_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                        const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_dq, const BwdTcArgs a) {
  constexpr int D = kDF;
  using L = LayoutF;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  BarsF *b = reinterpret_cast<BarsF *>(smem + L::kBar);
  const BwdParams &p = a.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // grid and row range as the dK/dV kernel's
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
  const int j_last = (j0 + kKeysA < g.nk ? j0 + kKeysA : g.nk) - 1;
  const int m_begin = row_begin(g.mask, j0, g.nq, g.nk) / kRowsA;
  const int m_end = (row_end(g.mask, g.window, j_last, g.nq, g.nk) + kRowsA - 1) / kRowsA;
  const int n_m = m_end > m_begin ? m_end - m_begin : 0;
  const int n_it = n_m * a.group;
  // Unbiased scores: warp 2 certifies the Q / dO tiles through ps_full
  // (measured 1.5% faster on training; with a bias the math is the longer
  // leg and ps_full would then wait for tiles two steps ahead, 5% slower).
  constexpr bool kWatch = !kBias && !kTab;

  if (threadIdx.x == 0) {
    mbar_init(&b->kv_full, 1);
    for (int s = 0; s < kStagesA; s++) {
      mbar_init(&b->qdo_full[s], 1);
      mbar_init(&b->qdo_empty[s], 1);
    }
    for (int s = 0; s < 2; s++) {
      mbar_init(&b->st_full[s], 1);
      mbar_init(&b->ps_full[s], kWatch ? 256 + 1 : 256);  // math warps (+ the tile watcher)
      mbar_init(&b->dq_full[s], 1);
      mbar_init(&b->dq_free[s], 128);
    }
    mbar_init(&b->mm_done, 1);
    mbar_init(&b->drain, 1);
    b->sync.limit_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    b->sync.abort = 0;
    b->sync.filled_one = b->sync.filled_a = b->sync.filled_b = b->sync.mma_issued = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&b->tmem_base, kTmemColsF);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = b->tmem_base;
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;

  const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV);
  const uint32_t sQ = smem_u32(smem + L::kQ), sDO = smem_u32(smem + L::kDO);
  const uint32_t sDS = smem_u32(smem + L::kDS);
  float *sRow = reinterpret_cast<float *>(smem + L::kRow);

  auto it_head = [&](int it) { return hk * a.group + (kTab ? it % a.group : it / n_m); };
  auto it_row0 = [&](int it) { return (m_begin + (kTab ? it / a.group : it % n_m)) * kRowsA; };

  if (warp < 4) {
    reg_dealloc<kRegCtl>();
    if (warp == 0 && lane == 0 && n_it > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      int filled = 0;  // Q / dO ring fills (stage = fill % kStagesA)
      mbar_arrive_expect_tx(&b->kv_full, 2 * L::kKV);
      for (int c = 0; c < L::kChunks; c++) {
        tma_load_3d(smem + L::kK + c * kChunkKV, &tm_k, &b->kv_full, c * 64, hk, g.k0 + j0);
        tma_load_3d(smem + L::kV + c * kChunkKV, &tm_v, &b->kv_full, c * 64, hk, g.k0 + j0);
      }
      for (int it = 0; it < n_it; it++) {
        const int st = it % kStagesA, u = it / kStagesA;
        const int h = it_head(it), tok = g.q0 + it_row0(it);
        if (it >= kStagesA && !wait_bar(&b->sync, &b->qdo_empty[st], (u - 1) & 1, p.err)) break;
        mbar_arrive_expect_tx(&b->qdo_full[st], 2 * L::kQT);
        filled++;
        for (int c = 0; c < L::kChunks; c++) {
          tma_load_3d(smem + L::kQ + st * L::kQT + c * kChunkQ, &tm_q, &b->qdo_full[st], c * 64, h, tok);
          tma_load_3d(smem + L::kDO + st * L::kQT + c * kChunkQ, &tm_do, &b->qdo_full[st], c * 64, h,
                      tok);
        }
      }
      b->sync.filled_one = 1;
      b->sync.filled_a = filled;
    } else if (kWatch && warp == 2 && lane == 0 && n_it > 0) {
      // Tile watcher: one more arrival on ps_full of step i once step
      // i + 2's Q / dO tiles have landed (and step i - 2's phase of the same
      // barrier has completed, so the arrival counts toward step i), so the
      // MMA thread, which issues step i + 2's S^T right after that barrier,
      // tests no TMA barrier: each test stalls it long enough for the
      // tensor pipe's short queue to drain.
      bool ok = true;
      for (int it = 0; ok && it < n_it; it++) {
        if (it + 2 < n_it)
          ok = wait_bar(&b->sync, &b->qdo_full[(it + 2) % kStagesA], ((it + 2) / kStagesA) & 1, p.err);
        if (ok && it >= 2) ok = wait_bar(&b->sync, &b->ps_full[it & 1], ((it - 2) >> 1) & 1, p.err);
        if (ok) mbar_arrive(&b->ps_full[it & 1]);
      }
    } else if (warp == 1 && lane == 0 && n_it > 0) {
      b->sync.mma_issued = 1;
      constexpr uint32_t idesc_s = idesc_f16_f32(128, kRowsA, 0, 0);
      constexpr uint32_t idesc_g = idesc_f16_f32(128, D, 0, 1);
      constexpr uint32_t idesc_q = idesc_f16_f32(D, kRowsA, 1, 1);
      const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024), dV0 = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dQk = smem_desc_sw128(sQ, 16, 1024), dDOk = smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dQm = smem_desc_sw128(sQ, kChunkQ, 1024);
      const uint64_t dDOm = smem_desc_sw128(sDO, kChunkQ, 1024);
      // K^T as an MN-major operand: d runs along the 128-byte swizzle rows,
      // the next 64 d values one chunk further, keys 8 rows per 1024 bytes
      const uint64_t dKm = smem_desc_sw128(sK, kChunkKV, 1024);
      // dS^T [128 keys][64 rows]: one 128-byte row per key (N = 64 fits one
      // swizzle row, so the leading offset is not used; kept small)
      const uint64_t dDSm = smem_desc_sw128(sDS, 16, 1024);
      auto issue_st = [&](uint64_t da, uint64_t db, uint32_t col) {
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
          const uint64_t oa = (uint64_t)((((kk >> 2) * kChunkKV) + (kk & 3) * 32) >> 4);
          const uint64_t ob = (uint64_t)((((kk >> 2) * kChunkQ) + (kk & 3) * 32) >> 4);
          mma_bf16_ss(tmem + col, da + oa, db + ob, idesc_s, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_grad = [&](uint32_t a_col, uint64_t db, uint32_t col, bool acc) {
#pragma unroll
        for (int kk = 0; kk < kRowsA / 16; kk++)
          mma_bf16_ts(tmem + col, tmem + a_col + 32 * (kk >> 1) + 8 * (kk & 1),
                      db + (uint64_t)((kk * 16 * 128) >> 4), idesc_g, (acc || kk > 0) ? 1u : 0u);
      };
      // dQ^T [d x 64 rows] = K^T [d x 128 keys] dS^T [128 keys x 64 rows]
      auto issue_dq = [&](uint32_t col) {
#pragma unroll
        for (int kk = 0; kk < kKeysA / 16; kk++) {
          const uint64_t o = (uint64_t)((kk * 16 * 128) >> 4);
          mma_bf16_ss(tmem + col, dKm + o, dDSm + o, idesc_q, kk > 0 ? 1u : 0u);
        }
      };
      auto qoff = [&](int s1) { return (uint64_t)((s1 * L::kQT) >> 4); };
      bool ok = wait_bar(&b->sync, &b->kv_full, 0, p.err) &&
                wait_bar(&b->sync, &b->qdo_full[0], 0, p.err);
      if (ok) {
        tc_fence_after();
        issue_st(dK0, dQk, kColS);
        issue_st(dV0, dDOk, kColDP);
        mma_commit(&b->st_full[0]);
      }
      if (ok && n_it > 1) {
        ok = wait_bar(&b->sync, &b->qdo_full[1], 0, p.err);
        if (ok) {
          tc_fence_after();
          issue_st(dK0, dQk + qoff(1), kColS + kRowsA);
          issue_st(dV0, dDOk + qoff(1), kColDP + kRowsA);
          mma_commit(&b->st_full[1]);
        }
      }
      // tb: the step's TMEM buffer (two), qs: its Q / dO stage (kStagesA)
      for (int it = 0; ok && it < n_it; it++) {
        const int tb = it & 1, qs = it % kStagesA;
        if (!wait_bar(&b->sync, &b->ps_full[tb], (it >> 1) & 1, p.err)) break;
        tc_fence_after();
        issue_dq(kColDP + tb * kRowsA);
        mma_commit(&b->dq_full[tb]);
        issue_grad(kColS + tb * kRowsA, dDOm + qoff(qs), kColDV, it > 0);
        issue_grad(kColS + tb * kRowsA + 16, dQm + qoff(qs), kColDK, it > 0);
        if (it + 1 == n_it) mma_commit(&b->mm_done);
        if (it + kStagesA < n_it) mma_commit(&b->qdo_empty[qs]);  // a later step refills it
        if (it + 2 < n_it) {  // kWatch: step it + 2's Q / dO landed, certified by ps_full
          const int q2 = (it + 2) % kStagesA, u2 = (it + 2) / kStagesA;
          if (!kWatch && !wait_bar(&b->sync, &b->qdo_full[q2], u2 & 1, p.err)) break;
          tc_fence_after();
          issue_st(dK0, dQk + qoff(q2), kColS + tb * kRowsA);
          if (!wait_bar(&b->sync, &b->dq_free[tb], (it >> 1) & 1, p.err)) break;
          tc_fence_after();
          issue_st(dV0, dDOk + qoff(q2), kColDP + tb * kRowsA);
          mma_commit(&b->st_full[tb]);
        }
      }
    }
  } else if (warp < 12) {
    reg_alloc<kRegMath>();
    const int wq = warp & 3;
    const int half = (warp - 4) >> 2;  // query rows [32 half, 32 half + 32) of each step
    const int r = wq * 32 + lane;      // key lane
    const int tid = threadIdx.x - 128;  // 0 .. 255; threads below 128 fetch row terms
    const int j = j0 + r;
    const int rb = key_row_begin(g.mask, j, g.nq, g.nk);
    const int re = key_row_end(g.mask, g.window, j, g.nq, g.nk);
    const bool tile_in = j0 + kKeysA <= g.nk;
    const int rb_last = key_row_begin(g.mask, j0 + kKeysA - 1, g.nq, g.nk);
    const int re_first = key_row_end(g.mask, g.window, j0, g.nq, g.nk);
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    // this key's 128-byte row of the dS^T copy; 16-byte chunk c of it lands
    // at chunk c ^ (key mod 8), the 128-byte swizzle the descriptor expects
    const uint32_t ds_row = sDS + (uint32_t)r * 128u;
    const CopyScales cs = copy_scales(p);
    const float c2 = cs.c2;
    bool ok = true;
    auto row_value = [&](int it) {
      const int c = tid & (kRowsA - 1);
      const int i = it_row0(it) + c;
      const size_t at = (size_t)it_head(it) * p.total_q + g.q0 + i;
      if (tid < kRowsA) return i < g.nq ? -p.lse2[at] : -INFINITY;
      return i < g.nq ? -p.delta[at] * cs.dsc : 0.f;
    };
    const bool fetcher = tid < 2 * kRowsA;
    float next_val = (n_it > 0 && fetcher) ? row_value(0) : 0.f;
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
    auto step = [&](int it, float (&bcur)[kTab ? 32 : 1], float (&bnext)[kTab ? 32 : 1]) {
      const int st = it & 1;
      const int i0 = it_row0(it);
      if (fetcher) sRow[st * 2 * kRowsA + tid] = next_val;
      math_group_sync();  // every math thread reaches it once per step, even after an abort
      if (fetcher && it + 1 < n_it) next_val = row_value(it + 1);
      const float *nlse2 = sRow + st * 2 * kRowsA;
      const float *nd = nlse2 + kRowsA;
      if constexpr (kTab) {
        if (it + 1 < n_it) load_bias(it + 1, bnext);
      }
      if (ok)
        ok = wait_bar(&b->sync, &b->st_full[st], (it >> 1) & 1, p.err);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) return;
      tc_fence_after();
      const bool step_full = tile_in && rb_last <= i0 && re_first >= i0 + kRowsA;
      const int c_lo = rb - i0, span = re > rb ? re - rb : 0;
      const uint64_t c2x2 = f2(c2, c2);
      const float slope2 = kBias ? __ldg(p.slopes + it_head(it)) * kLog2e : 0.f;
      const float bdist0 = (float)(j - i0 - causal_offset(g.mask, g.nq, g.nk));
      uint32_t pp[16], dd[16];
      uint32_t sv[32], dv[32];
      tmem_ld32(t_lane + kColS + st * kRowsA + half * 32, sv);
      tmem_ld32(t_lane + kColDP + st * kRowsA + half * 32, dv);
      tmem_wait_ld();
      auto body = [&](auto masked) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int c0 = half * 32 + e;
          float2 nl = *reinterpret_cast<const float2 *>(nlse2 + c0);
          const float2 ndd = *reinterpret_cast<const float2 *>(nd + c0);
          if constexpr (kBias) {
            nl.x += pos_bias2(slope2, bdist0, c0);
            nl.y += pos_bias2(slope2, bdist0, c0 + 1);
          }
          if constexpr (kTab) {
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
      // the dS^T copy for dQ^T: the previous step's dQ^T product must have
      // read it (complete long before, in practice)
      if (it > 0) {
        bool w = wait_bar(&b->sync, &b->dq_full[(it - 1) & 1], ((it - 1) >> 1) & 1, p.err);
        w = __all_sync(0xffffffffu, w);
        if (!w) {
          ok = false;
          return;
        }
      }
#pragma unroll
      for (int c = 0; c < 4; c++) {
        const uint32_t chunk = (uint32_t)((half * 4 + c) ^ (r & 7));
        st_shared_v4(ds_row + chunk * 16u, dd[4 * c], dd[4 * c + 1], dd[4 * c + 2], dd[4 * c + 3]);
      }
      fence_proxy_async_smem();  // generic-proxy writes visible to the tensor core
      // P^T, then dS^T, over this warp's 32 S^T columns: the A operands of
      // dV and dK, straight from tensor memory
      tmem_st16(t_lane + kColS + st * kRowsA + half * 32, pp);
      tmem_st16(t_lane + kColS + st * kRowsA + half * 32 + 16, dd);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&b->ps_full[st]);
    };
    float b0[kTab ? 32 : 1], b1[kTab ? 32 : 1];
    if constexpr (kTab) {
      if (n_it > 0) load_bias(0, b0);
      for (int it = 0; it < n_it; it += 2) {
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
    const int jt = g.k0 + (j < g.nk ? j : 0);
    __nv_bfloat16 *dkp = reinterpret_cast<__nv_bfloat16 *>(p.dk) + toff(p.sdk, jt, hk) + half * (D / 2);
    __nv_bfloat16 *dvp = reinterpret_cast<__nv_bfloat16 *>(p.dv) + toff(p.sdv, jt, hk) + half * (D / 2);
#pragma unroll
    for (int c = 0; c < D / 64; c++) {
      uint32_t kv32[32], vv32[32];
      if (have) {
        tmem_ld32(t_lane + kColDK + half * (D / 2) + c * 32, kv32);
        tmem_ld32(t_lane + kColDV + half * (D / 2) + c * 32, vv32);
        tmem_wait_ld();
      }
      if (j < g.nk) {
#pragma unroll
        for (int e = 0; e < 32; e += 8) {
          uint4 wk, wv;
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
  } else {
    reg_dealloc<kRegOut>();
    // dQ readout: thread = head-dim index (TMEM lane), 64 rows per step.
    // Each warp reduces its 32 features into the fp32 accumulator by TMA:
    // 32 rows at a time (two [16 rows x 32 fp32] shared tiles, row c of a
    // tile at 128 c bytes, one reduce-add each) once the tiles' previous
    // reduce-adds have read them; rows past the sequence add 0 (a 16-row
    // group wholly past it is skipped).  Only the warp itself syncs, so an
    // early exit cannot strand another warp.
    const int wq = warp & 3;
    const uint32_t t_lane = tmem + ((uint32_t)(wq * 32) << 16);
    float *sdq = reinterpret_cast<float *>(smem + L::kDQ + wq * L::kDQWarp);
    bool ok = true;
    for (int it = 0; it < n_it; it++) {
      const int tb = it & 1;
      if (ok) ok = wait_bar(&b->sync, &b->dq_full[tb], (it >> 1) & 1, p.err);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int i0 = it_row0(it);
      const int rows = g.nq - i0 < kRowsA ? g.nq - i0 : kRowsA;
      const int head = it_head(it);
#pragma unroll
      for (int hf = 0; hf < 2; hf++) {  // rows [32 hf, 32 hf + 32) of the step
        uint32_t v[32];
        tmem_ld32(t_lane + kColDP + tb * kRowsA + 32 * hf, v);
        tmem_wait_ld();
        if (hf == 1) {  // the step's dQ^T is out of tensor memory
          tc_fence_before();
          mbar_arrive(&b->dq_free[tb]);
        }
        if (32 * hf >= rows) continue;  // warp-uniform
        if (lane == 0) bulk_wait_read();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 32; c++)
          sdq[c * 32 + lane] = 32 * hf + c < rows ? __uint_as_float(v[c]) : 0.f;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, sdq, wq * 32, head, g.q0 + i0 + 32 * hf);
          if (32 * hf + 16 < rows)
            tma_reduce_add_3d(&tm_dq, sdq + 16 * 32, wq * 32, head, g.q0 + i0 + 32 * hf + 16);
          bulk_commit();
        }
      }
    }
    // the shared tiles stay allocated until the last reduce-adds have read them
    if (lane == 0) bulk_wait_read();
  }

  tc_fence_before();
  __syncthreads();
  // A block in which a wait gave up may still have copies and products in
  // flight: drain them before the tensor memory is freed.
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
    tmem_dealloc(tmem, kTmemColsF);
  }
}

// Zero the fp32 dQ accumulator (n4 float4 groups).
__global__ void zero_f32_kernel(float4 *p, size_t n4) {
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x)
    p[i] = z;
}

// dQ = accumulator x 2^-(s_v + s_do) x scale 2^-s_k, in bf16: eight
// elements per thread, every (token, query head) row of dq.
__global__ void dq_convert_kernel(const BwdParams p) {
  const size_t per_row = (size_t)p.d / 8;
  const size_t n = (size_t)p.total_q * p.hq * per_row;
  const CopyScales cs = copy_scales(p);
  const float f = cs.g * cs.gq;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t row = i / per_row;
    const int e = (int)(i - row * per_row) * 8;
    const int t = (int)(row / p.hq), h = (int)(row % p.hq);
    const float4 *src = reinterpret_cast<const float4 *>(p.dqacc + row * p.d + e);
    const float4 x = src[0], y = src[1];
    uint4 w;
    w.x = pack_bf16x2(x.x * f, x.y * f);
    w.y = pack_bf16x2(x.z * f, x.w * f);
    w.z = pack_bf16x2(y.x * f, y.y * f);
    w.w = pack_bf16x2(y.z * f, y.w * f);
    *reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(p.dq) + toff(p.sdq, t, h) + e) = w;
  }
}

template <bool kBias, bool kTab>
cudaError_t launch_fused_t(const BwdTcArgs &a, cudaStream_t st) {
  const BwdParams &p = a.p;
  const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap q64, do64, mk, mv, mdq;
  if (!make_map(&q64, p.q16, kDF, p.hq, p.total_q, 1, kRowsA, f16) ||
      !make_map(&do64, p.do16, kDF, p.hq, p.total_q, 1, kRowsA, f16) ||
      !make_map(&mk, p.k16, kDF, p.hkv, p.total_k, 1, kTileKeys, f16) ||
      !make_map(&mv, p.v16, kDF, p.hkv, p.total_k, 1, kTileKeys, f16) ||
      !make_map_f32(&mdq, p.dqacc, kDF, p.hq, p.total_q, 32, 16))
    return cudaErrorInvalidValue;
  static bool conf[64] = {false};
  cudaError_t e = set_smem(bwd_fused_tc_kernel<kBias, kTab>, LayoutF::kAlloc, conf);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)a.n_key_tiles * p.hkv * p.batch;
  if (grid >= (1LL << 31)) return cudaErrorInvalidValue;
  bwd_fused_tc_kernel<kBias, kTab><<<(unsigned)grid, kThreadsF, LayoutF::kAlloc, st>>>(q64, do64, mk, mv,
                                                                                        mdq, a);
  return cudaGetLastError();
}

}  // namespace

// The fused tensor-core backward after the preprocess (D and lse2 ready):
// zero the dQ accumulator, run the fused kernel, convert dQ.  head_dim 128.
cudaError_t launch_bwd_fused(const BwdParams &p, cudaStream_t st, char *desc, size_t desc_len) {
  BwdTcArgs a;
  a.p = p;
  a.group = p.hq / p.hkv;
  a.n_key_tiles = (p.max_k + kKeysA - 1) / kKeysA;
  a.n_row_tiles = 0;
  const long long ctas = (long long)a.n_key_tiles * p.hkv * p.batch;
  snprintf(desc, desc_len,
           "zero_rows+zero_rows+bwd_amax+bwd_pre+kv_to_f16%s+zero_f32+bwd_fused_tc_d%d%s+dq_convert "
           "ctas_fused=%lld",
           p.delta_ready ? "+fwd_tc2_delta" : "", p.d, p.btab ? "_btab" : "", ctas);
  if (p.d != kDF || !p.dqacc) return cudaErrorInvalidValue;
  const size_t n = (size_t)p.total_q * p.hq * p.d;
  if (n == 0) return cudaSuccess;
  const int sms = internal_sm_count();
  const size_t n4 = n / 4;
  size_t blocks = (n4 + 255) / 256;
  const size_t cap = (size_t)(sms > 0 ? sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  zero_f32_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<float4 *>(p.dqacc), n4);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (a.n_key_tiles > 0) {
    if (p.btab)
      e = launch_fused_t<false, true>(a, st);
    else if (p.slopes)
      e = launch_fused_t<true, false>(a, st);
    else
      e = launch_fused_t<false, false>(a, st);
    if (e != cudaSuccess) return e;
  }
  const size_t n8 = n / 8;
  blocks = (n8 + 255) / 256;
  if (blocks > cap) blocks = cap;
  dq_convert_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
