// plan.h -- host-side choice of the forward kernel plan.  Deterministic in
// its arguments and the device's SM count, so the workspace size query and
// the call agree.
#pragma once

#include <stddef.h>

#include "../../include/attn.h"

namespace attn {

enum PlanKind { PLAN_SIMT = 0, PLAN_TC = 1, PLAN_TC_SPLIT = 2 };

#ifndef ATTN_TC_FWD
#define ATTN_TC_FWD 0
#endif
constexpr bool kTensorCorePath = ATTN_TC_FWD != 0;

constexpr int kTileRows = 128;  // MMA rows per tile (tcgen05 M)
constexpr int kTileKeys = 128;  // keys per key tile (tcgen05 N of Q K^T)

struct TcPlan {
  int kind;
  int group;        // n_heads_q / n_heads_kv
  int pack;         // 1: a tile holds the `group` query heads of one KV head
  int tile_tokens;  // query tokens per tile: kTileRows, or kTileRows / group
  int n_m_tiles;    // tiles along the query axis per (sequence, head)
  int n_splits;     // key splits (1 unless kind == PLAN_TC_SPLIT)
};

// Tensor-core plan for bf16; the CUDA-core kernel for fp32.  When every query
// row of a KV-head group fits one tile (decode: a few queries against a long
// cache), the group's heads share the tile so each K/V tile is read once for
// all of them, and the keys are split across CTAs until the grid covers the
// GPU several times over; the splits are merged by a combine kernel.
inline TcPlan choose_fwd_plan(int batch, int max_q, int max_k, int total_q, int hq, int hkv,
                              int d, int window, attn_dtype dtype, int sms) {
  (void)total_q;
  (void)d;
  TcPlan p{};
  p.group = hq / hkv;
  p.n_splits = 1;
  if (dtype != ATTN_DTYPE_BF16 || !kTensorCorePath) {
    p.kind = PLAN_SIMT;
    return p;
  }
  p.kind = PLAN_TC;
  const bool can_pack = p.group > 1 && p.group <= 16 && (kTileRows % p.group) == 0;
  if (can_pack && (long long)max_q * p.group <= kTileRows) {
    p.pack = 1;
    p.tile_tokens = kTileRows / p.group;
  } else {
    p.pack = 0;
    p.tile_tokens = kTileRows;
  }
  p.n_m_tiles = (max_q + p.tile_tokens - 1) / p.tile_tokens;
  const long long ctas = (long long)batch * (p.pack ? hkv : hq) * p.n_m_tiles;
  if (ctas <= 0) return p;  // no query rows (an empty batch is a no-op): nothing to split
  int kv_tiles = (max_k + kTileKeys - 1) / kTileKeys;
  if (window > 0) {  // a bounded window: a tile's keys span window + tile_tokens - 1
    const long long span = (long long)window + p.tile_tokens - 1;
    const long long w_tiles = (span + kTileKeys - 1) / kTileKeys + 1;
    if (w_tiles < kv_tiles) kv_tiles = (int)w_tiles;
  }
  // Split the keys across CTAs for decode (packed heads), or when even the
  // prefill kernel's 256-row CTAs would leave most SMs idle.
  const long long prefill_ctas = (long long)batch * hq * ((max_q + 2 * kTileRows - 1) / (2 * kTileRows));
  const bool starved = p.pack ? ctas < 4LL * sms : 4 * prefill_ctas < sms;
  if (sms > 0 && starved && kv_tiles >= 8) {
    long long want = (8LL * sms + ctas - 1) / ctas;
    long long cap = kv_tiles / 4;  // at least four key tiles per split
    int n = (int)(want < cap ? want : cap);
    if (n > 64) n = 64;
    if (n >= 2) {
      p.kind = PLAN_TC_SPLIT;
      p.n_splits = n;
    }
  }
  return p;
}

inline size_t align_up256(size_t x) { return (x + 255) & ~(size_t)255; }

// Split-KV scratch: one fp32 partial output row and one partial logsumexp per
// (split, token, head).
inline size_t fwd_split_workspace(const TcPlan &p, int total_q, int hq, int d) {
  return align_up256((size_t)p.n_splits * total_q * hq * d * 4) +
         align_up256((size_t)p.n_splits * total_q * hq * 4);
}

}  // namespace attn
