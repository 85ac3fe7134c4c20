// bwd_tc.cuh -- pieces shared by the tensor-core backward kernels: launch
// arguments, bounded waits with a block-wide abort flag, the factors that
// undo the fp16 copies' power-of-two scaling, and the dK/dV tile shape.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"
#include "sm100.cuh"

namespace attn {
namespace {
using namespace sm100;

constexpr int kRowsA = 64;   // query rows per step
constexpr int kKeysA = 128;  // keys per CTA
// Q / dO ring depth: a stage is refilled only once the gradient products of
// its step have completed, so the ring must cover that round trip (MMA
// completion, the refill's TMA latency) with the steps queued behind it.
constexpr int kStagesA = 4;

struct BwdTcArgs {
  BwdParams p;
  int group;
  int n_key_tiles;  // dkdv grid x
  int n_row_tiles;  // dq grid x
};

struct Sync {
  uint64_t limit_ns;  // bound of every wait of this call
  int abort;
  // for a drain after an early exit: single-tile fills (0 / 1), ring fills
  // the producer issued, and whether the MMA thread issued any product
  int filled_one, filled_a, filled_b, mma_issued;
};

__device__ __forceinline__ bool wait_bar(Sync *sy, uint64_t *bar, uint32_t parity, int *err) {
  if (mbar_test_wait(bar, parity)) return true;  // already complete: the cheap path
  if (*reinterpret_cast<volatile int *>(&sy->abort)) return false;
  if (mbar_wait(bar, parity, sy->limit_ns)) return true;
  *reinterpret_cast<volatile int *>(&sy->abort) = 1;
  raise_error(err, ATTN_ERR_DEVICE_TIMEOUT);
  return false;
}

__device__ __forceinline__ void math_group_sync() {
  asm volatile("bar.sync 1, 256;" ::: "memory");
}

// Factors that undo the power-of-two scaling of the fp16 copies (scale
// exponents s_q, s_k, s_v, s_do from f16_copy_exponent): with Q' = 2^s_q Q
// and so on, S' = 2^(s_q + s_k) S, dP' = 2^(s_v + s_do) dP, and the products
// give dS' = 2^(s_v + s_do) dS, dV' = 2^s_do dV, dK' = 2^(s_v + s_do + s_q)
// dK / scale, dQ' = 2^(s_v + s_do + s_k) dQ / scale.  Every factor is a
// power of two (times the scale), so undoing them is exact.
struct CopyScales {
  float c2;    // S' -> log2 logit: scale log2(e) 2^-(s_q + s_k)
  float dsc;   // D -> dP' units: 2^(s_v + s_do)
  float bias;  // bias-tensor entry -> S' units: 2^(s_q + s_k) / scale
  float g;     // 2^-(s_v + s_do), the first factor of dK and dQ
  float gk, gq, gv;  // then dK: scale 2^-s_q, dQ: scale 2^-s_k; dV: 2^-s_do
};

__device__ __forceinline__ CopyScales copy_scales(const BwdParams &p) {
  const int sq = f16_copy_exponent(p.amax[kAmaxQ]), sk = f16_copy_exponent(p.amax[kAmaxK]);
  const int sv = f16_copy_exponent(p.amax[kAmaxV]), sd = f16_copy_exponent(p.amax[kAmaxDO]);
  CopyScales c;
  c.c2 = p.scale_log2 * exp2_int(-sq) * exp2_int(-sk);
  c.dsc = exp2_int(sv + sd);
  c.bias = (1.f / p.scale) * exp2_int(sq) * exp2_int(sk);
  c.g = exp2_int(-(sv + sd));
  c.gk = p.scale * exp2_int(-sq);
  c.gq = p.scale * exp2_int(-sk);
  c.gv = exp2_int(-sd);
  return c;
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes, bool *configured) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!configured[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace attn
