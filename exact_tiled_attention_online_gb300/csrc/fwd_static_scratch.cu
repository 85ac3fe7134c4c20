// fwd_static_scratch.cu -- attn_fwd_static_scratch: the forward for callers
// that cannot allocate device memory or pass a workspace (plug-ins inside a
// host runtime that owns a fixed memory plan and exposes no allocator, and
// serving loops where cudaMalloc is off limits once they run).  The split-KV
// decode's partial outputs live in one file-scope device array instead of a
// caller-provided workspace; the kernels are the ones attn_fwd launches.
#include <stdio.h>
#include <string.h>

#include "common.cuh"
#include "plan.h"

namespace attn {

cudaError_t launch_fwd_tc(const FwdParams &p, const TcPlan &plan, cudaStream_t st, char *desc,
                          size_t desc_len);
cudaError_t launch_combine(const FwdParams &p, const TcPlan &plan, cudaStream_t st);
int *internal_error_flag();
attn_status internal_check_sizes(int batch, int max_q, int max_k, int total_q, int total_k,
                                 int hq, int hkv, int d, int mask, int window, int dtype);
int internal_sm_count();
unsigned long long internal_wait_ns();
void internal_set_plan(const char *s);

// The scratch array: ATTN_STATIC_SCRATCH_BYTES on every device that loads the
// library.  Host code must not pass its name to a kernel (on the host it is a
// stand-in symbol, not a device address); the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[ATTN_STATIC_SCRATCH_BYTES];

// Device address of the scratch array on the current device, looked up once
// per device (the first call on a device should be made outside stream
// capture).  NULL when the lookup fails.
static void *static_scratch_ptr() {
  static void *cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) return nullptr;
    cache[dev] = ptr;
  }
  return cache[dev];
}

}  // namespace attn

using namespace attn;

extern "C" attn_status attn_fwd_static_scratch(
    const void *q, const void *k, const void *v, void *o, float *lse, float *o_f32,
    const int32_t *cu_q, const int32_t *cu_k, int batch, int max_q, int max_k, int total_q,
    int total_k, int hq, int hkv, int d, float scale, attn_mask_kind mask, int window,
    const float *bias_slopes, attn_dtype dtype, void *stream) {
  attn_status st = internal_check_sizes(batch, max_q, max_k, total_q, total_k, hq, hkv, d, mask,
                                        window, dtype);
  if (st != ATTN_OK) return st;
  if (batch == 0 || total_q == 0 || max_q == 0 || total_k == 0) {
    // No query rows (a no-op), or no keys (every row empty; no split plan):
    // attn_fwd handles both without any scratch.
    return attn_fwd(q, k, v, o, lse, o_f32, cu_q, cu_k, batch, max_q, max_k, total_q, total_k,
                    hq, hkv, d, scale, mask, window, bias_slopes, dtype, nullptr, 0, stream);
  }
  TcPlan plan = choose_fwd_plan(batch, max_q, max_k, total_q, hq, hkv, d, window, dtype,
                                internal_sm_count());
  if (plan.kind != PLAN_TC_SPLIT) {
    // Nothing to keep in scratch: the workspace-free attn_fwd path.
    return attn_fwd(q, k, v, o, lse, o_f32, cu_q, cu_k, batch, max_q, max_k, total_q, total_k,
                    hq, hkv, d, scale, mask, window, bias_slopes, dtype, nullptr, 0, stream);
  }
  if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (!cu_q || !cu_k || !q || !o || !k || !v) return ATTN_ERR_INVALID_ARG;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if (mis & 15) return ATTN_ERR_INVALID_ARG;
  if ((long long)batch * plan.n_splits > 65535) return ATTN_ERR_UNSUPPORTED;
  const size_t need = fwd_split_workspace(plan, total_q, hq, d);
  if (need > (size_t)ATTN_STATIC_SCRATCH_BYTES) return ATTN_ERR_SCRATCH_LIMIT;
  char *scratch = static_cast<char *>(static_scratch_ptr());
  int *err = internal_error_flag();
  if (!scratch || !err) return ATTN_ERR_CUDA;

  FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.o_f32 = o_f32;
  p.cu_q = cu_q; p.cu_k = cu_k;
  p.batch = batch; p.max_q = max_q; p.max_k = max_k; p.total_q = total_q; p.total_k = total_k;
  p.hq = hq; p.hkv = hkv; p.d = d; p.scale = scale; p.scale_log2 = scale * kLog2e;
  p.mask = mask;
  p.window = window;
  p.slopes = bias_slopes;
  p.sq = {(long long)hq * d, d};  // contiguous layouts
  p.sk = {(long long)hkv * d, d};
  p.sv = {(long long)hkv * d, d};
  p.so = {(long long)hq * d, d};
  p.err = err;
  p.wait_ns = internal_wait_ns();
  // Same carving as the caller-provided workspace of attn_fwd: partial
  // outputs first, partial logsumexps after them.
  p.o_part = reinterpret_cast<float *>(scratch);
  p.lse_part = reinterpret_cast<float *>(
      scratch + align_up256((size_t)plan.n_splits * total_q * hq * d * 4));
  p.n_splits = plan.n_splits;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  char desc[384];
  desc[0] = 0;
  cudaError_t ce = launch_fwd_tc(p, plan, cs, desc, sizeof(desc));
  if (ce == cudaSuccess) ce = launch_combine(p, plan, cs);
  char full[512];
  snprintf(full, sizeof(full), "%s [static scratch]%s%s", desc,
           ce == cudaSuccess ? "" : " [launch failed: ",
           ce == cudaSuccess ? "" : cudaGetErrorString(ce));
  if (ce != cudaSuccess) {
    const size_t n = strlen(full);
    snprintf(full + n, sizeof(full) - n, "]");
  }
  internal_set_plan(full);
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
