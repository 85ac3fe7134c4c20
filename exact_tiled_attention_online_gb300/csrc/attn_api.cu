// attn_api.cu -- the C ABI declared in include/attn.h: argument validation,
// plan selection, workspace carving and kernel launches.  Nothing here
// allocates memory; every buffer is the caller's.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "plan.h"

namespace attn {

cudaError_t launch_fwd_simt(const FwdParams &p, attn_dtype dtype, cudaStream_t st);
cudaError_t launch_bwd_simt(const BwdParams &p, attn_dtype dtype, cudaStream_t st);
cudaError_t launch_bwd_pre(const BwdParams &p, attn_dtype dtype, cudaStream_t st);
cudaError_t launch_kv_to_f16(const BwdParams &p, cudaStream_t st);
cudaError_t launch_bwd_amax(const BwdParams &p, cudaStream_t st);
cudaError_t launch_fwd_tc2_delta(const FwdParams &p, cudaStream_t st);
cudaError_t launch_bwd_tc(const BwdParams &p, cudaStream_t st, char *desc, size_t desc_len);
cudaError_t launch_bwd_fused(const BwdParams &p, cudaStream_t st, char *desc, size_t desc_len);
cudaError_t launch_fwd_tc(const FwdParams &p, const TcPlan &plan, cudaStream_t st,
                          char *desc, size_t desc_len);
cudaError_t launch_combine(const FwdParams &p, const TcPlan &plan, cudaStream_t st);
cudaError_t launch_fwd_tc2(const FwdParams &p, cudaStream_t st, char *desc, size_t desc_len);
cudaError_t launch_zero_rows(void *base, int T, int H, int d, Strides s, int elem,
                             cudaStream_t st);
cudaError_t launch_mask_probe(const int32_t *cu_q, const int32_t *cu_k, int batch, int max_q,
                              int max_k, int total_q, int total_k, int mask, int window,
                              int tile_rows, uint8_t *out, int *err, cudaStream_t st);

// The per-device error flag.  Device code reaches it through a pointer kernel
// argument; the host looks its address up once per device.
__device__ int g_device_error;

static int *device_error_ptr() {
  static int *cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int *>(ptr);
  }
  return cache[dev];
}

static thread_local char t_plan[512] = "none";

// Bound of every device wait, in ns (0: the kernels' 2 s default); set by
// attn_set_wait_limit_ns, read by every call.
static std::atomic<unsigned long long> g_wait_ns{0};

// Nonzero: the bf16 backward keeps to the two-kernel form, whose dQ is
// reproducible bit for bit (set by attn_set_deterministic).
static std::atomic<int> g_deterministic{0};

static void set_plan(const char *s) {
  snprintf(t_plan, sizeof(t_plan), "%s", s);
}

// ---------------------------------------------------------------------------
// Validation shared by every entry point.
// ---------------------------------------------------------------------------
static attn_status check_sizes(int batch, int max_q, int max_k, int total_q, int total_k,
                               int hq, int hkv, int d, int mask, int window, int dtype) {
  if (batch < 0 || max_q < 0 || max_k < 0 || total_q < 0 || total_k < 0)
    return ATTN_ERR_INVALID_ARG;
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (hq > 65535 || hkv > 65535 || batch > 65535) return ATTN_ERR_UNSUPPORTED;
  if (mask < ATTN_MASK_NONE || mask > ATTN_CAUSAL_BOTTOM_RIGHT) return ATTN_ERR_INVALID_ARG;
  if (window < 0 || (window > 0 && mask == ATTN_MASK_NONE)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_FP32) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (max_q > total_q || max_k > total_k) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// The layout of one tensor: the caller's strides, or contiguous THD.  false
// for a stride that is not positive or not a multiple of 16 bytes.
static bool pick_strides(const int64_t *given, int heads, int d, int elem, Strides *out) {
  if (!given) {
    out->ts = (long long)heads * d;
    out->hs = d;
    return true;
  }
  out->ts = given[0];
  out->hs = given[1];
  return out->ts > 0 && out->hs > 0 && (out->ts * elem) % 16 == 0 && (out->hs * elem) % 16 == 0;
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Backward workspace: D and lse2 [hq, total_q] fp32; for bf16 also scaled
// fp16 copies of q, dout ([total_q, hq, d]) and k, v ([total_k, hkv, d]) and
// the four tensors' largest magnitudes (256 bytes).
struct BwdLayout {
  size_t delta, lse2, q16, do16, k16, v16, amax, dqacc, total;
};
static BwdLayout bwd_layout(int total_q, int total_k, int hq, int hkv, int d, int dtype) {
  BwdLayout l{};
  const size_t rows = align256((size_t)hq * total_q * 4);
  l.delta = 0;
  l.lse2 = rows;
  size_t off = 2 * rows;
  if (dtype == ATTN_DTYPE_BF16) {
    const size_t qb = align256((size_t)total_q * hq * d * 2);
    const size_t kb = align256((size_t)total_k * hkv * d * 2);
    l.q16 = off;
    l.do16 = off + qb;
    l.k16 = off + 2 * qb;
    l.v16 = off + 2 * qb + kb;
    off += 2 * qb + 2 * kb;
    l.amax = off;
    off += 256;
    if (d == 128) {  // the fused backward's fp32 dQ accumulator
      l.dqacc = off;
      off += align256((size_t)total_q * hq * d * 4);
    }
  }
  l.total = off;
  return l;
}

// Internal helpers for the other entry-point file of the library.
int *internal_error_flag() { return device_error_ptr(); }
attn_status internal_check_sizes(int batch, int max_q, int max_k, int total_q, int total_k,
                                 int hq, int hkv, int d, int mask, int window, int dtype) {
  return check_sizes(batch, max_q, max_k, total_q, total_k, hq, hkv, d, mask, window, dtype);
}
int internal_sm_count() { return sm_count(); }
unsigned long long internal_wait_ns() { return g_wait_ns.load(std::memory_order_relaxed); }
void internal_set_plan(const char *s) { set_plan(s); }

}  // namespace attn

using namespace attn;

extern "C" {

int attn_version(void) { return 120; }

const char *attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported head_dim, dtype or size";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "a bounded device wait expired";
    case ATTN_ERR_DEVICE_BOUNDS: return "cu_seqlens inconsistent with the sizes passed";
    case ATTN_ERR_SCRATCH_LIMIT: return "problem needs more than the library's static scratch";
    case ATTN_ERR_DEVICE_RANGE: return "a backward input holds an infinity or NaN";
  }
  return "unknown status";
}

const char *attn_last_plan(void) { return t_plan; }

void attn_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns, std::memory_order_relaxed); }

void attn_set_deterministic(int on) { g_deterministic.store(on ? 1 : 0, std::memory_order_relaxed); }

int attn_get_deterministic(void) { return g_deterministic.load(std::memory_order_relaxed); }

size_t attn_fwd_workspace_size(int batch, int max_q, int max_k, int total_q, int hq, int hkv,
                               int d, int window, attn_dtype dtype) {
  // the window's value is checked here; its pairing with a causal kind is
  // the forward's check
  if (window < 0 || check_sizes(batch, max_q, max_k, total_q, max_k, hq, hkv, d,
                                ATTN_MASK_NONE, 0, dtype) != ATTN_OK)
    return (size_t)-1;
  TcPlan plan =
      choose_fwd_plan(batch, max_q, max_k, total_q, hq, hkv, d, window, dtype, sm_count());
  if (plan.kind != PLAN_TC_SPLIT) return 0;
  return fwd_split_workspace(plan, total_q, hq, d);
}

attn_status attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                     float *o_f32, const int32_t *cu_q, const int32_t *cu_k, int batch, int max_q, int max_k,
                     int total_q, int total_k, int hq, int hkv, int d, float scale,
                     attn_mask_kind mask, int window, const float *bias_slopes,
                     attn_dtype dtype, void *workspace, size_t workspace_bytes, void *stream) {
  return attn_fwd_ex(nullptr, nullptr, q, k, v, o, lse, o_f32, cu_q, cu_k, batch, max_q, max_k, total_q,
                     total_k, hq, hkv, d, scale, mask, window, bias_slopes, dtype, workspace,
                     workspace_bytes, stream);
}

// The explicit bias tensor's fields, or false for a malformed one.
static bool pick_btab(const attn_bias_tensor *b, const float **data, long long *ss, long long *hs,
                      long long *rs) {
  *data = nullptr;
  *ss = *hs = *rs = 0;
  if (!b) return true;
  if (!b->data || b->seq_stride < 0 || b->head_stride < 0 || b->row_stride < 0) return false;
  if (reinterpret_cast<uintptr_t>(b->data) & 3) return false;
  *data = b->data;
  *ss = b->seq_stride;
  *hs = b->head_stride;
  *rs = b->row_stride;
  return true;
}

attn_status attn_fwd_ex(const attn_strides *strides, const attn_bias_tensor *bias, const void *q, const void *k,
                        const void *v, void *o, float *lse, float *o_f32, const int32_t *cu_q,
                        const int32_t *cu_k, int batch, int max_q, int max_k, int total_q,
                        int total_k, int hq, int hkv, int d, float scale, attn_mask_kind mask,
                        int window, const float *bias_slopes, attn_dtype dtype,
                        void *workspace, size_t workspace_bytes, void *stream) {
  attn_status st =
      check_sizes(batch, max_q, max_k, total_q, total_k, hq, hkv, d, mask, window, dtype);
  if (st != ATTN_OK) return st;
  if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (batch > 0 && (!cu_q || !cu_k)) return ATTN_ERR_INVALID_ARG;
  if (total_q > 0 && (!q || !o)) return ATTN_ERR_INVALID_ARG;
  if (total_k > 0 && (!k || !v)) return ATTN_ERR_INVALID_ARG;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  FwdParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse; p.o_f32 = o_f32;
  p.cu_q = cu_q; p.cu_k = cu_k;
  p.batch = batch; p.max_q = max_q; p.max_k = max_k; p.total_q = total_q; p.total_k = total_k;
  p.hq = hq; p.hkv = hkv; p.d = d; p.scale = scale; p.scale_log2 = scale * kLog2e;
  p.mask = mask;
  p.window = window;
  p.slopes = bias_slopes;
  if (!pick_btab(bias, &p.btab, &p.bss, &p.bhs, &p.brs)) return ATTN_ERR_INVALID_ARG;
  const int elem = dtype == ATTN_DTYPE_FP32 ? 4 : 2;
  if (!pick_strides(strides ? strides->q : nullptr, hq, d, elem, &p.sq) ||
      !pick_strides(strides ? strides->k : nullptr, hkv, d, elem, &p.sk) ||
      !pick_strides(strides ? strides->v : nullptr, hkv, d, elem, &p.sv) ||
      !pick_strides(strides ? strides->o : nullptr, hq, d, elem, &p.so))
    return ATTN_ERR_INVALID_ARG;
  p.err = device_error_ptr();
  if (!p.err) return ATTN_ERR_CUDA;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  if (batch == 0 || total_q == 0 || max_q == 0) {
    set_plan("empty");
    return ATTN_OK;
  }
  TcPlan plan =
      choose_fwd_plan(batch, max_q, max_k, total_q, hq, hkv, d, window, dtype, sm_count());
  if (p.btab) {
    // bf16 with a positive scale and no slopes: the prefill kernel's bias-tensor
    // instance (the bias rides on the raw scores); otherwise the CUDA-core kernel
    const bool tab_tc = plan.kind != PLAN_SIMT && scale > 0.f && !bias_slopes;
    plan.kind = tab_tc ? PLAN_TC : PLAN_SIMT;
    plan.pack = false;
    plan.n_splits = 1;
  }
  if (plan.kind != PLAN_SIMT) {
    // TMA needs 16-byte aligned tensors; with no keys at all every row is
    // empty and the CUDA-core kernel writes the zeros and -inf directly.
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
    if (mis & 15) return ATTN_ERR_INVALID_ARG;
    if (total_k == 0) plan.kind = PLAN_SIMT;
    const long long gz = (long long)batch * plan.n_splits;
    if (gz > 65535) return ATTN_ERR_UNSUPPORTED;
  }
  char desc[384];
  desc[0] = 0;  // a launcher that fails early may leave it unwritten
  cudaError_t ce;
  if (plan.kind == PLAN_SIMT) {
    ce = launch_fwd_simt(p, dtype, cs);
    snprintf(desc, sizeof(desc), "fwd_simt_%s_d%d%s grid=(%d,%d,%d)",
             dtype == ATTN_DTYPE_FP32 ? "fp32" : "bf16", d, p.btab ? "_btab" : "",
             (max_q + 3) / 4, hq, batch);
  } else {
    if (plan.kind == PLAN_TC_SPLIT) {
      size_t need = fwd_split_workspace(plan, total_q, hq, d);
      if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
      if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return ATTN_ERR_INVALID_ARG;
      p.o_part = static_cast<float *>(workspace);
      p.lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                             align256((size_t)plan.n_splits * total_q * hq * d * 4));
      p.n_splits = plan.n_splits;
    }
    if (plan.kind == PLAN_TC && !plan.pack)
      ce = launch_fwd_tc2(p, cs, desc, sizeof(desc));  // prefill: two query tiles per CTA
    else
      ce = launch_fwd_tc(p, plan, cs, desc, sizeof(desc));
    if (ce == cudaSuccess && plan.kind == PLAN_TC_SPLIT) ce = launch_combine(p, plan, cs);
  }
  if (ce != cudaSuccess) {  // keep the runtime's reason with the plan
    const size_t n = strlen(desc);
    snprintf(desc + n, sizeof(desc) - n, " [launch failed: %s]", cudaGetErrorString(ce));
  }
  set_plan(desc);
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_bwd_workspace_size(int batch, int max_q, int max_k, int total_q, int total_k,
                               int hq, int hkv, int d, attn_dtype dtype) {
  if (check_sizes(batch, max_q, max_k, total_q, total_k, hq, hkv, d, ATTN_MASK_NONE, 0, dtype) !=
      ATTN_OK)
    return (size_t)-1;
  return bwd_layout(total_q, total_k, hq, hkv, d, dtype).total;
}

attn_status attn_bwd(const void *q, const void *k, const void *v, const void *o,
                     const float *lse, const float *o_f32, const void *dout, void *dq, void *dk, void *dv,
                     const int32_t *cu_q, const int32_t *cu_k, int batch, int max_q, int max_k,
                     int total_q, int total_k, int hq, int hkv, int d, float scale,
                     attn_mask_kind mask, int window, const float *bias_slopes,
                     attn_dtype dtype, void *workspace, size_t workspace_bytes, void *stream) {
  return attn_bwd_ex(nullptr, nullptr, q, k, v, o, lse, o_f32, dout, dq, dk, dv, cu_q, cu_k, batch, max_q,
                     max_k, total_q, total_k, hq, hkv, d, scale, mask, window, bias_slopes, dtype,
                     workspace, workspace_bytes, stream);
}

attn_status attn_bwd_ex(const attn_strides *strides, const attn_bias_tensor *bias, const void *q, const void *k,
                        const void *v, const void *o, const float *lse, const float *o_f32,
                        const void *dout, void *dq, void *dk, void *dv, const int32_t *cu_q,
                        const int32_t *cu_k, int batch, int max_q, int max_k, int total_q,
                        int total_k, int hq, int hkv, int d, float scale, attn_mask_kind mask,
                        int window, const float *bias_slopes, attn_dtype dtype,
                        void *workspace, size_t workspace_bytes, void *stream) {
  attn_status st =
      check_sizes(batch, max_q, max_k, total_q, total_k, hq, hkv, d, mask, window, dtype);
  if (st != ATTN_OK) return st;
  if (!isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (batch > 0 && (!cu_q || !cu_k)) return ATTN_ERR_INVALID_ARG;
  if (total_q > 0 && (!q || !o || !lse || !dout || !dq)) return ATTN_ERR_INVALID_ARG;
  if (total_k > 0 && (!k || !v || !dk || !dv)) return ATTN_ERR_INVALID_ARG;
  {  // a malformed bias tensor is an argument error before the workspace is looked at
    const float *bd;
    long long b0, b1, b2;
    if (!pick_btab(bias, &bd, &b0, &b1, &b2)) return ATTN_ERR_INVALID_ARG;
  }
  size_t need = attn_bwd_workspace_size(batch, max_q, max_k, total_q, total_k, hq, hkv, d, dtype);
  if (need > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return ATTN_ERR_INVALID_ARG;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  BwdParams p{};
  p.q = q; p.k = k; p.v = v; p.o = o; p.dout = dout; p.lse = lse; p.o_f32 = o_f32;
  p.dq = dq; p.dk = dk; p.dv = dv;
  p.cu_q = cu_q; p.cu_k = cu_k;
  p.batch = batch; p.max_q = max_q; p.max_k = max_k; p.total_q = total_q; p.total_k = total_k;
  p.hq = hq; p.hkv = hkv; p.d = d; p.scale = scale; p.scale_log2 = scale * kLog2e;
  p.mask = mask;
  p.window = window;
  p.slopes = bias_slopes;
  if (!pick_btab(bias, &p.btab, &p.bss, &p.bhs, &p.brs)) return ATTN_ERR_INVALID_ARG;
  const int elem = dtype == ATTN_DTYPE_FP32 ? 4 : 2;
  if (!pick_strides(strides ? strides->q : nullptr, hq, d, elem, &p.sq) ||
      !pick_strides(strides ? strides->k : nullptr, hkv, d, elem, &p.sk) ||
      !pick_strides(strides ? strides->v : nullptr, hkv, d, elem, &p.sv) ||
      !pick_strides(strides ? strides->o : nullptr, hq, d, elem, &p.so) ||
      !pick_strides(strides ? strides->dout : nullptr, hq, d, elem, &p.sdo) ||
      !pick_strides(strides ? strides->dq : nullptr, hq, d, elem, &p.sdq) ||
      !pick_strides(strides ? strides->dk : nullptr, hkv, d, elem, &p.sdk) ||
      !pick_strides(strides ? strides->dv : nullptr, hkv, d, elem, &p.sdv))
    return ATTN_ERR_INVALID_ARG;
  // the gradients are zeroed and written 16 bytes at a time
  if ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) |
       reinterpret_cast<uintptr_t>(dv)) & 15)
    return ATTN_ERR_INVALID_ARG;
  p.err = device_error_ptr();
  if (!p.err) return ATTN_ERR_CUDA;
  p.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  char *ws = static_cast<char *>(workspace);
  const BwdLayout wl = bwd_layout(total_q, total_k, hq, hkv, d, dtype);
  p.delta = reinterpret_cast<float *>(ws + wl.delta);
  p.lse2 = reinterpret_cast<float *>(ws + wl.lse2);
  if (batch == 0) {
    set_plan("empty");
    return ATTN_OK;
  }
  // Keys of no sequence (none when cu_k[batch] == total_k) and rows beyond
  // max_k are covered by the kernels; a zero fill first keeps dk/dv defined
  // even when the device flags inconsistent cu_seqlens.
  cudaError_t ce = cudaSuccess;
  if (total_k > 0) {  // every (token, head) row of dk and dv, whatever the strides
    ce = launch_zero_rows(dk, total_k, hkv, d, p.sdk, elem, cs);
    if (ce == cudaSuccess) ce = launch_zero_rows(dv, total_k, hkv, d, p.sdv, elem, cs);
  }
  char desc[320];
  desc[0] = 0;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(dout);
  // a bias tensor rides on the raw scores: tensor cores only with a positive
  // scale and no slopes
  const bool tc = dtype == ATTN_DTYPE_BF16 && kTensorCorePath && total_k > 0 && total_q > 0 &&
                  (mis & 15) == 0 && (!p.btab || (scale > 0.f && !bias_slopes));
  if (tc) {
    p.q16 = ws + wl.q16;
    p.do16 = ws + wl.do16;
    p.k16 = ws + wl.k16;
    p.v16 = ws + wl.v16;
    p.amax = reinterpret_cast<unsigned int *>(ws + wl.amax);
    // Without the forward's fp32 output, D_i = dO_i . O_i comes from a
    // forward pass that recomputes it (the rounded O would carry its bf16
    // error into every gradient through D).
    p.delta_ready = o_f32 ? 0 : 1;
    if (ce == cudaSuccess) ce = launch_bwd_amax(p, cs);
    if (ce == cudaSuccess) ce = launch_bwd_pre(p, dtype, cs);
    if (ce == cudaSuccess) ce = launch_kv_to_f16(p, cs);
    if (ce == cudaSuccess && !o_f32) {
      FwdParams fp{};
      fp.q = q; fp.k = k; fp.v = v;
      fp.cu_q = cu_q; fp.cu_k = cu_k;
      fp.batch = batch; fp.max_q = max_q; fp.max_k = max_k; fp.total_q = total_q;
      fp.total_k = total_k;
      fp.hq = hq; fp.hkv = hkv; fp.d = d; fp.scale = scale; fp.scale_log2 = p.scale_log2;
      fp.mask = mask;
      fp.window = window;
      fp.slopes = bias_slopes;
      fp.btab = p.btab; fp.bss = p.bss; fp.bhs = p.bhs; fp.brs = p.brs;
      fp.sq = p.sq; fp.sk = p.sk; fp.sv = p.sv;
      fp.err = p.err;
      fp.dout = dout; fp.sdo = p.sdo; fp.delta = p.delta;
      fp.wait_ns = p.wait_ns;
      ce = launch_fwd_tc2_delta(fp, cs);
    }
    if (ce == cudaSuccess) {
      if (d == 128 && !g_deterministic.load(std::memory_order_relaxed)) {
        p.dqacc = reinterpret_cast<float *>(ws + wl.dqacc);
        ce = launch_bwd_fused(p, cs, desc, sizeof(desc));
      } else {
        ce = launch_bwd_tc(p, cs, desc, sizeof(desc));
      }
    }
  } else {
    if (ce == cudaSuccess) ce = launch_bwd_simt(p, dtype, cs);
    snprintf(desc, sizeof(desc), "bwd_pre+bwd_dq_simt+bwd_dkdv_simt_%s_d%d%s",
             dtype == ATTN_DTYPE_FP32 ? "fp32" : "bf16", d, p.btab ? "_btab" : "");
  }
  set_plan(desc);
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_mask_probe(const int32_t *cu_q, const int32_t *cu_k, int batch, int max_q,
                            int max_k, int total_q, int total_k, attn_mask_kind mask,
                            int window, int tile_rows, uint8_t *out, void *stream) {
  attn_status st = check_sizes(batch, max_q, max_k, total_q, total_k, 1, 1, 64, mask, window,
                               ATTN_DTYPE_BF16);
  if (st != ATTN_OK) return st;
  if (tile_rows != 16 && tile_rows != 32 && tile_rows != 64 && tile_rows != 128)
    return ATTN_ERR_INVALID_ARG;
  if ((long long)total_q * total_k >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;
  if (batch > 0 && (!cu_q || !cu_k)) return ATTN_ERR_INVALID_ARG;
  if ((long long)total_q * total_k > 0 && !out) return ATTN_ERR_INVALID_ARG;
  int *err = device_error_ptr();
  if (!err) return ATTN_ERR_CUDA;
  if ((long long)total_q * total_k == 0) return ATTN_OK;
  cudaError_t ce = launch_mask_probe(cu_q, cu_k, batch, max_q, max_k, total_q, total_k, mask,
                                     window, tile_rows, out, err,
                                     static_cast<cudaStream_t>(stream));
  return ce == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status attn_get_device_error(void *stream) {
  int *flag = device_error_ptr();
  if (!flag) return ATTN_ERR_CUDA;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  return static_cast<attn_status>(v);
}

}  // extern "C"
