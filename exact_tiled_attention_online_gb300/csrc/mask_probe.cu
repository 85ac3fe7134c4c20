// mask_probe.cu -- writes the allowed-pair matrix that the tile planner and
// the per-lane predicate of common.cuh produce, so it can be compared bit for
// bit with an independent definition of the mask.
#include "common.cuh"
#include "plan.h"

namespace attn {

__global__ void mask_probe_kernel(const int32_t *cu_q, const int32_t *cu_k, int total_q,
                                  int total_k, int max_q, int max_k, int mask, int window,
                                  int tile_rows, uint8_t *out, int *err) {
  const int s = blockIdx.y;
  SeqGeom g = load_seq(cu_q, cu_k, s, total_q, total_k, max_q, max_k, mask, window);
  if (!g.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(err, ATTN_ERR_DEVICE_BOUNDS);
    return;
  }
  const int i0 = blockIdx.x * tile_rows;
  const KvRange kr = plan_kv_tiles(g.mask, g.window, g.nq, g.nk, i0, tile_rows, kTileKeys);
  for (int r = threadIdx.x; r < tile_rows; r += blockDim.x) {
    const int i = i0 + r;
    if (i >= g.nq) continue;  // out-of-range lane: no storage of its own
    uint8_t *row = out + (size_t)(g.q0 + i) * total_k + g.k0;
    for (int n = kr.n_begin; n < kr.n_end; n++)
      for (int c = 0; c < kTileKeys; c++) {
        const int j = n * kTileKeys + c;
        const bool ok = kr.full(n) ? true : lane_allowed(g.mask, g.window, i, j, g.nq, g.nk);
        if (ok) row[j] = 1;
      }
  }
}

cudaError_t launch_mask_probe(const int32_t *cu_q, const int32_t *cu_k, int batch, int max_q,
                              int max_k, int total_q, int total_k, int mask, int window,
                              int tile_rows, uint8_t *out, int *err, cudaStream_t st) {
  cudaError_t ce = cudaMemsetAsync(out, 0, (size_t)total_q * total_k, st);
  if (ce != cudaSuccess || batch == 0 || max_q == 0) return ce;
  dim3 grid((max_q + tile_rows - 1) / tile_rows, batch);
  mask_probe_kernel<<<grid, 128, 0, st>>>(cu_q, cu_k, total_q, total_k, max_q, max_k, mask,
                                          window, tile_rows, out, err);
  return cudaGetLastError();
}

}  // namespace attn
