// tma_map.h -- host-side construction of the TMA tensor maps the kernels use.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace attn {

// The driver's tensor-map encoder, looked up once through the runtime so the
// library does not link libcuda directly.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// A [T, H, D] 16-bit (bf16 or fp16) tensor seen as 3-D (d, head, token), loaded in boxes of
// 64 features x box_h heads x box_t tokens with the 128-byte swizzle (one
// 128-byte row per (token, head), the K-major layout tcgen05 descriptors
// expect).
// head_stride and token_stride are in elements (contiguous THD when they are
// D and H * D); the encoder checks that they are multiples of 16 bytes.
inline bool make_map(CUtensorMap *m, const void *base, int D, int H, int T, int box_h,
                     int box_t,
                     CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     long long head_stride = -1, long long token_stride = -1) {
  auto enc = tensor_map_encoder();
  if (!enc || T <= 0) return false;
  if (head_stride < 0) head_stride = D;
  if (token_stride < 0) token_stride = (long long)H * D;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)head_stride * 2, (cuuint64_t)token_stride * 2};
  cuuint32_t box[3] = {64u, (cuuint32_t)box_h, (cuuint32_t)box_t};
  cuuint32_t es[3] = {1u, 1u, 1u};
  CUresult r = enc(m, dt, 3, const_cast<void *>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A contiguous [T, H, D] fp32 tensor seen as 3-D (d, head, token), boxes of
// box_d features x 1 head x box_t tokens, no swizzle (rows of box_d floats
// packed in shared memory).
inline bool make_map_f32(CUtensorMap *m, float *base, int D, int H, int T, int box_d, int box_t) {
  auto enc = tensor_map_encoder();
  if (!enc || !base || T <= 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
  cuuint64_t strides[2] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4};
  cuuint32_t box[3] = {(cuuint32_t)box_d, 1u, (cuuint32_t)box_t};
  cuuint32_t es[3] = {1u, 1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An fp32 bias tensor seen as 3-D (key, row, sequence), element strides
// row_stride and seq_stride (0: the sequences share one set of entries),
// loaded in boxes of 32 keys x 128 rows with the 128-byte swizzle.  Entries
// past `keys`, `rows` or `seqs` read as 0.  false when the encoder rejects
// it (the base or a stride not a multiple of 16 bytes).
inline bool make_bias_map(CUtensorMap *m, const float *base, int keys, int rows, int seqs,
                          long long row_stride, long long seq_stride) {
  auto enc = tensor_map_encoder();
  if (!enc || !base || keys <= 0 || rows <= 0 || seqs <= 0 || row_stride <= 0 || seq_stride < 0)
    return false;
  if (seq_stride == 0) {
    seqs = 1;
    seq_stride = row_stride * rows;
  }
  cuuint64_t dims[3] = {(cuuint64_t)keys, (cuuint64_t)rows, (cuuint64_t)seqs};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride * 4, (cuuint64_t)seq_stride * 4};
  cuuint32_t box[3] = {32u, 128u, 1u};
  cuuint32_t es[3] = {1u, 1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace attn
