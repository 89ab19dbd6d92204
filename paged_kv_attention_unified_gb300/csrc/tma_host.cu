// Host side of TMA: tensor-map encoding through the driver entry point.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "ua_kernels.h"

namespace ua {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}
}  // namespace

cudaError_t encode_tiled_map(CUtensorMap* map, int elt_bytes, int rank, const void* base,
                             const uint64_t* dims, const uint64_t* strides_bytes,
                             const uint32_t* box, bool swizzle_128b, int l2_promotion) {
  auto encode = encode_fn();
  if (encode == nullptr) return cudaErrorNotSupported;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  const CUtensorMapDataType dt =
      elt_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUresult r =
      encode(map, dt, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, st, b, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle_128b ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             l2_promotion >= 256   ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
             : l2_promotion >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                   : CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_kv_page_map(CUtensorMap* map, const void* cache, int elt_bytes, int head_dim,
                               int num_kv_heads, int block_size, int64_t num_blocks,
                               int box_dims, int box_rows, bool swizzle_128b) {
  const uint64_t D = static_cast<uint64_t>(head_dim);
  const uint64_t e = static_cast<uint64_t>(elt_bytes);
  uint64_t dims[4] = {D, static_cast<uint64_t>(num_kv_heads), static_cast<uint64_t>(block_size),
                      static_cast<uint64_t>(num_blocks)};
  uint64_t strides[3] = {D * e, static_cast<uint64_t>(num_kv_heads) * D * e,
                         static_cast<uint64_t>(block_size) * num_kv_heads * D * e};
  uint32_t box[4] = {static_cast<uint32_t>(box_dims), 1, static_cast<uint32_t>(box_rows), 1};
  // L2 fetches no wider than one head's row: the neighbouring head's row
  // belongs to another CTA, which may read it only after it left L2.
  const int row_bytes = static_cast<int>(D * e);
  return encode_tiled_map(map, elt_bytes, 4, cache, dims, strides, box, swizzle_128b,
                          row_bytes >= 256 ? 256 : (row_bytes >= 128 ? 128 : 64));
}

}  // namespace ua
