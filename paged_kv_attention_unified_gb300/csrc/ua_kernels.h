// Launch entry points of the device kernels (host side of each .cu file).
#pragma once

#include <cuda_runtime.h>

#include "ua_device.cuh"

namespace ua {

// Split-KV decode kernel over p.tiles[0 .. p.num_tiles).
cudaError_t launch_decode(const KernelParams& p, int head_dim, int kv_dtype, cudaStream_t stream);

// Log-sum-exp combine of split partials into bf16 output rows.
cudaError_t launch_combine(const CombineParams& c, int head_dim, cudaStream_t stream);

// Test aid: copy the raw K/V rows each tile reads into dense buffers.
cudaError_t launch_gather_debug(const KernelParams& p, const int64_t* row_offsets, int head_dim,
                                int elt_bytes, void* k_out, void* v_out, cudaStream_t stream);

}  // namespace ua
