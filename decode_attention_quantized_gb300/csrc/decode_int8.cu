// decode_int8.cu -- instantiates the split-KV decode kernel for int8 cache codes
// (head_dim 64, 128, 256).  One translation unit per element type keeps the
// build parallel.
#include "decode.cuh"

namespace kvq {

cudaError_t launch_decode_int8(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                             int grid, int threads, size_t smem, cudaStream_t stream) {
  return launch_decode_t<KVQ_INT8>(head_dim, tk, tv, a, grid, threads, smem, stream);
}

cudaError_t occupancy_decode_int8(int head_dim, int threads, size_t smem, int* blocks_per_sm) {
  return occupancy_decode_t<KVQ_INT8>(head_dim, threads, smem, blocks_per_sm);
}

}  // namespace kvq
