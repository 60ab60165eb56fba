// decode_int8.cu -- instantiates the split-KV decode kernel for int8 cache codes
// (head_dim 64, 128, 256; grouped and, where it applies, wide consumer
// layouts).  One translation unit per element type keeps the build parallel.
#include "decode.cuh"

namespace kvq {

cudaError_t launch_decode_int8(int head_dim, int nt, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeArgs& a, int grid, int threads, size_t smem, cudaStream_t stream) {
  return dispatch_decode<KVQ_INT8, false>(head_dim, nt, &tk, &tv, &a, grid, threads, smem, stream, nullptr);
}

cudaError_t occupancy_decode_int8(int head_dim, int nt, int threads, size_t smem, int* blocks_per_sm) {
  return dispatch_decode<KVQ_INT8, true>(head_dim, nt, nullptr, nullptr, nullptr, 0, threads, smem, nullptr,
                                   blocks_per_sm);
}

}  // namespace kvq
