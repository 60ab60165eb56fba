// decode_qt_fp8.cu -- the query-tile kernel's fp8 instances (head_dim 128, 256).
#include "decode_qt.cuh"

namespace kvq {

cudaError_t launch_decode_qt_fp8(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                  int grid, size_t smem, cudaStream_t stream) {
  return dispatch_decode_qt<KVQ_FP8_E4M3>(head_dim, tk, tv, a, grid, smem, stream);
}

}  // namespace kvq
