// decode_tc_fp8.cu -- instantiates the tensor-memory decode kernel for fp8 e4m3
// cache codes (head_dim 128 and 256, 32 / 48 / 64 padded query rows).
#include "decode_tc.cuh"

namespace kvq {

cudaError_t launch_decode_tc_fp8(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream) {
  return dispatch_decode_tc<KVQ_FP8_E4M3, false>(head_dim, nr, tk, tv, a, grid, smem, stream);
}

}  // namespace kvq
