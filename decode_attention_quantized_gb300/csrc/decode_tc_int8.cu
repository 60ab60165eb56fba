// decode_tc_int8.cu -- instantiates the tensor-memory decode kernel for int8
// cache codes (head_dim 128 and 256, 32 / 48 / 64 padded query rows).
#include "decode_tc.cuh"

namespace kvq {

cudaError_t launch_decode_tc_int8(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream) {
  return dispatch_decode_tc<KVQ_INT8, false>(head_dim, nr, tk, tv, a, grid, smem, stream);
}

}  // namespace kvq
