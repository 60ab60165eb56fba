// decode_tc_int4.cu -- instantiates the tensor-memory decode kernel for int4
// cache codes (head_dim 128 and 256, 32 / 48 / 64 padded query rows).
#include "decode_tc.cuh"

namespace kvq {

cudaError_t launch_decode_tc_int4(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream) {
  return dispatch_decode_tc<KVQ_INT4, false>(head_dim, nr, tk, tv, a, grid, smem, stream);
}

}  // namespace kvq
