// decode_tc_grp_fp8.cu -- instantiates the tensor-memory decode kernel with
// group-wise scales for fp8 cache codes (head_dim 128 and 256, 32 / 48 / 64
// padded query rows); a translation unit of its own so that the build
// compiles it in parallel with the others.
#include "decode_tc.cuh"

namespace kvq {

cudaError_t launch_decode_tc_grp_fp8(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream) {
  return dispatch_decode_tc<KVQ_FP8_E4M3, true>(head_dim, nr, tk, tv, a, grid, smem, stream);
}

}  // namespace kvq
