// combine.cu -- fixed-order log-sum-exp merge of split-KV partials, exact
// head-sink rescale, static V scale and bf16 store.
//
// Flash-decoding with partials merged in a fixed order, so repeated decodes
// are bitwise identical: kv-quant-attn page, section "Method".  Head sink
// o *= 1/(1+exp(s_h - lse)): ApplyHeadSink in onnxruntime PR #29912.  The
// per-channel V scale applied to the output (the V half of the per-channel
// fold): onnxruntime PR #32515, Description.
//
// One warp per output row (b, t, query head); each lane owns D/32 consecutive
// channels.  Splits are visited in ascending key order by every lane.
#include <cuda_bf16.h>

#include "kvq_internal.h"
#include "ptx.cuh"

namespace kvq {
namespace {

template <int D>
__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int row_id = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int n_rows = a.batch * a.q_tokens * a.num_q_heads;
  if (row_id >= n_rows) return;
  const int hq = row_id % a.num_q_heads;
  const int t = (row_id / a.num_q_heads) % a.q_tokens;
  const int b = row_id / (a.num_q_heads * a.q_tokens);
  const int h = hq / a.group;
  const int r = t * a.group + (hq % a.group);  // row inside a work unit

  const int* prefix = a.plan + 4;
  const int i0 = prefix[b], i1 = prefix[b + 1];

  float m = -INFINITY;
  for (int it = i0 + lane; it < i1; it += 32) m = fmaxf(m, a.part_lse[((size_t)it * a.num_kv_heads + h) * a.rows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  float wsum = 0.0f;
  if (m != -INFINITY) {
    for (int it = i0; it < i1; ++it) {
      const size_t u = ((size_t)it * a.num_kv_heads + h) * a.rows + r;
      const float l2 = a.part_lse[u];
      if (l2 == -INFINITY) continue;
      const float w = ptx::fast_exp2(l2 - m);
      wsum += w;
      const float* po = a.part_o + u * D + lane * E;
      if constexpr (E % 4 == 0) {
#pragma unroll
        for (int e = 0; e < E; e += 4) {
          const float4 v = *reinterpret_cast<const float4*>(po + e);
          acc[e] += w * v.x;
          acc[e + 1] += w * v.y;
          acc[e + 2] += w * v.z;
          acc[e + 3] += w * v.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          const float2 v = *reinterpret_cast<const float2*>(po + e);
          acc[e] += w * v.x;
          acc[e + 1] += w * v.y;
        }
      }
    }
  }

  float lse_nat = -INFINITY;
  if (wsum > 0.0f) {
    const float inv = 1.0f / wsum;
    const float lse2 = m + ptx::fast_log2(wsum);
    lse_nat = lse2 * 0.69314718055994530942f;
    float f = inv;
    if (a.head_sink) f = inv / (1.0f + expf(a.head_sink[hq] - lse_nat));
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= f;
    if (a.v_mode == KVQ_SCALE_PER_TENSOR) {
      const float vs = a.v_scale[0];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= vs;
    } else if (a.v_mode == KVQ_SCALE_PER_CHANNEL) {
      const float* vs = a.v_scale + (size_t)h * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] *= vs[e];
    }
  }

  uint32_t packed[E / 2];
#pragma unroll
  for (int e = 0; e < E; e += 2) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(acc[e], acc[e + 1]);
    packed[e / 2] = *reinterpret_cast<const uint32_t*>(&v);
  }
  uint16_t* dst = a.out + (size_t)row_id * D + lane * E;
  if constexpr (E == 8) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  } else if constexpr (E == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  }
  if (a.lse_out && lane == 0) a.lse_out[row_id] = lse_nat;
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  const long long rows = (long long)a.batch * a.q_tokens * a.num_q_heads;
  const unsigned blocks = (unsigned)((rows + 7) / 8);
  switch (a.head_dim) {
    case 64: combine_kernel<64><<<blocks, 256, 0, stream>>>(a); break;
    case 128: combine_kernel<128><<<blocks, 256, 0, stream>>>(a); break;
    case 256: combine_kernel<256><<<blocks, 256, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace kvq
