// combine.cu -- fixed-order log-sum-exp merge of split-KV partials, exact
// head-sink rescale, static V scale and bf16 store.
//
// Flash-decoding with partials merged in a fixed order, so repeated decodes
// are bitwise identical: kv-quant-attn page, section "Method".  Head sink
// o *= 1/(1+exp(s_h - lse)): ApplyHeadSink in onnxruntime PR #29912.  The
// per-channel V scale applied to the output (the V half of the per-channel
// fold): onnxruntime PR #32515, Description.
//
// One CTA per output row (b, t, query head), or one warp per row for calls
// with many rows of few pieces; each lane owns D/32 consecutive channels.
#include <cuda_bf16.h>

#include "kvq_internal.h"
#include "ptx.cuh"

namespace kvq {
namespace {

constexpr int kCombineWarps = 8;

// The end of one row (every lane of one warp): the merged output acc (this
// lane's E channels) and weight sum against the row maximum m, the head sink,
// the static V scale, the bf16 store and the natural-log LSE.
template <int D>
__device__ __forceinline__ void combine_finish(const CombineArgs& a, int row_id, int hq, int h, int lane,
                                               float (&acc)[D / 32], float wsum, float m) {
  constexpr int E = D / 32;
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
  if (a.lse_out && lane == 0) a.lse_out[row_id] = lse_nat;
  if (lane * E >= a.out_dim) return;  // LATENT: only the leading v_head_size channels
  uint16_t* dst = a.out + (size_t)row_id * a.out_dim + lane * E;
  if constexpr (E == 8) {
    *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  } else if constexpr (E == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(packed[0], packed[1]);
  } else if constexpr (E == 2) {
    *reinterpret_cast<uint32_t*>(dst) = packed[0];
  } else {
    // head_dim 576: 18 channels a lane, the leading v_head_size (a multiple of
    // 8) written pair by pair
#pragma unroll
    for (int j = 0; j < E / 2; ++j)
      if (lane * E + 2 * j < a.out_dim) reinterpret_cast<uint32_t*>(dst)[j] = packed[j];
  }
}

// One CTA per output row; warp w folds pieces w, w + 8, ... (ascending), then
// warp 0 adds the eight warp sums in warp order.  Every split's weight is
// taken against the row's maximum log-sum-exp, so the result does not depend
// on how splits are spread over warps beyond that fixed order.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineArgs a) {
  constexpr int E = D / 32;
  __shared__ float s_acc[kCombineWarps][D];
  __shared__ float s_w[kCombineWarps];
  __shared__ float s_m[kCombineWarps];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row_id = blockIdx.x;
  const int hq = row_id % a.num_q_heads;
  const int t = (row_id / a.num_q_heads) % a.q_tokens;
  const int b = row_id / (a.num_q_heads * a.q_tokens);
  const int h = hq / a.group;
  const int r = t * a.group + (hq % a.group);  // row inside a work unit

  // pieces of segment s = b * Hkv + h are the CTAs whose cost ranges [x W,
  // (x + 1) W) meet the segment's tiles, which sit at cost positions
  // first tile + c s onward; the piece of CTA x sits in slot s + x
  const int W = a.plan[0], c = a.plan[2];
  const int* pre = a.plan + 4;
  const int nb = pre[b + 1] - pre[b];
  const int seg = b * a.num_kv_heads + h;
  const long long s_cost = (long long)pre[b] * a.num_kv_heads + (long long)h * nb + (long long)c * seg;
  const int i0 = nb > 0 ? seg + (int)(s_cost / W) : 0;
  const int i1 = nb > 0 ? seg + (int)((s_cost + nb - 1) / W) + 1 : 0;
  auto lse_of = [&](int slot) { return a.part_lse[(size_t)slot * a.rows + r]; };

  float m = -INFINITY;
  for (int it = i0 + threadIdx.x; it < i1; it += blockDim.x) m = fmaxf(m, lse_of(it));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_m[warp] = m;
  __syncthreads();
  m = s_m[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) m = fmaxf(m, s_m[w]);

  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  float wsum = 0.0f;
  if (m != -INFINITY) {
    for (int it = i0 + warp; it < i1; it += kCombineWarps) {
      const size_t u = (size_t)it * a.rows + r;
      const float l2 = a.part_lse[u];
      const float w = l2 == -INFINITY ? 0.0f : ptx::fast_exp2(l2 - m);
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
#pragma unroll
  for (int e = 0; e < E; ++e) s_acc[warp][lane * E + e] = acc[e];
  if (lane == 0) s_w[warp] = wsum;
  __syncthreads();
  if (warp != 0) return;

  wsum = s_w[0];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = s_acc[0][lane * E + e];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) {
    wsum += s_w[w];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] += s_acc[w][lane * E + e];
  }

  combine_finish<D>(a, row_id, hq, h, lane, acc, wsum, m);
}

// One warp per output row, kCombineWarps rows a CTA: for calls with many rows
// of few pieces each (a prefill chunk: B x C x Hq rows; a ragged decode
// batch), where a CTA per row leaves the GPU waiting on launch and latency
// and takes room the next step's decode could use.  The row's pieces are
// folded in slot order against the row's maximum, then combine_finish.
template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_rows_kernel(const CombineArgs a) {
  constexpr int E = D / 32;
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long row_ll = (long long)blockIdx.x * kCombineWarps + warp;
  if (row_ll >= (long long)a.batch * a.q_tokens * a.num_q_heads) return;
  const int row_id = (int)row_ll;
  const int hq = row_id % a.num_q_heads;
  const int t = (row_id / a.num_q_heads) % a.q_tokens;
  const int b = row_id / (a.num_q_heads * a.q_tokens);
  const int h = hq / a.group;
  const int r = t * a.group + (hq % a.group);
  const int W = a.plan[0], c = a.plan[2];
  const int* pre = a.plan + 4;
  const int nb = pre[b + 1] - pre[b];
  const int seg = b * a.num_kv_heads + h;
  const long long s_cost = (long long)pre[b] * a.num_kv_heads + (long long)h * nb + (long long)c * seg;
  const int i0 = nb > 0 ? seg + (int)(s_cost / W) : 0;
  const int i1 = nb > 0 ? seg + (int)((s_cost + nb - 1) / W) + 1 : 0;

  float m = -INFINITY;
  for (int it = i0 + lane; it < i1; it += 32) m = fmaxf(m, a.part_lse[(size_t)it * a.rows + r]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.0f;
  float wsum = 0.0f;
  if (m != -INFINITY) {
    // 32 pieces at a time: lane j takes the weight of piece base + j, the
    // warp then adds the pieces in order, loading four ahead of their FMAs
    for (int base = i0; base < i1; base += 32) {
      const int n = min(32, i1 - base);
      float wl = 0.0f;
      if (lane < n) {
        const float l2 = a.part_lse[(size_t)(base + lane) * a.rows + r];
        wl = l2 == -INFINITY ? 0.0f : ptx::fast_exp2(l2 - m);
      }
      float ws = wl;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
      wsum += ws;
      for (int j = 0; j < n; j += 4) {
        float v[4][E];
        float w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          w[q] = __shfl_sync(0xffffffffu, wl, (j + q) & 31);
          if (j + q < n) {
            const float* po = a.part_o + ((size_t)(base + j + q) * a.rows + r) * D + lane * E;
            if constexpr (E % 4 == 0) {
#pragma unroll
              for (int e = 0; e < E; e += 4) {
                const float4 t = *reinterpret_cast<const float4*>(po + e);
                v[q][e] = t.x;
                v[q][e + 1] = t.y;
                v[q][e + 2] = t.z;
                v[q][e + 3] = t.w;
              }
            } else {
#pragma unroll
              for (int e = 0; e < E; e += 2) {
                const float2 t = *reinterpret_cast<const float2*>(po + e);
                v[q][e] = t.x;
                v[q][e + 1] = t.y;
              }
            }
          } else {
            w[q] = 0.0f;
#pragma unroll
            for (int e = 0; e < E; ++e) v[q][e] = 0.0f;
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[e] += w[q] * v[q][e];
      }
    }
  }
  combine_finish<D>(a, row_id, hq, h, lane, acc, wsum, m);
}

// Sequence lengths of a prefill chunk's virtual sequences (one thread each).
__global__ void __launch_bounds__(256) prefill_lens_kernel(const int32_t* seq_lens, int32_t* out, int total, int n,
                                                           int C, int T) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  const int b = i / n, j = i - b * n;
  out[i] = max(0, seq_lens[b] - C + T * (j + 1));
}

// One thread waits on an mbarrier that nothing arrives on, with the bounded
// wait every pipeline wait uses, here given `limit_ns`: it must give up and
// flag KVQ_DEVERR_TIMEOUT, leaving the context usable.
__global__ void __launch_bounds__(32) wait_probe_kernel(unsigned int* err, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  ptx::mbar_init(&bar, 1);
  ptx::fence_mbar_init();
  if (!ptx::mbar_wait_slow(&bar, 0, limit_ns)) atomicOr(err, KVQ_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_probe(unsigned int* err, unsigned long long limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(err, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_prefill_lens(const int32_t* seq_lens, int32_t* out, int batch, int n, int C, int T,
                                cudaStream_t stream) {
  const int total = batch * n;
  return launch_pdl(prefill_lens_kernel, (unsigned)((total + 255) / 256), 256, 0, stream, seq_lens, out, total,
                    n, C, T);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream, bool warp_rows) {
  const long long rows = (long long)a.batch * a.q_tokens * a.num_q_heads;
  constexpr int threads = kCombineWarps * 32;
  if (warp_rows) {
    const unsigned blocks = (unsigned)((rows + kCombineWarps - 1) / kCombineWarps);
    switch (a.head_dim) {
      case 64: return launch_pdl(combine_rows_kernel<64>, blocks, threads, 0, stream, a);
      case 128: return launch_pdl(combine_rows_kernel<128>, blocks, threads, 0, stream, a);
      case 256: return launch_pdl(combine_rows_kernel<256>, blocks, threads, 0, stream, a);
      case 576: return launch_pdl(combine_rows_kernel<576>, blocks, threads, 0, stream, a);
      default: return cudaErrorInvalidValue;
    }
  }
  const unsigned blocks = (unsigned)rows;
  switch (a.head_dim) {
    case 64: return launch_pdl(combine_kernel<64>, blocks, threads, 0, stream, a);
    case 128: return launch_pdl(combine_kernel<128>, blocks, threads, 0, stream, a);
    case 256: return launch_pdl(combine_kernel<256>, blocks, threads, 0, stream, a);
    case 576: return launch_pdl(combine_kernel<576>, blocks, threads, 0, stream, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
