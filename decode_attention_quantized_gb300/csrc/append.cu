// append.cu -- quantize-on-write of new K/V rows into their paged-cache slots
// (ReshapeAndCache in onnxruntime PR #29912; per-row absmax scales as in the
// kv-quant-attn page, section "Method"; int4 two-per-byte packing as in
// onnxruntime PR #32515), optionally behind the fused QK-RMSNorm + RoPE
// prologue on K (QkNormRotaryTNH, PR #29912), which also runs alone on Q.
//
// Per-group scales (the group-wise scaling the kv-quant-attn page lists under
// "Requirements and limits" as not done there) apply the per-row rule to each
// run of group_size channels.
//
// One warp per (token, kv head, side): each lane holds D/32 consecutive
// channels, the row's absmax is a warp max-reduction (exact, order free; a
// group's over the lanes that hold it), the
// scale and every code use IEEE fp32 division (never a reciprocal multiply,
// which overflows for subnormal scales), codes round half to even.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kvq_internal.h"
#include "ptx.cuh"

namespace kvq {
namespace {

template <int E>
__device__ __forceinline__ void load_bf16(const uint16_t* p, float (&x)[E]) {
  if constexpr (E == 8) {
    uint4 v = *reinterpret_cast<const uint4*>(p);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else if constexpr (E == 4) {
    uint2 v = *reinterpret_cast<const uint2*>(p);
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xFFFF0000u);
  } else {
    // E even (2, or 18 at head_dim 576): 32-bit loads
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
      const uint32_t v = reinterpret_cast<const uint32_t*>(p)[i];
      x[2 * i] = __uint_as_float(v << 16);
      x[2 * i + 1] = __uint_as_float(v & 0xFFFF0000u);
    }
  }
}

template <int NB>
__device__ __forceinline__ void store_bytes(uint8_t* dst, const uint8_t (&b)[NB]) {
  if constexpr (NB == 8) {
    uint2 v;
    v.x = b[0] | (b[1] << 8) | (b[2] << 16) | ((uint32_t)b[3] << 24);
    v.y = b[4] | (b[5] << 8) | (b[6] << 16) | ((uint32_t)b[7] << 24);
    *reinterpret_cast<uint2*>(dst) = v;
  } else if constexpr (NB == 4) {
    *reinterpret_cast<uint32_t*>(dst) = b[0] | (b[1] << 8) | (b[2] << 16) | ((uint32_t)b[3] << 24);
  } else if constexpr (NB == 2) {
    *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(b[0] | (b[1] << 8));
  } else if constexpr (NB % 2 == 0) {
    // 18 bytes (head_dim 576): 16-bit stores
#pragma unroll
    for (int i = 0; i < NB / 2; ++i) reinterpret_cast<uint16_t*>(dst)[i] = (uint16_t)(b[2 * i] | (b[2 * i + 1] << 8));
  } else {
#pragma unroll
    for (int i = 0; i < NB; ++i) dst[i] = b[i];
  }
}

// Nearest bf16 to the float f, ties to even, as the float it denotes: add
// half a bf16 unit less one to the bit pattern, plus the kept lowest bit, and
// truncate (a carry into the exponent rounds up to the next binade or to
// infinity); NaN stays a quiet NaN.
__device__ __forceinline__ float bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return __uint_as_float(0x7FC00000u);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return __uint_as_float(u & 0xFFFF0000u);
}

// QK-RMSNorm, RoPE, then optionally the Walsh-Hadamard rotation, on one
// (token, head) row held by a warp, E channels per lane (channel lane * E +
// e), one bf16 rounding at the end
// (QkNormRotaryTNH, onnxruntime PR #29912, Summary of Changes).  The bf16
// result decides the quantized codes, so every step is one IEEE fp32
// operation in a fixed order: per-lane sums of squares in channel order, then
// a butterfly over lanes 16, 8, 4, 2, 1 (every lane ends with the same bits),
// r = 1 / sqrt(s / D + eps), y = (x * r) * w, and each rotated value as
// (y * cos) -+ (partner * sin) with both products rounded.  `ys` is this
// warp's staging row of 32 E floats, used to fetch each channel's rotation
// partner.  Returns false, after flagging KVQ_DEVERR_POSITION, when the
// token's position is outside the tables (the caller then writes nothing).
template <int E>
__device__ bool norm_rope_row(const NormRope& p, int n, int lane, float (&x)[E], float* ys, unsigned int* err) {
  constexpr int D = 32 * E;
  long long pos = 0;
  if (p.rd > 0) {
    pos = p.positions[n];
    if (pos < 0 || pos >= p.max_pos) {
      if (lane == 0) atomicOr(err, KVQ_DEVERR_POSITION);
      return false;
    }
  }
  if (p.w) {
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss = __fadd_rn(ss, __fmul_rn(x[e], x[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)D), p.eps)));
    float w[E];
    load_bf16<E>(p.w + lane * E, w);
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = __fmul_rn(__fmul_rn(x[e], r), w[e]);
  }
  if (p.rd > 0) {
#pragma unroll
    for (int e = 0; e < E; ++e) ys[lane * E + e] = x[e];
    __syncwarp();
    const int half = p.rd >> 1;
    const float* cs = p.cos_tab + (size_t)pos * half;
    const float* sn = p.sin_tab + (size_t)pos * half;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int c = lane * E + e, j = c - p.off;
      if (j >= 0 && j < p.rd) {
        const bool first = p.interleaved ? (j & 1) == 0 : j < half;
        const int i = p.interleaved ? j >> 1 : (first ? j : j - half);
        const int partner = p.interleaved ? (first ? c + 1 : c - 1) : (first ? c + half : c - half);
        const float co = cs[i], si = sn[i], o = ys[partner];
        x[e] = first ? __fsub_rn(__fmul_rn(x[e], co), __fmul_rn(o, si))
                     : __fadd_rn(__fmul_rn(x[e], co), __fmul_rn(o, si));
      }
    }
    __syncwarp();
  }
  if constexpr ((E & (E - 1)) == 0) {  // a power of two (the host checks head_dim)
  if (p.hadamard) {
    // Sylvester-order butterflies: span s pairs channels c and c + s (c & s
    // == 0) into (a + b, a - b); spans below E stay inside the lane, the rest
    // pair lane l with lane l ^ (s / E)
#pragma unroll
    for (int s = 1; s < E; s <<= 1) {
#pragma unroll
      for (int e = 0; e < E; ++e)
        if (!(e & s)) {
          const float a0 = x[e], b0 = x[e + s];
          x[e] = __fadd_rn(a0, b0);
          x[e + s] = __fsub_rn(a0, b0);
        }
    }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, x[e], m);
        x[e] = upper ? __fsub_rn(o, x[e]) : __fadd_rn(x[e], o);
      }
    }
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = __fmul_rn(x[e], p.had_scale);
  }
  }
#pragma unroll
  for (int e = 0; e < E; ++e) x[e] = bf16_rne(x[e]);
  return true;
}

template <int D>
__global__ void __launch_bounds__(256) append_kernel(const AppendArgs a) {
  constexpr int E = D / 32;  // channels per lane
  // the next kernel (a decode of these tokens) may be scheduled at once: it
  // waits for this grid, which waits for the one before it, before it reads
  // the rows written here or writes anything, so its early work overlaps
  // both this grid and the combine enqueued before it
  ptx::griddep_launch_dependents();
  ptx::griddep_wait();
  const int wg = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (wg >= a.n_tokens * a.num_kv_heads * 2) return;
  const int side = wg & 1;  // 0: K, 1: V
  if (side == 1 && a.latent) return;  // LATENT: the K row is also V
  const int n = (wg >> 1) / a.num_kv_heads;
  const int h = (wg >> 1) % a.num_kv_heads;
  const long long slot = a.slots[n];
  if (slot < 0) return;  // padding token
  if (slot >= a.capacity) {
    if (lane == 0) atomicOr(a.err, KVQ_DEVERR_SLOT);
    return;
  }
  const long long blk = slot >> a.log2_bs;
  const int row = (int)(slot & (a.block_size - 1));
  const size_t ridx = ((size_t)blk * a.num_kv_heads + h) * a.block_size + row;

  float x[E];
  load_bf16<E>((side ? a.v_new : a.k_new) + ((size_t)n * a.num_kv_heads + h) * D + lane * E, x);
  if (a.k_prologue) {
    // both sides of a token are skipped when its position is bad: the V warp
    // checks the position too (without flagging it twice)
    __shared__ float ys[8][D];
    if (side == 0) {
      if (!norm_rope_row<E>(a.pro, n, lane, x, ys[(threadIdx.x >> 5) & 7], a.err)) return;
    } else if (a.pro.rd > 0) {
      const long long pos = a.pro.positions[n];
      if (pos < 0 || pos >= a.pro.max_pos) return;
    }
  }

  const int mode = side ? a.v_mode : a.k_mode;
  float* sc = side ? a.v_scale : a.k_scale;
  const float qmax = a.dtype == KVQ_INT8 ? 127.0f : (a.dtype == KVQ_INT4 ? 7.0f : 448.0f);
  float s[E];
  if (mode == KVQ_SCALE_PER_ROW) {
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float rs = __fdiv_rn(amax, qmax);
#pragma unroll
    for (int e = 0; e < E; ++e) s[e] = rs;
    if (lane == 0) sc[ridx] = rs;
  } else if (mode == KVQ_SCALE_PER_GROUP) {
    // the same per run of G channels: G / E consecutive lanes hold a group
    const int gl = (1 << a.log2_group) / E;
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
    for (int o = gl >> 1; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float rs = __fdiv_rn(amax, qmax);
#pragma unroll
    for (int e = 0; e < E; ++e) s[e] = rs;
    if ((lane & (gl - 1)) == 0) sc[ridx * (size_t)(D >> a.log2_group) + lane / gl] = rs;
  } else if (mode == KVQ_SCALE_PER_TENSOR) {
    const float t = sc[0];
#pragma unroll
    for (int e = 0; e < E; ++e) s[e] = t;
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) s[e] = sc[(size_t)h * D + lane * E + e];
  }

  uint8_t* codes = side ? a.v_codes : a.k_codes;
  if (a.dtype == KVQ_INT4) {
    uint8_t b[E / 2];
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
      int c[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int e = 2 * j + u;
        c[u] = 0;
        if (s[e] != 0.0f) c[u] = min(7, max(-7, __float2int_rn(__fdiv_rn(x[e], s[e]))));
      }
      b[j] = (uint8_t)((c[0] & 0xF) | ((c[1] & 0xF) << 4));
    }
    store_bytes<E / 2>(codes + ridx * (D / 2) + lane * (E / 2), b);
  } else {
    uint8_t b[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      if (s[e] == 0.0f) {
        b[e] = 0;
      } else if (a.dtype == KVQ_INT8) {
        b[e] = (uint8_t)(int8_t)min(127, max(-127, __float2int_rn(__fdiv_rn(x[e], s[e]))));
      } else {
        b[e] = (uint8_t)__nv_cvt_float_to_fp8(__fdiv_rn(x[e], s[e]), __NV_SATFINITE, __NV_E4M3);
      }
    }
    store_bytes<E>(codes + ridx * D + lane * E, b);
  }
}

// kvq_norm_rope_apply: one warp per (token, head) row of x -> y.
template <int D>
__global__ void __launch_bounds__(256) norm_rope_kernel(const NormRopeArgs a) {
  constexpr int E = D / 32;
  __shared__ float ys[8][D];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int wg = (int)((blockIdx.x * (size_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (wg >= a.n_tokens * a.num_heads) return;
  const int n = wg / a.num_heads;
  const size_t off = (size_t)wg * D + lane * E;
  float x[E];
  load_bf16<E>(a.x + off, x);
  if (!norm_rope_row<E>(a.pro, n, lane, x, ys[(threadIdx.x >> 5) & 7], a.err)) return;
  uint16_t b[E];
#pragma unroll
  for (int e = 0; e < E; ++e) b[e] = (uint16_t)(__float_as_uint(x[e]) >> 16);  // exact: x is a bf16 value
  if constexpr (E == 8) {
    uint4 v;
    v.x = b[0] | ((uint32_t)b[1] << 16); v.y = b[2] | ((uint32_t)b[3] << 16);
    v.z = b[4] | ((uint32_t)b[5] << 16); v.w = b[6] | ((uint32_t)b[7] << 16);
    *reinterpret_cast<uint4*>(a.y + off) = v;
  } else if constexpr (E == 4) {
    uint2 v;
    v.x = b[0] | ((uint32_t)b[1] << 16); v.y = b[2] | ((uint32_t)b[3] << 16);
    *reinterpret_cast<uint2*>(a.y + off) = v;
  } else {
#pragma unroll
    for (int i = 0; i < E / 2; ++i)
      reinterpret_cast<uint32_t*>(a.y + off)[i] = b[2 * i] | ((uint32_t)b[2 * i + 1] << 16);
  }
}

}  // namespace

cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t stream) {
  const long long warps = (long long)a.n_tokens * a.num_heads;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  switch (a.head_dim) {
    case 64: return launch_pdl(norm_rope_kernel<64>, blocks, 256, 0, stream, a);
    case 128: return launch_pdl(norm_rope_kernel<128>, blocks, 256, 0, stream, a);
    case 256: return launch_pdl(norm_rope_kernel<256>, blocks, 256, 0, stream, a);
    case 576: return launch_pdl(norm_rope_kernel<576>, blocks, 256, 0, stream, a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
  const long long warps = (long long)a.n_tokens * a.num_kv_heads * 2;
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  switch (a.head_dim) {
    case 64: return launch_pdl(append_kernel<64>, blocks, 256, 0, stream, a);
    case 128: return launch_pdl(append_kernel<128>, blocks, 256, 0, stream, a);
    case 256: return launch_pdl(append_kernel<256>, blocks, 256, 0, stream, a);
    case 576: return launch_pdl(append_kernel<576>, blocks, 256, 0, stream, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
