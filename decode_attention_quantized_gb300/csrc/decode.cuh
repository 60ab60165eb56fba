// decode.cuh -- split-KV flash-decoding over a quantized paged KV cache.
//
// What it computes (one query row = (b, draft t, query head i), kv head
// h = i / G): logits s_j = sm_scale * <q, dequant(k_j)> for the keys the row
// sees, optional softcap, softmax, o = sum_j p_j dequant(v_j) / sum_j p_j.
// Sources: PagedAttention paged decode (onnxruntime PR #29912, Summary of
// Changes: split-KV, block-table aware, softcap, sliding window, on-the-fly
// dequantization); kv-quant-attn page, section "Method" (one block owns a
// (batch, kv head) pair and resolves every query head of the GQA group from
// one read; warps keep private (max, sumexp, accumulator) state with no
// barrier or atomic in the loop; partials merged in a fixed order); per-channel
// K scale folded into Q with a power-of-two normaliser (onnxruntime PR #32515,
// Description: the fold is exact, the normaliser keeps |q*s| <= |q|).
//
// Structure (one persistent CTA per SM slot):
//  * every CTA builds the same split plan from seq_lens in shared memory: the
//    (sequence, kv head) key ranges laid end to end in 64-key tiles, cut into
//    one equal slice per CTA; a piece of a range inside a slice is a split;
//  * one producer warp streams each unit's pages through a ring of shared
//    memory stages: TMA tensor copies (cp.async.bulk.tensor, 128/64/32-byte
//    swizzle) of the K and V code rows, the block id taken from the block
//    table as the copy's outer coordinate, plus 1-D bulk copies of per-row
//    scales; completion is counted on an mbarrier per stage;
//  * consumer warps (key warps x row groups of 8 query rows) take 16-key
//    sub-tiles: QK^T on tensor cores with keys as MMA-M and query rows as
//    MMA-N (ldmatrix of the codes, exact in-register code->f16 conversion),
//    online softmax in fp32, P moved into the PV operand layout with
//    movmatrix, PV with channels as MMA-M (ldmatrix.trans of the V codes);
//  * at the end of a unit the key warps of a row group merge their states
//    in a fixed chain through one shared slot and the last one writes the
//    unit's partial (base-2 log-sum-exp, normalized output) to the workspace.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "kvq_internal.h"
#include "pipeline.cuh"
#include "ptx.cuh"

namespace kvq {

namespace dev {

// Smallest e with 2^e >= x for finite x > 0 (read off the IEEE fields).
__device__ __forceinline__ int ceil_log2(float x) {
  const uint32_t u = __float_as_uint(x);
  int e = (int)((u >> 23) & 0xFFu) - 127;
  if (u & 0x7FFFFFu) e += 1;
  return e;
}

// r / G for 0 <= r < 2^16 and 1 <= G <= 64, given inv = fl(1/G): without an
// integer divide (a long dependent sequence on this GPU).  (r + 0.5) / G is at
// least 0.5 / G >= 2^-7 away from an integer, while the two roundings below
// move it by at most (r + 0.5) / G * 2^-23 < 2^-7, so the floor is exact.
__device__ __forceinline__ int div_small(int r, float inv) {
  return (int)(((float)r + 0.5f) * inv);
}

// 2^e for e in [-126, 127], exact.
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float((uint32_t)(e + 127) << 23); }

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Exact code -> f16 conversions producing MMA operand pairs (low half first).
// int8: bytes i, j of x = w ^ 0x80808080 placed under exponent byte 0x64
// (1024 + code + 128), minus 1152.
__device__ __forceinline__ uint32_t i8pair(uint32_t x, uint32_t sel) {
  return ptx::hsub2_u32(ptx::prmt(x, 0x64646464u, sel), 0x64806480u);
}
// int4: nibbles n, n+4 of x = w ^ 0x88888888 (shift = 4n) as 1024 + code + 8,
// minus 1032.
__device__ __forceinline__ uint32_t i4pair(uint32_t x, int shift) {
  return ptx::hsub2_u32(((x >> shift) & 0x000F000Fu) | 0x64006400u, 0x64086408u);
}
// e4m3: byte b = s.eeee.mmm moved to bits 15..8 of a half, then sign kept
// and eeee.mmm shifted right by one: exactly the f16 value b * 2^-8
// (subnormals included; the tensor-memory kernel's V path, which applies the
// 2^8 at its output).
__device__ __forceinline__ uint32_t f8pair(uint32_t w, uint32_t sel) {
  const uint32_t y = ptx::prmt(w, 0u, sel);
  return (y & 0x80008000u) | ((y >> 1) & 0x3F803F80u);
}

// e4m3 pair (bytes selected by sel into a 16-bit word) -> exact f16x2 by the
// hardware conversion.  kClamp: then max with -448 so that a NaN code (a
// stale byte past the sequence end, under a masked key) becomes finite.
template <bool kClamp = true>
__device__ __forceinline__ uint32_t f8cvt(uint32_t w, uint32_t sel) {
  const uint32_t x = ptx::prmt(w, 0u, sel);
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)(x & 0xFFFFu)));
  if constexpr (!kClamp) return d;
  uint32_t r;
  asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(d), "r"(0xDF00DF00u));
  return r;
}

template <bool B>
struct Flag {
  static constexpr bool value = B;
};

// tanh(x) = 1 - 2 / (e^{2x} + 1), from the definition; absolute error a few
// 1e-7 (ex2.approx and an approximate divide), saturating to +-1.
__device__ __forceinline__ float tanh_fast(float x) {
  return 1.0f - __fdividef(2.0f, ptx::fast_exp2(x * 2.8853900817779268f) + 1.0f);
}

// Exact e4m3x2 -> f16x2 (hardware conversion; the low byte goes to the low
// half).  Used for K only: a stale e4m3 NaN byte under a masked key can then
// only poison that key's own score, which the mask replaces.
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint16_t v) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
  return d;
}

// A fragment (keys x k-slots) of k-step t of a 16-byte code chunk for QK,
// from the ldmatrix words of keys g (wl) and g + 8 (wh), every code converted
// exactly (a zero code must give an exactly zero product whatever the scale).
template <int DT>
__device__ __forceinline__ void k_frag(uint32_t wl, uint32_t wh, int t, uint32_t (&A)[4]) {
  if constexpr (DT == KVQ_INT4) {
    const uint32_t xl = wl ^ 0x88888888u, xh = wh ^ 0x88888888u;
    A[0] = i4pair(xl, 8 * t);
    A[1] = i4pair(xh, 8 * t);
    A[2] = i4pair(xl, 8 * t + 4);
    A[3] = i4pair(xh, 8 * t + 4);
  } else if constexpr (DT == KVQ_INT8) {
    const uint32_t xl = wl ^ 0x80808080u, xh = wh ^ 0x80808080u;
    A[0] = i8pair(xl, 0x4140u);
    A[1] = i8pair(xh, 0x4140u);
    A[2] = i8pair(xl, 0x4342u);
    A[3] = i8pair(xh, 0x4342u);
  } else {
    A[0] = e4m3x2_f16x2((uint16_t)(wl & 0xFFFFu));
    A[1] = e4m3x2_f16x2((uint16_t)(wh & 0xFFFFu));
    A[2] = e4m3x2_f16x2((uint16_t)(wl >> 16));
    A[3] = e4m3x2_f16x2((uint16_t)(wh >> 16));
  }
}

// Output channel held by accumulator element e of channel tile mt in lane
// group g (the PV operand permutation chosen for the ldmatrix.trans layout).
template <int DT>
__device__ __forceinline__ int out_channel(int mt, int e, int g) {
  if constexpr (DT == KVQ_INT4)
    return 32 * (mt >> 1) + 4 * g + 2 * (mt & 1) + (e >> 1);
  else
    return 16 * mt + 2 * g + (e >> 1);
}

// Q operand of one query row rq (of the (b, h) work piece) for lane group c:
// the lane's channels in the MMA B-fragment permutation, per-channel K scale
// folded in under a power-of-two normaliser (|q * s| <= |q|), the row then
// normalised by the power of two just above its max so the f16 operand keeps
// its full mantissa.  Returns the logit factor for the row (sm_scale, tensor
// scale, both powers of two; times log2 e when no softcap follows),
// clamped to FLT_MAX so zero codes under a huge scale stay zero.  Rows past
// a.rows get q = 0.  Every lane of the warp must call it.
template <int DT, int D>
__device__ __forceinline__ float q_prologue(const DecodeArgs& a, int rq, int b, int h, int c,
                                            uint32_t (&qf)[D / 16][2]) {
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr int CPL = (DT == KVQ_INT4) ? 8 : 4;  // channels per 16-byte code chunk per lane
  constexpr int NQC = D / (4 * CPL);             // code chunks per row
  const int G = a.group, T = a.q_tokens, Hq = a.num_q_heads;
  const bool qvalid = rq < a.rows;
  const int tq = qvalid ? div_small(rq, __frcp_rn((float)G)) : 0, gq = qvalid ? rq - tq * G : 0;
  const uint16_t* qp = a.q + (((size_t)b * T + tq) * Hq + (size_t)h * G + gq) * D;
  float qv[NQC][CPL];
#pragma unroll
  for (int j = 0; j < NQC; ++j) {
    const int ch0 = j * 4 * CPL + c * CPL;
    if constexpr (CPL == 8) {
      const uint4 w = qvalid ? *reinterpret_cast<const uint4*>(qp + ch0) : make_uint4(0, 0, 0, 0);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qv[j][2 * i] = __uint_as_float(ww[i] << 16);
        qv[j][2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
      }
    } else {
      const uint2 w = qvalid ? *reinterpret_cast<const uint2*>(qp + ch0) : make_uint2(0, 0);
      qv[j][0] = __uint_as_float(w.x << 16);
      qv[j][1] = __uint_as_float(w.x & 0xFFFF0000u);
      qv[j][2] = __uint_as_float(w.y << 16);
      qv[j][3] = __uint_as_float(w.y & 0xFFFF0000u);
    }
  }
  int e_tot = 0;
  if (a.k_mode == KVQ_SCALE_PER_CHANNEL) {
    const float* ks = a.k_scale + (size_t)h * D;
    float km = 0.0f;
#pragma unroll
    for (int j = 0; j < NQC; ++j)
#pragma unroll
      for (int i = 0; i < CPL; ++i) km = fmaxf(km, fabsf(ks[j * 4 * CPL + c * CPL + i]));
    km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, 1));
    km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, 2));
    const int ek = km > 0.0f ? min(126, max(-126, ceil_log2(km))) : 0;
    const float sk = pow2i(-ek);
#pragma unroll
    for (int j = 0; j < NQC; ++j)
#pragma unroll
      for (int i = 0; i < CPL; ++i) qv[j][i] *= ks[j * 4 * CPL + c * CPL + i] * sk;
    e_tot += ek;
  }
  float qm = 0.0f;
#pragma unroll
  for (int j = 0; j < NQC; ++j)
#pragma unroll
    for (int i = 0; i < CPL; ++i) qm = fmaxf(qm, fabsf(qv[j][i]));
  qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, 1));
  qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, 2));
  const int eq = qm > 0.0f ? min(126, max(-126, ceil_log2(qm))) : 0;
  const float sq = pow2i(-eq);
  e_tot += eq;
#pragma unroll
  for (int j = 0; j < NQC; ++j) {
    if constexpr (DT == KVQ_INT4) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        qf[2 * j + t][0] = pack_h2(qv[j][2 * t] * sq, qv[j][2 * t + 4] * sq);
        qf[2 * j + t][1] = pack_h2(qv[j][2 * t + 1] * sq, qv[j][2 * t + 5] * sq);
      }
    } else {
      qf[j][0] = pack_h2(qv[j][0] * sq, qv[j][1] * sq);
      qf[j][1] = pack_h2(qv[j][2] * sq, qv[j][3] * sq);
    }
  }
  float base = a.sm_scale;
  if (a.k_mode == KVQ_SCALE_PER_TENSOR) base *= a.k_scale[0];
  float alpha = ldexpf(base, e_tot);
  if (a.softcap <= 0.0f) alpha *= kLog2e;
  return fminf(alpha, 3.4028234e38f);
}

}  // namespace dev

// Shared floats of the wide consumer layout with NT n-tiles per row half: the
// P buffer ([16 NT rows][64 keys] f16 = 16 NT x 32 floats), per-quarter row
// maxima and row sums ([4][16 NT] each), per-quarter V-scale maxima (+ pad to
// 32), the Q operand ([16 NT rows][D] f16) and the rows' logit factors (+ pad).
template <int NT, int D>
__host__ __device__ constexpr int wide_scratch_floats() {
  return NT > 0 ? 16 * NT * 32 + 2 * 4 * 16 * NT + 32 + 16 * NT * (D / 2) + ((16 * NT + 31) / 32) * 32 : 0;
}

// GS > 0: the grouped layout with the per-group scale paths for groups of GS
// channels compiled in (a kernel of its own per group size, so that its
// group boundaries are compile-time and the other modes carry none of it).
template <int DT, int D, int MINB, int NT, int GS>
__global__ void __launch_bounds__(288, MINB)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
  using Gm = Geo<DT, D>;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* ring = smem_raw + pad;

  const int n_cw = a.row_groups * a.key_warps;
  constexpr int kScrPerRg = (Gm::NMT * 4 + 4) * 32;  // floats: accumulators + (m, l) of one warp, [elem][lane]
  float* scr = reinterpret_cast<float*>(ring + (size_t)a.stages * a.stage_stride);
  const int scr_floats =
      NT > 0 ? wide_scratch_floats<NT, D>() : (a.key_warps > 1 ? a.row_groups * kScrPerRg : 0);
  int* pl_pre = reinterpret_cast<int*>(scr + scr_floats);  // [B + 1]
  int* pl_misc = pl_pre + a.batch + 1;                     // [4]
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(pl_misc + 4 + ((a.batch + 5) & 1));
  uint64_t* bar_empty = bar_full + a.stages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.q_tokens;

  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      ptx::mbar_init(&bar_full[s], 1);
      ptx::mbar_init(&bar_empty[s], (uint32_t)n_cw);
    }
    ptx::fence_mbar_init();
  }
  // With early reads (KVQ_DECODE_EARLY_INPUTS) the inputs the caller vouches
  // for (seq_lens, block table, q, static scales) are read before the wait on
  // the preceding grid on the stream: the producer waits before its first
  // cache read and the consumers before their first workspace write, so the
  // plan, the first block ids and the Q prologue overlap that grid's tail.
  // Without them build_slice waits first.
  const Slice<kTile> sp = build_slice<kTile>(a, pl_pre, pl_misc);
  const int t_begin = sp.t_begin, t_end = sp.t_end;
  auto piece = [&](int gt, int& b, int& h, int& k0, int& k1, int& L, int& slot, int& next) {
    sp.piece(a, gt, b, h, k0, k1, L, slot, next);
  };

  const bool k_row = a.k_mode == KVQ_SCALE_PER_ROW, v_row = a.v_mode == KVQ_SCALE_PER_ROW;

  // =============================================================== producer
  if (warp == n_cw) {
    produce<Gm, true>(a, sp, &tmk, &tmv, ring, bar_full, bar_empty, pl_pre, pl_misc);
    return;
  }

  if constexpr (NT > 0) {
    // ======================================================= wide consumers
    // For many query rows (17..48: drafts x GQA group).  8 warps = 4 key
    // quarters kq x 2 row halves rh of NT x 8 rows.  QK: warp (kq, rh) scores
    // keys [16 kq, 16 kq + 16) of each tile against its rows (each code is
    // converted by 2 warps, not by every row group); the per-row tile maxima
    // meet in shared memory so every warp applies the same running maximum;
    // P goes to a swizzled shared buffer; PV: warp (kq, rh) accumulates
    // channel quarter kq of its rows over all 64 keys.  The warps' outputs are
    // disjoint, so the end of a piece only sums the row sums.
    constexpr int RW = NT * 8, ROWS = 2 * RW;
    constexpr int QCH = Gm::NCH / 4;                     // code chunks of a channel quarter
    constexpr int MTW = (DT == KVQ_INT4 ? 2 : 1) * QCH;  // 16-channel tiles of a quarter
    float* s_max = scr + ROWS * 32;                      // [4][ROWS]
    float* s_l = s_max + 4 * ROWS;                       // [4][ROWS]
    float* s_vmax = s_l + 4 * ROWS;                      // [4]
    const uint32_t p_base = ptx::smem_u32(scr);          // P: [ROWS][64 keys] f16, 128-byte rows
    float* s_q = s_vmax + 32;                            // Q: [ROWS][D] f16 in MMA k-slot order
    const uint32_t q_base = ptx::smem_u32(s_q);
    float* s_alpha = s_q + ROWS * (D / 2);               // [ROWS] logit factors
    const int rh = warp & 1, kq = warp >> 1;
    // a row half past the unit's rows (8 or fewer rows: head_dim 576 with
    // few query heads) converts no codes and runs no MMAs; its warps still
    // meet the others at every barrier
    const bool idle = rh * RW >= a.rows;
    const int g = lane >> 2, c = lane & 3;
    const int G = a.group, W = a.window;
    const float inv_g = __frcp_rn((float)G);  // r / G by dev::div_small
    const float softcap = a.softcap;
    const float inv_cap = softcap > 0.0f ? 1.0f / softcap : 0.0f;
    const int ld_key = ((lane >> 3) & 1) * 8 + (lane & 7);
    const int ld_chunk = lane >> 4;
    // byte offset of P[row][key]: the 16-byte chunk index XOR (row & 7)
    auto p_off = [](int row, int key) -> uint32_t {
      return (uint32_t)(row * 128 + ((((key >> 3) ^ row) & 7) << 4) + (key & 7) * 2);
    };
    // byte offset of Q[row][k] (k = 16 * k-step + slot): 2D-byte rows, the
    // low three bits of the 16-byte chunk index XOR (row & 7)
    auto q_off = [](int row, int k) -> uint32_t {
      return (uint32_t)(row * 2 * D + ((((k >> 3) & ~7) | (((k >> 3) ^ row) & 7)) << 4) + (k & 7) * 2);
    };
    uint32_t it = 0;
    RingPos rp;
    bool ok = true;
    for (int gt = t_begin, next; gt < t_end; gt = next) {
      int b, h, k0, k1, L, u;
      piece(gt, b, h, k0, k1, L, u, next);
      // Q of n-tile kq of this half (warps kq < NT), stored in k-slot order so
      // that ldmatrix yields the B fragments; the rows' logit factors beside it
      if constexpr (D <= 256) {
        if (kq < NT) {
          const int row = rh * RW + kq * 8 + g;
          uint32_t qf[Gm::NMT][2];
          const float ag = dev::q_prologue<DT, D>(a, row, b, h, c, qf);
#pragma unroll
          for (int ks = 0; ks < Gm::NMT; ++ks) {
            ptx::st_shared_u32(q_base + q_off(row, ks * 16 + 2 * c), qf[ks][0]);
            ptx::st_shared_u32(q_base + q_off(row, ks * 16 + 8 + 2 * c), qf[ks][1]);
          }
          if (c == 0) s_alpha[row] = ag;
        }
      } else {
        // long rows: every warp takes k-step quarter kq of each row of its half
        // (the rows' maxima and the per-channel scales' maximum meet in shared
        // memory), the same arithmetic as q_prologue: q * (k_scale / 2^ek),
        // then / 2^eq, to f16 in the k-slot order
        static_assert(DT != KVQ_INT4, "8-bit codes");
        constexpr int KQ = D / 64;  // k-steps of a quarter
        const bool kc = a.k_mode == KVQ_SCALE_PER_CHANNEL;
        const float* ksp = a.k_scale + (size_t)h * D;
        auto row_ptr = [&](int r) {
          const int tq = dev::div_small(r, inv_g), gq = r - tq * G;
          return a.q + (((size_t)b * T + tq) * a.num_q_heads + (size_t)h * G + gq) * D;
        };
        auto load4 = [&](const uint16_t* qp, int j, float (&v)[4]) {
          const uint2 w = *reinterpret_cast<const uint2*>(qp + 16 * j + 4 * c);
          v[0] = __uint_as_float(w.x << 16);
          v[1] = __uint_as_float(w.x & 0xFFFF0000u);
          v[2] = __uint_as_float(w.y << 16);
          v[3] = __uint_as_float(w.y & 0xFFFF0000u);
        };
        float km = 0.0f;
        if (kc) {
#pragma unroll 3
          for (int j = kq * KQ; j < (kq + 1) * KQ; ++j)
#pragma unroll
            for (int i = 0; i < 4; ++i) km = fmaxf(km, fabsf(ksp[16 * j + 4 * c + i]));
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int r = rh * RW + nt * 8 + g;
          float m = 0.0f;
          if (r < a.rows) {
            const uint16_t* qp = row_ptr(r);
#pragma unroll 3
            for (int j = kq * KQ; j < (kq + 1) * KQ; ++j) {
              float v[4];
              load4(qp, j, v);
#pragma unroll
              for (int i = 0; i < 4; ++i) m = fmaxf(m, fabsf(kc ? v[i] * ksp[16 * j + 4 * c + i] : v[i]));
            }
          }
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
          m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
          if (c == 0) s_max[kq * ROWS + r] = m;
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
        if (lane == 0) s_vmax[warp] = km;  // eight slots
        ptx::named_bar_sync(1, 8 * 32);
        int ek = 0;
        if (kc) {
          float kmax = s_vmax[0];
#pragma unroll
          for (int w = 1; w < 8; ++w) kmax = fmaxf(kmax, s_vmax[w]);
          ek = kmax > 0.0f ? min(126, max(-126, dev::ceil_log2(kmax))) : 0;
        }
        const float sk = dev::pow2i(-ek);
        float base = a.sm_scale;
        if (a.k_mode == KVQ_SCALE_PER_TENSOR) base *= a.k_scale[0];
        if (softcap <= 0.0f) base *= kLog2e;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int r = rh * RW + nt * 8 + g;
          // (the quarters' maxima are of q * k_scale; times 2^-ek exactly)
          const float qm = fmaxf(fmaxf(s_max[r], s_max[ROWS + r]), fmaxf(s_max[2 * ROWS + r], s_max[3 * ROWS + r])) * sk;
          const int eq = qm > 0.0f ? min(126, max(-126, dev::ceil_log2(qm))) : 0;
          const float sq = dev::pow2i(-eq);
          const uint16_t* qp = row_ptr(r < a.rows ? r : 0);
#pragma unroll 3
          for (int j = kq * KQ; j < (kq + 1) * KQ; ++j) {
            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (r < a.rows) load4(qp, j, v);
            if (kc) {
#pragma unroll
              for (int i = 0; i < 4; ++i) v[i] *= ksp[16 * j + 4 * c + i] * sk;
            }
            ptx::st_shared_u32(q_base + q_off(r, 16 * j + 2 * c), dev::pack_h2(v[0] * sq, v[1] * sq));
            ptx::st_shared_u32(q_base + q_off(r, 16 * j + 8 + 2 * c), dev::pack_h2(v[2] * sq, v[3] * sq));
          }
          if (kq == 0 && c == 0) {
            float alpha = ldexpf(base, ek + eq);
            s_alpha[r] = fminf(alpha, 3.4028234e38f);
          }
        }
      }
      ptx::named_bar_sync(1, 8 * 32);
      float al[NT][2], m[NT][2], l[NT][2];
      int pos[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = rh * RW + nt * 8 + 2 * c + i;
          al[nt][i] = s_alpha[r];
          pos[nt][i] = r < a.rows ? L - T + dev::div_small(r, inv_g) : -1;
          m[nt][i] = -INFINITY;
          l[nt][i] = 0.0f;
        }
      }
      int F = v_row ? -126 : 0;  // V-scale normaliser exponent, the same in every warp
      float acc[MTW][NT][4];
#pragma unroll
      for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.0f;

      for (int key0 = k0; key0 < k1; key0 += kTile, ++it, rp.next(a.stages)) {
        const int stage = (int)rp.stage;
        if (ok) {
          ok = ptx::mbar_wait_bounded_inl(&bar_full[stage], rp.phase);
          if (!ok) atomicOr(a.err, KVQ_DEVERR_TIMEOUT);
        }
        const uint8_t* st = ring + (size_t)stage * a.stage_stride;
        const uint32_t sk_base = ptx::smem_u32(st);
        // LATENT (v_alias): V is the K codes and scales of the stage
        const uint32_t sv_base = sk_base + (a.v_alias ? 0 : Gm::CODE_BYTES);
        const float* ks_row = reinterpret_cast<const float*>(st + (a.v_alias ? 1 : 2) * Gm::CODE_BYTES);
        const float* vs_row = a.v_alias ? ks_row : ks_row + kTile;

        // ---- phase A: scores of this warp's 16 keys x NT n-tiles of rows
        const int kb = key0 + kq * kSub;
        const bool active = ok && kb < k1 && !idle;
        const int key_a = kb + g, key_b = key_a + 8;
        float x[NT][4];
        float vpa = 0.0f, vpb = 0.0f;
        if (active) {
          // long rows (head_dim 576: 36 k-steps) of one n-tile accumulate in
          // four independent chains, summed at the end, so the MMAs do not wait
          // on one another (with more n-tiles the extra registers spill)
          constexpr int NCHAIN = D > 256 && NT == 1 ? 4 : 1;
          float sacc[NCHAIN][NT][4];
#pragma unroll
          for (int ch = 0; ch < NCHAIN; ++ch)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) sacc[ch][nt][0] = sacc[ch][nt][1] = sacc[ch][nt][2] = sacc[ch][nt][3] = 0.0f;
          const uint32_t row_off = (uint32_t)(kq * kSub + ld_key) * Gm::SPAN;
          // B fragments of k-step ks for every n-tile of this half, from Q
          auto qfrag = [&](int ks, uint32_t (&bq)[NT][2]) {
            const int mi = lane >> 3;
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
              const int row = rh * RW + (2 * np + (mi >> 1)) * 8 + (lane & 7);
              uint32_t R[4];
              ptx::ldmatrix_x4(R, q_base + q_off(row, ks * 16 + (mi & 1) * 8));
              bq[2 * np][0] = R[0];
              bq[2 * np][1] = R[1];
              bq[2 * np + 1][0] = R[2];
              bq[2 * np + 1][1] = R[3];
            }
            if constexpr (NT % 2 == 1) {
              const int row = rh * RW + (NT - 1) * 8 + (lane & 7);
              uint32_t R[2];
              ptx::ldmatrix_x2(R, q_base + q_off(row, ks * 16 + (mi & 1) * 8));
              bq[NT - 1][0] = R[0];
              bq[NT - 1][1] = R[1];
            }
          };
#pragma unroll
          for (int kk = 0; kk < Gm::NCH / 2; ++kk) {
            const uint32_t byte = (uint32_t)(2 * kk + ld_chunk) * 16;
            const uint32_t addr =
                sk_base + (byte / Gm::SPAN) * (kTile * Gm::SPAN) + dev::swz<Gm::SPAN>(row_off + byte % Gm::SPAN);
            uint32_t R[4];
            ptx::ldmatrix_x4(R, addr);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int j = 2 * kk + h2;
              const uint32_t wl = R[2 * h2], wh = R[2 * h2 + 1];
              if constexpr (DT == KVQ_INT4) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                  uint32_t A[4];
                  dev::k_frag<DT>(wl, wh, t, A);
                  uint32_t bq[NT][2];
                  qfrag(2 * j + t, bq);
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt) ptx::mma_16816(sacc[0][nt], A, bq[nt][0], bq[nt][1]);
                }
              } else {
                uint32_t A[4];
                dev::k_frag<DT>(wl, wh, 0, A);
                uint32_t bq[NT][2];
                qfrag(j, bq);
                constexpr int chain = NCHAIN > 1 ? 1 : 0;  // (kk & 1) * 2 + h2 below when chained
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  ptx::mma_16816(sacc[chain ? ((kk & 1) * 2 + h2) % NCHAIN : 0][nt], A, bq[nt][0], bq[nt][1]);
              }
            }
          }
#pragma unroll
          for (int ch = 1; ch < NCHAIN; ++ch)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int e = 0; e < 4; ++e) sacc[0][nt][e] += sacc[ch][nt][e];
          float ksa = 1.0f, ksb = 1.0f;
          if (k_row) {
            ksa = ks_row[kq * kSub + g];
            ksb = ks_row[kq * kSub + g + 8];
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            x[nt][0] = sacc[0][nt][0] * al[nt][0] * ksa;
            x[nt][1] = sacc[0][nt][1] * al[nt][1] * ksa;
            x[nt][2] = sacc[0][nt][2] * al[nt][0] * ksb;
            x[nt][3] = sacc[0][nt][3] * al[nt][1] * ksb;
            if (softcap > 0.0f) {
#pragma unroll
              for (int e = 0; e < 4; ++e) x[nt][e] = softcap * dev::tanh_fast(x[nt][e] * inv_cap) * kLog2e;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = e < 2 ? key_a : key_b, p = pos[nt][e & 1];
              if (!(key <= p && (W == 0 || key > p - W))) x[nt][e] = -INFINITY;
            }
          }
          if (v_row) {
            vpa = key_a < L ? vs_row[kq * kSub + g] : 0.0f;
            vpb = key_b < L ? vs_row[kq * kSub + g + 8] : 0.0f;
          }
        } else {
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) x[nt][0] = x[nt][1] = x[nt][2] = x[nt][3] = -INFINITY;
        }
        // this warp's per-row maxima over its 16 keys, and its V-scale maximum
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            float t = fmaxf(x[nt][i], x[nt][i + 2]);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
            if (g == 0) s_max[kq * ROWS + rh * RW + nt * 8 + 2 * c + i] = t;
          }
        }
        if (v_row) {
          float vm = fmaxf(vpa, vpb);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
          if (rh == 0 && lane == 0) s_vmax[kq] = vm;
        }
        ptx::named_bar_sync(1, 8 * 32);

        // ---- phase B: the running maximum of every row over the 4 quarters
        float mu[NT][2], corr[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int row = rh * RW + nt * 8 + 2 * c + i;
            float tm = s_max[row];
#pragma unroll
            for (int q = 1; q < 4; ++q) tm = fmaxf(tm, s_max[q * ROWS + row]);
            const float mn = fmaxf(m[nt][i], tm);
            mu[nt][i] = mn == -INFINITY ? 0.0f : mn;
            corr[nt][i] = ptx::fast_exp2(m[nt][i] - mu[nt][i]);
            m[nt][i] = mn;
          }
        }
        float fs = 1.0f, inv = 1.0f;
        if (v_row) {
          const float vm = fmaxf(fmaxf(s_vmax[0], s_vmax[1]), fmaxf(s_vmax[2], s_vmax[3]));
          if (vm > 0.0f) {
            const int fn = min(126, max(-126, dev::ceil_log2(vm)));
            if (fn > F) {
              fs = (F - fn < -126) ? 0.0f : dev::pow2i(F - fn);
              F = fn;
            }
          }
          inv = dev::pow2i(-F);
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float p0 = ptx::fast_exp2(x[nt][0] - mu[nt][0]), p1 = ptx::fast_exp2(x[nt][1] - mu[nt][1]);
          const float p2 = ptx::fast_exp2(x[nt][2] - mu[nt][0]), p3 = ptx::fast_exp2(x[nt][3] - mu[nt][1]);
          l[nt][0] = l[nt][0] * corr[nt][0] + p0 + p2;
          l[nt][1] = l[nt][1] * corr[nt][1] + p1 + p3;
          if (active) {
            const float va = v_row ? vpa * inv : 1.0f, vb = v_row ? vpb * inv : 1.0f;
            // (keys x rows) -> (row g; keys 2c, 2c+1) of each 8-key half
            const uint32_t y0 = ptx::movmatrix_trans(dev::pack_h2(p0 * va, p1 * va));
            const uint32_t y1 = ptx::movmatrix_trans(dev::pack_h2(p2 * vb, p3 * vb));
            const int row = rh * RW + nt * 8 + g;
            ptx::st_shared_u32(p_base + p_off(row, kq * kSub + 2 * c), y0);
            ptx::st_shared_u32(p_base + p_off(row, kq * kSub + 8 + 2 * c), y1);
          }
        }
        {
          bool one = fs == 1.0f;
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) one = one && corr[nt][0] == 1.0f && corr[nt][1] == 1.0f;
          if (!__all_sync(0xffffffffu, one)) {
#pragma unroll
            for (int mt = 0; mt < MTW; ++mt)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                acc[mt][nt][0] *= corr[nt][0] * fs;
                acc[mt][nt][1] *= corr[nt][1] * fs;
                acc[mt][nt][2] *= corr[nt][0] * fs;
                acc[mt][nt][3] *= corr[nt][1] * fs;
              }
          }
        }
        ptx::named_bar_sync(1, 8 * 32);

        // ---- phase C: channel quarter kq of this half's rows over the tile
        for (int kg = 0; ok && !idle && kg < kTile / kSub; ++kg) {
          if (key0 + kg * kSub >= k1) break;  // that quarter wrote no P this tile
          uint32_t pb[NT][2];
          {
            const int mi = lane >> 3;  // x4: (n-tile pair, key half)
#pragma unroll
            for (int np = 0; np < NT / 2; ++np) {
              const int row = rh * RW + (2 * np + (mi >> 1)) * 8 + (lane & 7);
              uint32_t R[4];
              ptx::ldmatrix_x4(R, p_base + p_off(row, kg * kSub + (mi & 1) * 8));
              pb[2 * np][0] = R[0];
              pb[2 * np][1] = R[1];
              pb[2 * np + 1][0] = R[2];
              pb[2 * np + 1][1] = R[3];
            }
            if constexpr (NT % 2 == 1) {
              const int row = rh * RW + (NT - 1) * 8 + (lane & 7);
              uint32_t R[2];
              ptx::ldmatrix_x2(R, p_base + p_off(row, kg * kSub + (mi & 1) * 8));
              pb[NT - 1][0] = R[0];
              pb[NT - 1][1] = R[1];
            }
          }
          const uint32_t vrow_off = (uint32_t)(kg * kSub + ld_key) * Gm::SPAN;
#pragma unroll
          for (int jj = 0; jj < QCH / 2; ++jj) {
            const uint32_t byte = (uint32_t)(QCH * kq + 2 * jj + ld_chunk) * 16;
            const uint32_t addr =
                sv_base + (byte / Gm::SPAN) * (kTile * Gm::SPAN) + dev::swz<Gm::SPAN>(vrow_off + byte % Gm::SPAN);
            uint32_t R[4];
            ptx::ldmatrix_x4_trans(R, addr);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int jl = 2 * jj + h2;
              const uint32_t wl = R[2 * h2], wh = R[2 * h2 + 1];
              if constexpr (DT == KVQ_INT4) {
                const uint32_t xl = wl ^ 0x88888888u, xh = wh ^ 0x88888888u;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                  const uint32_t A[4] = {dev::i4pair(xl, 8 * t), dev::i4pair(xl, 8 * t + 4),
                                         dev::i4pair(xh, 8 * t), dev::i4pair(xh, 8 * t + 4)};
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt) ptx::mma_16816(acc[2 * jl + t][nt], A, pb[nt][0], pb[nt][1]);
                }
              } else {
                uint32_t A[4];
                if constexpr (DT == KVQ_INT8) {
                  const uint32_t xl = wl ^ 0x80808080u, xh = wh ^ 0x80808080u;
                  A[0] = dev::i8pair(xl, 0x4240u);
                  A[1] = dev::i8pair(xl, 0x4341u);
                  A[2] = dev::i8pair(xh, 0x4240u);
                  A[3] = dev::i8pair(xh, 0x4341u);
                } else {
                  A[0] = dev::f8cvt(wl, 0x0020u);
                  A[1] = dev::f8cvt(wl, 0x0031u);
                  A[2] = dev::f8cvt(wh, 0x0020u);
                  A[3] = dev::f8cvt(wh, 0x0031u);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) ptx::mma_16816(acc[jl][nt], A, pb[nt][0], pb[nt][1]);
              }
            }
          }
          if constexpr (QCH % 2 == 1) {
            // an odd last chunk of the quarter (head_dim 576: nine per quarter):
            // keys 0-7 and 8-15 of one chunk by a two-matrix load (lanes 0-15
            // give the row addresses)
            static_assert(DT != KVQ_INT4, "odd quarters only with 8-bit codes");
            constexpr int jl = QCH - 1;
            const uint32_t byte = (uint32_t)(QCH * kq + jl) * 16;
            const uint32_t addr =
                sv_base + (byte / Gm::SPAN) * (kTile * Gm::SPAN) + dev::swz<Gm::SPAN>(vrow_off + byte % Gm::SPAN);
            uint32_t R[2];
            ptx::ldmatrix_x2_trans(R, addr);
            uint32_t A[4];
            if constexpr (DT == KVQ_INT8) {
              const uint32_t xl = R[0] ^ 0x80808080u, xh = R[1] ^ 0x80808080u;
              A[0] = dev::i8pair(xl, 0x4240u);
              A[1] = dev::i8pair(xl, 0x4341u);
              A[2] = dev::i8pair(xh, 0x4240u);
              A[3] = dev::i8pair(xh, 0x4341u);
            } else {
              A[0] = dev::f8cvt(R[0], 0x0020u);
              A[1] = dev::f8cvt(R[0], 0x0031u);
              A[2] = dev::f8cvt(R[1], 0x0020u);
              A[3] = dev::f8cvt(R[1], 0x0031u);
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) ptx::mma_16816(acc[jl][nt], A, pb[nt][0], pb[nt][1]);
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bar_empty[stage]);
      }

      // ---- piece end: row sums over the 4 quarters, then each warp writes its
      // (rows, channel quarter) block of the normalized partial
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          float v = l[nt][i];
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (g == 0) s_l[kq * ROWS + rh * RW + nt * 8 + 2 * c + i] = v;
        }
      ptx::named_bar_sync(1, 8 * 32);
      // the tiles above may run while the preceding grid finishes; the
      // workspace is written only after it (no-op after the first)
      ptx::griddep_wait();
      float to_true = v_row ? dev::pow2i(F) : 1.0f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int r0 = rh * RW + nt * 8 + 2 * c, r1 = r0 + 1;
        float lt[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int row = r0 + i;
          lt[i] = s_l[row] + s_l[ROWS + row];
          lt[i] += s_l[2 * ROWS + row];
          lt[i] += s_l[3 * ROWS + row];
        }
        const float f0 = lt[0] > 0.0f ? to_true / lt[0] : 0.0f, f1 = lt[1] > 0.0f ? to_true / lt[1] : 0.0f;
        float* o0 = a.part_o + ((size_t)u * a.rows + r0) * D;
        float* o1 = o0 + D;
#pragma unroll
        for (int mt = 0; mt < MTW; ++mt) {
          const int mtg = (DT == KVQ_INT4 ? 2 * QCH * kq : QCH * kq) + mt;
          const int ch = dev::out_channel<DT>(mtg, 0, g);
          if (r0 < a.rows) *reinterpret_cast<float2*>(o0 + ch) = make_float2(acc[mt][nt][0] * f0, acc[mt][nt][2] * f0);
          if (r1 < a.rows) *reinterpret_cast<float2*>(o1 + ch) = make_float2(acc[mt][nt][1] * f1, acc[mt][nt][3] * f1);
        }
        if (kq == 0 && g == 0) {
          if (r0 < a.rows) a.part_lse[(size_t)u * a.rows + r0] = lt[0] > 0.0f ? m[nt][0] + ptx::fast_log2(lt[0]) : -INFINITY;
          if (r1 < a.rows) a.part_lse[(size_t)u * a.rows + r1] = lt[1] > 0.0f ? m[nt][1] + ptx::fast_log2(lt[1]) : -INFINITY;
        }
      }
      ptx::named_bar_sync(1, 8 * 32);
    }
    return;
  }

  // ============================================ consumers, grouped layout
  const int cw = warp;
  const int rg = cw % a.row_groups, kw = cw / a.row_groups;
  const int g = lane >> 2, c = lane & 3;
  const int G = a.group, Hq = a.num_q_heads;
  const float softcap = a.softcap;
  const float inv_cap = softcap > 0.0f ? 1.0f / softcap : 0.0f;
  // ldmatrix row address of this lane: matrix (lane >> 3) covers keys
  // 0-7 / 8-15 of the sub-tile and the even / odd 16-byte chunk of a pair
  const int ld_key = ((lane >> 3) & 1) * 8 + (lane & 7);
  const int ld_chunk = lane >> 4;
  // group-wise scales: a group is GS channels, i.e. GS / CH code chunks of
  // CH channels (16-byte chunks: 16 int8 / e4m3 codes or 32 int4 codes)
  constexpr bool GRP = GS > 0;
  const bool k_grp = GRP && a.k_mode == KVQ_SCALE_PER_GROUP, v_grp = GRP && a.v_mode == KVQ_SCALE_PER_GROUP;
  const bool v_sc = v_row || v_grp;  // V scales enter P under the normaliser 2^F
  constexpr int gmask = GRP ? GS - 1 : 0, NG = GRP ? D / GS : 1;
  const int ngk = a.sk_n;
  constexpr int CH = DT == KVQ_INT4 ? 32 : 16;
  uint32_t it = 0;
  RingPos rp;
  bool ok = true;

  for (int gt = t_begin, next; gt < t_end; gt = next) {
    int b, h, k0, k1, L, u;
    piece(gt, b, h, k0, k1, L, u, next);

    // ---- Q prologue: this lane's channels of query row g of the row group
    uint32_t qf[Gm::NMT][2];
    const float alpha_g = dev::q_prologue<DT, D>(a, rg * 8 + g, b, h, c, qf);
    const int r0 = rg * 8 + 2 * c, r1 = r0 + 1;
    // with a softcap the row factors also carry 1/softcap (clamped to FLT_MAX
    // like the factors themselves, so zero codes keep zero scores), and the
    // capped log2-domain logit is cap_l2 * tanh(x)
    const float cf = softcap > 0.0f ? inv_cap : 1.0f;
    const float al0 = fminf(__shfl_sync(0xffffffffu, alpha_g, (2 * c) * 4) * cf, 3.4028234e38f);
    const float al1 = fminf(__shfl_sync(0xffffffffu, alpha_g, (2 * c + 1) * 4) * cf, 3.4028234e38f);
    const float cap_l2 = softcap * kLog2e;
    const float inv_g = __frcp_rn((float)G);
    const int pos0 = r0 < a.rows ? L - T + dev::div_small(r0, inv_g) : -1;
    const int pos1 = r1 < a.rows ? L - T + dev::div_small(r1, inv_g) : -1;
    const int W = a.window;

    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    int F = v_sc ? -126 : 0;  // V-scale normaliser exponent (warp uniform)
    float acc[Gm::NMT][4];
#pragma unroll
    for (int mt = 0; mt < Gm::NMT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;

    for (int key0 = k0; key0 < k1; key0 += kTile, ++it, rp.next(a.stages)) {
      // (the head_dim 128 group-scale instances keep the division: with the
      // counter their code ran at half speed)
      constexpr bool kDiv = GRP && D < 256;
      const int stage = kDiv ? (int)(it % (uint32_t)a.stages) : (int)rp.stage;
      if (ok) {
        ok = ptx::mbar_wait_bounded_inl(&bar_full[stage], kDiv ? (it / a.stages) & 1 : rp.phase);
        if (!ok) atomicOr(a.err, KVQ_DEVERR_TIMEOUT);
      }
      const uint8_t* st = ring + (size_t)stage * a.stage_stride;
      const uint32_t sk_base = ptx::smem_u32(st);
      // LATENT (v_alias): V is the K codes and scales of the stage
      const uint32_t sv_base = sk_base + (a.v_alias ? 0 : Gm::CODE_BYTES);
      const float* ks_row = reinterpret_cast<const float*>(st + (a.v_alias ? 1 : 2) * Gm::CODE_BYTES);
      const float* vs_row = a.v_alias ? ks_row : ks_row + kTile * (GRP && ngk > 1 ? ngk : 1);
      for (int sub = kw; ok && sub < kTile / kSub; sub += a.key_warps) {
        const int kb = key0 + sub * kSub;
        if (kb >= k1) break;
        const uint32_t row_off = (uint32_t)(sub * kSub + ld_key) * Gm::SPAN;

        // ---- S = K Q^T for 16 keys x 8 rows (keys are MMA-M).  Per-group K:
        // each group's partial dot product is scaled by its keys' group scales
        // into gx as soon as the group's last chunk is in.
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        float gx[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < Gm::NCH / 2; ++kk) {
          const uint32_t byte = (uint32_t)(2 * kk + ld_chunk) * 16;
          const uint32_t addr =
              sk_base + (byte / Gm::SPAN) * (kTile * Gm::SPAN) + dev::swz<Gm::SPAN>(row_off + byte % Gm::SPAN);
          uint32_t R[4];
          ptx::ldmatrix_x4(R, addr);
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            const int j = 2 * kk + h2;
            const uint32_t wl = R[2 * h2], wh = R[2 * h2 + 1];
            if constexpr (DT == KVQ_INT4) {
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                uint32_t A[4];
                dev::k_frag<DT>(wl, wh, t, A);
                if (t == 0)
                  ptx::mma_16816(sa, A, qf[2 * j + t][0], qf[2 * j + t][1]);
                else
                  ptx::mma_16816(sb, A, qf[2 * j + t][0], qf[2 * j + t][1]);
              }
            } else {
              uint32_t A[4];
              dev::k_frag<DT>(wl, wh, 0, A);
              if (h2 == 0)
                ptx::mma_16816(sa, A, qf[j][0], qf[j][1]);
              else
                ptx::mma_16816(sb, A, qf[j][0], qf[j][1]);
            }
            if (k_grp && (((j + 1) * CH) & gmask) == 0) {
              const int grp = (j + 1) * CH / (GRP ? GS : 1) - 1;
              const float ga = ks_row[(sub * kSub + g) * NG + grp];
              const float gb = ks_row[(sub * kSub + g + 8) * NG + grp];
              gx[0] = fmaf(sa[0] + sb[0], ga, gx[0]);
              gx[1] = fmaf(sa[1] + sb[1], ga, gx[1]);
              gx[2] = fmaf(sa[2] + sb[2], gb, gx[2]);
              gx[3] = fmaf(sa[3] + sb[3], gb, gx[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) sa[e] = sb[e] = 0.0f;
            }
          }
        }
        if (k_grp) {
#pragma unroll
          for (int e = 0; e < 4; ++e) sa[e] = gx[e];
        }

        // ---- logits: element e -> key kb + g (+8 for e >= 2), row 2c (+1 for odd e)
        const int key_a = kb + g, key_b = key_a + 8;
        float ksa = 1.0f, ksb = 1.0f;
        if (k_row) {
          ksa = ks_row[sub * kSub + g];
          ksb = ks_row[sub * kSub + g + 8];
        }
        float x[4] = {(sa[0] + sb[0]) * al0, (sa[1] + sb[1]) * al1, (sa[2] + sb[2]) * al0, (sa[3] + sb[3]) * al1};
        if (k_row) {
          x[0] *= ksa;
          x[1] *= ksa;
          x[2] *= ksb;
          x[3] *= ksb;
        }
        if (softcap > 0.0f) {
#pragma unroll
          for (int e = 0; e < 4; ++e) x[e] = cap_l2 * dev::tanh_fast(x[e]);
        }
        // a sub-tile whose keys every query position sees (below the first
        // draft, inside every row's window) needs no mask; padding rows then
        // keep finite scores, which only feed their own unwritten outputs
        if (!(kb + kSub - 1 <= L - T && (W == 0 || kb > L - 1 - W))) {
          const bool va0 = key_a <= pos0 && (W == 0 || key_a > pos0 - W);
          const bool va1 = key_a <= pos1 && (W == 0 || key_a > pos1 - W);
          const bool vb0 = key_b <= pos0 && (W == 0 || key_b > pos0 - W);
          const bool vb1 = key_b <= pos1 && (W == 0 || key_b > pos1 - W);
          x[0] = va0 ? x[0] : -INFINITY;
          x[1] = va1 ? x[1] : -INFINITY;
          x[2] = vb0 ? x[2] : -INFINITY;
          x[3] = vb1 ? x[3] : -INFINITY;
        }

        // ---- online softmax (rows 2c, 2c+1; reduce over the 8 key lanes) with
        // lazy reference maxima: m moves (to the exact running maximum) only
        // when a score of the sub-tile exceeds it by more than 8, so P <= 2^8
        // in f16 and most sub-tiles skip the reduction and the rescale
        float t0 = fmaxf(x[0], x[2]), t1 = fmaxf(x[1], x[3]);
        float c0 = 1.0f, c1 = 1.0f;
        if (__any_sync(0xffffffffu, t0 > m0 + 8.0f || t1 > m1 + 8.0f)) {
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, o));
            t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, o));
          }
          const float mn0 = fmaxf(m0, t0), mn1 = fmaxf(m1, t1);
          c0 = ptx::fast_exp2(m0 - (mn0 == -INFINITY ? 0.0f : mn0));
          c1 = ptx::fast_exp2(m1 - (mn1 == -INFINITY ? 0.0f : mn1));
          m0 = mn0;
          m1 = mn1;
        }
        const float mu0 = m0 == -INFINITY ? 0.0f : m0;
        const float mu1 = m1 == -INFINITY ? 0.0f : m1;
        const float p0 = ptx::fast_exp2(x[0] - mu0), p1 = ptx::fast_exp2(x[1] - mu1);
        const float p2 = ptx::fast_exp2(x[2] - mu0), p3 = ptx::fast_exp2(x[3] - mu1);
        l0 = l0 * c0 + p0 + p2;
        l1 = l1 * c1 + p1 + p3;

        // ---- per-row (per-group) V scales enter P (each channel group's P),
        // normalised by 2^F >= their maximum; keys past the sequence end get
        // scale 0 (their scale slots may hold anything)
        float vsa = 1.0f, vsb = 1.0f, fs = 1.0f, vinv = 1.0f;
        if (v_sc) {
          float ua = 0.0f, ub = 0.0f;
          if (GRP && v_grp) {
#pragma unroll
            for (int gi = 0; gi < NG; ++gi) {
              if (key_a < L) ua = fmaxf(ua, vs_row[(sub * kSub + g) * NG + gi]);
              if (key_b < L) ub = fmaxf(ub, vs_row[(sub * kSub + g + 8) * NG + gi]);
            }
          } else {
            ua = key_a < L ? vs_row[sub * kSub + g] : 0.0f;
            ub = key_b < L ? vs_row[sub * kSub + g + 8] : 0.0f;
          }
          float vm = fmaxf(ua, ub);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
          if (vm > 0.0f) {
            const int fn = min(126, max(-126, dev::ceil_log2(vm)));
            if (fn > F) {
              fs = (F - fn < -126) ? 0.0f : dev::pow2i(F - fn);
              F = fn;
            }
          }
          vinv = dev::pow2i(-F);
          vsa = ua * vinv;
          vsb = ub * vinv;
        }
        const float rs0 = c0 * fs, rs1 = c1 * fs;
        if (!__all_sync(0xffffffffu, rs0 == 1.0f && rs1 == 1.0f)) {
#pragma unroll
          for (int mt = 0; mt < Gm::NMT; ++mt) {
            acc[mt][0] *= rs0;
            acc[mt][1] *= rs1;
            acc[mt][2] *= rs0;
            acc[mt][3] *= rs1;
          }
        }
        // P (keys x rows) -> PV operand (rows x keys) by an 8x8 transpose
        const uint32_t pb0 = ptx::movmatrix_trans(v_sc ? dev::pack_h2(p0 * vsa, p1 * vsa) : dev::pack_h2(p0, p1));
        const uint32_t pb1 = ptx::movmatrix_trans(v_sc ? dev::pack_h2(p2 * vsb, p3 * vsb) : dev::pack_h2(p2, p3));

        // ---- O += V^T P^T for all channels (channels are MMA-M).  Every key
        // below the sequence end holds a code the quantizer wrote (never NaN);
        // only a sub-tile reaching past it can meet stale e4m3 NaN bytes, and
        // only there are the V codes clamped.
        auto pv = [&](auto clamp) {
          uint32_t qb0 = pb0, qb1 = pb1;  // this channel group's P (per-group V scales)
#pragma unroll
          for (int jj = 0; jj < Gm::NCH / 2; ++jj) {
            const uint32_t byte = (uint32_t)(2 * jj + ld_chunk) * 16;
            const uint32_t addr =
                sv_base + (byte / Gm::SPAN) * (kTile * Gm::SPAN) + dev::swz<Gm::SPAN>(row_off + byte % Gm::SPAN);
            uint32_t R[4];
            ptx::ldmatrix_x4_trans(R, addr);
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int j = 2 * jj + h2;
              const uint32_t wl = R[2 * h2], wh = R[2 * h2 + 1];
              if (v_grp && ((j * CH) & gmask) == 0) {
                const int grp = j * CH / (GRP ? GS : 1);
                const float ga = key_a < L ? vs_row[(sub * kSub + g) * NG + grp] * vinv : 0.0f;
                const float gb = key_b < L ? vs_row[(sub * kSub + g + 8) * NG + grp] * vinv : 0.0f;
                qb0 = ptx::movmatrix_trans(dev::pack_h2(p0 * ga, p1 * ga));
                qb1 = ptx::movmatrix_trans(dev::pack_h2(p2 * gb, p3 * gb));
              }
              if constexpr (DT == KVQ_INT4) {
                const uint32_t xl = wl ^ 0x88888888u, xh = wh ^ 0x88888888u;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                  const uint32_t A[4] = {dev::i4pair(xl, 8 * t), dev::i4pair(xl, 8 * t + 4), dev::i4pair(xh, 8 * t),
                                         dev::i4pair(xh, 8 * t + 4)};
                  ptx::mma_16816(acc[2 * j + t], A, qb0, qb1);
                }
              } else {
                uint32_t A[4];
                if constexpr (DT == KVQ_INT8) {
                  const uint32_t xl = wl ^ 0x80808080u, xh = wh ^ 0x80808080u;
                  A[0] = dev::i8pair(xl, 0x4240u);
                  A[1] = dev::i8pair(xl, 0x4341u);
                  A[2] = dev::i8pair(xh, 0x4240u);
                  A[3] = dev::i8pair(xh, 0x4341u);
                } else {
                  constexpr bool kC = decltype(clamp)::value;
                  A[0] = dev::f8cvt<kC>(wl, 0x0020u);
                  A[1] = dev::f8cvt<kC>(wl, 0x0031u);
                  A[2] = dev::f8cvt<kC>(wh, 0x0020u);
                  A[3] = dev::f8cvt<kC>(wh, 0x0031u);
                }
                ptx::mma_16816(acc[j], A, qb0, qb1);
              }
            }
          }
        };
        if constexpr (DT == KVQ_FP8_E4M3) {
          if (kb + kSub <= L) pv(dev::Flag<false>{}); else pv(dev::Flag<true>{});
        } else {
          pv(dev::Flag<false>{});
        }
      }
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bar_empty[stage]);
    }

    // ---- unit end: the key warps of a row group merge their states in a
    // fixed chain (warp 0 into 1, the result into 2, ...) through one shared
    // slot per row group; the last warp of the chain writes the partial
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, o);
      l1 += __shfl_xor_sync(0xffffffffu, l1, o);
    }
    float to_true = v_sc ? dev::pow2i(F) : 1.0f;  // acc * to_true = sum_j p_j dequant(v_j)
    float* slot = scr + rg * kScrPerRg;
    for (int k = 1; k < a.key_warps; ++k) {
      if (kw == k - 1) {
#pragma unroll
        for (int mt = 0; mt < Gm::NMT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) slot[(mt * 4 + e) * 32 + lane] = acc[mt][e] * to_true;
        slot[(Gm::NMT * 4 + 0) * 32 + lane] = m0;
        slot[(Gm::NMT * 4 + 1) * 32 + lane] = m1;
        slot[(Gm::NMT * 4 + 2) * 32 + lane] = l0;
        slot[(Gm::NMT * 4 + 3) * 32 + lane] = l1;
      }
      ptx::named_bar_sync(1, (uint32_t)n_cw * 32);
      if (kw == k) {
        const float pm0 = slot[(Gm::NMT * 4 + 0) * 32 + lane], pm1 = slot[(Gm::NMT * 4 + 1) * 32 + lane];
        const float pl0 = slot[(Gm::NMT * 4 + 2) * 32 + lane], pl1 = slot[(Gm::NMT * 4 + 3) * 32 + lane];
        const float M0 = fmaxf(m0, pm0), M1 = fmaxf(m1, pm1);
        const float a0 = M0 == -INFINITY ? 0.0f : ptx::fast_exp2(m0 - M0);
        const float b0 = M0 == -INFINITY ? 0.0f : ptx::fast_exp2(pm0 - M0);
        const float a1 = M1 == -INFINITY ? 0.0f : ptx::fast_exp2(m1 - M1);
        const float b1 = M1 == -INFINITY ? 0.0f : ptx::fast_exp2(pm1 - M1);
#pragma unroll
        for (int mt = 0; mt < Gm::NMT; ++mt) {
          acc[mt][0] = acc[mt][0] * to_true * a0 + slot[(mt * 4 + 0) * 32 + lane] * b0;
          acc[mt][1] = acc[mt][1] * to_true * a1 + slot[(mt * 4 + 1) * 32 + lane] * b1;
          acc[mt][2] = acc[mt][2] * to_true * a0 + slot[(mt * 4 + 2) * 32 + lane] * b0;
          acc[mt][3] = acc[mt][3] * to_true * a1 + slot[(mt * 4 + 3) * 32 + lane] * b1;
        }
        l0 = l0 * a0 + pl0 * b0;
        l1 = l1 * a1 + pl1 * b1;
        m0 = M0;
        m1 = M1;
        to_true = 1.0f;
      }
      ptx::named_bar_sync(1, (uint32_t)n_cw * 32);
    }
    if (kw == a.key_warps - 1) {
      // the tiles above may run while the preceding grid finishes; the
      // workspace is written only after it (no-op after the first)
      ptx::griddep_wait();
      const float f0 = l0 > 0.0f ? to_true / l0 : 0.0f, f1 = l1 > 0.0f ? to_true / l1 : 0.0f;
      const int rr0 = rg * 8 + 2 * c, rr1 = rr0 + 1;
      float* o0 = a.part_o + ((size_t)u * a.rows + rr0) * D;
      float* o1 = o0 + D;
#pragma unroll
      for (int mt = 0; mt < Gm::NMT; ++mt) {
        const int ch = dev::out_channel<DT>(mt, 0, g);
        if (rr0 < a.rows) *reinterpret_cast<float2*>(o0 + ch) = make_float2(acc[mt][0] * f0, acc[mt][2] * f0);
        if (rr1 < a.rows) *reinterpret_cast<float2*>(o1 + ch) = make_float2(acc[mt][1] * f1, acc[mt][3] * f1);
      }
      if (g == 0) {
        if (rr0 < a.rows) a.part_lse[(size_t)u * a.rows + rr0] = l0 > 0.0f ? m0 + ptx::fast_log2(l0) : -INFINITY;
        if (rr1 < a.rows) a.part_lse[(size_t)u * a.rows + rr1] = l1 > 0.0f ? m1 + ptx::fast_log2(l1) : -INFINITY;
      }
    }
  }
}

// Raises (never lowers) the kernel's dynamic shared-memory limit on the
// current device; shared by the occupancy query and the launch so that a
// query for a small plan cannot undercut a larger plan launched later.
template <int DT, int D, int MINB, int NT, int GS>
cudaError_t ensure_smem(size_t smem) {
  static int smem_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_set[dev] < (int)smem) {
    e = cudaFuncSetAttribute(decode_kernel<DT, D, MINB, NT, GS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    smem_set[dev] = (int)smem;
  }
  return cudaSuccess;
}

template <int DT, int D, int MINB, int NT, int GS>
cudaError_t launch_decode_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int grid,
                            int threads, size_t smem, cudaStream_t stream) {
  cudaError_t e = ensure_smem<DT, D, MINB, NT, GS>(smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(decode_kernel<DT, D, MINB, NT, GS>, grid, threads, smem, stream, tk, tv, a);
}

template <int DT, int D, int MINB, int NT, int GS>
cudaError_t occupancy_decode_d(int threads, size_t smem, int* blocks_per_sm) {
  cudaError_t e = ensure_smem<DT, D, MINB, NT, GS>(smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, decode_kernel<DT, D, MINB, NT, GS>,
                                                       threads, smem);
}

// The wide layout needs a channel quarter of at least two 16-byte code chunks.
template <int DT, int D>
constexpr bool wide_ok() { return Geo<DT, D>::NCH >= 8; }

template <int D_, int MINB_, int NT_, int GS_ = 0>
struct KernelCfg {
  static constexpr int d = D_, minb = MINB_, nt = NT_, gs = GS_;
};

// Dispatch on head_dim and on nt (0: grouped layout; -32, -64, -128: grouped
// layout with per-group scales of that many channels; 2, 3: wide layout; head
// dim 576, 8-bit codes only: the wide layout with nt = 1, 2 or 3).
template <int DT, bool Query>
cudaError_t dispatch_decode(int head_dim, int nt, const CUtensorMap* tk, const CUtensorMap* tv, const DecodeArgs* a,
                            int grid, int threads, size_t smem, cudaStream_t stream, int* blocks_per_sm) {
  auto go = [&](auto cfg) -> cudaError_t {
    using K = decltype(cfg);
    if constexpr (Query)
      return occupancy_decode_d<DT, K::d, K::minb, K::nt, K::gs>(threads, smem, blocks_per_sm);
    else
      return launch_decode_d<DT, K::d, K::minb, K::nt, K::gs>(*tk, *tv, *a, grid, threads, smem, stream);
  };
  auto by_nt = [&](auto dtag) -> cudaError_t {
    constexpr int d = decltype(dtag)::value;
    if (nt == 0) return go(KernelCfg<d, d == 256 ? 1 : 2, 0>{});
    if (nt == -32) return go(KernelCfg<d, d == 256 ? 1 : 2, 0, 32>{});
    if (nt == -64) return go(KernelCfg<d, d == 256 ? 1 : 2, 0, 64>{});
    if constexpr (d >= 128) {
      if (nt == -128) return go(KernelCfg<d, d == 256 ? 1 : 2, 0, 128>{});
    }
    if constexpr (wide_ok<DT, d>()) {
      if (nt == 2) return go(KernelCfg<d, 1, 2>{});
      if (nt == 3) return go(KernelCfg<d, 1, 3>{});
    }
    return cudaErrorInvalidValue;
  };
  switch (head_dim) {
    case 64: return by_nt(std::integral_constant<int, 64>{});
    case 128: return by_nt(std::integral_constant<int, 128>{});
    case 256: return by_nt(std::integral_constant<int, 256>{});
    case 576:
      if constexpr (DT != KVQ_INT4) {
        if (nt == 1) return go(KernelCfg<576, 2, 1>{});  // two CTAs per SM (96 registers)
        if (nt == 2) return go(KernelCfg<576, 1, 2>{});
        if (nt == 3) return go(KernelCfg<576, 1, 3>{});
      }
      return cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvq
