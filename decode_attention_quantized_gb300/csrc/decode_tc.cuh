// decode_tc.cuh -- split-KV decode for many query rows per kv head (17..64:
// draft tokens x GQA group) on the tcgen05 tensor cores, accumulators in
// tensor memory (TMEM).
//
// Same computation, split plan, partial format and producer as decode.cuh
// (PagedAttention paged decode, onnxruntime PR #29912; kv-quant-attn page,
// section "Method"; per-channel fold, onnxruntime PR #32515).  With keys as
// the MMA M dimension (128 keys per tile) and the NR padded query rows as N:
//
//   S^T [128 keys x NR]    = K [128 keys x D]          . Q [NR x D]^T
//   O^T [128 ch x NR] (+)= V^T [128 ch x 128 keys] . P [NR x 128 keys]^T   (per 128-channel half)
//   l   [* x NR]     (+)= 1 [128 x 16 keys]         . P^T                  (row sums)
//
// A (K, V^T, ones) lives in TMEM, written there straight from the code stages
// by the dequantizing warps (tcgen05.st), so the f16 copies of K and V never
// touch shared memory; B (Q, P) is in shared memory in the 128-byte swizzle.
// The row sums come from the tensor core too, over the same f16 weights the
// PV product uses; a per-row V scale is folded into V^T (with a power-of-two
// normaliser), so P holds plain softmax weights.
//
// Warp roles (15 warps):
//   0-3   softmax: S^T of a tile out of TMEM in one round trip (one key per
//         thread), scale / softcap / mask, P into shared memory; exact row
//         maxima (and a rescale of O, l) only when a logit exceeds its row's
//         reference maximum by more than 8 (P <= 2^8 in f16, fp32
//         accumulators); also the Q prologue and the epilogue of each piece
//   4-7   K dequant: one key row per thread -> f16 K columns in TMEM, in two
//         channel halves, each released by its half of QK^T
//   8-11  V dequant: ldmatrix.trans fragments -> V^T in TMEM (16x256b
//         stores), per 128-channel half; a per-row V scale is folded in
//   12    TMA producer of the code stages (shared with decode.cuh)
//   13    TMEM allocation; issues QK^T into a double-buffered S^T
//   14    issues PV and the row sums
// MMAs are issued by an elected lane of a converged warp, four k-steps per
// asm block; bounded waits poll once inline and loop out of line.  The
// code is kept compact (rolled loops where registers allow): fifteen
// warps on four schedulers run six different loops, and a kernel whose
// hot code outgrows the instruction caches stalls on instruction fetch.
#pragma once

#include "decode.cuh"

namespace kvq {

template <int DT, int D, int NR>
struct TcCfg {
  using Gm = Geo<DT, D, kTcKeys>;
  static constexpr int NH = D / 128;  // 128-channel halves of V^T and O^T
  // TMEM columns (32-bit)
  static constexpr int K_COL = 0;                 // [128 key lanes x D channels], f16 pairs
  static constexpr int V_COL = K_COL + D / 2;     // NH x [128 channel lanes x 128 keys], f16 pairs
  static constexpr int O_COL = V_COL + NH * 64;   // NH x [128 channel lanes x NR rows], fp32
  static constexpr int S_COL = O_COL + NH * NR;   // 2 x [128 key lanes x NR rows], fp32
  static constexpr int L_COL = S_COL + 2 * NR;    // row sums (every lane holds a copy)
  static constexpr int ONE_COL = L_COL + NR;      // 8 columns of f16 ones: A of the row-sum product
  static constexpr int TMEM_COLS = 512;
  static_assert(D == 128 || D == 256, "head_dim 128 or 256");
  static_assert(NR % 16 == 0 && NR >= 32 && NR <= 64, "N of an M=128 MMA: multiple of 16");
  static_assert(ONE_COL + 8 <= TMEM_COLS, "TMEM columns");
  static constexpr int P_BYTES = NR * 2 * kTcKeys;  // one P buffer
};

namespace dev {

// Tile-local key k -> its K index in the PV product.  The V^T fragments put,
// in each 16-key group, keys 2c, 2c+1 at K indices 4c, 4c+1 and keys
// 2c+8, 2c+9 at 4c+2, 4c+3 (c = 0..3); P is stored in the same order.
__device__ __forceinline__ int pv_kpos(int k) {
  return (k & ~15) | (((k & 7) >> 1) << 2) | (((k >> 3) & 1) << 1) | (k & 1);
}

// Channel of O^T lane `lane` of lane quarter q in channel half h.  Lane tile
// lt = lane / 16 of the quarter holds a 16-channel A fragment whose row i
// (= lane % 16) is channel 2g + (i >> 3) of a 16-byte 8-bit code chunk, or
// channel 4g + 2 lt + (i >> 3) of a 16-byte int4 chunk (g = i & 7).
template <int DT>
__device__ __forceinline__ int tc_out_channel(int h, int q, int lane) {
  const int lt = lane >> 4, i = lane & 15, g = i & 7, rs = i >> 3;
  if constexpr (DT == KVQ_INT4)
    return 32 * (4 * h + q) + 4 * g + 2 * lt + rs;
  else
    return 16 * (8 * h + 2 * q + lt) + 2 * g + rs;
}

// int4 nibble pairs -> f16 pairs in one LOP3 + one subtraction each.  The
// field (w & mask) is XORed with the offset 8 (two's complement -> code + 8)
// and given the exponent byte 0x64 (1024 + field): nibbles at bits 0 / 16
// give (code + 8) + 1024, minus 1032 -> code; nibbles at bits 4 / 20 give
// 16 (code + 8) + 1024, minus 1152 -> 16 code.  Both exact; a zero code
// gives an exact zero.
__device__ __forceinline__ uint32_t i4lo(uint32_t w) {
  return ptx::hsub2_u32((w & 0x000F000Fu) ^ 0x64086408u, 0x64086408u);
}
__device__ __forceinline__ uint32_t i4hi16(uint32_t w) {
  return ptx::hsub2_u32((w & 0x00F000F0u) ^ 0x64806480u, 0x64806480u);
}

// Odd int4 channels (the high nibble of each byte) come out of the
// conversions above times 16: Q carries 1/16 for them and the output is
// scaled by 1/16 (both exact).
template <int DT>
__host__ __device__ constexpr float odd_channel_factor() {
  return DT == KVQ_INT4 ? 0.0625f : 1.0f;
}

// One 16-byte chunk of a key's code row -> its f16 values as K columns
// (K index = column * 2 + half).  8-bit: channels in order.  int4: each
// 32-bit word (channels 8i..8i+7, even channel in the low nibble) gives the
// pairs (8i+n, 8i+n+4), n = 0..3, odd n times 16, so K index 8i + 2n + e
// holds channel 8i + n + 4e; Q is stored in the same order.
template <int DT>
__device__ __forceinline__ void k_cols(const uint4 w4, uint32_t* v) {
  const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (DT == KVQ_INT4) {
      const uint32_t y = w[i] >> 8;
      v[4 * i] = i4lo(w[i]);
      v[4 * i + 1] = i4hi16(w[i]);
      v[4 * i + 2] = i4lo(y);
      v[4 * i + 3] = i4hi16(y);
    } else if constexpr (DT == KVQ_INT8) {
      const uint32_t x = w[i] ^ 0x80808080u;
      v[2 * i] = i8pair(x, 0x4140u);
      v[2 * i + 1] = i8pair(x, 0x4342u);
    } else {
      v[2 * i] = e4m3x2_f16x2((uint16_t)(w[i] & 0xFFFFu));
      v[2 * i + 1] = e4m3x2_f16x2((uint16_t)(w[i] >> 16));
    }
  }
}

// The four 16x256b registers of one 16-key group of a V^T lane tile, from the
// ldmatrix.trans words of keys 0-7 (wl) and 8-15 (wh): A-fragment rows
// g / g+8 (two channels) x keys (2c, 2c+1) and (2c+8, 2c+9), placed as
// (lane g, col 2c), (lane g, col 2c+1), (lane g+8, col 2c), (lane g+8,
// col 2c+1).  t selects the int4 channel pair of the chunk (row g+8, the odd
// channel, times 16).  Every code maps to a finite f16 (e4m3 by the NaN-free
// bit move, value * 2^-8).
template <int DT>
__device__ __forceinline__ void v_frag(uint32_t wl, uint32_t wh, int t, uint32_t* r) {
  uint32_t a0, a1, a2, a3;
  if constexpr (DT == KVQ_INT4) {
    const uint32_t xl = t ? wl >> 8 : wl, xh = t ? wh >> 8 : wh;
    a0 = i4lo(xl);
    a1 = i4hi16(xl);
    a2 = i4lo(xh);
    a3 = i4hi16(xh);
  } else if constexpr (DT == KVQ_INT8) {
    const uint32_t xl = wl ^ 0x80808080u, xh = wh ^ 0x80808080u;
    a0 = i8pair(xl, 0x4240u);
    a1 = i8pair(xl, 0x4341u);
    a2 = i8pair(xh, 0x4240u);
    a3 = i8pair(xh, 0x4341u);
  } else {
    a0 = f8pair(wl, 0x2404u);
    a1 = f8pair(wl, 0x3414u);
    a2 = f8pair(wh, 0x2404u);
    a3 = f8pair(wh, 0x3414u);
  }
  r[0] = a0;
  r[1] = a2;
  r[2] = a1;
  r[3] = a3;
}

// The slow path of a bounded wait: polls until the phase completes, or on a
// timeout (or an earlier one anywhere in the CTA) sets the CTA's abort flag
// and KVQ_DEVERR_TIMEOUT and returns.
static __device__ __noinline__ void wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                                  unsigned int* err) {
  if (*abort_flag) return;
  if (!ptx::mbar_wait_slow(bar, parity)) {
    *abort_flag = 1;
    atomicOr(err, KVQ_DEVERR_TIMEOUT);
  }
}

// N columns of this warp's TMEM lane quarter (x16 loads, one wait).  The
// empty asm statements tie every register to the wait, so that no use of a
// loaded value is scheduled before the load has completed.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[N]) {
  static_assert(N % 16 == 0, "16-column loads");
  uint32_t u[N];
#pragma unroll
  for (int j = 0; j < N / 16; ++j) ptx::tmem_ld16(taddr + 16 * j, *reinterpret_cast<uint32_t(*)[16]>(u + 16 * j));
  ptx::tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < N; ++i) {
    asm volatile("" : "+r"(u[i]));
    v[i] = __uint_as_float(u[i]);
  }
}

template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const float (&v)[N]) {
  static_assert(N % 16 == 0, "16-column stores");
#pragma unroll
  for (int j = 0; j < N / 16; ++j) {
    uint32_t u[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(v[16 * j + i]);
    ptx::tmem_st16(taddr + 16 * j, u);
  }
}

}  // namespace dev

template <int DT, int D, int NR, bool GRP>
__global__ void __launch_bounds__(kTcWarps * 32, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const DecodeArgs a) {
  using C = TcCfg<DT, D, NR>;
  using Gm = typename C::Gm;
  constexpr int KT = kTcKeys;
  constexpr int kSoftmax = 0, kDqK = 4, kDqV = 8, kProducer = 12, kMma = 13, kMmaPv = 14;
  constexpr int NKS = D / 16;  // k-steps of QK^T; the K tile is freed in two channel halves
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* base = smem_raw + pad;
  const TcSmem lay = tc_smem_layout(D, Gm::DP, NR, a.stages, a.batch, a.stage_stride);
  uint8_t* ring = base + lay.ring;
  uint8_t* q_s = base + lay.q;
  uint8_t* p_s = base + lay.p;
  float* f_alpha = reinterpret_cast<float*>(base + lay.scr);  // [NR] logit factor of each row
  int* i_pos = reinterpret_cast<int*>(f_alpha + NR);           // [NR] last key each row sees (-1: padding)
  float* f_red = reinterpret_cast<float*>(i_pos + NR);         // [4][NR] tile row maxima per softmax warp
  float* f_mu = f_red + 4 * NR;                                 // [4][NR] exponent offsets, a copy per warp
  float* f_corr = f_mu + 4 * NR;                                // [4][NR] rescale factors, a copy per warp
  float* f_vmax = f_corr + 4 * NR;                              // [2][8] by tile parity: overflow flags, V-scale maxima
  int* pl_pre = reinterpret_cast<int*>(base + lay.pre);
  int* pl_misc = pl_pre + a.batch + 1;
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(base + lay.bars);
  uint64_t* bar_empty = bar_full + a.stages;
  uint64_t* b_qk = bar_empty + a.stages;  // [2] S^T buffer written by QK^T (K columns free)
  uint64_t* b_sfree = b_qk + 2;           // [2] S^T buffer consumed by the softmax warps
  uint64_t* b_kh0 = b_qk + 4;             // first half of QK^T done: K channel half 0 free
  uint64_t* b_kfull = b_qk + 5;           // [2] K channel half in TMEM
  uint64_t* b_vh = b_qk + 7;              // [2] PV of a V^T channel half done: that half free
  uint64_t* b_vfull = b_qk + 9;           // [2] V^T channel half in TMEM
  uint64_t* b_pfull = b_qk + 11;          // [2] P buffer written (and O rescaled)
  uint64_t* b_pv = b_qk + 13;             // [2] PV + row sums of a tile complete
  uint64_t* b_qfull = b_qk + 15;          // Q of a piece written
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + lay.slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      ptx::mbar_init(&bar_full[s], 1);
      ptx::mbar_init(&bar_empty[s], 12);  // K, V and softmax warps
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&b_qk[i], 1);
      ptx::mbar_init(&b_sfree[i], 4);
      ptx::mbar_init(&b_kfull[i], 4);
      ptx::mbar_init(&b_vh[i], 1);
      ptx::mbar_init(&b_vfull[i], 4);
      ptx::mbar_init(&b_pfull[i], 4);
      ptx::mbar_init(&b_pv[i], 1);
    }
    ptx::mbar_init(b_kh0, 1);
    ptx::mbar_init(b_qfull, 4);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMma) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tc_fence_before();
  }
  // With early reads (KVQ_DECODE_EARLY_INPUTS) the inputs the caller vouches
  // for (seq_lens, block table, q, static scales) are read before the wait on
  // the preceding grid on the stream: the producer waits before its first
  // cache read, the softmax warps before their first workspace write (the
  // other roles touch only shared memory and TMEM), so the plan, the first
  // block ids and the Q prologue overlap that grid's tail.  Without them
  // build_slice waits first.
  const Slice<KT> sp = build_slice<KT>(a, pl_pre, pl_misc);
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Bounded wait; after the first timeout every later wait of the CTA is
  // skipped (results are garbage, flagged KVQ_DEVERR_TIMEOUT, and the CTA
  // still reaches its end).  Only the first poll is inlined.
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (!ptx::mbar_try_wait(bar, parity)) dev::wait_or_abort(bar, parity, abort_flag, a.err);
  };
  const bool k_row = a.k_mode == KVQ_SCALE_PER_ROW, v_row = a.v_mode == KVQ_SCALE_PER_ROW;
  // group-wise scales (a stage holds K's [KT][nk] and V's [KT][nv] of them;
  // only the GRP instances carry their code)
  const bool k_grp = GRP && a.k_mode == KVQ_SCALE_PER_GROUP, v_grp = GRP && a.v_mode == KVQ_SCALE_PER_GROUP;
  const int nk = a.sk_n, nv = a.sv_n, lg = a.log2_gs;
  // V scales in a stage, and the stage stride (compile-time without groups)
  const uint32_t v_sc_off = 2 * Gm::CODE_BYTES + KT * 4 * (GRP && nk > 1 ? nk : 1);
  const uint32_t stage_bytes = GRP ? (uint32_t)a.stage_stride : (uint32_t)Gm::STAGE_STRIDE;
  // logits take a per-key factor; V^T columns carry scales under the normaliser 2^F
  const bool k_sc = k_row || k_grp, v_sc = v_row || v_grp;

  if (warp == kProducer) {
    // ============================================================ producer
    produce<Gm, false>(a, sp, &tmk, &tmv, ring, bar_full, bar_empty, pl_pre, pl_misc);
  } else if (warp >= kDqK && warp < kDqK + 4) {
    // ========================================================== K dequant
    // thread = key 32 q + lane of the tile = TMEM lane of the K operand; the
    // two channel halves are written (and freed by QK^T) one after the other,
    // each converted before the wait for the QK^T that frees it.  Per-group K
    // scales: the key's columns carry code * s_g / 2^E, 2^E the power of two
    // at or above its largest group scale (the softmax multiplies the logit
    // by 2^E, as by a per-row scale)
    const int q = warp - kDqK, kk = 32 * q + lane;
    const uint32_t t_k = tmem + ((uint32_t)(32 * q) << 16) + C::K_COL;
    constexpr int HCH = Gm::NCH / 2;  // 16-byte chunks of a channel half
    uint32_t it = 0;
    RingPos rp;
    for (int gt = sp.t_begin, next; gt < sp.t_end; gt = next) {
      int b, h, k0, k1, L, u;
      sp.piece(a, gt, b, h, k0, k1, L, u, next);
      for (int key0 = k0; key0 < k1; key0 += KT, ++it, rp.next(a.stages)) {
        const uint32_t stage = rp.stage;
        wait(&bar_full[stage], rp.phase);
        const uint8_t* st = ring + (size_t)stage * stage_bytes;
        const float* kgs = reinterpret_cast<const float*>(st + 2 * Gm::CODE_BYTES) + kk * nk;
        float kinv = 0.0f;
        if (k_grp) {
          float mx = 0.0f;
          for (int g = 0; g < nk; ++g) mx = fmaxf(mx, kgs[g]);
          kinv = mx > 0.0f ? dev::pow2i(-min(126, max(-126, dev::ceil_log2(mx)))) : 0.0f;
        }
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          // the half's codes are read and converted before the wait for the
          // previous QK^T, so only the TMEM stores follow its completion
          constexpr int CW = DT == KVQ_INT4 ? 16 : 8;  // K columns per 16-byte chunk
          uint4 w[HCH];
#pragma unroll
          for (int jj = 0; jj < HCH; ++jj) {
            const uint32_t byte = (uint32_t)(half * HCH + jj) * 16;
            w[jj] = *reinterpret_cast<const uint4*>(
                st + (byte / Gm::SPAN) * (KT * Gm::SPAN) + dev::swz<Gm::SPAN>(kk * Gm::SPAN + byte % Gm::SPAN));
          }
          uint32_t v[HCH * CW];
#pragma unroll
          for (int jj = 0; jj < HCH; ++jj) dev::k_cols<DT>(w[jj], v + CW * jj);
          if (k_grp) {
            constexpr int CHC = DT == KVQ_INT4 ? 32 : 16;  // channels of a 16-byte chunk (one group)
#pragma unroll
            for (int jj = 0; jj < HCH; ++jj) {
              const float r = kgs[((half * HCH + jj) * CHC) >> lg] * kinv;
              const uint32_t rr = dev::pack_h2(r, r);
#pragma unroll
              for (int m = 0; m < CW; ++m) v[CW * jj + m] = ptx::hmul2_u32(v[CW * jj + m], rr);
            }
          }
          if (it > 0) {
            if (half == 0) wait(b_kh0, (it - 1) & 1);                        // QK^T(t-1) read channel half 0
            else wait(&b_qk[(it - 1) & 1], ((it - 1) >> 1) & 1);             // QK^T(t-1) complete
          }
          ptx::tc_fence_after();
          // the half's HCH * CW columns (32 or 64) in one store
          if constexpr (HCH * CW == 64)
            ptx::tmem_st64(t_k + HCH * CW * half, v);
          else
            ptx::tmem_st32(t_k + HCH * CW * half, v);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&b_kfull[half]);
        }
        if (lane == 0) ptx::mbar_arrive(&bar_empty[stage]);
      }
    }
  } else if (warp >= kDqV && warp < kDqV + 4) {
    // ========================================================== V dequant
    // lane quarter q of each 128-channel half: two 16-lane tiles of V^T.
    // Per-row V scale: the columns of key k carry vs_k / 2^F, F the power of
    // two at or above the largest scale of the piece so far (keys past the
    // sequence end get 0); the softmax warps track the same F.  Per-group: the
    // same with the scale of the group of this warp's channels (the 32
    // channels a lane quarter holds in one half lie in one group), F over
    // every group of the piece's keys.
    const int q = warp - kDqV;
    const int ld_key = ((lane >> 3) & 1) * 8 + (lane & 7), ld_chunk = lane >> 4;
    const int c = lane & 3;
    uint32_t it = 0;
    RingPos rp;
    for (int gt = sp.t_begin, next; gt < sp.t_end; gt = next) {
      int b, h, k0, k1, L, u;
      sp.piece(a, gt, b, h, k0, k1, L, u, next);
      int F = -126;
      for (int key0 = k0; key0 < k1; key0 += KT, ++it, rp.next(a.stages)) {
        const uint32_t stage = rp.stage;
        wait(&bar_full[stage], rp.phase);
        const uint8_t* st = ring + (size_t)stage * stage_bytes;
        const uint32_t sv = ptx::smem_u32(st) + Gm::CODE_BYTES;
        const float* vsp = reinterpret_cast<const float*>(st + v_sc_off);
        uint32_t s_lo[8], s_hi[8];
        float vinv = 0.0f;
        // the scale pairs of keys (2c, 2c + 1) and (2c + 8, 2c + 9) of each
        // 16-key group, scale index j of a key = key * stride + j
        auto v_pairs = [&](int stride, int j) {
#pragma unroll
          for (int kg = 0; kg < 8; ++kg) {
            const int ka = 16 * kg + 2 * c, kb = ka + 8;
            s_lo[kg] = dev::pack_h2(key0 + ka < L ? vsp[ka * stride + j] * vinv : 0.0f,
                                    key0 + ka + 1 < L ? vsp[(ka + 1) * stride + j] * vinv : 0.0f);
            s_hi[kg] = dev::pack_h2(key0 + kb < L ? vsp[kb * stride + j] * vinv : 0.0f,
                                    key0 + kb + 1 < L ? vsp[(kb + 1) * stride + j] * vinv : 0.0f);
          }
        };
        if (v_row || v_grp) {
          float vm = 0.0f;
#pragma unroll
          for (int i = 0; i < KT / 32; ++i)
            if (key0 + 32 * i + lane < L) {
              if (v_row) {
                vm = fmaxf(vm, vsp[32 * i + lane]);
              } else {
                for (int g = 0; g < nv; ++g) vm = fmaxf(vm, vsp[(32 * i + lane) * nv + g]);
              }
            }
          vm = ptx::redux_max(vm);
          if (vm > 0.0f) F = max(F, min(126, max(-126, dev::ceil_log2(vm))));
          vinv = dev::pow2i(-F);
          if (v_row) v_pairs(1, 0);
        }
#pragma unroll 1
        for (int hh = 0; hh < C::NH; ++hh) {
          if (v_grp) v_pairs(nv, (128 * hh + 32 * q) >> lg);
          uint32_t f0[32], f1[32];  // lane tiles 0 / 1: 8 key groups x 4 registers
          if constexpr (DT == KVQ_INT4) {
            // chunk 4 hh + q (32 channels): tile t = channel pair t of each 4
            const uint32_t byte = (uint32_t)(4 * hh + q) * 16;
#pragma unroll
            for (int kp = 0; kp < 4; ++kp) {
              const int row = 32 * kp + (lane >> 3) * 8 + (lane & 7);
              const uint32_t addr = sv + (byte / Gm::SPAN) * (KT * Gm::SPAN) +
                                    dev::swz<Gm::SPAN>((uint32_t)row * Gm::SPAN + byte % Gm::SPAN);
              uint32_t R[4];
              ptx::ldmatrix_x4_trans(R, addr);
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                dev::v_frag<DT>(R[2 * e], R[2 * e + 1], 0, &f0[4 * (2 * kp + e)]);
                dev::v_frag<DT>(R[2 * e], R[2 * e + 1], 1, &f1[4 * (2 * kp + e)]);
              }
            }
          } else {
            // chunks 8 hh + 2 q (tile 0) and + 1 (tile 1), 16 channels each
#pragma unroll
            for (int kg = 0; kg < 8; ++kg) {
              const uint32_t byte = (uint32_t)(8 * hh + 2 * q + ld_chunk) * 16;
              const int row = 16 * kg + ld_key;
              const uint32_t addr = sv + (byte / Gm::SPAN) * (KT * Gm::SPAN) +
                                    dev::swz<Gm::SPAN>((uint32_t)row * Gm::SPAN + byte % Gm::SPAN);
              uint32_t R[4];
              ptx::ldmatrix_x4_trans(R, addr);
              dev::v_frag<DT>(R[0], R[1], 0, &f0[4 * kg]);
              dev::v_frag<DT>(R[2], R[3], 0, &f1[4 * kg]);
            }
          }
          if (v_row || v_grp) {
#pragma unroll
            for (int kg = 0; kg < 8; ++kg) {
              f0[4 * kg] = ptx::hmul2_u32(f0[4 * kg], s_lo[kg]);
              f0[4 * kg + 1] = ptx::hmul2_u32(f0[4 * kg + 1], s_hi[kg]);
              f0[4 * kg + 2] = ptx::hmul2_u32(f0[4 * kg + 2], s_lo[kg]);
              f0[4 * kg + 3] = ptx::hmul2_u32(f0[4 * kg + 3], s_hi[kg]);
              f1[4 * kg] = ptx::hmul2_u32(f1[4 * kg], s_lo[kg]);
              f1[4 * kg + 1] = ptx::hmul2_u32(f1[4 * kg + 1], s_hi[kg]);
              f1[4 * kg + 2] = ptx::hmul2_u32(f1[4 * kg + 2], s_lo[kg]);
              f1[4 * kg + 3] = ptx::hmul2_u32(f1[4 * kg + 3], s_hi[kg]);
            }
          }
          if (it > 0) wait(&b_vh[hh], (it - 1) & 1);  // PV(t-1) has read this channel half
          ptx::tc_fence_after();
          const uint32_t t_v = tmem + C::V_COL + 64 * hh;
          ptx::tmem_st16x256_x8(t_v + ((uint32_t)(32 * q) << 16), f0);
          ptx::tmem_st16x256_x8(t_v + ((uint32_t)(32 * q + 16) << 16), f1);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&b_vfull[hh]);
        }
        if (lane == 0) ptx::mbar_arrive(&bar_empty[stage]);
      }
    }
  } else if (warp == kMma || warp == kMmaPv) {
    // ================================================================ MMA
    // Two issuing warps on different schedulers: warp kMma issues QK^T of
    // every tile, warp kMmaPv its PV and row sums (their TMEM regions and
    // shared operands are disjoint; the softmax orders the two).  Each warp
    // runs its loop whole and converged; one elected lane issues every MMA
    // and commit.  Runs of 4 k-steps (one 128-byte swizzle row of B) are one
    // asm block; each operand half is released as soon as the MMAs that
    // read it complete.
    constexpr uint32_t idesc = ptx::idesc_f16_f32(128, NR);
    const uint64_t q_desc = ptx::smem_desc_sw128(ptx::smem_u32(q_s));
    const uint32_t q_lo = (uint32_t)q_desc, d_hi = (uint32_t)(q_desc >> 32);
    const uint32_t p_lo = (uint32_t)ptx::smem_desc_sw128(ptx::smem_u32(p_s));
    constexpr uint32_t kSlabDesc = (NR * 128) >> 4;  // descriptor step between 64-element K slabs
    const bool qk_warp = warp == kMma;
    uint32_t it = 0;
    int pc = 0;
    for (int gt = sp.t_begin, next; gt < sp.t_end; gt = next, ++pc) {
      int b, h, k0, k1, L, u;
      sp.piece(a, gt, b, h, k0, k1, L, u, next);
      for (int key0 = k0; key0 < k1; key0 += KT, ++it) {
        const bool first = key0 == k0;
        if (qk_warp) {
          // ---- QK^T of tile `it` (two channel halves, each committed)
          if (first) wait(b_qfull, pc & 1);
          if (it >= 2) wait(&b_sfree[it & 1], ((it - 2) >> 1) & 1);  // the softmax is done with this S buffer
          const uint32_t s_col = tmem + C::S_COL + (it & 1) * NR;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            wait(&b_kfull[half], it & 1);
            __syncwarp();
            ptx::tc_fence_after();
#pragma unroll 1
            for (int sl = half * (D / 128); sl < (half + 1) * (D / 128); ++sl)
              ptx::mma_f16_ts_x4(s_col, tmem + C::K_COL + 32 * sl, 8, q_lo + sl * kSlabDesc, d_hi, idesc,
                                 sl > 0 ? 1u : 0u);
            ptx::mma_commit(half == 0 ? b_kh0 : &b_qk[it & 1]);
          }
        } else {
          // ---- PV and row sums of tile `it`.  A piece's first PV overwrites
          // O and l: the softmax warps read the previous piece's out before
          // they release that tile's P buffer.
          wait(&b_pfull[it & 1], (it >> 1) & 1);
          __syncwarp();
          ptx::tc_fence_after();
          const uint32_t pb = p_lo + (it & 1) * (C::P_BYTES >> 4);
          const uint32_t acc0 = first ? 0u : 1u;
#pragma unroll 1
          for (int sl = 0; sl < 2; ++sl)
            ptx::mma_f16_ts_x4(tmem + C::L_COL, tmem + C::ONE_COL, 0, pb + sl * kSlabDesc, d_hi, idesc,
                               sl ? 1u : acc0);
#pragma unroll 1
          for (int hh = 0; hh < C::NH; ++hh) {
            wait(&b_vfull[hh], it & 1);
            __syncwarp();
            ptx::tc_fence_after();
#pragma unroll 1
            for (int sl = 0; sl < 2; ++sl)
              ptx::mma_f16_ts_x4(tmem + C::O_COL + hh * NR, tmem + C::V_COL + 64 * hh + 32 * sl, 8,
                                 pb + sl * kSlabDesc, d_hi, idesc, sl ? 1u : acc0);
            ptx::mma_commit(&b_vh[hh]);
          }
          ptx::mma_commit(&b_pv[it & 1]);
        }
      }
    }
    if (it > 0) {
      // every MMA this warp issued has completed before TMEM can be released
      const uint32_t last = it - 1;
      uint64_t* done = qk_warp ? &b_qk[last & 1] : &b_pv[last & 1];
      if (!ptx::mbar_wait_bounded(done, (last >> 1) & 1) && lane == 0) atomicOr(a.err, KVQ_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ============================================================ softmax
    const int q = warp - kSoftmax;
    const int kk = 32 * q + lane;  // tile-local key of this thread = TMEM lane of S^T
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q) << 16);
    const int G = a.group, T = a.q_tokens, Hq = a.num_q_heads, W = a.window, rows = a.rows;
    const float inv_g = __frcp_rn((float)G);  // r / G by dev::div_small
    const float softcap = a.softcap;
    const float inv_cap = softcap > 0.0f ? 1.0f / softcap : 0.0f;
    // where this key's P goes in a P buffer: slab of 64 K indices, 16-byte
    // chunk and byte inside the 128-byte row (the row's chunk index is XORed
    // with row & 7, the 128-byte swizzle)
    const int kpos = dev::pv_kpos(kk);
    uint32_t p_st[8];  // byte offset of this key in rows r = 8 i + j, minus r * 128
    {
      const uint32_t p_chunk = (uint32_t)(kpos & 63) >> 3, p_in = ((uint32_t)(kpos & 7)) * 2;
#pragma unroll
      for (int j = 0; j < 8; ++j) p_st[j] = (uint32_t)(kpos >> 6) * (NR * 128) + (((p_chunk ^ (uint32_t)j) & 7u) << 4) + p_in;
    }
    {
      uint32_t ones[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ones[i] = 0x3C003C00u;  // f16 1.0 pairs
      ptx::tmem_st8(t_lane + C::ONE_COL, ones);
      ptx::tmem_wait_st();
    }
    // Q prologue geometry: 8 channels per lane, D / 8 lanes per row, RPP rows
    // per warp pass, NQR rows per thread
    constexpr int LPR = D / 8, RPP = 32 / LPR, NQR = NR / (4 * RPP);
    const int rsub = lane / LPR, cl = lane % LPR;

    // Epilogue of a piece: O and row sums out of TMEM 16 rows at a time (the
    // sums and both O channel halves of a chunk in one TMEM round trip), the
    // normalized partial and its base-2 log-sum-exp to the workspace.  Run
    // once per piece, so kept small (its code is cold by then).
    auto epilogue = [&](int u, uint32_t last, float m0, float m1, int F) {
      wait(&b_pv[last & 1], (last >> 1) & 1);
      ptx::tc_fence_after();
      float to_true = v_sc ? dev::pow2i(F) : 1.0f;
      if constexpr (DT == KVQ_FP8_E4M3) to_true *= 256.0f;
      float* lse = a.part_lse + (size_t)u * rows;
#pragma unroll 1
      for (int r0 = 0; r0 < rows; r0 += 16) {
        uint32_t lu[16], ou[C::NH][16];
        ptx::tmem_ld16(t_lane + C::L_COL + r0, lu);
#pragma unroll
        for (int hh = 0; hh < C::NH; ++hh) ptx::tmem_ld16(t_lane + C::O_COL + hh * NR + r0, ou[hh]);
        ptx::tmem_wait_ld();
        // every lane holds all 16 sums; lane j + (r0 & 31) takes row r0 + j's
        const int j = lane - (r0 & 31);
        float lj = 0.0f, inv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          asm volatile("" : "+r"(lu[i]));
          const float l = __uint_as_float(lu[i]);
          lj = j == i ? l : lj;
          inv[i] = l > 0.0f ? to_true * ptx::fast_rcp(l) : 0.0f;
        }
        if (q == 0 && j >= 0 && j < 16 && r0 + j < rows)
          lse[r0 + j] = lj > 0.0f ? (r0 + j < 32 ? m0 : m1) + ptx::fast_log2(lj) : -INFINITY;
#pragma unroll
        for (int hh = 0; hh < C::NH; ++hh) {
          const int ch = dev::tc_out_channel<DT>(hh, q, lane);
          const float cf = (ch & 1) ? dev::odd_channel_factor<DT>() : 1.0f;
          float* dst = a.part_o + ((size_t)u * rows + r0) * D + ch;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            asm volatile("" : "+r"(ou[hh][i]));
            if (r0 + i < rows) dst[(size_t)i * D] = __uint_as_float(ou[hh][i]) * inv[i] * cf;
          }
        }
      }
      ptx::tc_fence_before();
    };

    uint32_t it = 0;
    RingPos rp;
    int pc = 0;
    int e_u = 0, e_F = 0;  // the previous piece, for its epilogue
    uint32_t e_last = 0;
    float e_mu0 = 0.0f, e_mu1 = 0.0f;
    for (int gt = sp.t_begin, next = 0;; gt = next, ++pc) {
      const bool more = gt < sp.t_end;
      int b = 0, h = 0, k0 = 0, k1 = 0, L = 0, u = 0;
      if (more) sp.piece(a, gt, b, h, k0, k1, L, u, next);
      // every softmax warp is done with the previous piece's row factors
      ptx::named_bar_sync(1, 128);

      // ---- Q of this piece (this warp waited for the previous piece's last
      // QK^T, so the buffer is free): per-channel K scale folded in under a
      // power-of-two normaliser, each row normalised by the power of two just
      // above its maximum, f16 in the MMA's K order, 128-byte swizzle.  Every
      // row this thread converts is loaded first (one round trip), and the
      // rows are converted with their reductions interleaved.
      if (more) {
        const bool kc = a.k_mode == KVQ_SCALE_PER_CHANNEL;
        uint4 raw[NQR];
#pragma unroll
        for (int i = 0; i < NQR; ++i) {
          const int r = (q + 4 * i) * RPP + rsub;
          const int t = dev::div_small(r, inv_g);
          raw[i] = r < rows ? ptx::ldg_nc_v4(a.q + (((size_t)b * T + t) * Hq + (size_t)h * G + r - t * G) * D + 8 * cl)
                            : make_uint4(0, 0, 0, 0);
        }
        float ksv[8];
        int ek = 0;
        if (kc) {
          const float4* ksp = reinterpret_cast<const float4*>(a.k_scale + (size_t)h * D + 8 * cl);
          const float4 s0 = __ldg(ksp), s1 = __ldg(ksp + 1);
          ksv[0] = s0.x; ksv[1] = s0.y; ksv[2] = s0.z; ksv[3] = s0.w;
          ksv[4] = s1.x; ksv[5] = s1.y; ksv[6] = s1.z; ksv[7] = s1.w;
          float km = 0.0f;
#pragma unroll
          for (int i = 0; i < 8; ++i) km = fmaxf(km, fabsf(ksv[i]));
#pragma unroll
          for (int o = 1; o < LPR; o <<= 1) km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
          ek = km > 0.0f ? min(126, max(-126, dev::ceil_log2(km))) : 0;
          const float sk = dev::pow2i(-ek);
#pragma unroll
          for (int i = 0; i < 8; ++i) ksv[i] *= sk;
        }
        float base = a.sm_scale;
        if (a.k_mode == KVQ_SCALE_PER_TENSOR) base *= a.k_scale[0];
        if (softcap <= 0.0f) base *= kLog2e;
#pragma unroll
        for (int i = 0; i < NQR; ++i) {
          const int r = (q + 4 * i) * RPP + rsub;
          float qv[8];
          const uint32_t ww[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[2 * j] = __uint_as_float(ww[j] << 16);
            qv[2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
          }
          if (kc) {
#pragma unroll
            for (int j = 0; j < 8; ++j) qv[j] *= ksv[j];
          }
          float qm = 0.0f;
#pragma unroll
          for (int j = 0; j < 8; ++j) qm = fmaxf(qm, fabsf(qv[j]));
          if constexpr (LPR == 32) {
            qm = ptx::redux_max(qm);  // one row per warp
          } else {
#pragma unroll
            for (int o = 1; o < LPR; o <<= 1) qm = fmaxf(qm, __shfl_xor_sync(0xffffffffu, qm, o));
          }
          const int eq = qm > 0.0f ? min(126, max(-126, dev::ceil_log2(qm))) : 0;
          const float sq = dev::pow2i(-eq);
          uint32_t w[4];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            if constexpr (DT == KVQ_INT4) {
              const float f = (m & 1) ? sq * dev::odd_channel_factor<DT>() : sq;  // channels m, m + 4
              w[m] = dev::pack_h2(qv[m] * f, qv[m + 4] * f);
            } else {
              w[m] = dev::pack_h2(qv[2 * m] * sq, qv[2 * m + 1] * sq);
            }
          }
          uint8_t* dst = q_s + (cl >> 3) * (NR * 128) + r * 128 + ((((uint32_t)cl & 7u) ^ ((uint32_t)r & 7u)) << 4);
          *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
          if (cl == 0) {
            // alpha = base * 2^(ek + eq) as two exact power-of-two steps (each
            // exponent within the normal range), finite, and > 0 so that
            // alpha * (-inf) stays -inf
            const int e = ek + eq, e1 = e / 2;
            const float al = fmaxf(fminf(base * dev::pow2i(e1) * dev::pow2i(e - e1), 3.4028234e38f), 1e-30f);
            const bool valid = r < rows;
            f_alpha[r] = valid ? al : 1.0f;
            i_pos[r] = valid ? L - T + dev::div_small(r, inv_g) : -1;
          }
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_qfull);
      }
      // before the first tile (not only before the first workspace write, as
      // in the other kernels): this kernel holds a whole SM, and its tiles
      // run early only at the cost of the preceding grid's last CTAs
      ptx::griddep_wait();
      if (pc > 0) epilogue(e_u, e_last, e_mu0, e_mu1, e_F);
      if (!more) break;
      ptx::named_bar_sync(1, 128);  // this piece's row factors are visible

      float mu0 = -INFINITY, mu1 = -INFINITY;  // reference maxima of rows lane, lane + 32
      int F = v_sc ? -126 : 0;                 // V-scale normaliser exponent
      for (int key0 = k0; key0 < k1; key0 += KT, ++it, rp.next(a.stages)) {
        const bool first = key0 == k0;
        const uint32_t stage = rp.stage;
        const uint32_t s_col = t_lane + C::S_COL + (it & 1) * NR;
        wait(&b_qk[it & 1], (it >> 1) & 1);
        ptx::tc_fence_after();

        const int key = key0 + kk;
        float ks = 1.0f, vs = 0.0f;  // vs only sets the normaliser F here; V^T carries the scale
        if (k_sc || v_sc) {
          wait(&bar_full[stage], rp.phase);
          const uint8_t* st = ring + (size_t)stage * stage_bytes;
          const float* sc = reinterpret_cast<const float*>(st + 2 * Gm::CODE_BYTES);
          const float* scv = reinterpret_cast<const float*>(st + v_sc_off);
          if (k_row) {
            ks = sc[kk];
          } else if (k_grp) {
            // the power of two the K dequant divided this key's columns by
            float mx = 0.0f;
            for (int g = 0; g < nk; ++g) mx = fmaxf(mx, sc[kk * nk + g]);
            ks = mx > 0.0f ? dev::pow2i(min(126, max(-126, dev::ceil_log2(mx)))) : 1.0f;
          }
          if (key < L) {
            if (v_row) {
              vs = scv[kk];
            } else if (v_grp) {
              for (int g = 0; g < nv; ++g) vs = fmaxf(vs, scv[kk * nv + g]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bar_empty[stage]);

        // S^T of this tile: all NR columns in one TMEM round trip (TMEM reads
        // queue behind the tensor core's accumulator traffic).  logits: y =
        // S * k_scale (the row factor alpha is applied in the exponent), or
        // the softcapped log2-domain logit (alpha = 1); masked keys -inf.
        // The S buffer is held until the tile's reference maxima are settled:
        // the slow path below reads it a second time.
        const bool full = (key0 + KT - 1 <= L - T) && (W == 0 || key0 >= L - W);
        float y[NR];
        auto logits = [&]() {
          dev::tmem_ld_cols<NR>(s_col, y);
          if (softcap > 0.0f) {
#pragma unroll
            for (int r = 0; r < NR; r += 4) {
              const float4 a4 = *reinterpret_cast<const float4*>(f_alpha + r);
              y[r] = softcap * dev::tanh_fast(y[r] * ks * a4.x * inv_cap) * kLog2e;
              y[r + 1] = softcap * dev::tanh_fast(y[r + 1] * ks * a4.y * inv_cap) * kLog2e;
              y[r + 2] = softcap * dev::tanh_fast(y[r + 2] * ks * a4.z * inv_cap) * kLog2e;
              y[r + 3] = softcap * dev::tanh_fast(y[r + 3] * ks * a4.w * inv_cap) * kLog2e;
            }
          } else if (k_sc) {
#pragma unroll
            for (int r = 0; r < NR; ++r) y[r] *= ks;
          }
          if (!full) {
#pragma unroll
            for (int r = 0; r < NR; r += 4) {
              const int4 p4 = *reinterpret_cast<const int4*>(i_pos + r);
              const int ps[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (!(key <= ps[i] && (W == 0 || key > ps[i] - W))) y[r + i] = -INFINITY;
            }
          }
        };
        // y -> the exponent z = alpha * y - mu, in place (f_mu holds -mu)
        auto to_exponent = [&]() {
#pragma unroll
          for (int r = 0; r < NR; r += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(f_mu + q * NR + r);
            const float4 a4 = softcap > 0.0f ? make_float4(1.0f, 1.0f, 1.0f, 1.0f)
                                             : *reinterpret_cast<const float4*>(f_alpha + r);
            y[r] = fmaf(y[r], a4.x, m4.x);
            y[r + 1] = fmaf(y[r + 1], a4.y, m4.y);
            y[r + 2] = fmaf(y[r + 2], a4.z, m4.z);
            y[r + 3] = fmaf(y[r + 3], a4.w, m4.w);
          }
        };
        logits();

        // ---- does any logit of the tile exceed its row's reference maximum by
        // more than 8 (P > 2^8)?  f_mu holds -mu (1e30 for a row with no key
        // yet, so that any unmasked key trips the check while a masked one
        // still gives exp2(-inf) = 0).  Only then (and on a piece's first
        // tile) are exact tile maxima taken and the references moved.
        to_exponent();
        float dm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four short chains, not one long one
#pragma unroll
        for (int r = 0; r < NR; ++r) dm[r & 3] = fmaxf(dm[r & 3], y[r]);
        const float dmax = fmaxf(fmaxf(dm[0], dm[1]), fmaxf(dm[2], dm[3]));
        const bool ovf = __any_sync(0xffffffffu, dmax > 8.0f);
        float* f_flag = f_vmax + 8 * (it & 1);  // [4] overflow flags, [4] V-scale maxima; by tile parity
        {
          const float vm = v_sc ? ptx::redux_max(vs) : 0.0f;
          if (lane == 0) {
            f_flag[q] = ovf ? 1.0f : 0.0f;
            f_flag[4 + q] = vm;
          }
        }
        ptx::named_bar_sync(1, 128);
        const bool slow = first || (f_flag[0] + f_flag[1] + f_flag[2] + f_flag[3]) > 0.0f;

        // V-scale normaliser (the dequant warps track the same F)
        float fs = 1.0f;
        if (v_sc) {
          const float vm = fmaxf(fmaxf(f_flag[4], f_flag[5]), fmaxf(f_flag[6], f_flag[7]));
          if (vm > 0.0f) {
            const int fn = min(126, max(-126, dev::ceil_log2(vm)));
            if (fn > F) {
              fs = (F - fn < -126) ? 0.0f : dev::pow2i(F - fn);
              F = fn;
            }
          }
        }
        float c0 = 1.0f, c1 = 1.0f;
        if (slow) {
          logits();  // y again, from the held S buffer
          // tile maxima per row (of y; alpha > 0 keeps the order)
#pragma unroll
          for (int r = 0; r < NR; r += 4) {
            const float t0 = ptx::redux_max(y[r]), t1 = ptx::redux_max(y[r + 1]);
            const float t2 = ptx::redux_max(y[r + 2]), t3 = ptx::redux_max(y[r + 3]);
            if (lane == 0) *reinterpret_cast<float4*>(f_red + q * NR + r) = make_float4(t0, t1, t2, t3);
          }
          ptx::named_bar_sync(1, 128);
          // reference maxima (lane holds rows lane and lane + 32) and the
          // factors that bring O and l to them
          auto update = [&](int r, float& mu, float& corr) {
            float t = fmaxf(fmaxf(f_red[r], f_red[NR + r]), fmaxf(f_red[2 * NR + r], f_red[3 * NR + r]));
            if (softcap <= 0.0f) t *= f_alpha[r];
            if (t > mu + 8.0f) {
              corr = mu == -INFINITY ? 1.0f : ptx::fast_exp2(mu - t);  // a row with no key yet holds zeros
              mu = t;
            }
          };
          if (lane < rows) update(lane, mu0, c0);
          if (lane + 32 < rows) update(lane + 32, mu1, c1);
          if (lane < NR) {
            // padding rows (zero Q, no output) get offset 0 and never trip
            f_mu[q * NR + lane] = lane >= rows ? 0.0f : (mu0 == -INFINITY ? 1e30f : -mu0);
            f_corr[q * NR + lane] = c0;
          }
          if (lane + 32 < NR) {
            f_mu[q * NR + lane + 32] = lane + 32 >= rows ? 0.0f : (mu1 == -INFINITY ? 1e30f : -mu1);
            f_corr[q * NR + lane + 32] = c1;
          }
          __syncwarp();
          to_exponent();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&b_sfree[it & 1]);  // the QK^T after next may overwrite S
        const bool need = !first && (fs != 1.0f || (slow && __any_sync(0xffffffffu, c0 != 1.0f || c1 != 1.0f)));
        if (need && !slow) {
          // only the V-scale normaliser grew: O alone is rescaled
          if (lane < NR) f_corr[q * NR + lane] = 1.0f;
          if (lane + 32 < NR) f_corr[q * NR + lane + 32] = 1.0f;
          __syncwarp();
        }

        // ---- P = exp2(z), f16, 16 rows at a time
        if (it >= 2) wait(&b_pv[it & 1], ((it - 2) >> 1) & 1);  // PV of tile it - 2 has read this buffer
        uint8_t* pbuf = p_s + (it & 1) * C::P_BYTES;
#pragma unroll
        for (int r0 = 0; r0 < NR; r0 += 16) {
          __half2 hp[8];
#pragma unroll
          for (int i = 0; i < 16; i += 2)
            hp[i / 2] = __floats2half2_rn(ptx::fast_exp2(y[r0 + i]), ptx::fast_exp2(y[r0 + i + 1]));
          uint8_t* prow = pbuf + r0 * 128;
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            *reinterpret_cast<__half*>(prow + i * 128 + p_st[i & 7]) = hp[i / 2].x;
            *reinterpret_cast<__half*>(prow + (i + 1) * 128 + p_st[(i + 1) & 7]) = hp[i / 2].y;
          }
        }
        ptx::fence_proxy_async_smem();

        // bring O and l to the new reference maxima (rare: a maximum moved by
        // more than 2^8), and O to a grown V-scale normaliser
        if (need) {
          wait(&b_pv[(it - 1) & 1], ((it - 1) >> 1) & 1);  // the previous PV has landed
          ptx::tc_fence_after();
#pragma unroll 1
          for (int hh = 0; hh <= C::NH; ++hh) {
            const uint32_t col = t_lane + (hh < C::NH ? C::O_COL + hh * NR : C::L_COL);
            const float f = hh < C::NH ? fs : 1.0f;
#pragma unroll 1
            for (int r0 = 0; r0 < NR; r0 += 16) {
              float o[16];
              dev::tmem_ld_cols<16>(col + r0, o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] *= f_corr[q * NR + r0 + i] * f;
              dev::tmem_st_cols<16>(col + r0, o);
            }
          }
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&b_pfull[it & 1]);
      }
      e_u = u;
      e_last = it - 1;
      e_mu0 = mu0;
      e_mu1 = mu1;
      e_F = F;
    }
  }

  // every role ends here; TMEM is released once no warp can touch it
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Raises (never lowers) the kernel's dynamic shared-memory limit on the
// current device, then launches one CTA per grid slot.
template <int DT, int D, int NR, bool GRP>
cudaError_t launch_decode_tc_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int grid,
                               size_t smem, cudaStream_t stream) {
  static int smem_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_set[dev] < (int)smem) {
    e = cudaFuncSetAttribute(decode_tc_kernel<DT, D, NR, GRP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set[dev] = (int)smem;
  }
  return launch_pdl(decode_tc_kernel<DT, D, NR, GRP>, grid, kTcWarps * 32, smem, stream, tk, tv, a);
}

// head_dim 256: nr 32 or 48; head_dim 128: nr 32, 48 or 64.
template <int DT, bool GRP>
cudaError_t dispatch_decode_tc(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream) {
  if (head_dim == 256) {
    if (nr == 32) return launch_decode_tc_d<DT, 256, 32, GRP>(tk, tv, a, grid, smem, stream);
    if (nr == 48) return launch_decode_tc_d<DT, 256, 48, GRP>(tk, tv, a, grid, smem, stream);
  } else if (head_dim == 128) {
    if (nr == 32) return launch_decode_tc_d<DT, 128, 32, GRP>(tk, tv, a, grid, smem, stream);
    if (nr == 48) return launch_decode_tc_d<DT, 128, 48, GRP>(tk, tv, a, grid, smem, stream);
    if (nr == 64) return launch_decode_tc_d<DT, 128, 64, GRP>(tk, tv, a, grid, smem, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
