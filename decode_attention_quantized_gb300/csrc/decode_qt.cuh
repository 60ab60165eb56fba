// decode_qt.cuh -- attention of many query rows per kv head over the quantized
// paged cache on the tcgen05 tensor cores, with the query rows as the MMA's M
// dimension: the tiled kernel of a prefill chunk (kv-quant-attn page,
// "Requirements and limits": prefill wants a tiled attention kernel; chunked
// prefill over the paged cache, onnxruntime PR #29912 and PR #32515 testing).
//
// A work unit is one (sequence, kv head) of up to 128 query rows, row r =
// token t * G + head g of the GQA group, token t seeing the keys up to its own
// position (causal within the chunk) and the window.  Same split plan,
// producer, 64-key stage layout and partial format as decode.cuh:
//
//   S [128 rows x 64 keys] = Q [128 x D] . K [64 x D]^T    A = Q in TMEM, B = K (f16, shared, K-major)
//   O [128 rows x D]    (+)= P [128 x 64] . V [64 x D]      A = P in TMEM, B = V (f16, shared, MN-major)
//
// Each key tile's codes are dequantized once into f16 tiles in shared memory
// (double-buffered, the 128-byte swizzle); one byte layout -- key rows of
// 128-byte, 64-channel slabs -- serves K as a K-major B operand and V as an
// MN-major one.  The softmax is one thread per query row: its row of S comes
// out of TMEM whole (and the S buffer is released at once, so QK^T of the
// next tile can run while the softmax works), its running maximum and sum
// stay in registers, and its weights P go back to TMEM (two buffers) as the A
// operand of PV.  Shared memory carries only the code stages and the f16
// tiles: with 128 rows per tile the kernel is bound by shared-memory
// bandwidth (the dequant warps' reads and writes and the MMAs' B operands).
//
// Warp roles (15 warps, 480 threads):
//   0-3   softmax, row 32 w + lane: the piece's Q (per-channel K scale folded
//         in, a power-of-two normaliser per row) into TMEM; S -> P with lazy
//         row maxima (exact maxima and an O rescale only when a row's maximum
//         grows by more than 2^8); the epilogue of each piece
//   4-7   K dequant, key 32 (w & 1) + lane of the tile, channel half w >> 1
//   8-11  V dequant, the same split; a per-row V scale is folded in as
//         vs / 2^F, F the power of two at or above the piece's largest so far
//   12    TMA producer of the code stages (shared with decode.cuh)
//   13    TMEM allocation; issues QK^T
//   14    issues PV (as soon as a tile's P is written, whatever QK^T waits for)
// A warp whose 32 rows are all padding (a unit of fewer than 128 rows) does
// no softmax work: it only keeps its barrier arrivals in step.
#pragma once

#include "decode_tc.cuh"

namespace kvq {

template <int DT, int D>
struct QtCfg {
  using Gm = Geo<DT, D, kTile>;
  static constexpr int KT = kTile;
  static constexpr int SLAB = KT * 128;            // bytes of one 64-channel slab of an f16 tile
  static constexpr int TILE = (D / 64) * SLAB;     // bytes of one f16 tile (K or V)
  // TMEM columns (32-bit); lanes are query rows
  static constexpr int Q_COL = 0;                  // [128 rows x D] f16 pairs
  static constexpr int O_COL = D / 2;              // [128 rows x D] fp32
  static constexpr int NSB = D == 128 ? 2 : 1;     // S buffers (one at head_dim 256: TMEM is full)
  static constexpr int S_COL = O_COL + D;          // NSB x [128 rows x 64 keys] fp32
  static constexpr int P_COL = S_COL + NSB * KT;   // 2 x [128 rows x 64 keys] f16 pairs
  static constexpr int TMEM_COLS = 512;
  static_assert(D == 128 || D == 256, "head_dim 128 or 256");
  static_assert(P_COL + KT <= TMEM_COLS, "TMEM columns");
};

namespace dev {

// One 16-byte chunk of a key's V code row -> f16 pairs in the same order as
// k_cols (the MN-major V tile's N index); e4m3 by the NaN-free bit move
// (value * 2^-8; 2^8 is applied at the output), so that stale bytes under a
// masked key stay finite and their zero weight gives exact zeros.
template <int DT>
__device__ __forceinline__ void v_cols(const uint4 w4, uint32_t* v) {
  if constexpr (DT == KVQ_FP8_E4M3) {
    const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = f8pair(w[i], 0x1404u);
      v[2 * i + 1] = f8pair(w[i], 0x3424u);
    }
  } else {
    k_cols<DT>(w4, v);
  }
}

// Address of 16-byte f16 chunk c (K or N index 8c .. 8c + 7) of key row kk in
// an f16 tile: 64-element slabs of [KT rows][128 B], the chunk index XORed
// with kk & 7 (the tensor core's 128-byte swizzle).
template <int SLAB>
__device__ __forceinline__ uint32_t qt_chunk(uint32_t tile, int kk, int c) {
  return tile + (uint32_t)(c >> 3) * SLAB + (uint32_t)kk * 128u + ((((uint32_t)c & 7u) ^ ((uint32_t)kk & 7u)) << 4);
}

}  // namespace dev

template <int DT, int D>
__global__ void __launch_bounds__(kQtWarps * 32, 1)
    decode_qt_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const DecodeArgs a) {
  using C = QtCfg<DT, D>;
  using Gm = typename C::Gm;
  constexpr int KT = C::KT;
  constexpr int kDqK = 4, kDqV = 8, kProducer = 12, kMma = 13, kMmaPv = 14;
  constexpr int NSB = C::NSB;
  constexpr float kLog2e = 1.4426950408889634f;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* base = smem_raw + pad;
  const QtSmem lay = qt_smem_layout(D, a.stages, a.batch, a.stage_stride);
  uint8_t* ring = base + lay.ring;
  const uint32_t kf = ptx::smem_u32(base + lay.kf), vf = ptx::smem_u32(base + lay.vf);
  float* ksb = reinterpret_cast<float*>(base + lay.sc);  // [4][KT] K scales of tile it, at it & 3
  int* fexp = reinterpret_cast<int*>(ksb + 4 * KT);       // [4] V-normaliser exponent of tile it, at it & 3
  int* pl_pre = reinterpret_cast<int*>(base + lay.pre);
  int* pl_misc = pl_pre + a.batch + 1;
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(base + lay.bars);
  uint64_t* bar_empty = bar_full + a.stages;
  uint64_t* b_qk = bar_empty + a.stages;  // [NSB] QK^T of tile it complete: S buffer it % NSB written
  uint64_t* b_sfree = b_qk + 2;           // [NSB] that S buffer read by the softmax warps
  uint64_t* b_kfree = b_qk + 4;           // [2] QK^T of tile it complete: K tile it & 1 free
  uint64_t* b_kfull = b_qk + 6;           // [2] K f16 tile written
  uint64_t* b_vfull = b_qk + 8;           // [2] V f16 tile written
  uint64_t* b_pfull = b_qk + 10;          // [2] P of tile it written to P buffer it & 1 (and O rescaled)
  uint64_t* b_pv = b_qk + 12;             // [2] PV of tile it complete: P buffer and V tile it & 1 free
  uint64_t* b_qfull = b_qk + 14;          // Q of a piece in TMEM
  uint64_t* b_ksc = b_qk + 15;            // [4] K scales of tile it in ksb slot it & 3 (per-row K)
  uint64_t* b_fx = b_qk + 19;             // [4] V normaliser of tile it in fexp slot it & 3 (per-row V)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + lay.slot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      ptx::mbar_init(&bar_full[s], 1);
      ptx::mbar_init(&bar_empty[s], 8);  // K and V dequant warps
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&b_qk[i], 1);
      ptx::mbar_init(&b_sfree[i], 4);
      ptx::mbar_init(&b_kfree[i], 1);
      ptx::mbar_init(&b_kfull[i], 4);
      ptx::mbar_init(&b_vfull[i], 4);
      ptx::mbar_init(&b_pfull[i], 4);
      ptx::mbar_init(&b_pv[i], 1);
    }
    ptx::mbar_init(b_qfull, 4);
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(&b_ksc[i], 2);  // the two K warps of channel half 0
      ptx::mbar_init(&b_fx[i], 1);   // the first V warp
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kMma) {
    ptx::tmem_alloc(tmem_slot, C::TMEM_COLS);
    ptx::tc_fence_before();
  }
  const Slice<KT> sp = build_slice<KT>(a, pl_pre, pl_misc);
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Bounded wait: after a timeout every later wait of the CTA is skipped, the
  // results are flagged, and the CTA reaches its end.
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    if (!ptx::mbar_try_wait(bar, parity)) dev::wait_or_abort(bar, parity, abort_flag, a.err);
  };
  const bool k_row = a.k_mode == KVQ_SCALE_PER_ROW, v_row = a.v_mode == KVQ_SCALE_PER_ROW;

  if (warp == kProducer) {
    // ============================================================ producer
    produce<Gm, false>(a, sp, &tmk, &tmv, ring, bar_full, bar_empty, pl_pre, pl_misc);
  } else if (warp >= kDqK && warp < kDqV + 4) {
    // ==================================================== K and V dequant
    // thread: key kk of the tile, channel half hf; its code chunks are read
    // and converted before the wait for the MMA that frees the f16 tile, so
    // only the shared stores follow that wait
    const bool is_v = warp >= kDqV;
    const int q = warp - (is_v ? kDqV : kDqK);
    const int kk = 32 * (q & 1) + lane, hf = q >> 1;
    constexpr int HB = Gm::DP / 2;                  // code bytes of a channel half
    constexpr int NCC = HB / 16;                    // 16-byte code chunks of a half
    constexpr int CW = DT == KVQ_INT4 ? 16 : 8;     // f16 pairs per code chunk
    const uint32_t f16_base = is_v ? vf : kf;
    uint64_t* b_free = is_v ? b_pv : b_kfree;
    uint64_t* b_full = is_v ? b_vfull : b_kfull;
    const uint32_t code_off = is_v ? (uint32_t)Gm::CODE_BYTES : 0u;
    uint32_t it = 0;
    RingPos rp;
    for (int gt = sp.t_begin, next; gt < sp.t_end; gt = next) {
      int b, h, k0, k1, L, u;
      sp.piece(a, gt, b, h, k0, k1, L, u, next);
      int F = -126;  // V-scale normaliser exponent of the piece
      for (int key0 = k0; key0 < k1; key0 += KT, ++it, rp.next(a.stages)) {
        const uint32_t stage = rp.stage;
        const uint32_t buf = it & 1;
        wait(&bar_full[stage], rp.phase);
        const uint8_t* st = ring + (size_t)stage * a.stage_stride;
        uint4 w[NCC];
#pragma unroll
        for (int j = 0; j < NCC; ++j) {
          const uint32_t byte = (uint32_t)(hf * HB + 16 * j);
          w[j] = *reinterpret_cast<const uint4*>(st + code_off + (byte / Gm::SPAN) * (KT * Gm::SPAN) +
                                                 dev::swz<Gm::SPAN>((uint32_t)kk * Gm::SPAN + byte % Gm::SPAN));
        }
        // this key's per-row scale, and (V) the tile's largest before the
        // sequence end; then the stage goes back to the producer
        float sc = 0.0f, vm = 0.0f;
        if (is_v ? v_row : k_row) {
          const float* scp = reinterpret_cast<const float*>(st + 2 * Gm::CODE_BYTES + (is_v ? KT * 4 : 0));
          sc = scp[kk];
          if (is_v) {
            if (key0 + lane < L) vm = scp[lane];
            if (key0 + 32 + lane < L) vm = fmaxf(vm, scp[32 + lane]);
          }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bar_empty[stage]);
        uint32_t s2 = 0;
        if (is_v && v_row) {
          vm = ptx::redux_max(vm);
          if (vm > 0.0f) F = max(F, min(126, max(-126, dev::ceil_log2(vm))));
          const float s = key0 + kk < L ? sc * dev::pow2i(-F) : 0.0f;
          s2 = dev::pack_h2(s, s);
          // F of this tile for the softmax warps, before the conversion and
          // the wait for the V tile: the softmax needs the normaliser, not
          // the tile.  Slot it & 3 was last read by the softmax of tile
          // it - 4, which finished before the PV of tile it - 3 that this
          // warp waited for on its previous tile.
          if (q == 0) {
            if (lane == 0) fexp[it & 3] = F;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&b_fx[it & 3]);
          }
        }
        uint32_t v[NCC * CW];
#pragma unroll
        for (int j = 0; j < NCC; ++j) {
          if (is_v) dev::v_cols<DT>(w[j], v + CW * j);
          else dev::k_cols<DT>(w[j], v + CW * j);
        }
        if (is_v && v_row) {
#pragma unroll
          for (int m = 0; m < NCC * CW; ++m) v[m] = ptx::hmul2_u32(v[m], s2);
        }
        if (it >= 2) wait(&b_free[buf], ((it - 2) >> 1) & 1);  // the MMA two tiles back has read this tile
        const uint32_t tile = f16_base + buf * C::TILE;
#pragma unroll
        for (int c = 0; c < NCC * CW / 4; ++c) {
          const uint32_t addr = dev::qt_chunk<C::SLAB>(tile, kk, hf * (D / 16) + c);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[4 * c]), "r"(v[4 * c + 1]),
                       "r"(v[4 * c + 2]), "r"(v[4 * c + 3])
                       : "memory");
        }
        // the softmax of tile `it` reads the K scales in slot it & 3 after
        // b_ksc; the slot was last read by the softmax of tile it - 4, which
        // completed before the MMA two tiles back that this warp waited for,
        // so the slot's barrier is never more than one phase ahead of its reader
        if (hf == 0 && !is_v && k_row) ksb[(it & 3) * KT + kk] = sc;
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&b_full[buf]);
          if (!is_v && k_row && hf == 0) ptx::mbar_arrive(&b_ksc[it & 3]);
        }
      }
    }
  } else if (warp == kMma || warp == kMmaPv) {
    // ================================================================ MMA
    // Warp kMma issues QK^T of every tile (A = Q in TMEM, B = the K tile),
    // warp kMmaPv its PV (A = P, B = the V tile); one elected lane of each
    // converged warp issues.  A piece's first PV overwrites O: the softmax
    // warps read the previous piece's O before they release that tile's P.
    constexpr uint32_t idesc_qk = ptx::idesc_f16_f32(128, KT);
    constexpr uint32_t idesc_pv = ptx::idesc_f16_f32(128, D) | (1u << 16);  // B MN-major
    const uint64_t kd = ptx::smem_desc_sw128(kf);
    const uint32_t k_lo = (uint32_t)kd, d_hi = (uint32_t)(kd >> 32);
    const uint32_t v_lo = (uint32_t)ptx::smem_desc_sw128_mn(vf, C::SLAB);
    const bool qk_warp = warp == kMma;
    // PV of tile j (A = P, B = its V tile); the first of a piece overwrites O
    auto issue_pv = [&](uint32_t j, bool first) {
      const uint32_t buf = j & 1;
      wait(&b_pfull[buf], (j >> 1) & 1);
      wait(&b_vfull[buf], (j >> 1) & 1);
      __syncwarp();
      ptx::tc_fence_after();
      ptx::mma_f16_ts_x4_step(tmem + C::O_COL, tmem + C::P_COL + (KT / 2) * buf, 8, v_lo + buf * (C::TILE >> 4),
                              (16 * 128) >> 4, d_hi, idesc_pv, first ? 0u : 1u);
      ptx::mma_commit(&b_pv[buf]);
    };
    uint32_t it = 0;
    int pc = 0;
    for (int gt = sp.t_begin, next; gt < sp.t_end; gt = next, ++pc) {
      int b, h, k0, k1, L, u;
      sp.piece(a, gt, b, h, k0, k1, L, u, next);
      for (int key0 = k0; key0 < k1; key0 += KT, ++it) {
        const bool first = key0 == k0;
        const uint32_t buf = it & 1;
        if (qk_warp) {
          const uint32_t sb = it % NSB;
          if (first) wait(b_qfull, pc & 1);
          wait(&b_kfull[buf], (it >> 1) & 1);
          if (it >= NSB) wait(&b_sfree[sb], ((it - NSB) / NSB) & 1);  // the softmax has read that S buffer
          __syncwarp();
          ptx::tc_fence_after();
#pragma unroll 1
          for (int sl = 0; sl < D / 64; ++sl)
            ptx::mma_f16_ts_x4(tmem + C::S_COL + KT * sb, tmem + C::Q_COL + 32 * sl, 8,
                               k_lo + ((buf * C::TILE + sl * C::SLAB) >> 4), d_hi, idesc_qk, sl > 0 ? 1u : 0u);
          ptx::mma_commit(&b_qk[sb]);
          ptx::mma_commit(&b_kfree[buf]);
        } else {
          issue_pv(it, first);
        }
      }
    }
    if (it > 0) {
      // every MMA this warp issued has completed before TMEM can be released
      const uint32_t last = it - 1;
      uint64_t* done = qk_warp ? &b_kfree[last & 1] : &b_pv[last & 1];
      if (!ptx::mbar_wait_bounded(done, (last >> 1) & 1) && lane == 0) atomicOr(a.err, KVQ_DEVERR_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ============================================================ softmax
    const int q = warp;
    const int r = 32 * q + lane;  // query row = TMEM lane
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q) << 16);
    const int G = a.group, T = a.q_tokens, Hq = a.num_q_heads, W = a.window, rows = a.rows;
    const float softcap = a.softcap;
    const float inv_cap = softcap > 0.0f ? 1.0f / softcap : 0.0f;
    const bool valid = r < rows;
    const bool pad_warp = 32 * q >= rows;  // every row of this warp is padding
    const int t_row = valid ? dev::div_small(r, __frcp_rn((float)G)) : 0;

    // Epilogue of a piece: O out of TMEM 16 columns at a time, normalized,
    // to the workspace with the base-2 log-sum-exp.
    auto epilogue = [&](int u, uint32_t last, float mu, float l, int F) {
      wait(&b_pv[last & 1], (last >> 1) & 1);
      if (pad_warp) return;
      ptx::tc_fence_after();
      float to_true = v_row ? dev::pow2i(F) : 1.0f;
      if constexpr (DT == KVQ_FP8_E4M3) to_true *= 256.0f;
      const float inv = l > 0.0f ? to_true / l : 0.0f;
      if (valid) a.part_lse[(size_t)u * rows + r] = l > 0.0f ? mu + ptx::fast_log2(l) : -INFINITY;
      float* dst = a.part_o + ((size_t)u * rows + r) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 16) {
        float o[16];
        dev::tmem_ld_cols<16>(t_lane + C::O_COL + c0, o);
        if (!valid) continue;
        float x[16];
        if constexpr (DT == KVQ_INT4) {
          // N index 8 i + 2 m + e holds channel 8 i + m + 4 e, odd m times 16
#pragma unroll
          for (int g8 = 0; g8 < 2; ++g8)
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const float cf = (m & 1) ? dev::odd_channel_factor<DT>() : 1.0f;
              x[8 * g8 + m] = o[8 * g8 + 2 * m] * inv * cf;
              x[8 * g8 + m + 4] = o[8 * g8 + 2 * m + 1] * inv * cf;
            }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) x[i] = o[i] * inv;
        }
#pragma unroll
        for (int i = 0; i < 16; i += 4) *reinterpret_cast<float4*>(dst + c0 + i) = make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
      }
      ptx::tc_fence_before();
    };

    uint32_t it = 0;
    int pc = 0;
    int e_u = 0, e_F = 0;  // the previous piece, for its epilogue
    uint32_t e_last = 0;
    float e_mu = 0.0f, e_l = 0.0f;
    float alpha = 1.0f;
    int pos = -1;
    for (int gt = sp.t_begin, next = 0;; gt = next, ++pc) {
      const bool more = gt < sp.t_end;
      int b = 0, h = 0, k0 = 0, k1 = 0, L = 0, u = 0;
      if (more) sp.piece(a, gt, b, h, k0, k1, L, u, next);

      // ---- Q of this piece (every QK^T of the previous piece has completed:
      // this thread waited for its last S): the per-channel K scale folded in
      // under a power-of-two normaliser, the row normalised by the power of
      // two at or above its maximum, f16 pairs in the K order of the K tile.
      if (more && !pad_warp) {
        const bool kc = a.k_mode == KVQ_SCALE_PER_CHANNEL;
        const uint16_t* src = a.q + (((size_t)b * T + t_row) * Hq + (size_t)h * G + (r - t_row * G)) * D;
        const float* ksp = a.k_scale + (size_t)h * D;
        int ek = 0;
        if (kc) {
          // the largest per-channel K scale: a warp-wide maximum (one round trip)
          float km = 0.0f;
#pragma unroll
          for (int c = 4 * lane; c < D; c += 128) {
            const float4 s4 = __ldg(reinterpret_cast<const float4*>(ksp + c));
            km = fmaxf(fmaxf(km, fmaxf(fabsf(s4.x), fabsf(s4.y))), fmaxf(fabsf(s4.z), fabsf(s4.w)));
          }
          km = ptx::redux_max(km);
          ek = km > 0.0f ? min(126, max(-126, dev::ceil_log2(km))) : 0;
        }
        const float sk = dev::pow2i(-ek);
        // one 8-channel chunk of the row (raw bf16 pairs), the K scale folded in
        auto unpack = [&](const uint4 raw, int c8, float (&qv)[8]) {
          const uint32_t ww[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[2 * j] = __uint_as_float(ww[j] << 16);
            qv[2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
          }
          if (kc) {
            const float4 s0 = __ldg(reinterpret_cast<const float4*>(ksp + 8 * c8));
            const float4 s1 = __ldg(reinterpret_cast<const float4*>(ksp + 8 * c8 + 4));
            qv[0] *= s0.x * sk; qv[1] *= s0.y * sk; qv[2] *= s0.z * sk; qv[3] *= s0.w * sk;
            qv[4] *= s1.x * sk; qv[5] *= s1.y * sk; qv[6] *= s1.z * sk; qv[7] *= s1.w * sk;
          }
        };
        // the row's maximum: its chunks loaded in batches of 16 (every load
        // of a batch in flight at once; the row sits in L2, pulled there by
        // the producer while the previous piece ran)
        constexpr int NCH8 = D / 8, BAT = NCH8 < 16 ? NCH8 : 16;
        float qm = 0.0f;
#pragma unroll 1
        for (int c0 = 0; c0 < NCH8; c0 += BAT) {
          uint4 raw[BAT];
#pragma unroll
          for (int i = 0; i < BAT; ++i) raw[i] = valid ? ptx::ldg_nc_v4(src + 8 * (c0 + i)) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int i = 0; i < BAT; ++i) {
            float qv[8];
            unpack(raw[i], c0 + i, qv);
#pragma unroll
            for (int j = 0; j < 8; ++j) qm = fmaxf(qm, fabsf(qv[j]));
          }
        }
        const int eq = qm > 0.0f ? min(126, max(-126, dev::ceil_log2(qm))) : 0;
        const float sq = dev::pow2i(-eq);
        // again (cached now), normalised and packed, 32 channels per TMEM store
#pragma unroll 1
        for (int c32 = 0; c32 < D / 32; ++c32) {
          uint4 raw[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) raw[i] = valid ? ptx::ldg_nc_v4(src + 8 * (4 * c32 + i)) : make_uint4(0, 0, 0, 0);
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float qv[8];
            unpack(raw[i], 4 * c32 + i, qv);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              if constexpr (DT == KVQ_INT4) {
                const float f = (m & 1) ? sq * dev::odd_channel_factor<DT>() : sq;  // channels m, m + 4
                w[4 * i + m] = dev::pack_h2(qv[m] * f, qv[m + 4] * f);
              } else {
                w[4 * i + m] = dev::pack_h2(qv[2 * m] * sq, qv[2 * m + 1] * sq);
              }
            }
          }
          ptx::tmem_st16(t_lane + C::Q_COL + 16 * c32, w);
        }
        ptx::tmem_wait_st();
        float base = a.sm_scale;
        if (a.k_mode == KVQ_SCALE_PER_TENSOR) base *= a.k_scale[0];
        if (softcap <= 0.0f) base *= kLog2e;
        // alpha = base * 2^(ek + eq) in two exact power-of-two steps, finite
        // and > 0 (so that alpha * -inf stays -inf)
        const int e = ek + eq, e1 = e / 2;
        alpha = valid ? fmaxf(fminf(base * dev::pow2i(e1) * dev::pow2i(e - e1), 3.4028234e38f), 1e-30f) : 1.0f;
        pos = valid ? L - T + t_row : -1;
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(b_qfull);
      } else if (more) {
        // padding rows: their Q (and so S, P and O) is never read
        if (lane == 0) ptx::mbar_arrive(b_qfull);
      }
      if (pc > 0) {
        // the previous piece's tiles may have run while the preceding grid
        // finished; the workspace is written only after it
        ptx::griddep_wait();
        epilogue(e_u, e_last, e_mu, e_l, e_F);
      }
      if (!more) break;

      float mu = -INFINITY;         // reference maximum of this row (log2 units)
      float l0 = 0.0f, l1 = 0.0f;   // its weight sum, in two halves (even and odd keys)
      int F = -126;                 // V-scale normaliser exponent
      for (int key0 = k0; key0 < k1; key0 += KT, ++it) {
        const bool first = key0 == k0;
        const uint32_t buf = it & 1, sb = it % NSB;
        wait(&b_qk[sb], (it / NSB) & 1);
        if (pad_warp) {
          // rows past the unit: no S, no P (their O rows are never read);
          // the arrivals follow the same waits as everyone else's, so that
          // each barrier phase still collects one arrival per warp
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&b_sfree[sb]);
          if (it >= 2) wait(&b_pv[buf], ((it - 2) >> 1) & 1);
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(&b_pfull[buf]);
          continue;
        }
        ptx::tc_fence_after();
        float y[KT];
        dev::tmem_ld_cols<KT>(t_lane + C::S_COL + KT * sb, y);

        // logits in log2 units: y = S * k_scale * alpha (softcapped), masked
        // keys -inf; the products two at a time (f32x2)
        if (k_row) {
          wait(&b_ksc[it & 3], (it >> 2) & 1);
          const float* ksc = ksb + (it & 3) * KT;
          const float am = softcap > 0.0f ? 1.0f : alpha;
#pragma unroll
          for (int k = 0; k < KT; k += 4) {
            const float4 s4 = *reinterpret_cast<const float4*>(ksc + k);
            float a0, a1, a2, a3;
            ptx::mul_x2(a0, a1, s4.x, s4.y, am, am);
            ptx::mul_x2(a2, a3, s4.z, s4.w, am, am);
            ptx::mul_x2(y[k], y[k + 1], y[k], y[k + 1], a0, a1);
            ptx::mul_x2(y[k + 2], y[k + 3], y[k + 2], y[k + 3], a2, a3);
          }
        } else if (softcap <= 0.0f) {
#pragma unroll
          for (int k = 0; k < KT; k += 2) ptx::mul_x2(y[k], y[k + 1], y[k], y[k + 1], alpha, alpha);
        }
        // S is in registers and the K scales are read: the buffer may take
        // the QK^T two tiles on
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&b_sfree[sb]);
        if (softcap > 0.0f) {
          const float ac = alpha * inv_cap;
#pragma unroll
          for (int k = 0; k < KT; ++k) y[k] = softcap * dev::tanh_fast(y[k] * ac) * kLog2e;
        }
        float fs = 1.0f;  // growth of the V-scale normaliser
        if (v_row) {
          wait(&b_fx[it & 3], (it >> 2) & 1);  // this tile's V normaliser is in fexp
          const int fn = fexp[it & 3];
          if (fn > F) {
            fs = (F - fn < -126) ? 0.0f : dev::pow2i(F - fn);
            F = fn;
          }
        }
        const bool full = key0 + KT - 1 <= pos && (W == 0 || key0 > pos - W);
        if (!full) {
#pragma unroll
          for (int k = 0; k < KT; ++k) {
            const int key = key0 + k;
            if (!(key <= pos && (W == 0 || key > pos - W))) y[k] = -INFINITY;
          }
        }
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int k = 0; k < KT; k += 4) {
          mx0 = ptx::max3(mx0, y[k], y[k + 1]);
          mx1 = ptx::max3(mx1, y[k + 2], y[k + 3]);
        }
        const float m = fmaxf(mx0, mx1);
        // move the reference only when the tile's maximum exceeds it by more
        // than 8 (P <= 2^8 in f16); a row with no key yet holds zeros in O
        float corr = 1.0f;
        bool resc = false;
        if (m > mu + 8.0f) {
          if (mu != -INFINITY) {
            corr = ptx::fast_exp2(mu - m);
            resc = !first;
          }
          mu = m;
        }
        l0 *= corr;
        l1 *= corr;
        resc = resc || (fs != 1.0f && !first);
        // P = exp2(y - mu), f16 pairs; the sums take the fp32 weights
        const float nmu = mu == -INFINITY ? 0.0f : -mu;
        uint32_t p[KT / 2];
#pragma unroll
        for (int k = 0; k < KT; k += 2) {
          float z0, z1;
          ptx::add_x2(z0, z1, y[k], y[k + 1], nmu, nmu);
          const float e0 = ptx::fast_exp2(z0), e1 = ptx::fast_exp2(z1);
          ptx::add_x2(l0, l1, l0, l1, e0, e1);
          p[k / 2] = dev::pack_h2(e0, e1);
        }
        // this tile's P buffer is free once the PV two tiles back has landed
        if (it >= 2) wait(&b_pv[buf], ((it - 2) >> 1) & 1);
        if (__any_sync(0xffffffffu, resc)) {
          // bring this warp's rows of O to the new reference and normaliser
          // (after the previous PV has landed)
          wait(&b_pv[(it - 1) & 1], ((it - 1) >> 1) & 1);
          ptx::tc_fence_after();
          const float f = resc ? corr * fs : 1.0f;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 16) {
            float o[16];
            dev::tmem_ld_cols<16>(t_lane + C::O_COL + c0, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= f;
            dev::tmem_st_cols<16>(t_lane + C::O_COL + c0, o);
          }
        }
        ptx::tmem_st16(t_lane + C::P_COL + (KT / 2) * buf, *reinterpret_cast<uint32_t(*)[16]>(p));
        ptx::tmem_st16(t_lane + C::P_COL + (KT / 2) * buf + 16, *reinterpret_cast<uint32_t(*)[16]>(p + 16));
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&b_pfull[buf]);
      }
      e_u = u;
      e_last = it - 1;
      e_mu = mu;
      e_l = l0 + l1;
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
template <int DT, int D>
cudaError_t launch_decode_qt_d(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int grid,
                               size_t smem, cudaStream_t stream) {
  static int smem_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (smem_set[dev] < (int)smem) {
    e = cudaFuncSetAttribute(decode_qt_kernel<DT, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    smem_set[dev] = (int)smem;
  }
  return launch_pdl(decode_qt_kernel<DT, D>, grid, kQtWarps * 32, smem, stream, tk, tv, a);
}

template <int DT>
cudaError_t dispatch_decode_qt(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                               int grid, size_t smem, cudaStream_t stream) {
  if (head_dim == 256) return launch_decode_qt_d<DT, 256>(tk, tv, a, grid, smem, stream);
  if (head_dim == 128) return launch_decode_qt_d<DT, 128>(tk, tv, a, grid, smem, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
