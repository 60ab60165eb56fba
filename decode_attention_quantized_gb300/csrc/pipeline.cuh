// pipeline.cuh -- the parts every decode kernel shares: the geometry of a
// shared-memory stage of quantized code rows, the tile-balanced split plan
// that each CTA builds from seq_lens, the walk over the pieces of a CTA's
// slice, and the producer warp that streams code pages through a ring of
// mbarrier-guarded stages with TMA.
//
// Split-KV over a paged cache: PagedAttention paged decode (onnxruntime PR
// #29912, Summary of Changes: split-KV, block-table aware); one block owns a
// (batch, kv head) key range and partials are merged in a fixed order
// (kv-quant-attn page, section "Method").
#pragma once

#include "kvq_internal.h"
#include "ptx.cuh"

namespace kvq {

constexpr int round_up_c(int x, int m) { return (x + m - 1) / m * m; }

// One stage holds KT keys: the K code rows, then the V code rows, each as
// SLABS column slabs of [KT rows][SPAN bytes] in the TMA swizzle, then KT K
// scales and KT V scales (fp32, per-row mode only).  STAGE_STRIDE always
// leaves room for the scales (the tensor-memory kernel's ring); the mma.sync
// kernel and the producer step by DecodeArgs::stage_stride, which the host
// sizes without the scale area when neither side has per-row scales.
template <int DT, int D_, int KT = kTile>
struct Geo {
  static constexpr int D = D_;
  static constexpr int DP = DT == KVQ_INT4 ? D_ / 2 : D_;  // bytes per cached row
  // TMA box inner bytes = swizzle span: the widest of 128 / 64 / 32 bytes that
  // divides the row (a 576-byte row is nine 64-byte slabs)
  static constexpr int SPAN = DP % 128 == 0 ? 128 : (DP % 64 == 0 ? 64 : 32);
  static constexpr int SLABS = DP / SPAN;                // column slabs per row
  static constexpr int NCH = DP / 16;                    // 16-byte chunks per row
  static constexpr int NMT = D_ / 16;                      // 16-channel MMA tiles
  static constexpr int KEYS = KT;                        // keys per stage
  static constexpr int CODE_BYTES = KT * DP;             // one side of one stage
  static constexpr int STAGE_STRIDE = round_up_c(2 * CODE_BYTES + 2 * KT * 4, 1024);
};

namespace dev {

// byte offset o inside a slab of SPAN-byte rows -> swizzled offset written by
// the TMA unit (16-byte granule index XOR row-group bits 7.., period 8 rows).
template <int SPAN>
__device__ __forceinline__ uint32_t swz(uint32_t o) {
  return o ^ (((o >> 7) & (SPAN / 16 - 1)) << 4);
}

}  // namespace dev

// Ring position of a running tile counter it: stage = it mod S and the phase
// bit (it / S) & 1, kept by one add and one compare per tile instead of a
// division by the run-time stage count.
struct RingPos {
  uint32_t stage = 0, phase = 0;
  __device__ __forceinline__ void next(uint32_t S) {
    if (++stage == S) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// The split plan.  Segment s = b * Hkv + h is sequence b's key range
// [lo_b, L_b) for kv head h: n_b = ceil((L_b - lo_b) / KT) tiles.  The
// segments laid end to end in s order make `total` tiles.  Each CTA also
// pays a fixed time per piece it starts (the query prologue, the merge and
// the partial write), worth `c` tiles (DecodeArgs::piece_cost): so on a cost
// line each segment occupies its n_b tiles followed by c units of gap, and
// CTA x takes the cost range [x W, (x + 1) W), W = ceil(total cost / grid).
// A CTA whose range straddles a segment change takes c fewer tiles; c = 0 is
// the plain equal-tiles split.  The piece of segment s in CTA x writes its
// partial to slot s + x: distinct for every piece and contiguous over the
// pieces of one segment (the combine walks them in that order).
template <int KT>
struct Slice {
  const int* pre;  // shared [B + 1]: tile prefix over sequences
  int lim, t_begin, t_end;

  // key range [lo, L) of sequence b: L clamped to the capacity bound, lo the
  // first key any query row sees (window) rounded down to the tile
  __device__ __forceinline__ void seq_range(const DecodeArgs& a, int b, int& L, int& lo) const {
    L = a.seq_lens[b];
    L = L < 0 ? 0 : (L > lim ? lim : L);
    lo = 0;
    if (a.window > 0) lo = max(0, L - a.q_tokens - a.window + 1);
    lo &= ~(KT - 1);
  }

  // the piece that starts at global tile gt: sequence, kv head, key range
  // [k0, k1), sequence length, partial slot, and the global tile after it
  __device__ __forceinline__ void piece(const DecodeArgs& a, int gt, int& b, int& h, int& k0, int& k1, int& L,
                                        int& slot, int& next) const {
    const int Hkv = a.num_kv_heads;
    int lo = 0, hi = a.batch - 1;  // last b with pre[b] * Hkv <= gt (skips empty sequences)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] * Hkv <= gt) lo = mid; else hi = mid - 1;
    }
    b = lo;
    const int nb = pre[b + 1] - pre[b];
    const int off = gt - pre[b] * Hkv;
    h = off / nb;
    const int t0 = off - h * nb;
    next = min(gt - t0 + nb, t_end);
    int klo;
    seq_range(a, b, L, klo);
    k0 = klo + t0 * KT;
    k1 = min(klo + (t0 + next - gt) * KT, L);
    slot = b * Hkv + h + (int)blockIdx.x;
  }
};

// Builds the plan in shared memory (pl_pre [B + 1], pl_misc [4]); every
// thread of the CTA calls it.  It reads only seq_lens: with early_reads
// (KVQ_DECODE_EARLY_INPUTS) before the wait on the preceding grid, else after
// it; the producer publishes the plan to the workspace after that wait
// (publish_slice).  Flags seq_lens outside [0, capacity].
template <int KT>
__device__ Slice<KT> build_slice(const DecodeArgs& a, int* pl_pre, int* pl_misc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = a.batch, Hkv = a.num_kv_heads;
  const int cap = a.max_blocks_per_seq * a.block_size;
  if (!a.early_reads) ptx::griddep_wait();  // seq_lens may come from the preceding grid
  Slice<KT> sp;
  sp.pre = pl_pre;
  sp.lim = (a.max_seq_len > 0 && a.max_seq_len < cap) ? a.max_seq_len : cap;
  for (int b = tid; b < B; b += blockDim.x) {
    const int raw = a.seq_lens[b];
    if ((raw < 0 || raw > sp.lim) && blockIdx.x == 0) atomicOr(a.err, KVQ_DEVERR_SEQ_LEN);
    int L, lo;
    sp.seq_range(a, b, L, lo);
    pl_pre[b] = (max(0, L - lo) + KT - 1) / KT;  // tiles, for now
  }
  __syncthreads();
  const int c = a.piece_cost;
  if (warp == 0) {
    const int seg = (B + 31) / 32;
    const int s0 = min(B, lane * seg), s1 = min(B, s0 + seg);
    int cnt = 0;
    for (int b = s0; b < s1; ++b) cnt += pl_pre[b];
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - cnt;
    for (int b = s0; b < s1; ++b) {
      const int n = pl_pre[b];
      pl_pre[b] = run;
      run += n;
    }
    if (lane == 31) {
      const int total = incl * Hkv;
      const long long cost = total > 0 ? (long long)total + (long long)c * (B * Hkv - 1) : 0;
      pl_pre[B] = incl;
      pl_misc[0] = (int)max(1LL, (cost + gridDim.x - 1) / gridDim.x);
      pl_misc[1] = total;
      pl_misc[2] = (int)cost;
    }
  }
  __syncthreads();
  // the combine may be scheduled now; it waits for this grid to complete
  ptx::griddep_launch_dependents();
  const int W = pl_misc[0], total = pl_misc[1], cost = pl_misc[2];
  // first tile at or after cost position p
  auto tile_at = [&](long long p) -> int {
    if (p >= cost) return total;
    int lo = 0, hi = B - 1;  // last b whose first segment starts at or before p
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)pl_pre[mid] * Hkv + (long long)c * mid * Hkv <= p) lo = mid; else hi = mid - 1;
    }
    const int nb = pl_pre[lo + 1] - pl_pre[lo];
    const long long base = (long long)pl_pre[lo] * Hkv + (long long)c * lo * Hkv;
    const int h = (int)min((long long)(Hkv - 1), (p - base) / (nb + c));
    const long long off = p - base - (long long)h * (nb + c);
    return pl_pre[lo] * Hkv + h * nb + (int)min(off, (long long)nb);
  };
  sp.t_begin = tile_at((long long)blockIdx.x * W);
  sp.t_end = max(sp.t_begin, tile_at((long long)(blockIdx.x + 1) * W));
  return sp;
}

// CTA 0 copies the plan into the workspace for the combine (one warp, after
// the wait on the preceding grid: that grid may still read the workspace).
__device__ __forceinline__ void publish_slice(const DecodeArgs& a, const int* pl_pre, const int* pl_misc) {
  if (blockIdx.x != 0) return;
  const int lane = threadIdx.x & 31;
  for (int i = lane; i <= a.batch; i += 32) a.plan[4 + i] = pl_pre[i];
  if (lane == 0) {
    a.plan[0] = pl_misc[0];
    a.plan[1] = pl_misc[1];
    a.plan[2] = a.piece_cost;
    a.plan[3] = a.units_max;
  }
}

// The producer warp.  The whole warp fetches a piece's block ids 32 pages at
// a time (one coalesced load per 32 pages, the next batch loaded while the
// current one is used) and hands them to lane 0 by shuffles.  With early
// reads the first piece's ids are read before the wait on the preceding grid;
// the cache is read, and the plan published, only after it -- except, with
// early cache reads (KVQ_DECODE_EARLY_CACHE), the stages before the one that
// holds the step's new tokens.  Lane 0 waits for a free stage and issues,
// per page segment of the stage, one TMA tensor copy per (slab, side) with
// the block id as the outer coordinate, plus 1-D bulk copies of the per-row
// scales.  kBurst: the whole stage's block ids are resolved first and its
// copies go out in one unrolled burst under a single expect-tx arrival (the
// mma.sync kernel, whose stages of small pages want a short issue path).
// Otherwise the segment loop stays rolled, each segment adding its bytes to
// the transaction count, with one arrival after the last (the tensor-memory
// kernel, whose fifteen warps share four schedulers and which stalls on
// instruction fetch when its code grows).  A block id outside
// [0, num_blocks) is flagged and its rows are not loaded.  Returns after
// every copy it issued has landed, so the CTA never exits with a copy in
// flight.
template <class Gm, bool kBurst>
__device__ void produce(const DecodeArgs& a, const Slice<Gm::KEYS>& sp, const CUtensorMap* tmk,
                        const CUtensorMap* tmv, uint8_t* ring, uint64_t* bar_full, uint64_t* bar_empty,
                        const int* pl_pre, const int* pl_misc) {
  constexpr int KT = Gm::KEYS;
  const int lane = threadIdx.x & 31;
  bool waited = false;
  auto gate = [&]() {
    if (waited) return;
    ptx::griddep_wait();
    publish_slice(a, pl_pre, pl_misc);
    waited = true;
  };
  // per-row / per-group scales: nk (nv) floats per K (V) row, K's [KT][nk]
  // after the codes, V's [KT][nv] at KT * max(1, nk) floats after that.  With
  // v_alias (LATENT) a stage holds the K side only: no V codes, no V scales.
  const int nk = a.sk_n, nv = a.v_alias ? 0 : a.sv_n;
  const uint32_t sc_off = (a.v_alias ? 1 : 2) * Gm::CODE_BYTES;
  const uint32_t v_sc = sc_off + KT * 4 * (nk > 1 ? nk : 1);
  const int Hkv = a.num_kv_heads;
  const int seg_rows = min(a.block_size, kTile);  // rows of one TMA box
  const uint32_t seg_bytes = (uint32_t)seg_rows * ((a.v_alias ? 1 : 2) * Gm::DP + 4 * nk + 4 * nv);
  const uint32_t S = (uint32_t)a.stages;
  uint32_t it = 0;
  RingPos rp;
  int ok = 1;
  for (int gt = sp.t_begin, next; gt < sp.t_end; gt = next) {
    int b, h, k0, k1, L, slot;
    sp.piece(a, gt, b, h, k0, k1, L, slot, next);
    const int32_t* bt = a.block_table + (size_t)(b / a.bt_div) * a.max_blocks_per_seq;
    const int p_last = (k1 - 1) >> a.log2_bs;
    int base = k0 >> a.log2_bs;
    int my_id = base + lane <= p_last ? bt[base + lane] : -1;
    // the next 32 ids are in flight while these are used, so a batch change
    // does not stall the copies on a block-table read
    int nx_id = base + 32 + lane <= p_last ? bt[base + 32 + lane] : -1;
    // with early cache reads only the stage holding the step's new tokens
    // waits for the preceding grid (which may be writing those rows)
    if (!a.early_cache) gate();
    if (gt != sp.t_begin) {
      // the consumers read this piece's query rows once the previous piece
      // ends; the producer runs a ring ahead of them, so it pulls those rows
      // into L2 now (G heads of one kv head are contiguous per token)
      const int lines = a.group * Gm::D * 2 / 128;
      for (int i = lane; i < a.q_tokens * lines; i += 32) {
        const int t = i / lines, c = i - t * lines;
        ptx::prefetch_l2(a.q + (((size_t)b * a.q_tokens + t) * a.num_q_heads + (size_t)h * a.group) * Gm::D + c * 64);
      }
    }
    for (int key0 = k0; key0 < k1; key0 += KT, ++it, rp.next(S)) {
      const int stage = (int)rp.stage;
      if (a.early_cache && key0 + KT > L - a.q_tokens) gate();
      if (lane == 0 && it >= S && ok) {
        ok = (kBurst ? ptx::mbar_wait_bounded_inl(&bar_empty[stage], rp.phase ^ 1u)
                     : ptx::mbar_wait_bounded(&bar_empty[stage], rp.phase ^ 1u)) ? 1 : 0;
        if (!ok) atomicOr(a.err, KVQ_DEVERR_TIMEOUT);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      uint8_t* st = ring + (size_t)stage * a.stage_stride;
      const int kend = ok ? min(key0 + KT, k1) : key0;  // nothing is loaded after a timeout
      if constexpr (kBurst) {
        // the stage's block ids first (whole warp), then one burst of copies
        // from lane 0 under a single expect-tx arrival
        int blk[KT / 16];
        uint32_t bytes = 0;
  #pragma unroll
        for (int s = 0; s < KT / 16; ++s) {
          blk[s] = -1;
          const int skey = key0 + s * seg_rows;
          if (skey >= kend) continue;
          const int page = skey >> a.log2_bs;
          if (page - base >= 32) {
            base += 32;
            my_id = nx_id;
            nx_id = base + 32 + lane <= p_last ? bt[base + 32 + lane] : -1;
          }
          const int id = __shfl_sync(0xffffffffu, my_id, page - base);
          if (id < 0 || id >= a.num_blocks) {
            if (lane == 0) atomicOr(a.err, KVQ_DEVERR_BLOCK_ID);
            continue;
          }
          blk[s] = id;
          bytes += seg_bytes;
        }
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(&bar_full[stage], bytes);
  #pragma unroll
          for (int s = 0; s < KT / 16; ++s) {
            if (blk[s] < 0) continue;
            const int row0 = (key0 + s * seg_rows) & (a.block_size - 1);
  #pragma unroll
            for (int sl = 0; sl < Gm::SLABS; ++sl) {
              uint8_t* dk = st + sl * (KT * Gm::SPAN) + s * seg_rows * Gm::SPAN;
              ptx::tma_load_4d(dk, tmk, sl * Gm::SPAN, row0, h, blk[s], &bar_full[stage]);
              if (!a.v_alias)
                ptx::tma_load_4d(dk + Gm::CODE_BYTES, tmv, sl * Gm::SPAN, row0, h, blk[s], &bar_full[stage]);
            }
            const size_t srow = ((size_t)blk[s] * Hkv + h) * a.block_size + row0;
            if (nk)
              ptx::bulk_load(st + sc_off + s * seg_rows * 4 * nk, a.k_scale + srow * nk,
                             seg_rows * 4 * nk, &bar_full[stage]);
            if (nv)
              ptx::bulk_load(st + v_sc + s * seg_rows * 4 * nv, a.v_scale + srow * nv, seg_rows * 4 * nv,
                             &bar_full[stage]);
          }
        }
      } else {
#pragma unroll 1
        for (int skey = key0; skey < kend; skey += seg_rows) {
          const int page = skey >> a.log2_bs;
          if (page - base >= 32) {
            base += 32;
            my_id = nx_id;
            nx_id = base + 32 + lane <= p_last ? bt[base + 32 + lane] : -1;
          }
          const int id = __shfl_sync(0xffffffffu, my_id, page - base);
          if (lane == 0) {
            if (id < 0 || id >= a.num_blocks) {
              atomicOr(a.err, KVQ_DEVERR_BLOCK_ID);
            } else {
              const int s = (skey - key0) / seg_rows;
              const int row0 = skey & (a.block_size - 1);
              ptx::mbar_expect_tx(&bar_full[stage], seg_bytes);
#pragma unroll
              for (int sl = 0; sl < Gm::SLABS; ++sl) {
                uint8_t* dk = st + sl * (KT * Gm::SPAN) + s * seg_rows * Gm::SPAN;
                ptx::tma_load_4d(dk, tmk, sl * Gm::SPAN, row0, h, id, &bar_full[stage]);
                if (!a.v_alias)
                  ptx::tma_load_4d(dk + Gm::CODE_BYTES, tmv, sl * Gm::SPAN, row0, h, id, &bar_full[stage]);
              }
              const size_t srow = ((size_t)id * Hkv + h) * a.block_size + row0;
              if (nk)
                ptx::bulk_load(st + sc_off + s * seg_rows * 4 * nk, a.k_scale + srow * nk,
                               seg_rows * 4 * nk, &bar_full[stage]);
              if (nv)
                ptx::bulk_load(st + v_sc + s * seg_rows * 4 * nv, a.v_scale + srow * nv, seg_rows * 4 * nv,
                               &bar_full[stage]);
            }
          }
        }
        if (lane == 0) ptx::mbar_arrive(&bar_full[stage]);
      }
      __syncwarp();
    }
  }
  gate();  // (an empty slice still publishes the plan from CTA 0)
  // let every copy this warp issued land before the CTA can exit
  if (lane == 0) {
    for (uint32_t s = 0; s < S && s < it; ++s) {
      const uint32_t last = it - 1 - ((it - 1 - s) % S);
      if (!ptx::mbar_wait_bounded(&bar_full[s], (last / S) & 1)) atomicOr(a.err, KVQ_DEVERR_TIMEOUT);
    }
  }
  __syncwarp();
}

}  // namespace kvq
