// kvq_internal.h -- launch arguments and launchers shared between the host
// shim (api.cu) and the kernel translation units.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "kvq.h"

namespace kvq {

constexpr int kTile = 64;       // keys per pipeline stage (4 sub-tiles of 16)
constexpr int kSub = 16;        // keys per MMA sub-tile
constexpr int kMaxBatch = 1024; // sequences whose split plan fits in shared memory
constexpr int kMaxStages = 8;

// The QK-RMSNorm + RoPE prologue (kvq_norm_rope, host-validated).
struct NormRope {
  const uint16_t* w;        // bf16 bits [D] or null (no RMSNorm)
  float eps;
  const float* cos_tab;     // [max_pos, rd / 2]
  const float* sin_tab;
  const int64_t* positions; // [N] (rd > 0)
  int rd, off, interleaved, max_pos;
  int hadamard;             // Walsh-Hadamard rotation after RoPE
  float had_scale;          // fl32(1 / fl32(sqrt(D)))
};

struct AppendArgs {
  const uint16_t* k_new;  // bf16 bits [N, Hkv, D]
  const uint16_t* v_new;
  const int64_t* slots;   // [N]
  uint8_t* k_codes;
  uint8_t* v_codes;
  float* k_scale;
  float* v_scale;
  long long capacity;     // num_blocks * block_size
  int n_tokens, num_kv_heads, head_dim, block_size, log2_bs;
  int dtype, k_mode, v_mode;
  int log2_group;           // PER_GROUP sides: log2 of the channels per scale group
  unsigned int* err;
  int k_prologue;           // apply `pro` to the K rows before quantizing them
  int latent;               // LATENT layout: only the K rows are written
  NormRope pro;
};

struct NormRopeArgs {
  const uint16_t* x;        // bf16 bits [N, H, D]
  uint16_t* y;
  int n_tokens, num_heads, head_dim;
  unsigned int* err;
  NormRope pro;
};

struct DecodeArgs {
  const uint16_t* q;            // bf16 bits [B, T, Hq, D]
  const int32_t* block_table;   // [B, max_blocks_per_seq]
  const int32_t* seq_lens;      // [B]
  const float* k_scale;         // PER_ROW / PER_GROUP array or static scales
  const float* v_scale;
  int k_mode, v_mode;
  int sk_n, sv_n;     // fp32 scales per cached row of K / V: 1 PER_ROW, groups PER_GROUP, 0 static
                      // (the mma.sync kernel's group size is its instance's)
  int log2_gs;        // PER_GROUP: log2 of the channels per group (the tensor-memory kernel); else 0
  int num_blocks, block_size, log2_bs, num_kv_heads;
  int batch, num_q_heads, q_tokens, group, rows, max_blocks_per_seq, max_seq_len;
  float sm_scale, softcap;
  int window;
  int row_groups, key_warps, stages;
  int stage_stride;  // bytes between ring stages (a multiple of 1024)
  int units_max;    // partial slots (grid + batch * Hkv)
  int piece_cost;   // tiles' worth of time a CTA spends on each piece change (split planning)
  int bt_div;       // block-table row of sequence b is b / bt_div (prefill: virtual sequences)
  int v_alias;      // LATENT on the mma.sync kernel: a stage holds the K codes (and K scales) only,
                    // and V is read from them (one copy of each cache row per key)
  int early_reads;  // 1: read seq_lens, block table and q before the wait on the preceding grid
  int early_cache;  // 1: also load cache rows older than the step's new tokens before that wait
  int* plan;        // workspace: [0] cost per CTA, [1] total tiles, [2] piece cost, [3] slots, then tile prefix[B+1]
  float* part_lse;  // [units_max, rows]   base-2 log-sum-exp of each piece
  float* part_o;    // [units_max, rows, D] normalized piece output
  unsigned int* err;
};

struct CombineArgs {
  const int* plan;
  const float* part_lse;
  const float* part_o;
  const float* head_sink;  // [Hq] or null
  const float* v_scale;    // static V scale (PER_TENSOR [1] / PER_CHANNEL [Hkv, D]) or null
  int v_mode;
  uint16_t* out;           // bf16 bits [B, T, Hq, out_dim]
  float* lse_out;          // [B, T, Hq] or null
  int batch, q_tokens, num_q_heads, num_kv_heads, group, rows, head_dim;
  int out_dim;             // channels written per row: head_dim, or v_head_size (LATENT)
};

// The tensor-memory decode kernel (many query rows per kv head): 128 keys per
// stage and per MMA tile, 15 warps, and its shared-memory layout (byte offsets
// from the 1024-aligned base; the host adds 1024 bytes of alignment slack).
constexpr int kTcKeys = 128;
constexpr int kTcWarps = 15;

struct TcSmem {
  int ring, q, p, scr, pre, bars, slot, total;
};

// One stage: the K and V code rows of kTcKeys keys, then K's [kTcKeys][nk] and
// V's [kTcKeys][nv] fp32 scales (nk, nv = scales per cached row: 1 per-row,
// D / group_size per-group; a side with static scales still keeps one slot per
// key), in 1 KB multiples.
__host__ __device__ constexpr int tc_stage_stride(int row_bytes, int nk = 1, int nv = 1) {
  return (2 * kTcKeys * row_bytes + kTcKeys * 4 * ((nk > 1 ? nk : 1) + (nv > 1 ? nv : 1)) + 1023) / 1024 * 1024;
}

// ring: stages x stage stride; q: [D/64 slabs][nr rows][128 B] f16; p: two
// [2 slabs][nr rows][128 B] f16 buffers; scr: row factors, positions and the
// per-warp row maxima / reference maxima / rescale factors; pre: split plan;
// bars: mbarriers; slot: TMEM address + abort flag.
__host__ __device__ constexpr TcSmem tc_smem_layout(int head_dim, int row_bytes, int nr, int stages, int batch,
                                                    int stage_stride) {
  TcSmem s{};
  s.ring = 0;
  s.q = stages * stage_stride;
  s.p = s.q + nr * 2 * head_dim;
  s.scr = s.p + 2 * nr * 2 * kTcKeys;
  s.pre = s.scr + (2 * nr + 3 * 4 * nr + 16) * 4;
  s.bars = (s.pre + (batch + 5) * 4 + 7) / 8 * 8;
  s.slot = s.bars + (2 * stages + 24) * 8;
  s.total = s.slot + 16;
  return s;
}

// The query-tile kernel (query rows as the MMA's M dimension: a prefill
// chunk's tokens x the GQA group, up to 128 rows per kv head): 64-key stages
// (the mma.sync kernel's ring), 14 warps, f16 K and V tiles double-buffered in
// shared memory.  Byte offsets from the 1024-aligned base.
constexpr int kQtWarps = 15;
constexpr int kQtRows = 128;

struct QtSmem {
  int ring, kf, vf, sc, pre, bars, slot, total;
};

// ring: stages x stage stride; kf, vf: two [D/64 slabs][kTile keys][128 B] f16
// tiles each; sc: four [kTile] K scales and four V-normaliser exponents (the
// per-row scales a tile's softmax needs, copied out of the stage so that the
// stage is released early); pre: split plan; bars: mbarriers; slot: TMEM
// address + abort flag.
__host__ __device__ constexpr QtSmem qt_smem_layout(int head_dim, int stages, int batch, int stage_stride) {
  QtSmem s{};
  s.ring = 0;
  s.kf = stages * stage_stride;
  s.vf = s.kf + 2 * (head_dim / 64) * kTile * 128;
  s.sc = s.vf + 2 * (head_dim / 64) * kTile * 128;
  s.pre = s.sc + 4 * kTile * 4 + 4 * 4;
  s.bars = (s.pre + (batch + 5) * 4 + 7) / 8 * 8;
  s.slot = s.bars + (2 * stages + 16) * 8;
  s.total = s.slot + 16;
  return s;
}

// Launches a kernel with programmatic stream serialization: it may start while
// the previous kernel on the stream finishes, and every kvq kernel waits
// (griddepcontrol.wait) before its first global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_norm_rope(const NormRopeArgs& a, cudaStream_t stream);
// The bounded-wait check: one wait that runs out after limit_ns.
cudaError_t launch_wait_probe(unsigned int* err, unsigned long long limit_ns, cudaStream_t stream);
// warp_rows: one warp per output row (many rows of few pieces: a prefill
// chunk, a ragged decode batch) instead of one CTA per row.
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream, bool warp_rows = false);
// out[b * n + j] = max(0, seq_lens[b] - C + T (j + 1)) for the n = C / T groups
// of a prefill chunk (virtual sequences of T tokens).
cudaError_t launch_prefill_lens(const int32_t* seq_lens, int32_t* out, int batch, int n, int C, int T,
                                cudaStream_t stream);
cudaError_t launch_decode_int8(int head_dim, int nt, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeArgs& a, int grid, int threads, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_fp8(int head_dim, int nt, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeArgs& a, int grid, int threads, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_int4(int head_dim, int nt, const CUtensorMap& tk, const CUtensorMap& tv,
                               const DecodeArgs& a, int grid, int threads, size_t smem, cudaStream_t stream);

// Tensor-memory layout for nr padded query rows (32, 48; 64 with head_dim 128).
cudaError_t launch_decode_tc_int8(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_tc_fp8(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                 const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_tc_int4(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream);
// The same with group-wise scales on either side.
cudaError_t launch_decode_tc_grp_int8(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                      const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_tc_grp_fp8(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                     const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_tc_grp_int4(int head_dim, int nr, const CUtensorMap& tk, const CUtensorMap& tv,
                                      const DecodeArgs& a, int grid, size_t smem, cudaStream_t stream);

// The query-tile kernel (head_dim 128 or 256; no group-wise scales).
cudaError_t launch_decode_qt_int8(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                  int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_qt_fp8(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                 int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_decode_qt_int4(int head_dim, const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                  int grid, size_t smem, cudaStream_t stream);

cudaError_t occupancy_decode_int8(int head_dim, int nt, int threads, size_t smem, int* blocks_per_sm);
cudaError_t occupancy_decode_fp8(int head_dim, int nt, int threads, size_t smem, int* blocks_per_sm);
cudaError_t occupancy_decode_int4(int head_dim, int nt, int threads, size_t smem, int* blocks_per_sm);

}  // namespace kvq
