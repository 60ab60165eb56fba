/*
 * kvq.h -- decode attention over a quantized, paged KV cache (GB300, sm_103a).
 *
 * A C ABI: plain structs, pointers and sizes.  Every device pointer is caller
 * owned; the library never allocates, frees, or synchronizes the stream it is
 * given (kvq_get_device_error is the one call that waits, and says so).  All
 * compute calls are asynchronous on `stream` and take their grid and workspace
 * extents from host-side shapes only, so a sequence of calls can be captured
 * in a CUDA graph.
 *
 * The operations follow these pages:
 *  - onnxruntime issue #29783 (quantized KV cache in GroupQueryAttention):
 *    per-token scales, quantize the appended token on write, dequantize on
 *    read, no fp16 copy of the past.
 *  - onnxruntime PR #29912 "[CUDA] PagedAttention: quantized KV cache, XQA
 *    decode, MLA, QK-Norm and head sink", Summary of Changes: slot_mapping,
 *    head_sink, k_scale / v_scale with PER_TENSOR / PER_CHANNEL granularity,
 *    int8 / float8e4m3fn cache types, ReshapeAndCache (quantize on write),
 *    split-KV paged decode with softcap and sliding window, ApplyHeadSink, and
 *    the attention_metadata upper bound that keeps a step capturable.
 *  - onnxruntime PR #32515 "[CUDA] Add INT4 paged KV cache with per-channel
 *    scales", Description: int4 packed two per byte, cache head dimension
 *    (head_size+1)/2, per-channel scale folded into Q and re-applied to the
 *    output, speculative decode with several query tokens.
 *  - "kv-quant-attn" page, sections "Method" and "Correctness": per-row absmax
 *    scales, one block per (batch, kv head) resolving the whole GQA group from
 *    one read, warp-private softmax state, fixed-order merge (bitwise
 *    reproducible), GQA ratio at most 8, head dimension at most 256; section
 *    "Requirements and limits": the group-wise scaling it leaves undone, here
 *    as PER_GROUP.
 *
 * Data layout (all tensors dense, row-major, innermost last):
 *   codes       uint8  [num_blocks, num_kv_heads, block_size, Dp]
 *               Dp = head_dim (int8, e4m3) or head_dim/2 (int4: channel 2j in
 *               the low nibble of byte j, channel 2j+1 in the high nibble,
 *               two's-complement nibbles)
 *   PER_ROW     scales fp32 [num_blocks, num_kv_heads, block_size]
 *   PER_TENSOR  scale  fp32 [1]
 *   PER_CHANNEL scales fp32 [num_kv_heads, head_dim]
 *   PER_GROUP   scales fp32 [num_blocks, num_kv_heads, block_size, head_dim / group_size]
 *   cache slot  s = block * block_size + row
 *   q, out      bf16   [batch, q_tokens, num_q_heads, head_dim]
 *   k_new/v_new bf16   [n_tokens, num_kv_heads, head_dim]
 *   block_table int32  [batch, max_blocks_per_seq]
 *   seq_lens    int32  [batch]   (each includes the q_tokens new tokens)
 *   lse_out     fp32   [batch, q_tokens, num_q_heads] (natural log)
 *
 * Supported on the GPU path: head_dim in {64, 128, 256}, and 576 for a LATENT
 * cache (absorbed MLA, e.g. 512 latent + 64 rotary channels) with int8 or
 * e4m3 codes and per-row, per-tensor or per-channel scales, at most 48 query
 * rows per kv head; num_q_heads a multiple of num_kv_heads with a ratio of at
 * most 8; q_tokens in [1, 8]; block_size a power of two >= 16; batch <= 1024.
 * Pointers 16-byte aligned.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_API __attribute__((visibility("default")))

/* A cudaStream_t (the same type: a pointer to the runtime's stream object);
 * NULL is the legacy default stream. */
typedef struct CUstream_st* kvq_stream_t;

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,         /* bad enum, shape, null or misaligned pointer */
  KVQ_ERR_UNSUPPORTED = 2,         /* valid, but outside what the GPU path covers */
  KVQ_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < kvq_decode_workspace_size */
  KVQ_ERR_CUDA = 4,                /* a CUDA runtime call or a launch failed */
  KVQ_ERR_DEVICE_TIMEOUT = 5       /* a bounded device-side wait gave up */
} kvq_status;

/* Cache element types (PR #29912: int8, float8e4m3fn; PR #32515: packed int4). */
typedef enum { KVQ_INT8 = 1, KVQ_FP8_E4M3 = 2, KVQ_INT4 = 3 } kvq_dtype;

/* Scale granularity: PER_ROW is one absmax scale per (token, kv head) row,
 * computed on append (kv-quant-attn "Method"; issue #29783 per-token);
 * PER_TENSOR and PER_CHANNEL are static caller-given scales (PR #29912);
 * PER_GROUP applies the PER_ROW rule to each run of kvq_cache.group_size
 * consecutive channels of a row, one scale per group (the group-wise scaling
 * the kv-quant-attn page lists under "Requirements and limits" as not done
 * there, which would narrow the int4 error around outlier channels). */
typedef enum {
  KVQ_SCALE_PER_ROW = 1,
  KVQ_SCALE_PER_TENSOR = 2,
  KVQ_SCALE_PER_CHANNEL = 3,
  KVQ_SCALE_PER_GROUP = 4
} kvq_scale_mode;

/* Device-side data violations, OR-ed into a per-device flag word.  The
 * offending access is skipped (never trapped); outputs that depend on it are
 * unspecified.  Read with kvq_get_device_error. */
#define KVQ_DEVERR_SLOT 0x1u      /* append: slot_mapping[n] >= num_blocks * block_size */
#define KVQ_DEVERR_BLOCK_ID 0x2u  /* decode: block_table entry outside [0, num_blocks) */
#define KVQ_DEVERR_SEQ_LEN 0x4u   /* decode: seq_len < 0, > capacity, or > max_seq_len */
#define KVQ_DEVERR_TIMEOUT 0x8u   /* a bounded pipeline wait gave up */
#define KVQ_DEVERR_POSITION 0x10u /* norm/RoPE prologue: position outside [0, max_position) */

/* Cache layouts (PR #29912, kv_cache_layout and v_head_size): SEPARATE K and V
 * caches, or LATENT (absorbed MLA): one cache whose rows serve as K, and whose
 * leading v_head_size channels serve as V. */
typedef enum { KVQ_LAYOUT_SEPARATE = 0, KVQ_LAYOUT_LATENT = 1 } kvq_layout;

/* The paged cache: one descriptor per layer (kv-quant-attn "Usage": one cache
 * object per layer).  All pointers are device memory owned by the caller.
 * k_scale / v_scale: PER_ROW fp32 [num_blocks, Hkv, block_size] or PER_GROUP
 * fp32 [num_blocks, Hkv, block_size, head_dim / group_size] arrays written by
 * kvq_append (16-byte aligned), or the static scales (PER_TENSOR [1],
 * PER_CHANNEL [Hkv, head_dim]; finite and > 0: the precondition the PR #447
 * scale loader checks). */
typedef struct {
  int32_t dtype;        /* kvq_dtype */
  int32_t k_mode;       /* kvq_scale_mode of K */
  int32_t v_mode;       /* kvq_scale_mode of V */
  int32_t num_blocks;   /* pool size in blocks */
  int32_t block_size;   /* tokens per block (power of two >= 16) */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_dim;     /* D */
  void* k_codes;        /* uint8 [num_blocks, Hkv, block_size, Dp] */
  void* v_codes;
  float* k_scale;
  float* v_scale;
  int32_t layout;       /* kvq_layout; LATENT: v_codes, v_scale, v_mode are ignored (V is the K
                           row, with K's scales) and may be NULL / 0; kvq_append writes K only
                           and ignores v_new; kvq_combine writes out [B, T, Hq, v_head_size] */
  int32_t v_head_size;  /* LATENT: channels of V, a multiple of 8 in [8, head_dim]; 0 = head_dim
                           (the pages' DeepSeek-V3 example: head_dim 576, v_head_size 512) */
  int32_t group_size;   /* PER_GROUP on either side: channels per scale group, 32, 64 or 128
                           and at most head_dim (one group size for both sides); otherwise
                           ignored.  Decode with a PER_GROUP side runs on the mma.sync
                           kernel's grouped layout for every query-row count. */
} kvq_cache;

/* One decode call (PagedAttention's inputs, PR #29912 Summary of Changes). */
typedef struct {
  int32_t batch;              /* B (<= 1024) */
  int32_t num_q_heads;        /* Hq; Hq / Hkv <= 8; query head i reads kv head i / (Hq/Hkv) */
  int32_t q_tokens;           /* T in [1, 8]: 1, or 1 + drafts (PR #32515, speculative
                                 decode); draft t sits at position seq_len - T + t and
                                 sees keys 0..that position (causal among drafts) */
  int32_t max_blocks_per_seq; /* block_table row length; capacity = it * block_size */
  int32_t max_seq_len;        /* host upper bound on seq_lens, like attention_metadata
                                 [max_kv_len] (PR #29912); 0 = capacity.  Sizes the grid,
                                 never read back from the device. */
  float sm_scale;             /* logit scale; <= 0 selects 1/sqrt(head_dim) */
  float softcap;              /* > 0: logit s -> softcap * tanh(s / softcap); 0 = off */
  int32_t window;             /* > 0: keep the `window` most recent keys up to and
                                 including the query position; 0 = off */
  uint32_t flags;             /* KVQ_DECODE_* bits below; 0 = the defaults */
} kvq_decode_params;

/* kvq_decode_params.flags.
 *
 * KVQ_DECODE_EARLY_INPUTS: every kvq kernel may start while the kernel enqueued
 * just before it on the stream finishes (programmatic dependent launch).  By
 * default kvq_decode reads nothing until that preceding kernel has completed.
 * With this bit it reads q, block_table, seq_lens and the static scales
 * (PER_TENSOR / PER_CHANNEL) while the preceding kernel is still running, and
 * waits only before it reads the cache and writes the workspace: the split plan
 * and the query prologue then overlap that kernel's tail.  Set it only when
 * none of those inputs is written by the operation enqueued just before
 * kvq_decode on the stream: e.g. they were copied from the host, or that
 * operation is kvq_append (which writes only the cache) and the one before
 * the append writes none of them either (kvq_append lets the decode start
 * while that one finishes: a kvq_combine, say, which writes only out and
 * lse).  It must not be set when that operation is kvq_norm_rope_apply
 * producing q, or any kernel that writes q, block_table or seq_lens.
 *
 * KVQ_DECODE_NO_TCGEN05: keep shapes of 17..64 query rows per kv head on the
 * mma.sync kernel's layouts instead of the tensor-memory (tcgen05) kernel
 * (for comparing the two; results agree within the parity tolerance). */
#define KVQ_DECODE_EARLY_INPUTS 0x1u
#define KVQ_DECODE_NO_TCGEN05 0x2u
/* KVQ_DECODE_EARLY_CACHE (with KVQ_DECODE_EARLY_INPUTS): the operation
 * enqueued just before kvq_decode writes no cache row other than the step's
 * new tokens (positions seq_lens[b] - q_tokens .. seq_lens[b] - 1): e.g. it
 * is kvq_append of exactly those tokens, or it writes no cache at all.  The
 * decode then loads every older row while that operation is still running and
 * waits for it only before the 64- or 128-key tile that holds the new tokens,
 * so the first cache reads overlap its tail.  Without KVQ_DECODE_EARLY_INPUTS
 * the bit has no effect. */
#define KVQ_DECODE_EARLY_CACHE 0x4u

/* Human-readable name of a status code (static storage). */
KVQ_API const char* kvq_status_string(kvq_status status);

/* kvq_append -- quantize-on-write of new K/V rows into their cache slots
 * (ReshapeAndCache, PR #29912; per-row absmax, kv-quant-attn "Method";
 * int4 nibble packing, PR #32515).
 * For each token n and kv head h, the D bf16 values of k_new[n, h, :] (and of
 * v_new) are quantized: PER_ROW scale = absmax / qmax (IEEE fp32 division,
 * qmax 127 / 7 / 448, an all-zero row stores scale 0 and zero codes; PER_GROUP
 * the same over each group of group_size channels), then
 * code = clamp(round_half_even(x / scale), -qmax, qmax) for int8 / int4, or
 * the nearest e4m3 value (ties to even, finite overflow saturated to 448).
 * slot_mapping int64 [n_tokens] (device): slot < 0 skips the token (padding);
 * slot >= num_blocks * block_size sets KVQ_DEVERR_SLOT and skips it.
 * Rows already in the cache are never touched.  n_tokens == 0 is a no-op.
 * Its kernel lets the next kernel on the stream be scheduled at once (that
 * kernel may then run while this one and the one before it finish); every
 * kvq kernel waits for its predecessor before it reads what that one writes,
 * so only a decode with KVQ_DECODE_EARLY_INPUTS reads anything early. */
KVQ_API kvq_status kvq_append(const kvq_cache* cache, const void* k_new, const void* v_new,
                              const int64_t* slot_mapping, int32_t n_tokens,
                              kvq_stream_t stream);

/* The prologue before the cache write: QK-RMSNorm, then RoPE (QkNormRotaryTNH
 * in onnxruntime PR #29912, Summary of Changes: q_norm_weight / k_norm_weight
 * inputs, qk_norm_epsilon with default 1e-6, rotary_offset, which rotates
 * channels [rotary_offset, rotary_offset + rotary_dim)).  For each (token,
 * head) row x of head_dim bf16 values:
 *   RMSNorm (norm_weight != NULL): y_d = (x_d * r) * w_d,
 *     r = 1 / sqrt(sum_d x_d^2 / head_dim + eps);
 *   RoPE (rotary_dim > 0): the pair (a, b) of angle index i in
 *     [0, rotary_dim/2) becomes (a cos - b sin, b cos + a sin), with
 *     cos = cos_cache[pos, i], sin = sin_cache[pos, i] for the token's
 *     position pos; pairs are (off + i, off + i + rotary_dim/2) (half split)
 *     or (off + 2i, off + 2i + 1) (rotary_interleaved);
 * then one round-to-nearest-even to bf16 per value.  Arithmetic is IEEE fp32,
 * one rounding per operation in a fixed order, so results are reproducible
 * bit for bit: with E = head_dim / 32, the squares of channels
 * l*E .. l*E + E - 1 are summed in order into partial l (l = 0..31), then for
 * o = 16, 8, 4, 2, 1 each partial l becomes partial l + partial (l xor o);
 * each rotated value is (y * cos) -+ (partner * sin) with both products
 * rounded.  The pages fix neither the rotation layout nor the tables: both
 * are the caller's, as here. */
typedef struct {
  const void* norm_weight;    /* bf16 [head_dim] (device), or NULL: no RMSNorm */
  float norm_eps;             /* <= 0 selects 1e-6 */
  int32_t rotary_dim;         /* 0: no RoPE; else even, rotary_offset + rotary_dim <= head_dim */
  int32_t rotary_offset;      /* first rotated channel (>= 0) */
  int32_t rotary_interleaved; /* 0: half-split pairs; 1: adjacent pairs */
  const float* cos_cache;     /* fp32 [max_position, rotary_dim/2] (device) */
  const float* sin_cache;     /* fp32 [max_position, rotary_dim/2] (device) */
  int32_t max_position;       /* rows of the tables (> 0 when rotary_dim > 0) */
  int32_t hadamard;           /* 1: then rotate the row by the orthonormal Walsh-Hadamard
                                 matrix (Sylvester order, entry (i, j) =
                                 (-1)^popcount(i & j) / sqrt(head_dim)): butterflies of
                                 span 1, 2, 4, ... in fp32, then times
                                 fl32(1 / fl32(sqrt(head_dim))).  Apply it to Q and K alike:
                                 dot products are unchanged while an outlier channel is
                                 spread over the row before quantization (the rotation
                                 PR #32515 names as the follow-up for the int4 cache) */
} kvq_norm_rope;

/* kvq_norm_rope_apply -- the prologue on x [n_tokens, num_heads, head_dim]
 * bf16 (device) into y (same shape; y == x is allowed), e.g. the queries
 * before kvq_decode.  positions int64 [n_tokens] (device; may be NULL when
 * rotary_dim == 0): a position outside [0, max_position) sets
 * KVQ_DEVERR_POSITION and leaves that token's rows of y unwritten.
 * head_dim in {64, 128, 256, 576} (the Hadamard rotation: powers of two only);
 * x, y 16-byte aligned. */
KVQ_API kvq_status kvq_norm_rope_apply(const kvq_norm_rope* prologue, const void* x, void* y,
                                       const int64_t* positions, int32_t n_tokens,
                                       int32_t num_heads, int32_t head_dim, kvq_stream_t stream);

/* kvq_append_norm_rope -- kvq_append with the prologue fused in front of the
 * K quantizer: each K row is normalized and rotated as kvq_norm_rope_apply
 * would (same fp32 arithmetic, same bf16 rounding) and the resulting bf16 row
 * is quantized exactly as kvq_append quantizes its input; V rows are
 * quantized as given (the prologue acts on Q and K only).  A token with a
 * negative slot is skipped; one whose position is outside the tables sets
 * KVQ_DEVERR_POSITION and neither its K nor its V rows are written. */
KVQ_API kvq_status kvq_append_norm_rope(const kvq_cache* cache, const kvq_norm_rope* k_prologue,
                                        const void* k_new, const void* v_new,
                                        const int64_t* slot_mapping, const int64_t* positions,
                                        int32_t n_tokens, kvq_stream_t stream);

/* Bytes of workspace kvq_decode needs for these shapes on the current device
 * (split partials and the device-side split plan).  Host-only arithmetic plus
 * one cached device-attribute query. */
KVQ_API kvq_status kvq_decode_workspace_size(const kvq_cache* cache,
                                             const kvq_decode_params* params,
                                             size_t* workspace_bytes);

/* kvq_decode -- split-KV flash-decoding over the quantized pages
 * (PagedAttention paged decode, PR #29912; kv-quant-attn "Method").
 * Reads q, block_table, seq_lens and the cache on the device, dequantizes on
 * the fly, and writes per-split partials (log-sum-exp and normalized output)
 * plus the split plan into `workspace` (device, caller owned, at least
 * kvq_decode_workspace_size bytes, 256-byte aligned).  The result is
 * completed by kvq_combine with the same cache, params and workspace on the
 * same stream.  Per query row, logits are sm_scale * <q, k_j>, capped by
 * softcap, masked to keys j <= pos (and j > pos - window when set).
 * The kvq kernels let the next kernel on the stream start early
 * (programmatic dependent launch); kvq_decode itself waits for the preceding
 * kernel to complete before it reads any input, unless params->flags has
 * KVQ_DECODE_EARLY_INPUTS (see there for when that is allowed). */
KVQ_API kvq_status kvq_decode(const kvq_cache* cache, const kvq_decode_params* params,
                              const void* q, const int32_t* block_table,
                              const int32_t* seq_lens, void* workspace,
                              size_t workspace_bytes, kvq_stream_t stream);

/* kvq_combine -- fixed-order log-sum-exp merge of the split partials
 * (kv-quant-attn "Method": partials merged in a fixed order, bitwise
 * reproducible), then the exact head-sink rescale o *= 1/(1+exp(s_h - lse))
 * (ApplyHeadSink, PR #29912), the static V scale (PER_TENSOR, or PER_CHANNEL
 * per output channel: the fold of PR #32515), and a round-to-nearest-even
 * bf16 store to out [B, T, Hq, D].
 * head_sink fp32 [Hq] or NULL; lse_out fp32 [B, T, Hq] or NULL (natural-log
 * LSE of the logits, before the sink; -inf for an empty key set, whose output
 * row is zero). */
KVQ_API kvq_status kvq_combine(const kvq_cache* cache, const kvq_decode_params* params,
                               const void* workspace, size_t workspace_bytes,
                               const float* head_sink, void* out, float* lse_out,
                               kvq_stream_t stream);

/* kvq_prefill -- attention of a chunk of C = params->q_tokens new query tokens
 * per sequence over the quantized cache (chunked prefill / prompt attention:
 * PR #29912 and PR #32515 testing name prefill and chunked prefill; the head
 * sink applies as in decode).  The chunk's K/V rows are appended first
 * (kvq_append); token c of sequence b sits at position seq_lens[b] - C + c
 * and sees keys 0..that position (and the window, when set).  q, out bf16
 * [B, C, Hq, D]; lse_out fp32 [B, C, Hq] or NULL; head_sink as in
 * kvq_combine.  The chunk is cut into groups of T tokens (virtual
 * sequences; sequence b's j-th group sees the prefix seq_lens[b] - C + T
 * (j + 1)), run as one attention pass and one combine; B * C / T <= 1024.
 * With head_dim 128 or 256, no group-wise scales and KVQ_DECODE_NO_TCGEN05
 * unset, T is the largest divisor of C with T x (Hq / Hkv) <= 128 when that
 * gives at least 64 query rows per kv head: a group's rows are the M
 * dimension of tcgen05 MMAs and each key tile of its prefix is dequantized
 * once for all of them (the kv-quant-attn page, "Requirements and limits":
 * prefill wants a tiled attention kernel).  Otherwise T is the largest of 8,
 * 4, 2, 1 dividing C and the groups run on the decode kernels.  Each group
 * reads its prefix, so a chunk costs C / T passes over the cache, shared
 * through L2 where they coincide.  C >= 1 (no upper bound besides the
 * virtual batch).  workspace: at least kvq_prefill_workspace_size bytes,
 * 256-byte aligned. */
KVQ_API kvq_status kvq_prefill_workspace_size(const kvq_cache* cache, const kvq_decode_params* params,
                                              size_t* workspace_bytes);
KVQ_API kvq_status kvq_prefill(const kvq_cache* cache, const kvq_decode_params* params, const void* q,
                               const int32_t* block_table, const int32_t* seq_lens, const float* head_sink,
                               void* out, float* lse_out, void* workspace, size_t workspace_bytes,
                               kvq_stream_t stream);

/* kvq_attend_noalloc -- kvq_decode then kvq_combine, with the split-partial
 * scratch in a library-owned 16 MiB device array instead of a caller
 * workspace.  The pages have no counterpart: this exists for callers that
 * cannot allocate device memory where they run attention (a plugin inside a
 * runtime that owns all device memory and offers no scratch allocator, or a
 * loop that must not pay cudaMalloc's implicit synchronization).  It allocates
 * and frees nothing.  Arguments and results are those of kvq_decode and
 * kvq_combine; KVQ_ERR_WORKSPACE_TOO_SMALL when the shapes need more than
 * 16 MiB of scratch (kvq_decode_workspace_size tells).  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture.  The array holds the previous
 * call's contents and is shared by all calls on the device: calls that
 * overlap on the GPU (different streams without ordering) race. */
KVQ_API kvq_status kvq_attend_noalloc(const kvq_cache* cache, const kvq_decode_params* params,
                                      const void* q, const int32_t* block_table,
                                      const int32_t* seq_lens, const float* head_sink, void* out,
                                      float* lse_out, kvq_stream_t stream);

/* kvq_check_wait_timeout -- failure-detection check of the bounded waits.
 * Launches one thread that waits on an mbarrier nothing ever arrives on, with
 * the same bounded wait the decode pipelines use (there bounded at 1.5 s),
 * here given limit_us microseconds (1 .. 2,000,000).  The wait gives up,
 * KVQ_DEVERR_TIMEOUT is set in the device flag word, and the context stays
 * usable: kvq_get_device_error then returns KVQ_ERR_DEVICE_TIMEOUT.  Nothing
 * is faulted or trapped.  Asynchronous on `stream`. */
KVQ_API kvq_status kvq_check_wait_timeout(uint32_t limit_us, kvq_stream_t stream);

/* Reads the current device's KVQ_DEVERR_* flag word into *flags (host).  This
 * call synchronizes `stream` before reading.  clear != 0 resets the word. */
KVQ_API kvq_status kvq_get_device_error(uint32_t* flags, int32_t clear, kvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
