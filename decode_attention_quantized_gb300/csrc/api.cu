// api.cu -- the C ABI of include/kvq.h: host-side validation, split planning,
// TMA descriptor encoding and kernel launches.  No allocation, no host sync
// (except kvq_get_device_error, which says so), no device data read back.
#include <cmath>
#include <cstring>
#include <mutex>

#include "kvq_internal.h"

namespace kvq {

// Per-device flag word for data violations (KVQ_DEVERR_*).
__device__ unsigned int g_error_word;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool init = false;
  int sms = 0;
  unsigned int* err = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

kvq_status current_device(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVQ_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVQ_ERR_CUDA;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_error_word) != cudaSuccess) return KVQ_ERR_CUDA;
    d.init = true;
  }
  *out = &d;
  return KVQ_OK;
}

kvq_status encoder(PFN_cuTensorMapEncodeTiled_v12000* out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return KVQ_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = g_encode;
  return KVQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}
int row_bytes(const kvq_cache* c) { return c->dtype == KVQ_INT4 ? c->head_dim / 2 : c->head_dim; }
// fp32 scales per cached row of a side in mode m (0: static scales)
int scales_per_row(const kvq_cache* c, int m) {
  return m == KVQ_SCALE_PER_ROW ? 1 : (m == KVQ_SCALE_PER_GROUP && c->group_size > 0 ? c->head_dim / c->group_size : 0);
}
bool any_group(const kvq_cache* c) {
  return c->k_mode == KVQ_SCALE_PER_GROUP || c->v_mode == KVQ_SCALE_PER_GROUP;
}

kvq_status check_cache(const kvq_cache* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->dtype < KVQ_INT8 || c->dtype > KVQ_INT4) return KVQ_ERR_INVALID_ARG;
  for (int m : {c->k_mode, c->v_mode})
    if (m < KVQ_SCALE_PER_ROW || m > KVQ_SCALE_PER_GROUP) return KVQ_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0) return KVQ_ERR_INVALID_ARG;
  if (!pow2(c->block_size) || c->block_size < 16 || c->block_size > (1 << 20)) return KVQ_ERR_INVALID_ARG;
  if ((long long)c->num_blocks * c->block_size > (1LL << 31) - 1) return KVQ_ERR_INVALID_ARG;
  // head_dim 576 (absorbed MLA: 512 latent + 64 rotary channels): LATENT with
  // 8-bit codes and per-row or static scales, on the mma.sync wide layout
  const bool latent576 = c->head_dim == 576 && c->layout == KVQ_LAYOUT_LATENT && c->dtype != KVQ_INT4 &&
                         c->k_mode != KVQ_SCALE_PER_GROUP;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256 && !latent576) return KVQ_ERR_UNSUPPORTED;
  if (!c->k_codes || !c->v_codes || !c->k_scale || !c->v_scale) return KVQ_ERR_INVALID_ARG;
  if (!aligned(c->k_codes, 16) || !aligned(c->v_codes, 16)) return KVQ_ERR_INVALID_ARG;
  if (!aligned(c->k_scale, scales_per_row(c, c->k_mode) ? 16 : 4)) return KVQ_ERR_INVALID_ARG;
  if (!aligned(c->v_scale, scales_per_row(c, c->v_mode) ? 16 : 4)) return KVQ_ERR_INVALID_ARG;
  if (c->k_mode == KVQ_SCALE_PER_GROUP || c->v_mode == KVQ_SCALE_PER_GROUP) {
    const int g = c->group_size;
    if ((g != 32 && g != 64 && g != 128) || g > c->head_dim) return KVQ_ERR_INVALID_ARG;
  }
  return KVQ_OK;
}

// The effective descriptor: a LATENT cache reads V from the K codes and
// scales (the leading v_head_size channels are kept by the combine);
// v_head_size is filled in for both layouts.  Then the usual checks.
kvq_status resolve_cache(const kvq_cache* c, kvq_cache* eff) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  *eff = *c;
  if (c->layout == KVQ_LAYOUT_LATENT) {
    eff->v_codes = c->k_codes;
    eff->v_scale = c->k_scale;
    eff->v_mode = c->k_mode;
    const int dv = c->v_head_size == 0 ? c->head_dim : c->v_head_size;
    if (dv < 8 || dv > c->head_dim || dv % 8) return KVQ_ERR_INVALID_ARG;
    eff->v_head_size = dv;
  } else if (c->layout == KVQ_LAYOUT_SEPARATE) {
    if (c->v_head_size != 0 && c->v_head_size != c->head_dim) return KVQ_ERR_INVALID_ARG;
    eff->v_head_size = c->head_dim;
  } else {
    return KVQ_ERR_INVALID_ARG;
  }
  return check_cache(eff);
}

// qt: the query-tile layout of kvq_prefill's virtual sequences, whose
// tokens x group may reach kQtRows rows (any token count); else at most 8
// tokens of at most 8 query heads per kv head.
kvq_status check_params(const kvq_cache* c, const kvq_decode_params* p, bool qt = false) {
  if (!p) return KVQ_ERR_INVALID_ARG;
  if (p->batch < 0 || p->num_q_heads <= 0 || p->q_tokens <= 0 || p->max_blocks_per_seq <= 0 ||
      p->max_seq_len < 0 || p->window < 0)
    return KVQ_ERR_INVALID_ARG;
  if (p->num_q_heads % c->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(p->sm_scale) || !std::isfinite(p->softcap) || p->softcap < 0.0f) return KVQ_ERR_INVALID_ARG;
  if (p->flags & ~(KVQ_DECODE_EARLY_INPUTS | KVQ_DECODE_NO_TCGEN05 | KVQ_DECODE_EARLY_CACHE))
    return KVQ_ERR_INVALID_ARG;
  if ((long long)p->max_blocks_per_seq * c->block_size > (1LL << 30)) return KVQ_ERR_INVALID_ARG;
  if (p->num_q_heads / c->num_kv_heads > 8 || p->batch > kMaxBatch) return KVQ_ERR_UNSUPPORTED;
  if (qt ? (long long)p->q_tokens * (p->num_q_heads / c->num_kv_heads) > kQtRows : p->q_tokens > 8)
    return KVQ_ERR_UNSUPPORTED;
  // the tile space of all (sequence, kv head) ranges must index with int
  const long long tiles = (long long)p->max_blocks_per_seq * c->block_size / kTile + 1;
  if ((long long)p->batch * c->num_kv_heads * tiles >= (1LL << 31)) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

// Split planning: the time a CTA spends on each piece change, in tiles of
// its kernel (measured: 3 balances best for both kernels; the ragged mixed
// workload's decode went from 249 to 206 us, paged from 120 to 118 us, spec
// from 67.8 to 64.8 us).
constexpr int kTcPieceCost = 3;
// The query-tile kernel: a piece change (Q prologue, epilogue, pipeline
// refill) costs about 8 of its tiles; its ring is capped at 3 stages (with
// 7-8 stages at head_dim 128, a quarter of the CTAs of a ragged batch ran
// 3-4x slower than the rest; 3 stages measured balanced and fastest).
constexpr int kQtPieceCost = 8;
constexpr int kQtMaxStages = 3;
constexpr int kPieceCost = 3;

// Launch shape of the decode kernel and the workspace it implies.
struct Plan {
  int rows, row_groups, key_warps, nt, tc_nr, qt, threads, stages, grid, units_max;
  size_t stride, smem, ws_plan, ws_lse, ws_o, ws_total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// K and V code rows of one stage, then room for the K and V per-row or
// per-group scales only when a side has them (a 16-row fp8 stage of head_dim
// 128 is then 16 KB, so four CTAs with three stages each fit on an SM): K's
// [kTile][sk_n] floats, then V's [kTile][sv_n] at kTile * max(1, sk_n)
// floats.  A LATENT cache on the mma.sync kernel (alias) keeps the K side
// only: V is read from it.  1 KB multiples keep every stage on the 128-byte
// swizzle's alignment.
size_t stage_stride(const kvq_cache* c, bool alias) {
  const size_t code = (size_t)kTile * row_bytes(c);
  const int nk = scales_per_row(c, c->k_mode), nv = alias ? 0 : scales_per_row(c, c->v_mode);
  const size_t sc = (nk || nv) ? (size_t)kTile * 4 * ((nk > 1 ? nk : 1) + (alias ? 0 : (nv > 1 ? nv : 1))) : 0;
  return ((alias ? 1 : 2) * code + sc + 1023) / 1024 * 1024;
}

size_t fixed_smem(const kvq_cache* c, int row_groups, int key_warps, int nt, int batch, int stages) {
  size_t s = 1024;  // alignment slack of the ring
  if (nt > 0)  // wide layout: P buffer, row maxima / sums, Q operand, logit factors
    s += (size_t)(16 * nt * 32 + 2 * 4 * 16 * nt + 32 + 16 * nt * (c->head_dim / 2) + (16 * nt + 31) / 32 * 32) * 4;
  else if (key_warps > 1)
    s += (size_t)row_groups * (c->head_dim / 16 * 4 + 4) * 32 * 4;  // merge slot per row group
  s += ((size_t)batch + 5 + ((batch + 5) & 1)) * 4;                                  // split plan
  s += (size_t)stages * 2 * 8;                                                       // mbarriers
  return s;
}

// The mma.sync kernel instance: the plan's consumer layout nt (0 grouped, 2 / 3
// wide), or -group_size for the grouped layout with per-group scales.
int kernel_nt(const kvq_cache* c, const Plan& P) { return any_group(c) ? -c->group_size : P.nt; }

cudaError_t occupancy(const kvq_cache* c, int nt, int threads, size_t smem, int* n) {
  switch (c->dtype) {
    case KVQ_INT8: return occupancy_decode_int8(c->head_dim, nt, threads, smem, n);
    case KVQ_FP8_E4M3: return occupancy_decode_fp8(c->head_dim, nt, threads, smem, n);
    default: return occupancy_decode_int4(c->head_dim, nt, threads, smem, n);
  }
}

// The tensor-memory kernel takes 17..48 query rows per kv head at head_dim
// 256 and 17..64 at head_dim 128 (its TMEM columns bound rows x head_dim);
// KVQ_DECODE_NO_TCGEN05 keeps such shapes on the mma.sync layouts.
int tc_rows(const kvq_cache* c, const kvq_decode_params* p, int rows) {
  if (p->flags & KVQ_DECODE_NO_TCGEN05) return 0;
  if (rows < 17) return 0;
  if (c->head_dim == 256 && rows <= 48) return rows <= 32 ? 32 : 48;
  if (c->head_dim == 128 && rows <= 64) return rows <= 32 ? 32 : (rows <= 48 ? 48 : 64);
  return 0;
}

kvq_status make_plan_tc(const kvq_cache* c, const kvq_decode_params* p, const DeviceInfo& dev, Plan* P) {
  const int B = p->batch > 0 ? p->batch : 1;
  const int dp = row_bytes(c);
  const int stride = tc_stage_stride(dp, scales_per_row(c, c->k_mode), scales_per_row(c, c->v_mode));
  constexpr size_t kMaxSmem = 227 * 1024;  // per CTA
  int stages = 0;
  for (int s = kMaxStages; s >= 2 && stages == 0; --s)
    if ((size_t)tc_smem_layout(c->head_dim, dp, P->tc_nr, s, B, stride).total + 1024 <= kMaxSmem) stages = s;
  if (stages == 0) return KVQ_ERR_UNSUPPORTED;
  P->stages = stages;
  P->stride = (size_t)stride;
  P->smem = (size_t)tc_smem_layout(c->head_dim, dp, P->tc_nr, stages, B, stride).total + 1024;
  P->threads = kTcWarps * 32;
  P->row_groups = 0;
  P->key_warps = 0;
  P->nt = 0;
  const long long cap = (long long)p->max_blocks_per_seq * c->block_size;
  const long long maxlen = (p->max_seq_len > 0 && p->max_seq_len < cap) ? p->max_seq_len : cap;
  long long grid = dev.sms;  // one CTA per SM: it holds all of the SM's tensor memory
  const long long useful = (long long)B * c->num_kv_heads * ((maxlen + kTcKeys - 1) / kTcKeys + 1);
  if (grid > useful) grid = useful;
  P->grid = (int)(grid < 1 ? 1 : grid);
  return KVQ_OK;
}

// Whether kvq_prefill takes the query-tile kernel: head_dim 128 or 256, no
// group-wise scales, the tcgen05 kernels allowed.
bool qt_ok(const kvq_cache* c, const kvq_decode_params* p) {
  return !(p->flags & KVQ_DECODE_NO_TCGEN05) && (c->head_dim == 128 || c->head_dim == 256) && !any_group(c);
}

// The query-tile kernel: one CTA per SM (it holds all of the SM's TMEM), the
// mma.sync kernel's 64-key stages, as many of them as fit beside the two
// double-buffered f16 tiles.
kvq_status make_plan_qt(const kvq_cache* c, const kvq_decode_params* p, const DeviceInfo& dev, Plan* P) {
  const int B = p->batch > 0 ? p->batch : 1;
  const size_t stride = stage_stride(c, false);
  constexpr size_t kMaxSmem = 227 * 1024;  // per CTA
  int stages = 0;
  for (int s = kQtMaxStages; s >= 2 && stages == 0; --s)
    if ((size_t)qt_smem_layout(c->head_dim, s, B, (int)stride).total + 1024 <= kMaxSmem) stages = s;
  if (stages == 0) return KVQ_ERR_UNSUPPORTED;
  P->qt = 1;
  P->stages = stages;
  P->stride = stride;
  P->smem = (size_t)qt_smem_layout(c->head_dim, stages, B, (int)stride).total + 1024;
  P->threads = kQtWarps * 32;
  const long long cap = (long long)p->max_blocks_per_seq * c->block_size;
  const long long maxlen = (p->max_seq_len > 0 && p->max_seq_len < cap) ? p->max_seq_len : cap;
  long long grid = dev.sms;
  const long long useful = (long long)B * c->num_kv_heads * ((maxlen + kTile - 1) / kTile + 1);
  if (grid > useful) grid = useful;
  P->grid = (int)(grid < 1 ? 1 : grid);
  return KVQ_OK;
}

kvq_status make_plan_uncached(const kvq_cache* c, const kvq_decode_params* p, const DeviceInfo& dev, bool qt,
                              Plan* out) {
  Plan P{};
  const int G = p->num_q_heads / c->num_kv_heads;
  P.rows = G * p->q_tokens;
  if (qt) {
    if (!qt_ok(c, p) || P.rows > kQtRows) return KVQ_ERR_UNSUPPORTED;
    if (kvq_status s = make_plan_qt(c, p, dev, &P)) return s;
    const int B = p->batch > 0 ? p->batch : 1;
    P.units_max = P.grid + B * c->num_kv_heads;
    P.ws_plan = align256((size_t)(4 + B + 1) * 4);
    P.ws_lse = align256((size_t)P.units_max * P.rows * 4);
    P.ws_o = (size_t)P.units_max * P.rows * c->head_dim * 4;
    P.ws_total = P.ws_plan + P.ws_lse + P.ws_o;
    *out = P;
    return KVQ_OK;
  }
  P.tc_nr = tc_rows(c, p, P.rows);
  if (P.tc_nr) {
    if (kvq_status s = make_plan_tc(c, p, dev, &P)) return s;
    const int B = p->batch > 0 ? p->batch : 1;
    P.units_max = P.grid + B * c->num_kv_heads;
    P.ws_plan = align256((size_t)(4 + B + 1) * 4);
    P.ws_lse = align256((size_t)P.units_max * P.rows * 4);
    P.ws_o = (size_t)P.units_max * P.rows * c->head_dim * 4;
    P.ws_total = P.ws_plan + P.ws_lse + P.ws_o;
    *out = P;
    return KVQ_OK;
  }
  P.row_groups = (P.rows + 7) / 8;
  P.key_warps = P.row_groups <= 2 ? 4 : (P.row_groups <= 4 ? 2 : 1);
  // 17..48 rows (e.g. drafts x GQA group): the wide layout, 4 key quarters x 2
  // row halves of nt n-tiles, when a channel quarter spans >= 2 code chunks;
  // head_dim 576 takes it for every row count up to 48 (its rows are too long
  // for one warp's registers)
  const bool wide_fits = c->dtype == KVQ_INT4 ? c->head_dim == 256 : c->head_dim >= 128;
  if (c->head_dim == 576) {
    if (P.rows > 48) return KVQ_ERR_UNSUPPORTED;
    P.nt = (P.row_groups + 1) / 2;
  } else {
    P.nt = (wide_fits && !any_group(c) && P.row_groups >= 3 && P.row_groups <= 6) ? (P.row_groups + 1) / 2 : 0;
  }
  if (P.nt > 0) {
    P.row_groups = 2;
    P.key_warps = 4;
  }
  const int n_cw = P.row_groups * P.key_warps;
  P.threads = 32 * (n_cw + 1);
  const int B = p->batch > 0 ? p->batch : 1;
  const size_t stride = stage_stride(c, c->layout == KVQ_LAYOUT_LATENT);
  P.stride = stride;
  // the most CTAs per SM whose ring still holds >= 3 stages (more warps per
  // SM hide more latency); one CTA with >= 2 stages as the last resort
  int occ = 0;
  for (int target : {4, 3, 2, 1}) {
    // per-SM shared memory is 228 KiB with 1 KiB reserved per resident CTA
    const size_t budget = (size_t)228 * 1024 / target - 1024;
    const size_t fixed = fixed_smem(c, P.row_groups, P.key_warps, P.nt, B, 0);
    // head_dim 576 stages are 37 KB: two CTAs of two stages each still keep
    // 148 KB in flight per SM, and twice the warps hide more latency
    const int min_stages = target > 1 && c->head_dim != 576 ? 3 : 2;
    if (fixed + (size_t)min_stages * (stride + 16) > budget) continue;
    int stages = (int)((budget - fixed) / (stride + 16));
    stages = stages > kMaxStages ? kMaxStages : stages;
    const size_t smem = fixed_smem(c, P.row_groups, P.key_warps, P.nt, B, stages) + (size_t)stages * stride;
    int n = 0;
    if (occupancy(c, kernel_nt(c, P), P.threads, smem, &n) != cudaSuccess) return KVQ_ERR_CUDA;
    if (n >= target) {
      occ = target;
      P.stages = stages;
      P.smem = smem;
      break;
    }
  }
  if (occ == 0) return KVQ_ERR_UNSUPPORTED;
  const long long cap = (long long)p->max_blocks_per_seq * c->block_size;
  const long long maxlen = (p->max_seq_len > 0 && p->max_seq_len < cap) ? p->max_seq_len : cap;
  long long grid = (long long)dev.sms * occ;
  const long long useful = (long long)B * c->num_kv_heads * ((maxlen + kTile - 1) / kTile + 1);
  if (grid > useful) grid = useful;
  P.grid = (int)(grid < 1 ? 1 : grid);
  P.units_max = P.grid + B * c->num_kv_heads;  // partial slots: segment + CTA index
  P.ws_plan = align256((size_t)(4 + B + 1) * 4);
  P.ws_lse = align256((size_t)P.units_max * P.rows * 4);
  P.ws_o = (size_t)P.units_max * P.rows * c->head_dim * 4;
  P.ws_total = P.ws_plan + P.ws_lse + P.ws_o;
  *out = P;
  return KVQ_OK;
}

// The launch plan depends only on shapes and the device; calls with the same
// shapes reuse it (no occupancy query on the hot path).
struct PlanKey {
  int dev, dtype, k_mode, v_mode, group_size, head_dim, num_kv_heads, block_size, batch, num_q_heads,
      q_tokens, max_blocks_per_seq, max_seq_len, no_tc, layout, qt;
  bool operator==(const PlanKey& o) const { return std::memcmp(this, &o, sizeof(PlanKey)) == 0; }
};
constexpr int kPlanCache = 64;
PlanKey g_plan_keys[kPlanCache];
Plan g_plans[kPlanCache];
int g_plan_count = 0, g_plan_next = 0;

kvq_status make_plan(const kvq_cache* c, const kvq_decode_params* p, const DeviceInfo& dev, Plan* out,
                     bool qt = false) {
  PlanKey k;
  std::memset(&k, 0, sizeof k);
  if (cudaGetDevice(&k.dev) != cudaSuccess) return KVQ_ERR_CUDA;
  k.dtype = c->dtype;
  k.k_mode = c->k_mode;
  k.v_mode = c->v_mode;
  k.group_size = any_group(c) ? c->group_size : 0;
  k.head_dim = c->head_dim;
  k.num_kv_heads = c->num_kv_heads;
  k.block_size = c->block_size;
  k.batch = p->batch;
  k.num_q_heads = p->num_q_heads;
  k.q_tokens = p->q_tokens;
  k.max_blocks_per_seq = p->max_blocks_per_seq;
  k.max_seq_len = p->max_seq_len;
  k.no_tc = (p->flags & KVQ_DECODE_NO_TCGEN05) ? 1 : 0;
  k.layout = c->layout;
  k.qt = qt ? 1 : 0;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_plan_count; ++i)
      if (g_plan_keys[i] == k) {
        *out = g_plans[i];
        return KVQ_OK;
      }
  }
  Plan P;
  if (kvq_status s = make_plan_uncached(c, p, dev, qt, &P)) return s;
  std::lock_guard<std::mutex> lk(g_mu);
  const int slot = g_plan_count < kPlanCache ? g_plan_count++ : (g_plan_next++ % kPlanCache);
  g_plan_keys[slot] = k;
  g_plans[slot] = P;
  *out = P;
  return KVQ_OK;
}

kvq_status encode_codes_map(const kvq_cache* c, void* base, CUtensorMap* tm) {
  PFN_cuTensorMapEncodeTiled_v12000 enc;
  if (kvq_status s = encoder(&enc)) return s;
  const int dp = row_bytes(c);
  const int span = dp % 128 == 0 ? 128 : (dp % 64 == 0 ? 64 : 32);  // a 576-byte row: nine 64-byte slabs
  const cuuint64_t dims[4] = {(cuuint64_t)dp, (cuuint64_t)c->block_size, (cuuint64_t)c->num_kv_heads,
                              (cuuint64_t)c->num_blocks};
  const cuuint64_t strides[3] = {(cuuint64_t)dp, (cuuint64_t)dp * c->block_size,
                                 (cuuint64_t)dp * c->block_size * c->num_kv_heads};
  const cuuint32_t box[4] = {(cuuint32_t)span, (cuuint32_t)(c->block_size < kTile ? c->block_size : kTile), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA; }

// Host checks of a norm/RoPE prologue for rows of head_dim channels; fills
// the kernel-side descriptor.
kvq_status check_norm_rope(const kvq_norm_rope* p, int head_dim, const int64_t* positions, NormRope* out) {
  if (!p) return KVQ_ERR_INVALID_ARG;
  if (p->norm_weight && !aligned(p->norm_weight, 16)) return KVQ_ERR_INVALID_ARG;
  if (!(p->norm_eps == p->norm_eps)) return KVQ_ERR_INVALID_ARG;  // NaN
  const int rd = p->rotary_dim, off = p->rotary_offset;
  if (rd < 0 || (rd & 1) || off < 0 || (long long)off + rd > head_dim) return KVQ_ERR_INVALID_ARG;
  if (rd > 0 && (!p->cos_cache || !p->sin_cache || !positions || p->max_position <= 0 ||
                 !aligned(p->cos_cache, 4) || !aligned(p->sin_cache, 4) || !aligned(positions, 8)))
    return KVQ_ERR_INVALID_ARG;
  NormRope r{};
  r.w = static_cast<const uint16_t*>(p->norm_weight);
  r.eps = p->norm_eps > 0.0f ? p->norm_eps : 1e-6f;
  r.cos_tab = p->cos_cache;
  r.sin_tab = p->sin_cache;
  r.positions = positions;
  r.rd = rd;
  r.off = off;
  r.interleaved = p->rotary_interleaved ? 1 : 0;
  r.max_pos = rd > 0 ? p->max_position : 0;
  if (p->hadamard != 0 && p->hadamard != 1) return KVQ_ERR_INVALID_ARG;
  if (p->hadamard && (head_dim & (head_dim - 1))) return KVQ_ERR_UNSUPPORTED;  // a power of two
  r.hadamard = p->hadamard;
  r.had_scale = 1.0f / std::sqrt((float)head_dim);
  *out = r;
  return KVQ_OK;
}

kvq_status append_common(const kvq_cache* cache, const kvq_norm_rope* k_prologue, const void* k_new,
                         const void* v_new, const int64_t* slot_mapping, const int64_t* positions,
                         int32_t n_tokens, kvq_stream_t stream) {
  kvq_cache eff_;
  if (kvq_status s = resolve_cache(cache, &eff_)) return s;
  cache = &eff_;
  if (n_tokens < 0) return KVQ_ERR_INVALID_ARG;
  NormRope pro{};
  if (k_prologue)
    if (kvq_status s = check_norm_rope(k_prologue, cache->head_dim, positions, &pro)) return s;
  if (n_tokens == 0) return KVQ_OK;
  const bool latent = cache->layout == KVQ_LAYOUT_LATENT;  // V is the K row: v_new unused
  if (!k_new || (!v_new && !latent) || !slot_mapping) return KVQ_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || (v_new && !aligned(v_new, 16)) || !aligned(slot_mapping, 8))
    return KVQ_ERR_INVALID_ARG;
  if ((long long)n_tokens * cache->num_kv_heads * 2 > (1LL << 31) - 1) return KVQ_ERR_INVALID_ARG;
  DeviceInfo* dev;
  if (kvq_status s = current_device(&dev)) return s;
  AppendArgs a{};
  a.k_new = static_cast<const uint16_t*>(k_new);
  a.v_new = static_cast<const uint16_t*>(v_new);
  a.slots = slot_mapping;
  a.k_codes = static_cast<uint8_t*>(cache->k_codes);
  a.v_codes = static_cast<uint8_t*>(cache->v_codes);
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.capacity = (long long)cache->num_blocks * cache->block_size;
  a.n_tokens = n_tokens;
  a.num_kv_heads = cache->num_kv_heads;
  a.head_dim = cache->head_dim;
  a.block_size = cache->block_size;
  a.log2_bs = ilog2(cache->block_size);
  a.dtype = cache->dtype;
  a.k_mode = cache->k_mode;
  a.v_mode = cache->v_mode;
  a.log2_group = any_group(cache) ? ilog2(cache->group_size) : 0;
  a.err = dev->err;
  a.k_prologue = k_prologue ? 1 : 0;
  a.latent = latent ? 1 : 0;
  a.pro = pro;
  return from_cuda(launch_append(a, reinterpret_cast<cudaStream_t>(stream)));
}

// kvq_decode with the block-table row of sequence b at b / bt_div.  With
// early_reads 1, q, the block table, seq_lens and the static scales are read
// before the wait on the preceding grid (KVQ_DECODE_EARLY_INPUTS); with 0,
// every input is read after it (the default, and kvq_prefill's virtual
// sequences, whose lengths that grid writes).
kvq_status decode_impl(const kvq_cache* cache, const kvq_decode_params* params, const void* q,
                       const int32_t* block_table, const int32_t* seq_lens, int bt_div, int early_reads,
                       bool qt, void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
  kvq_cache eff_;
  if (kvq_status s = resolve_cache(cache, &eff_)) return s;
  cache = &eff_;
  if (kvq_status s = check_params(cache, params, qt)) return s;
  if (params->batch == 0) return KVQ_OK;
  if (!q || !block_table || !seq_lens || !workspace) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(workspace, 256))
    return KVQ_ERR_INVALID_ARG;
  DeviceInfo* dev;
  if (kvq_status s = current_device(&dev)) return s;
  Plan P;
  if (kvq_status s = make_plan(cache, params, *dev, &P, qt)) return s;
  if (workspace_bytes < P.ws_total) return KVQ_ERR_WORKSPACE_TOO_SMALL;

  alignas(64) CUtensorMap tk, tv;
  if (kvq_status s = encode_codes_map(cache, cache->k_codes, &tk)) return s;
  if (kvq_status s = encode_codes_map(cache, cache->v_codes, &tv)) return s;

  DecodeArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.k_mode = cache->k_mode;
  a.v_mode = cache->v_mode;
  a.sk_n = scales_per_row(cache, cache->k_mode);
  a.sv_n = scales_per_row(cache, cache->v_mode);
  a.log2_gs = any_group(cache) ? ilog2(cache->group_size) : 0;
  a.num_blocks = cache->num_blocks;
  a.block_size = cache->block_size;
  a.log2_bs = ilog2(cache->block_size);
  a.num_kv_heads = cache->num_kv_heads;
  a.batch = params->batch;
  a.num_q_heads = params->num_q_heads;
  a.q_tokens = params->q_tokens;
  a.group = params->num_q_heads / cache->num_kv_heads;
  a.rows = P.rows;
  a.max_blocks_per_seq = params->max_blocks_per_seq;
  a.max_seq_len = params->max_seq_len;
  a.sm_scale = params->sm_scale > 0.0f ? params->sm_scale : 1.0f / std::sqrt((float)cache->head_dim);
  a.softcap = params->softcap;
  a.window = params->window;
  a.row_groups = P.row_groups;
  a.key_warps = P.key_warps;
  a.stages = P.stages;
  a.stage_stride = (int)P.stride;
  a.units_max = P.units_max;
  // a piece change (query prologue, merge and partial write, refill of the
  // role pipeline) is charged as a few tiles when the split is planned
  a.piece_cost = P.qt ? kQtPieceCost : (P.tc_nr ? kTcPieceCost : kPieceCost);
  a.bt_div = bt_div;
  // the mma.sync kernel reads a LATENT cache's V from the K codes it loaded
  // (the tensor-memory kernels load both sides)
  a.v_alias = (cache->layout == KVQ_LAYOUT_LATENT && !P.tc_nr && !P.qt) ? 1 : 0;
  a.early_reads = early_reads;
  a.early_cache = (early_reads && (params->flags & KVQ_DECODE_EARLY_CACHE)) ? 1 : 0;
  char* ws = static_cast<char*>(workspace);
  a.plan = reinterpret_cast<int*>(ws);
  a.part_lse = reinterpret_cast<float*>(ws + P.ws_plan);
  a.part_o = reinterpret_cast<float*>(ws + P.ws_plan + P.ws_lse);
  a.err = dev->err;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (P.qt) {
    switch (cache->dtype) {
      case KVQ_INT8: e = launch_decode_qt_int8(cache->head_dim, tk, tv, a, P.grid, P.smem, st); break;
      case KVQ_FP8_E4M3: e = launch_decode_qt_fp8(cache->head_dim, tk, tv, a, P.grid, P.smem, st); break;
      default: e = launch_decode_qt_int4(cache->head_dim, tk, tv, a, P.grid, P.smem, st); break;
    }
  } else if (P.tc_nr && any_group(cache)) {
    switch (cache->dtype) {
      case KVQ_INT8: e = launch_decode_tc_grp_int8(cache->head_dim, P.tc_nr, tk, tv, a, P.grid, P.smem, st); break;
      case KVQ_FP8_E4M3: e = launch_decode_tc_grp_fp8(cache->head_dim, P.tc_nr, tk, tv, a, P.grid, P.smem, st); break;
      default: e = launch_decode_tc_grp_int4(cache->head_dim, P.tc_nr, tk, tv, a, P.grid, P.smem, st); break;
    }
  } else if (P.tc_nr) {
    switch (cache->dtype) {
      case KVQ_INT8: e = launch_decode_tc_int8(cache->head_dim, P.tc_nr, tk, tv, a, P.grid, P.smem, st); break;
      case KVQ_FP8_E4M3: e = launch_decode_tc_fp8(cache->head_dim, P.tc_nr, tk, tv, a, P.grid, P.smem, st); break;
      default: e = launch_decode_tc_int4(cache->head_dim, P.tc_nr, tk, tv, a, P.grid, P.smem, st); break;
    }
  } else {
    switch (cache->dtype) {
      case KVQ_INT8: e = launch_decode_int8(cache->head_dim, kernel_nt(cache, P), tk, tv, a, P.grid, P.threads, P.smem, st); break;
      case KVQ_FP8_E4M3: e = launch_decode_fp8(cache->head_dim, kernel_nt(cache, P), tk, tv, a, P.grid, P.threads, P.smem, st); break;
      default: e = launch_decode_int4(cache->head_dim, kernel_nt(cache, P), tk, tv, a, P.grid, P.threads, P.smem, st); break;
    }
  }
  return from_cuda(e);
}

// A prefill chunk of C tokens per sequence as virtual decode sequences of T
// tokens each, n = C / T per sequence.  On the query-tile kernel (qt), T is
// the largest divisor of C whose T x G rows fit its 128-row tile, when that
// gives at least 64 rows; otherwise the decode kernels take the largest of
// 8, 4, 2, 1 dividing C.
kvq_status prefill_shape(const kvq_cache* c, const kvq_decode_params* p, kvq_decode_params* v, int* n,
                         bool* qt) {
  if (!p || p->q_tokens < 1 || p->batch < 0) return KVQ_ERR_INVALID_ARG;
  const int C = p->q_tokens;
  const int G = c->num_kv_heads > 0 && p->num_q_heads % c->num_kv_heads == 0 ? p->num_q_heads / c->num_kv_heads : 0;
  int T = 8;
  *qt = false;
  if (G > 0 && qt_ok(c, p)) {
    int tq = kQtRows / G;
    if (tq > C) tq = C;
    while (C % tq) --tq;
    if (tq * G >= 64) {
      T = tq;
      *qt = true;
    }
  }
  if (!*qt)
    while (C % T) T >>= 1;
  const long long vb = (long long)p->batch * (C / T);
  if (vb > kMaxBatch) return KVQ_ERR_UNSUPPORTED;
  *v = *p;
  v->batch = (int32_t)vb;
  v->q_tokens = T;
  *n = C / T;
  return KVQ_OK;
}

// kvq_combine over the plan of decode_impl (qt: the query-tile layout of a
// prefill's virtual sequences).
kvq_status combine_impl(const kvq_cache* cache, const kvq_decode_params* params, bool qt, const void* workspace,
                        size_t workspace_bytes, const float* head_sink, void* out, float* lse_out,
                        kvq_stream_t stream, bool warp_rows = false) {
  kvq_cache eff_;
  if (kvq_status s = resolve_cache(cache, &eff_)) return s;
  cache = &eff_;
  if (kvq_status s = check_params(cache, params, qt)) return s;
  if (params->batch == 0) return KVQ_OK;
  if (!workspace || !out) return KVQ_ERR_INVALID_ARG;
  if (!aligned(workspace, 256) || !aligned(out, 16) || (lse_out && !aligned(lse_out, 4)) ||
      (head_sink && !aligned(head_sink, 4)))
    return KVQ_ERR_INVALID_ARG;
  DeviceInfo* dev;
  if (kvq_status s = current_device(&dev)) return s;
  Plan P;
  if (kvq_status s = make_plan(cache, params, *dev, &P, qt)) return s;
  if (workspace_bytes < P.ws_total) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  const char* ws = static_cast<const char*>(workspace);
  CombineArgs a{};
  a.plan = reinterpret_cast<const int*>(ws);
  a.part_lse = reinterpret_cast<const float*>(ws + P.ws_plan);
  a.part_o = reinterpret_cast<const float*>(ws + P.ws_plan + P.ws_lse);
  a.head_sink = head_sink;
  a.v_mode = cache->v_mode;
  // per-row and per-group V scales are applied inside the decode kernel
  a.v_scale = (cache->v_mode == KVQ_SCALE_PER_ROW || cache->v_mode == KVQ_SCALE_PER_GROUP) ? nullptr
                                                                                          : cache->v_scale;
  a.out = static_cast<uint16_t*>(out);
  a.lse_out = lse_out;
  a.batch = params->batch;
  a.q_tokens = params->q_tokens;
  a.num_q_heads = params->num_q_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.group = params->num_q_heads / cache->num_kv_heads;
  a.rows = P.rows;
  a.head_dim = cache->head_dim;
  a.out_dim = cache->v_head_size;
  // a warp per row when the rows have about 16 pieces or fewer on average
  // (the pieces are the grid's slices plus one per segment); a CTA per row
  // for few rows of many pieces (one long sequence split over the GPU)
  const long long segs = (long long)params->batch * cache->num_kv_heads;
  if ((long long)P.units_max <= 16 * segs) warp_rows = true;
  return from_cuda(launch_combine(a, reinterpret_cast<cudaStream_t>(stream), warp_rows));
}


kvq_status decode_workspace_size(const kvq_cache* cache, const kvq_decode_params* params, bool qt,
                                 size_t* workspace_bytes) {
  kvq_cache eff_;
  if (kvq_status s = resolve_cache(cache, &eff_)) return s;
  cache = &eff_;
  if (kvq_status s = check_params(cache, params, qt)) return s;
  if (!workspace_bytes) return KVQ_ERR_INVALID_ARG;
  DeviceInfo* dev;
  if (kvq_status s = current_device(&dev)) return s;
  Plan P;
  if (kvq_status s = make_plan(cache, params, *dev, &P, qt)) return s;
  *workspace_bytes = P.ws_total;
  return KVQ_OK;
}

}  // namespace
}  // namespace kvq

using namespace kvq;

extern "C" {

KVQ_API const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape or type";
    case KVQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_DEVICE_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

KVQ_API kvq_status kvq_append(const kvq_cache* cache, const void* k_new, const void* v_new,
                              const int64_t* slot_mapping, int32_t n_tokens, kvq_stream_t stream) {
  return append_common(cache, nullptr, k_new, v_new, slot_mapping, nullptr, n_tokens, stream);
}

KVQ_API kvq_status kvq_append_norm_rope(const kvq_cache* cache, const kvq_norm_rope* k_prologue,
                                        const void* k_new, const void* v_new, const int64_t* slot_mapping,
                                        const int64_t* positions, int32_t n_tokens, kvq_stream_t stream) {
  if (!k_prologue) return KVQ_ERR_INVALID_ARG;
  return append_common(cache, k_prologue, k_new, v_new, slot_mapping, positions, n_tokens, stream);
}

KVQ_API kvq_status kvq_norm_rope_apply(const kvq_norm_rope* prologue, const void* x, void* y,
                                       const int64_t* positions, int32_t n_tokens, int32_t num_heads,
                                       int32_t head_dim, kvq_stream_t stream) {
  if (head_dim != 64 && head_dim != 128 && head_dim != 256 && head_dim != 576) return KVQ_ERR_UNSUPPORTED;
  if (n_tokens < 0 || num_heads <= 0) return KVQ_ERR_INVALID_ARG;
  NormRopeArgs a{};
  if (kvq_status s = check_norm_rope(prologue, head_dim, positions, &a.pro)) return s;
  if (n_tokens == 0) return KVQ_OK;
  if (!x || !y || !aligned(x, 16) || !aligned(y, 16)) return KVQ_ERR_INVALID_ARG;
  if ((long long)n_tokens * num_heads > (1LL << 31) - 1) return KVQ_ERR_INVALID_ARG;
  DeviceInfo* dev;
  if (kvq_status s = current_device(&dev)) return s;
  a.x = static_cast<const uint16_t*>(x);
  a.y = static_cast<uint16_t*>(y);
  a.n_tokens = n_tokens;
  a.num_heads = num_heads;
  a.head_dim = head_dim;
  a.err = dev->err;
  return from_cuda(launch_norm_rope(a, reinterpret_cast<cudaStream_t>(stream)));
}

KVQ_API kvq_status kvq_decode_workspace_size(const kvq_cache* cache, const kvq_decode_params* params,
                                             size_t* workspace_bytes) {
  return decode_workspace_size(cache, params, false, workspace_bytes);
}

KVQ_API kvq_status kvq_decode(const kvq_cache* cache, const kvq_decode_params* params, const void* q,
                              const int32_t* block_table, const int32_t* seq_lens, void* workspace,
                              size_t workspace_bytes, kvq_stream_t stream) {
  const int early = (params && (params->flags & KVQ_DECODE_EARLY_INPUTS)) ? 1 : 0;
  return decode_impl(cache, params, q, block_table, seq_lens, 1, early, false, workspace, workspace_bytes,
                     stream);
}

KVQ_API kvq_status kvq_combine(const kvq_cache* cache, const kvq_decode_params* params, const void* workspace,
                               size_t workspace_bytes, const float* head_sink, void* out, float* lse_out,
                               kvq_stream_t stream) {
  return combine_impl(cache, params, false, workspace, workspace_bytes, head_sink, out, lse_out, stream);
}

KVQ_API kvq_status kvq_prefill_workspace_size(const kvq_cache* cache, const kvq_decode_params* params,
                                              size_t* workspace_bytes) {
  if (!workspace_bytes) return KVQ_ERR_INVALID_ARG;
  kvq_cache eff_;
  if (kvq_status s = resolve_cache(cache, &eff_)) return s;
  kvq_decode_params v;
  int n = 0;
  bool qt = false;
  if (kvq_status s = prefill_shape(&eff_, params, &v, &n, &qt)) return s;
  size_t ws = 0;
  if (kvq_status s = decode_workspace_size(&eff_, &v, qt, &ws)) return s;
  *workspace_bytes = align256((size_t)v.batch * 4) + ws;
  return KVQ_OK;
}

KVQ_API kvq_status kvq_prefill(const kvq_cache* cache, const kvq_decode_params* params, const void* q,
                               const int32_t* block_table, const int32_t* seq_lens, const float* head_sink,
                               void* out, float* lse_out, void* workspace, size_t workspace_bytes,
                               kvq_stream_t stream) {
  kvq_cache eff_;
  if (kvq_status s = resolve_cache(cache, &eff_)) return s;
  cache = &eff_;
  kvq_decode_params v;
  int n = 0;
  bool qt = false;
  if (kvq_status s = prefill_shape(cache, params, &v, &n, &qt)) return s;
  if (kvq_status s = check_params(cache, &v, qt)) return s;
  if (params->batch == 0) return KVQ_OK;
  if (!q || !block_table || !seq_lens || !workspace || !out) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(workspace, 256) ||
      !aligned(out, 16) || (lse_out && !aligned(lse_out, 4)) || (head_sink && !aligned(head_sink, 4)))
    return KVQ_ERR_INVALID_ARG;
  size_t need = 0;
  if (kvq_status s = kvq_prefill_workspace_size(cache, params, &need)) return s;
  if (workspace_bytes < need) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  // the virtual sequences' lengths head the workspace; the decode reads them
  // only after it has waited for the kernel that writes them
  const size_t head = align256((size_t)v.batch * 4);
  int32_t* lens = static_cast<int32_t*>(workspace);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaError_t e = launch_prefill_lens(seq_lens, lens, params->batch, n, params->q_tokens, v.q_tokens, st))
    return from_cuda(e);
  char* ws = static_cast<char*>(workspace) + head;
  if (kvq_status s = decode_impl(cache, &v, q, block_table, lens, n, 0, qt, ws, workspace_bytes - head, stream))
    return s;
  // a chunk's B x C x Hq rows have few pieces each: one warp per row
  return combine_impl(cache, &v, qt, ws, workspace_bytes - head, head_sink, out, lse_out, stream, true);
}

KVQ_API kvq_status kvq_check_wait_timeout(uint32_t limit_us, kvq_stream_t stream) {
  if (limit_us == 0 || limit_us > 2000000u) return KVQ_ERR_INVALID_ARG;
  DeviceInfo* dev;
  if (kvq_status s = current_device(&dev)) return s;
  return from_cuda(launch_wait_probe(dev->err, 1000ull * limit_us, reinterpret_cast<cudaStream_t>(stream)));
}

KVQ_API kvq_status kvq_get_device_error(uint32_t* flags, int32_t clear, kvq_stream_t stream) {
  if (!flags) return KVQ_ERR_INVALID_ARG;
  DeviceInfo* dev;
  if (kvq_status s = current_device(&dev)) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return KVQ_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, dev->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return KVQ_ERR_CUDA;
  if (clear && cudaMemset(dev->err, 0, sizeof v) != cudaSuccess) return KVQ_ERR_CUDA;
  *flags = v;
  return (v & KVQ_DEVERR_TIMEOUT) ? KVQ_ERR_DEVICE_TIMEOUT : KVQ_OK;
}

}  // extern "C"
