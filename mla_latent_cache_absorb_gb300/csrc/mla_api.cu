// The C ABI of libmla: host validation, workspace layout, split plan and kernel launches.
// Every entry point validates on the host before enqueueing anything; kernels report what
// only the GPU can see through the workspace's error word.
#include <cmath>
#include <algorithm>
#include <atomic>
#include <cstring>
#include <limits>

#include "common.cuh"

namespace mla {

static bool checked_mul(uint64_t a, uint64_t b, uint64_t* out) {
  if (a != 0 && b > std::numeric_limits<uint64_t>::max() / a) return false;
  *out = a * b;
  return true;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static size_t act_size(int dt) { return dt == MLA_BF16 ? 2 : 4; }

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Dimensions and dtypes shared by every call.
static mla_status check_cfg(const mla_config* cfg) {
  if (cfg == nullptr) return MLA_ERR_INVALID_ARG;
  if (cfg->n_heads < 1 || cfg->kv_lora < 1 || cfg->qk_nope < 1 || cfg->qk_rope < 2 ||
      (cfg->qk_rope & 1) || cfg->v_head < 1)
    return MLA_ERR_INVALID_ARG;
  if (cfg->act_dtype != MLA_F32 && cfg->act_dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
  if (cfg->kv_b_dtype != MLA_F32 && cfg->kv_b_dtype != MLA_BF16 && cfg->kv_b_dtype != MLA_Q8_0 &&
      cfg->kv_b_dtype != MLA_Q4_AFFINE)
    return MLA_ERR_INVALID_ARG;
  if (cfg->kv_b_dtype == MLA_Q8_0 && (cfg->kv_lora % 32) != 0) return MLA_ERR_BAD_KV_B;
  if (cfg->kv_b_dtype == MLA_Q4_AFFINE && (cfg->kv_lora % 64) != 0) return MLA_ERR_BAD_KV_B;
  if (cfg->page_size < 0) return MLA_ERR_INVALID_ARG;
  if (cfg->page_size == 0 && cfg->rows_per_seq < 1) return MLA_ERR_INVALID_ARG;
  if (cfg->page_size > 0 && cfg->max_pages_per_seq < 1) return MLA_ERR_INVALID_ARG;
  if (!(cfg->softmax_scale > 0.f) || !std::isfinite(cfg->softmax_scale)) return MLA_ERR_INVALID_ARG;
  // implementation limits of the kernels (row staged per thread / per CTA)
  if (cfg->kv_lora + cfg->qk_rope > 2048 || cfg->qk_nope > 512 || cfg->kv_lora > 4096)
    return MLA_ERR_UNSUPPORTED;
  // row stride must keep 16-byte alignment for vectorised row access
  if (((int64_t)(cfg->kv_lora + cfg->qk_rope) * (int64_t)act_size(cfg->act_dtype)) % 16 != 0)
    return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

static mla_status check_cache(const mla_config* cfg, const mla_cache* cache, int B) {
  if (cache == nullptr || cache->rows == nullptr || cache->n_physical_rows < 1) return MLA_ERR_INVALID_ARG;
  if (!aligned(cache->rows, 16)) return MLA_ERR_INVALID_ARG;
  if (cfg->page_size > 0) {
    if (cache->page_table == nullptr) return MLA_ERR_INVALID_ARG;
  } else {
    uint64_t need;
    if (!checked_mul((uint64_t)B, (uint64_t)cfg->rows_per_seq, &need)) return MLA_ERR_INVALID_ARG;
    if ((uint64_t)cache->n_physical_rows < need) return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

static std::atomic<uint64_t> g_wait_ns{kWaitDrainNs};

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

int device_sms() {
  static std::atomic<int> cached[64] = {};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) {
    n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

int simt_heads_per_cta(const mla_config& cfg);

// The split plan: how many row splits per sequence, how many rows each, and where the
// workspace keeps the fused query rows and the per-split partials.
// tokens > 1: cfg.n_heads counts tokens x (heads of kv_b) per sequence, token-major; the SM-pair
// kernel (one head per row of its tile, no per-head row limit) is not used then.
static mla_status make_plan(const mla_config& cfg, int B, DecodePlan* p, int tokens = 1) {
  const int sms = device_sms();
  if (sms <= 0) return MLA_ERR_CUDA;
  std::memset(p, 0, sizeof(*p));
  if (tokens < 1 || cfg.n_heads % tokens != 0) return MLA_ERR_INVALID_ARG;
  p->tokens = tokens;
  p->kvb_heads = cfg.n_heads / tokens;
  p->capacity = cfg.page_size == 0 ? cfg.rows_per_seq : (int64_t)cfg.max_pages_per_seq * cfg.page_size;
  const int max_pairs = tokens == 1 && attn_pair_supported(cfg) ? attn_pair_max_pairs() : -1;
  if (max_pairs > 0) {
    // 128 heads: one cluster of two CTAs per SM pair, the 64-row tile list split evenly over
    // the pairs that fit on the device at once
    p->path = PATH_PAIR;
    p->heads_per_cta = cfg.n_heads;
    p->n_groups = 1;
    p->ctas_per_group = max_pairs < sms / 2 ? max_pairs : sms / 2;
    if (p->ctas_per_group < 1) p->ctas_per_group = 1;
    const int64_t max_tiles = (int64_t)B * ((p->capacity + 63) / 64);
    if (max_tiles < p->ctas_per_group) p->ctas_per_group = (int)max_tiles;
    p->splits = p->ctas_per_group;
    p->chunk_rows = 0;
    p->part_groups = 1;
    p->part_hpg = cfg.n_heads;
    p->n_slots = p->ctas_per_group + B - 1;
  } else if (attn_tc_supported(cfg)) {
    // tensor-core path: one CTA per SM, each head group's tile list split evenly over its CTAs
    p->path = PATH_TC;
    p->heads_per_cta = tc_heads_per_cta(cfg.n_heads);
    p->n_groups = (cfg.n_heads + p->heads_per_cta - 1) / p->heads_per_cta;
    p->ctas_per_group = sms / p->n_groups > 0 ? sms / p->n_groups : 1;
    // never more CTAs than the batch can have 128-row tiles
    const int64_t max_tiles = (int64_t)B * ((p->capacity + 127) / 128);
    if (max_tiles < p->ctas_per_group) p->ctas_per_group = (int)max_tiles;
    p->splits = p->ctas_per_group;
    p->chunk_rows = 0;
    p->part_groups = p->n_groups;
    p->part_hpg = p->heads_per_cta;
    p->n_slots = p->ctas_per_group + B - 1;
  } else {
    // CUDA-core path: grid (split, sequence, head group) with equal row splits
    p->path = PATH_SIMT;
    p->heads_per_cta = simt_heads_per_cta(cfg);
    p->n_groups = (cfg.n_heads + p->heads_per_cta - 1) / p->heads_per_cta;
    const int64_t tile = 16;
    const int64_t per_seq_ctas = (int64_t)B * p->n_groups;
    int64_t want = (2 * sms + per_seq_ctas - 1) / per_seq_ctas;
    if (want < 1) want = 1;
    if (want > 64) want = 64;
    int64_t chunk = (p->capacity + want - 1) / want;
    chunk = ((chunk + tile - 1) / tile) * tile;
    p->chunk_rows = chunk;
    p->splits = (int)((p->capacity + chunk - 1) / chunk);
    p->part_groups = 1;
    p->part_hpg = cfg.n_heads;
    p->n_slots = B * p->splits;
  }

  const size_t row = (size_t)(cfg.kv_lora + cfg.qk_rope);
  const size_t n_part = (size_t)p->part_groups * p->n_slots * p->part_hpg;
  size_t off = sizeof(WsHeader);
  p->off_qabs = off;
  off = align256(off + (size_t)B * cfg.n_heads * row * act_size(cfg.act_dtype));
  p->off_qres = off;
  if (cfg.act_dtype == MLA_BF16) off = align256(off + (size_t)B * cfg.n_heads * row * 2);
  p->off_po = off;
  off = align256(off + n_part * cfg.kv_lora * sizeof(float));
  p->off_plse = off;
  off = align256(off + n_part * sizeof(float));
  p->off_meta = off;
  off = align256(off + (size_t)B * 2 * sizeof(int32_t));
  p->small = decode_small_supported(cfg, B, tokens) ? 1 : 0;
  if (p->small) {
    const size_t rows_q = (size_t)B * cfg.n_heads;
    p->off_sq = off;
    off = align256(off + rows_q * row * sizeof(float));
    p->off_sp = off;
    off = align256(off + rows_q * (size_t)decode_small_max_chunks(cfg) * (cfg.kv_lora + 4) * sizeof(float));
    p->off_sw = off;
    off = align256(off + rows_q * (size_t)(cfg.kv_lora / 64) * cfg.v_head * sizeof(float));
    p->off_sc = off;
    off = align256(off + rows_q * sizeof(uint32_t));
  }
  p->total = off;
  return MLA_OK;
}

cudaError_t ensure_smem(const void* func, int bytes) {
  // per host thread: no locking, and setting the attribute again from another thread is harmless
  struct Entry { const void* f; int dev; int bytes; };
  thread_local Entry table[128];
  thread_local int n = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (table[i].f == func && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  for (int i = 0; i < n; ++i)
    if (table[i].f == func && table[i].dev == dev) { table[i].bytes = bytes; return cudaSuccess; }
  if (n < 128) table[n++] = Entry{func, dev, bytes};
  return cudaSuccess;
}

static mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

// A projection's in_dim against its weight dtype: a multiple of 8 (16-byte vectors of x), of 32
// for Q8_0 blocks, of 64 for the 4-bit groups.
static bool proj_in_dim_ok(int64_t k, int dt) {
  if (k < 8 || k > (int64_t(1) << 30) || k % 8 != 0) return false;
  if (dt == MLA_Q8_0) return k % 32 == 0;
  if (dt == MLA_Q4_AFFINE) return k % 64 == 0;
  return dt == MLA_F32 || dt == MLA_BF16;
}

static mla_status check_proj(const mla_config* cfg, const mla_proj* pj, int B) {
  mla_status st = check_cfg(cfg);
  if (st != MLA_OK) return st;
  if (pj == nullptr || B < 1) return MLA_ERR_INVALID_ARG;
  if (pj->w_dtype != MLA_F32 && pj->w_dtype != MLA_BF16 && pj->w_dtype != MLA_Q8_0 &&
      pj->w_dtype != MLA_Q4_AFFINE)
    return MLA_ERR_UNSUPPORTED;
  if (!proj_in_dim_ok(pj->hidden, pj->w_dtype) || pj->q_lora < 0) return MLA_ERR_INVALID_ARG;
  if (pj->q_lora > 0 && !proj_in_dim_ok(pj->q_lora, pj->w_dtype)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

static mla_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || !aligned(ws, 256)) return MLA_ERR_WORKSPACE;
  if (ws_bytes < need) return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_POS_MISMATCH: return "append position does not match the sequence length";
    case MLA_ERR_CACHE_FULL: return "append position beyond the cache capacity";
    case MLA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MLA_ERR_TIMEOUT: return "a bounded device wait timed out";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_BAD_SEQ_LEN: return "sequence length below 1 or above the cache capacity";
    case MLA_ERR_BAD_PAGE: return "page-table entry out of range";
    case MLA_ERR_BAD_KV_B: return "kv_b dtype, shape or size does not match the configuration";
  }
  return "unknown status";
}

int32_t mla_abi_version(void) { return 1; }

uint64_t mla_set_wait_limit_ns(uint64_t ns) {
  return g_wait_ns.exchange(ns == 0 ? kWaitDrainNs : ns, std::memory_order_relaxed);
}

mla_status mla_yarn_inv_freq(int32_t rope_dim, double theta, double factor, int32_t orig_max_pos,
                             double beta_fast, double beta_slow, double* out_host) {
  if (out_host == nullptr || rope_dim < 2 || (rope_dim & 1) || !(theta > 1.0) || orig_max_pos < 1)
    return MLA_ERR_INVALID_ARG;
  const int half = rope_dim / 2;
  const double d = static_cast<double>(rope_dim);
  double lo = 0, hi = 1;
  const bool yarn = factor > 1.0;
  if (yarn) {
    if (!(beta_fast > 0) || !(beta_slow > 0)) return MLA_ERR_INVALID_ARG;
    const double two_pi = 6.283185307179586476925286766559;
    // correction dimension: the pair index whose wavelength fits n_rot turns into the
    // original context
    auto corr = [&](double n_rot) {
      return d * std::log(static_cast<double>(orig_max_pos) / (n_rot * two_pi)) / (2.0 * std::log(theta));
    };
    lo = std::floor(corr(beta_fast));
    hi = std::ceil(corr(beta_slow));
    if (lo < 0) lo = 0;
    if (hi > d - 1) hi = d - 1;
    if (lo == hi) hi += 0.001;
  }
  for (int i = 0; i < half; ++i) {
    const double base = std::pow(theta, -2.0 * i / d);
    if (!yarn) {
      out_host[i] = base;
      continue;
    }
    double r = (i - lo) / (hi - lo);
    r = r < 0 ? 0 : (r > 1 ? 1 : r);
    out_host[i] = base / factor * r + base * (1.0 - r);
  }
  return MLA_OK;
}

double mla_yarn_mscale(double factor, double coeff) {
  return factor <= 1.0 ? 1.0 : 1.0 + 0.1 * coeff * std::log(factor);
}

float mla_softmax_scale(int32_t qk_nope, int32_t qk_rope, double mscale) {
  if (qk_nope < 0 || qk_rope < 0 || qk_nope + qk_rope < 1) return 0.f;
  return static_cast<float>(mscale * mscale / std::sqrt(static_cast<double>(qk_nope + qk_rope)));
}

mla_status mla_validate_kv_b(int32_t dtype, int64_t rows, int64_t cols, uint64_t size_bytes,
                             int32_t heads, int32_t nope, int32_t kv_lora, int32_t v_dim) {
  if (heads < 1 || nope < 1 || kv_lora < 1 || v_dim < 1) return MLA_ERR_INVALID_ARG;
  if (dtype != MLA_F32 && dtype != MLA_BF16 && dtype != MLA_Q8_0 && dtype != MLA_Q4_AFFINE) return MLA_ERR_BAD_KV_B;
  uint64_t exp_rows;
  if (!checked_mul((uint64_t)heads, (uint64_t)nope + (uint64_t)v_dim, &exp_rows)) return MLA_ERR_BAD_KV_B;
  if (rows < 0 || cols < 0 || (uint64_t)rows != exp_rows || cols != kv_lora) return MLA_ERR_BAD_KV_B;
  uint64_t row_bytes;
  if (dtype == MLA_Q8_0) {
    if (kv_lora % 32 != 0) return MLA_ERR_BAD_KV_B;
    if (!checked_mul((uint64_t)(kv_lora / 32), 34u, &row_bytes)) return MLA_ERR_BAD_KV_B;
  } else if (dtype == MLA_Q4_AFFINE) {
    if (kv_lora % 64 != 0) return MLA_ERR_BAD_KV_B;
    // codes (cols / 2 bytes) plus a bf16 scale and bias per 64 columns
    row_bytes = (uint64_t)kv_lora / 2 + (uint64_t)(kv_lora / 64) * 4u;
  } else {
    if (!checked_mul((uint64_t)kv_lora, dtype == MLA_BF16 ? 2u : 4u, &row_bytes)) return MLA_ERR_BAD_KV_B;
  }
  uint64_t total;
  if (!checked_mul(exp_rows, row_bytes, &total)) return MLA_ERR_BAD_KV_B;
  return total == size_bytes ? MLA_OK : MLA_ERR_BAD_KV_B;
}

uint64_t mla_kv_b_bytes(const mla_config* cfg) {
  if (cfg == nullptr || cfg->n_heads < 1 || cfg->qk_nope < 1 || cfg->v_head < 1 || cfg->kv_lora < 1) return 0;
  uint64_t rows, row_bytes, total;
  if (!checked_mul((uint64_t)cfg->n_heads, (uint64_t)cfg->qk_nope + (uint64_t)cfg->v_head, &rows)) return 0;
  if (cfg->kv_b_dtype == MLA_Q8_0) {
    if (cfg->kv_lora % 32) return 0;
    row_bytes = (uint64_t)(cfg->kv_lora / 32) * 34u;
  } else if (cfg->kv_b_dtype == MLA_Q4_AFFINE) {
    if (cfg->kv_lora % 64) return 0;
    row_bytes = (uint64_t)cfg->kv_lora / 2 + (uint64_t)(cfg->kv_lora / 64) * 4u;
  } else if (cfg->kv_b_dtype == MLA_BF16) {
    row_bytes = (uint64_t)cfg->kv_lora * 2u;
  } else if (cfg->kv_b_dtype == MLA_F32) {
    row_bytes = (uint64_t)cfg->kv_lora * 4u;
  } else {
    return 0;
  }
  if (!checked_mul(rows, row_bytes, &total)) return 0;
  return total;
}

mla_status mla_append_workspace_size(const mla_config* cfg, int32_t B, size_t* bytes) {
  mla_status st = check_cfg(cfg);
  if (st != MLA_OK) return st;
  if (B < 1 || bytes == nullptr) return MLA_ERR_INVALID_ARG;
  *bytes = align256(sizeof(WsHeader) + (size_t)B * (cfg->kv_lora + cfg->qk_rope) * sizeof(float));
  return MLA_OK;
}

mla_status mla_decode_workspace_size(const mla_config* cfg, int32_t B, size_t* bytes) {
  mla_status st = check_cfg(cfg);
  if (st != MLA_OK) return st;
  if (B < 1 || bytes == nullptr) return MLA_ERR_INVALID_ARG;
  DecodePlan p;
  st = make_plan(*cfg, B, &p);
  if (st != MLA_OK) return st;
  *bytes = p.total;
  return MLA_OK;
}

mla_status mla_decode_plan(const mla_config* cfg, int32_t B, mla_plan_info* info) {
  mla_status st = check_cfg(cfg);
  if (st != MLA_OK) return st;
  if (B < 1 || info == nullptr) return MLA_ERR_INVALID_ARG;
  DecodePlan p;
  st = make_plan(*cfg, B, &p);
  if (st != MLA_OK) return st;
  info->kernel = p.path;
  info->heads_per_cta = p.heads_per_cta;
  info->head_groups = p.n_groups;
  info->splits = p.splits;
  info->rows_per_split = p.chunk_rows;   // 0: tiles are balanced across CTAs instead
  info->capacity = p.capacity;
  if (p.small) {   // mla_decode_attn runs the one-launch path
    info->kernel = 3;
    info->heads_per_cta = cfg->n_heads;
    info->head_groups = 1;
    info->splits = decode_small_grid(*cfg, B);
    info->rows_per_split = 32;
  }
  return MLA_OK;
}

mla_status mla_cache_append(const mla_config* cfg, const mla_cache* cache, const void* kv_in,
                            const void* w_kva, int32_t hidden, const float* norm_w,
                            const int32_t* positions, const int32_t* seq_lens, int32_t B,
                            void* workspace, size_t ws_bytes, mla_stream_t stream) {
  mla_status st = check_cfg(cfg);
  if (st != MLA_OK) return st;
  if (B < 1 || kv_in == nullptr || norm_w == nullptr || positions == nullptr) return MLA_ERR_INVALID_ARG;
  if (cfg->rope_inv_freq == nullptr) return MLA_ERR_INVALID_ARG;
  st = check_cache(cfg, cache, B);
  if (st != MLA_OK) return st;
  if (w_kva != nullptr) {
    if (hidden < 8 || hidden % 8 != 0 || !aligned(kv_in, 16) || !aligned(w_kva, 16)) return MLA_ERR_INVALID_ARG;
  }
  size_t need;
  st = mla_append_workspace_size(cfg, B, &need);
  if (st != MLA_OK) return st;
  st = check_ws(workspace, ws_bytes, need);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  WsHeader* hdr = static_cast<WsHeader*>(workspace);
  const float* kva = static_cast<const float*>(kv_in);
  if (w_kva != nullptr) {
    float* kva_ws = reinterpret_cast<float*>(static_cast<char*>(workspace) + sizeof(WsHeader));
    st = cuda_status(launch_proj(kv_in, cfg->act_dtype == MLA_BF16, hidden, B, cfg->act_dtype, w_kva,
                                 cfg->kv_lora + cfg->qk_rope, kva_ws, false, nullptr, 0, nullptr, false, s));
    if (st != MLA_OK) return st;
    kva = kva_ws;
  }
  return cuda_status(launch_append_finish(*cfg, *cache, kva, norm_w, positions, seq_lens, B, hdr,
                                          w_kva != nullptr, s));
}

static mla_status decode_prologue(const mla_config* cfg, int32_t B, void* workspace, size_t ws_bytes,
                                  DecodePlan* plan) {
  mla_status st = check_cfg(cfg);
  if (st != MLA_OK) return st;
  if (B < 1) return MLA_ERR_INVALID_ARG;
  st = make_plan(*cfg, B, plan);
  if (st != MLA_OK) return st;
  return check_ws(workspace, ws_bytes, plan->total);
}

}  // extern "C"

namespace {

// The three stages, enqueued with a plan already made and arguments already checked.

// ordered: launch the absorb without programmatic serialization, so that it starts only after
// all earlier work on the stream has completed
mla_status enqueue_absorb(const mla_config* cfg, const DecodePlan& plan, const void* q, const void* kv_b,
                          const int32_t* positions, int32_t B, void* workspace, bool ordered, cudaStream_t s) {
  void* q_abs = static_cast<char*>(workspace) + plan.off_qabs;
  void* q_res = cfg->act_dtype == MLA_BF16 ? static_cast<char*>(workspace) + plan.off_qres : nullptr;
  if (absorb_tc_supported(*cfg, B))
    return cuda_status(launch_absorb_tc(*cfg, q, kv_b, positions, q_abs, q_res, B, static_cast<WsHeader*>(workspace),
                                        !ordered, s));
  return cuda_status(launch_absorb(*cfg, q, kv_b, positions, q_abs, q_res, B, !ordered, s));
}

// kv_early: the kernel just before is an ordered absorb (enqueue_absorb with ordered = true)
mla_status enqueue_partial(const mla_config* cfg, const DecodePlan& plan, const mla_cache* cache,
                           const int32_t* seq_lens, int32_t B, void* workspace, bool kv_early, cudaStream_t s) {
  char* ws = static_cast<char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  float* po = reinterpret_cast<float*>(ws + plan.off_po);
  float* pl = reinterpret_cast<float*>(ws + plan.off_plse);
  int32_t* meta = reinterpret_cast<int32_t*>(ws + plan.off_meta);
  const void* q_res = cfg->act_dtype == MLA_BF16 ? ws + plan.off_qres : nullptr;
  if (plan.path == PATH_PAIR)
    return cuda_status(
        launch_attn_pair(*cfg, *cache, plan, seq_lens, ws + plan.off_qabs, q_res, po, pl, meta, B, hdr, kv_early, s));
  if (plan.path == PATH_TC)
    return cuda_status(
        launch_attn_tc(*cfg, *cache, plan, seq_lens, ws + plan.off_qabs, q_res, po, pl, meta, B, hdr, kv_early, s));
  return cuda_status(launch_attn_simt(*cfg, *cache, plan, seq_lens, ws + plan.off_qabs, q_res, po, pl, meta, B, hdr, s));
}

mla_status enqueue_combine(const mla_config* cfg, const DecodePlan& plan, const void* kv_b, float* out, float* lse,
                           int32_t B, void* workspace, cudaStream_t s) {
  char* ws = static_cast<char*>(workspace);
  const int32_t* meta = reinterpret_cast<const int32_t*>(ws + plan.off_meta);
  const float* po = reinterpret_cast<const float*>(ws + plan.off_po);
  const float* pl = reinterpret_cast<const float*>(ws + plan.off_plse);
  // the tensor-core attention scores used bf16 latent queries: correct the LSE for the residual
  const void* q_res = plan.path != PATH_SIMT ? ws + plan.off_qres : nullptr;
  if (combine_tc_supported(*cfg, B))
    return cuda_status(launch_combine_tc(*cfg, plan, kv_b, meta, po, pl, q_res, out, lse, B,
                                         reinterpret_cast<WsHeader*>(ws), s));
  return cuda_status(launch_combine(*cfg, plan, kv_b, meta, po, pl, q_res, out, lse, B, s));
}

mla_status check_absorb_args(const mla_config* cfg, const void* q, const void* kv_b, const int32_t* positions) {
  if (q == nullptr || kv_b == nullptr) return MLA_ERR_INVALID_ARG;
  if (positions != nullptr && cfg->rope_inv_freq == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_b, 16)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status mla_decode_absorb(const mla_config* cfg, const void* q, const void* kv_b,
                             const int32_t* positions, int32_t B, void* workspace, size_t ws_bytes,
                             mla_stream_t stream) {
  DecodePlan plan;
  mla_status st = decode_prologue(cfg, B, workspace, ws_bytes, &plan);
  if (st != MLA_OK) return st;
  st = check_absorb_args(cfg, q, kv_b, positions);
  if (st != MLA_OK) return st;
  return enqueue_absorb(cfg, plan, q, kv_b, positions, B, workspace, false, reinterpret_cast<cudaStream_t>(stream));
}

mla_status mla_decode_partial(const mla_config* cfg, const mla_cache* cache, const int32_t* seq_lens,
                              int32_t B, void* workspace, size_t ws_bytes, mla_stream_t stream) {
  DecodePlan plan;
  mla_status st = decode_prologue(cfg, B, workspace, ws_bytes, &plan);
  if (st != MLA_OK) return st;
  if (seq_lens == nullptr) return MLA_ERR_INVALID_ARG;
  st = check_cache(cfg, cache, B);
  if (st != MLA_OK) return st;
  return enqueue_partial(cfg, plan, cache, seq_lens, B, workspace, false, reinterpret_cast<cudaStream_t>(stream));
}

mla_status mla_decode_combine(const mla_config* cfg, const void* kv_b, const int32_t* seq_lens,
                              float* out, float* lse, int32_t B, void* workspace, size_t ws_bytes,
                              mla_stream_t stream) {
  DecodePlan plan;
  mla_status st = decode_prologue(cfg, B, workspace, ws_bytes, &plan);
  if (st != MLA_OK) return st;
  if (kv_b == nullptr || out == nullptr) return MLA_ERR_INVALID_ARG;
  (void)seq_lens;   // the partial stage recorded each sequence's slots (and validity) in meta
  if (!aligned(kv_b, 16)) return MLA_ERR_INVALID_ARG;
  return enqueue_combine(cfg, plan, kv_b, out, lse, B, workspace, reinterpret_cast<cudaStream_t>(stream));
}

mla_status mla_decode_attn(const mla_config* cfg, const void* q, const void* kv_b, const mla_cache* cache,
                           const int32_t* seq_lens, const int32_t* positions, float* out, float* lse,
                           int32_t B, void* workspace, size_t ws_bytes, mla_stream_t stream) {
  // validate everything before the first launch, so a bad argument enqueues nothing; the plan
  // is made once for the three stages
  DecodePlan plan;
  mla_status st = decode_prologue(cfg, B, workspace, ws_bytes, &plan);
  if (st != MLA_OK) return st;
  st = check_absorb_args(cfg, q, kv_b, positions);
  if (st != MLA_OK) return st;
  if (seq_lens == nullptr || out == nullptr) return MLA_ERR_INVALID_ARG;
  st = check_cache(cfg, cache, B);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (plan.small) {
    // tiny batches: the whole decode in one launch
    char* ws = static_cast<char*>(workspace);
    return cuda_status(launch_decode_small(*cfg, *cache, q, kv_b, seq_lens, positions, out, lse, B,
                                           reinterpret_cast<float*>(ws + plan.off_sq),
                                           reinterpret_cast<float*>(ws + plan.off_sp),
                                           reinterpret_cast<float*>(ws + plan.off_sw),
                                           reinterpret_cast<unsigned int*>(ws + plan.off_sc),
                                           reinterpret_cast<WsHeader*>(ws), s));
  }
  // Long attentions (at the cache's capacity, at least four 128-row tiles per CTA, or eight
  // 64-row tiles per CTA pair): the absorb starts once everything before it on the stream, the
  // cache append above all, has completed, and the attention then streams cache rows while the
  // absorb still runs. Short ones keep the absorb's own overlap with the kernels before it,
  // which is worth more to them.
  const int64_t tiles128 = (int64_t)B * ((plan.capacity + 127) / 128);
  const int64_t tiles64 = (int64_t)B * ((plan.capacity + 63) / 64);
  const bool early = (plan.path == PATH_TC && tiles128 >= 4 * (int64_t)plan.ctas_per_group) ||
                     (plan.path == PATH_PAIR && tiles64 >= 8 * (int64_t)plan.ctas_per_group);
  st = enqueue_absorb(cfg, plan, q, kv_b, positions, B, workspace, early, s);
  if (st != MLA_OK) return st;
  st = enqueue_partial(cfg, plan, cache, seq_lens, B, workspace, early, s);
  if (st != MLA_OK) return st;
  return enqueue_combine(cfg, plan, kv_b, out, lse, B, workspace, s);
}

mla_status mla_get_device_error(const void* workspace, int32_t* seq_out, mla_stream_t stream) {
  if (workspace == nullptr) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  int32_t h[2];
  if (cudaMemcpy(h, workspace, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (seq_out != nullptr) *seq_out = h[1];
  return static_cast<mla_status>(h[0]);
}

mla_status mla_clear_device_error(void* workspace, mla_stream_t stream) {
  if (workspace == nullptr) return MLA_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(WsHeader), reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

// The layer projections' workspace: a 256-byte header (the device error word) and, as a call
// needs them, the float32 q_lat rows, the bf16 hi / lo halves of a float32 input (tensor-core
// path) and the split partials of the tensor-core GEMMs (reused by the calls of one front end,
// which run in stream order).
struct ProjWs {
  ProjTcPlan pa, pb;            // front end: first launch (q_a or q, with kv_a), q_b; o_proj: pa
  size_t off_qlat, off_hi, off_lo, off_part, total;
};

size_t align_up256(size_t x) { return (x + 255) & ~size_t(255); }

mla_status front_end_ws(const mla_config* cfg, const mla_proj* pj, int32_t B, ProjWs* w) {
  const int64_t q_rows = (int64_t)cfg->n_heads * (cfg->qk_nope + cfg->qk_rope);
  // the kv_a rows count in the plan whether or not they are computed, so that q's column slices
  // (and so its rounding) do not depend on it
  const int64_t kva_rows = cfg->kv_lora + cfg->qk_rope;
  const bool chain = pj->q_lora > 0;
  const bool xb = cfg->act_dtype == MLA_BF16;
  w->pa = proj_tc_plan(chain ? pj->q_lora : q_rows, kva_rows, pj->hidden, B, false, xb ? pj->w_dtype : -1);
  w->pb = chain ? proj_tc_plan(q_rows, 0, pj->q_lora, B, true, pj->w_dtype) : ProjTcPlan{};
  size_t off = sizeof(WsHeader);
  w->off_qlat = off;
  if (chain) off = align_up256(off + (size_t)B * pj->q_lora * sizeof(float));
  w->off_hi = off;
  if (w->pb.use) off = align_up256(off + (size_t)B * pj->q_lora * 2);
  w->off_lo = off;
  if (w->pb.use) off = align_up256(off + (size_t)B * pj->q_lora * 2);
  w->off_part = off;
  const int64_t part = std::max<int64_t>(w->pa.use ? w->pa.part_floats : 0, w->pb.use ? w->pb.part_floats : 0);
  off = align_up256(off + (size_t)part * sizeof(float));
  w->total = off;
  return MLA_OK;
}

mla_status o_proj_ws(const mla_config* cfg, const mla_proj* pj, int32_t B, ProjWs* w) {
  const int64_t k = (int64_t)cfg->n_heads * cfg->v_head;
  w->pa = proj_tc_plan(pj->hidden, 0, (int)k, B, true, pj->w_dtype);
  w->pb = ProjTcPlan{};
  size_t off = sizeof(WsHeader);
  w->off_qlat = off;
  w->off_hi = off;
  if (w->pa.use) off = align_up256(off + (size_t)B * k * 2);
  w->off_lo = off;
  if (w->pa.use) off = align_up256(off + (size_t)B * k * 2);
  w->off_part = off;
  off = align_up256(off + (size_t)(w->pa.use ? w->pa.part_floats : 0) * sizeof(float));
  w->total = off;
  return MLA_OK;
}

}  // namespace

extern "C" {

mla_status mla_front_end_workspace_size(const mla_config* cfg, const mla_proj* pj, int32_t B, size_t* bytes) {
  mla_status st = check_proj(cfg, pj, B);
  if (st != MLA_OK) return st;
  if (bytes == nullptr) return MLA_ERR_INVALID_ARG;
  ProjWs w;
  st = front_end_ws(cfg, pj, B, &w);
  if (st != MLA_OK) return st;
  *bytes = w.total;
  return MLA_OK;
}

mla_status mla_o_proj_workspace_size(const mla_config* cfg, const mla_proj* pj, int32_t B, size_t* bytes) {
  mla_status st = check_proj(cfg, pj, B);
  if (st != MLA_OK) return st;
  if (bytes == nullptr) return MLA_ERR_INVALID_ARG;
  if (!proj_in_dim_ok((int64_t)cfg->n_heads * cfg->v_head, pj->w_dtype)) return MLA_ERR_INVALID_ARG;
  ProjWs w;
  st = o_proj_ws(cfg, pj, B, &w);
  if (st != MLA_OK) return st;
  *bytes = w.total;
  return MLA_OK;
}

mla_status mla_proj_launches(const mla_config* cfg, const mla_proj* pj, int32_t B, int32_t* front_end,
                             int32_t* o_proj) {
  mla_status st = check_proj(cfg, pj, B);
  if (st != MLA_OK) return st;
  ProjWs w;
  if (front_end != nullptr) {
    st = front_end_ws(cfg, pj, B, &w);
    if (st != MLA_OK) return st;
    int n = 1 + (w.pa.use && w.pa.splits > 1 ? 1 : 0);                // q_a (or q) with kv_a
    if (pj->q_lora > 0) n += 2 + (w.pb.use && w.pb.splits > 1 ? 1 : 0);  // norm, q_b
    *front_end = n;
  }
  if (o_proj != nullptr) {
    if (!proj_in_dim_ok((int64_t)cfg->n_heads * cfg->v_head, pj->w_dtype)) return MLA_ERR_INVALID_ARG;
    st = o_proj_ws(cfg, pj, B, &w);
    if (st != MLA_OK) return st;
    *o_proj = w.pa.use ? 2 + (w.pa.splits > 1 ? 1 : 0) : 1;           // halves, GEMM, reduction
  }
  return MLA_OK;
}

mla_status mla_front_end(const mla_config* cfg, const mla_proj* pj, const void* x, void* q, float* kva,
                         int32_t B, void* workspace, size_t ws_bytes, mla_stream_t stream) {
  mla_status st = check_proj(cfg, pj, B);
  if (st != MLA_OK) return st;
  if (x == nullptr || q == nullptr || pj->w_q == nullptr || !aligned(x, 16) || !aligned(pj->w_q, 16))
    return MLA_ERR_INVALID_ARG;
  if (kva != nullptr && (pj->w_kva == nullptr || !aligned(pj->w_kva, 16))) return MLA_ERR_INVALID_ARG;
  const bool chain = pj->q_lora > 0;
  if (chain && (pj->w_q_a == nullptr || pj->q_a_norm_w == nullptr || !aligned(pj->w_q_a, 16) ||
                !(pj->q_norm_eps >= 0.f) || !std::isfinite(pj->q_norm_eps)))
    return MLA_ERR_INVALID_ARG;
  ProjWs w;
  st = front_end_ws(cfg, pj, B, &w);
  if (st != MLA_OK) return st;
  st = check_ws(workspace, ws_bytes, w.total);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  WsHeader* hdr = reinterpret_cast<WsHeader*>(ws);
  float* part = reinterpret_cast<float*>(ws + w.off_part);
  const bool xb = cfg->act_dtype == MLA_BF16;
  const int64_t q_rows = (int64_t)cfg->n_heads * (cfg->qk_nope + cfg->qk_rope);
  const int64_t kva_rows = cfg->kv_lora + cfg->qk_rope;
  const void* w1 = kva != nullptr ? pj->w_kva : nullptr;
  // first launch: q (or q_lat) and kv_a from x, one read of x
  void* y0 = chain ? static_cast<void*>(ws + w.off_qlat) : q;
  const int64_t rows0 = chain ? pj->q_lora : q_rows;
  const bool y0_bf16 = !chain && xb;
  if (w.pa.use)
    st = cuda_status(launch_proj_tc(w.pa, x, nullptr, pj->hidden, B, chain ? pj->w_q_a : pj->w_q, rows0, y0, y0_bf16,
                                    w1, kva_rows, kva, false, part, hdr, s));
  else
    st = cuda_status(launch_proj(x, xb, pj->hidden, B, pj->w_dtype, chain ? pj->w_q_a : pj->w_q, rows0, y0, y0_bf16,
                                 w1, kva_rows, kva, false, s));
  if (st != MLA_OK || !chain) return st;
  float* q_lat = reinterpret_cast<float*>(ws + w.off_qlat);
  uint16_t* hi = reinterpret_cast<uint16_t*>(ws + w.off_hi);
  uint16_t* lo = reinterpret_cast<uint16_t*>(ws + w.off_lo);
  st = cuda_status(launch_rms_norm_rows(q_lat, pj->q_a_norm_w, pj->q_lora, B, pj->q_norm_eps, s,
                                        w.pb.use ? hi : nullptr, w.pb.use ? lo : nullptr));
  if (st != MLA_OK) return st;
  if (w.pb.use)
    return cuda_status(launch_proj_tc(w.pb, hi, lo, pj->q_lora, B, pj->w_q, q_rows, q, xb, nullptr, 0, nullptr, false,
                                      part, hdr, s));
  return cuda_status(launch_proj(q_lat, false, pj->q_lora, B, pj->w_dtype, pj->w_q, q_rows, q, xb, nullptr, 0,
                                 nullptr, false, s));
}

mla_status mla_o_proj(const mla_config* cfg, const mla_proj* pj, const float* attn, float* y, int32_t B,
                      void* workspace, size_t ws_bytes, mla_stream_t stream) {
  mla_status st = check_proj(cfg, pj, B);
  if (st != MLA_OK) return st;
  const int64_t k = (int64_t)cfg->n_heads * cfg->v_head;
  if (!proj_in_dim_ok(k, pj->w_dtype)) return MLA_ERR_INVALID_ARG;
  if (attn == nullptr || y == nullptr || pj->w_o == nullptr || !aligned(attn, 16) || !aligned(pj->w_o, 16))
    return MLA_ERR_INVALID_ARG;
  ProjWs w;
  st = o_proj_ws(cfg, pj, B, &w);
  if (st != MLA_OK) return st;
  st = check_ws(workspace, ws_bytes, w.total);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  if (!w.pa.use)
    return cuda_status(launch_proj(attn, false, (int)k, B, pj->w_dtype, pj->w_o, pj->hidden, y, false, nullptr, 0,
                                   nullptr, false, s));
  uint16_t* hi = reinterpret_cast<uint16_t*>(ws + w.off_hi);
  uint16_t* lo = reinterpret_cast<uint16_t*>(ws + w.off_lo);
  st = cuda_status(launch_split_hi_lo(attn, (int64_t)B * k, hi, lo, s));
  if (st != MLA_OK) return st;
  return cuda_status(launch_proj_tc(w.pa, hi, lo, (int)k, B, pj->w_o, pj->hidden, y, false, nullptr, 0, nullptr, false,
                                    reinterpret_cast<float*>(ws + w.off_part), reinterpret_cast<WsHeader*>(ws), s));
}

// ---- several query tokens per sequence -------------------------------------------------------
// The T tokens of a sequence attend as T x H heads of one sequence (token-major), so every
// staged row tile serves all of them; the absorb sees B x T query rows of H heads.

static mla_status multi_cfg(const mla_config* cfg, int32_t tokens, mla_config* out) {
  mla_status st = check_cfg(cfg);
  if (st != MLA_OK) return st;
  if (tokens < 1 || tokens > 64 || (int64_t)tokens * cfg->n_heads > 65536) return MLA_ERR_INVALID_ARG;
  *out = *cfg;
  out->n_heads = tokens * cfg->n_heads;
  return MLA_OK;
}

mla_status mla_decode_multi_workspace_size(const mla_config* cfg, int32_t tokens, int32_t B, size_t* bytes) {
  if (tokens == 1) return mla_decode_workspace_size(cfg, B, bytes);
  mla_config vc;
  mla_status st = multi_cfg(cfg, tokens, &vc);
  if (st != MLA_OK) return st;
  if (B < 1 || bytes == nullptr) return MLA_ERR_INVALID_ARG;
  DecodePlan p;
  st = make_plan(vc, B, &p, tokens);
  if (st != MLA_OK) return st;
  *bytes = p.total;
  return MLA_OK;
}

mla_status mla_decode_attn_multi(const mla_config* cfg, int32_t tokens, const void* q, const void* kv_b,
                                 const mla_cache* cache, const int32_t* seq_lens, const int32_t* positions,
                                 float* out, float* lse, int32_t B, void* workspace, size_t ws_bytes,
                                 mla_stream_t stream) {
  if (tokens == 1)
    return mla_decode_attn(cfg, q, kv_b, cache, seq_lens, positions, out, lse, B, workspace, ws_bytes, stream);
  mla_config vc;
  mla_status st = multi_cfg(cfg, tokens, &vc);
  if (st != MLA_OK) return st;
  if (B < 1 || (int64_t)B * tokens >= (int64_t(1) << 31)) return MLA_ERR_INVALID_ARG;
  DecodePlan plan;
  st = make_plan(vc, B, &plan, tokens);
  if (st != MLA_OK) return st;
  st = check_ws(workspace, ws_bytes, plan.total);
  if (st != MLA_OK) return st;
  st = check_absorb_args(cfg, q, kv_b, positions);
  if (st != MLA_OK) return st;
  if (seq_lens == nullptr || out == nullptr) return MLA_ERR_INVALID_ARG;
  st = check_cache(&vc, cache, B);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t tiles128 = (int64_t)B * ((plan.capacity + 127) / 128);
  const bool early = plan.path == PATH_TC && tiles128 >= 4 * (int64_t)plan.ctas_per_group;
  // absorb: B x T query rows of H heads (query row b*T + i sits at positions[b] + i); the fused
  // rows land as [B][T*H][C+R], the attention's T*H heads per sequence
  void* q_abs = static_cast<char*>(workspace) + plan.off_qabs;
  void* q_res = cfg->act_dtype == MLA_BF16 ? static_cast<char*>(workspace) + plan.off_qres : nullptr;
  const int bq = B * tokens;
  if (absorb_tc_supported(*cfg, bq))
    st = cuda_status(launch_absorb_tc(*cfg, q, kv_b, positions, q_abs, q_res, bq, static_cast<WsHeader*>(workspace),
                                      !early, s, tokens));
  else
    st = cuda_status(launch_absorb(*cfg, q, kv_b, positions, q_abs, q_res, bq, !early, s, tokens));
  if (st != MLA_OK) return st;
  st = enqueue_partial(&vc, plan, cache, seq_lens, B, workspace, early, s);
  if (st != MLA_OK) return st;
  return enqueue_combine(&vc, plan, kv_b, out, lse, B, workspace, s);
}

}  // extern "C"
