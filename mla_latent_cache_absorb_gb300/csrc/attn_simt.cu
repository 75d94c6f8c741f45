// Split attention over the compressed cache rows on CUDA cores (float32 arithmetic).
//
// turbospark-runtime 0.3.0, src/families/deepseek2/attn.rs, MQA attention over the compressed
// rows: the key is the whole row [kv_lat ; k_pe], the value is its first kv_lora elements, all
// heads read the same rows. moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs,
// mla_sdpa_folded over cache_len = pos + 1 rows.
//
// This is the general path: any dimensions, float32 or bf16 storage. Grid (split, sequence,
// head group); a CTA stages a tile of rows (as float32) once for all of its heads, keeps an
// online softmax per head and writes the split's normalised latent sum and log-sum-exp.
#include "common.cuh"

#include <math_constants.h>

namespace mla {

constexpr int SIMT_THREADS = 256;
constexpr int SIMT_TT = 16;          // rows per staged tile
constexpr int SIMT_MAXO = 16;        // (head, latent) outputs per thread

struct SimtArgs {
  RowMap map;
  const void* rows;
  const int32_t* seq_lens;
  const void* q_abs;
  const uint16_t* q_res;   // bf16 rounding residual of q_abs (bf16 rows) or nullptr
  float* part_o;
  float* part_lse;
  int32_t* meta;
  WsHeader* hdr;
  int H, C, R, hpb, S;
  int64_t chunk;
  float scale;
  // query tokens per sequence (heads token-major, kvb_heads per token): head m sees the rows
  // before L - tokens + 1 + m / kvb_heads
  int tokens, kvb_heads;
};

template <int DT>
__global__ void __launch_bounds__(SIMT_THREADS) attn_simt_kernel(SimtArgs a) {
  using T = typename Act<DT>::T;
  extern __shared__ float sm[];
  pdl_trigger();
  pdl_wait();   // fused query rows from the absorb, the appended row, partials the combine reads
  const int s = blockIdx.x, b = blockIdx.y, g = blockIdx.z;
  const int row = a.C + a.R;
  const int h0 = g * a.hpb;
  const int nh = min(a.hpb, a.H - h0);
  const int64_t L = a.seq_lens[b];
  const bool len_ok = (L >= 1 && L >= a.tokens && L <= a.map.capacity());
  if (threadIdx.x == 0 && s == 0 && g == 0) {
    // slots of sequence b for the combine stage: b*S .. b*S + ceil(L/chunk) - 1
    a.meta[2 * b] = b * a.S;
    a.meta[2 * b + 1] = len_ok ? (int)((L + a.chunk - 1) / a.chunk) : 0;
    if (!len_ok) set_error(a.hdr, MLA_ERR_BAD_SEQ_LEN, b);
  }
  if (!len_ok) return;  // the combine stage writes NaN for this sequence
  const int64_t t0 = (int64_t)s * a.chunk;
  const int64_t t1 = min(L, t0 + a.chunk);
  float* po = a.part_o + (((int64_t)b * a.S + s) * a.H + h0) * a.C;
  float* pl = a.part_lse + ((int64_t)b * a.S + s) * a.H + h0;
  if (t0 >= t1) return;   // beyond this sequence: the combine stage never reads this slot

  float* q_s = sm;                          // [hpb][row]
  float* tile = q_s + a.hpb * row;          // [TT][row]
  float* p_s = tile + SIMT_TT * row;        // [hpb][TT]
  float* m_s = p_s + a.hpb * SIMT_TT;       // [hpb]
  float* l_s = m_s + a.hpb;                 // [hpb]
  float* al_s = l_s + a.hpb;                // [hpb]
  int* bad_s = reinterpret_cast<int*>(al_s + a.hpb);

  const T* qa = static_cast<const T*>(a.q_abs);
  for (int i = threadIdx.x; i < nh * row; i += SIMT_THREADS) {
    const int64_t qi = ((int64_t)b * a.H + h0) * row + i;
    q_s[i] = Act<DT>::load(qa, qi) + (a.q_res != nullptr ? bf16_bits_to_f32(a.q_res[qi]) : 0.f);
  }
  for (int i = threadIdx.x; i < a.hpb; i += SIMT_THREADS) {
    m_s[i] = -CUDART_INF_F;
    l_s[i] = 0.f;
  }
  if (threadIdx.x == 0) *bad_s = 0;

  const int n_out = nh * a.C;
  float acc[SIMT_MAXO];
#pragma unroll
  for (int k = 0; k < SIMT_MAXO; ++k) acc[k] = 0.f;

  const T* rows = static_cast<const T*>(a.rows);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t tb = t0; tb < t1; tb += SIMT_TT) {
    const int nt = (int)min((int64_t)SIMT_TT, t1 - tb);
    __syncthreads();
    for (int i = threadIdx.x; i < nt * row; i += SIMT_THREADS) {
      const int tt = i / row, d = i % row;
      const int64_t pr = a.map.phys(b, tb + tt);
      if (pr < 0) { *bad_s = 1; continue; }
      tile[i] = Act<DT>::load(rows, pr * row + d);
    }
    __syncthreads();
    if (*bad_s) {
      if (threadIdx.x == 0) set_error(a.hdr, MLA_ERR_BAD_PAGE, b);
      for (int i = threadIdx.x; i < nh; i += SIMT_THREADS) pl[i] = CUDART_NAN_F;
      return;
    }
    // scores: one warp per (head, row) pair
    for (int pr = warp; pr < nh * SIMT_TT; pr += SIMT_THREADS / 32) {
      const int hh = pr / SIMT_TT, tt = pr % SIMT_TT;
      float d = 0.f;
      if (tt < nt)
        for (int k = lane; k < row; k += 32) d = fmaf(q_s[hh * row + k], tile[tt * row + k], d);
      d = warp_sum(d);
      const bool seen = tt < nt && tb + tt < L - a.tokens + 1 + (h0 + hh) / a.kvb_heads;
      if (lane == 0) p_s[hh * SIMT_TT + tt] = seen ? d * a.scale : -CUDART_INF_F;
    }
    __syncthreads();
    // online softmax, one thread per head
    for (int hh = threadIdx.x; hh < nh; hh += SIMT_THREADS) {
      float mx = m_s[hh];
      for (int tt = 0; tt < nt; ++tt) mx = fmaxf(mx, p_s[hh * SIMT_TT + tt]);
      // exp(-inf) = 0 on the first tile; a head that sees no row yet keeps its zero sums
      const float alpha = mx == -CUDART_INF_F ? 1.f : expf(m_s[hh] - mx);
      float sum = 0.f;
      for (int tt = 0; tt < SIMT_TT; ++tt) {
        const float sc = p_s[hh * SIMT_TT + tt];
        const float p = (tt < nt && sc != -CUDART_INF_F) ? expf(sc - mx) : 0.f;
        p_s[hh * SIMT_TT + tt] = p;
        sum += p;
      }
      l_s[hh] = l_s[hh] * alpha + sum;
      m_s[hh] = mx;
      al_s[hh] = alpha;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < SIMT_MAXO; ++k) {
      const int idx = threadIdx.x + k * SIMT_THREADS;
      if (idx < n_out) {
        const int hh = idx / a.C, c = idx % a.C;
        float o = acc[k] * al_s[hh];
        for (int tt = 0; tt < nt; ++tt) o = fmaf(p_s[hh * SIMT_TT + tt], tile[tt * row + c], o);
        acc[k] = o;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < SIMT_MAXO; ++k) {
    const int idx = threadIdx.x + k * SIMT_THREADS;
    if (idx < n_out) {
      const int hh = idx / a.C, c = idx % a.C;
      // l = 0: no row of this split is visible to the head: O = 0, lse = -inf (weight 0)
      po[(int64_t)hh * a.C + c] = l_s[hh] > 0.f ? acc[k] / l_s[hh] : 0.f;
    }
  }
  for (int hh = threadIdx.x; hh < nh; hh += SIMT_THREADS)
    pl[hh] = l_s[hh] > 0.f ? m_s[hh] + logf(l_s[hh]) : -CUDART_INF_F;
}

int simt_heads_per_cta(const mla_config& cfg) {
  int hpb = (SIMT_THREADS * SIMT_MAXO) / cfg.kv_lora;
  if (hpb > cfg.n_heads) hpb = cfg.n_heads;
  if (hpb > 16) hpb = 16;
  return hpb < 1 ? 1 : hpb;
}

size_t simt_smem_bytes(const mla_config& cfg, int hpb) {
  const int row = cfg.kv_lora + cfg.qk_rope;
  return sizeof(float) * ((size_t)hpb * row + (size_t)SIMT_TT * row + (size_t)hpb * SIMT_TT + 3 * hpb + 1);
}

cudaError_t launch_attn_simt(const mla_config& cfg, const mla_cache& cache, const DecodePlan& plan,
                             const int32_t* seq_lens, const void* q_abs, const void* q_res, float* part_o,
                             float* part_lse, int32_t* meta, int B, WsHeader* hdr, cudaStream_t st) {
  SimtArgs a;
  a.map = RowMap{cache.page_table, cfg.page_size, cfg.max_pages_per_seq, cfg.rows_per_seq,
                 cache.n_physical_rows};
  a.rows = cache.rows;
  a.seq_lens = seq_lens;
  a.q_abs = q_abs;
  a.q_res = static_cast<const uint16_t*>(q_res);
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.meta = meta;
  a.hdr = hdr;
  a.H = cfg.n_heads; a.C = cfg.kv_lora; a.R = cfg.qk_rope;
  a.hpb = plan.heads_per_cta;
  a.S = plan.splits;
  a.chunk = plan.chunk_rows;
  a.scale = cfg.softmax_scale;
  a.tokens = plan.tokens;
  a.kvb_heads = plan.kvb_heads;
  if (a.tokens < 1 || a.kvb_heads < 1 || a.tokens * a.kvb_heads != cfg.n_heads) return cudaErrorInvalidValue;
  dim3 grid(plan.splits, B, plan.n_groups);
  const size_t smem = simt_smem_bytes(cfg, plan.heads_per_cta);
  cudaError_t e;
  if (cfg.act_dtype == MLA_BF16) {
    e = ensure_smem((const void*)attn_simt_kernel<MLA_BF16>, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_simt_kernel<MLA_BF16>, grid, dim3(SIMT_THREADS), smem, st, a);
  } else {
    e = ensure_smem((const void*)attn_simt_kernel<MLA_F32>, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_simt_kernel<MLA_F32>, grid, dim3(SIMT_THREADS), smem, st, a);
  }
}

}  // namespace mla
