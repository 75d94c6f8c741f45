// Cache append: optional kv_a projection, RMSNorm over the latent, consecutive-pair YaRN
// RoPE over the k_pe tail, one rounding into the cache row.
//
// turbospark-runtime 0.3.0, src/families/deepseek2/attn.rs, encode_mla_attention_block:
// kv_a straight into the compressed row [latent ; k_pe], norm over kv_lora in place, RoPE of
// the pe tail in place with the same (consecutive-element) pairing as q.
// moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs, mla_attn_layer_forward_gpu: KV-A
// chain, kv_a_layernorm, YaRN RoPE of k_pe, append of row[pos]; PosMismatch / CacheFull guards.
//
// Here the finished row is produced in registers (float32) and written once, so the cache
// never holds a half-finished row and the value is rounded to the cache dtype only once. The
// kv_a projection itself, when asked for, is the layer-projection GEMV of proj.cu.
#include "common.cuh"

namespace mla {

// ---- finish: norm + rope + store, one CTA per sequence ---------------------------------------
constexpr int FIN_THREADS = 128;
constexpr int FIN_MAX_PER_THREAD = 16;   // row elements per thread: C+R <= 2048

template <int DT>
__global__ void __launch_bounds__(FIN_THREADS)
append_finish_kernel(mla_config cfg, RowMap map, typename Act<DT>::T* __restrict__ rows_out,
                     const float* __restrict__ kva, const float* __restrict__ norm_w,
                     const int32_t* __restrict__ positions, const int32_t* __restrict__ seq_lens,
                     WsHeader* hdr, int kva_dep) {
  pdl_trigger();
  const int b = blockIdx.x;
  const int C = cfg.kv_lora, R = cfg.qk_rope, row = C + R;
  // every load that does not depend on another goes out first: the row (unless the projection
  // kernel just before produces it), the norm weights, this thread's RoPE pair and frequency,
  // the position and the length
  float v[FIN_MAX_PER_THREAD], wn[FIN_MAX_PER_THREAD];
  const float* src = kva + (int64_t)b * row;
  const bool has_pair = threadIdx.x < R / 2;
  float x0 = 0.f, x1 = 0.f;
  auto load_row = [&]() {
#pragma unroll
    for (int k = 0; k < FIN_MAX_PER_THREAD; ++k) {
      const int i = threadIdx.x + k * FIN_THREADS;
      v[k] = (i < row) ? src[i] : 0.f;
    }
    if (has_pair) {
      x0 = src[C + 2 * threadIdx.x];
      x1 = src[C + 2 * threadIdx.x + 1];
    }
  };
  if (!kva_dep) load_row();
#pragma unroll
  for (int k = 0; k < FIN_MAX_PER_THREAD; ++k) {
    const int i = threadIdx.x + k * FIN_THREADS;
    wn[k] = (i < C) ? norm_w[i] : 0.f;
  }
  const int pos = positions[b];
  const int len = seq_lens != nullptr ? seq_lens[b] : pos;
  // this thread's RoPE angle, before the wait (float64 arithmetic is slow on this GPU: the
  // frequency is split into a float pair once and the angle formed in float where that holds)
  float rc = 1.f, rs = 0.f;
  if (has_pair) {
    float fh, fl;
    rope_freq_split(cfg.rope_inv_freq, threadIdx.x, &fh, &fl);
    rope_cs_split(cfg.rope_inv_freq, fh, fl, threadIdx.x, pos, &rc, &rs);
  }
  pdl_wait();   // the cache row may still be read by the previous step's attention
  if (kva_dep) load_row();
  if (len != pos) {
    if (threadIdx.x == 0) set_error(hdr, MLA_ERR_POS_MISMATCH, b);
    return;
  }
  if (pos < 0 || (int64_t)pos >= map.capacity()) {
    if (threadIdx.x == 0) set_error(hdr, MLA_ERR_CACHE_FULL, b);
    return;
  }
  const int64_t pr = map.phys(b, pos);
  if (pr < 0 || pr >= map.n_phys) {
    if (threadIdx.x == 0) set_error(hdr, MLA_ERR_BAD_PAGE, b);
    return;
  }

  __shared__ float red[FIN_THREADS / 32];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < FIN_MAX_PER_THREAD; ++k) {
    const int i = threadIdx.x + k * FIN_THREADS;
    if (i < C) ss = fmaf(v[k], v[k], ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < FIN_THREADS / 32; ++w) tot += red[w];
  const float inv_rms = 1.0f / sqrtf(tot / static_cast<float>(C) + cfg.rms_eps);

  typename Act<DT>::T* dst = rows_out + pr * row;
#pragma unroll
  for (int k = 0; k < FIN_MAX_PER_THREAD; ++k) {
    const int i = threadIdx.x + k * FIN_THREADS;
    if (i < C) Act<DT>::store(dst, i, v[k] * inv_rms * wn[k]);
  }
  // RoPE over the pe tail: one thread per pair (2i, 2i+1)
  if (has_pair) {
    Act<DT>::store(dst, C + 2 * threadIdx.x, x0 * rc - x1 * rs);
    Act<DT>::store(dst, C + 2 * threadIdx.x + 1, x0 * rs + x1 * rc);
  }
  for (int i = threadIdx.x + FIN_THREADS; i < R / 2; i += FIN_THREADS) {   // R / 2 > 128 only
    float c, s;
    rope_cs(cfg.rope_inv_freq, i, pos, &c, &s);
    const float y0 = src[C + 2 * i], y1 = src[C + 2 * i + 1];
    Act<DT>::store(dst, C + 2 * i, y0 * c - y1 * s);
    Act<DT>::store(dst, C + 2 * i + 1, y0 * s + y1 * c);
  }
}

cudaError_t launch_append_finish(const mla_config& cfg, const mla_cache& cache, const float* kva,
                                 const float* norm_w, const int32_t* positions,
                                 const int32_t* seq_lens, int B, WsHeader* hdr, bool kva_dep, cudaStream_t st) {
  RowMap map{cache.page_table, cfg.page_size, cfg.max_pages_per_seq, cfg.rows_per_seq,
             cache.n_physical_rows};
  if (cfg.act_dtype == MLA_BF16)
    return launch_pdl(append_finish_kernel<MLA_BF16>, dim3(B), dim3(FIN_THREADS), 0, st, cfg, map,
                      static_cast<uint16_t*>(cache.rows), kva, norm_w, positions, seq_lens, hdr, (int)kva_dep);
  return launch_pdl(append_finish_kernel<MLA_F32>, dim3(B), dim3(FIN_THREADS), 0, st, cfg, map,
                    static_cast<float*>(cache.rows), kva, norm_w, positions, seq_lens, hdr, (int)kva_dep);
}

}  // namespace mla
