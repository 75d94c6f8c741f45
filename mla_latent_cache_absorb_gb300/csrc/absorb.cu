// Absorb: q'[b,h,c] = sum_n q_nope[b,h,n] * W_UK[h][n,c], written with the rotated q_pe as the
// fused query row [q' ; q_pe] (act dtype) that the attention stage reads.
//
// moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs, folded SDPA chain: q_prime from the
// nope rows of kv_b (kv_b_per_head = nope + v_head_dim). turbospark-runtime 0.3.0,
// src/families/deepseek2/attn.rs: q_pe windows roped BEFORE the absorb gathers them into the
// fused [q' ; q_pe] rows.
//
// Per head this is a small GEMM (M = kv_lora, N = B, K = nope) whose cost is reading W_UK once;
// each CTA owns one head and a 64-column slice of the latent, stages that slice of W_UK
// (dequantised to float32) and the head's q_nope for a block of sequences in shared memory.
#include "common.cuh"

namespace mla {

constexpr int ABS_THREADS = 256;
constexpr int ABS_COLS = 64;     // latent columns per CTA
constexpr int ABS_BCHUNK = 32;   // sequences per shared-memory pass

// at most 64 registers: four CTAs share an SM (the grid is heads x 8 column blocks, often more
// than one wave)
template <int DT>
__global__ void __launch_bounds__(ABS_THREADS, 4)
absorb_kernel(mla_config cfg, const typename Act<DT>::T* __restrict__ q, const void* __restrict__ kv_b,
              const int32_t* __restrict__ positions, typename Act<DT>::T* __restrict__ q_abs,
              typename Act<DT>::T* __restrict__ q_res, int B, int pos_t) {
  // value v goes out as its storage rounding, and (bf16 only) the rounding residual to q_res
  auto put = [&](int64_t i, float v) {
    Act<DT>::store(q_abs, i, v);
    if (q_res != nullptr) Act<DT>::store(q_res, i, v - Act<DT>::rounded(v));
  };
  extern __shared__ float sm[];
  pdl_trigger();
  const int H = cfg.n_heads, C = cfg.kv_lora, N = cfg.qk_nope, R = cfg.qk_rope, V = cfg.v_head;
  const int h = blockIdx.x;
  const int c0 = blockIdx.y * ABS_COLS;
  const int qrow = N + R, arow = C + R;
  // sequences per shared-memory pass: no more than the batch has, so that small batches leave
  // room for more CTAs per SM
  const int bchunk = min(ABS_BCHUNK, B);
  float* w_s = sm;                          // [N][ABS_COLS]
  float* q_s = sm + N * ABS_COLS;           // [bchunk][N]
  float* red_s = q_s + bchunk * N;          // [4][bchunk][ABS_COLS] partial sums over nope quarters
  const int tid = threadIdx.x;

  // Loads of the first pass go out together: this thread's q_pe pair (the head's B*R/2 pairs
  // are shared out over the CTAs of the head), its q_nope elements of the first sequence chunk,
  // then the W_UK slice; nothing waits for a load before all of them are in flight.
  const int n_pairs = B * (R / 2);
  const int pair0 = blockIdx.y * ABS_THREADS + tid;
  const int pair_stride = gridDim.y * ABS_THREADS;
  float px0 = 0.f, px1 = 0.f;
  int ppos = 0;
  double pinv = 0.0;
  if (pair0 < n_pairs) {
    const int b = pair0 / (R / 2), p = pair0 % (R / 2);
    const int64_t qi = ((int64_t)b * H + h) * qrow + N + 2 * p;
    px0 = Act<DT>::load(q, qi);
    px1 = Act<DT>::load(q, qi + 1);
    if (positions != nullptr) {
      ppos = positions[b / pos_t] + b % pos_t;
      pinv = cfg.rope_inv_freq[p];
    }
  }
  constexpr int QPRE = 16;                  // q_nope elements prefetched per thread
  const int nb0 = min(ABS_BCHUNK, B);
  float qv[QPRE];
#pragma unroll
  for (int u = 0; u < QPRE; ++u) {
    const int i = tid + u * ABS_THREADS;
    qv[u] = 0.f;
    if (i < nb0 * N) qv[u] = Act<DT>::load(q, ((int64_t)(i / N) * H + h) * qrow + i % N);
  }
  const int64_t wrow0 = (int64_t)h * (N + V);
  stage_kv_b_rows(w_s, ABS_COLS, kv_b, cfg.kv_b_dtype, wrow0, N, c0, min(ABS_COLS, C - c0), C, ABS_THREADS,
                  (int64_t)cfg.n_heads * (cfg.qk_nope + cfg.v_head));
  pdl_wait();   // the fused query rows may still be read by the previous step's attention

  // q_pe: rotate at positions[b] (or copy when positions == NULL) into the row's tail
  for (int i = pair0; i < n_pairs; i += pair_stride) {
    const int b = i / (R / 2), p = i % (R / 2);
    if (i != pair0) {
      const int64_t qi = ((int64_t)b * H + h) * qrow + N + 2 * p;
      px0 = Act<DT>::load(q, qi);
      px1 = Act<DT>::load(q, qi + 1);
      if (positions != nullptr) {
        ppos = positions[b / pos_t] + b % pos_t;
        pinv = cfg.rope_inv_freq[p];
      }
    }
    const int64_t ai = ((int64_t)b * H + h) * arow + C + 2 * p;
    if (positions != nullptr) {
      float c, s;
      rope_cs_value(pinv, ppos, &c, &s);
      put(ai, px0 * c - px1 * s);
      put(ai + 1, px0 * s + px1 * c);
    } else {
      put(ai, px0);
      put(ai + 1, px1);
    }
  }

  // thread (cc, part): latent column c0 + cc, nope quarter `part`, every sequence of the chunk;
  // the four quarter sums are added in a fixed order afterwards
  const int cc = tid % ABS_COLS;
  const int part = tid / ABS_COLS;   // 0..3
  const int n_lo = part * N / 4, n_hi = (part + 1) * N / 4;
  for (int b0 = 0; b0 < B; b0 += bchunk) {
    const int nb = min(bchunk, B - b0);
    __syncthreads();
    if (b0 == 0) {
#pragma unroll
      for (int u = 0; u < QPRE; ++u) {
        const int i = tid + u * ABS_THREADS;
        if (i < nb * N) q_s[i] = qv[u];
      }
      for (int i = tid + QPRE * ABS_THREADS; i < nb * N; i += ABS_THREADS)
        q_s[i] = Act<DT>::load(q, ((int64_t)(i / N) * H + h) * qrow + i % N);
    } else {
      for (int i = tid; i < nb * N; i += ABS_THREADS) {
        const int bb = i / N, n = i % N;
        q_s[bb * N + n] = Act<DT>::load(q, ((int64_t)(b0 + bb) * H + h) * qrow + n);
      }
    }
    __syncthreads();
    for (int bb = 0; bb < nb; ++bb) {
      float acc = 0.f;
      for (int n = n_lo; n < n_hi; ++n) acc = fmaf(q_s[bb * N + n], w_s[n * ABS_COLS + cc], acc);
      red_s[(part * bchunk + bb) * ABS_COLS + cc] = acc;
    }
    __syncthreads();
    for (int i = tid; i < nb * ABS_COLS; i += ABS_THREADS) {
      const int bb = i / ABS_COLS, c = i % ABS_COLS;
      if (c0 + c < C) {
        const float* r = red_s + bb * ABS_COLS + c;
        const float v = ((r[0] + r[bchunk * ABS_COLS]) + r[2 * bchunk * ABS_COLS]) + r[3 * bchunk * ABS_COLS];
        put(((int64_t)(b0 + bb) * H + h) * arow + c0 + c, v);
      }
    }
  }
}

cudaError_t launch_absorb(const mla_config& cfg, const void* q, const void* kv_b,
                          const int32_t* positions, void* q_abs, void* q_res, int B, bool pdl, cudaStream_t st,
                          int pos_t) {
  if (pos_t < 1) return cudaErrorInvalidValue;
  dim3 grid(cfg.n_heads, (cfg.kv_lora + ABS_COLS - 1) / ABS_COLS);
  const size_t bchunk = (size_t)(B < ABS_BCHUNK ? B : ABS_BCHUNK);
  const size_t smem = sizeof(float) * ((size_t)cfg.qk_nope * ABS_COLS + bchunk * cfg.qk_nope + 4 * bchunk * ABS_COLS);
  if (cfg.act_dtype == MLA_BF16) {
    auto k = absorb_kernel<MLA_BF16>;
    cudaError_t e = ensure_smem((const void*)k, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(pdl, k, grid, dim3(ABS_THREADS), smem, st, cfg, static_cast<const uint16_t*>(q), kv_b, positions,
                      static_cast<uint16_t*>(q_abs), static_cast<uint16_t*>(q_res), B, pos_t);
  } else {
    auto k = absorb_kernel<MLA_F32>;
    cudaError_t e = ensure_smem((const void*)k, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(pdl, k, grid, dim3(ABS_THREADS), smem, st, cfg, static_cast<const float*>(q), kv_b, positions,
                      static_cast<float*>(q_abs), static_cast<float*>(nullptr), B, pos_t);
  }
}

}  // namespace mla
