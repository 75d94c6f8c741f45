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

template <int DT>
__global__ void __launch_bounds__(ABS_THREADS)
absorb_kernel(mla_config cfg, const typename Act<DT>::T* __restrict__ q, const void* __restrict__ kv_b,
              const int32_t* __restrict__ positions, typename Act<DT>::T* __restrict__ q_abs,
              typename Act<DT>::T* __restrict__ q_res, int B) {
  // value v goes out as its storage rounding, and (bf16 only) the rounding residual to q_res
  auto put = [&](int64_t i, float v) {
    Act<DT>::store(q_abs, i, v);
    if (q_res != nullptr) Act<DT>::store(q_res, i, v - Act<DT>::load(q_abs, i));
  };
  extern __shared__ float sm[];
  const int H = cfg.n_heads, C = cfg.kv_lora, N = cfg.qk_nope, R = cfg.qk_rope, V = cfg.v_head;
  const int h = blockIdx.x;
  const int c0 = blockIdx.y * ABS_COLS;
  const int qrow = N + R, arow = C + R;
  float* w_s = sm;                          // [N][ABS_COLS]
  float* q_s = sm + N * ABS_COLS;           // [ABS_BCHUNK][N]

  const int64_t wrow0 = (int64_t)h * (N + V);
  stage_kv_b_rows(w_s, ABS_COLS, kv_b, cfg.kv_b_dtype, wrow0, N, c0, min(ABS_COLS, C - c0), C, ABS_THREADS);

  const int cc = threadIdx.x % ABS_COLS;
  const int bsub = threadIdx.x / ABS_COLS;   // 0..3
  for (int b0 = 0; b0 < B; b0 += ABS_BCHUNK) {
    const int nb = min(ABS_BCHUNK, B - b0);
    __syncthreads();
    for (int i = threadIdx.x; i < nb * N; i += ABS_THREADS) {
      const int bb = i / N, n = i % N;
      q_s[bb * N + n] = Act<DT>::load(q, ((int64_t)(b0 + bb) * H + h) * qrow + n);
    }
    __syncthreads();
    if (c0 + cc < C) {
      for (int bb = bsub; bb < nb; bb += ABS_THREADS / ABS_COLS) {
        float acc = 0.f;
        for (int n = 0; n < N; ++n) acc = fmaf(q_s[bb * N + n], w_s[n * ABS_COLS + cc], acc);
        put(((int64_t)(b0 + bb) * H + h) * arow + c0 + cc, acc);
      }
    }
  }

  // q_pe: rotate at positions[b] (or copy when positions == NULL) into the row's tail
  if (blockIdx.y == 0) {
    for (int i = threadIdx.x; i < B * (R / 2); i += ABS_THREADS) {
      const int b = i / (R / 2), p = i % (R / 2);
      const int64_t qi = ((int64_t)b * H + h) * qrow + N + 2 * p;
      const int64_t ai = ((int64_t)b * H + h) * arow + C + 2 * p;
      const float x0 = Act<DT>::load(q, qi), x1 = Act<DT>::load(q, qi + 1);
      if (positions != nullptr) {
        float c, s;
        rope_cs(cfg.rope_inv_freq, p, positions[b], &c, &s);
        put(ai, x0 * c - x1 * s);
        put(ai + 1, x0 * s + x1 * c);
      } else {
        put(ai, x0);
        put(ai + 1, x1);
      }
    }
  }
}

cudaError_t launch_absorb(const mla_config& cfg, const void* q, const void* kv_b,
                          const int32_t* positions, void* q_abs, void* q_res, int B, cudaStream_t st) {
  dim3 grid(cfg.n_heads, (cfg.kv_lora + ABS_COLS - 1) / ABS_COLS);
  const size_t smem = sizeof(float) * ((size_t)cfg.qk_nope * ABS_COLS + (size_t)ABS_BCHUNK * cfg.qk_nope);
  if (cfg.act_dtype == MLA_BF16) {
    auto k = absorb_kernel<MLA_BF16>;
    cudaError_t e = ensure_smem((const void*)k, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, ABS_THREADS, smem, st>>>(cfg, static_cast<const uint16_t*>(q), kv_b, positions,
                                       static_cast<uint16_t*>(q_abs), static_cast<uint16_t*>(q_res), B);
  } else {
    auto k = absorb_kernel<MLA_F32>;
    cudaError_t e = ensure_smem((const void*)k, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<grid, ABS_THREADS, smem, st>>>(cfg, static_cast<const float*>(q), kv_b, positions,
                                       static_cast<float*>(q_abs), nullptr, B);
  }
  return cudaGetLastError();
}

}  // namespace mla
