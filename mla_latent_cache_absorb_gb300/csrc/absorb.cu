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

  // The W_UK slice is staged before the dependency wait; after it, this thread's q_pe pair (the
  // head's B*R/2 pairs are shared out over the CTAs of the head) and its q_nope elements of the
  // first sequence chunk go out together.
  const int n_pairs = B * (R / 2);
  const int pair0 = blockIdx.y * ABS_THREADS + tid;
  const int pair_stride = gridDim.y * ABS_THREADS;
  float px0 = 0.f, px1 = 0.f;
  int ppos = 0;
  double pinv = 0.0;
  if (pair0 < n_pairs && positions != nullptr) {
    const int b = pair0 / (R / 2), p = pair0 % (R / 2);
    ppos = positions[b / pos_t] + b % pos_t;
    pinv = cfg.rope_inv_freq[p];
  }
  const int64_t wrow0 = (int64_t)h * (N + V);
  stage_kv_b_rows(w_s, ABS_COLS, kv_b, cfg.kv_b_dtype, wrow0, N, c0, min(ABS_COLS, C - c0), C, ABS_THREADS,
                  (int64_t)cfg.n_heads * (cfg.qk_nope + cfg.v_head));
  // q may be written by a kernel two or more launches back (the front end): every read of it
  // comes after the wait for the previous kernel, which completes only after that one's own wait
  pdl_wait();
  if (pair0 < n_pairs) {
    const int b = pair0 / (R / 2), p = pair0 % (R / 2);
    const int64_t qi = ((int64_t)b * H + h) * qrow + N + 2 * p;
    px0 = Act<DT>::load(q, qi);
    px1 = Act<DT>::load(q, qi + 1);
  }
  constexpr int QPRE = 16;                  // q_nope elements loaded together per thread
  const int nb0 = min(ABS_BCHUNK, B);
  float qv[QPRE];
#pragma unroll
  for (int u = 0; u < QPRE; ++u) {
    const int i = tid + u * ABS_THREADS;
    qv[u] = 0.f;
    if (i < nb0 * N) qv[u] = Act<DT>::load(q, ((int64_t)(i / N) * H + h) * qrow + i % N);
  }

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

// ---- small batches (B <= 8), bf16 or Q8_0 kv_b: the weights stream in as raw bytes ----
// One CTA per (head, 256 latent columns). Before the dependency wait every thread issues its
// share of the slice of W_UK as 16-byte cp.async pieces of the raw rows (Q8_0: 272 bytes, bf16:
// 512 bytes per row), so the whole slice is in flight at once; the q_nope rows come after the
// wait. Thread (column quad cq, row quarter rq) decodes its four columns of 32 rows from shared
// memory (Q8_0: the codes' bytes go into the mantissa of 2^23 and 2^23 + 128 is subtracted,
// exact, then times the block scale) and accumulates all sequences; the four quarter sums are
// added in a fixed order.
constexpr int ABS_S_THREADS = 256;
constexpr int ABS_S_COLS = 256;
constexpr int ABS_S_BMAX = 8;

template <int DT, int WDT, int BT>   // BT: sequences of the batch rounded up to 1, 2, 4 or 8
__global__ void __launch_bounds__(ABS_S_THREADS, 2)
absorb_small_kernel(mla_config cfg, const typename Act<DT>::T* __restrict__ q, const uint8_t* __restrict__ kv_b,
                    const int32_t* __restrict__ positions, typename Act<DT>::T* __restrict__ q_abs,
                    typename Act<DT>::T* __restrict__ q_res, int B, int pos_t) {
  auto put = [&](int64_t i, float v) {
    Act<DT>::store(q_abs, i, v);
    if (q_res != nullptr) Act<DT>::store(q_res, i, v - Act<DT>::rounded(v));
  };
  extern __shared__ __align__(16) uint8_t sm_raw[];
  pdl_trigger();
  const int H = cfg.n_heads, C = cfg.kv_lora, N = cfg.qk_nope, R = cfg.qk_rope, V = cfg.v_head;
  const int h = blockIdx.x, lh = blockIdx.y;
  const int qrow = N + R, arow = C + R;
  constexpr int RB = WDT == MLA_Q8_0 ? ABS_S_COLS / 32 * 34 : ABS_S_COLS * 2;   // raw bytes of a row slice
  const int64_t row_bytes = WDT == MLA_Q8_0 ? (int64_t)(C / 32) * 34 : (int64_t)C * 2;
  uint8_t* w_s = sm_raw;                                              // [N][RB]
  float* q_s = reinterpret_cast<float*>(sm_raw + N * RB);             // [B][N]
  float* red_s = q_s + ABS_S_BMAX * N;                                // [4][B][256]
  const int tid = threadIdx.x;

  // the slice of W_UK: rows h (N + V) .. + N, bytes lh RB .. + RB of each
  {
    const uint8_t* src0 = kv_b + (int64_t)h * (N + V) * row_bytes + (int64_t)lh * RB;
    constexpr int PPR = RB / 16;   // pieces per row
    for (int i = tid; i < N * PPR; i += ABS_S_THREADS) {
      const int r = i / PPR, pc = i - r * PPR;
      const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(w_s + r * RB + pc * 16));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src0 + r * row_bytes + pc * 16)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  // this CTA's share of the q_pe pairs (the head's B R/2 pairs over its C/256 CTAs); the
  // frequencies as float pairs, before the dependency wait (positions and frequencies are inputs)
  __shared__ float f_hi[32], f_lo[32];   // R <= 64
  const int n_pairs = B * (R / 2);
  const int pair_stride = gridDim.y * ABS_S_THREADS;
  const int pair0 = lh * ABS_S_THREADS + tid;
  if (positions != nullptr && tid < R / 2) rope_freq_split(cfg.rope_inv_freq, tid, &f_hi[tid], &f_lo[tid]);
  pdl_wait();   // q may come from the kernel before; the fused rows may still be read by the previous step
  __syncthreads();
  // every load of q first (this thread's q_nope elements and its first pair), then the stores
  constexpr int QPT = (ABS_S_BMAX * 128 + ABS_S_THREADS - 1) / ABS_S_THREADS;
  float qn[QPT];
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = tid + u * ABS_S_THREADS;
    qn[u] = (i < B * N) ? Act<DT>::load(q, ((int64_t)(i / N) * H + h) * qrow + i % N) : 0.f;
  }
  float px0 = 0.f, px1 = 0.f;
  if (pair0 < n_pairs) {
    const int b = pair0 / (R / 2), p = pair0 % (R / 2);
    const int64_t qi = ((int64_t)b * H + h) * qrow + N + 2 * p;
    px0 = Act<DT>::load(q, qi);
    px1 = Act<DT>::load(q, qi + 1);
  }
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    const int i = tid + u * ABS_S_THREADS;
    if (i < BT * N) q_s[i] = qn[u];   // sequences past B: zero
  }
  for (int i = pair0; i < n_pairs; i += pair_stride) {
    const int b = i / (R / 2), p = i % (R / 2);
    float x0 = px0, x1 = px1, c = 1.f, s = 0.f;
    if (i != pair0) {
      const int64_t qi = ((int64_t)b * H + h) * qrow + N + 2 * p;
      x0 = Act<DT>::load(q, qi);
      x1 = Act<DT>::load(q, qi + 1);
    }
    if (positions != nullptr) rope_cs_split(cfg.rope_inv_freq, f_hi[p], f_lo[p], p, positions[b / pos_t] + b % pos_t, &c, &s);
    const int64_t ai = ((int64_t)b * H + h) * arow + C + 2 * p;
    if (positions != nullptr) {
      put(ai, x0 * c - x1 * s);
      put(ai + 1, x0 * s + x1 * c);
    } else {
      put(ai, x0);
      put(ai + 1, x1);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  const int cq = tid & 63, rq = tid >> 6;
  const int nq = N / 4;
  // packed float pairs: columns (4 cq, 4 cq + 1) and (4 cq + 2, 4 cq + 3)
  float2 acc[BT][2];
#pragma unroll
  for (int b = 0; b < BT; ++b) acc[b][0] = acc[b][1] = make_float2(0.f, 0.f);
#pragma unroll 4
  for (int n = rq * nq; n < (rq + 1) * nq; ++n) {
    float2 w0, w1;
    if (WDT == MLA_Q8_0) {
      const uint8_t* blk = w_s + n * RB + (cq >> 3) * 34;
      const uint16_t* c16 = reinterpret_cast<const uint16_t*>(blk + 2 + 4 * (cq & 7));
      const uint32_t codes = ((uint32_t)c16[0] | ((uint32_t)c16[1] << 16)) ^ 0x80808080u;
      const float d = __half2float(*reinterpret_cast<const __half*>(blk));
      const float2 bias = make_float2(-8388736.0f, -8388736.0f), dd = make_float2(d, d);
      w0 = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(codes, 0x4B000000u, 0x7650u)),
                                             __uint_as_float(__byte_perm(codes, 0x4B000000u, 0x7651u))),
                                 bias),
                      dd);
      w1 = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(codes, 0x4B000000u, 0x7652u)),
                                             __uint_as_float(__byte_perm(codes, 0x4B000000u, 0x7653u))),
                                 bias),
                      dd);
    } else {
      const uint2 u = *reinterpret_cast<const uint2*>(w_s + n * RB + 8 * cq);
      w0 = make_float2(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u));
      w1 = make_float2(__uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
    }
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const float qv = q_s[b * N + n];
      const float2 q2 = make_float2(qv, qv);
      acc[b][0] = __ffma2_rn(q2, w0, acc[b][0]);
      acc[b][1] = __ffma2_rn(q2, w1, acc[b][1]);
    }
  }
#pragma unroll
  for (int b = 0; b < BT; ++b)
    if (b < B)
      *reinterpret_cast<float4*>(red_s + (rq * ABS_S_BMAX + b) * ABS_S_COLS + 4 * cq) =
          make_float4(acc[b][0].x, acc[b][0].y, acc[b][1].x, acc[b][1].y);
  __syncthreads();
  for (int i = tid; i < B * ABS_S_COLS; i += ABS_S_THREADS) {
    const int b = i / ABS_S_COLS, col = i % ABS_S_COLS;
    const float* r = red_s + b * ABS_S_COLS + col;
    const float v = ((r[0] + r[ABS_S_BMAX * ABS_S_COLS]) + r[2 * ABS_S_BMAX * ABS_S_COLS]) + r[3 * ABS_S_BMAX * ABS_S_COLS];
    put(((int64_t)b * H + h) * arow + lh * ABS_S_COLS + col, v);
  }
}

static bool absorb_small_fits(const mla_config& cfg, int B) {
  return B >= 1 && B <= ABS_S_BMAX && (cfg.kv_b_dtype == MLA_BF16 || cfg.kv_b_dtype == MLA_Q8_0) &&
         cfg.kv_lora % ABS_S_COLS == 0 && cfg.qk_nope % 4 == 0 && cfg.qk_nope <= 128 && cfg.qk_rope <= 64;
}

template <int DT, int WDT, int BT>
static cudaError_t launch_absorb_small_bt(const mla_config& cfg, const void* q, const void* kv_b, const int32_t* positions,
                                       void* q_abs, void* q_res, int B, bool pdl, cudaStream_t st, int pos_t) {
  using T = typename Act<DT>::T;
  constexpr int RB = WDT == MLA_Q8_0 ? ABS_S_COLS / 32 * 34 : ABS_S_COLS * 2;
  const size_t smem = (size_t)cfg.qk_nope * RB + sizeof(float) * ((size_t)ABS_S_BMAX * cfg.qk_nope + 4 * ABS_S_BMAX * ABS_S_COLS);
  auto k = absorb_small_kernel<DT, WDT, BT>;
  cudaError_t e = ensure_smem((const void*)k, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(cfg.n_heads, cfg.kv_lora / ABS_S_COLS);
  return launch_kernel(pdl, k, grid, dim3(ABS_S_THREADS), smem, st, cfg, static_cast<const T*>(q),
                       static_cast<const uint8_t*>(kv_b), positions, static_cast<T*>(q_abs), static_cast<T*>(q_res), B,
                       pos_t);
}

template <int DT, int WDT>
static cudaError_t launch_absorb_small(const mla_config& cfg, const void* q, const void* kv_b, const int32_t* positions,
                                       void* q_abs, void* q_res, int B, bool pdl, cudaStream_t st, int pos_t) {
  if (B <= 1) return launch_absorb_small_bt<DT, WDT, 1>(cfg, q, kv_b, positions, q_abs, q_res, B, pdl, st, pos_t);
  if (B <= 2) return launch_absorb_small_bt<DT, WDT, 2>(cfg, q, kv_b, positions, q_abs, q_res, B, pdl, st, pos_t);
  if (B <= 4) return launch_absorb_small_bt<DT, WDT, 4>(cfg, q, kv_b, positions, q_abs, q_res, B, pdl, st, pos_t);
  return launch_absorb_small_bt<DT, WDT, 8>(cfg, q, kv_b, positions, q_abs, q_res, B, pdl, st, pos_t);
}

cudaError_t launch_absorb(const mla_config& cfg, const void* q, const void* kv_b,
                          const int32_t* positions, void* q_abs, void* q_res, int B, bool pdl, cudaStream_t st,
                          int pos_t) {
  if (pos_t < 1) return cudaErrorInvalidValue;
  if (absorb_small_fits(cfg, B)) {
    const bool q8 = cfg.kv_b_dtype == MLA_Q8_0;
    if (cfg.act_dtype == MLA_BF16)
      return q8 ? launch_absorb_small<MLA_BF16, MLA_Q8_0>(cfg, q, kv_b, positions, q_abs, q_res, B, pdl, st, pos_t)
                : launch_absorb_small<MLA_BF16, MLA_BF16>(cfg, q, kv_b, positions, q_abs, q_res, B, pdl, st, pos_t);
    return q8 ? launch_absorb_small<MLA_F32, MLA_Q8_0>(cfg, q, kv_b, positions, q_abs, nullptr, B, pdl, st, pos_t)
              : launch_absorb_small<MLA_F32, MLA_BF16>(cfg, q, kv_b, positions, q_abs, nullptr, B, pdl, st, pos_t);
  }
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
