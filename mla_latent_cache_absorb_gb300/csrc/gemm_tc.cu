// Tensor-core absorb and up-projection for bf16 kv_b with kv_lora 512 and nope / v_head 128.
//
// moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs, folded SDPA chain: q_prime (the nope
// rows of kv_b, per head) and out_per_head (the v rows, skipping nope); turbospark-runtime 0.3.0,
// src/families/deepseek2/attn.rs, absorb into fused [q' ; q_pe] rows and v-combine.
//
// Both stages are, per head, a GEMM whose cost is reading the head's 128 KB slice of kv_b once:
//   absorb:  q'^T[c, b]  = W_UK,h^T[c, n] . q_nope^T[n, b]   (M = 2 x 128 latent, N = batch, K = 128)
//   combine: out^T[j, b] = W_UV,h[j, c]   . vc^T[c, b]       (M = 128, N = batch, K = 512)
// The weight slice arrives by TMA in the 128-byte swizzle layout and is the A operand (MN-major
// for W_UK^T, K-major for W_UV); the batch is the N dimension, so one CTA per head (and batch
// chunk) issues a handful of tcgen05 MMAs with the fp32 accumulator in TMEM.
// The combine first merges the split partials into vc (float32) and feeds it as two bf16 terms,
// hi and lo, stacked into one N = 64 operand for its 32 sequences (the two accumulator halves
// are added in the epilogue), so the up-projection keeps close to float32 accuracy on the bf16
// tensor path. The absorb pads its batch chunk to a multiple of 16.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <math_constants.h>

namespace mla {

namespace {

constexpr int G_THREADS = 128;
// Main-loop waits use the launch's wait_ns; drains of a copy or MMAs already issued always get
// the full kWaitDrainNs, so nothing is in flight when a CTA leaves or frees tensor memory.
constexpr uint64_t G_DRAIN = kWaitDrainNs;
constexpr int ABS_TC_BCHUNK = 64;
constexpr int CMB_TC_BCHUNK = 32;
constexpr int CMB_TC_THREADS = 512;   // 4 merge items per thread, loads of 2 items x 4 slots in flight
constexpr int ABS_TC_SMEM = 4 * 16384 + 2 * 8192 + 1024;
constexpr int CMB_TC_WSMEM = 8 * 16384 + 8 * 8192;   // W_UV + vc hi/lo

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint16_t bf16_bits(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&h);
}

struct AbsorbTcArgs {
  const uint16_t* q;        // [B][H][N+R] bf16
  uint16_t* q_abs;          // [B][H][C+R] bf16
  uint16_t* q_res;          // [B][H][C+R] bf16 rounding residual of q_abs
  const int32_t* positions;
  const double* inv_freq;
  WsHeader* hdr;
  uint64_t wait_ns;
  int B, H, N, R, V, C;
  int pos_t;                // query tokens per sequence: row b's position is positions[b / pos_t] + b % pos_t
};

// grid (H, 2 latent halves, batch chunks of 64); 128 threads
__global__ void __launch_bounds__(G_THREADS, 1)
absorb_tc_kernel(const __grid_constant__ CUtensorMap w_map, AbsorbTcArgs a) {
  extern __shared__ uint8_t dyn_raw[];
  __shared__ uint64_t bar_w, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int failed;
  uint8_t* dyn = align1024(dyn_raw);
  uint8_t* ws = dyn;                 // 4 blocks [128 n rows x 64 latent] (MN-major A)
  uint8_t* qs = dyn + 4 * 16384;     // 2 blocks [64 b rows x 64 n] (K-major B)
  __shared__ float rope_hi[32], rope_lo[32];   // the RoPE frequencies as float pairs (rope <= 64)
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, lh = blockIdx.y, b0 = blockIdx.z * ABS_TC_BCHUNK;
  const int nb = min(ABS_TC_BCHUNK, a.B - b0);
  const int NB = (nb + 15) & ~15;
  const int qrow = a.N + a.R, arow = a.C + a.R;

  if (tid == 0) {
    failed = 0;
    tc::mbar_init(&bar_w, 1);
    tc::mbar_init(&bar_mma, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 128);
    tc::tmem_relinquish();
  }
  const bool rope_f32 = a.positions != nullptr && a.R <= 64;
  if (rope_f32 && tid < a.R / 2) {
    const double inv = a.inv_freq[tid];
    const float hi = __double2float_rn(inv);
    rope_hi[tid] = hi;
    rope_lo[tid] = __double2float_rn(inv - static_cast<double>(hi));
  }
  tc::tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    tc::mbar_arrive_expect_tx(&bar_w, 4 * 16384);
    for (int cb = 0; cb < 4; ++cb)
      tc::tma_load_2d(ws + cb * 16384, &w_map, 256 * lh + 64 * cb, h * (a.N + a.V), &bar_w);
  }
  // q may be written by a kernel two or more launches back (the front end): every read of it
  // comes after the wait for the previous kernel, which completes only after that one's own wait
  pdl_wait();
  // q_nope rows of this batch chunk, 128-byte swizzled, zero rows past the batch (all of a
  // thread's loads are issued before its first store)
  {
    constexpr int QI = ABS_TC_BCHUNK * 16 / G_THREADS;
    uint4 v[QI];
#pragma unroll
    for (int m = 0; m < QI; ++m) {
      const int i = tid + m * G_THREADS;
      const int r = i >> 4, ch = i & 15, kb = ch >> 3, c8 = ch & 7;
      v[m] = make_uint4(0, 0, 0, 0);
      if (r < nb) v[m] = *reinterpret_cast<const uint4*>(a.q + ((size_t)(b0 + r) * a.H + h) * qrow + kb * 64 + c8 * 8);
    }
#pragma unroll
    for (int m = 0; m < QI; ++m) {
      const int i = tid + m * G_THREADS;
      const int r = i >> 4, ch = i & 15, kb = ch >> 3, c8 = ch & 7;
      *reinterpret_cast<uint4*>(qs + kb * 8192 + tc::sw128_offset(r, c8)) = v[m];
    }
  }
  tc::fence_proxy_async_smem();
  __syncwarp();
  __syncthreads();
  if (tid == 0) {
    if (!tc::mbar_wait(&bar_w, 0, a.wait_ns)) {
      failed = 1;
      set_error(a.hdr, MLA_ERR_TIMEOUT, b0);
      tc::mbar_wait(&bar_w, 0, G_DRAIN);   // the weight copy must land before the CTA leaves
    } else {
      tc::tc_fence_after();
      const uint32_t idesc = tc::idesc_bf16_f32(128, NB, 1, 0);
      const uint32_t w0 = tc::smem_u32(ws), q0 = tc::smem_u32(qs);
      for (int mc = 0; mc < 2; ++mc)
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = tc::sdesc_sw128(w0 + (2 * mc) * 16384 + kk * 2048, 16384, 1024);
          const uint64_t bd = tc::sdesc_sw128(q0 + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024);
          tc::mma_f16_ss(tmem + mc * 64, ad, bd, idesc, kk > 0);
        }
    }
    tc::mma_commit(&bar_mma);   // arrives once every MMA issued above has completed
  }
  // rotated q_pe into the row's tail, while the MMAs run: the batch chunk's pairs are shared
  // by the CTAs of the two latent halves; a thread loads all of its pairs (and positions)
  // before using any
  {
    const int hr = a.R / 2;
    const int npairs = nb * hr;
    const int pb = lh == 0 ? 0 : npairs / 2, pe = lh == 0 ? npairs / 2 : npairs;
    constexpr int RI = (ABS_TC_BCHUNK * 32 / 2 + G_THREADS - 1) / G_THREADS;   // rope <= 64
    uint32_t xv[RI];
    int pv[RI];
#pragma unroll
    for (int m = 0; m < RI; ++m) {
      const int i = pb + tid + m * G_THREADS;
      xv[m] = 0;
      pv[m] = 0;
      if (i < pe) {
        const int bb = i / hr, p = i - bb * hr;
        xv[m] = *reinterpret_cast<const uint32_t*>(a.q + ((size_t)(b0 + bb) * a.H + h) * qrow + a.N + 2 * p);
        if (a.positions != nullptr) pv[m] = a.positions[(b0 + bb) / a.pos_t] + (b0 + bb) % a.pos_t;
      }
    }
    auto rotate = [&](int i, uint32_t x, int pos) {
      const int bb = i / hr, p = i - bb * hr;
      const size_t ai = ((size_t)(b0 + bb) * a.H + h) * arow + a.C + 2 * p;
      const float x0 = __uint_as_float(x << 16), x1 = __uint_as_float(x & 0xFFFF0000u);
      float y0 = x0, y1 = x1;
      if (a.positions != nullptr) {
        float c, sn;
        if (rope_f32 && pos >= 0 && pos < ROPE_F32_MAX_POS && rope_hi[p] > 0.f && rope_hi[p] <= 1.f)
          rope_cs_f32(rope_hi[p], rope_lo[p], pos, &c, &sn);
        else
          rope_cs(a.inv_freq, p, pos, &c, &sn);
        y0 = x0 * c - x1 * sn;
        y1 = x0 * sn + x1 * c;
      }
      const uint16_t h0 = bf16_bits(y0), h1 = bf16_bits(y1);
      *reinterpret_cast<uint32_t*>(a.q_abs + ai) = (uint32_t)h0 | ((uint32_t)h1 << 16);
      *reinterpret_cast<uint32_t*>(a.q_res + ai) =
          (uint32_t)bf16_bits(y0 - bf16_bits_to_f32(h0)) | ((uint32_t)bf16_bits(y1 - bf16_bits_to_f32(h1)) << 16);
    };
#pragma unroll
    for (int m = 0; m < RI; ++m) {
      const int i = pb + tid + m * G_THREADS;
      if (i < pe) rotate(i, xv[m], pv[m]);
    }
    // rope widths above 64 leave pairs for a plain loop
    for (int i = pb + tid + RI * G_THREADS; i < pe; i += G_THREADS) {
      const int bb = i / hr, p = i - bb * hr;
      rotate(i, *reinterpret_cast<const uint32_t*>(a.q + ((size_t)(b0 + bb) * a.H + h) * qrow + a.N + 2 * p),
             a.positions != nullptr ? a.positions[(b0 + bb) / a.pos_t] + (b0 + bb) % a.pos_t : 0);
    }
  }
  __syncwarp();   // lanes 1-31 of warp 0 wait for lane 0
  // warp-uniform: the TMEM loads below are warp-collective
  bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&bar_mma, 0, a.wait_ns) &&
                                       !*reinterpret_cast<volatile int*>(&failed));
  if (!ok) {
    if (lane == 0 && atomicExch(&failed, 1) == 0) set_error(a.hdr, MLA_ERR_TIMEOUT, b0);
    // whatever happened, every MMA issued has to complete before tensor memory is freed
    tc::mbar_wait(&bar_mma, 0, G_DRAIN);
  }
  tc::tc_fence_after();
  __syncwarp();
  __syncthreads();
  ok = !*reinterpret_cast<volatile int*>(&failed);
  if (!ok) {
    // this CTA's fused query entries (its sequences, head h, latent half lh) become NaN, so
    // their scores, and the sequences' outputs, do too
    for (int i = tid; i < nb * 256; i += G_THREADS) {
      const size_t ai = ((size_t)(b0 + i / 256) * a.H + h) * arow + 256 * lh + (i % 256);
      a.q_abs[ai] = 0x7FC0;
      a.q_res[ai] = 0;
    }
  } else {
    // Lane = latent column, TMEM column = sequence: each warp transposes its 32 x 32 block
    // through shared memory (the B operand's space, free once the MMAs are done) so that every
    // lane then writes 16-byte pieces of 8 consecutive latent columns of one sequence.
    uint16_t* hi_s = reinterpret_cast<uint16_t*>(qs + warp * 4096);   // [32 sequences][32 columns]
    uint16_t* lo_s = hi_s + 32 * 32;
    for (int mc = 0; mc < 2; ++mc) {
      const int cw = 256 * lh + 128 * mc + 32 * warp;   // this warp's first latent column
      for (int col0 = 0; col0 < NB; col0 += 32) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + mc * 64 + col0, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float v = __uint_as_float(r[j]);
          const uint16_t hi = bf16_bits(v);
          hi_s[j * 32 + lane] = hi;
          lo_s[j * 32 + lane] = bf16_bits(v - bf16_bits_to_f32(hi));
        }
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int chunk = lane + 32 * i, bj = chunk >> 2, g = chunk & 3;
          const int b = col0 + bj;
          if (b < nb) {
            const size_t ai = ((size_t)(b0 + b) * a.H + h) * arow + cw + 8 * g;
            *reinterpret_cast<uint4*>(a.q_abs + ai) = *reinterpret_cast<const uint4*>(hi_s + bj * 32 + 8 * g);
            *reinterpret_cast<uint4*>(a.q_res + ai) = *reinterpret_cast<const uint4*>(lo_s + bj * 32 + 8 * g);
          }
        }
        __syncwarp();
      }
    }
  }
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 128);
  }
}

struct CombineTcArgs {
  const int32_t* meta;
  const float* part_o;
  const float* part_lse;
  float* out;
  float* lse;
  const uint16_t* q_res;    // bf16 query residual [B][H][C+R] (LSE correction) or nullptr
  float scale;
  WsHeader* hdr;
  uint64_t wait_ns;
  int H, C, N, V, R, B, hpg, n_slots, max_slots;
  int kvb_heads;            // heads of kv_b: head h up-projects through W_UV of head h % kvb_heads
};

// grid (H, batch chunks of 32); 512 threads
__global__ void __launch_bounds__(CMB_TC_THREADS, 1)
combine_tc_kernel(const __grid_constant__ CUtensorMap w_map, CombineTcArgs a) {
  extern __shared__ uint8_t dyn_raw[];
  __shared__ uint64_t bar_w, bar_mma;
  __shared__ uint32_t tmem_base;
  __shared__ int failed;
  __shared__ float lse_s[CMB_TC_BCHUNK];
  __shared__ int first_s[CMB_TC_BCHUNK], cnt_s[CMB_TC_BCHUNK];
  uint8_t* dyn = align1024(dyn_raw);
  uint8_t* wu = dyn;                           // 8 blocks [128 j rows x 64 c] (K-major A)
  // 8 blocks [64 rows x 64 c] (K-major B): rows 0-31 the bf16 high parts of vc for the 32
  // sequences, rows 32-63 their low parts, so one N=64 MMA per k-step takes both
  uint8_t* vb = dyn + 8 * 16384;
  float* dres = reinterpret_cast<float*>(vb + 8 * 8192);   // [32][64] partial vc . res
  float* wt_s = dres + CMB_TC_BCHUNK * 64;                  // [32][max_slots]
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x, b0 = blockIdx.y * CMB_TC_BCHUNK;
  const int nb = min(CMB_TC_BCHUNK, a.B - b0);
  const int pg = h / a.hpg, hh = h % a.hpg;
  auto lse_at = [&](int slot) { return ((int64_t)pg * a.n_slots + slot) * a.hpg + hh; };

  if (tid == 0) {
    failed = 0;
    tc::mbar_init(&bar_w, 1);
    tc::mbar_init(&bar_mma, 1);
    tc::fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 64);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    tc::mbar_arrive_expect_tx(&bar_w, 8 * 16384);
    for (int kb = 0; kb < 8; ++kb)
      tc::tma_load_2d(wu + kb * 16384, &w_map, 64 * kb, (h % a.kvb_heads) * (a.N + a.V) + a.N, &bar_w);
  }
  pdl_wait();   // the partials and meta come from the attention kernel
  // split weights: 16 lanes per sequence, every sequence of the chunk at once, the first
  // slots' LSEs kept in registers so the partials' LSEs are read from memory once
  static_assert(CMB_TC_THREADS / 16 == CMB_TC_BCHUNK, "one 16-lane group per sequence");
  {
    constexpr int KEEP = 4;
    const int bb = tid >> 4, l16 = tid & 15;
    int first = 0, ns = 0;
    if (bb < nb) {
      first = a.meta[2 * (b0 + bb)];
      ns = min(a.meta[2 * (b0 + bb) + 1], a.max_slots);
    }
    float v[KEEP];
    float mx = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < KEEP; ++k) {
      const int s = l16 + 16 * k;
      v[k] = (s < ns) ? a.part_lse[lse_at(first + s)] : -CUDART_INF_F;
      mx = fmaxf(mx, v[k]);
    }
    for (int s = l16 + 16 * KEEP; s < ns; s += 16) mx = fmaxf(mx, a.part_lse[lse_at(first + s)]);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < KEEP; ++k)
      if (l16 + 16 * k < ns) tot += expf(v[k] - mx);
    for (int s = l16 + 16 * KEEP; s < ns; s += 16) tot += expf(a.part_lse[lse_at(first + s)] - mx);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
    const float l = (ns > 0) ? mx + logf(tot) : CUDART_NAN_F;
#pragma unroll
    for (int k = 0; k < KEEP; ++k)
      if (l16 + 16 * k < ns) wt_s[bb * a.max_slots + l16 + 16 * k] = expf(v[k] - l);
    for (int s = l16 + 16 * KEEP; s < ns; s += 16)
      wt_s[bb * a.max_slots + s] = expf(a.part_lse[lse_at(first + s)] - l);
    if (l16 == 0) {
      lse_s[bb] = l;
      first_s[bb] = first;
      cnt_s[bb] = ns;
    }
  }
  __syncwarp();
  __syncthreads();
  // vc = sum_s w_s O_s as bf16 hi + lo, 8 latent columns per item, 128-byte swizzled. Item
  // (bb, ch) = sequence bb, latent columns 8*ch..8*ch+7; a thread takes items of one column
  // group and four sequences, two at a time, with the loads of up to four slots of both items
  // (and their query residuals) issued before any is used.
  constexpr int MU = 2, SU = 4;
  const int ch = tid & 63, kb = ch >> 3, c8 = ch & 7;
  for (int m0 = 0; m0 < CMB_TC_BCHUNK / (CMB_TC_THREADS / 64); m0 += MU) {
    int bbv[MU], nsv[MU], fv[MU];
    float acc[MU][8];
    uint4 resv[MU];
#pragma unroll
    for (int u = 0; u < MU; ++u) {
      bbv[u] = (tid >> 6) + (CMB_TC_THREADS / 64) * (m0 + u);
      const bool live = bbv[u] < nb && !isnan(lse_s[bbv[u]]);
      nsv[u] = live ? cnt_s[bbv[u]] : 0;
      fv[u] = first_s[bbv[u]];
      resv[u] = make_uint4(0, 0, 0, 0);
      if (a.q_res != nullptr && bbv[u] < nb)
        resv[u] = *reinterpret_cast<const uint4*>(a.q_res + ((size_t)(b0 + bbv[u]) * a.H + h) * (a.C + a.R) + ch * 8);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[u][e] = 0.f;
    }
    int smax = 0;
#pragma unroll
    for (int u = 0; u < MU; ++u) smax = max(smax, nsv[u]);
    for (int s0 = 0; s0 < smax; s0 += SU) {
      float4 x[MU][SU][2];
#pragma unroll
      for (int u = 0; u < MU; ++u)
#pragma unroll
        for (int v = 0; v < SU; ++v) {
          x[u][v][0] = x[u][v][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (s0 + v < nsv[u]) {
            const float4* src = reinterpret_cast<const float4*>(a.part_o + lse_at(fv[u] + s0 + v) * a.C + ch * 8);
            x[u][v][0] = src[0];
            x[u][v][1] = src[1];
          }
        }
#pragma unroll
      for (int u = 0; u < MU; ++u)
#pragma unroll
        for (int v = 0; v < SU; ++v) {
          const float w = (s0 + v < nsv[u]) ? wt_s[bbv[u] * a.max_slots + s0 + v] : 0.f;
          if (w != 0.f) {   // empty slots carry weight 0 and unwritten data: skip, never 0 * x
            acc[u][0] = fmaf(w, x[u][v][0].x, acc[u][0]); acc[u][1] = fmaf(w, x[u][v][0].y, acc[u][1]);
            acc[u][2] = fmaf(w, x[u][v][0].z, acc[u][2]); acc[u][3] = fmaf(w, x[u][v][0].w, acc[u][3]);
            acc[u][4] = fmaf(w, x[u][v][1].x, acc[u][4]); acc[u][5] = fmaf(w, x[u][v][1].y, acc[u][5]);
            acc[u][6] = fmaf(w, x[u][v][1].z, acc[u][6]); acc[u][7] = fmaf(w, x[u][v][1].w, acc[u][7]);
          }
        }
    }
#pragma unroll
    for (int u = 0; u < MU; ++u) {
      const int bb = bbv[u];
      if (bb < nb && isnan(lse_s[bb])) {
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[u][e] = CUDART_NAN_F;
      }
      if (a.q_res != nullptr) {
        const uint32_t w[4] = {resv[u].x, resv[u].y, resv[u].z, resv[u].w};
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          d += acc[u][2 * e] * __uint_as_float(w[e] << 16) + acc[u][2 * e + 1] * __uint_as_float(w[e] & 0xFFFF0000u);
        dres[bb * 64 + ch] = (bb < nb) ? d : 0.f;
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint16_t h0 = bf16_bits(acc[u][2 * e]), h1 = bf16_bits(acc[u][2 * e + 1]);
        const uint16_t l0 = bf16_bits(acc[u][2 * e] - bf16_bits_to_f32(h0));
        const uint16_t l1 = bf16_bits(acc[u][2 * e + 1] - bf16_bits_to_f32(h1));
        hi[e] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        lo[e] = (uint32_t)l0 | ((uint32_t)l1 << 16);
      }
      *reinterpret_cast<uint4*>(vb + kb * 8192 + tc::sw128_offset(bb, c8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(vb + kb * 8192 + tc::sw128_offset(bb + 32, c8)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
  tc::fence_proxy_async_smem();
  __syncwarp();
  __syncthreads();
  if (a.q_res != nullptr) {
    // first-order LSE correction for the bf16 latent queries the scores used:
    // lse += scale * vc . res, summed in a fixed order (one warp per sequence)
    for (int bb = warp; bb < nb; bb += CMB_TC_THREADS / 32) {
      float d = dres[bb * 64 + lane] + dres[bb * 64 + 32 + lane];
      d = warp_sum(d);
      if (lane == 0) lse_s[bb] += a.scale * d;
    }
    __syncwarp();
    __syncthreads();
  }
  if (tid == 0) {
    if (!tc::mbar_wait(&bar_w, 0, a.wait_ns)) {
      failed = 1;
      set_error(a.hdr, MLA_ERR_TIMEOUT, b0);
      tc::mbar_wait(&bar_w, 0, G_DRAIN);   // the weight copy must land before the CTA leaves
    } else {
      tc::tc_fence_after();
      // D[j, 0..31] = W . vc_hi, D[j, 32..63] = W . vc_lo; the epilogue adds the halves
      const uint32_t idesc = tc::idesc_bf16_f32(128, 64, 0, 0);
      const uint32_t w0 = tc::smem_u32(wu), v0 = tc::smem_u32(vb);
      for (int kb = 0; kb < 8; ++kb)
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_f16_ss(tmem, tc::sdesc_sw128(w0 + kb * 16384 + kk * 32, 16, 1024),
                         tc::sdesc_sw128(v0 + kb * 8192 + kk * 32, 16, 1024), idesc, (kb | kk) != 0);
    }
    tc::mma_commit(&bar_mma);
  }
  __syncwarp();
  // warp-uniform: the TMEM loads below are warp-collective; warps 0-3 read the 128 TMEM lanes
  if (warp < 4 && !__all_sync(0xffffffffu, tc::mbar_wait(&bar_mma, 0, a.wait_ns) &&
                                               !*reinterpret_cast<volatile int*>(&failed))) {
    if (lane == 0 && atomicExch(&failed, 1) == 0) set_error(a.hdr, MLA_ERR_TIMEOUT, b0);
    // every MMA issued has to complete before tensor memory is freed
    tc::mbar_wait(&bar_mma, 0, G_DRAIN);
  }
  tc::tc_fence_after();
  __syncwarp();
  __syncthreads();
  const bool ok = !*reinterpret_cast<volatile int*>(&failed);
  if (!ok) {
    // the chunk's outputs for head h become NaN
    for (int i = tid; i < nb * a.V; i += CMB_TC_THREADS)
      a.out[((size_t)(b0 + i / a.V) * a.H + h) * a.V + (i % a.V)] = CUDART_NAN_F;
    __syncthreads();
    if (tid < nb) lse_s[tid] = CUDART_NAN_F;
  } else if (warp < 4) {
    uint32_t r[32], rl[32];
    tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), r);
    tc::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 32, rl);
    tc::tmem_wait_ld();
    const int j = 32 * warp + lane;
#pragma unroll
    for (int b = 0; b < 32; ++b)
      if (b < nb) a.out[((size_t)(b0 + b) * a.H + h) * a.V + j] = __uint_as_float(r[b]) + __uint_as_float(rl[b]);
  }
  if (a.lse != nullptr)
    for (int bb = tid; bb < nb; bb += CMB_TC_THREADS) a.lse[(size_t)(b0 + bb) * a.H + h] = lse_s[bb];
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 64);
  }
}

}  // namespace

// The tensor-core absorb / combine take bf16 kv_b with kv_lora 512 and 128-row W_UK / W_UV
// blocks, and batches large enough to fill an MMA's N dimension.
bool absorb_tc_supported(const mla_config& cfg, int B) {
  return cfg.act_dtype == MLA_BF16 && cfg.kv_b_dtype == MLA_BF16 && cfg.kv_lora == 512 && cfg.qk_nope == 128 &&
         B >= 8 && (int64_t)cfg.n_heads * (cfg.qk_nope + cfg.v_head) < (int64_t(1) << 31);
}

bool combine_tc_supported(const mla_config& cfg, int B) {
  return cfg.kv_b_dtype == MLA_BF16 && cfg.kv_lora == 512 && cfg.v_head == 128 && B >= 8 &&
         (int64_t)cfg.n_heads * (cfg.qk_nope + cfg.v_head) < (int64_t(1) << 31);
}

cudaError_t launch_absorb_tc(const mla_config& cfg, const void* q, const void* kv_b, const int32_t* positions,
                             void* q_abs, void* q_res, int B, WsHeader* hdr, bool pdl, cudaStream_t st,
                             int pos_t) {
  if (pos_t < 1) return cudaErrorInvalidValue;
  CUtensorMap w_map;
  if (!make_map_2d_bf16(&w_map, kv_b, 512, (uint64_t)cfg.n_heads * (cfg.qk_nope + cfg.v_head), 64, 128))
    return cudaErrorInvalidValue;
  AbsorbTcArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.q_abs = static_cast<uint16_t*>(q_abs);
  a.q_res = static_cast<uint16_t*>(q_res);
  a.positions = positions;
  a.inv_freq = cfg.rope_inv_freq;
  a.hdr = hdr;
  a.wait_ns = wait_limit_ns();
  a.B = B; a.H = cfg.n_heads; a.N = cfg.qk_nope; a.R = cfg.qk_rope; a.V = cfg.v_head; a.C = cfg.kv_lora;
  a.pos_t = pos_t;
  cudaError_t e = ensure_smem((const void*)absorb_tc_kernel, ABS_TC_SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(cfg.n_heads, 2, (B + ABS_TC_BCHUNK - 1) / ABS_TC_BCHUNK);
  return launch_kernel(pdl, absorb_tc_kernel, grid, dim3(G_THREADS), ABS_TC_SMEM, st, w_map, a);
}

cudaError_t launch_combine_tc(const mla_config& cfg, const DecodePlan& plan, const void* kv_b,
                              const int32_t* meta, const float* part_o, const float* part_lse, const void* q_res,
                              float* out, float* lse, int B, WsHeader* hdr, cudaStream_t st) {
  // cfg.n_heads = plan.tokens query tokens x plan.kvb_heads heads of kv_b
  if (plan.kvb_heads < 1 || plan.kvb_heads * plan.tokens != cfg.n_heads) return cudaErrorInvalidValue;
  CUtensorMap w_map;
  if (!make_map_2d_bf16(&w_map, kv_b, 512, (uint64_t)plan.kvb_heads * (cfg.qk_nope + cfg.v_head), 64, 128))
    return cudaErrorInvalidValue;
  CombineTcArgs a;
  a.meta = meta; a.part_o = part_o; a.part_lse = part_lse; a.out = out; a.lse = lse; a.hdr = hdr;
  a.q_res = static_cast<const uint16_t*>(q_res);
  a.scale = cfg.softmax_scale;
  a.wait_ns = wait_limit_ns();
  a.H = cfg.n_heads; a.C = cfg.kv_lora; a.N = cfg.qk_nope; a.V = cfg.v_head; a.R = cfg.qk_rope; a.B = B;
  a.hpg = plan.part_hpg; a.n_slots = plan.n_slots;
  a.kvb_heads = plan.kvb_heads;
  a.max_slots = plan.path != PATH_SIMT ? plan.ctas_per_group : plan.splits;
  const int smem = CMB_TC_WSMEM + 1024 + CMB_TC_BCHUNK * (64 + a.max_slots) * (int)sizeof(float);
  cudaError_t e = ensure_smem((const void*)combine_tc_kernel, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(cfg.n_heads, (B + CMB_TC_BCHUNK - 1) / CMB_TC_BCHUNK);
  return launch_pdl(combine_tc_kernel, grid, dim3(CMB_TC_THREADS), (size_t)smem, st, w_map, a);
}

}  // namespace mla
