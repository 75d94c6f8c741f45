// Combine + up-project: merge the splits of each (sequence, head) by log-sum-exp, then
// out[b,h,:] = W_UV,h * vc[b,h,:].
//
// moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs, out_per_head (v_combine through the
// v rows of kv_b, skipping the nope rows). turbospark-runtime 0.3.0,
// src/families/deepseek2/attn.rs, encode_mla_v_combine (Q8_0 W_UV). The split + COMBINE pass
// structure follows turbospark-runtime 0.3.0, src/families/gptoss/attn.rs.
//
// Grid (head, slice of V, block of 8 sequences); the V-slices per head are as few as still give
// about one CTA per SM, since every slice merges the partials again. Each CTA merges the splits
// of its sequences for its head into float32 latent vectors (every thread keeps several partial
// loads in flight; with few sequences the slots are shared out over several threads and summed
// in a fixed order), then, 32 outputs at a time, stages those rows of W_UV (dequantised) in
// shared memory and forms the dot products one warp per pair of outputs with the lanes across
// the latent.
#include "common.cuh"

#include <math_constants.h>

namespace mla {

constexpr int CMB_THREADS = 512;
constexpr int CMB_VJ = 32;      // V outputs per CTA
constexpr int CMB_BC = 8;       // sequences per CTA
constexpr int CMB_RES_MAX = 512; // latent widths whose query residual is staged in shared memory
constexpr int CMB_U = 8;        // partial loads in flight per thread

struct CombineArgs {
  const void* kv_b;
  const int32_t* meta;      // [B][2]: first partial slot, slot count (0 = invalid sequence)
  const float* part_o;      // [groups][n_slots][hpg][C]
  const float* part_lse;    // [groups][n_slots][hpg]
  float* out;
  float* lse;
  const uint16_t* q_res;    // bf16 query residual [B][H][C+R] or nullptr (no LSE correction)
  float scale;
  int kv_b_dtype;
  int H, C, N, V, R, B;
  int hpg, n_slots, max_slots;
  int vper;                 // outputs per CTA (a multiple of CMB_VJ): the merge is done once per CTA
  int kvb_heads;            // heads of kv_b: head h up-projects through W_UV of head h % kvb_heads
};

// out[b0 + bb, h, j0 + j] = W_UV row j . vc[bb] for bb < nb <= NBT: one warp per pair of outputs
// (CMB_VJ outputs per pass), lane `lane` taking the latent float4s lane, lane + 32, ... of both
// rows (rows of w_s and vc_s are zero past C up to `stride`), so each vc element read from
// shared memory serves two outputs; fixed-order warp reductions; 2 x NBT accumulators per lane.
static_assert(CMB_THREADS / 32 * 2 == CMB_VJ, "one warp per pair of outputs of a chunk");
template <int NBT>
__device__ __forceinline__ void combine_outputs(const CombineArgs& a, const float* w_s, const float* vc_s, int stride,
                                                int nb, int nj, int b0, int h, int j0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ja = 2 * warp, jb = ja + 1;
  float acc[2][NBT];
#pragma unroll
  for (int bb = 0; bb < NBT; ++bb) acc[0][bb] = acc[1][bb] = 0.f;
  if (ja < nj) {
    const float4* wa = reinterpret_cast<const float4*>(w_s + ja * stride);
    // a row past nj (odd nj) holds stale data: its sums are computed and dropped
    const float4* wb = reinterpret_cast<const float4*>(w_s + jb * stride);
    const float4* vc4 = reinterpret_cast<const float4*>(vc_s);
    const int s4 = stride / 4;
#pragma unroll 1
    for (int c4 = lane; c4 < s4; c4 += 32) {
      const float4 x = wa[c4], y = wb[c4];
#pragma unroll
      for (int bb = 0; bb < NBT; ++bb) {
        if (bb < nb) {
          const float4 v = vc4[bb * s4 + c4];
          acc[0][bb] = fmaf(x.x, v.x, fmaf(x.y, v.y, fmaf(x.z, v.z, fmaf(x.w, v.w, acc[0][bb]))));
          acc[1][bb] = fmaf(y.x, v.x, fmaf(y.y, v.y, fmaf(y.z, v.z, fmaf(y.w, v.w, acc[1][bb]))));
        }
      }
    }
  }
#pragma unroll
  for (int bb = 0; bb < NBT; ++bb) {
    const float va = warp_sum(acc[0][bb]), vb = warp_sum(acc[1][bb]);
    if (lane == 0 && bb < nb) {
      const int64_t o = ((int64_t)(b0 + bb) * a.H + h) * a.V + j0;
      if (ja < nj) a.out[o + ja] = va;
      if (jb < nj) a.out[o + jb] = vb;
    }
  }
}

__global__ void __launch_bounds__(CMB_THREADS, 2) combine_kernel(CombineArgs a) {
  extern __shared__ float sm[];
  pdl_trigger();
  const int h = blockIdx.x;
  const int jbeg = blockIdx.y * a.vper;
  const int jend = min(a.V, jbeg + a.vper);
  const int b0 = blockIdx.z * CMB_BC;
  const int nb = min(CMB_BC, a.B - b0);
  const int C = a.C;
  const int C4 = (C + 3) / 4;               // latent in groups of 4
  float* w_s = sm;                          // [CMB_VJ][4*C4]
  float* vc_s = w_s + CMB_VJ * 4 * C4;      // [CMB_BC][4*C4]
  float4* red_s = reinterpret_cast<float4*>(vc_s + CMB_BC * 4 * C4);   // [CMB_THREADS]
  float* wt_s = reinterpret_cast<float*>(red_s + CMB_THREADS);         // [CMB_BC][max_slots]
  float* lse_s = wt_s + CMB_BC * a.max_slots;                          // [CMB_BC]
  int* first_s = reinterpret_cast<int*>(lse_s + CMB_BC);               // [CMB_BC]
  int* cnt_s = first_s + CMB_BC;                                        // [CMB_BC]
  uint16_t* res_s = reinterpret_cast<uint16_t*>(cnt_s + CMB_BC);        // [CMB_BC][C] when C <= 512
  const int pg = h / a.hpg, hh = h % a.hpg;
  auto lse_at = [&](int slot) { return ((int64_t)pg * a.n_slots + slot) * a.hpg + hh; };

  // W_UV rows of the first 32-output chunk (the rest follow after the merge)
  const int64_t wrow0 = (int64_t)(h % a.kvb_heads) * (a.N + a.V) + a.N;
  const int64_t kv_rows = (int64_t)a.kvb_heads * (a.N + a.V);
  stage_kv_b_rows(w_s, 4 * C4, a.kv_b, a.kv_b_dtype, wrow0 + jbeg, min(CMB_VJ, jend - jbeg), 0, C, C, CMB_THREADS,
                  kv_rows);
  pdl_wait();   // the partials and meta come from the attention kernel
  // Loads that do not depend on one another go out together: each warp's sequence metadata
  // and the query residual (for the first-order LSE correction below); the partial LSEs follow
  // one memory round trip later.
  static_assert(CMB_BC <= CMB_THREADS / 32, "one warp per sequence of the block");
  constexpr int RES_PER = CMB_BC * CMB_RES_MAX / CMB_THREADS;   // residual elements per thread
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int first = 0, ns = 0;
  if (warp < nb) {
    first = a.meta[2 * (b0 + warp)];
    ns = min(a.meta[2 * (b0 + warp) + 1], a.max_slots);
  }
  const bool res_pre = a.q_res != nullptr && C <= CMB_RES_MAX;
  uint16_t rv[RES_PER];
  if (res_pre) {
#pragma unroll
    for (int u = 0; u < RES_PER; ++u) {
      const int i = threadIdx.x + u * CMB_THREADS;
      rv[u] = (i < nb * C) ? a.q_res[((int64_t)(b0 + i / C) * a.H + h) * (C + a.R) + i % C] : 0;
    }
  }
  // split weights exp(lse_s - lse): one warp per sequence, each lane's first slot kept in a register
  if (warp < nb) {
    const float v0 = (lane < ns) ? a.part_lse[lse_at(first + lane)] : -CUDART_INF_F;
    float mx = v0;
    for (int s = lane + 32; s < ns; s += 32) mx = fmaxf(mx, a.part_lse[lse_at(first + s)]);
    mx = warp_max(mx);
    float tot = (lane < ns) ? expf(v0 - mx) : 0.f;
    for (int s = lane + 32; s < ns; s += 32) tot += expf(a.part_lse[lse_at(first + s)] - mx);
    tot = warp_sum(tot);
    const float l = (ns > 0) ? mx + logf(tot) : CUDART_NAN_F;
    if (lane < ns) wt_s[warp * a.max_slots + lane] = expf(v0 - l);
    for (int s = lane + 32; s < ns; s += 32) wt_s[warp * a.max_slots + s] = expf(a.part_lse[lse_at(first + s)] - l);
    if (lane == 0) {
      lse_s[warp] = l;
      first_s[warp] = first;
      cnt_s[warp] = ns;
    }
  }
  if (res_pre) {
#pragma unroll
    for (int u = 0; u < RES_PER; ++u) {
      const int i = threadIdx.x + u * CMB_THREADS;
      if (i < nb * C) res_s[i] = rv[u];
    }
  }
  __syncthreads();

  // vc[bb][4g..4g+3] = sum_s w_s * O_s; item = (bb, g); `split` threads share an item's slots
  const int nitems = nb * C4;
  int split = 1;
  while (split < 8 && 2 * split * nitems <= CMB_THREADS) split *= 2;
  const bool vec = (C % 4) == 0;
  for (int it = threadIdx.x; it < nitems * split; it += CMB_THREADS) {
    const int item = it % nitems, sp = it / nitems;
    const int bb = item / C4, g = item % C4;
    const int ns = cnt_s[bb], first = first_s[bb];
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = sp; s0 < ns; s0 += split * CMB_U) {
      float4 x[CMB_U];
#pragma unroll
      for (int u = 0; u < CMB_U; ++u) {
        const int s = s0 + u * split;
        x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s < ns) {
          const float* src = a.part_o + lse_at(first + s) * C + 4 * g;
          if (vec) {
            x[u] = *reinterpret_cast<const float4*>(src);
          } else {
            x[u].x = src[0];
            if (4 * g + 1 < C) x[u].y = src[1];
            if (4 * g + 2 < C) x[u].z = src[2];
            if (4 * g + 3 < C) x[u].w = src[3];
          }
        }
      }
#pragma unroll
      for (int u = 0; u < CMB_U; ++u) {
        const int s = s0 + u * split;
        const float w = (s < ns) ? wt_s[bb * a.max_slots + s] : 0.f;
        if (w != 0.f) {   // empty slots carry weight 0 and unwritten data: skip, never 0 * x
          acc.x = fmaf(w, x[u].x, acc.x);
          acc.y = fmaf(w, x[u].y, acc.y);
          acc.z = fmaf(w, x[u].z, acc.z);
          acc.w = fmaf(w, x[u].w, acc.w);
        }
      }
    }
    if (split == 1) {
      if (isnan(lse_s[bb])) acc = make_float4(CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F);
      reinterpret_cast<float4*>(vc_s)[bb * C4 + g] = acc;
    } else {
      red_s[it] = acc;
    }
  }
  if (split > 1) {
    __syncthreads();
    for (int item = threadIdx.x; item < nitems; item += CMB_THREADS) {
      const int bb = item / C4;
      float4 v = red_s[item];
      for (int sp = 1; sp < split; ++sp) {   // fixed order: results do not depend on timing
        const float4 t = red_s[sp * nitems + item];
        v.x += t.x; v.y += t.y; v.z += t.z; v.w += t.w;
      }
      if (isnan(lse_s[bb])) v = make_float4(CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F);
      reinterpret_cast<float4*>(vc_s)[item] = v;
    }
  }
  __syncthreads();
  // lse, written by the first V-slice's CTA, one warp per sequence (no barrier: nothing else
  // reads lse_s from here on). When the scores used bf16 latent queries q_hi = q' - res, to
  // first order the exact log-sum-exp is lse + scale * (sum_t p_t kv_lat_t) . res
  // = lse + scale * vc . res.
  if (blockIdx.y == 0 && a.lse != nullptr) {
    for (int bb = warp; bb < nb; bb += CMB_THREADS / 32) {
      float l = lse_s[bb];
      if (a.q_res != nullptr) {
        const uint16_t* res = res_pre ? res_s + bb * C : a.q_res + ((int64_t)(b0 + bb) * a.H + h) * (C + a.R);
        float d = 0.f;
        for (int c = lane; c < C; c += 32) d = fmaf(vc_s[bb * 4 * C4 + c], bf16_bits_to_f32(res[c]), d);
        d = warp_sum(d);
        l += a.scale * d;
      }
      if (lane == 0) a.lse[(int64_t)(b0 + bb) * a.H + h] = l;
    }
  }
  // out[b, h, j0 + j] for all sequences of the block, the CTA's outputs in chunks of 32 W_UV rows
  for (int j0 = jbeg; j0 < jend; j0 += CMB_VJ) {
    const int nj = min(CMB_VJ, jend - j0);
    if (j0 != jbeg) {
      __syncthreads();   // the previous chunk's dot products are done with w_s
      stage_kv_b_rows(w_s, 4 * C4, a.kv_b, a.kv_b_dtype, wrow0 + j0, nj, 0, C, C, CMB_THREADS, kv_rows);
      __syncthreads();
    }
    if (nb == 1) {
      combine_outputs<1>(a, w_s, vc_s, 4 * C4, nb, nj, b0, h, j0);
    } else if (nb == 2) {
      combine_outputs<2>(a, w_s, vc_s, 4 * C4, nb, nj, b0, h, j0);
    } else {
      // more than two sequences: passes of two over the W_UV rows (more accumulators a lane
      // would not fit the register budget of two CTAs per SM)
      for (int p0 = 0; p0 < nb; p0 += 2)
        combine_outputs<2>(a, w_s, vc_s + p0 * (4 * C4), 4 * C4, min(2, nb - p0), nj, b0 + p0, h, j0);
    }
  }
}

// ---- small batches (B <= 8), bf16 or Q8_0 kv_b: one CTA per head ----
// Before the dependency wait every thread issues its share of the head's W_UV rows as raw
// 16-byte cp.async pieces (the whole [V][row] slice in flight at once). After it: one warp per
// sequence forms the slot weights; each thread merges one (sequence, 4 latent columns) item
// with all its slots' loads in flight (sixteen at a time, summed in slot order); one warp per
// output row then decodes its W_UV row from shared memory (lane l: columns 16 l .. 16 l + 15)
// against the merged rows it holds in registers, with fixed-order warp sums.
constexpr int CMB_S_THREADS = 512;
constexpr int CMB_S_BMAX = 8;
constexpr int CMB_S_U = 16;
constexpr int CMB_S_MAXS = 256;
constexpr int CMB_S_VP = 18;       // lane pitch of the merged rows in shared memory (floats)   // slots a sequence may span at most (weights from registers)

template <int WDT, int BT>
__global__ void __launch_bounds__(CMB_S_THREADS, 1) combine_small_kernel(CombineArgs a) {
  extern __shared__ __align__(16) uint8_t sm_raw[];
  pdl_trigger();
  const int h = blockIdx.x;
  const int B = a.B, C = a.C, V = a.V;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int RB = WDT == MLA_Q8_0 ? C / 32 * 34 : C * 2;   // raw bytes of a W_UV row
  uint8_t* w_s = sm_raw;                                                       // [V][RB]
  // merged rows, lane-major for the output phase: [BT][32 lanes][18] (lane l's columns
  // C/32 l .. at 18 l: a row of 64-bit loads across the lanes hits distinct bank pairs)
  float* vc_s = reinterpret_cast<float*>(sm_raw + (((size_t)V * RB + 15) & ~(size_t)15));
  float* wt_s = vc_s + BT * 32 * CMB_S_VP;                                     // [BT][max_slots]
  float* lse_s = wt_s + BT * a.max_slots;                                      // [BT]
  int* first_s = reinterpret_cast<int*>(lse_s + BT);                           // [BT]
  int* cnt_s = first_s + BT;                                                   // [BT]
  const int pg = h / a.hpg, hh = h % a.hpg;
  auto lse_at = [&](int slot) { return ((int64_t)pg * a.n_slots + slot) * a.hpg + hh; };

  {   // W_UV rows of head h % kvb_heads, raw
    const uint8_t* src0 = static_cast<const uint8_t*>(a.kv_b) + ((int64_t)(h % a.kvb_heads) * (a.N + V) + a.N) * RB;
    const int ppr = RB / 16;
    for (int i = tid; i < V * ppr; i += CMB_S_THREADS) {
      const int r = i / ppr, pc = i - r * ppr;
      const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(w_s + r * RB + pc * 16));
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src0 + (int64_t)r * RB + pc * 16)
                   : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  pdl_wait();   // the partials and meta come from the attention kernel
  __shared__ float dres_s[CMB_S_BMAX][4];   // per sequence: vc . residual, by 32-item group
  if (tid < B) {
    first_s[tid] = a.meta[2 * tid];
    cnt_s[tid] = min(a.meta[2 * tid + 1], a.max_slots);
  }
  __syncthreads();

  // vc[b][4 g .. 4 g + 3] = sum_s w_s O_s (slots in order), item (b, g) = it. The first batch of a
  // thread's slot loads (and its query residual) goes out before the slot weights are formed.
  const int C4 = C / 4;
  const bool use_res = a.q_res != nullptr;
  for (int it0 = 0; it0 < BT * C4; it0 += CMB_S_THREADS) {
    const int it = it0 + tid;
    const bool live = it < B * C4;
    const int b = live ? it / C4 : 0, g = it - b * C4;
    const int ns = live ? cnt_s[b] : 0, first = first_s[b];
    float4 x[CMB_S_U];
#pragma unroll
    for (int u = 0; u < CMB_S_U; ++u)
      x[u] = u < ns ? __ldcg(reinterpret_cast<const float4*>(a.part_o + lse_at(first + u) * C) + g)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    uint2 res = make_uint2(0u, 0u);
    if (live && use_res)
      res = *reinterpret_cast<const uint2*>(a.q_res + ((int64_t)b * a.H + h) * (C + a.R) + 4 * g);
    if (it0 == 0) {
      // slot weights exp(lse_s - lse): one warp per sequence, every LSE loaded once
      if (warp < B) {
        const int wn = cnt_s[warp], wf = first_s[warp];
        float lv[CMB_S_MAXS / 32];
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < CMB_S_MAXS / 32; ++k) {
          const int sl = lane + 32 * k;
          lv[k] = sl < wn ? a.part_lse[lse_at(wf + sl)] : -CUDART_INF_F;
          mx = fmaxf(mx, lv[k]);
        }
        mx = warp_max(mx);
        float tot = 0.f;
#pragma unroll
        for (int k = 0; k < CMB_S_MAXS / 32; ++k)
          if (lane + 32 * k < wn) tot += expf(lv[k] - mx);
        tot = warp_sum(tot);
        const float l = (wn > 0) ? mx + logf(tot) : CUDART_NAN_F;
#pragma unroll
        for (int k = 0; k < CMB_S_MAXS / 32; ++k)
          if (lane + 32 * k < wn) wt_s[warp * a.max_slots + lane + 32 * k] = expf(lv[k] - l);
        if (lane == 0) lse_s[warp] = l;
      }
      __syncthreads();
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += CMB_S_U) {
      if (s0 > 0) {
#pragma unroll
        for (int u = 0; u < CMB_S_U; ++u)
          x[u] = s0 + u < ns ? __ldcg(reinterpret_cast<const float4*>(a.part_o + lse_at(first + s0 + u) * C) + g)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < CMB_S_U; ++u) {
        const float w = s0 + u < ns ? wt_s[b * a.max_slots + s0 + u] : 0.f;
        if (w != 0.f) {   // empty slots carry weight 0 and unwritten data: skip, never 0 * x
          acc.x = fmaf(w, x[u].x, acc.x);
          acc.y = fmaf(w, x[u].y, acc.y);
          acc.z = fmaf(w, x[u].z, acc.z);
          acc.w = fmaf(w, x[u].w, acc.w);
        }
      }
    }
    if (it < BT * C4) {
      if (!live) acc = make_float4(0.f, 0.f, 0.f, 0.f);   // sequences past B
      else if (isnan(lse_s[b])) acc = make_float4(CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F, CUDART_NAN_F);
      const int bb = it / C4, col = 4 * (it - bb * C4), cpl = C / 32;
      float* dst = vc_s + (bb * 32 + col / cpl) * CMB_S_VP + col % cpl;
      *reinterpret_cast<float2*>(dst) = make_float2(acc.x, acc.y);
      *reinterpret_cast<float2*>(dst + 2) = make_float2(acc.z, acc.w);
    }
    // vc . residual of this item, summed over the warp's 32 items (all of sequence b: C4 is a
    // multiple of 32), in a fixed order
    float d = 0.f;
    if (live && use_res)
      d = ((acc.x * __uint_as_float(res.x << 16) + acc.y * __uint_as_float(res.x & 0xFFFF0000u)) +
           acc.z * __uint_as_float(res.y << 16)) + acc.w * __uint_as_float(res.y & 0xFFFF0000u);
    d = warp_sum(d);
    if (lane == 0 && live) dres_s[b][(g >> 5) & 3] = d;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // lse: with bf16 latent queries q_hi = q' - res the exact log-sum-exp is, to first order,
  // lse + scale * vc . res
  if (a.lse != nullptr && tid < B) {
    float l = lse_s[tid];
    if (use_res) {
      float d = 0.f;
      for (int k = 0; k < C4 / 32; ++k) d += dres_s[tid][k];
      l += a.scale * d;
    }
    a.lse[(int64_t)tid * a.H + h] = l;
  }

  // out[b, h, v]: warp per row v, lane l over latent columns cpl l .. cpl l + cpl - 1, the
  // sequences' merged rows held in registers four at a time; the four sums meet in a
  // transpose-reduce (lanes trade halves at distances 16 and 8, then add at 4, 2, 1)
  const int cpl = C / 32;   // columns per lane: 8 or 16
#pragma unroll 1
  for (int b0 = 0; b0 < BT; b0 += 4) {
    float2 vr[4][8];
#pragma unroll
    for (int b = 0; b < 4; ++b)
#pragma unroll
      for (int e = 0; e < 8; ++e)
        vr[b][e] = (b0 + b < BT && 2 * e < cpl)
                       ? *reinterpret_cast<const float2*>(vc_s + ((b0 + b) * 32 + lane) * CMB_S_VP + 2 * e)
                       : make_float2(0.f, 0.f);
    for (int v = warp; v < V; v += CMB_S_THREADS / 32) {
      float2 w[8];
      if (WDT == MLA_Q8_0) {
        // the lane's columns lie in block (cpl lane) / 32, from element (cpl lane) % 32
        const int c0 = cpl * lane;
        const uint8_t* blk = w_s + v * RB + (c0 >> 5) * 34;
        const float d = __half2float(*reinterpret_cast<const __half*>(blk));
        const float2 dd = make_float2(d, d), bias = make_float2(-8388736.0f, -8388736.0f);
        const uint16_t* c16 = reinterpret_cast<const uint16_t*>(blk + 2 + (c0 & 31));
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint32_t cc = (2 * e < cpl ? (uint32_t)c16[e] : 0u) ^ 0x8080u;   // absent columns: code 0
          w[e] = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(cc, 0x4B000000u, 0x7650u)),
                                                   __uint_as_float(__byte_perm(cc, 0x4B000000u, 0x7651u))),
                                       bias),
                            dd);
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(w_s + v * RB + 2 * cpl * lane);
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          const uint4 u = q4 * 8 < cpl ? src[q4] : make_uint4(0, 0, 0, 0);
          const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) w[4 * q4 + e] = make_float2(__uint_as_float(uw[e] << 16), __uint_as_float(uw[e] & 0xFFFF0000u));
        }
      }
      float y[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 8; ++e) y2 = __ffma2_rn(w[e], vr[b][e], y2);
        y[b] = y2.x + y2.y;
      }
      const bool c = (lane & 16) != 0, dd8 = (lane & 8) != 0;
      const float w0 = (c ? y[2] : y[0]) + __shfl_xor_sync(0xffffffffu, c ? y[0] : y[2], 16);
      const float w1 = (c ? y[3] : y[1]) + __shfl_xor_sync(0xffffffffu, c ? y[1] : y[3], 16);
      float z = (dd8 ? w1 : w0) + __shfl_xor_sync(0xffffffffu, dd8 ? w0 : w1, 8);
      z += __shfl_xor_sync(0xffffffffu, z, 4);
      z += __shfl_xor_sync(0xffffffffu, z, 2);
      z += __shfl_xor_sync(0xffffffffu, z, 1);
      const int bb = b0 + 2 * (int)c + (int)dd8;   // the sequence this lane's sum belongs to
      if ((lane & 7) == 0 && bb < B) a.out[((int64_t)bb * a.H + h) * V + v] = z;
    }
  }
}

static bool combine_small_fits(const mla_config& cfg, int B, int max_slots) {
  return B >= 1 && B <= CMB_S_BMAX && (cfg.kv_b_dtype == MLA_BF16 || cfg.kv_b_dtype == MLA_Q8_0) &&
         (cfg.kv_lora == 256 || cfg.kv_lora == 512) && cfg.v_head <= 512 && max_slots >= 1 && max_slots <= CMB_S_MAXS;
}

template <int WDT, int BT>
static cudaError_t launch_combine_small_bt(const CombineArgs& a, cudaStream_t st) {
  const int RB = WDT == MLA_Q8_0 ? a.C / 32 * 34 : a.C * 2;
  const size_t smem = (((size_t)a.V * RB + 15) & ~(size_t)15) +
                      sizeof(float) * ((size_t)BT * 32 * CMB_S_VP + (size_t)BT * a.max_slots + 3 * BT);
  auto k = combine_small_kernel<WDT, BT>;
  cudaError_t e = ensure_smem((const void*)k, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(a.H), dim3(CMB_S_THREADS), smem, st, a);
}

template <int WDT>
static cudaError_t launch_combine_small(const CombineArgs& a, cudaStream_t st) {
  if (a.B <= 1) return launch_combine_small_bt<WDT, 1>(a, st);
  if (a.B <= 2) return launch_combine_small_bt<WDT, 2>(a, st);
  if (a.B <= 4) return launch_combine_small_bt<WDT, 4>(a, st);
  return launch_combine_small_bt<WDT, 8>(a, st);
}

cudaError_t launch_combine(const mla_config& cfg, const DecodePlan& plan, const void* kv_b,
                           const int32_t* meta, const float* part_o, const float* part_lse, const void* q_res,
                           float* out, float* lse, int B, cudaStream_t st) {
  CombineArgs a;
  a.kv_b = kv_b; a.meta = meta; a.part_o = part_o; a.part_lse = part_lse;
  a.out = out; a.lse = lse; a.kv_b_dtype = cfg.kv_b_dtype;
  a.q_res = static_cast<const uint16_t*>(q_res);
  a.scale = cfg.softmax_scale;
  a.H = cfg.n_heads; a.C = cfg.kv_lora; a.N = cfg.qk_nope; a.V = cfg.v_head; a.R = cfg.qk_rope; a.B = B;
  a.hpg = plan.part_hpg; a.n_slots = plan.n_slots;
  if (plan.kvb_heads < 1 || plan.kvb_heads * plan.tokens != cfg.n_heads) return cudaErrorInvalidValue;
  a.kvb_heads = plan.kvb_heads;
  // most slots one sequence can span: splits (CUDA-core path) or CTAs per group (tensor path)
  a.max_slots = plan.path != PATH_SIMT ? plan.ctas_per_group : plan.splits;
  if (combine_small_fits(cfg, B, a.max_slots)) {
    const int RB = cfg.kv_b_dtype == MLA_Q8_0 ? cfg.kv_lora / 32 * 34 : cfg.kv_lora * 2;
    const int bt = B <= 1 ? 1 : B <= 2 ? 2 : B <= 4 ? 4 : 8;
    const size_t smem = (((size_t)cfg.v_head * RB + 15) & ~(size_t)15) +
                        sizeof(float) * ((size_t)bt * 32 * CMB_S_VP + (size_t)bt * a.max_slots + 3 * bt);
    if (smem <= 227 * 1024)
      return cfg.kv_b_dtype == MLA_Q8_0 ? launch_combine_small<MLA_Q8_0>(a, st) : launch_combine_small<MLA_BF16>(a, st);
  }
  // V-slices per head: enough CTAs to cover the SMs, but every slice merges the partials again
  const int chunks = (cfg.v_head + CMB_VJ - 1) / CMB_VJ;
  const int64_t base_ctas = (int64_t)cfg.n_heads * ((B + CMB_BC - 1) / CMB_BC);
  int sms = device_sms();
  if (sms <= 0) sms = 152;
  int vsplit = (int)((sms + base_ctas - 1) / base_ctas);
  vsplit = vsplit < 1 ? 1 : (vsplit > chunks ? chunks : vsplit);
  a.vper = ((chunks + vsplit - 1) / vsplit) * CMB_VJ;
  dim3 grid(cfg.n_heads, (cfg.v_head + a.vper - 1) / a.vper, (B + CMB_BC - 1) / CMB_BC);
  const size_t c4 = 4 * (size_t)((cfg.kv_lora + 3) / 4);
  const size_t smem = sizeof(float) * ((size_t)CMB_VJ * c4 + (size_t)CMB_BC * c4 + 4 * (size_t)CMB_THREADS +
                                       (size_t)CMB_BC * a.max_slots + 3 * CMB_BC) +
                      sizeof(uint16_t) * (size_t)CMB_BC * CMB_RES_MAX;
  cudaError_t e = ensure_smem((const void*)combine_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(combine_kernel, grid, dim3(CMB_THREADS), smem, st, a);
}

}  // namespace mla
