// Shared device helpers and the internal launch interface of libmla.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

// ---- workspace header (first 256 bytes of every workspace) ---------------------------------
struct WsHeader {
  int32_t code;   // first device error recorded (mla_status), 0 = none
  int32_t seq;    // sequence index it concerns
  int32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// ---- programmatic dependent launch -------------------------------------------------------------
// Every kernel of a step is launched so that it may start while the kernel before it on the
// stream is still running: it lets its own successor start at once (pdl_trigger) and, before
// touching anything an earlier kernel of the library writes or still reads, waits until its
// predecessor has completed (pdl_wait). Because every kernel waits before it completes, the
// predecessor's completion implies that of all earlier kernels. Launched without the attribute
// (launch_kernel with pdl = false), a kernel starts only after all earlier work on the stream has
// completed and its pdl_wait is a no-op.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&lc, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  return launch_kernel(true, kernel, grid, block, smem, st, static_cast<Args&&>(args)...);
}

// Bounded waits inside the kernels. A wait for copies or MMAs already issued (a drain before a
// CTA exits) always gets kWaitDrainNs; a main-loop wait gets the limit current when the kernel
// was enqueued, wait_limit_ns() (kWaitDrainNs unless mla_set_wait_limit_ns changed it).
constexpr uint64_t kWaitDrainNs = 200ull * 1000 * 1000;
uint64_t wait_limit_ns();

__device__ __forceinline__ void set_error(WsHeader* hdr, int code, int seq) {
  if (atomicCAS(&hdr->code, 0, code) == 0) atomicExch(&hdr->seq, seq);
}

// ---- element access -------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <int DT> struct Act;
template <> struct Act<MLA_F32> {
  using T = float;
  static __device__ __forceinline__ float load(const T* p, int64_t i) { return p[i]; }
  static __device__ __forceinline__ void store(T* p, int64_t i, float v) { p[i] = v; }
  static __device__ __forceinline__ float rounded(float v) { return v; }   // the stored value
};
template <> struct Act<MLA_BF16> {
  using T = uint16_t;
  static __device__ __forceinline__ float load(const T* p, int64_t i) { return bf16_bits_to_f32(p[i]); }
  static __device__ __forceinline__ void store(T* p, int64_t i, float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    p[i] = *reinterpret_cast<uint16_t*>(&h);
  }
  static __device__ __forceinline__ float rounded(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
};

// One kv_b element (row r, column c) in any weight dtype; `rows` is the matrix's row count (the
// 4-bit format keeps its scales and biases after all the codes). Q8_0: fp16 scale then 32
// codes per 34-byte block, value = scale * code (exact in float32). Q4_AFFINE: 8 codes per
// little-endian 32-bit word (code j in bits 4j..4j+3), a bf16 scale and bias per 64 columns,
// value = scale * code + bias.
__device__ __forceinline__ float kv_b_load(const void* kv_b, int dtype, int64_t r, int c, int C, int64_t rows) {
  if (dtype == MLA_BF16) {
    return bf16_bits_to_f32(static_cast<const uint16_t*>(kv_b)[r * C + c]);
  } else if (dtype == MLA_F32) {
    return static_cast<const float*>(kv_b)[r * C + c];
  } else if (dtype == MLA_Q8_0) {
    const uint8_t* blk = static_cast<const uint8_t*>(kv_b) + r * (int64_t)(C / 32) * 34 + (c / 32) * 34;
    uint16_t dbits = static_cast<uint16_t>(blk[0]) | (static_cast<uint16_t>(blk[1]) << 8);
    float d = __half2float(__ushort_as_half(dbits));
    return d * static_cast<float>(static_cast<int8_t>(blk[2 + (c & 31)]));
  } else {
    const uint32_t w = static_cast<const uint32_t*>(kv_b)[(r * C + c) / 8];
    const uint16_t* sb = reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(kv_b) + rows * (int64_t)(C / 2));
    const int64_t g = r * (C / 64) + c / 64;
    return fmaf(bf16_bits_to_f32(sb[g]), static_cast<float>((w >> (4 * (c & 7))) & 15u),
                bf16_bits_to_f32(sb[rows * (C / 64) + g]));
  }
}

// Eight consecutive kv_b elements of row r from column c as float32 (zero past ncols_left):
// one 16-byte load for bf16, two for f32, the 8 codes plus the block scale for Q8_0, one word
// plus its group's scale and bias for Q4_AFFINE.
__device__ __forceinline__ void kv_b_load8(float v[8], const void* kv_b, int dtype, int64_t r, int c,
                                           int ncols_left, int C, int64_t rows) {
  if (ncols_left >= 8 && (C % 8) == 0) {
    if (dtype == MLA_BF16) {
      const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(kv_b) + r * C + c);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        v[2 * e] = __uint_as_float(w[e] << 16);
        v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
      }
    } else if (dtype == MLA_F32) {
      const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(kv_b) + r * C + c);
      const float4 a = src[0], b = src[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else if (dtype == MLA_Q8_0) {
      // a block starts at an even byte offset (34 bytes each), so the scale and the codes are
      // read as 16-bit words (little endian: the lower byte is the lower element)
      const uint16_t* blk = reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(kv_b) +
                                                              r * (int64_t)(C / 32) * 34 + (c / 32) * 34);
      const float d = __half2float(__ushort_as_half(blk[0]));
      const int o = 1 + (c & 31) / 2;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint16_t w = blk[o + e];
        v[2 * e] = d * static_cast<float>(static_cast<int8_t>(w & 0xFF));
        v[2 * e + 1] = d * static_cast<float>(static_cast<int8_t>(w >> 8));
      }
    } else {
      const uint32_t w = static_cast<const uint32_t*>(kv_b)[(r * C + c) / 8];
      const uint16_t* sb =
          reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(kv_b) + rows * (int64_t)(C / 2));
      const int64_t g = r * (C / 64) + c / 64;
      const float sc = bf16_bits_to_f32(sb[g]), bi = bf16_bits_to_f32(sb[rows * (C / 64) + g]);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = fmaf(sc, static_cast<float>((w >> (4 * e)) & 15u), bi);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (e < ncols_left) ? kv_b_load(kv_b, dtype, r, c + e, C, rows) : 0.f;
  }
}

// Stage kv_b rows [r0, r0 + nrows) x columns [c0, c0 + ncols) as float32 into dst (row stride
// dst_stride floats; columns past ncols, up to a multiple of 8, are zero), in items of 8
// columns; each thread issues the loads of four items before it stores any of them. `rows` is
// the whole matrix's row count.
__device__ __forceinline__ void stage_kv_b_rows(float* dst, int dst_stride, const void* kv_b, int dtype,
                                                int64_t r0, int nrows, int c0, int ncols, int C, int nthreads,
                                                int64_t rows) {
  constexpr int U = 4;   // items in flight per thread
  const int ngrp = (ncols + 7) / 8;
  const int total = nrows * ngrp;
  for (int base = threadIdx.x; base < total; base += nthreads * U) {
    float v[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * nthreads;
      if (i < total) {
        const int r = i / ngrp, g = i % ngrp;
        kv_b_load8(v[u], kv_b, dtype, r0 + r, c0 + 8 * g, ncols - 8 * g, C, rows);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * nthreads;
      if (i < total) {
        const int r = i / ngrp, g = i % ngrp;
        float* d = dst + r * dst_stride + 8 * g;
        if (8 * g + 8 <= dst_stride && (reinterpret_cast<uintptr_t>(d) & 15) == 0) {
          reinterpret_cast<float4*>(d)[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
          reinterpret_cast<float4*>(d)[1] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (8 * g + e < dst_stride) d[e] = v[u][e];
        }
      }
    }
  }
}

// Logical row t of sequence b -> physical row, or -1 when it would lie outside the pool: a
// negative page id, a page that does not fit in n_phys rows (the product is formed in 64 bits,
// so no page id can wrap it back into range), or a contiguous row at or past n_phys.
struct RowMap {
  const int32_t* page_table;
  int32_t page_size;
  int32_t max_pages;
  int64_t rows_per_seq;
  int64_t n_phys;
  __device__ __forceinline__ int64_t phys(int b, int64_t t) const {
    if (page_size == 0) {
      const int64_t r = (int64_t)b * rows_per_seq + t;
      return (t >= 0 && r < n_phys) ? r : -1;
    }
    const int64_t pg = page_table[(int64_t)b * max_pages + t / page_size];
    if (pg < 0 || (pg + 1) * (int64_t)page_size > n_phys) return -1;
    return pg * page_size + t % page_size;
  }
  __host__ __device__ __forceinline__ int64_t capacity() const {
    return page_size == 0 ? rows_per_seq : (int64_t)max_pages * page_size;
  }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// RoPE angle for pair i at position pos. The angle pos * inv_freq[i] is formed in float64 and
// reduced to [-pi, pi] there (a - 2*pi*round(a / 2*pi)), so positions in the hundreds of
// thousands keep full accuracy; the reduced angle then goes to the float sincos.
__device__ __forceinline__ void rope_cs_value(double inv_freq, int pos, float* c, float* s) {
  const double two_pi = 6.283185307179586476925286766559;
  const double a = static_cast<double>(pos) * inv_freq;
  const double turns = rint(a * (1.0 / two_pi));
  const float r = static_cast<float>(fma(-turns, two_pi, a));
  sincosf(r, s, c);
}

__device__ __forceinline__ void rope_cs(const double* inv_freq, int i, int pos, float* c, float* s) {
  rope_cs_value(inv_freq[i], pos, c, s);
}

// The same angle in float arithmetic only (double throughput is very low on this GPU), for a
// frequency given as two floats inv_hi + inv_lo with 0 < inv_hi <= 1 and 0 <= pos < ROPE_F32_MAX_POS:
// the product pos * inv as an unevaluated sum a_hi + a_lo (the FMA yields the rounding error of
// pos * inv_hi exactly), then a three-term Cody-Waite reduction by 2 pi = P1 + P2 + P3 with
// P1 = 201/32 (8 significant bits, so k * P1 is exact for quotients k < 2^16 and a_hi - k * P1
// is exact), P2 and P3 the float roundings of the successive remainders: about 5e-7 rad of
// absolute error. The reduced angle lies in [-pi, pi] (to rounding), where the hardware sine and
// cosine approximations are accurate to about 2^-21 absolute.
constexpr int ROPE_F32_MAX_POS = 1 << 18;
__device__ __forceinline__ void rope_cs_f32(float inv_hi, float inv_lo, int pos, float* c, float* s) {
  const float x = static_cast<float>(pos);                 // exact: pos < 2^24
  const float a_hi = x * inv_hi;
  const float a_lo = fmaf(x, inv_hi, -a_hi) + x * inv_lo;
  const float k = rintf(a_hi * 0.15915494f);               // whole turns
  float r = fmaf(-k, 6.28125f, a_hi);
  r = fmaf(-k, 1.9353071693331003e-3f, r);
  r = fmaf(-k, 1.0253131677018246e-11f, r);
  __sincosf(r + a_lo, s, c);
}

// The frequency of pair i as an unevaluated float sum hi + lo (two float64 operations, done once
// per pair in a kernel's prologue: float64 arithmetic is slow on this GPU).
__device__ __forceinline__ void rope_freq_split(const double* inv_freq, int i, float* hi, float* lo) {
  const double inv = inv_freq[i];
  const float h = __double2float_rn(inv);
  *hi = h;
  *lo = __double2float_rn(inv - static_cast<double>(h));
}
// The RoPE angle of pair i at pos: in float arithmetic from (hi, lo) where that form holds
// (0 < hi <= 1, 0 <= pos < ROPE_F32_MAX_POS), else in float64 from inv_freq.
__device__ __forceinline__ void rope_cs_split(const double* inv_freq, float hi, float lo, int i, int pos, float* c,
                                              float* s) {
  if (pos >= 0 && pos < ROPE_F32_MAX_POS && hi > 0.f && hi <= 1.f)
    rope_cs_f32(hi, lo, pos, c, s);
  else
    rope_cs(inv_freq, i, pos, c, s);
}

// ---- decode plan: how the rows of a sequence are split, and the workspace layout -------------
struct DecodePlan {
  int path;              // PATH_SIMT or PATH_TC
  int heads_per_cta;     // heads sharing one staged row tile in one CTA
  int n_groups;          // ceil(H / heads_per_cta)
  int splits;            // CUDA-core path: row splits per sequence
  int64_t chunk_rows;    // CUDA-core path: rows per split (a multiple of its row tile)
  int64_t capacity;      // maximum rows a sequence can attend
  int ctas_per_group;    // tensor-core paths: CTAs (pair path: CTA pairs) sharing one tile list
  // query tokens per sequence: the attention and combine see tokens * kvb_heads heads per
  // sequence (token-major); head m up-projects through W_UV of head m % kvb_heads and sees the
  // rows before L - tokens + 1 + m / kvb_heads
  int tokens, kvb_heads;
  // partials: part_o[g][slot][hh][C], part_lse[g][slot][hh] for part_groups x n_slots slots of
  // part_hpg heads; meta[b] = {first slot, slot count} of sequence b (count 0: invalid length)
  int part_groups, part_hpg, n_slots;
  // q_res: bf16 rounding residual of the fused query rows (bf16 activations only)
  size_t off_qabs, off_qres, off_po, off_plse, off_meta, total;
  // one-launch decode for tiny batches (decode_small.cu), used by mla_decode_attn when set;
  // its float32 queries, chunk partials, slice shares of out and per-head counters follow the
  // staged layout
  int small;
  size_t off_sq, off_sp, off_sw, off_sc;
};
enum { PATH_SIMT = 0, PATH_TC = 1, PATH_PAIR = 2 };

// one-launch decode for tiny batches: absorb, attention over 32-row chunks, merge and W_UV in
// one grid with bounded grid-wide barriers (decode_small.cu)
bool decode_small_supported(const mla_config& cfg, int B, int tokens);
int64_t decode_small_max_chunks(const mla_config& cfg);
int decode_small_grid(const mla_config& cfg, int B);
cudaError_t launch_decode_small(const mla_config& cfg, const mla_cache& cache, const void* q, const void* kv_b,
                                const int32_t* seq_lens, const int32_t* positions, float* out, float* lse, int B,
                                float* qf, float* part, float* wshare, unsigned int* head_cnt, WsHeader* hdr,
                                cudaStream_t st);

// True when the CUDA driver's tensor-map encoder could be found (looked up once per process).
bool tma_encoder_available();
// 2D bf16 TMA map over a row-major [rows, inner] tensor (inner elements contiguous) with
// boxes of box_inner x box_rows and the 128-byte swizzle (64-byte with swizzle_bytes = 64, for
// boxes 32 elements wide). False when the CUDA driver entry point is unavailable or the encoding
// is rejected.
bool make_map_2d_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows, int swizzle_bytes = 128);
bool make_map_row_blocks_bf16(CUtensorMap* m, const void* base, uint64_t row_elems, uint64_t rows,
                              uint32_t n_blocks, uint32_t box_rows, uint32_t box_blocks);

// Raise a kernel's dynamic shared memory limit once per (kernel, device), so that repeated
// launches (and launches under stream capture) make no attribute calls.
cudaError_t ensure_smem(const void* func, int bytes);
// Multiprocessor count of the current device (cached per device), or -1 on a CUDA error.
int device_sms();

// host launchers (defined in the kernel files)
cudaError_t launch_append_finish(const mla_config& cfg, const mla_cache& cache, const float* kva,
                                 const float* norm_w, const int32_t* positions,
                                 const int32_t* seq_lens, int B, WsHeader* hdr, bool kva_dep, cudaStream_t st);
// pdl = false: the absorb starts only after all earlier work on the stream has completed
// pos_t: query tokens per sequence; the position of query row b is positions[b / pos_t] + b % pos_t
cudaError_t launch_absorb(const mla_config& cfg, const void* q, const void* kv_b,
                          const int32_t* positions, void* q_abs, void* q_res, int B, bool pdl, cudaStream_t st,
                          int pos_t = 1);
cudaError_t launch_attn_simt(const mla_config& cfg, const mla_cache& cache, const DecodePlan& plan,
                             const int32_t* seq_lens, const void* q_abs, const void* q_res, float* part_o,
                             float* part_lse, int32_t* meta, int B, WsHeader* hdr, cudaStream_t st);
// kv_early: the kernel launched just before is an absorb launched with pdl = false, so cache rows
// may be read before the dependency wait (only the queries wait for the absorb)
cudaError_t launch_attn_tc(const mla_config& cfg, const mla_cache& cache, const DecodePlan& plan,
                           const int32_t* seq_lens, const void* q_abs, const void* q_res, float* part_o,
                           float* part_lse, int32_t* meta, int B, WsHeader* hdr, bool kv_early, cudaStream_t st);
bool attn_tc_supported(const mla_config& cfg);
// 128 heads on a pair of SMs (a cluster of two CTAs, 64-row tiles)
bool attn_pair_supported(const mla_config& cfg);
// cluster pairs of the pair kernel that fit on the current device at once, or -1
int attn_pair_max_pairs();
cudaError_t launch_attn_pair(const mla_config& cfg, const mla_cache& cache, const DecodePlan& plan,
                             const int32_t* seq_lens, const void* q_abs, const void* q_res, float* part_o,
                             float* part_lse, int32_t* meta, int B, WsHeader* hdr, bool kv_early, cudaStream_t st);
int tc_heads_per_cta(int H);
bool absorb_tc_supported(const mla_config& cfg, int B);
bool combine_tc_supported(const mla_config& cfg, int B);
cudaError_t launch_absorb_tc(const mla_config& cfg, const void* q, const void* kv_b, const int32_t* positions,
                             void* q_abs, void* q_res, int B, WsHeader* hdr, bool pdl, cudaStream_t st,
                             int pos_t = 1);
// q_res != nullptr: the partials came from bf16 latent queries; the combine adds the first-order
// LSE correction softmax_scale * (vc . q_res[latent]) for the residual the scores did not see.
cudaError_t launch_combine_tc(const mla_config& cfg, const DecodePlan& plan, const void* kv_b,
                              const int32_t* meta, const float* part_o, const float* part_lse, const void* q_res,
                              float* out, float* lse, int B, WsHeader* hdr, cudaStream_t st);
// projections (proj.cu): y = W x for one or two weight matrices sharing x [B, K]
cudaError_t launch_proj(const void* x, bool x_bf16, int K, int B, int w_dtype, const void* w0, int64_t rows0,
                        void* y0, bool y0_bf16, const void* w1, int64_t rows1, void* y1, bool y1_bf16,
                        cudaStream_t st);
cudaError_t launch_rms_norm_rows(float* x, const float* w, int K, int B, float eps, cudaStream_t st,
                                 uint16_t* hi = nullptr, uint16_t* lo = nullptr);
// tensor-core projections (bf16 weights, up to 128/256 sequences), see proj.cu
struct ProjTcPlan {
  bool use;
  int xsplit, BP, NB, nkb, kb_per_split, splits, stages;
  int64_t tiles0, tiles1, part_floats;
};
ProjTcPlan proj_tc_plan(int64_t rows0, int64_t rows1, int K, int B, bool x_f32, int w_dtype);
cudaError_t launch_proj_tc(const ProjTcPlan& p, const void* x, const void* x_lo, int K, int B, const void* w0,
                           int64_t rows0, void* y0, bool y0_bf16, const void* w1, int64_t rows1, void* y1,
                           bool y1_bf16, float* part, WsHeader* hdr, cudaStream_t st);
cudaError_t launch_split_hi_lo(const float* x, int64_t n, uint16_t* hi, uint16_t* lo, cudaStream_t st);
cudaError_t launch_combine(const mla_config& cfg, const DecodePlan& plan, const void* kv_b,
                           const int32_t* meta, const float* part_o, const float* part_lse, const void* q_res,
                           float* out, float* lse, int B, cudaStream_t st);

}  // namespace mla
