// The projections around the decode step: the layer's front end (the Q chain q_a ->
// q_a_layernorm -> q_b, or one direct q projection, plus kv_a from the same input) and o_proj
// after the up-projection.
//
// moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs, mla_attn_layer_forward_gpu: Q chain
// (q_a_proj matvec, RMSNorm of q_lat over q_lora_rank, q_b_proj matvec), KV-A chain
// (kv_a_proj_with_mqa matvec), o_proj final matvec; turbospark-runtime 0.3.0,
// src/families/deepseek2/attn.rs, encode_mla_attention_block: Q_PROJ GEMV of the normed hidden
// state, O_PROJ GEMV of the combined heads.
//
// Each projection is y[b, r] = sum_k W[r, k] x[b, k], a weight stream: every weight is read from
// memory once per pass of 8 sequences and used for 8 multiply-adds per sequence of the pass. A
// warp owns 4 consecutive rows and one slice of the columns; each lane takes 8 consecutive
// columns per 256-column step (one 16-byte load per row for bf16 weights, the 8 codes and their
// block scale for Q8_0, one word and its group's scale and bias for the 4-bit format), so the
// x values it loads serve all 4 rows. The 32 per-lane sums of a warp (4 rows x 8 sequences) are
// reduced by a butterfly that halves the live values at each of its five steps (31 shuffles
// for all 32 sums, lane l ending with sum l), then the column slices of a row group are added
// in slice order through shared memory. Every sum has a fixed order, so results are
// run-to-run identical. One launch can serve two matrices that read the same x (q_a or q, and
// kv_a): the CTAs past the first matrix's take the second's rows.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <math_constants.h>

namespace mla {

namespace {

// bf16 bit pattern of v, round to nearest even
__device__ __forceinline__ uint16_t pt_bf16_bits(float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  return *reinterpret_cast<uint16_t*>(&h);
}

constexpr int PJ_WARPS = 8;
constexpr int PJ_THREADS = 32 * PJ_WARPS;
constexpr int PJ_RW = 4;     // rows per warp
constexpr int PJ_BP = 8;     // sequences per pass
constexpr int PJ_STEP = 256; // columns per warp step (32 lanes x 8)
static_assert(PJ_RW * PJ_BP == 32, "one reduced sum per lane");

struct ProjArgs {
  const void* w[2];      // [rows, K] in the weight dtype
  int64_t rows[2];
  void* y[2];            // [B, rows]: float32, or bf16 where y_bf16
  int y_bf16[2];
  int64_t ctas0;         // CTAs serving matrix 0; the rest serve matrix 1
  const void* x;         // [B, K] float32 or bf16, 16-byte aligned
  int K, B;
  int ksplit;            // warps sharing a row group's columns (1, 2, 4 or 8)
};

template <bool XBF>
__device__ __forceinline__ void load_x8(float v[8], const void* x, int64_t off) {
  if (XBF) {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = __uint_as_float(w[e] << 16);
      v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// v[i] summed over the warp's lanes for all 32 i at once: after the step with offset o, a lane
// keeps the half of its values selected by its bit o (added to the partner's copy of that
// half), so lane l finally holds the sum of every lane's v[l].
__device__ __forceinline__ float warp_sum32_scatter(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? v[i] : v[i + n / 2];
      const float keep = up ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

// Eight consecutive weights of one row as loaded (raw), decoded to float32 only when used, so
// that the loads of two column steps can be in flight at once without holding 64 floats.
template <int WD> struct Raw8;
template <> struct Raw8<MLA_BF16> {
  uint4 u;
  __device__ __forceinline__ void load(const void* W, int64_t r, int k, int K, int64_t) {
    u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(W) + r * K + k);
  }
  __device__ __forceinline__ void zero() { u = make_uint4(0, 0, 0, 0); }
  __device__ __forceinline__ void get(float v[8]) const {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = __uint_as_float(w[e] << 16);
      v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
};
template <> struct Raw8<MLA_F32> {
  float4 a, b;
  __device__ __forceinline__ void load(const void* W, int64_t r, int k, int K, int64_t) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(W) + r * K + k);
    a = p[0];
    b = p[1];
  }
  __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
  __device__ __forceinline__ void get(float v[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};
// Q8_0: 34-byte blocks (fp16 scale, 32 int8 codes) along the row; a block starts at an even
// byte offset, so the scale and the codes are read as 16-bit words (lower byte = lower column)
template <> struct Raw8<MLA_Q8_0> {
  uint32_t c01, c23;   // the 8 codes
  float d;
  __device__ __forceinline__ void load(const void* W, int64_t r, int k, int K, int64_t) {
    const uint16_t* blk = reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(W) +
                                                            r * (int64_t)(K / 32) * 34 + (k / 32) * 34);
    const int o = 1 + (k & 31) / 2;
    d = __half2float(__ushort_as_half(blk[0]));
    c01 = (uint32_t)blk[o] | ((uint32_t)blk[o + 1] << 16);
    c23 = (uint32_t)blk[o + 2] | ((uint32_t)blk[o + 3] << 16);
  }
  __device__ __forceinline__ void zero() { c01 = c23 = 0; d = 0.f; }
  __device__ __forceinline__ void get(float v[8]) const {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[e] = d * (float)(int8_t)(c01 >> (8 * e));
      v[4 + e] = d * (float)(int8_t)(c23 >> (8 * e));
    }
  }
};
// 4-bit affine: 8 codes per little-endian word (code j in bits 4j..4j+3), then after all the
// codes the bf16 scales and then the bf16 biases, one of each per 64 columns of a row
template <> struct Raw8<MLA_Q4_AFFINE> {
  uint32_t w;
  float sc, bi;
  __device__ __forceinline__ void load(const void* W, int64_t r, int k, int K, int64_t rows) {
    w = static_cast<const uint32_t*>(W)[(r * K + k) / 8];
    const uint16_t* sb = reinterpret_cast<const uint16_t*>(static_cast<const uint8_t*>(W) + rows * (int64_t)(K / 2));
    const int64_t g = r * (K / 64) + k / 64;
    sc = bf16_bits_to_f32(sb[g]);
    bi = bf16_bits_to_f32(sb[rows * (K / 64) + g]);
  }
  __device__ __forceinline__ void zero() { w = 0; sc = bi = 0.f; }
  __device__ __forceinline__ void get(float v[8]) const {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = fmaf(sc, (float)((w >> (4 * e)) & 15u), bi);
  }
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async8(void* smem, const void* gmem) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Shared-memory x chunk of one round (PJ_ROUND columns of up to PJ_BP sequences). float32: the
// 8 values a lane uses in a step are stored as two 16-byte halves 512 bytes apart (half h of
// lane l at h*128 + 4*l floats of the step), so each quarter-warp's 16-byte reads cover all 32
// banks; bf16: a lane's 8 values are one 16-byte run, already conflict-free.
constexpr int PJ_ROUND = 4 * PJ_STEP;   // columns per round

template <bool XBF>
__device__ __forceinline__ void stage_x_round(uint8_t* xs, const void* x, int64_t b0, int nb, int K, int c0) {
  constexpr int EB = XBF ? 2 : 4;            // bytes per element
  constexpr int PC = 16 / EB;                // columns per 16-byte piece
  constexpr int PPS = PJ_ROUND / PC;         // pieces per sequence in a round
  const int cols = min(PJ_ROUND, K - c0);
  const int npieces = nb * PPS;
  for (int i = threadIdx.x; i < npieces; i += PJ_THREADS) {
    const int j = i / PPS, p = i % PPS;
    if (p * PC >= cols) continue;
    const uint8_t* src = static_cast<const uint8_t*>(x) + ((b0 + j) * (int64_t)K + c0 + p * PC) * EB;
    int dst;   // element offset within the sequence's round
    if (XBF) {
      dst = p * PC;
    } else {
      const int st = p / 64, q = p % 64;      // 64 pieces of 4 floats per step
      dst = st * PJ_STEP + (q & 1) * 128 + (q >> 1) * 4;
    }
    cp_async16(xs + ((int64_t)j * PJ_ROUND + dst) * EB, src);
  }
}

template <bool XBF>
__device__ __forceinline__ void load_x8_smem(float v[8], const uint8_t* xs, int j, int st_in_round, int lane) {
  if (XBF) {
    const uint4 u = *reinterpret_cast<const uint4*>(xs + ((int64_t)j * PJ_ROUND + st_in_round * PJ_STEP + lane * 8) * 2);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[2 * e] = __uint_as_float(w[e] << 16);
      v[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
    }
  } else {
    const float* base = reinterpret_cast<const float*>(xs) + (int64_t)j * PJ_ROUND + st_in_round * PJ_STEP + lane * 4;
    const float4 a = *reinterpret_cast<const float4*>(base);
    const float4 b = *reinterpret_cast<const float4*>(base + 128);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// CTA: 8 warps = (8 / S) row groups of 4 rows x S column slices. The columns go by rounds of
// 4 steps (1024 columns); in a round, slice s takes steps s, s+S, ... of it. The round's x
// values (PJ_BP sequences) are copied into shared memory with cp.async one round ahead; each
// warp keeps the raw weights of its next step in flight while it computes the current one.
template <int WD, bool XBF>
__global__ void __launch_bounds__(PJ_THREADS, 2) proj_gemv_kernel(const __grid_constant__ ProjArgs a) {
  extern __shared__ __align__(16) uint8_t xs_raw[];
  __shared__ float red[PJ_WARPS][32];
  constexpr int EB = XBF ? 2 : 4;
  constexpr int XS_BUF = PJ_BP * PJ_ROUND * EB;   // bytes of one round buffer
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.ksplit, g = warp / S, s = warp % S;
  const bool second = blockIdx.x >= a.ctas0;
  const int64_t cta = second ? blockIdx.x - a.ctas0 : blockIdx.x;
  const int64_t rows = second ? a.rows[1] : a.rows[0];
  const void* W = second ? a.w[1] : a.w[0];
  void* Y = second ? a.y[1] : a.y[0];
  const bool ybf = second ? a.y_bf16[1] != 0 : a.y_bf16[0] != 0;
  const int K = a.K;
  const int64_t r0 = (cta * (PJ_WARPS / S) + g) * PJ_RW;
  const int nrounds = (K + PJ_ROUND - 1) / PJ_ROUND;
  const int spr = 4 / S;                 // steps per warp per round
  bool row_ok[PJ_RW];
#pragma unroll
  for (int r = 0; r < PJ_RW; ++r) row_ok[r] = r0 + r < rows;
  // the warp's n-th step: round n / spr, step s + S * (n % spr) of it
  auto step_col = [&](int n) { return (n / spr) * PJ_ROUND + (s + S * (n % spr)) * PJ_STEP + lane * 8; };
  const int nsteps = nrounds * spr;
  auto load_raw = [&](Raw8<WD> (&raw)[PJ_RW], int n) {
    const int k = step_col(n);
#pragma unroll
    for (int r = 0; r < PJ_RW; ++r) {
      if (n < nsteps && k < K && row_ok[r]) raw[r].load(W, r0 + r, k, K, rows);
      else raw[r].zero();
    }
  };

  // weights are not produced by an earlier kernel: the first step's loads go out before the wait
  Raw8<WD> cur[PJ_RW];
  load_raw(cur, 0);
  pdl_wait();   // x may be the previous kernel's output, and y may still be read by it

  for (int b0 = 0; b0 < a.B; b0 += PJ_BP) {
    const int nb = min(PJ_BP, a.B - b0);
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    stage_x_round<XBF>(xs_raw, a.x, b0, nb, K, 0);
    cp_async_commit();
    int n = 0;
    for (int t = 0; t < nrounds; ++t) {
      if (t + 1 < nrounds) stage_x_round<XBF>(xs_raw + ((t + 1) & 1) * XS_BUF, a.x, b0, nb, K, (t + 1) * PJ_ROUND);
      cp_async_commit();
      cp_async_wait<1>();
      __syncthreads();
      const uint8_t* xr = xs_raw + (t & 1) * XS_BUF;
      for (int q = 0; q < spr; ++q, ++n) {
        Raw8<WD> nxt[PJ_RW];
        // next step: the pass's next one, or the first one of the next pass
        load_raw(nxt, n + 1 < nsteps ? n + 1 : (b0 + PJ_BP < a.B ? 0 : nsteps));
        const int k = step_col(n);
        if (k < K) {
          float w[PJ_RW][8];
#pragma unroll
          for (int r = 0; r < PJ_RW; ++r) cur[r].get(w[r]);
#pragma unroll
          for (int j = 0; j < PJ_BP; ++j) {
            if (j < nb) {
              float xv[8];
              load_x8_smem<XBF>(xv, xr, j, s + S * q, lane);
#pragma unroll
              for (int r = 0; r < PJ_RW; ++r)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r * PJ_BP + j] = fmaf(w[r][e], xv[e], acc[r * PJ_BP + j]);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < PJ_RW; ++r) cur[r] = nxt[r];
      }
      __syncthreads();   // every warp is done with this buffer before the copy two rounds on
    }
    red[warp][lane] = warp_sum32_scatter(acc, lane);
    __syncthreads();
    if (s == 0) {
      float v = 0.f;
      for (int t = 0; t < S; ++t) v += red[warp + t][lane];
      const int r = lane / PJ_BP, j = lane % PJ_BP;
      if (r0 + r < rows && j < nb) {
        const int64_t o = (int64_t)(b0 + j) * rows + r0 + r;
        if (ybf) {
          __nv_bfloat16 hv = __float2bfloat16_rn(v);
          static_cast<uint16_t*>(Y)[o] = *reinterpret_cast<uint16_t*>(&hv);
        } else {
          static_cast<float*>(Y)[o] = v;
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
}

// ---- bf16 / float32 weights: a per-lane cp.async ring -------------------------------------
// Each lane copies its own 16 bytes (bf16: 8 columns; float32: two pieces) of each of its warp's
// 4 rows for a step straight into shared memory and later reads back exactly those bytes, so
// the ring needs no barrier: cp.async.wait_group orders a lane's own copies. D steps are in
// flight per warp. x goes through one shared buffer per round (16 KB: 1024 bf16 or 512 float32
// columns of 8 sequences), loaded into registers a round ahead and stored between the
// round's two barriers.
// Quantised weights (Q8_0, 4-bit affine) go through the same ring as raw bytes, when K is a
// multiple of 256 (whole steps; every run below starts on a 16- or 8-byte boundary): a step of
// a row is 8 Q8_0 blocks (8 x 34 = 272 bytes, 17 pieces of 16 bytes), or 128 bytes of 4-bit
// codes plus the row's 4 bf16 scales and 4 bf16 biases (two 8-byte pieces). The warp's pieces
// are shared out over its lanes, so a lane decodes bytes other lanes copied: a __syncwarp after
// the wait makes them visible, and one after the step's use frees the slot for reuse.
// SLOT: bytes of one step of the warp's 4 rows; D: steps in flight per warp.
template <int WD> struct Ring;
template <> struct Ring<MLA_BF16> { static constexpr int D = 4, LB = 16, SLOT = PJ_RW * 32 * 16; };
template <> struct Ring<MLA_F32> { static constexpr int D = 2, LB = 32, SLOT = PJ_RW * 32 * 32; };
template <> struct Ring<MLA_Q8_0> { static constexpr int D = 8, LB = 0, SLOT = PJ_RW * 272; };
template <> struct Ring<MLA_Q4_AFFINE> { static constexpr int D = 8, LB = 0, SLOT = PJ_RW * (128 + 16); };

template <bool XBF> struct XRound {
  static constexpr int EB = XBF ? 2 : 4;
  static constexpr int COLS = XBF ? 1024 : 512;        // columns per round
  static constexpr int STEPS = COLS / PJ_STEP;          // steps per round (4 or 2)
  static constexpr int PC = 16 / EB;                    // columns per 16-byte piece
  static constexpr int PPS = COLS / PC;                 // pieces per sequence (128)
  static constexpr int BYTES = PJ_BP * COLS * EB;       // 16 KB
  static constexpr int PPT = PJ_BP * PPS / PJ_THREADS;  // pieces per thread (4)
};

template <int WD, bool XBF>
constexpr int ring_smem_bytes() {
  return XRound<XBF>::BYTES + PJ_WARPS * Ring<WD>::D * Ring<WD>::SLOT;
}

template <int WD, bool XBF>
__global__ void __launch_bounds__(PJ_THREADS, 2) proj_gemv_ring_kernel(const __grid_constant__ ProjArgs a) {
  using XR = XRound<XBF>;
  constexpr int D = Ring<WD>::D, LB = Ring<WD>::LB, SLOT = Ring<WD>::SLOT, EW = WD == MLA_BF16 ? 2 : 4;
  constexpr bool QUANT = WD == MLA_Q8_0 || WD == MLA_Q4_AFFINE;
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ float red[PJ_WARPS][32];
  uint8_t* xs = sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = sm + XR::BYTES + warp * (D * SLOT);
  pdl_trigger();
  const int S = a.ksplit, g = warp / S, s = warp % S;
  const bool second = blockIdx.x >= a.ctas0;
  const int64_t cta = second ? blockIdx.x - a.ctas0 : blockIdx.x;
  const int64_t rows = second ? a.rows[1] : a.rows[0];
  const uint8_t* W = static_cast<const uint8_t*>(second ? a.w[1] : a.w[0]);
  void* Y = second ? a.y[1] : a.y[0];
  const bool ybf = second ? a.y_bf16[1] != 0 : a.y_bf16[0] != 0;
  const int K = a.K;
  const int64_t r0 = (cta * (PJ_WARPS / S) + g) * PJ_RW;
  const int nrounds = (K + XR::COLS - 1) / XR::COLS;
  const int lg_s = S == 1 ? 0 : (S == 2 ? 1 : 2);          // S is 1, 2 or 4
  const int lg_spr = (XBF ? 2 : 1) - lg_s;                  // steps of a warp per round
  const int spr = 1 << lg_spr;
  const int nsteps = nrounds << lg_spr;
  // each row's first byte (rows past the matrix point at its first row and copy nothing)
  const uint8_t* wrow[PJ_RW];
  bool row_ok[PJ_RW];
#pragma unroll
  for (int r = 0; r < PJ_RW; ++r) {
    row_ok[r] = r0 + r < rows;
    const int64_t rr = row_ok[r] ? r0 + r : 0;
    wrow[r] = W + rr * (int64_t)K * EW + lane * 8 * EW;   // bf16 / float32
  }
  // 4-bit: the scales and the biases of all rows follow the codes
  const uint8_t* q4_sc = W + rows * (int64_t)(K / 2);
  const uint8_t* q4_bi = q4_sc + rows * (int64_t)(K / 64) * 2;
  auto step_col = [&](int n) {
    return (n >> lg_spr) * XR::COLS + ((s + ((n & (spr - 1)) << lg_s)) * PJ_STEP) + lane * 8;
  };
  // step n's weights into ring slot n % D (rows or columns outside the matrix are not copied:
  // their slot bytes are never used for a stored result); always closes one commit group
  auto issue = [&](int n) {
    if (n < nsteps) {
      const int k = step_col(n);
      if (k < K) {
        if constexpr (WD == MLA_Q8_0) {
          // 68 pieces: piece i = (row i / 17, 16-byte piece i % 17), lane i % 32
          uint8_t* slot = ring + (n % D) * SLOT;
          const int64_t boff = (int64_t)((k - lane * 8) / 32) * 34;
#pragma unroll
          for (int u = 0; u < 3; ++u) {
            const int i = lane + 32 * u;
            const int r = i / 17, pc = i % 17;   // lane-dependent row: addressed directly
            if (i < PJ_RW * 17 && r0 + r < rows)
              cp_async16(slot + r * 272 + 16 * pc, W + (r0 + r) * (int64_t)(K / 32) * 34 + boff + 16 * pc);
          }
        } else if constexpr (WD == MLA_Q4_AFFINE) {
          // codes: lane l copies piece l % 8 of row l / 8; lanes 0-7 also the scales (rows
          // 0-3) or the biases (rows 0-3) of the step's four 64-column groups
          uint8_t* slot = ring + (n % D) * SLOT;
          const int k0 = k - lane * 8;
          const int r = lane >> 3, pc = lane & 7;   // lane-dependent row: addressed directly
          if (r0 + r < rows) cp_async16(slot + r * 128 + 16 * pc, W + (r0 + r) * (int64_t)(K / 2) + k0 / 2 + 16 * pc);
          if (lane < 8) {
            const int rr = lane & 3;
            if (r0 + rr < rows) {
              const int64_t g = (r0 + rr) * (int64_t)(K / 64) + k0 / 64;
              cp_async8(slot + PJ_RW * 128 + (lane >> 2) * 32 + rr * 8, (lane < 4 ? q4_sc : q4_bi) + g * 2);
            }
          }
        } else {
          uint8_t* slot = ring + (n % D) * SLOT + lane * LB;
          const int koff = (k - lane * 8) * EW;
#pragma unroll
          for (int r = 0; r < PJ_RW; ++r) {
            if (row_ok[r]) {
#pragma unroll
              for (int h = 0; h < LB / 16; ++h) cp_async16(slot + r * 32 * LB + 16 * h, wrow[r] + koff + 16 * h);
            }
          }
        }
      }
    }
    cp_async_commit();
  };
  uint4 xreg[XR::PPT];
  auto x_load = [&](int64_t b0, int nb, int t) {
    const int c0 = t * XR::COLS;
#pragma unroll
    for (int i = 0; i < XR::PPT; ++i) {
      const int piece = threadIdx.x + i * PJ_THREADS;
      const int j = piece / XR::PPS, p = piece % XR::PPS;
      xreg[i] = make_uint4(0, 0, 0, 0);
      if (j < nb && c0 + p * XR::PC < K)
        xreg[i] = *reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.x) +
                                                  ((b0 + j) * (int64_t)K + c0 + p * XR::PC) * XR::EB);
    }
  };
  auto x_store = [&]() {
#pragma unroll
    for (int i = 0; i < XR::PPT; ++i) {
      const int piece = threadIdx.x + i * PJ_THREADS;
      const int j = piece / XR::PPS, p = piece % XR::PPS;
      int dst;   // element offset within the sequence's round (float32: halves 128 floats apart)
      if (XBF) {
        dst = p * XR::PC;
      } else {
        const int st = p / 64, q = p % 64;
        dst = st * PJ_STEP + (q & 1) * 128 + (q >> 1) * 4;
      }
      *reinterpret_cast<uint4*>(xs + ((int64_t)j * XR::COLS + dst) * XR::EB) = xreg[i];
    }
  };

  // the weights are no other kernel's output: the first steps' copies start before the wait
#pragma unroll
  for (int i = 0; i < D - 1; ++i) issue(i);
  pdl_wait();   // x may be the previous kernel's output, and y may still be read by it

  for (int b0 = 0; b0 < a.B; b0 += PJ_BP) {
    const int nb = min(PJ_BP, a.B - b0);
    if (b0 > 0) {
#pragma unroll
      for (int i = 0; i < D - 1; ++i) issue(i);
    }
    x_load(b0, nb, 0);
    x_store();
    __syncthreads();
    if (nrounds > 1) x_load(b0, nb, 1);
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    int n = 0;
    for (int t = 0; t < nrounds; ++t) {
      for (int q = 0; q < spr; ++q, ++n) {
        issue(n + D - 1);
        cp_async_wait<D - 1>();
        if constexpr (QUANT) __syncwarp();   // the other lanes' pieces of this step have landed
        const int k = step_col(n);
        if (k < K) {
          const uint8_t* slot = ring + (n % D) * SLOT;
          float w[PJ_RW][8];
#pragma unroll
          for (int r = 0; r < PJ_RW; ++r) {
            if constexpr (WD == MLA_Q8_0) {
              // lane l: block l / 4 of the step, codes 8 (l % 4) .. +7, as 16-bit-aligned bytes
              const uint8_t* blk = slot + r * 272 + (lane >> 2) * 34;
              const float d = __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(blk)));
              const uint32_t o = (uint32_t)(blk - slot) + 2 + 8 * (lane & 3);   // even
              const uint32_t* wp = reinterpret_cast<const uint32_t*>(slot + (o & ~3u));
              const uint32_t sh = (o & 3u) * 8;                                  // 0 or 16
              // the third word only when the codes straddle it (the last block's last lane
              // would otherwise read past the row)
              const uint32_t w0 = wp[0], w1 = wp[1], w2 = sh ? wp[2] : 0u;
              // the sign bit of every code flipped, then each byte placed in the mantissa of
              // 2^23 (one byte permute) and 2^23 + 128 taken off: exactly the signed code, with
              // no int-to-float conversion (those issue at a quarter of the FMA rate)
              const uint32_t c01 = __funnelshift_r(w0, w1, sh) ^ 0x80808080u;
              const uint32_t c23 = __funnelshift_r(w1, w2, sh) ^ 0x80808080u;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                w[r][e] = d * (__uint_as_float(__byte_perm(c01, 0x4B000000u, 0x7650u | e)) - 8388736.0f);
                w[r][4 + e] = d * (__uint_as_float(__byte_perm(c23, 0x4B000000u, 0x7650u | e)) - 8388736.0f);
              }
            } else if constexpr (WD == MLA_Q4_AFFINE) {
              const uint32_t cw = *reinterpret_cast<const uint32_t*>(slot + r * 128 + lane * 4);
              const uint16_t* sb = reinterpret_cast<const uint16_t*>(slot + PJ_RW * 128);
              const float sc = bf16_bits_to_f32(sb[r * 4 + (lane >> 3)]);
              const float bi = bf16_bits_to_f32(sb[16 + r * 4 + (lane >> 3)]);
              // each code in the mantissa of 2^23 and 2^23 taken off (exact, no conversion)
#pragma unroll
              for (int e = 0; e < 8; ++e)
                w[r][e] = fmaf(sc, __uint_as_float(((cw >> (4 * e)) & 15u) | 0x4B000000u) - 8388608.0f, bi);
            } else if constexpr (WD == MLA_BF16) {
              const uint4 u = *reinterpret_cast<const uint4*>(slot + (r * 32 + lane) * LB);
              const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                w[r][2 * e] = __uint_as_float(ww[e] << 16);
                w[r][2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
              }
            } else {
              const float4 u0 = *reinterpret_cast<const float4*>(slot + (r * 32 + lane) * LB);
              const float4 u1 = *reinterpret_cast<const float4*>(slot + (r * 32 + lane) * LB + 16);
              w[r][0] = u0.x; w[r][1] = u0.y; w[r][2] = u0.z; w[r][3] = u0.w;
              w[r][4] = u1.x; w[r][5] = u1.y; w[r][6] = u1.z; w[r][7] = u1.w;
            }
          }
          const int sr = s + S * q;   // step within the round
#pragma unroll
          for (int j = 0; j < PJ_BP; ++j) {
            if (j < nb) {
              float xv[8];
              if (XBF) {
                const uint4 u = *reinterpret_cast<const uint4*>(xs + ((int64_t)j * XR::COLS + sr * PJ_STEP + lane * 8) * 2);
                const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  xv[2 * e] = __uint_as_float(ww[e] << 16);
                  xv[2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
                }
              } else {
                const float* base = reinterpret_cast<const float*>(xs) + (int64_t)j * XR::COLS + sr * PJ_STEP + lane * 4;
                const float4 u0 = *reinterpret_cast<const float4*>(base);
                const float4 u1 = *reinterpret_cast<const float4*>(base + 128);
                xv[0] = u0.x; xv[1] = u0.y; xv[2] = u0.z; xv[3] = u0.w;
                xv[4] = u1.x; xv[5] = u1.y; xv[6] = u1.z; xv[7] = u1.w;
              }
#pragma unroll
              for (int r = 0; r < PJ_RW; ++r)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[r * PJ_BP + j] = fmaf(w[r][e], xv[e], acc[r * PJ_BP + j]);
            }
          }
        }
        if constexpr (QUANT) __syncwarp();   // every lane is done with this slot before it is refilled
      }
      __syncthreads();   // every warp is done with this round's x
      if (t + 1 < nrounds) {
        x_store();
        __syncthreads();
        if (t + 2 < nrounds) x_load(b0, nb, t + 2);
      }
    }
    cp_async_wait<0>();
    red[warp][lane] = warp_sum32_scatter(acc, lane);
    __syncthreads();
    if (s == 0) {
      float v = 0.f;
      for (int t = 0; t < S; ++t) v += red[warp + t][lane];
      const int r = lane / PJ_BP, j = lane % PJ_BP;
      if (r0 + r < rows && j < nb) {
        const int64_t o = (int64_t)(b0 + j) * rows + r0 + r;
        if (ybf) {
          __nv_bfloat16 hv = __float2bfloat16_rn(v);
          static_cast<uint16_t*>(Y)[o] = *reinterpret_cast<uint16_t*>(&hv);
        } else {
          static_cast<float*>(Y)[o] = v;
        }
      }
    }
    __syncthreads();
  }
}

template <bool XBF>
constexpr int proj_smem_bytes() { return 2 * PJ_BP * PJ_ROUND * (XBF ? 2 : 4); }

// In place: x[b, :] = x[b, :] / sqrt(mean(x[b, :]^2) + eps) * w, one CTA per vector; the sum
// of squares is formed in a fixed order (thread partials, warp butterflies, then the 8 warp
// sums in warp order).
// With hi != nullptr the normalised values go out as bf16 hi and lo [B, K] instead (x unchanged).
__global__ void __launch_bounds__(PJ_THREADS) rms_norm_rows_kernel(float* x, const float* w, int K, float eps,
                                                                   uint16_t* hi, uint16_t* lo) {
  __shared__ float part[PJ_WARPS];
  pdl_trigger();
  pdl_wait();
  float* xb = x + (int64_t)blockIdx.x * K;
  float ss = 0.f;
  for (int k = threadIdx.x; k < K; k += PJ_THREADS) ss = fmaf(xb[k], xb[k], ss);
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < PJ_WARPS; ++i) tot += part[i];
  const float inv = rsqrtf(tot / (float)K + eps);
  for (int k = threadIdx.x; k < K; k += PJ_THREADS) {
    const float v = xb[k] * inv * w[k];
    if (hi == nullptr) {
      xb[k] = v;
    } else {
      const int64_t o = (int64_t)blockIdx.x * K + k;
      const uint16_t h = pt_bf16_bits(v);
      hi[o] = h;
      lo[o] = pt_bf16_bits(v - bf16_bits_to_f32(h));
    }
  }
}

// bf16 / float32 weights always take the ring; quantised ones when their steps are whole
constexpr bool proj_uses_ring(int wd, int K) {
  return wd == MLA_BF16 || wd == MLA_F32 || ((wd == MLA_Q8_0 || wd == MLA_Q4_AFFINE) && K % 256 == 0);
}

template <int WD, bool XBF>
cudaError_t launch_proj_x(const ProjArgs& a, int64_t blocks, cudaStream_t st) {
  if (proj_uses_ring(WD, a.K)) {
    constexpr int bytes = ring_smem_bytes<WD, XBF>();
    const cudaError_t e = ensure_smem(reinterpret_cast<const void*>(proj_gemv_ring_kernel<WD, XBF>), bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(proj_gemv_ring_kernel<WD, XBF>, dim3((unsigned)blocks), dim3(PJ_THREADS), bytes, st, a);
  } else {
    const cudaError_t e = ensure_smem(reinterpret_cast<const void*>(proj_gemv_kernel<WD, XBF>), proj_smem_bytes<XBF>());
    if (e != cudaSuccess) return e;
    return launch_pdl(proj_gemv_kernel<WD, XBF>, dim3((unsigned)blocks), dim3(PJ_THREADS), proj_smem_bytes<XBF>(), st, a);
  }
}

template <int WD>
cudaError_t launch_proj_dt(const ProjArgs& a, bool x_bf16, int64_t blocks, cudaStream_t st) {
  return x_bf16 ? launch_proj_x<WD, true>(a, blocks, st) : launch_proj_x<WD, false>(a, blocks, st);
}

// ---- bf16 weights, up to 128 sequences: tcgen05 ------------------------------------------------
// y[b, r] = sum_k W[r, k] x[b, k] as D[r, b] = W_tile . X^T on the tensor cores: a CTA owns 128 rows
// of W (the M = 128 operand, K-major, 64-column blocks by TMA in the 128-byte swizzle) and one
// slice of the columns (split-K); the batch is the N operand: the bf16 input rows, or, for a
// float32 input, its bf16 hi rows then its bf16 lo rows (x = hi + lo to about 2^-16), whose two
// accumulator halves the epilogue adds. A four-stage ring of (W block, X block) pairs feeds one
// MMA-issuing thread (two to four stages, as many as keep a CTA within half of the shared
// memory, so that two CTAs share an SM); the fp32 accumulator [128 rows x N] lives in tensor
// memory; four warps read it out. With one slice the result goes straight to y; otherwise each slice writes its
// partial sums and a second kernel adds the slices in order. Warp 0 issues the TMA loads, warp 1
// owns tensor memory and issues the MMAs, warps 2-5 (one per tensor-memory lane quarter) run
// the epilogue. Every wait is bounded; on a timeout the CTA records MLA_ERR_TIMEOUT, drains what
// it issued, frees tensor memory and writes NaN for the outputs it owns.
constexpr int PT_STAGES = 4;             // at most
constexpr int PT_SMEM_HALF = 110 * 1024; // stages of one CTA: two CTAs fit an SM
constexpr uint64_t G_DRAIN_NS = kWaitDrainNs;
constexpr int PT_THREADS = 192;
constexpr int PT_A_BYTES = 128 * 128;   // 128 rows x 64 bf16 columns

struct ProjTcArgs {
  int64_t tiles0;        // 128-row tiles of matrix 0; tiles past it belong to matrix 1
  int64_t rows[2];
  void* y[2];            // [B, rows]: float32, or bf16 where y_bf16
  int y_bf16[2];
  float* part;           // [splits][B][rows0 + rows1] float32 partial sums (splits > 1)
  int K, B;
  int NB;                // MMA N: the padded batch (bf16 input) or twice it (hi ; lo)
  int BP;                // padded batch: rows of one X half in shared memory
  int xsplit;            // 1: X is hi and lo (two maps), accumulator halves added
  int splits, kb_per_split, nkb;
  int stages;            // ring depth (2 to PT_STAGES)
  WsHeader* hdr;
  uint64_t wait_ns;
};

__global__ void __launch_bounds__(PT_THREADS, 1)
proj_tc_kernel(const __grid_constant__ CUtensorMap w0_map, const __grid_constant__ CUtensorMap w1_map,
               const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap xlo_map,
               const ProjTcArgs a) {
  extern __shared__ uint8_t pt_raw[];
  __shared__ uint64_t full[PT_STAGES], empty[PT_STAGES], mma_done;
  __shared__ uint32_t tmem_base;
  __shared__ int failed;
  uint8_t* dyn = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(pt_raw) + 1023) & ~uintptr_t(1023));
  const int b_bytes = a.NB * 128;
  const int stage_bytes = PT_A_BYTES + b_bytes;
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool second = blockIdx.x >= a.tiles0;
  const int64_t r0 = (second ? blockIdx.x - a.tiles0 : blockIdx.x) * 128;
  const int64_t rows = second ? a.rows[1] : a.rows[0];
  const CUtensorMap* wmap = second ? &w1_map : &w0_map;
  const int split = blockIdx.y;
  const int kb0 = split * a.kb_per_split, kb1 = min(a.nkb, kb0 + a.kb_per_split);
  const int nkb = kb1 - kb0;
  const uint32_t tcols = a.NB <= 64 ? 64 : (a.NB <= 128 ? 128 : 256);
  const int NS = a.stages;
  if (tid == 0) {
    failed = 0;
    for (int i = 0; i < NS; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
    }
    tc::mbar_init(&mma_done, 1);
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_base, tcols);
    tc::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(wmap);
    tc::tma_prefetch_desc(&x_map);
    if (a.xsplit) tc::tma_prefetch_desc(&xlo_map);
  }
  tc::tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      // the weights are no other kernel's output: the first blocks of W go out before the
      // dependency wait (their bytes expected without an arrival, so a stage completes only once
      // its input block, armed with the arrival below, has landed too), the input's after it
      const int pre = min(nkb, NS);
      for (int i = 0; i < pre; ++i) {
        tc::mbar_expect_tx(&full[i], PT_A_BYTES);
        tc::tma_load_2d(dyn + i * stage_bytes, wmap, 64 * (kb0 + i), (int32_t)r0, &full[i]);
      }
      pdl_wait();
      bool ok = true;
      int last = -1;
      for (int i = 0; i < nkb && ok; ++i) {
        const int st = i % NS;
        uint8_t* sa = dyn + st * stage_bytes;
        if (i >= NS) {
          if (!tc::mbar_wait(&empty[st], (uint32_t)(((i / NS) - 1) & 1), a.wait_ns)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&full[st], stage_bytes);
          tc::tma_load_2d(sa, wmap, 64 * (kb0 + i), (int32_t)r0, &full[st]);
        } else {
          tc::mbar_arrive_expect_tx(&full[st], stage_bytes - PT_A_BYTES);
        }
        tc::tma_load_2d(sa + PT_A_BYTES, &x_map, 64 * (kb0 + i), 0, &full[st]);
        if (a.xsplit) tc::tma_load_2d(sa + PT_A_BYTES + a.BP * 128, &xlo_map, 64 * (kb0 + i), 0, &full[st]);
        last = i;
      }
      if (!ok && atomicExch(&failed, 1) == 0) set_error(a.hdr, MLA_ERR_TIMEOUT, 0);
      // the loads issued must land before the CTA leaves: wait for the stages of the last ones
      // (every prefetched weight block has its input block issued: no wait precedes those)
      for (int i = max(0, last - NS + 1); i <= last; ++i)
        tc::mbar_wait(&full[i % NS], (uint32_t)((i / NS) & 1), G_DRAIN_NS);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, a.NB, 0, 0);
      bool ok = true;
      for (int i = 0; i < nkb; ++i) {
        const int st = i % NS;
        if (!tc::mbar_wait(&full[st], (uint32_t)((i / NS) & 1), a.wait_ns) ||
            *reinterpret_cast<volatile int*>(&failed)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t sa = tc::smem_u32(dyn + st * stage_bytes);
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_f16_ss(tmem, tc::sdesc_sw128(sa + kk * 32, 16, 1024),
                         tc::sdesc_sw128(sa + PT_A_BYTES + kk * 32, 16, 1024), idesc, (i | kk) != 0);
        tc::mma_commit(&empty[st]);
      }
      if (!ok && atomicExch(&failed, 1) == 0) set_error(a.hdr, MLA_ERR_TIMEOUT, 0);
      tc::mma_commit(&mma_done);   // arrives once every MMA issued has completed
    }
  } else {
    // ======================= epilogue: warps 2-5, lane quarter warp % 4 =======================
    const int q = warp & 3;
    const int64_t r = r0 + 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&mma_done, 0, a.wait_ns + G_DRAIN_NS));
    ok = ok && !*reinterpret_cast<volatile int*>(&failed);
    ok = __all_sync(0xffffffffu, ok);
    tc::tc_fence_after();
    const int nout = a.xsplit ? a.BP : a.NB;
    const int y_col = (int)(second ? a.rows[0] : 0);
    const int64_t rows_all = a.rows[0] + a.rows[1];
    for (int c0 = 0; c0 < nout; c0 += 32) {
      uint32_t v[32], w[32];
      if (ok) {
        tc::tmem_ld32(tmem + lane_base + c0, v);
        if (a.xsplit) tc::tmem_ld32(tmem + lane_base + a.BP + c0, w);
        tc::tmem_wait_ld();
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int b = c0 + j;
        if (b >= a.B || r >= rows) continue;
        float val = CUDART_NAN_F;
        if (ok) val = __uint_as_float(v[j]) + (a.xsplit ? __uint_as_float(w[j]) : 0.f);
        if (a.splits > 1) {
          a.part[((int64_t)split * a.B + b) * rows_all + y_col + r] = val;
        } else {
          void* Y = second ? a.y[1] : a.y[0];
          const bool ybf = second ? a.y_bf16[1] != 0 : a.y_bf16[0] != 0;
          if (ybf) static_cast<uint16_t*>(Y)[(int64_t)b * rows + r] = pt_bf16_bits(val);
          else static_cast<float*>(Y)[(int64_t)b * rows + r] = val;
        }
      }
    }
  }
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, tcols);
  }
}

// y[b, r] = sum over the slices, in slice order (one thread per output)
__global__ void __launch_bounds__(256) proj_reduce_kernel(const float* __restrict__ part, int splits, int B,
                                                          int64_t rows0, int64_t rows1, void* y0, int y0_bf16,
                                                          void* y1, int y1_bf16) {
  pdl_trigger();
  pdl_wait();
  const int64_t rows_all = rows0 + rows1;
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (i >= (int64_t)B * rows_all) return;
  const int64_t b = i / rows_all, c = i % rows_all;
  float v = 0.f;
  for (int s = 0; s < splits; ++s) v += part[((int64_t)s * B + b) * rows_all + c];
  const bool second = c >= rows0;
  const int64_t r = second ? c - rows0 : c, rows = second ? rows1 : rows0;
  void* Y = second ? y1 : y0;
  if (second ? y1_bf16 : y0_bf16) static_cast<uint16_t*>(Y)[b * rows + r] = pt_bf16_bits(v);
  else static_cast<float*>(Y)[b * rows + r] = v;
}

// x [B, K] float32 -> bf16 hi = rn(x) and lo = rn(x - hi), each [B, K] (x = hi + lo to ~2^-16)
__global__ void __launch_bounds__(256) split_hi_lo_kernel(const float* __restrict__ x, int64_t n,
                                                          uint16_t* __restrict__ hi, uint16_t* __restrict__ lo) {
  pdl_trigger();
  pdl_wait();
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (i >= n) return;
  const float v = x[i];
  const uint16_t h = pt_bf16_bits(v);
  hi[i] = h;
  lo[i] = pt_bf16_bits(v - bf16_bits_to_f32(h));
}

}  // namespace

cudaError_t launch_proj(const void* x, bool x_bf16, int K, int B, int w_dtype, const void* w0, int64_t rows0,
                        void* y0, bool y0_bf16, const void* w1, int64_t rows1, void* y1, bool y1_bf16,
                        cudaStream_t st) {
  ProjArgs a;
  a.w[0] = w0; a.rows[0] = rows0; a.y[0] = y0; a.y_bf16[0] = y0_bf16 ? 1 : 0;
  a.w[1] = w1; a.rows[1] = w1 != nullptr ? rows1 : 0; a.y[1] = y1; a.y_bf16[1] = y1_bf16 ? 1 : 0;
  a.x = x;
  a.K = K;
  a.B = B;
  // Split the columns among more warps (at most the steps of a round: 4, or 2 for float32 x on
  // the ring kernel) only while the grid stays under two CTAs per SM.
  const int64_t target = 2 * (int64_t)device_sms();
  const int s_max = (!x_bf16 && proj_uses_ring(w_dtype, K)) ? 2 : 4;
  int S = 1;
  while (S < s_max) {
    const int64_t rows_per_cta = (int64_t)(PJ_WARPS / S) * PJ_RW;
    if ((a.rows[0] + rows_per_cta - 1) / rows_per_cta + (a.rows[1] + rows_per_cta - 1) / rows_per_cta >= target)
      break;
    S *= 2;
  }
  a.ksplit = S;
  const int64_t rows_per_cta = (int64_t)(PJ_WARPS / S) * PJ_RW;
  a.ctas0 = (a.rows[0] + rows_per_cta - 1) / rows_per_cta;
  const int64_t blocks = a.ctas0 + (a.rows[1] + rows_per_cta - 1) / rows_per_cta;
  if (blocks < 1 || blocks >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  switch (w_dtype) {
    case MLA_F32: return launch_proj_dt<MLA_F32>(a, x_bf16, blocks, st);
    case MLA_BF16: return launch_proj_dt<MLA_BF16>(a, x_bf16, blocks, st);
    case MLA_Q8_0: return launch_proj_dt<MLA_Q8_0>(a, x_bf16, blocks, st);
    case MLA_Q4_AFFINE: return launch_proj_dt<MLA_Q4_AFFINE>(a, x_bf16, blocks, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rms_norm_rows(float* x, const float* w, int K, int B, float eps, cudaStream_t st,
                                 uint16_t* hi, uint16_t* lo) {
  return launch_pdl(rms_norm_rows_kernel, dim3((unsigned)B), dim3(PJ_THREADS), 0, st, x, w, K, eps, hi, lo);
}


ProjTcPlan proj_tc_plan(int64_t rows0, int64_t rows1, int K, int B, bool x_f32, int w_dtype) {
  ProjTcPlan p = ProjTcPlan{};
  // Under 16 sequences only a large matrix pays for the extra launches (the input's halves, the
  // slice reduction) and the fill of the ring: at 4 sequences a 235 MB matrix streams 1.4x faster
  // than on the CUDA cores, a 30 MB one no faster.
  const int64_t w_bytes = (rows0 + rows1) * (int64_t)K * 2;
  p.use = w_dtype == MLA_BF16 && (B >= 16 || w_bytes >= (int64_t(64) << 20)) && B <= (x_f32 ? 128 : 256) &&
          K >= 64 && K % 8 == 0 && rows0 + rows1 > 0 && rows0 + rows1 < (int64_t(1) << 31);
  if (!p.use) return p;
  p.xsplit = x_f32 ? 1 : 0;
  p.BP = x_f32 ? ((B + 7) / 8) * 8 : ((B + 15) / 16) * 16;
  p.NB = x_f32 ? 2 * p.BP : p.BP;
  p.tiles0 = (rows0 + 127) / 128;
  p.tiles1 = (rows1 + 127) / 128;
  p.nkb = (K + 63) / 64;
  const int stage_bytes = PT_A_BYTES + p.NB * 128;
  p.stages = PT_SMEM_HALF / stage_bytes;
  if (p.stages > PT_STAGES) p.stages = PT_STAGES;
  if (p.stages < 2) p.stages = 2;
  const int64_t tiles = p.tiles0 + p.tiles1;
  int sms = device_sms();
  if (sms <= 0) sms = 152;
  // Column slices: the CTAs are spread evenly over the SMs, each streams its slice's 64-column
  // blocks plus a pipeline fill of about eight blocks; more than one slice adds the partial sums'
  // round trip (8 bytes per output and slice, counted in 16 KB weight blocks per SM). Pick the
  // count that minimises the busiest SM's load (the fewest slices among equals), each slice at
  // least four blocks.
  int64_t best = -1, best_cost = 0;
  for (int64_t sp = 1; sp <= (p.nkb >= 8 ? p.nkb / 4 : 1); ++sp) {
    const int64_t kb = (p.nkb + sp - 1) / sp;
    const int64_t part_blocks = sp > 1 ? (sp * (int64_t)B * (rows0 + rows1) * 8) / (PT_A_BYTES * (int64_t)sms) : 0;
    const int64_t cost = ((tiles * sp + sms - 1) / sms) * (kb + 8) + part_blocks;
    if (best < 0 || cost < best_cost) {
      best = sp;
      best_cost = cost;
    }
  }
  p.kb_per_split = (int)((p.nkb + best - 1) / best);
  p.splits = (p.nkb + p.kb_per_split - 1) / p.kb_per_split;
  p.part_floats = p.splits > 1 ? (int64_t)p.splits * B * (rows0 + rows1) : 0;
  return p;
}

cudaError_t launch_proj_tc(const ProjTcPlan& p, const void* x, const void* x_lo, int K, int B, const void* w0,
                           int64_t rows0, void* y0, bool y0_bf16, const void* w1, int64_t rows1, void* y1,
                           bool y1_bf16, float* part, WsHeader* hdr, cudaStream_t st) {
  if (!p.use || (p.splits > 1 && part == nullptr) || (p.xsplit && x_lo == nullptr)) return cudaErrorInvalidValue;
  if (w1 == nullptr) rows1 = 0;
  CUtensorMap w0m, w1m, xm, xlm;
  if (!make_map_2d_bf16(&w0m, w0, (uint64_t)K, (uint64_t)rows0, 64, 128)) return cudaErrorInvalidValue;
  if (rows1 > 0) {
    if (!make_map_2d_bf16(&w1m, w1, (uint64_t)K, (uint64_t)rows1, 64, 128)) return cudaErrorInvalidValue;
  } else {
    w1m = w0m;
  }
  const uint32_t xbox = (uint32_t)(p.xsplit ? p.BP : p.NB);
  if (!make_map_2d_bf16(&xm, x, (uint64_t)K, (uint64_t)B, 64, xbox)) return cudaErrorInvalidValue;
  if (p.xsplit) {
    if (!make_map_2d_bf16(&xlm, x_lo, (uint64_t)K, (uint64_t)B, 64, xbox)) return cudaErrorInvalidValue;
  } else {
    xlm = xm;
  }
  ProjTcArgs a;
  a.tiles0 = p.tiles0;
  a.rows[0] = rows0;
  a.rows[1] = rows1;
  a.y[0] = y0;
  a.y[1] = y1;
  a.y_bf16[0] = y0_bf16 ? 1 : 0;
  a.y_bf16[1] = y1_bf16 ? 1 : 0;
  a.part = part;
  a.K = K;
  a.B = B;
  a.NB = p.NB;
  a.BP = p.BP;
  a.xsplit = p.xsplit;
  a.splits = p.splits;
  a.kb_per_split = p.kb_per_split;
  a.nkb = p.nkb;
  a.stages = p.stages;
  a.hdr = hdr;
  a.wait_ns = wait_limit_ns();
  const int smem = p.stages * (PT_A_BYTES + p.NB * 128) + 1024;
  cudaError_t e = ensure_smem(reinterpret_cast<const void*>(proj_tc_kernel), smem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = p.tiles0 + (rows1 > 0 ? p.tiles1 : 0);
  e = launch_pdl(proj_tc_kernel, dim3((unsigned)tiles, (unsigned)p.splits), dim3(PT_THREADS), (size_t)smem, st, w0m,
                 w1m, xm, xlm, a);
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t n = (int64_t)B * (rows0 + rows1);
  return launch_pdl(proj_reduce_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, (const float*)part,
                    p.splits, B, rows0, rows1, y0, y0_bf16 ? 1 : 0, y1, y1_bf16 ? 1 : 0);
}

cudaError_t launch_split_hi_lo(const float* x, int64_t n, uint16_t* hi, uint16_t* lo, cudaStream_t st) {
  return launch_pdl(split_hi_lo_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, x, n, hi, lo);
}

}  // namespace mla
