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

namespace mla {

namespace {

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
template <int WD> struct Ring;
template <> struct Ring<MLA_BF16> { static constexpr int D = 4, LB = 16; };
template <> struct Ring<MLA_F32> { static constexpr int D = 2, LB = 32; };

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
  return XRound<XBF>::BYTES + PJ_WARPS * Ring<WD>::D * PJ_RW * 32 * Ring<WD>::LB;
}

template <int WD, bool XBF>
__global__ void __launch_bounds__(PJ_THREADS, 2) proj_gemv_ring_kernel(const __grid_constant__ ProjArgs a) {
  using XR = XRound<XBF>;
  constexpr int D = Ring<WD>::D, LB = Ring<WD>::LB, EW = WD == MLA_BF16 ? 2 : 4;
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ float red[PJ_WARPS][32];
  uint8_t* xs = sm;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* ring = sm + XR::BYTES + warp * (D * PJ_RW * 32 * LB);
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
    wrow[r] = W + (row_ok[r] ? (r0 + r) * (int64_t)K * EW : 0) + lane * 8 * EW;
  }
  auto step_col = [&](int n) {
    return (n >> lg_spr) * XR::COLS + ((s + ((n & (spr - 1)) << lg_s)) * PJ_STEP) + lane * 8;
  };
  // step n's weights into ring slot n % D (rows or columns outside the matrix are not copied:
  // their slot bytes are never used for a stored result); always closes one commit group
  auto issue = [&](int n) {
    if (n < nsteps) {
      const int k = step_col(n);
      if (k < K) {
        uint8_t* slot = ring + (n % D) * (PJ_RW * 32 * LB) + lane * LB;
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
        const int k = step_col(n);
        if (k < K) {
          const uint8_t* slot = ring + (n % D) * (PJ_RW * 32 * LB);
          float w[PJ_RW][8];
#pragma unroll
          for (int r = 0; r < PJ_RW; ++r) {
            if (WD == MLA_BF16) {
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
__global__ void __launch_bounds__(PJ_THREADS) rms_norm_rows_kernel(float* x, const float* w, int K, float eps) {
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
  for (int k = threadIdx.x; k < K; k += PJ_THREADS) xb[k] = xb[k] * inv * w[k];
}

template <int WD, bool XBF>
cudaError_t launch_proj_x(const ProjArgs& a, int64_t blocks, cudaStream_t st) {
  if constexpr (WD == MLA_BF16 || WD == MLA_F32) {
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
  // Split the columns among more warps (at most the steps of a round: 4, or 2 for float32 x
  // under bf16 / float32 weights) only while the grid stays under two CTAs per SM.
  const int64_t target = 2 * (int64_t)device_sms();
  const int s_max = (!x_bf16 && (w_dtype == MLA_BF16 || w_dtype == MLA_F32)) ? 2 : 4;
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

cudaError_t launch_rms_norm_rows(float* x, const float* w, int K, int B, float eps, cudaStream_t st) {
  return launch_pdl(rms_norm_rows_kernel, dim3((unsigned)B), dim3(PJ_THREADS), 0, st, x, w, K, eps);
}

}  // namespace mla
