// One-launch decode for tiny batches: absorb, split attention and LSE-merge combine with the
// W_UV up-projection in a single grid, phases separated by grid-wide barriers, all in float32
// on the CUDA cores.
//
// moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs, folded SDPA chain (q_prime from the
// nope rows of kv_b, SDPA over the compressed rows, out_per_head through the v rows of kv_b);
// turbospark-runtime 0.3.0, src/families/deepseek2/attn.rs, absorb -> MQA attention over the
// compressed rows [kv_lat ; k_pe] -> v-combine.
//
// For a handful of query rows (B x H <= 64, H <= 32) the staged path is four dependent kernels whose
// boundaries and set-up cost more than their work. Here the grid (one CTA per SM at most) runs:
//   1. absorb: q'[b,h,c] = sum_n q_nope[b,h,n] W_UK,h[n,c] in float32, 64 latent columns per
//      item, and the RoPE of q_pe; W_UK is read into registers before the dependency wait, and
//      the rows of the CTA's first chunk are already on their way (bulk copies).
//   2. attention: each sequence is cut into 32-row chunks (boundaries fixed by the sequence's
//      own length, so a sequence's result does not depend on the rest of the batch); a CTA
//      takes chunks g, g + G, ... and writes, per chunk and head, the chunk's maximum, sum and
//      unnormalised output row. A warp serves heads w, w + 8, ...; lanes own 16-byte column
//      pieces of the rows, the scores of 8 rows come together in a transpose-reduce, and the
//      products run as packed float pairs.
//   3. merge and W_UV: per (sequence, head, 64 latent columns) the chunks' partials in chunk
//      order, and that slice's share of out = W_UV o (W_UV read before the dependency wait);
//      the last slice of a head to finish adds the shares in slice order and writes out, lse.
// The two barriers count arrivals in the workspace header (zero before a call; the last CTA
// out resets them). Every wait is bounded: a CTA whose wait runs out records MLA_ERR_TIMEOUT
// and writes NaN for the outputs it owns.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int SM_THREADS = 256;
constexpr int SM_WARPS = SM_THREADS / 32;
constexpr int SM_CHUNK = 32;            // rows per attention chunk (one per lane)
constexpr int SM_MAX_HPW = 4;           // heads per warp at most (H <= 32)
constexpr int SM_MAX_CHUNKS = 256;     // 32-row chunks of a sequence at most (capacity <= 8192)
constexpr int SM_MAX_CPL = 16;          // latent columns per lane at most (two 8-column pieces: C <= 512)

struct SmallArgs {
  const uint16_t* q;        // [B][H][N + R] bf16
  const uint16_t* kv_b;     // [H][N + V][C] bf16
  const uint16_t* rows;     // cache rows [n_phys][C + R] bf16
  RowMap map;
  const int32_t* seq_lens;
  const int32_t* positions; // or nullptr
  const double* inv_freq;
  float* out;               // [B][H][V]
  float* lse;               // [B][H] or nullptr
  float* qf;                // [B][H][C + R] float32 fused queries
  float* wshare;            // [B][H][C / 64][V]: each latent slice's share of out
  unsigned int* head_cnt;   // [B * H] finished slices per head (zeroed in phase 1)
  float* part;              // [B][max_chunks][H][C + 4]: output row, max (log2 units), sum, 2 zeros
                            // (rows of C + 4 floats keep every float4 access 16-byte aligned)
  WsHeader* hdr;
  int B, H, C, R, N, V, max_chunks;
  float scale_log2;
  uint64_t wait_ns;
};

// Arrival counters of the two barriers and of the exit, in the header's spare words.
__device__ __forceinline__ unsigned int* sm_counter(WsHeader* hdr, int i) {
  return reinterpret_cast<unsigned int*>(&hdr->pad[8 + i]);
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of the G CTAs in two halves: every thread's writes before grid_arrive are
// visible to every thread after the matching grid_wait; work in between overlaps the wait.
__device__ __forceinline__ void grid_arrive(unsigned int* ctr) {
  __syncthreads();
  // release: the CTA's writes (ordered before this thread by the block barrier) become visible
  // to every CTA that acquires the count
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
}
// False (for the whole CTA) when the wait ran out.
__device__ bool grid_wait(unsigned int* ctr, unsigned int G, uint64_t limit_ns, int* flag_s) {
  if (threadIdx.x == 0) {
    const uint64_t t0 = tc::global_ns();
    int ok = 1;
    while (ld_acquire_gpu(ctr) < G) {
      if (tc::global_ns() - t0 > limit_ns) {
        ok = 0;
        break;
      }
    }
    *flag_s = ok;
  }
  __syncthreads();
  return *flag_s != 0;
}
__device__ __forceinline__ bool grid_barrier(unsigned int* ctr, unsigned int G, uint64_t limit_ns, int* flag_s) {
  grid_arrive(ctr);
  return grid_wait(ctr, G, limit_ns, flag_s);
}

__device__ __forceinline__ float bf16f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Warp-level bf16 tensor-core steps (m16n8k16, float32 accumulate) and the shared-memory
// fragment loads that feed them (four 8x8 bf16 matrices; lane l gives the row address of
// matrix l / 8).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t r[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}
__device__ __forceinline__ void mma_bf16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
               "{%0, %1, %2, %3};"
               : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi): the pair carries 16 significant bits.
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16* hi, __nv_bfloat16* lo) {
  *hi = __float2bfloat16_rn(x);
  *lo = __float2bfloat16_rn(x - __bfloat162float(*hi));
}

// Global -> shared bulk copy completing on an mbarrier of this CTA (both addresses and the size
// multiples of 16 bytes).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

// Chunks of a sequence of length L (0 when the length is out of range).
__device__ __forceinline__ int seq_chunks(const SmallArgs& a, int L) {
  if (L < 1 || L > a.map.capacity()) return 0;
  return (L + SM_CHUNK - 1) / SM_CHUNK;
}

// Warp 0: the rows of chunk k into rows_s ([32][C + R] bf16). Lane r maps row r of the chunk;
// each run of consecutive physical rows goes in one bulk copy (a contiguous cache or a page
// gives one copy per chunk), all completing on `bar`. *bad_s says whether a row lay outside
// the pool (not copied).
__device__ __forceinline__ void issue_chunk_rows(const SmallArgs& a, const int* cfirst, const int* len, int k,
                                                 uint8_t* rows_s, uint64_t* bar, int* bad_s) {
  const int lane = threadIdx.x & 31;
  int b = 0;
  while (b + 1 < a.B && cfirst[b + 1] <= k) ++b;
  const int t0 = (k - cfirst[b]) * SM_CHUNK;
  const int nr = min(SM_CHUNK, len[b] - t0);
  const int64_t pr = lane < nr ? a.map.phys(b, (int64_t)t0 + lane) : -1;
  const int64_t prev = __shfl_up_sync(0xffffffffu, pr, 1);
  const bool good = pr >= 0;
  const bool start = good && (lane == 0 || prev < 0 || prev + 1 != pr);
  const unsigned int goodm = __ballot_sync(0xffffffffu, good), startm = __ballot_sync(0xffffffffu, start);
  const unsigned int want = nr >= 32 ? 0xffffffffu : ((1u << nr) - 1u);
  const uint32_t bytes = (uint32_t)(a.C + a.R) * 2u;
  if (lane == 0) {
    *bad_s = goodm != want;
    tc::mbar_arrive_expect_tx(bar, (uint32_t)__popc(goodm) * bytes);
  }
  __syncwarp();
  if (start) {   // the run ends at the next start or at the first row without a physical row
    const unsigned int above = lane == 31 ? 0u : (0xffffffffu << (lane + 1));
    const unsigned int stops = (startm | ~goodm) & above;
    const int end = stops ? __ffs(stops) - 1 : 32;
    bulk_g2s(rows_s + (size_t)lane * bytes, a.rows + pr * (a.C + a.R), (uint32_t)(end - lane) * bytes, bar);
  }
}

// The landed rows of a chunk (raw [32][C + R]) into the padded tile (row pitch C + R + 8, so
// the eight row addresses of a fragment load fall in distinct banks); rows at or past nr are
// zero, so they add nothing to P V.
__device__ __forceinline__ void relayout_rows(const uint8_t* raw, uint8_t* tile, int CR, int nr) {
  const int pieces = CR / 8;
  for (int i = threadIdx.x; i < SM_CHUNK * pieces; i += SM_THREADS) {
    const int r = i / pieces, pc = i - r * pieces;
    const uint4 v = r < nr ? *reinterpret_cast<const uint4*>(raw + (size_t)(r * CR + pc * 8) * 2) : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(tile + (size_t)(r * (CR + 8) + pc * 8) * 2) = v;
  }
}

// rows of chunk k of the batch (k < the chunk total), its sequence and index in the sequence
__device__ __forceinline__ int chunk_rows(int B, const int* cfirst, const int* len, int k, int* b_out, int* j_out) {
  int b = 0;
  while (b + 1 < B && cfirst[b + 1] <= k) ++b;
  *b_out = b;
  *j_out = k - cfirst[b];
  return min(SM_CHUNK, len[b] - (k - cfirst[b]) * SM_CHUNK);
}

template <int HPW>   // heads per warp: ceil(H / 8)
__global__ void __launch_bounds__(SM_THREADS, 1) decode_small_kernel(const __grid_constant__ SmallArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];   // chunk rows (raw and padded), queries, scores, P
  __shared__ float w_s[SM_MAX_CHUNKS];               // merge: chunk weights
  __shared__ float ol_s[64];                         //        merged latent slice
  __shared__ int flag_s;
  __shared__ int cfirst_s[65];          // chunk prefix over the sequences (B <= 64)
  __shared__ int len_s[64];             // their lengths
  __shared__ float red_s[4][64];
  __shared__ float wred_s[SM_WARPS];
  __shared__ uint64_t rows_bar;
  __shared__ int rows_bad_s;
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned int G = gridDim.x;
  const int g = blockIdx.x;
  const int B = a.B, H = a.H, C = a.C, R = a.R, N = a.N, V = a.V;
  const int CR = C + R, NV = N + V;
  constexpr int MT = HPW > 2 ? 2 : 1;   // 16-head tiles of the tensor-core steps
  constexpr int HM = 16 * MT;
  const int CRP = CR + 8;               // padded row pitch (elements) of the tile, queries
  uint8_t* rows_s = smem;                                                        // raw [32][CR]
  __nv_bfloat16* tile_s = reinterpret_cast<__nv_bfloat16*>(smem + SM_CHUNK * CR * 2);   // [32][CRP]
  __nv_bfloat16* q_s = tile_s + SM_CHUNK * CRP;                                  // [2][HM][CRP] hi, lo
  float* sc_s = reinterpret_cast<float*>(q_s + 2 * HM * CRP);                    // [8][HM][32] column parts
  __nv_bfloat16* p_s = reinterpret_cast<__nv_bfloat16*>(sc_s + SM_WARPS * HM * SM_CHUNK);  // [2][HM][40]
  constexpr int PP = SM_CHUNK + 8;      // P row pitch
  bool ok = true;

  // ---- before the dependency wait: chunk layout and weights (no earlier kernel writes them) ----
  if (tid == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      const int L = a.seq_lens[b];
      len_s[b] = L;
      cfirst_s[b] = acc;
      acc += seq_chunks(a, L);
    }
    cfirst_s[B] = acc;
    tc::mbar_init(&rows_bar, 1);
    tc::fence_mbar_init();
  }
  for (int i = tid; i < (HM - H) * CRP; i += SM_THREADS) {   // padding heads: zero queries and P
    q_s[H * CRP + i] = __float2bfloat16_rn(0.f);
    q_s[(HM + H) * CRP + i] = __float2bfloat16_rn(0.f);
  }
  for (int i = tid; i < (HM - H) * PP; i += SM_THREADS) {
    p_s[H * PP + i] = __float2bfloat16_rn(0.f);
    p_s[(HM + H) * PP + i] = __float2bfloat16_rn(0.f);
  }
  const int n_items1 = B * H * (C / 64);   // absorb and merge items: (sequence, head, 64 latent columns)
  // the first absorb item's W_UK slice: column cc * 64 + (tid & 63), nope rows of quarter tid >> 6
  const int nq = N / 4;
  float wuk[32];
  if (g < n_items1) {
    const int h = (g / (C / 64)) % H, cc = g % (C / 64);
    const int c = cc * 64 + (tid & 63), n0 = (tid >> 6) * nq;
#pragma unroll
    for (int i = 0; i < 32; ++i)
      wuk[i] = i < nq ? bf16f(a.kv_b[((int64_t)h * NV + n0 + i) * C + c]) : 0.f;
  }
  // the first merge item's W_UV slice: row tid >> 1, latent columns cc * 64 + (tid & 1) * 32 .. + 31
  uint32_t wuv[16];
  if (g < n_items1) {
    const int h = (g / (C / 64)) % H, cc = g % (C / 64), v = tid >> 1;
    const uint4* src = reinterpret_cast<const uint4*>(a.kv_b + ((int64_t)h * NV + N + v) * C + cc * 64 + (tid & 1) * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 u = v < V ? src[i] : make_uint4(0, 0, 0, 0);
      wuv[4 * i] = u.x; wuv[4 * i + 1] = u.y; wuv[4 * i + 2] = u.z; wuv[4 * i + 3] = u.w;
    }
  }
  // the RoPE frequencies as float pairs (inputs, read before the wait)
  __shared__ float f_hi[32], f_lo[32];   // R <= 64
  if (a.positions != nullptr && tid < R / 2) rope_freq_split(a.inv_freq, tid, &f_hi[tid], &f_lo[tid]);
  pdl_wait();   // q and the appended cache row come from earlier kernels; the workspace and out
                // may still be read by them
  __syncthreads();
  const int total_chunks = cfirst_s[B];
  // the rows of this CTA's first chunk land while the absorb runs
  uint32_t rows_par = 0;
  bool rows_pending = g < total_chunks;
  if (rows_pending && warp == 0) issue_chunk_rows(a, cfirst_s, len_s, g, rows_s, &rows_bar, &rows_bad_s);
  if (g == 0) {   // lengths out of range: that sequence's outputs come out NaN (no chunks)
    for (int b = tid; b < B; b += SM_THREADS)
      if (cfirst_s[b + 1] == cfirst_s[b]) set_error(a.hdr, MLA_ERR_BAD_SEQ_LEN, b);
    for (int i = tid; i < B * H; i += SM_THREADS) a.head_cnt[i] = 0u;   // used after two barriers
  }

  // ================================ 1. absorb ================================
  for (int it = g; it < n_items1; it += G) {
    const int b = it / (H * (C / 64)), h = (it / (C / 64)) % H, cc = it % (C / 64);
    const int c = cc * 64 + (tid & 63), n0 = (tid >> 6) * nq;
    const uint16_t* qn = a.q + ((int64_t)b * H + h) * (N + R);
    float acc = 0.f;
    if (it == g) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (i < nq) acc = fmaf(bf16f(qn[n0 + i]), wuk[i], acc);
    } else {
      for (int i = 0; i < nq; ++i) acc = fmaf(bf16f(qn[n0 + i]), bf16f(a.kv_b[((int64_t)h * NV + n0 + i) * C + c]), acc);
    }
    red_s[tid >> 6][tid & 63] = acc;
    __syncthreads();
    float* qf = a.qf + ((int64_t)b * H + h) * CR;
    if (tid < 64) qf[cc * 64 + tid] = ((red_s[0][tid] + red_s[1][tid]) + red_s[2][tid]) + red_s[3][tid];
    if (cc == 0 && tid >= 64 && tid < 64 + R / 2) {
      const int p = tid - 64;
      const float x0 = bf16f(qn[N + 2 * p]), x1 = bf16f(qn[N + 2 * p + 1]);
      if (a.positions != nullptr) {
        float cv, sv;
        rope_cs_split(a.inv_freq, f_hi[p], f_lo[p], p, a.positions[b], &cv, &sv);
        qf[C + 2 * p] = x0 * cv - x1 * sv;
        qf[C + 2 * p + 1] = x0 * sv + x1 * cv;
      } else {
        qf[C + 2 * p] = x0;
        qf[C + 2 * p + 1] = x1;
      }
    }
    __syncthreads();
  }
  grid_arrive(sm_counter(a.hdr, 0));
  // while the other CTAs finish their absorb: the first chunk's rows into the padded tile, and
  // the next chunk's copy issued into the raw buffer
  bool cur_bad = false;
  if (rows_pending) {
    const bool landed = tc::mbar_wait(&rows_bar, rows_par, a.wait_ns);
    if (__syncthreads_and(landed)) {
      rows_pending = false;
      rows_par ^= 1u;
      cur_bad = rows_bad_s != 0;
      int b0, j0;
      relayout_rows(rows_s, reinterpret_cast<uint8_t*>(tile_s), CR, chunk_rows(B, cfirst_s, len_s, g, &b0, &j0));
      __syncthreads();
      if (g + (int)G < total_chunks) {
        if (warp == 0) issue_chunk_rows(a, cfirst_s, len_s, g + (int)G, rows_s, &rows_bar, &rows_bad_s);
        rows_pending = true;
      }
    } else {
      ok = false;
    }
  }
  ok = grid_wait(sm_counter(a.hdr, 0), G, a.wait_ns, &flag_s) && ok;

  // ================================ 2. attention over 32-row chunks ================================
  // On the tensor cores, warp-level bf16 steps with float32 accumulation. The float32 queries
  // and probabilities each go in as two bf16 operands (hi + lo), the cache rows exactly.
  //   scores: S[h, r] = q'_h . row_r; warp w takes an eighth of the (C + R) / 16 column steps
  //           for all 32 rows; the eight parts meet in shared memory.
  //   softmax: warp w, heads w, w + 8, ...: lane r holds row r; max, probabilities, sum.
  //   output: O[h, c] = sum_r P[h, r] row_r[c]; warp w takes latent columns w C/8 .. + C/8.
  const uint32_t tile_a = tc::smem_u32(tile_s), q_a = tc::smem_u32(q_s), p_a = tc::smem_u32(p_s);
  const int grp = lane >> 2, tig = lane & 3;
  const int KS = CR / 16;
  int q_seq = -1;
  for (int k = g; ok && k < total_chunks; k += G) {
    int b, j;
    const int nr = chunk_rows(B, cfirst_s, len_s, k, &b, &j);
    float* part = a.part + ((int64_t)b * a.max_chunks + j) * H * (C + 4);
    if (k != g) {   // a later chunk: its copy was issued when the previous tile was made
      const bool landed = tc::mbar_wait(&rows_bar, rows_par, a.wait_ns);
      if (!__syncthreads_and(landed)) {
        ok = false;
        break;
      }
      rows_pending = false;
      rows_par ^= 1u;
      cur_bad = rows_bad_s != 0;
      relayout_rows(rows_s, reinterpret_cast<uint8_t*>(tile_s), CR, nr);
      __syncthreads();
      if (k + (int)G < total_chunks) {
        if (warp == 0) issue_chunk_rows(a, cfirst_s, len_s, k + (int)G, rows_s, &rows_bar, &rows_bad_s);
        rows_pending = true;
      }
    }
    if (b != q_seq) {   // this sequence's fused queries (written by other CTAs before the barrier)
      const float4* src = reinterpret_cast<const float4*>(a.qf + (int64_t)b * H * CR);
      const int n4 = CR / 4;
      for (int i = tid; i < H * n4; i += SM_THREADS) {
        const int h = i / n4, c4 = i - h * n4;
        const float4 v = __ldcg(src + i);
        __nv_bfloat16 hi[4], lo[4];
        split_bf16(v.x, &hi[0], &lo[0]);
        split_bf16(v.y, &hi[1], &lo[1]);
        split_bf16(v.z, &hi[2], &lo[2]);
        split_bf16(v.w, &hi[3], &lo[3]);
        *reinterpret_cast<uint2*>(q_s + h * CRP + 4 * c4) = *reinterpret_cast<const uint2*>(hi);
        *reinterpret_cast<uint2*>(q_s + (HM + h) * CRP + 4 * c4) = *reinterpret_cast<const uint2*>(lo);
      }
      q_seq = b;
    }
    __syncthreads();
    if (cur_bad) {   // a row outside the pool: the merge of the sequence's heads comes out NaN
      if (tid == 0) set_error(a.hdr, MLA_ERR_BAD_PAGE, b);
      for (int i = tid; i < H; i += SM_THREADS) {
        part[(int64_t)i * (C + 4) + C] = 0.f;
        part[(int64_t)i * (C + 4) + C + 1] = CUDART_NAN_F;
      }
    } else {
      // ---- scores: warp w takes column steps w KS/8 .. (w+1) KS/8 - 1 of all 32 rows ----
      {
        const int ks0 = warp * KS / SM_WARPS, ks1 = (warp + 1) * KS / SM_WARPS;
        float acc[2][4][MT][4];   // [hi, lo][8-row tile][head tile]
#pragma unroll
        for (int x = 0; x < 2; ++x)
#pragma unroll
          for (int y = 0; y < 4; ++y)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[x][y][mt][e] = 0.f;
        // B (two tiles per load): rows 8 (2 i + lane / 16) + (lane & 7), columns ks*16 + 8 (lane / 8 & 1);
        // A: head row (lane & 7) + 8 (lane / 8 & 1), columns ks*16 + 8 (lane / 16)
        const uint32_t b_lane = tile_a + (uint32_t)((((lane >> 4) * 8 + (lane & 7)) * CRP + 8 * ((lane >> 3) & 1)) * 2);
        const uint32_t a_lane = q_a + (uint32_t)((((lane & 7) + 8 * ((lane >> 3) & 1)) * CRP + 8 * (lane >> 4)) * 2);
        for (int ks = ks0; ks < ks1; ++ks) {
          uint32_t bf[2][4];
          ldsm_x4(b_lane + ks * 32, bf[0]);                              // row tiles 0, 1
          ldsm_x4(b_lane + (uint32_t)(16 * CRP * 2) + ks * 32, bf[1]);   // row tiles 2, 3
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            uint32_t ah[4], al[4];
            ldsm_x4(a_lane + (uint32_t)((mt * 16 * CRP + ks * 16) * 2), ah);
            ldsm_x4(a_lane + (uint32_t)(((HM + mt * 16) * CRP + ks * 16) * 2), al);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
              const uint32_t b0 = bf[nt >> 1][2 * (nt & 1)], b1 = bf[nt >> 1][2 * (nt & 1) + 1];
              mma_bf16(acc[0][nt][mt], ah, b0, b1);
              mma_bf16(acc[1][nt][mt], al, b0, b1);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            float* s0 = sc_s + (warp * HM + mt * 16 + grp) * SM_CHUNK + nt * 8 + 2 * tig;
            *reinterpret_cast<float2*>(s0) =
                make_float2(acc[0][nt][mt][0] + acc[1][nt][mt][0], acc[0][nt][mt][1] + acc[1][nt][mt][1]);
            *reinterpret_cast<float2*>(s0 + 8 * SM_CHUNK) =
                make_float2(acc[0][nt][mt][2] + acc[1][nt][mt][2], acc[0][nt][mt][3] + acc[1][nt][mt][3]);
          }
      }
      __syncthreads();
      // ---- softmax over the chunk's rows, per head ----
#pragma unroll
      for (int jj = 0; jj < HPW; ++jj) {
        const int h = warp + SM_WARPS * jj;
        if (h < H) {
          float sum = 0.f;   // the eight column parts, in order
#pragma unroll
          for (int w = 0; w < SM_WARPS; ++w) sum += sc_s[(w * HM + h) * SM_CHUNK + lane];
          const float sc = lane < nr ? sum * a.scale_log2 : -CUDART_INF_F;
          const float m = warp_max(sc);
          const float pv = lane < nr ? ex2(sc - m) : 0.f;
          const float l = warp_sum(pv);
          split_bf16(pv, &p_s[h * PP + lane], &p_s[(HM + h) * PP + lane]);
          if (lane == 0) reinterpret_cast<float4*>(part + (int64_t)h * (C + 4))[C / 4] = make_float4(m, l, 0.f, 0.f);
        }
      }
      __syncthreads();
      // ---- output rows: latent columns of this warp ----
      {
        const int tpw = C / 64;   // 8-column tiles per warp
        uint32_t pf[2][2][MT][4];   // [column step][hi, lo][head tile]
#pragma unroll
        for (int ks = 0; ks < 2; ++ks)
#pragma unroll
          for (int hl = 0; hl < 2; ++hl)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
              ldsm_x4(p_a + (uint32_t)((((hl * HM + mt * 16) + (lane & 7) + 8 * ((lane >> 3) & 1)) * PP + ks * 16 +
                                        8 * (lane >> 4)) * 2),
                      pf[ks][hl][mt]);
#pragma unroll 2
        for (int jt = 0; jt < tpw; ++jt) {
          const int n0 = (warp * tpw + jt) * 8;
          uint32_t bv[4];   // rows 0-7, 8-15, 16-23, 24-31 of columns n0 .. n0 + 7, transposed
          ldsm_x4_trans(tile_a + (uint32_t)((lane * CRP + n0) * 2), bv);
          float acc[2][MT][4];
#pragma unroll
          for (int hl = 0; hl < 2; ++hl)
#pragma unroll
            for (int mt = 0; mt < MT; ++mt)
#pragma unroll
              for (int e = 0; e < 4; ++e) acc[hl][mt][e] = 0.f;
#pragma unroll
          for (int ks = 0; ks < 2; ++ks)
#pragma unroll
            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
              for (int mt = 0; mt < MT; ++mt) mma_bf16(acc[hl][mt], pf[ks][hl][mt], bv[2 * ks], bv[2 * ks + 1]);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int h = mt * 16 + grp;
            if (h < H)
              *reinterpret_cast<float2*>(part + (int64_t)h * (C + 4) + n0 + 2 * tig) =
                  make_float2(acc[0][mt][0] + acc[1][mt][0], acc[0][mt][1] + acc[1][mt][1]);
            if (h + 8 < H)
              *reinterpret_cast<float2*>(part + (int64_t)(h + 8) * (C + 4) + n0 + 2 * tig) =
                  make_float2(acc[0][mt][2] + acc[1][mt][2], acc[0][mt][3] + acc[1][mt][3]);
          }
        }
      }
    }
    __syncthreads();   // the tile, scores and P are reused by the next chunk
  }
  if (ok) ok = grid_barrier(sm_counter(a.hdr, 1), G, a.wait_ns, &flag_s);

  // ================================ 3. merge and W_UV ================================
  // Item (sequence, head, 64 latent columns): the chunks' partials merged in chunk order, then
  // that slice's share of out[b,h,:] = W_UV,h o (W_UV of the first item read before the
  // dependency wait). The last of a head's C/64 items to finish (a counter per head) adds the
  // shares in slice order and writes out and lse: no further barrier.
  __shared__ __align__(16) float colred_s[16][64];
  __shared__ int last_s;
  for (int it = g; it < n_items1; it += G) {
    const int b = it / (H * (C / 64)), h = (it / (C / 64)) % H, cc = it % (C / 64);
    const int nch = cfirst_s[b + 1] - cfirst_s[b];
    float* share = a.wshare + ((int64_t)(b * H + h) * (C / 64) + cc) * V;
    float M = CUDART_NAN_F, Ls = CUDART_NAN_F;
    if (!ok) {   // a CTA whose wait ran out: its shares are NaN
      for (int v = tid; v < V; v += SM_THREADS) share[v] = CUDART_NAN_F;
    } else {
      const float* pb = a.part + (int64_t)b * a.max_chunks * H * (C + 4) + (int64_t)h * (C + 4);
      const int64_t cstride = (int64_t)H * (C + 4);   // between chunks
      // every load at once: the maximum and sum of chunk tid, columns 4 * (tid & 15) .. + 3 of
      // chunks (tid >> 4) + 16 i
      float2 ml = make_float2(-CUDART_INF_F, 0.f);
      if (tid < nch) ml = __ldcg(reinterpret_cast<const float2*>(pb + tid * cstride + C));
      const int quad = tid & 15, grp = tid >> 4;
      float4 t[SM_MAX_CHUNKS / 16];
#pragma unroll
      for (int i = 0; i < SM_MAX_CHUNKS / 16; ++i) {
        const int kk = grp + 16 * i;
        t[i] = kk < nch ? __ldcg(reinterpret_cast<const float4*>(pb + kk * cstride + cc * 64) + quad)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      const float mx = warp_max(ml.x);
      if (lane == 0) wred_s[warp] = mx;
      __syncthreads();
      M = wred_s[0];
      for (int w = 1; w < SM_WARPS; ++w) M = fmaxf(M, wred_s[w]);
      __syncthreads();
      const float wk = tid < nch ? ex2(ml.x - M) : 0.f;
      if (tid < nch) w_s[tid] = wk;
      const float pl = warp_sum(wk * ml.y);
      if (lane == 0) wred_s[warp] = pl;
      __syncthreads();
      Ls = 0.f;
      for (int w = 0; w < SM_WARPS; ++w) Ls += wred_s[w];
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int i = 0; i < SM_MAX_CHUNKS / 16; ++i) {
        const int kk = grp + 16 * i;
        if (kk < nch) {
          const float w = w_s[kk];
          acc.x = fmaf(w, t[i].x, acc.x); acc.y = fmaf(w, t[i].y, acc.y);
          acc.z = fmaf(w, t[i].z, acc.z); acc.w = fmaf(w, t[i].w, acc.w);
        }
      }
      reinterpret_cast<float4*>(colred_s[grp])[quad] = acc;
      __syncthreads();
      if (tid < 64) {
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < 16; ++q) sum += colred_s[q][tid];
        ol_s[tid] = sum / Ls;
      }
      __syncthreads();
      // the slice's share of out: row tid >> 1, half tid & 1 of the 64 columns
      const int v = tid >> 1;
      uint32_t wv[16];
      if (it == g) {
#pragma unroll
        for (int i = 0; i < 16; ++i) wv[i] = wuv[i];
      } else {
        const uint4* wsrc =
            reinterpret_cast<const uint4*>(a.kv_b + ((int64_t)h * NV + N + v) * C + cc * 64 + (tid & 1) * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 u = v < V ? wsrc[i] : make_uint4(0, 0, 0, 0);
          wv[4 * i] = u.x; wv[4 * i + 1] = u.y; wv[4 * i + 2] = u.z; wv[4 * i + 3] = u.w;
        }
      }
      const float* o = ol_s + (tid & 1) * 32;
      float y = 0.f;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        y = fmaf(__uint_as_float(wv[i] << 16), o[2 * i], y);
        y = fmaf(__uint_as_float(wv[i] & 0xFFFF0000u), o[2 * i + 1], y);
      }
      y += __shfl_xor_sync(0xffffffffu, y, 1);
      if ((tid & 1) == 0 && v < V) share[v] = y;
    }
    // the last of the head's slices adds the shares
    __syncthreads();
    if (tid == 0) {   // acquire-release: the shares written before are seen by the last slice
      unsigned int prev;
      asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&a.head_cnt[b * H + h]) : "memory");
      last_s = prev == (unsigned int)(C / 64 - 1);
    }
    __syncthreads();
    if (last_s) {
      const float* sh0 = a.wshare + (int64_t)(b * H + h) * (C / 64) * V;
      const bool valid = nch > 0;   // a length out of range: NaN
      for (int v = tid; v < V; v += SM_THREADS) {
        float y = 0.f;
        for (int s2 = 0; s2 < C / 64; ++s2) y += __ldcg(sh0 + s2 * V + v);
        a.out[((int64_t)b * H + h) * V + v] = valid ? y : CUDART_NAN_F;
      }
      if (tid == 0 && a.lse != nullptr)
        a.lse[(int64_t)b * H + h] = valid ? (M + __log2f(Ls)) * 0.69314718055994530942f : CUDART_NAN_F;
    }
    __syncthreads();   // w_s, ol_s, colred_s, wred_s and last_s are reused by the next item
  }
  if (!ok && tid == 0) set_error(a.hdr, MLA_ERR_TIMEOUT, 0);

  // ---- leave: a row copy still in flight (a wait that ran out) gets one more bounded wait ----
  if (rows_pending && tid == 0) tc::mbar_wait(&rows_bar, rows_par, kWaitDrainNs);
  // ---- the last CTA out resets the counters for the next call ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(sm_counter(a.hdr, 2), 1u) == G - 1) {
      for (int i = 0; i < 3; ++i) atomicExch(sm_counter(a.hdr, i), 0u);
      __threadfence();
    }
  }
}

}  // namespace

int64_t decode_small_max_chunks(const mla_config& cfg) {
  const int64_t cap = cfg.page_size == 0 ? cfg.rows_per_seq : (int64_t)cfg.max_pages_per_seq * cfg.page_size;
  return (cap + SM_CHUNK - 1) / SM_CHUNK;
}

// CTAs of the grid: one per chunk of the longest batch or per absorb / merge item (sequence, head,
// 64 latent columns), whichever is more, at most one per SM.
int decode_small_grid(const mla_config& cfg, int B) {
  const int sms = device_sms();
  const int64_t chunks = (int64_t)B * decode_small_max_chunks(cfg);
  const int64_t items = (int64_t)B * cfg.n_heads * (cfg.kv_lora / 64);
  const int64_t want = chunks > items ? chunks : items;
  return (int)(want < sms ? want : sms);
}

bool decode_small_supported(const mla_config& cfg, int B, int tokens) {
  const int64_t cap = cfg.page_size == 0 ? cfg.rows_per_seq : (int64_t)cfg.max_pages_per_seq * cfg.page_size;
  const bool dims = tokens == 1 && cfg.act_dtype == MLA_BF16 && cfg.kv_b_dtype == MLA_BF16 && B >= 1 &&
                    (int64_t)B * cfg.n_heads <= 64 && cfg.n_heads <= SM_WARPS * SM_MAX_HPW &&
                    cfg.kv_lora % 128 == 0 && cfg.kv_lora <= 32 * SM_MAX_CPL &&
                    (cfg.kv_lora + cfg.qk_rope) % 8 == 0 && cfg.qk_rope <= 64 && cfg.qk_rope % 16 == 0 &&
                    cfg.qk_nope % 4 == 0 && cfg.qk_nope <= 128 && cfg.v_head % 16 == 0 && cfg.v_head <= 128 &&
                    cap >= 1 && cap <= (int64_t)SM_CHUNK * SM_MAX_CHUNKS;
  if (!dims) return false;
  const int G = decode_small_grid(cfg, B);
  if (G < 1) return false;
  // Against the staged kernels with the tensor-core attention (rows of 512 + 64), the one launch
  // wins while its CTAs take few rounds: measured on one GB300 it takes ~14.6 us with one round
  // of absorb / merge items and one of 32-row chunks, ~4.6 us more per further round of items and
  // ~3.3 us per further round of chunks, against ~21-25 us staged. Otherwise (the staged path's
  // CUDA-core attention) it is always the faster.
  const int64_t items = (int64_t)B * cfg.n_heads * (cfg.kv_lora / 64);
  const int64_t chunks = (int64_t)B * decode_small_max_chunks(cfg);
  const int64_t rounds = (items + G - 1) / G + (chunks + G - 1) / G;
  const bool staged_tc = cfg.kv_lora == 512 && cfg.qk_rope == 64;
  return !staged_tc || rounds <= 3;
}

cudaError_t launch_decode_small(const mla_config& cfg, const mla_cache& cache, const void* q, const void* kv_b,
                                const int32_t* seq_lens, const int32_t* positions, float* out, float* lse, int B,
                                float* qf, float* part, float* wshare, unsigned int* head_cnt, WsHeader* hdr,
                                cudaStream_t st) {
  SmallArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.kv_b = static_cast<const uint16_t*>(kv_b);
  a.rows = static_cast<const uint16_t*>(cache.rows);
  a.map = RowMap{cache.page_table, cfg.page_size, cfg.max_pages_per_seq, cfg.rows_per_seq, cache.n_physical_rows};
  a.seq_lens = seq_lens;
  a.positions = positions;
  a.inv_freq = cfg.rope_inv_freq;
  a.out = out;
  a.lse = lse;
  a.qf = qf;
  a.part = part;
  a.wshare = wshare;
  a.head_cnt = head_cnt;
  a.hdr = hdr;
  a.B = B;
  a.H = cfg.n_heads;
  a.C = cfg.kv_lora;
  a.R = cfg.qk_rope;
  a.N = cfg.qk_nope;
  a.V = cfg.v_head;
  a.max_chunks = (int)decode_small_max_chunks(cfg);
  a.scale_log2 = cfg.softmax_scale * 1.4426950408889634f;
  a.wait_ns = wait_limit_ns();
  const int hpw = (cfg.n_heads + SM_WARPS - 1) / SM_WARPS;
  const int CR = cfg.kv_lora + cfg.qk_rope, hm = hpw > 2 ? 32 : 16;
  // raw rows, padded tile, queries (hi, lo), the scores' eight column parts, P (hi, lo)
  const int smem = SM_CHUNK * CR * 2 + SM_CHUNK * (CR + 8) * 2 + 2 * hm * (CR + 8) * 2 + SM_WARPS * hm * SM_CHUNK * 4 +
                   2 * hm * (SM_CHUNK + 8) * 2;
  void (*kern)(SmallArgs) = hpw == 1 ? decode_small_kernel<1> : hpw == 2 ? decode_small_kernel<2> : decode_small_kernel<4>;
  cudaError_t e = ensure_smem((const void*)kern, smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3((unsigned)decode_small_grid(cfg, B)), dim3(SM_THREADS), (size_t)smem, st, a);
}

}  // namespace mla
