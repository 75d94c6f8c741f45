// Split attention over compressed bf16 cache rows for 128 heads on a pair of SMs: a cluster of
// two CTAs on the 5th-generation tensor cores (tcgen05), exchanging partial scores and
// probabilities through distributed shared memory.
//
// turbospark-runtime 0.3.0, src/families/deepseek2/attn.rs, MQA attention over the compressed
// rows (key = whole row [kv_lat ; k_pe], value = its first kv_lora elements, all heads read the
// same rows); moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs, mla_sdpa_folded.
//
// Shape: rows of 576 = 512 latent + 64 rope, bf16, 128 heads. CTA c (0 or 1) of a pair streams,
// for every 64-row tile, latent columns [256c, 256c + 256) and rope columns [512 + 32c, +32) of
// each row (36 KB) into a three-stage ring. It holds the queries of all 128 heads for those
// columns: the latent part in tensor memory (the A operand of QK^T), the rope part in shared
// memory twice, as the bf16 rotated q_pe and as its bf16 rounding residual, so the rope score is
// exact to about 2^-16. Per tile it computes the partial scores
//     S_c = Q_c . K_c^T      (M = 128 heads, N = 64 rows, K = 256 + 2 x 32)   in tensor memory
// and S = S_0 + S_1. CTA c owns the softmax of heads [64c, 64c + 64): its threads for the other
// 64 heads stage their partial scores in shared memory and one bulk copy sends them into the
// peer's shared memory; the own-head threads add the peer's partial to their own, keep the
// running maximum and sum, and write their heads' rows of P (bf16, 128 heads x 64 rows, the A
// operand of PV) into this CTA's P buffer, and one bulk copy writes the same rows into the
// peer's P buffer. Each CTA then accumulates its latent half of the output for all 128 heads,
//     O_c += P . V_c         (M = 128 heads, N = 256 latent, K = 64 rows)
// in tensor memory. Every cache row is read from memory once per pair; the pair exchanges 24 KB
// per tile in each direction.
//
// Softmax: two threads per head (heads are the MMA rows; each thread holds 32 of the tile's 64
// scores of its head), log2 domain, with a running maximum that is only raised when a score
// exceeds it by more than 2^16; then the output rows of that head are rescaled in both CTAs (the
// rescale factor travels with the probabilities).
//
// Work split: the 64-row tiles of all sequences form one list, with a few units of switch cost
// ahead of each sequence; pair k takes the k-th equal share of it, crossing sequence boundaries.
// Each (pair, sequence) piece writes a partial (O normalised, lse) into slot k + b; CTA c writes
// latent columns [256c, 256c + 256) of every head and the lse of its own heads.
//
// Roles (384 threads). Warps 0-7 access tensor memory, warp w the lane quarter w mod 4 (32 heads):
// on this CTA's own heads, warps of both sets run the softmax (one half of the tile's rows each)
// and the epilogue of those heads; on the peer's heads, warps 0-3 send this CTA's partial scores
// and warps 4-7 take the peer's rescale factors, rescale those heads' output rows and write their
// epilogue. All eight warps also load each segment's latent queries into tensor memory (half of
// a head's columns each). Of warps 8-11, one issues the TMA loads and one owns tensor memory and
// issues the MMAs (one thread), polling and issuing whichever of the next QK^T and the next PV is
// ready; both sit on the sub-partitions of the peer-head warps. A third forwards the score grants
// to the peer, so that no softmax thread waits on a remote arrival. Every wait is bounded; on a
// timeout the CTA records MLA_ERR_TIMEOUT and tells its peer, every role stops, transfers in
// flight in both directions are drained, and tensor memory is freed.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <math_constants.h>

namespace mla {

namespace {

constexpr int AP_TILE = 64;                             // rows per tile (MMA N of QK^T, K of PV)
constexpr int AP_HEADS = 128;                           // MMA M
constexpr int AP_BLK = AP_TILE * 128;                   // 8 KB: 64 rows x 64 latent columns (128-byte rows)
constexpr int AP_RBLK = AP_TILE * 64;                   // 4 KB: 64 rows x 32 rope columns (64-byte rows)
constexpr int AP_STAGE = 4 * AP_BLK + AP_RBLK;          // 36 KB
constexpr int AP_STAGES = 3;
constexpr int AP_QR = AP_HEADS * 64;                    // 8 KB: 128 heads x 32 rope columns
constexpr int AP_SBUF = 64 * AP_TILE * 4;               // 16 KB: 64 heads' partial scores of a tile
constexpr int AP_PBUF = AP_HEADS * 128;                 // 16 KB: P, 128 heads x 64 rows bf16
// shared memory: rope queries (hi, lo), stages, received and sent scores (two each), P (two)
constexpr int AP_OFF_STAGES = 2 * AP_QR;
constexpr int AP_OFF_SRECV = AP_OFF_STAGES + AP_STAGES * AP_STAGE;
constexpr int AP_OFF_SSEND = AP_OFF_SRECV + 2 * AP_SBUF;
constexpr int AP_OFF_P = AP_OFF_SSEND + 2 * AP_SBUF;
constexpr int AP_SMEM_DYN = AP_OFF_P + 2 * AP_PBUF + 1024;
constexpr int AP_THREADS = 384;
// warps 8-11 sit one on each SM sub-partition (warp w on sub-partition w mod 4); the TMA and MMA
// roles take the two whose sub-partitions hold the peer-head warps, so that their polling never
// competes with this CTA's softmax warps (which sit on the sub-partitions of their lane quarters)
__device__ __forceinline__ int ap_tma_warp(uint32_t c) { return c == 0 ? 10 : 8; }
__device__ __forceinline__ int ap_mma_warp(uint32_t c) { return c == 0 ? 11 : 9; }
// one of the two remaining warps forwards the score grants: a remote arrival with release
// semantics takes the issuing thread about half a microsecond, which must not hold up the softmax
__device__ __forceinline__ int ap_fwd_warp(uint32_t c) { return c == 0 ? 8 : 10; }
constexpr uint32_t AP_S_COL = 0;     // S: two buffers of 64 columns
constexpr uint32_t AP_Q_COL = 128;   // latent queries: 128 columns of bf16 pairs (256 latent)
constexpr uint32_t AP_O_COL = 256;   // O: 256 columns
constexpr uint32_t AP_TMEM_COLS = 512;
// log2 units: p may reach 2^16 before a rescale (bf16 P and the float32 sums hold that with room
// to spare: at most 2^16 x 2^17 rows x |v| per sum); at 2^8 the YaRN-scaled scores of the long
// Q8_0 workload crossed it on a tenth of the tiles, each costing a wait for PV and an O rescale
constexpr float AP_RESCALE = 16.0f;
constexpr uint64_t AP_DRAIN = kWaitDrainNs;
// named barriers: own-head softmax threads (128), score senders (64), factor receivers (64)
constexpr int AP_BAR_OWN = 1, AP_BAR_SEND = 2, AP_BAR_RECV = 3;
constexpr int AP_N_OWN = 128, AP_N_SEND = 64, AP_N_RECV = 64;
constexpr uint32_t AP_PX_BYTES = 64 * 128 + 64 * 4;    // one CTA's rows of P + its rescale factors

struct PairArgs {
  RowMap map;
  const int32_t* seq_lens;
  const uint16_t* q_abs;  // [B][128][576] bf16 fused query rows
  float* part_o;          // [n_slots][128][512]
  float* part_lse;        // [n_slots][128]
  int32_t* meta;          // [B][2]: first slot, slot count
  WsHeader* hdr;
  int B, n_pairs, n_slots;
  float scale_log2;
  uint64_t wait_ns;
  int kv_early;           // cache rows may be read before the dependency wait (see attn_tc.cu)
};

struct __align__(16) PairSmem {
  uint64_t full[AP_STAGES], empty[AP_STAGES];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_free[2];
  uint64_t srecv_full[2];   // the peer's partial scores of tile n landed in buffer n & 1
  uint64_t srecv_grant[2];  // the peer has read buffer n & 1 of our partial scores
  uint64_t srecv_read[2];   // this CTA's softmax has read the peer's scores of tile n (buffer n & 1)
  uint64_t pfree[2];        // PV of tile n in both CTAs done: P buffer n & 1 free (two arrivals)
  uint64_t px_full[2];      // the peer's rows of P and its factors for tile n landed (buffer n & 1)
  uint64_t l_full[2];       // the peer's 1/l of segment j landed in l_recv[j & 1]
  uint64_t pv_ready[2];     // P of tile n is written and O rescaled
  uint64_t pv_done[2];      // PV of tile n has completed (this CTA)
  uint64_t o_full, o_empty;
  uint64_t mma_fin;
  uint32_t tmem_base;
  int abort;
  int seg_b0;
  long long seg_p0;
  int bad_page[4];          // by segment mod 4: the producer runs at most three tiles ahead
  int sent[3];              // transfers this CTA issued to its peer: scores, P, 1/l
  int got[3];               // transfers of the peer this CTA consumed
  int peer_sent[3];         // written by the peer before the final cluster barriers
  // bulk-copied: 16-byte aligned
  __align__(16) float alpha_send[2][64];
  __align__(16) float alpha_recv[2][64];
  float l_recv[2][64];
  float xch[2][64];         // own heads: the two half-row threads' partial maxima (and sums)
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// OR of `v` over the `count` threads of named barrier `id`, returned to all of them.
__device__ __forceinline__ bool group_vote_or(bool v, int id, int count) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "barrier.red.or.pred po, %2, %3, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(id), "r"(count)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void group_bar(int id, int count) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// A bounded wait that also gives up once this CTA (or its peer, which tells it) has aborted.
// `cluster`: acquire at cluster scope, for barriers the peer completes.
__device__ __forceinline__ bool wait_bar(PairSmem& s, uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                         bool cluster = false) {
  const uint64_t t0 = tc::global_ns();
  for (uint32_t i = 0;; ++i) {
    if (cluster ? tc::mbar_try_wait_cluster(bar, parity) : tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 15) == 15) {
      if (*reinterpret_cast<volatile int*>(&s.abort)) return false;
      if (tc::global_ns() - t0 > limit_ns) return false;
    }
  }
}

// A wait of a thread group (named barrier `id`, `count` threads): every thread polls, then the
// group agrees on the outcome so its threads always leave (or stay in) their loops together.
__device__ __forceinline__ bool group_wait(PairSmem& s, uint64_t* bar, uint32_t parity, int id, int count,
                                           uint64_t limit_ns, bool cluster = false) {
  const bool ok = wait_bar(s, bar, parity, limit_ns, cluster);
  __syncwarp();
  return !group_vote_or(!ok, id, count);
}

// Record the first failure of this CTA and tell the peer, whose waits then give up too.
__device__ __forceinline__ void pair_fail(PairSmem& s, WsHeader* hdr, int b, uint32_t peer) {
  if (atomicExch(&s.abort, 1) == 0) {
    set_error(hdr, MLA_ERR_TIMEOUT, b);
    tc::st_cluster_u32(tc::mapa(tc::smem_u32(&s.abort), peer), 1);
  }
}

__device__ __forceinline__ long long seq_tiles(const PairArgs& a, int b) {
  const long long L = a.seq_lens[b];
  if (L < 1 || L > a.map.capacity()) return 0;
  return (L + AP_TILE - 1) / AP_TILE;
}

// The work list the pairs share is measured in tiles, plus AP_SEG_COST units ahead of each
// sequence: a pair that starts a new sequence within its share pays for the switch (the next
// queries, the previous segment's epilogue, a cold exchange chain: ~5-7 us), so it takes that
// many fewer tiles and the pairs end closer together (3, 4 and 5 units measured: 4 was best).
// Sequence b occupies [v_b, v_b + AP_SEG_COST + n_b) of the list, its tiles the last n_b units.
constexpr long long AP_SEG_COST = 4;
__device__ __forceinline__ long long seq_width(const PairArgs& a, int b) {
  const long long n = seq_tiles(a, b);
  return n > 0 ? n + AP_SEG_COST : 0;
}

// Segment iterator over the (sequence, tile range) pieces of a pair's share [r0, r1) of the
// work list; p is the list position where sequence b starts.
struct PairSegIter {
  int b;
  long long p;
  long long r0, r1;
  __device__ bool next(const PairArgs& a, int* sb, int* t_lo, int* t_hi) {
    while (b < a.B && p < r1) {
      const long long n = seq_tiles(a, b);
      const long long p_t = p + AP_SEG_COST;   // list position of the sequence's first tile
      const long long lo = max(r0, p_t), hi = min(r1, p_t + n);
      const int cur = b;
      ++b;
      p += n > 0 ? n + AP_SEG_COST : 0;
      if (hi > lo) {
        *sb = cur;
        *t_lo = (int)(lo - p_t);
        *t_hi = (int)(hi - p_t);
        return true;
      }
    }
    return false;
  }
};

// Swizzled 16-byte chunk k of head row hl in a buffer of rows of `row_bytes` (chunk index XOR
// the row index mod 8, so eight consecutive rows hit eight different bank groups).
__device__ __forceinline__ uint32_t swz(uint32_t hl, uint32_t k, uint32_t row_bytes) {
  return hl * row_bytes + ((k ^ (hl & 7u)) << 4);
}

// Latent queries of head lane `h` of sequence `sb`: latent columns [col0, col0 + 128) of this
// CTA's half into tensor-memory columns t_q + col0 / 2 onwards (bf16 pairs, 32 columns a store).
// All 256 bytes are requested at once, so the load costs one memory round trip. Warp-collective
// (tcgen05.st).
__device__ __forceinline__ void load_q_lat(const PairArgs& a, uint32_t c, int sb, int h, int col0, uint32_t t_q) {
  const uint4* src =
      reinterpret_cast<const uint4*>(a.q_abs + ((size_t)sb * AP_HEADS + h) * 576 + 256 * c + col0);
  uint4 v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = src[i];
#pragma unroll
  for (int hb = 0; hb < 2; ++hb) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      r[4 * i] = v[8 * hb + i].x;
      r[4 * i + 1] = v[8 * hb + i].y;
      r[4 * i + 2] = v[8 * hb + i].z;
      r[4 * i + 3] = v[8 * hb + i].w;
    }
    tc::tmem_st32(t_q + (uint32_t)(col0 / 2 + 32 * hb), r);
  }
}

__global__ void __launch_bounds__(AP_THREADS, 1)
attn_pair_kernel(const __grid_constant__ CUtensorMap rows_map, const __grid_constant__ CUtensorMap rope_map,
                 const __grid_constant__ CUtensorMap qrope_map, const __grid_constant__ CUtensorMap qres_map,
                 PairArgs a) {
  extern __shared__ uint8_t dyn_raw[];
  __shared__ PairSmem s;
  pdl_trigger();
  uint8_t* dyn = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* qrope = dyn;                                // [hi ; lo] x [128 heads x 32 columns], 64-byte swizzle
  uint8_t* stages = dyn + AP_OFF_STAGES;               // 3 x (4 latent blocks + 1 rope block)
  uint8_t* srecv = dyn + AP_OFF_SRECV;                 // 2 x [64 own heads][64 rows] fp32, swizzled
  uint8_t* ssend = dyn + AP_OFF_SSEND;                 // 2 x [64 peer heads][64 rows] fp32, swizzled
  uint8_t* pbuf = dyn + AP_OFF_P;                      // 2 x [128 heads][64 rows] bf16, 128-byte swizzle
  long long* scan = reinterpret_cast<long long*>(stages);   // prologue scratch
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t c = tc::cluster_ctarank();
  const uint32_t peer = c ^ 1u;
  const int pair = blockIdx.x >> 1;

  // ---- length of the work list (block scan over per-thread chunks of sequences) ----
  const int chunk = (a.B + AP_THREADS - 1) / AP_THREADS;
  const int cb0 = min(a.B, tid * chunk), cb1 = min(a.B, cb0 + chunk);
  long long mine = 0;
  for (int b = cb0; b < cb1; ++b) mine += seq_width(a, b);
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) scan[warp] = incl;
  if (tid == 0) {
    s.abort = 0;
    s.seg_b0 = a.B;
    s.seg_p0 = 0;
    for (int i = 0; i < 4; ++i) s.bad_page[i] = 0;
    for (int i = 0; i < 3; ++i) s.sent[i] = s.got[i] = s.peer_sent[i] = 0;
  }
  __syncwarp();
  __syncthreads();
  long long before = incl - mine, T = 0;
#pragma unroll
  for (int w = 0; w < AP_THREADS / 32; ++w) {
    const long long v = scan[w];
    if (w < warp) before += v;
    T += v;
  }
  const long long r0 = (T * pair) / a.n_pairs, r1 = (T * (pair + 1)) / a.n_pairs;
  if (r0 < r1) {
    if (tid == 0) {
      for (int i = 0; i < AP_STAGES; ++i) {
        tc::mbar_init(&s.full[i], 1);
        tc::mbar_init(&s.empty[i], 1);
      }
      // the latent queries from the own-head, score-sender and receiver threads, the rope queries
      // by TMA
      tc::mbar_init(&s.q_full, AP_N_OWN + AP_N_SEND + AP_N_RECV + 1);
      tc::mbar_init(&s.q_empty, 1);
      for (int i = 0; i < 2; ++i) {
        tc::mbar_init(&s.s_full[i], 1);
        tc::mbar_init(&s.s_free[i], AP_N_OWN + AP_N_SEND);
        tc::mbar_init(&s.srecv_full[i], 1);
        tc::mbar_init(&s.srecv_grant[i], 1);
        tc::mbar_init(&s.pfree[i], 2);
        tc::mbar_init(&s.px_full[i], 1);
        tc::mbar_init(&s.l_full[i], 1);
        tc::mbar_init(&s.pv_ready[i], AP_N_OWN + AP_N_RECV);
        tc::mbar_init(&s.pv_done[i], 1);
        // the first transfer into each buffer is expected from the start; later ones are
        // re-armed by the receiving threads before they let the peer send into it again
        tc::mbar_arrive_expect_tx(&s.srecv_full[i], AP_SBUF);
        tc::mbar_arrive_expect_tx(&s.px_full[i], AP_PX_BYTES);
        tc::mbar_arrive_expect_tx(&s.l_full[i], 64 * 4);
      }
      tc::mbar_init(&s.srecv_read[0], 1);
      tc::mbar_init(&s.srecv_read[1], 1);
      tc::mbar_init(&s.o_full, 1);
      tc::mbar_init(&s.o_empty, AP_N_OWN + AP_N_RECV);
      tc::mbar_init(&s.mma_fin, 1);
      tc::fence_mbar_init();
    }
    if (warp == ap_mma_warp(c)) {
      tc::tmem_alloc(&s.tmem_base, AP_TMEM_COLS);
      tc::tmem_relinquish();
    }
    if (warp == ap_tma_warp(c) && lane == 0) {
      tc::tma_prefetch_desc(&rows_map);
      tc::tma_prefetch_desc(&rope_map);
      tc::tma_prefetch_desc(&qrope_map);
      tc::tma_prefetch_desc(&qres_map);
    }
  }
  // the thread whose chunk holds list position r0 finds the first sequence of the pair's share
  if (r0 < r1 && before <= r0 && r0 < before + mine) {
    long long p = before;
    for (int b = cb0; b < cb1; ++b) {
      const long long n = seq_width(a, b);
      if (r0 < p + n) {
        s.seg_b0 = b;
        s.seg_p0 = p;
        break;
      }
      p += n;
    }
  }
  if (!a.kv_early) pdl_wait();
  // CTA 0 of pair 0 publishes, per sequence, which partial slots the combine must merge: those
  // of the pairs whose shares hold the sequence's first tile (list position x) to its last
  // (x + n - 1); pair k holds [T k / n_pairs, T (k + 1) / n_pairs)
  if (blockIdx.x == 0) {
    long long p = before;
    for (int b = cb0; b < cb1; ++b) {
      const long long n = seq_tiles(a, b);
      int first = 0, count = 0;
      if (n > 0) {
        const long long x = p + AP_SEG_COST;
        const long long kf = ((x + 1) * a.n_pairs + T - 1) / T - 1;
        const long long kl = ((x + n) * a.n_pairs + T - 1) / T - 1;
        first = (int)(kf + b);
        count = (int)(kl - kf + 1);
      } else {
        set_error(a.hdr, MLA_ERR_BAD_SEQ_LEN, b);
      }
      a.meta[2 * b] = first;
      a.meta[2 * b + 1] = count;
      p += seq_width(a, b);
    }
  }
  if (r0 >= r1) {
    // both CTAs of the pair leave here (they computed the same range); no shared memory of the
    // peer is touched
    pdl_wait();
    if (c == 0 && before <= r0 && r0 < before + mine) {
      long long p = before;
      for (int b = cb0; b < cb1; ++b) {
        const long long n = seq_width(a, b);
        if (r0 < p + n) {
          // an empty share strictly inside the sequence's tiles lies in its slot interval
          if (p + AP_SEG_COST < r0) {
            float* pl = a.part_lse + (size_t)(pair + b) * AP_HEADS;
            for (int h = 0; h < AP_HEADS; ++h) pl[h] = -CUDART_INF_F;
          }
          break;
        }
        p += n;
      }
    }
    return;
  }

  tc::fence_proxy_async_smem();   // the prologue's generic writes precede the TMA writes
  tc::tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc::tc_fence_after();
  // the peer's barriers are initialised and armed before either CTA sends anything
  tc::cluster_sync();
  const uint32_t tmem = s.tmem_base;
  PairSegIter it{s.seg_b0, s.seg_p0, r0, r1};
  int fail_b = s.seg_b0;

  if (warp == ap_tma_warp(c)) {
    // ================================ TMA producer ================================
    if (lane == 0) {
      int sb = 0, tlo, thi, seg = 0;
      long long n = 0;
      long long last_n[AP_STAGES];
      for (int i = 0; i < AP_STAGES; ++i) last_n[i] = -1;
      int q_loaded = -1;
      bool ok = true;
      const uint64_t kv_policy = tc::l2_policy_evict_first();
      auto load_q = [&]() -> bool {
        if (seg > 0 && !wait_bar(s, &s.q_empty, (seg - 1) & 1, a.wait_ns)) return false;
        tc::mbar_arrive_expect_tx(&s.q_full, 2 * AP_QR);
        const int qrow = sb * AP_HEADS;
        tc::tma_load_2d(qrope, &qrope_map, 512 + 32 * (int)c, qrow, &s.q_full);
        tc::tma_load_2d(qrope + AP_QR, &qres_map, 512 + 32 * (int)c, qrow, &s.q_full);
        q_loaded = seg;
        return true;
      };
      while (ok && it.next(a, &sb, &tlo, &thi)) {
        fail_b = sb;
        // A segment's rope queries replace the previous segment's once its last QK^T is done
        // (q_empty); that wait comes after the segment's first tile is on its way, so that the
        // tile's load overlaps the end of the previous segment instead of following it.
        bool q_pending = true;
        for (int t = tlo; t < thi && ok; ++t) {
          const int st = (int)(n % AP_STAGES);
          // the row lookup (a page-table read) goes before the wait for a free stage, which
          // lies on the loop from PV of tile n - 3 to QK^T of tile n
          int64_t pr = a.map.phys(sb, (int64_t)t * AP_TILE);
          if (n >= AP_STAGES && !wait_bar(s, &s.empty[st], (uint32_t)(((n / AP_STAGES) - 1) & 1), a.wait_ns)) {
            ok = false;
            break;
          }
          if (pr < 0) {   // out-of-range page id: load a valid row, flag the segment
            atomicExch(&s.bad_page[seg & 3], 1);
            set_error(a.hdr, MLA_ERR_BAD_PAGE, sb);
            pr = 0;
          }
          uint8_t* dst = stages + st * AP_STAGE;
          tc::mbar_arrive_expect_tx(&s.full[st], AP_STAGE);
          // this CTA's four 64-column latent blocks in one copy (four [64 rows][64] tiles)
          tc::tma_load_3d_hint(dst, &rows_map, 0, (int32_t)pr, 4 * (int)c, &s.full[st], kv_policy);
          tc::tma_load_2d_hint(dst + 4 * AP_BLK, &rope_map, 512 + 32 * (int)c, (int32_t)pr, &s.full[st], kv_policy);
          last_n[st] = n;
          if (q_pending) {
            q_pending = false;
            if (a.kv_early && seg == 0) pdl_wait();
            if (!load_q()) ok = false;
          }
          if (ok) ++n;
        }
        if (ok) ++seg;
      }
      if (!ok) pair_fail(s, a.hdr, fail_b, peer);
      // every copy issued has landed before the CTA goes on to leave
      for (int i = 0; i < AP_STAGES; ++i)
        if (last_n[i] >= 0) tc::mbar_wait(&s.full[i], (uint32_t)((last_n[i] / AP_STAGES) & 1), AP_DRAIN);
      if (q_loaded >= 0) tc::mbar_wait(&s.q_full, (uint32_t)(q_loaded & 1), AP_DRAIN);
    }
  } else if (warp == ap_mma_warp(c)) {
    // ================================ MMA issuer ================================
    // QK^T of tile n needs its stage loaded, its S buffer read out (tile n - 2) and, on a
    // segment's first tile, the segment's queries; PV of tile n needs P of tile n (both CTAs'
    // rows) and, on a segment's first tile, the previous segment's O read out. The thread polls
    // both without blocking and issues whichever is ready; QK^T runs ahead as far as the stages
    // and the two S buffers allow.
    if (a.kv_early) pdl_wait();
    if (lane == 0) {
      const uint32_t idesc_qk = tc::idesc_bf16_f32(AP_HEADS, AP_TILE, 0, 0);
      const uint32_t idesc_pv = tc::idesc_bf16_f32(AP_HEADS, 256, 0, 1);
      const uint32_t qr0 = tc::smem_u32(qrope), st0 = tc::smem_u32(stages), p0 = tc::smem_u32(pbuf);
      bool ok = true;
      struct Cursor {
        PairSegIter it;
        int sb, tlo, thi, t, seg;
        long long n;
        bool live;
        __device__ void start(const PairArgs& a) {
          seg = 0;
          n = 0;
          live = it.next(a, &sb, &tlo, &thi);
          t = tlo;
        }
        __device__ void step(const PairArgs& a) {
          ++n;
          if (++t < thi) return;
          live = it.next(a, &sb, &tlo, &thi);
          t = tlo;
          ++seg;
        }
      };
      Cursor cq{it, 0, 0, 0, 0, 0, 0, false}, cp{it, 0, 0, 0, 0, 0, 0, false};
      cq.start(a);
      cp.start(a);
      uint64_t t_idle = tc::global_ns();
      while (cp.live) {
        bool progressed = false;
        if (cq.live) {
          const int st = (int)(cq.n % AP_STAGES);
          const bool first = cq.t == cq.tlo;
          if ((!first || tc::mbar_test_wait(&s.q_full, cq.seg & 1)) &&
              tc::mbar_test_wait(&s.full[st], (uint32_t)((cq.n / AP_STAGES) & 1)) &&
              (cq.n < 2 || tc::mbar_test_wait(&s.s_free[cq.n & 1], (uint32_t)(((cq.n >> 1) - 1) & 1)))) {
            tc::tc_fence_after();
            const uint32_t d = tmem + AP_S_COL + (uint32_t)(cq.n & 1) * AP_TILE;
            const uint32_t sa = st0 + st * AP_STAGE;
            // latent: A = queries in tensor memory, B = the stage's four 64-column blocks
            for (int ks = 0; ks < 16; ++ks)
              tc::mma_f16_ts(d, tmem + AP_Q_COL + 8 * ks,
                             tc::sdesc_sw128(sa + (ks >> 2) * AP_BLK + (ks & 3) * 32, 16, 1024), idesc_qk, ks != 0);
            // rope: the rotated q_pe, then its residual, against the stage's 32 rope columns
            for (int ks = 0; ks < 4; ++ks)
              tc::mma_f16_ss(d, tc::sdesc(qr0 + (ks >> 1) * AP_QR + (ks & 1) * 32, 16, 512, 4),
                             tc::sdesc(sa + 4 * AP_BLK + (ks & 1) * 32, 16, 512, 4), idesc_qk, 1);
            tc::mma_commit(&s.s_full[cq.n & 1]);
            if (cq.t + 1 == cq.thi) tc::mma_commit(&s.q_empty);
            cq.step(a);
            progressed = true;
          }
        }
        if (cp.n < cq.n) {
          const bool first = cp.t == cp.tlo, last = cp.t + 1 == cp.thi;
          const int b = (int)(cp.n & 1);
          if (tc::mbar_test_wait(&s.pv_ready[b], (uint32_t)((cp.n >> 1) & 1)) &&
              tc::mbar_try_wait_cluster(&s.px_full[b], (uint32_t)((cp.n >> 1) & 1)) &&
              (!first || cp.seg == 0 || tc::mbar_test_wait(&s.o_empty, (uint32_t)((cp.seg - 1) & 1)))) {
            tc::tc_fence_after();
            const int st = (int)(cp.n % AP_STAGES);
            // A = P (128 heads x 64 rows, K-major), B = V: the stage's four latent blocks,
            // N = 256 across them (MN-major, 8 KB apart)
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_f16_ss(tmem + AP_O_COL, tc::sdesc_sw128(p0 + b * AP_PBUF + kk * 32, 16, 1024),
                             tc::sdesc_sw128(st0 + st * AP_STAGE + kk * 2048, AP_BLK, 1024), idesc_pv,
                             !(first && kk == 0));
            tc::mma_commit(&s.empty[st]);
            tc::mma_commit(&s.pv_done[b]);
            tc::mma_commit_mc(&s.pfree[b], 0x3);   // this P buffer is free here and in the peer
            if (last) tc::mma_commit(&s.o_full);
            fail_b = cp.sb;
            cp.step(a);
            progressed = true;
          }
        }
        if (progressed) {
          t_idle = tc::global_ns();
        } else if (*reinterpret_cast<volatile int*>(&s.abort) || tc::global_ns() - t_idle > a.wait_ns) {
          ok = false;
          break;
        }
      }
      if (!ok) pair_fail(s, a.hdr, fail_b, peer);
      // every MMA issued must finish before tensor memory is released
      tc::mma_commit(&s.mma_fin);
      tc::mbar_wait(&s.mma_fin, 0, AP_DRAIN);
    }
  } else if (warp == ap_fwd_warp(c)) {
    // ================================ score-grant forwarder ================================
    // once this CTA's softmax has read the peer's partial scores of tile n out of buffer n & 1,
    // arm that buffer for tile n + 2 and tell the peer it may send into it
    if (lane == 0) {
      const uint32_t pr_srecv_grant = tc::mapa(tc::smem_u32(&s.srecv_grant[0]), peer);
      int sb = 0, tlo, thi;
      long long n = 0;
      bool ok = true;
      while (ok && it.next(a, &sb, &tlo, &thi)) {
        fail_b = sb;
        for (int t = tlo; t < thi; ++t, ++n) {
          const int b = (int)(n & 1);
          if (!wait_bar(s, &s.srecv_read[b], (uint32_t)((n >> 1) & 1), a.wait_ns)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&s.srecv_full[b], AP_SBUF);
          tc::mbar_arrive_remote(pr_srecv_grant + 8 * b);
        }
      }
      if (!ok) pair_fail(s, a.hdr, fail_b, peer);
    }
  } else if (warp < 8) {
    // ======================= tensor-memory lane quarters: softmax and exchange =======================
    if (a.kv_early) pdl_wait();
    const int q = warp & 3;                              // lane quarter
    const int set = warp >> 2;                           // 0: warps 0-3, 1: warps 4-7
    const int h = 32 * q + lane;                         // head = tensor-memory lane
    const bool own = (uint32_t)(q >> 1) == c;            // this CTA's heads
    const int hl = h & 63;                               // head index within its CTA's 64
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const uint32_t t_s = tmem + lane_base + AP_S_COL, t_q = tmem + lane_base + AP_Q_COL;
    const uint32_t t_o = tmem + lane_base + AP_O_COL;
    int sb = 0, tlo, thi, seg = 0;
    long long n = 0;
    bool ok = true;
    // tcgen05.ld / tcgen05.st are warp-collective: a warp rescales when any of its lanes (heads)
    // needs it, the others multiply by 1; the decision is never taken per lane.
    auto rescale_o = [&](float alpha, int c0, int nc) {
      __syncwarp();
      for (int cb = c0; cb < c0 + nc; cb += 32) {
        uint32_t r[32];
        tc::tmem_ld32(t_o + cb, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
        tc::tmem_st32(t_o + cb, r);
      }
    };
    // columns [c0, c0 + nc) of this lane's O, times inv, to po
    auto store_o = [&](float* po, float inv, int c0, int nc) {
      __syncwarp();
      for (int cb = c0; cb < c0 + nc; cb += 32) {
        uint32_t r[32];
        tc::tmem_ld32(t_o + cb, r);
        tc::tmem_wait_ld();
        // a lane writes its own head's row: one 32-byte sector per store
#pragma unroll
        for (int j = 0; j < 32; j += 8)
          tc::st_global_v8(po + cb + j, __uint_as_float(r[j]) * inv, __uint_as_float(r[j + 1]) * inv,
                           __uint_as_float(r[j + 2]) * inv, __uint_as_float(r[j + 3]) * inv,
                           __uint_as_float(r[j + 4]) * inv, __uint_as_float(r[j + 5]) * inv,
                           __uint_as_float(r[j + 6]) * inv, __uint_as_float(r[j + 7]) * inv);
      }
    };
    // The next segment's latent queries of this thread into L2 while this segment runs (the
    // lines that `queries` below loads at its end).
    auto prefetch_next = [&]() {
      PairSegIter pk = it;
      int qb, x0, x1;
      if (!pk.next(a, &qb, &x0, &x1)) return;
      const char* p =
          reinterpret_cast<const char*>(a.q_abs + ((size_t)qb * AP_HEADS + h) * 576 + 256 * c + 128 * set);
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p + 128));
    };
    // this thread's share of the latent queries of sequence qb, then arrival on q_full: half of
    // its head's 256 columns (the two warps on each lane quarter split them by `set`)
    auto queries = [&](int qb) {
      __syncwarp();
      tc::tc_fence_after();
      load_q_lat(a, c, qb, h, 128 * set, t_q);
      tc::tmem_wait_st();
      tc::tc_fence_before();
      tc::mbar_arrive(&s.q_full);
    };
    if (own) {
      // ---------------- softmax of this CTA's head h, rows [32 set, 32 set + 32) of each tile ----------------
      const int k = set;
      uint8_t* prow = pbuf + h * 128;                    // this head's row of P (buffer 0)
      const uint32_t pr_pbuf = tc::mapa(tc::smem_u32(pbuf), peer);
      const uint32_t pr_alpha = tc::mapa(tc::smem_u32(&s.alpha_recv[0][0]), peer);
      const uint32_t pr_px_full = tc::mapa(tc::smem_u32(&s.px_full[0]), peer);
      const uint32_t pr_l = tc::mapa(tc::smem_u32(&s.l_recv[0][0]), peer);
      const uint32_t pr_l_full0 = tc::mapa(tc::smem_u32(&s.l_full[0]), peer);
      const bool leader = hl == 0 && k == 0;
      int n_sent = 0, n_got = 0, l_sent = 0;
      float m = -CUDART_INF_F, l = 0.f;                  // running max (log2 units), this half's sum
      {
        PairSegIter pk = it;
        int qb, x0, x1;
        if (pk.next(a, &qb, &x0, &x1)) queries(qb);
      }
      while (ok && it.next(a, &sb, &tlo, &thi)) {
        fail_b = sb;
        const long long L = a.seq_lens[sb];
        m = -CUDART_INF_F;
        l = 0.f;
        prefetch_next();
        for (int t = tlo; t < thi; ++t, ++n) {
          const bool first = t == tlo, last = t + 1 == thi;
          const int b = (int)(n & 1);
          const int nvalid = (int)min((long long)AP_TILE, L - (long long)t * AP_TILE);
          if (!group_wait(s, &s.s_full[b], (uint32_t)((n >> 1) & 1), AP_BAR_OWN, AP_N_OWN, a.wait_ns)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          uint32_t r[32];
          tc::tmem_ld32(t_s + (uint32_t)b * AP_TILE + 32 * k, r);
          tc::tmem_wait_ld();
          tc::tc_fence_before();
          tc::mbar_arrive(&s.s_free[b]);
          if (nvalid < AP_TILE) {
            // rows past the sequence: zero this CTA's latent columns of them, so that
            // 0 * (stale or NaN) cannot reach O (QK^T of the tile has completed: s_full above)
            uint8_t* stg = stages + (int)(n % AP_STAGES) * AP_STAGE;
            const int nz = (AP_TILE - nvalid) * 4 * 8;
            for (int i = hl + 64 * k; i < nz; i += AP_N_OWN) {
              const int row = nvalid + i / 32, blk = (i / 8) & 3, ch = i & 7;
              *reinterpret_cast<uint4*>(stg + blk * AP_BLK + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            }
            tc::fence_proxy_async_smem();
          }
          if (!group_wait(s, &s.srecv_full[b], (uint32_t)((n >> 1) & 1), AP_BAR_OWN, AP_N_OWN, a.wait_ns, true)) {
            ok = false;
            break;
          }
          float sv[32];
          const uint8_t* rb = srecv + b * AP_SBUF;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const float4 v = *reinterpret_cast<const float4*>(rb + swz(hl, 8 * k + kk, 256));
            sv[4 * kk + 0] = __uint_as_float(r[4 * kk + 0]) + v.x;
            sv[4 * kk + 1] = __uint_as_float(r[4 * kk + 1]) + v.y;
            sv[4 * kk + 2] = __uint_as_float(r[4 * kk + 2]) + v.z;
            sv[4 * kk + 3] = __uint_as_float(r[4 * kk + 3]) + v.w;
          }
          ++n_got;
          float mt = -CUDART_INF_F;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            sv[j] = 32 * k + j < nvalid ? sv[j] * a.scale_log2 : -CUDART_INF_F;
            mt = fmaxf(mt, sv[j]);
          }
          s.xch[k][hl] = mt;
          group_bar(AP_BAR_OWN, AP_N_OWN);   // the received scores are read; both halves' maxima are in
          if (leader) tc::mbar_arrive(&s.srecv_read[b]);   // the forwarder re-arms and grants
          mt = fmaxf(s.xch[0][hl], s.xch[1][hl]);   // the same in both halves: same decisions
          float alpha = 1.f;
          if (first || mt > m + AP_RESCALE) {
            const float mn = fmaxf(m, mt);
            if (!first) alpha = ex2(m - mn);
            l *= alpha;
            m = mn;
          }
          uint32_t pk[16];
          float ps = 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float p0 = 32 * k + j < nvalid ? ex2(sv[j] - m) : 0.f;
            const float p1 = 32 * k + j + 1 < nvalid ? ex2(sv[j + 1] - m) : 0.f;
            ps += p0 + p1;
            pk[j >> 1] = pack_bf16x2(p0, p1);
          }
          l += ps;
          // P buffer b (here and in the peer) is free once PV of tile n - 2 is done in both CTAs
          if (n >= 2 && !group_wait(s, &s.pfree[b], (uint32_t)(((n >> 1) - 1) & 1), AP_BAR_OWN, AP_N_OWN,
                                    a.wait_ns, true)) {
            ok = false;
            break;
          }
          // this head's 32 probabilities: 16-byte chunks 4k..4k+3 of its 128-byte row of P
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            *reinterpret_cast<uint4*>(prow + b * AP_PBUF + (((4 * k + kk) ^ (h & 7)) << 4)) =
                make_uint4(pk[4 * kk], pk[4 * kk + 1], pk[4 * kk + 2], pk[4 * kk + 3]);
          if (k == 0) s.alpha_send[b][hl] = alpha;
          tc::fence_proxy_async_smem();
          // O may be rescaled once PV of tile n - 1 is done (the group decides together)
          if (group_vote_or(alpha != 1.f, AP_BAR_OWN, AP_N_OWN)) {
            if (!group_wait(s, &s.pv_done[(n - 1) & 1], (uint32_t)(((n - 1) >> 1) & 1), AP_BAR_OWN, AP_N_OWN,
                            a.wait_ns)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            rescale_o(alpha, 128 * k, 128);
            tc::tmem_wait_st();
          }
          group_bar(AP_BAR_OWN, AP_N_OWN);   // this CTA's rows of P and the factors are written
          if (leader) {
            tc::bulk_s2s(pr_pbuf + b * AP_PBUF + 64 * c * 128, tc::smem_u32(pbuf + b * AP_PBUF + 64 * c * 128),
                         64 * 128, pr_px_full + 8 * b);
            tc::bulk_s2s(pr_alpha + b * 256, tc::smem_u32(&s.alpha_send[b][0]), 256, pr_px_full + 8 * b);
          }
          ++n_sent;
          tc::tc_fence_before();
          tc::mbar_arrive(&s.pv_ready[b]);
          if (last) {
            // QK^T of the segment completed before its last scores were read: the latent queries
            // may be replaced by the next segment's, off the path of this tile's probabilities and
            // overlapping the wait for its PV
            PairSegIter pk = it;
            int qb, x0, x1;
            if (pk.next(a, &qb, &x0, &x1)) queries(qb);
            // ---- epilogue of the segment: this head's lse and its half of O ----
            s.xch[k][hl] = l;
            group_bar(AP_BAR_OWN, AP_N_OWN);
            const float lt = s.xch[0][hl] + s.xch[1][hl];
            const float inv = 1.0f / lt;
            if (k == 0) {
              tc::st_async_b32(pr_l + 4 * ((seg & 1) * 64 + hl), __float_as_uint(inv), pr_l_full0 + 8 * (seg & 1));
              ++l_sent;
            }
            if (!group_wait(s, &s.o_full, (uint32_t)(seg & 1), AP_BAR_OWN, AP_N_OWN, a.wait_ns)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const int slot = pair + sb;
            if (k == 0) {
              const bool bad = *reinterpret_cast<volatile int*>(&s.bad_page[seg & 3]) != 0;
              a.part_lse[(size_t)slot * AP_HEADS + h] =
                  bad ? CUDART_NAN_F : (m + __log2f(lt)) * 0.69314718055994530942f;
            }
            store_o(a.part_o + ((size_t)slot * AP_HEADS + h) * 512 + 256 * c, inv, 128 * k, 128);
            tc::tc_fence_before();
            group_bar(AP_BAR_OWN, AP_N_OWN);   // bad_page read, xch free
            if (leader) s.bad_page[seg & 3] = 0;
            tc::mbar_arrive(&s.o_empty);
          }
        }
        if (!ok) break;
        ++seg;
      }
      if (!ok) pair_fail(s, a.hdr, fail_b, peer);
      if (leader) {
        s.sent[1] = n_sent;   // P
        s.sent[2] = l_sent;
        s.got[0] = n_got;     // scores
      }
    } else if (set == 0) {
      // ---------------- the peer's head h: send this CTA's partial scores ----------------
      const uint32_t pr_srecv = tc::mapa(tc::smem_u32(srecv), peer);
      const uint32_t pr_srecv_full = tc::mapa(tc::smem_u32(&s.srecv_full[0]), peer);
      int n_sent = 0;
      {
        PairSegIter pk = it;
        int qb, x0, x1;
        if (pk.next(a, &qb, &x0, &x1)) queries(qb);
      }
      while (ok && it.next(a, &sb, &tlo, &thi)) {
        fail_b = sb;
        prefetch_next();
        for (int t = tlo; t < thi; ++t, ++n) {
          const int b = (int)(n & 1);
          if (!group_wait(s, &s.s_full[b], (uint32_t)((n >> 1) & 1), AP_BAR_SEND, AP_N_SEND, a.wait_ns)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          uint32_t ra[32], rb[32];
          tc::tmem_ld32(t_s + (uint32_t)b * AP_TILE, ra);
          tc::tmem_ld32(t_s + (uint32_t)b * AP_TILE + 32, rb);
          tc::tmem_wait_ld();
          tc::tc_fence_before();
          tc::mbar_arrive(&s.s_free[b]);
          // the peer has read what we sent into this buffer two tiles ago (and so the bulk copy
          // out of our staging buffer b has completed)
          if (n >= 2 && !group_wait(s, &s.srecv_grant[b], (uint32_t)(((n >> 1) - 1) & 1), AP_BAR_SEND, AP_N_SEND,
                                    a.wait_ns, true)) {
            ok = false;
            break;
          }
          uint8_t* sbuf = ssend + b * AP_SBUF;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            *reinterpret_cast<uint4*>(sbuf + swz(hl, kk, 256)) = make_uint4(ra[4 * kk], ra[4 * kk + 1], ra[4 * kk + 2],
                                                                           ra[4 * kk + 3]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            *reinterpret_cast<uint4*>(sbuf + swz(hl, 8 + kk, 256)) = make_uint4(rb[4 * kk], rb[4 * kk + 1],
                                                                               rb[4 * kk + 2], rb[4 * kk + 3]);
          tc::fence_proxy_async_smem();
          group_bar(AP_BAR_SEND, AP_N_SEND);
          if (hl == 0)
            tc::bulk_s2s(pr_srecv + b * AP_SBUF, tc::smem_u32(sbuf), AP_SBUF, pr_srecv_full + 8 * b);
          ++n_sent;
          if (t + 1 == thi) {
            // the segment's QK^T is complete (its last scores are read): load the next one's
            // queries once this tile's scores are on their way to the peer
            PairSegIter pk = it;
            int qb, x0, x1;
            if (pk.next(a, &qb, &x0, &x1)) queries(qb);
          }
        }
        if (!ok) break;
        ++seg;
      }
      if (!ok) pair_fail(s, a.hdr, fail_b, peer);
      if (hl == 0) s.sent[0] = n_sent;   // scores
    } else {
      // ---------------- the peer's head h: its rescale factors, epilogue ----------------
      int n_got = 0, l_got = 0;
      {
        PairSegIter pk = it;
        int qb, x0, x1;
        if (pk.next(a, &qb, &x0, &x1)) queries(qb);
      }
      while (ok && it.next(a, &sb, &tlo, &thi)) {
        fail_b = sb;
        prefetch_next();
        for (int t = tlo; t < thi; ++t, ++n) {
          const bool last = t + 1 == thi;
          const int b = (int)(n & 1);
          if (!group_wait(s, &s.px_full[b], (uint32_t)((n >> 1) & 1), AP_BAR_RECV, AP_N_RECV, a.wait_ns, true)) {
            ok = false;
            break;
          }
          const float alpha = s.alpha_recv[b][hl];
          ++n_got;
          group_bar(AP_BAR_RECV, AP_N_RECV);   // every receiver has read its factor
          // re-armed before this CTA's PV of tile n can run, and so before the peer may send into
          // this buffer again (it waits for that PV)
          if (hl == 0) tc::mbar_arrive_expect_tx(&s.px_full[b], AP_PX_BYTES);
          if (group_vote_or(alpha != 1.f, AP_BAR_RECV, AP_N_RECV)) {
            if (!group_wait(s, &s.pv_done[(n - 1) & 1], (uint32_t)(((n - 1) >> 1) & 1), AP_BAR_RECV, AP_N_RECV,
                            a.wait_ns)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            rescale_o(alpha, 0, 256);
            tc::tmem_wait_st();
          }
          tc::tc_fence_before();
          tc::mbar_arrive(&s.pv_ready[b]);
          if (last) {
            // The peer's probabilities of this tile came from this CTA's scores of it, so the
            // segment's QK^T has completed: the second half of the next segment's queries.
            PairSegIter pk = it;
            int qb, x0, x1;
            if (pk.next(a, &qb, &x0, &x1)) queries(qb);
            // ---- epilogue of the segment for the peer's head: its 1/l comes from the peer ----
            if (!group_wait(s, &s.o_full, (uint32_t)(seg & 1), AP_BAR_RECV, AP_N_RECV, a.wait_ns)) {
              ok = false;
              break;
            }
            if (!group_wait(s, &s.l_full[seg & 1], (uint32_t)((seg >> 1) & 1), AP_BAR_RECV, AP_N_RECV, a.wait_ns,
                            true)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const float inv = s.l_recv[seg & 1][hl];
            ++l_got;
            group_bar(AP_BAR_RECV, AP_N_RECV);
            if (hl == 0) tc::mbar_arrive_expect_tx(&s.l_full[seg & 1], 64 * 4);
            const int slot = pair + sb;
            store_o(a.part_o + ((size_t)slot * AP_HEADS + h) * 512 + 256 * c, inv, 0, 256);
            tc::tc_fence_before();
            tc::mbar_arrive(&s.o_empty);
          }
        }
        if (!ok) break;
        ++seg;
      }
      if (!ok) pair_fail(s, a.hdr, fail_b, peer);
      if (hl == 0) {
        s.got[1] = n_got;     // P
        s.got[2] = l_got;
      }
    }
  }

  // ---- leave: no transfer may still be landing in either CTA's shared memory ----
  __syncwarp();
  tc::tc_fence_before();
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < 3; ++i) tc::st_cluster_u32(tc::mapa(tc::smem_u32(&s.peer_sent[i]), peer), (uint32_t)s.sent[i]);
  __syncwarp();   // the cluster barrier is warp-collective: warp 0 reconverges after thread 0's stores
  tc::cluster_sync();
  if (tid == 0) {
    // every transfer the peer issued into this CTA has landed (each has its phase armed: the peer
    // only sends after this CTA has armed the barrier and released the buffer)
    for (int k = s.got[0]; k < s.peer_sent[0]; ++k)
      tc::mbar_wait_cluster(&s.srecv_full[k & 1], (uint32_t)((k >> 1) & 1), AP_DRAIN);
    for (int k = s.got[1]; k < s.peer_sent[1]; ++k)
      tc::mbar_wait_cluster(&s.px_full[k & 1], (uint32_t)((k >> 1) & 1), AP_DRAIN);
    for (int k = s.got[2]; k < s.peer_sent[2]; ++k)
      tc::mbar_wait_cluster(&s.l_full[k & 1], (uint32_t)((k >> 1) & 1), AP_DRAIN);
  }
  __syncwarp();
  tc::cluster_sync();
  if (warp == ap_mma_warp(c)) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, AP_TMEM_COLS);
  }
  // After an abort some partials are missing or stale: mark this CTA's heads invalid in every
  // slot of the pair's share (lse = NaN), so the affected outputs come out NaN.
  if (*reinterpret_cast<volatile int*>(&s.abort)) {
    PairSegIter jt{s.seg_b0, s.seg_p0, r0, r1};
    int jb = 0, jlo, jhi;
    while (jt.next(a, &jb, &jlo, &jhi))
      for (int hh = tid; hh < 64; hh += AP_THREADS)
        a.part_lse[(size_t)(pair + jb) * AP_HEADS + 64 * c + hh] = CUDART_NAN_F;
  }
}

}  // namespace

bool attn_pair_supported(const mla_config& cfg) {
  return cfg.act_dtype == MLA_BF16 && cfg.kv_lora == 512 && cfg.qk_rope == 64 && cfg.n_heads == AP_HEADS &&
         (cfg.page_size == 0 || cfg.page_size % AP_TILE == 0) && tma_encoder_available();
}

static cudaLaunchConfig_t pair_launch_config(int grid, cudaStream_t st, cudaLaunchAttribute* at, bool pdl) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(AP_THREADS);
  lc.dynamicSmemBytes = AP_SMEM_DYN;
  lc.stream = st;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = pdl ? 2 : 1;
  return lc;
}

// Pairs of SMs that can hold the kernel at once (one cluster of two CTAs each), per device.
int attn_pair_max_pairs() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  if (ensure_smem((const void*)attn_pair_kernel, AP_SMEM_DYN) != cudaSuccess) return -1;
  cudaLaunchAttribute at[2];
  const int sms = device_sms();
  cudaLaunchConfig_t lc = pair_launch_config(2 * (sms / 2 > 0 ? sms / 2 : 1), nullptr, at, false);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void*)attn_pair_kernel, &lc) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();
    return -1;
  }
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

cudaError_t launch_attn_pair(const mla_config& cfg, const mla_cache& cache, const DecodePlan& plan,
                             const int32_t* seq_lens, const void* q_abs, const void* q_res, float* part_o,
                             float* part_lse, int32_t* meta, int B, WsHeader* hdr, bool kv_early, cudaStream_t st) {
  if (cache.n_physical_rows >= (int64_t(1) << 31) || (int64_t)B * cfg.n_heads >= (int64_t(1) << 31))
    return cudaErrorInvalidValue;
  if (q_res == nullptr) return cudaErrorInvalidValue;
  CUtensorMap rows_map, rope_map, qrope_map, qres_map;
  if (!make_map_row_blocks_bf16(&rows_map, cache.rows, 576, (uint64_t)cache.n_physical_rows, 8, AP_TILE, 4) ||
      !make_map_2d_bf16(&rope_map, cache.rows, 576, (uint64_t)cache.n_physical_rows, 32, AP_TILE, 64) ||
      !make_map_2d_bf16(&qrope_map, q_abs, 576, (uint64_t)B * cfg.n_heads, 32, AP_HEADS, 64) ||
      !make_map_2d_bf16(&qres_map, q_res, 576, (uint64_t)B * cfg.n_heads, 32, AP_HEADS, 64))
    return cudaErrorInvalidValue;
  PairArgs a;
  a.map = RowMap{cache.page_table, cfg.page_size, cfg.max_pages_per_seq, cfg.rows_per_seq, cache.n_physical_rows};
  a.seq_lens = seq_lens;
  a.q_abs = static_cast<const uint16_t*>(q_abs);
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.meta = meta;
  a.hdr = hdr;
  a.B = B;
  a.n_pairs = plan.ctas_per_group;
  a.n_slots = plan.n_slots;
  a.scale_log2 = cfg.softmax_scale * 1.4426950408889634f;
  a.wait_ns = wait_limit_ns();
  a.kv_early = kv_early ? 1 : 0;
  cudaError_t e = ensure_smem((const void*)attn_pair_kernel, AP_SMEM_DYN);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute at[2];
  cudaLaunchConfig_t lc = pair_launch_config(2 * plan.ctas_per_group, st, at, true);
  return cudaLaunchKernelEx(&lc, attn_pair_kernel, rows_map, rope_map, qrope_map, qres_map, a);
}

}  // namespace mla
