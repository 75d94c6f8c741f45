// Split attention over compressed bf16 cache rows on the 5th-generation tensor cores (tcgen05).
//
// turbospark-runtime 0.3.0, src/families/deepseek2/attn.rs, MQA attention over the compressed
// rows (key = whole row [kv_lat ; k_pe], value = its first kv_lora elements, all heads read the
// same rows); moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs, mla_sdpa_folded.
//
// Shape: rows of 576 = 512 latent + 64 rope, bf16. One CTA per SM streams 128-row tiles of the
// cache through shared memory with TMA and computes, for a group of HG heads at once (HG = 64;
// 16 or 32 when the model has that few heads),
//     S^T = K_tile . Q^T          (M = 128 rows, N = HG heads, K = 576)    K-major operands
//     O^T += V_tile^T . P^T       (M = 4 x 128 latent, N = HG heads, K = 128 rows)  MN-major
// with both accumulators in TMEM (S^T 2 x HG columns, O^T 4 x HG columns). The row tile is the
// A operand of both products, so every staged row is shared by all heads of the group and read
// from shared memory twice. The tile's nine 64-column blocks live in nine 16 KB slots; the rope slot
// is reused for P^T once QK^T has read it, and each pair of latent slots is handed back to the
// TMA producer as soon as its 128-column chunk of PV has completed, so the next tile streams in
// while this one finishes.
//
// Softmax: one thread per tile row in each of one or two warpgroups (HG = 64: two, each owning
// 32 heads, so two warps share every SM sub-partition), log2 domain, with a per-head running
// maximum that is only raised when a score exceeds it by more than 2^16: the exact column max
// (a cross-thread reduction) and the rescale of O^T in TMEM happen on the first tile of a
// segment and on those rare tiles only. Each thread keeps per-head partial sums of p; they are
// reduced once per segment.
//
// Work split: the tiles of all sequences form one list per head group; CTA k of a group takes
// the k-th equal share of it (crossing sequence boundaries), so every SM gets the same number of
// tiles whatever the length mix. Each (CTA, sequence) piece writes a partial (O normalised, lse)
// into slot k + b, and the combine stage merges the slots of a sequence.
//
// Roles: warps 0-1 issue the TMA loads (alternate 64-column blocks of each tile; one issuing
// thread alone streams well below what an SM can take in), warp 2 owns TMEM and issues the MMAs
// (one thread), the remaining warps do the softmax and the epilogue. Every mbarrier wait is
// bounded; on a timeout the CTA records MLA_ERR_TIMEOUT, every role stops, and TMEM is freed
// before exit.
#include "common.cuh"
#include "tc_ptx.cuh"

#include <climits>
#include <cudaTypedefs.h>
#include <math_constants.h>

namespace mla {

namespace {

constexpr int TC_TILE = 128;       // rows per tile (MMA M)
constexpr int TC_KB = 9;           // 64-column blocks per row (576 / 64)
constexpr int TC_LAT_KB = 8;       // latent blocks (512 / 64)
constexpr int TC_SLOT_BYTES = TC_TILE * 128;   // 16 KB
constexpr int TC_PRODUCERS = 2;   // TMA producer warps (a single issuing thread tops out near 45 GB/s)
constexpr int TC_MMA_WARP = TC_PRODUCERS;
constexpr int TC_SM_WARP0 = TC_PRODUCERS + 1;   // first softmax warp
// Drain waits (copies and MMAs already issued, before the CTA exits) always get the full
// limit; the main-loop waits get the launch's wait_ns (normally the same 200 ms).
constexpr uint64_t WAIT_NS = kWaitDrainNs;

// Per head-group width HG (the MMA N: 16, 32 or 64 heads per CTA).
template <int HG>
struct Cfg {
  static constexpr int QBLK_BYTES = HG * 128;                 // one 64-column block of Q
  // Q blocks: 9 of the bf16 fused query rows + the bf16 residual of the rope block, so the
  // rope part of every score is exact to ~2^-16 (hi + lo)
  static constexpr int Q_BLOCKS = TC_KB + 1;
  // softmax warpgroups: each owns HW = HG / NWG heads of every tile row (four warps, one per
  // TMEM lane quarter)
  static constexpr int NWG = HG == 64 ? 2 : 1;
  static constexpr int HW = HG / NWG;
  static constexpr int THREADS = 32 * TC_SM_WARP0 + 128 * NWG;
  static constexpr int SMEM_DYN = TC_KB * TC_SLOT_BYTES + Q_BLOCKS * QBLK_BYTES + 1024;
  static constexpr uint32_t O_COL = 0;                        // O^T chunks: 4 x HG columns
  static constexpr uint32_t S_COL = 4 * HG;                   // S^T buffers: 2 x HG columns
  static constexpr uint32_t TMEM_COLS = HG == 64 ? 512 : (HG == 32 ? 256 : 128);
  static constexpr int P_ROW = 2 * HG;                        // bytes of one P^T row (bf16)
  // P^T is MN-major with rows of P_ROW bytes: 128-, 64- or 32-byte swizzle
  static constexpr uint32_t P_LAYOUT = HG == 64 ? 2u : (HG == 32 ? 4u : 6u);
  static __device__ __forceinline__ uint32_t p_offset(uint32_t row, uint32_t chunk) {
    if (HG == 64) return row * 128u + ((chunk ^ (row & 7u)) << 4);
    if (HG == 32) return row * 64u + ((chunk ^ ((row >> 1) & 3u)) << 4);
    return row * 32u + ((chunk ^ ((row >> 2) & 1u)) << 4);
  }
};
constexpr int TC_HG_MAX = 64;
constexpr float RESCALE_THRESHOLD = 16.0f;  // log2 units: p may reach 2^16 before a rescale

struct TcArgs {
  RowMap map;
  const int32_t* seq_lens;
  float* part_o;          // [G][n_slots][64][C]
  float* part_lse;        // [G][n_slots][64]
  int32_t* meta;          // [B][2]: first slot, slot count
  WsHeader* hdr;
  int B, H, G, ncg, n_slots;
  float scale_log2;
  uint64_t wait_ns;       // limit of the main-loop waits
  // 1: the kernel launched just before this one started only after all earlier work on the
  // stream had completed, and writes no cache row; cache rows may then be read before the
  // dependency wait (only the queries wait for it)
  int kv_early;
  // query tokens per sequence (heads token-major, kvb_heads per token): head m sees the rows
  // before L - tokens + 1 + m / kvb_heads; one token: every head sees the L rows
  int tokens, kvb_heads;
};

struct Smem {
  static constexpr int TC_HG = TC_HG_MAX;   // arrays sized for the widest group
  uint64_t full[TC_KB], empty[TC_KB];
  uint64_t q_full, q_empty;
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, o_done, o_empty, mma_fin;
  uint32_t tmem_base;
  int abort;
  int seg_b0;
  long long seg_p0;
  int bad_page[2][2];     // [segment parity][warpgroup]: the producers run at most one segment ahead
  float red[4][TC_HG];
  float m2[TC_HG];        // running max per head, log2 units
  float alpha[TC_HG];     // rescale factors (then 1/l in the epilogue)
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// OR of `v` over the 128 threads of softmax warpgroup `wg` (named barrier 1 + wg), returned to
// all of them.
__device__ __forceinline__ bool softmax_vote_or(bool v, int wg) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\t"
      "setp.ne.u32 pi, %1, 0;\n\t"
      "barrier.red.or.pred po, %2, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"((uint32_t)v), "r"(1 + wg)
      : "memory");
  return out != 0;
}

__device__ __forceinline__ void softmax_bar(int wg) {
  __syncwarp();
  asm volatile("barrier.sync %0, 128;" ::"r"(1 + wg) : "memory");
}


__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Tiles a sequence contributes (0 for an invalid length: below one row per query token, or
// past the capacity).
__device__ __forceinline__ long long seq_tiles(const TcArgs& a, int b) {
  const long long L = a.seq_lens[b];
  if (L < a.tokens || L < 1 || L > a.map.capacity()) return 0;
  return (L + TC_TILE - 1) / TC_TILE;
}

// Tile range [r0, r1) of CTA k among ncg CTAs sharing T tiles.
__device__ __forceinline__ void cta_range(long long T, int k, int ncg, long long* r0, long long* r1) {
  *r0 = (T * k) / ncg;
  *r1 = (T * (k + 1)) / ncg;
}

// A bounded wait (limit_ns) that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_bar(Smem& s, uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = tc::global_ns();
  for (uint32_t i = 0;; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 15) == 15) {
      if (*reinterpret_cast<volatile int*>(&s.abort)) return false;
      if (tc::global_ns() - t0 > limit_ns) return false;
    }
  }
}

// Softmax-side wait: every softmax thread polls the barrier itself (a warp whose lane 0 alone
// polled would run split afterwards: collective operations then serialise and the warp's
// arrivals at the group barrier stop lining up), then the warpgroup's 128 threads agree on the
// outcome, so they always leave (or stay in) their loops together and never strand a barrier.
__device__ __forceinline__ bool softmax_wait(Smem& s, uint64_t* bar, uint32_t parity, int wg, uint64_t limit_ns) {
  const bool ok = wait_bar(s, bar, parity, limit_ns);
  __syncwarp();
  return !softmax_vote_or(!ok, wg);
}

__device__ __forceinline__ void fail(Smem& s, WsHeader* hdr, int b) {
  if (atomicExch(&s.abort, 1) == 0) set_error(hdr, MLA_ERR_TIMEOUT, b);
}

// Segment iterator: walks the (sequence, tile range) pieces of this CTA's share.
struct SegIter {
  int b;
  long long p;      // first global tile of sequence b
  long long r0, r1; // this CTA's range
  __device__ bool next(const TcArgs& a, int* sb, int* t_lo, int* t_hi) {
    while (b < a.B && p < r1) {
      const long long n = seq_tiles(a, b);
      const long long lo = max(r0, p), hi = min(r1, p + n);
      const int cur = b;
      const long long pb = p;
      ++b;
      p += n;
      if (hi > lo) {
        *sb = cur;
        *t_lo = (int)(lo - pb);
        *t_hi = (int)(hi - pb);
        return true;
      }
    }
    return false;
  }
};

template <int HG>
__global__ void __launch_bounds__(Cfg<HG>::THREADS, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap rows_map, const __grid_constant__ CUtensorMap q_map,
               const __grid_constant__ CUtensorMap qres_map, TcArgs a) {
  extern __shared__ uint8_t dyn_raw[];
  __shared__ Smem s;
  pdl_trigger();
  uint8_t* dyn = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* slots = dyn;                                 // 9 x 16 KB
  uint8_t* qs = dyn + TC_KB * TC_SLOT_BYTES;            // 10 Q blocks
  // prologue scratch: the slots are free until the first TMA load
  long long* scan = reinterpret_cast<long long*>(slots);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.x % a.G;
  const int k = blockIdx.x / a.G;

  // ---- every thread: total tile count (block scan over per-thread chunks of sequences) ----------
  constexpr int NT = Cfg<HG>::THREADS;
  const int chunk = (a.B + NT - 1) / NT;
  const int cb0 = min(a.B, tid * chunk), cb1 = min(a.B, cb0 + chunk);
  long long mine = 0;
  for (int b = cb0; b < cb1; ++b) mine += seq_tiles(a, b);
  long long incl = mine;   // inclusive scan within the warp, then across the six warp totals
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
    s.bad_page[0][0] = s.bad_page[0][1] = 0;
    s.bad_page[1][0] = s.bad_page[1][1] = 0;
  }
  __syncwarp();
  __syncthreads();
  long long before = incl - mine, T = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    const long long v = scan[w];
    if (w < warp) before += v;
    T += v;
  }
  long long r0, r1;
  cta_range(T, k, a.ncg, &r0, &r1);
  // on-chip set-up (barriers, TMEM, tensor-map prefetch) overlaps the previous kernel
  if (r0 < r1) {
    if (tid == 0) {
      for (int i = 0; i < TC_KB; ++i) {
        tc::mbar_init(&s.full[i], 1);
        tc::mbar_init(&s.empty[i], 1);
      }
      tc::mbar_init(&s.q_full, 1);
      tc::mbar_init(&s.q_empty, 1);
      for (int i = 0; i < 2; ++i) {
        tc::mbar_init(&s.s_full[i], 1);
        tc::mbar_init(&s.s_empty[i], 128 * Cfg<HG>::NWG);
      }
      tc::mbar_init(&s.p_full, 128 * Cfg<HG>::NWG);
      tc::mbar_init(&s.o_done, 1);
      tc::mbar_init(&s.o_empty, 128 * Cfg<HG>::NWG);
      tc::mbar_init(&s.mma_fin, 1);
      tc::fence_mbar_init();
    }
    if (warp == TC_MMA_WARP) {
      tc::tmem_alloc(&s.tmem_base, Cfg<HG>::TMEM_COLS);
      tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
      tc::tma_prefetch_desc(&rows_map);
      tc::tma_prefetch_desc(&q_map);
      tc::tma_prefetch_desc(&qres_map);
    }
  }
  // the thread whose chunk holds tile r0 finds the first sequence of this CTA's share (the
  // lengths are the caller's input: no kernel of the step writes them)
  if (r0 < r1 && before <= r0 && r0 < before + mine) {
    long long p = before;
    for (int b = cb0; b < cb1; ++b) {
      const long long n = seq_tiles(a, b);
      if (r0 < p + n) {
        s.seg_b0 = b;
        s.seg_p0 = p;
        if constexpr (HG < 64) {   // narrow groups: few heads, short latency-bound attentions
          // Warm L2 and the address translation for this CTA's first tile while the kernel
          // before runs. A prefetch delivers nothing to this SM, and L2 stays coherent with any
          // write to those rows (the appended one) made before the loads that follow the wait.
          if (!a.kv_early) {
            const long long L = a.seq_lens[b], t0 = (r0 - p) * TC_TILE;
            for (int j = 0; j < 2; ++j) {
              const long long lt = t0 + 64 * j;
              const int64_t pr = lt < L ? a.map.phys(b, lt) : -1;
              if (pr >= 0)
                for (int kb = 0; kb < TC_KB; ++kb) tc::tma_prefetch_l2_2d(&rows_map, kb * 64, (int32_t)pr);
            }
          }
        }
        break;
      }
      p += n;
    }
  }
  // Everything below reads what the absorb / append kernels wrote (query rows, the new cache
  // row) or writes what the previous step's combine may still read (meta, partials). In the
  // early mode the only kernel that can still be running is the absorb, which began after all
  // earlier work (append, previous combine) had completed: then only the query loads wait.
  if (!a.kv_early) pdl_wait();
  // CTA 0 of group 0 publishes, per sequence, which partial slots the combine must merge
  if (blockIdx.x == 0) {
    long long p = before;
    for (int b = cb0; b < cb1; ++b) {
      const long long n = seq_tiles(a, b);
      int first = 0, count = 0;
      if (n > 0) {
        // covering CTAs: smallest k with r1_k > p, largest k with r0_k < p + n
        const long long kf = ((p + 1) * a.ncg + T - 1) / T - 1;
        const long long kl = ((p + n) * a.ncg + T - 1) / T - 1;
        first = (int)(kf + b);
        count = (int)(kl - kf + 1);
      } else {
        set_error(a.hdr, MLA_ERR_BAD_SEQ_LEN, b);
      }
      a.meta[2 * b] = first;
      a.meta[2 * b + 1] = count;
      p += n;
    }
  }
  if (r0 >= r1) {
    // Wait even in the early mode: a grid completes only after its predecessor has, also when
    // no CTA has a share.
    pdl_wait();
    // No share. If the empty range sits strictly inside a sequence, this CTA's slot lies in
    // that sequence's slot interval: mark it empty (lse = -inf, weight 0 in the combine).
    if (before <= r0 && r0 < before + mine) {
      long long p = before;
      for (int b = cb0; b < cb1; ++b) {
        const long long n = seq_tiles(a, b);
        if (r0 < p + n) {
          if (p < r0) {
            float* pl = a.part_lse + (size_t)(g * a.n_slots + k + b) * HG;
            for (int h = 0; h < HG; ++h) pl[h] = -CUDART_INF_F;
          }
          break;
        }
        p += n;
      }
    }
    return;   // uniform: every thread computed the same range
  }

  tc::fence_proxy_async_smem();   // the prologue's generic writes to the slots precede TMA writes
  tc::tc_fence_before();
  __syncwarp();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  SegIter it{s.seg_b0, s.seg_p0, r0, r1};

  if (warp < TC_PRODUCERS) {
    // ============================ TMA producers ============================
    // Producer p issues the blocks kb = p, p + 2, ... of every tile (the loads of one tile are
    // spread over two issuing threads); producer 0 also loads each segment's queries.
    if (lane == 0) {
      const int pw = warp;
      int sb = 0, tlo, thi;
      int seg = 0;
      long long n = 0;            // global tile counter of this CTA
      long long last_n[TC_KB];    // last tile loaded into each slot (for the abort drain)
      for (int kb = 0; kb < TC_KB; ++kb) last_n[kb] = -1;
      int q_loaded = -1;
      bool ok = true;
      // cache rows are read once per head group, by CTAs that run side by side: mark them first
      // to leave L2, so that the split partials this kernel writes stay there for the combine
      const uint64_t kv_policy = tc::l2_policy_evict_first();
      auto load_q = [&]() -> bool {
        if (seg > 0 && !wait_bar(s, &s.q_empty, (seg - 1) & 1, a.wait_ns)) return false;
        tc::mbar_arrive_expect_tx(&s.q_full, Cfg<HG>::Q_BLOCKS * Cfg<HG>::QBLK_BYTES);
        const int qrow = sb * a.H + g * HG;
        for (int kb = 0; kb < TC_KB; ++kb)
          tc::tma_load_2d(qs + kb * Cfg<HG>::QBLK_BYTES, &q_map, kb * 64, qrow, &s.q_full);
        tc::tma_load_2d(qs + TC_KB * Cfg<HG>::QBLK_BYTES, &qres_map, TC_LAT_KB * 64, qrow, &s.q_full);
        q_loaded = seg;
        return true;
      };
      while (ok && it.next(a, &sb, &tlo, &thi)) {
        // early mode: the first tile's rows go out before the wait for the absorb's queries
        const bool defer_q = a.kv_early && seg == 0;
        if (pw == 0 && !defer_q && !load_q()) { ok = false; break; }
        const long long L = a.seq_lens[sb];
        for (int t = tlo; t < thi && ok; ++t) {
          const long long t0 = (long long)t * TC_TILE;
          // physical first row of each 64-row half; halves past the sequence are skipped
          int y[2];
          uint32_t bytes = 0;
          for (int j = 0; j < 2; ++j) {
            const long long lt = t0 + 64 * j;
            y[j] = -1;
            if (lt < L) {
              int64_t pr = a.map.phys(sb, lt);
              if (pr < 0) {   // out-of-range page id: load a valid row, flag the segment
                for (int w = 0; w < Cfg<HG>::NWG; ++w) atomicExch(&s.bad_page[seg & 1][w], 1);
                set_error(a.hdr, MLA_ERR_BAD_PAGE, sb);
                pr = 0;
              }
              y[j] = (int)pr;
              bytes += 64 * 128;
            }
          }
          // latent blocks 0..7 in order, the rope block (8) last: the order QK^T consumes them
          for (int kb = pw; kb < TC_KB; kb += TC_PRODUCERS) {
            if (n > 0 && !wait_bar(s, &s.empty[kb], (uint32_t)((n - 1) & 1), a.wait_ns)) { ok = false; break; }
            tc::mbar_arrive_expect_tx(&s.full[kb], bytes);
            for (int j = 0; j < 2; ++j)
              if (y[j] >= 0)
                tc::tma_load_2d_hint(slots + kb * TC_SLOT_BYTES + j * 64 * 128, &rows_map, kb * 64, y[j],
                                     &s.full[kb], kv_policy);
            last_n[kb] = n;
          }
          if (ok && pw == 0 && defer_q && t == tlo) {
            pdl_wait();
            if (!load_q()) ok = false;
          }
          if (ok) ++n;
        }
        if (ok) ++seg;
      }
      if (!ok) fail(s, a.hdr, sb);
      // Wait (bounded) for every copy this thread issued, so none lands after the CTA exits:
      // after an abort of any role the last tiles may never have been consumed. In a clean run
      // they have all landed already and these waits return at once.
      for (int kb = pw; kb < TC_KB; kb += TC_PRODUCERS)
        if (last_n[kb] >= 0) tc::mbar_wait(&s.full[kb], (uint32_t)(last_n[kb] & 1), WAIT_NS);
      if (q_loaded >= 0) tc::mbar_wait(&s.q_full, (uint32_t)(q_loaded & 1), WAIT_NS);
    }
  } else if (warp == TC_MMA_WARP) {
    // ================================ MMA issuer ================================
    if (a.kv_early) pdl_wait();   // only the producers run ahead of the absorb
    if (lane == 0) {
      const uint32_t idesc_qk = tc::idesc_bf16_f32(TC_TILE, HG, 0, 0);
      const uint32_t idesc_pv = tc::idesc_bf16_f32(128, HG, 1, 1);
      const uint32_t slot0 = tc::smem_u32(slots), q0 = tc::smem_u32(qs);
      int sb = 0, tlo, thi;
      int seg = 0;
      long long n = 0;
      bool ok = true;
      while (ok && it.next(a, &sb, &tlo, &thi)) {
        if (!wait_bar(s, &s.q_full, seg & 1, a.wait_ns)) { ok = false; break; }
        tc::tc_fence_after();
        for (int t = tlo; t < thi; ++t, ++n) {
          const int sbuf = (int)(n & 1);
          const uint32_t s_tmem = tmem + Cfg<HG>::S_COL + sbuf * HG;
          if (n >= 2 && !wait_bar(s, &s.s_empty[sbuf], (uint32_t)(((n >> 1) - 1) & 1), a.wait_ns)) { ok = false; break; }
          tc::tc_fence_after();
          for (int i = 0; i < TC_KB; ++i) {
            const int kb = (i < TC_LAT_KB) ? i : TC_LAT_KB;
            if (!wait_bar(s, &s.full[kb], (uint32_t)(n & 1), a.wait_ns)) { ok = false; break; }
            tc::tc_fence_after();
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = tc::sdesc_sw128(slot0 + kb * TC_SLOT_BYTES + kk * 32, 16, 1024);
              const uint64_t bd = tc::sdesc_sw128(q0 + kb * Cfg<HG>::QBLK_BYTES + kk * 32, 16, 1024);
              tc::mma_f16_ss(s_tmem, ad, bd, idesc_qk, (i | kk) != 0);
            }
          }
          if (!ok) break;
          // the rope block once more against the residual of the rope queries (hi + lo)
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t ad = tc::sdesc_sw128(slot0 + TC_LAT_KB * TC_SLOT_BYTES + kk * 32, 16, 1024);
            const uint64_t bd = tc::sdesc_sw128(q0 + TC_KB * Cfg<HG>::QBLK_BYTES + kk * 32, 16, 1024);
            tc::mma_f16_ss(s_tmem, ad, bd, idesc_qk, 1);
          }
          tc::mma_commit(&s.s_full[sbuf]);
          if (t + 1 == thi) tc::mma_commit(&s.q_empty);
          // PV needs P^T (slot 8) and, on a segment's first tile, the previous O^T read out
          if (!wait_bar(s, &s.p_full, (uint32_t)(n & 1), a.wait_ns)) { ok = false; break; }
          if (t == tlo && seg > 0 && !wait_bar(s, &s.o_empty, (uint32_t)((seg - 1) & 1), a.wait_ns)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t p_addr = slot0 + TC_LAT_KB * TC_SLOT_BYTES;
          for (int cc = 0; cc < 4; ++cc) {
            const uint32_t a_base = slot0 + (2 * cc) * TC_SLOT_BYTES;
            for (int j = 0; j < TC_TILE / 16; ++j) {
              const uint64_t ad = tc::sdesc_sw128(a_base + j * 2048, TC_SLOT_BYTES, 1024);
              const uint64_t bd = tc::sdesc(p_addr + j * 16 * Cfg<HG>::P_ROW, TC_SLOT_BYTES, 8 * Cfg<HG>::P_ROW,
                                            Cfg<HG>::P_LAYOUT);
              tc::mma_f16_ss(tmem + Cfg<HG>::O_COL + cc * HG, ad, bd, idesc_pv, !(t == tlo && j == 0));
            }
            tc::mma_commit(&s.empty[2 * cc]);
            tc::mma_commit(&s.empty[2 * cc + 1]);
          }
          tc::mma_commit(&s.empty[TC_LAT_KB]);
          tc::mma_commit(&s.o_done);
        }
        ++seg;
      }
      if (!ok) fail(s, a.hdr, sb);
      // every MMA issued must finish before TMEM is released
      tc::mma_commit(&s.mma_fin);
      tc::mbar_wait(&s.mma_fin, 0, WAIT_NS);
    }
  } else {
    // ================================ softmax + epilogue ================================
    // Warpgroup wg owns heads [h0, h0 + HW) of every row: its own running maxima, votes and
    // rescales (TMEM columns and P^T chunks of those heads only), its own named barrier.
    constexpr int HW = Cfg<HG>::HW;
    const int wg = (warp - TC_SM_WARP0) >> 2;
    const int h0 = wg * HW;
    const int q = warp & 3;                  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;           // tile row (and O^T latent row within a chunk)
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    if (a.kv_early) pdl_wait();   // only the producers run ahead of the absorb
    const int sidx = (tid - 32 * TC_SM_WARP0) & 127;   // 0..127 within the warpgroup
    int sb = 0, tlo, thi;
    int seg = 0;
    long long n = 0;
    bool ok = true;
    constexpr int CW = HW < 32 ? HW : 32;    // TMEM columns per load
    constexpr int NCH = HW / CW;
    float lp[HW];                            // this row's share of each owned head's sum of p
    uint8_t* prow = slots + TC_LAT_KB * TC_SLOT_BYTES;   // P^T lives in the rope slot
    while (ok && it.next(a, &sb, &tlo, &thi)) {
      const long long L = a.seq_lens[sb];
#pragma unroll
      for (int h = 0; h < HW; ++h) lp[h] = 0.f;
      if (sidx < HW) s.m2[h0 + sidx] = -CUDART_INF_F;
      for (int t = tlo; t < thi; ++t, ++n) {
        const int sbuf = (int)(n & 1);
        const uint32_t s_addr = tmem + lane_base + Cfg<HG>::S_COL + sbuf * HG + h0;
        if (!softmax_wait(s, &s.s_full[sbuf], (uint32_t)((n >> 1) & 1), wg, a.wait_ns)) { ok = false; break; }
        tc::tc_fence_after();
        // Row validity per head: a row at or past L is nobody's; one before L - tokens + 1 is
        // every head's; in between, head m of the sequence sees it iff m >= hthr (the heads of
        // the later tokens). Column j of this group is head g * HG + j of the sequence.
        const long long rg = (long long)t * TC_TILE + row;
        const long long lim0 = L - a.tokens + 1;
        const bool valid = rg < L;
        const int hthr = !valid ? INT_MAX : (rg < lim0 ? 0 : (int)(rg - lim0 + 1) * a.kvb_heads);
        const int hcol0 = g * HG + h0;   // sequence head of this warpgroup's column 0
        const bool first = (t == tlo);
        // PV of the previous tile has completed (its commit preceded this tile's QK commit);
        // waiting keeps the o_done phases in step for every softmax thread
        if (n > 0 && !softmax_wait(s, &s.o_done, (uint32_t)((n - 1) & 1), wg, a.wait_ns)) { ok = false; break; }
        tc::tc_fence_after();
        // pass 1: does any score exceed its head's running max by more than the threshold?
        // (TMEM loads are warp-collective: every lane loads, validity only gates the arithmetic)
        bool need = first;
        for (int half = 0; half < NCH; ++half) {
          uint32_t r[CW];
          tc::tmem_ld<CW>(s_addr + half * CW, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < CW; ++j)
            if (hcol0 + half * CW + j >= hthr)
              need |= fmaf(__uint_as_float(r[j]), a.scale_log2, -s.m2[h0 + half * CW + j]) > RESCALE_THRESHOLD;
        }
        __syncwarp();
        if (softmax_vote_or(need, wg)) {
          // exact per-head maximum over the tile's valid rows; raise the running max
          for (int half = 0; half < NCH; ++half) {
            uint32_t r[CW];
            tc::tmem_ld<CW>(s_addr + half * CW, r);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < CW; ++j) {
              float v = hcol0 + half * CW + j >= hthr ? __uint_as_float(r[j]) * a.scale_log2 : -CUDART_INF_F;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
              if (lane == 0) s.red[q][h0 + half * CW + j] = v;
            }
          }
          softmax_bar(wg);
          if (sidx < HW) {
            const int h = h0 + sidx;
            const float mt = fmaxf(fmaxf(s.red[0][h], s.red[1][h]), fmaxf(s.red[2][h], s.red[3][h]));
            const float mo = s.m2[h];
            const float mn = fmaxf(mo, mt);
            // a head with no visible row yet keeps its (zero) sums: factor 1, not ex2(-inf + inf)
            s.alpha[h] = first ? 0.f : (mn == -CUDART_INF_F ? 1.f : ex2(mo - mn));
            s.m2[h] = mn;
          }
          softmax_bar(wg);
#pragma unroll
          for (int h = 0; h < HW; ++h) lp[h] *= s.alpha[h0 + h];
          if (!first) {
            // rescale the four O^T chunks this thread's TMEM lane holds, owned heads only (PV
            // of the previous tile has completed, see the o_done wait above)
            for (int cc = 0; cc < 4; ++cc) {
              for (int half = 0; half < NCH; ++half) {
                uint32_t r[CW];
                const uint32_t ta = tmem + lane_base + Cfg<HG>::O_COL + cc * HG + h0 + half * CW;
                tc::tmem_ld<CW>(ta, r);
                tc::tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < CW; ++j)
                  r[j] = __float_as_uint(__uint_as_float(r[j]) * s.alpha[h0 + half * CW + j]);
                tc::tmem_st<CW>(ta, r);
              }
            }
            tc::tmem_wait_st();
          }
        }
        // pass 2: probabilities, partial sums, and this row's owned chunks of P^T (MN-major,
        // swizzled rows of 2*HG bytes) into the rope slot, which TMA (async proxy) wrote and
        // QK^T has finished reading
        tc::fence_proxy_async_smem();
        for (int half = 0; half < NCH; ++half) {
          uint32_t r[CW];
          tc::tmem_ld<CW>(s_addr + half * CW, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int c4 = 0; c4 < CW / 8; ++c4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = c4 * 8 + 2 * e;
              const int h = half * CW + j;
              float p0 = 0.f, p1 = 0.f;
              if (hcol0 + h >= hthr) p0 = ex2(fmaf(__uint_as_float(r[j]), a.scale_log2, -s.m2[h0 + h]));
              if (hcol0 + h + 1 >= hthr) p1 = ex2(fmaf(__uint_as_float(r[j + 1]), a.scale_log2, -s.m2[h0 + h + 1]));
              lp[h] += p0;
              lp[h + 1] += p1;
              w[e] = pack_bf16x2(p0, p1);
            }
            *reinterpret_cast<uint4*>(prow + Cfg<HG>::p_offset(row, (h0 + half * CW) / 8 + c4)) =
                make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        // S^T of this tile is fully read: the MMA warp may reuse the buffer
        tc::tc_fence_before();
        tc::mbar_arrive(&s.s_empty[sbuf]);
        if (!valid) {
          // rows past the sequence: zero their latent so 0 * (stale or NaN) cannot reach O^T
          // (the warpgroups share the eight latent slots)
          const uint4 z = make_uint4(0, 0, 0, 0);
          for (int kb = wg; kb < TC_LAT_KB; kb += Cfg<HG>::NWG)
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8)
              *reinterpret_cast<uint4*>(slots + kb * TC_SLOT_BYTES + row * 128 + c8 * 16) = z;
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        tc::mbar_arrive(&s.p_full);
      }
      if (!ok) break;
      // ---- epilogue of the segment: wait for its last PV, normalise, write the partial ----
      if (!softmax_wait(s, &s.o_done, (uint32_t)((n - 1) & 1), wg, a.wait_ns)) { ok = false; break; }
      tc::tc_fence_after();
#pragma unroll
      for (int h = 0; h < HW; ++h) {
        float v = lp[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) s.red[q][h0 + h] = v;
      }
      softmax_bar(wg);
      const int slot = k + sb;
      const int nh = min(HG, a.H - g * HG);
      if (sidx < HW) {
        const int h = h0 + sidx;
        const float l = s.red[0][h] + s.red[1][h] + s.red[2][h] + s.red[3][h];
        // l = 0: no row of this piece is visible to the head (a later token's row range):
        // O stays 0 and lse = -inf, weight 0 in the combine
        s.alpha[h] = l > 0.f ? 1.0f / l : 0.f;
        if (h < nh) {
          const bool bad = *reinterpret_cast<volatile int*>(&s.bad_page[seg & 1][wg]) != 0;
          a.part_lse[(size_t)(g * a.n_slots + slot) * HG + h] =
              bad ? CUDART_NAN_F : (s.m2[h] + __log2f(l)) * 0.69314718055994530942f;
        }
      }
      softmax_bar(wg);
      float* po = a.part_o + ((size_t)(g * a.n_slots + slot) * HG) * 512;
      for (int cc = 0; cc < 4; ++cc) {
        for (int half = 0; half < NCH; ++half) {
          uint32_t r[CW];
          tc::tmem_ld<CW>(tmem + lane_base + Cfg<HG>::O_COL + cc * HG + h0 + half * CW, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < CW; ++j) {
            const int h = h0 + half * CW + j;
            if (h < nh) po[(size_t)h * 512 + cc * 128 + row] = __uint_as_float(r[j]) * s.alpha[h];
          }
        }
      }
      tc::tc_fence_before();
      softmax_bar(wg);   // this warpgroup's s.red / s.alpha / s.m2 free; its threads have read bad_page
      if (sidx == 0) s.bad_page[seg & 1][wg] = 0;
      __syncwarp();
      tc::mbar_arrive(&s.o_empty);
      ++seg;
    }
    if (!ok) fail(s, a.hdr, sb);
  }

  __syncwarp();   // lanes that skipped a role wait here for their lane 0
  tc::tc_fence_before();
  __syncthreads();
  if (warp == TC_MMA_WARP) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, Cfg<HG>::TMEM_COLS);
  }
  // After an abort some of this CTA's partials are missing or stale: mark every partial slot
  // of its share invalid (lse = NaN), so the affected sequences' outputs come out NaN. The
  // slots are this CTA's alone; every role has stopped (the barrier above).
  if (*reinterpret_cast<volatile int*>(&s.abort)) {
    SegIter jt{s.seg_b0, s.seg_p0, r0, r1};
    int sb = 0, tlo, thi;
    while (jt.next(a, &sb, &tlo, &thi))
      for (int h = tid; h < HG; h += Cfg<HG>::THREADS)
        a.part_lse[(size_t)(g * a.n_slots + k + sb) * HG + h] = CUDART_NAN_F;
  }
}

}  // namespace

namespace {

// 2D bf16 map over `rows` rows of 576 elements, boxes of 64 columns x 64 rows, 128-byte swizzle.
bool make_rows_map(CUtensorMap* m, const void* base, uint64_t rows) {
  return make_map_2d_bf16(m, base, 576, rows, 64, 64);
}

}  // namespace

bool attn_tc_supported(const mla_config& cfg) {
  return cfg.act_dtype == MLA_BF16 && cfg.kv_lora == 512 && cfg.qk_rope == 64 &&
         (cfg.page_size == 0 || cfg.page_size % 64 == 0) && tma_encoder_available();
}

// Heads per CTA for H heads: the narrowest group width (16, 32 or 64) that holds all heads,
// else 64-head groups. Narrow groups write proportionally smaller partials.
int tc_heads_per_cta(int H) {
  return H <= 16 ? 16 : (H <= 32 ? 32 : 64);
}


cudaError_t launch_attn_tc(const mla_config& cfg, const mla_cache& cache, const DecodePlan& plan,
                           const int32_t* seq_lens, const void* q_abs, const void* q_res, float* part_o,
                           float* part_lse, int32_t* meta, int B, WsHeader* hdr, bool kv_early, cudaStream_t st) {
  if (cache.n_physical_rows >= (int64_t(1) << 31) || (int64_t)B * cfg.n_heads >= (int64_t(1) << 31))
    return cudaErrorInvalidValue;
  CUtensorMap rows_map, q_map;
  if (!make_rows_map(&rows_map, cache.rows, (uint64_t)cache.n_physical_rows)) return cudaErrorInvalidValue;
  CUtensorMap qres_map;
  if (q_res == nullptr) return cudaErrorInvalidValue;
  if (!make_map_2d_bf16(&q_map, q_abs, 576, (uint64_t)B * cfg.n_heads, 64, (uint32_t)plan.heads_per_cta) ||
      !make_map_2d_bf16(&qres_map, q_res, 576, (uint64_t)B * cfg.n_heads, 64, (uint32_t)plan.heads_per_cta))
    return cudaErrorInvalidValue;
  TcArgs a;
  a.map = RowMap{cache.page_table, cfg.page_size, cfg.max_pages_per_seq, cfg.rows_per_seq, cache.n_physical_rows};
  a.seq_lens = seq_lens;
  a.part_o = part_o;
  a.part_lse = part_lse;
  a.meta = meta;
  a.hdr = hdr;
  a.B = B;
  a.H = cfg.n_heads;
  a.G = plan.n_groups;
  a.ncg = plan.ctas_per_group;
  a.n_slots = plan.n_slots;
  a.scale_log2 = cfg.softmax_scale * 1.4426950408889634f;
  a.kv_early = kv_early ? 1 : 0;
  a.wait_ns = wait_limit_ns();
  a.tokens = plan.tokens;
  a.kvb_heads = plan.kvb_heads;
  if (a.tokens < 1 || a.kvb_heads < 1 || a.tokens * a.kvb_heads != cfg.n_heads) return cudaErrorInvalidValue;
  const int grid = plan.n_groups * plan.ctas_per_group;
  cudaError_t e;
  switch (plan.heads_per_cta) {
    case 64:
      e = ensure_smem((const void*)attn_tc_kernel<64>, Cfg<64>::SMEM_DYN);
      if (e != cudaSuccess) return e;
      e = launch_pdl(attn_tc_kernel<64>, dim3(grid), dim3(Cfg<64>::THREADS), Cfg<64>::SMEM_DYN, st, rows_map, q_map,
                     qres_map, a);
      break;
    case 32:
      e = ensure_smem((const void*)attn_tc_kernel<32>, Cfg<32>::SMEM_DYN);
      if (e != cudaSuccess) return e;
      e = launch_pdl(attn_tc_kernel<32>, dim3(grid), dim3(Cfg<32>::THREADS), Cfg<32>::SMEM_DYN, st, rows_map, q_map,
                     qres_map, a);
      break;
    case 16:
      e = ensure_smem((const void*)attn_tc_kernel<16>, Cfg<16>::SMEM_DYN);
      if (e != cudaSuccess) return e;
      e = launch_pdl(attn_tc_kernel<16>, dim3(grid), dim3(Cfg<16>::THREADS), Cfg<16>::SMEM_DYN, st, rows_map, q_map,
                     qres_map, a);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return e;
}

}  // namespace mla
