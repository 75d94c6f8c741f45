/*
 * mla.h -- C ABI for one decode step of Multi-head Latent Attention (MLA) over a
 * compressed latent KV cache, on an NVIDIA GB300 (sm_103a).
 *
 * Two calls carry the method (mla_front_end and mla_o_proj, further down, add the layer's
 * projections before and after them):
 *   mla_cache_append  writes each sequence's new compressed row [kv_lat ; k_pe] into the
 *                     cache: optional kv_a projection, RMSNorm over the latent part,
 *                     consecutive-pair YaRN RoPE over the k_pe tail.
 *   mla_decode_attn   absorbs q_nope through W_UK into latent space, attends over every
 *                     cached row with all heads sharing each row (split over the sequence),
 *                     merges the splits by log-sum-exp and up-projects through W_UV.
 *
 * Sources (docs.rs source pages):
 *   moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs -- mla_attn_layer_forward_gpu:
 *     KV chain, YaRN RoPE of q_pe and k_pe, cache append, folded SDPA chain
 *     (q_prime -> mla_sdpa_folded -> out_per_head), softmax scale, error set.
 *   turbospark-runtime 0.3.0, src/families/deepseek2/attn.rs -- encode_mla_attention_block:
 *     the fused cache row, in-place norm and RoPE, absorb, MQA attention over compressed
 *     rows, v-combine; validate_q8_0_matrix.
 *
 * Conventions for every call:
 *   - Dimensions: H heads, C = kv_lora, N = qk_nope, R = qk_rope, V = v_head, a cache row
 *     holds C+R elements: [kv_lat (C) ; k_pe (R)].
 *   - Pointers marked "device" are CUDA device (or managed) pointers on the current device;
 *     "host" pointers are plain host memory. The caller owns every buffer; the library
 *     allocates no device memory and keeps no per-call state (mla_decode_attn_noalloc,
 *     at the end, uses one fixed device array that is part of the library).
 *   - Calls marked "async" only validate on the host and enqueue kernels on `stream`;
 *     they return before the GPU work ends and never synchronise. The kernels are launched
 *     with programmatic stream serialization (mla_decode_attn's first kernel at times
 *     excepted, see there): each lets the next kernel on the stream launch early and waits
 *     for its predecessor before touching data another kernel produces. A
 *     caller's own kernel launched right after with that same launch attribute must execute
 *     griddepcontrol.wait before it reads a call's outputs; ordinary launches, copies and events
 *     wait for completion as usual. Errors found on the
 *     host return before anything is enqueued. Conditions only the GPU can see (a bad
 *     length, a position that does not match the cache length, a page id out of range)
 *     set a sticky error word in the call's workspace; the affected sequence's outputs
 *     are written as NaN and the other sequences are unaffected. Read it with
 *     mla_get_device_error. Kernels never trap.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (same handle as cudaStream_t / CUstream). NULL = the legacy default stream. */
typedef struct CUstream_st* mla_stream_t;

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null pointer, bad dimension, misaligned pointer, B < 1 */
  MLA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (dtype / dimension combination) */
  MLA_ERR_POS_MISMATCH = 3,  /* device: append position != the sequence's current length */
  MLA_ERR_CACHE_FULL = 4,    /* device: append position beyond the cache's capacity */
  MLA_ERR_WORKSPACE = 5,     /* workspace NULL, misaligned or smaller than required */
  MLA_ERR_TIMEOUT = 6,       /* device: a bounded wait inside a kernel ran out */
  MLA_ERR_CUDA = 7,          /* a CUDA runtime call failed (launch, attribute, no device) */
  MLA_ERR_BAD_SEQ_LEN = 8,   /* device: seq_len < 1 or above the cache's capacity */
  MLA_ERR_BAD_PAGE = 9,      /* device: page-table entry outside [0, n_physical_rows/page_size) */
  MLA_ERR_BAD_KV_B = 10      /* kv_b dtype / shape / byte size contract broken */
} mla_status;

typedef enum mla_dtype {
  MLA_F32 = 0,
  MLA_BF16 = 1,
  /* Q8_0: 34-byte blocks of 32 elements along a row: an fp16 scale d (little endian)
   * then 32 int8 codes q; element value d*q. Weights only (kv_b). */
  MLA_Q8_0 = 2,
  /* 4-bit affine, groups of 64 (moeflux mla_attn_forward.rs: a 4-bit projection is
   * weight + scales + biases, group size 64; gpu_matvec.rs MatvecSpec: packed weight,
   * bf16 scales, bf16 biases). One buffer holding, for an [rows, cols] matrix: the codes
   * as rows*cols/8 little-endian uint32 words (row-major; code j of a word, bits 4j..4j+3,
   * is column 8w+j), then scales [rows, cols/64] bf16, then biases [rows, cols/64] bf16.
   * Element value scale*q + bias, q in 0..15. Weights only (kv_b); cols % 64 == 0. */
  MLA_Q4_AFFINE = 3
} mla_dtype;

typedef struct mla_config {
  int32_t n_heads;            /* H >= 1 */
  int32_t kv_lora;            /* C >= 1 (a multiple of 32 when kv_b is Q8_0) */
  int32_t qk_nope;            /* N >= 1 */
  int32_t qk_rope;            /* R >= 2, even */
  int32_t v_head;             /* V >= 1 */
  int32_t act_dtype;          /* mla_dtype, F32 or BF16: q and the cache rows */
  int32_t kv_b_dtype;         /* mla_dtype, F32, BF16, Q8_0 or Q4_AFFINE */
  float softmax_scale;        /* mscale^2 / sqrt(N+R); see mla_softmax_scale */
  float rms_eps;              /* RMSNorm epsilon of the latent norm (append only) */
  int32_t page_size;          /* 0: contiguous rows per sequence; else rows per page (>= 1) */
  int32_t max_pages_per_seq;  /* paged: width of a page-table row */
  int64_t rows_per_seq;       /* contiguous: rows reserved per sequence (its capacity) */
  const double* rope_inv_freq;/* device [R/2] float64 per-pair inverse frequencies,
                                 e.g. from mla_yarn_inv_freq; may be NULL only for a
                                 decode call whose q_pe is already rotated */
} mla_config;

/* The cache: physical rows plus, when paged, the page table.
 * Contiguous: logical row t of sequence b is physical row b*rows_per_seq + t.
 * Paged: logical row t of sequence b is physical row
 *        page_table[b*max_pages_per_seq + t/page_size]*page_size + t%page_size. */
typedef struct mla_cache {
  void* rows;                 /* device [n_physical_rows, C+R] in act_dtype, row-major,
                                 16-byte aligned; rows are C+R contiguous elements */
  const int32_t* page_table;  /* device [B, max_pages_per_seq] int32, or NULL (contiguous) */
  int64_t n_physical_rows;    /* rows in `rows` (bounds every address the kernels form) */
} mla_cache;

/* ---- host-only helpers (no GPU needed) ------------------------------------------------ */

/* Human-readable name of a status. Never NULL. */
const char* mla_status_string(mla_status s);

/* ABI revision of this header (bumped on any incompatible change). */
int32_t mla_abi_version(void);

/* YaRN per-pair inverse frequencies, float64, into out_host[rope_dim/2].
 * moeflux mla_attn_forward.rs, MlaYarnTables::new (table from rope_dim, theta, factor,
 * original max position, beta_fast, beta_slow); turbospark gptoss attn.rs module doc
 * (a per-pair table, because the ramp is not one theta). Pair i has base frequency
 * theta^(-2i/rope_dim); for factor > 1 pairs below the beta_fast correction dimension
 * keep it, pairs above the beta_slow one are divided by factor, linear ramp between
 * (YaRN's NTK-by-parts). factor <= 1 gives plain RoPE.
 * Errors: INVALID_ARG for rope_dim < 2 or odd, theta <= 1, orig_max_pos < 1, NULL out. */
mla_status mla_yarn_inv_freq(int32_t rope_dim, double theta, double factor,
                             int32_t orig_max_pos, double beta_fast, double beta_slow,
                             double* out_host);

/* YaRN magnitude scale: 1 + 0.1*coeff*ln(factor) for factor > 1, else 1.
 * turbospark deepseek2 attn.rs, attention scale comment. */
double mla_yarn_mscale(double factor, double coeff);

/* Softmax scale mscale^2 / sqrt(qk_nope + qk_rope) (moeflux mla_attn_forward.rs,
 * folded SDPA chain: 1/sqrt(qk_head_dim) * mscale * mscale). Returns 0 on bad dims. */
float mla_softmax_scale(int32_t qk_nope, int32_t qk_rope, double mscale);

/* The kv_b contract (turbospark deepseek2 attn.rs, validate_q8_0_matrix, generalised to
 * all four weight dtypes): shape must be (heads*(nope+v_dim), kv_lora); for Q8_0
 * kv_lora must be a non-zero multiple of 32, for Q4_AFFINE of 64; size_bytes must equal
 * the packed size, computed with overflow-checked multiplies. Returns OK, BAD_KV_B or
 * INVALID_ARG. */
mla_status mla_validate_kv_b(int32_t dtype, int64_t rows, int64_t cols, uint64_t size_bytes,
                             int32_t heads, int32_t nope, int32_t kv_lora, int32_t v_dim);

/* Bytes of a kv_b tensor for cfg (0 on invalid cfg or overflow). kv_b is row-major
 * [H*(N+V), C]: per head its N rows of W_UK then its V rows of W_UV
 * (moeflux mla_attn_forward.rs: kv_b_per_head = nope + v_head_dim; out_per_head skips
 * the nope rows). */
uint64_t mla_kv_b_bytes(const mla_config* cfg);

/* ---- workspace sizing (needs a CUDA device: the split plan depends on its SM count) ---- */

/* Bytes of device workspace mla_cache_append needs for B sequences (with or without the
 * kv_a projection). Writes *bytes; returns INVALID_ARG / CUDA on failure. */
mla_status mla_append_workspace_size(const mla_config* cfg, int32_t B, size_t* bytes);

/* Bytes of device workspace mla_decode_attn (and its three stages) needs for B sequences
 * on the current device. The split plan is fixed by (cfg, B, device), so a workspace sized
 * here fits every call with the same cfg and B. */
mla_status mla_decode_workspace_size(const mla_config* cfg, int32_t B, size_t* bytes);

/* The split plan mla_decode_attn uses for (cfg, B) on the current device. */
typedef struct mla_plan_info {
  int32_t kernel;          /* attention kernel: 0 = CUDA-core (any dims, f32 or bf16),
                              1 = tcgen05 tensor-core (bf16 rows of 576 = 512 + 64), one CTA
                              per SM and head group, 128-row tiles,
                              2 = tcgen05 on SM pairs (bf16 rows of 576, exactly 128 heads):
                              a cluster of two CTAs shares each 64-row tile, one latent half
                              each; `splits` then counts CTA pairs,
                              3 = one launch for tiny batches (bf16, one query row per
                              sequence, B * H <= 64, H <= 32, capacity <= 8192, and few
                              enough chunks and heads that the grid takes them in about one
                              round): absorb, attention over 32-row chunks, merge and W_UV
                              in a single grid separated by grid-wide barriers; `splits`
                              then counts the grid's CTAs */
  int32_t heads_per_cta;   /* heads that share each staged row tile (kernel 2: per CTA pair) */
  int32_t head_groups;     /* ceil(H / heads_per_cta) */
  int32_t splits;          /* row splits per sequence (partials kept in the workspace) */
  int64_t rows_per_split;  /* rows each split covers (a multiple of the row tile) */
  int64_t capacity;        /* most rows one sequence can attend */
} mla_plan_info;

/* Fills *info with the plan for (cfg, B). Host-only query; needs a CUDA device. */
mla_status mla_decode_plan(const mla_config* cfg, int32_t B, mla_plan_info* info);

/* ---- failure detection --------------------------------------------------------------------
 * Every wait inside the tensor-core kernels (on a TMA copy, an MMA, another role of the same
 * CTA) is bounded: when it runs out, the kernel records MLA_ERR_TIMEOUT in the workspace,
 * every role of the CTA stops, copies and MMAs already issued are drained, tensor memory is
 * freed, and the outputs the CTA owns are written as NaN (their sequences' out and lse become
 * NaN). The limit of the main-loop waits is a process-wide setting, read when a call enqueues
 * its kernels (a captured graph keeps the value of its capture); the drains always keep
 * 200 ms. Sets the limit in nanoseconds (0 restores the default, 200 ms) and returns the
 * previous one. A limit far below a kernel's natural waits makes it time out on purpose: that
 * is how the timeout path is tested. Thread-safe; host-only. */
uint64_t mla_set_wait_limit_ns(uint64_t ns);

/* ---- the method ----------------------------------------------------------------------- */

/* Append one new row per sequence, in place (async).
 * turbospark deepseek2 attn.rs, encode_mla_attention_block: kv_a straight into the cache
 * row, RMSNorm over kv_lora in place, RoPE of the pe tail in place with the q pairing;
 * moeflux mla_attn_forward.rs: KV-A chain, kv_a_layernorm, YaRN RoPE of k_pe, append of
 * row[pos], guards PosMismatch and CacheFull.
 *   kv_in      device. w_kva == NULL: [B, C+R] float32 kv_a rows (the projection's output).
 *              w_kva != NULL: [B, hidden] hidden states in act_dtype.
 *   w_kva      device [C+R, hidden] in act_dtype, row-major, or NULL.
 *   hidden     columns of w_kva (ignored when w_kva == NULL; a multiple of 8 otherwise).
 *   norm_w     device [C] float32 RMSNorm weight.
 *   positions  device [B] int32: the row index each sequence writes and the RoPE position.
 *   seq_lens   device [B] int32 current lengths, or NULL. When given, positions[b] must
 *              equal seq_lens[b] (device error POS_MISMATCH otherwise). The call never
 *              changes lengths: the caller advances them.
 * For each b the finished row is y[0:C] = x[0:C]/sqrt(mean(x[0:C]^2)+eps)*norm_w and
 * y[C:C+R] = RoPE(x[C:C+R], positions[b]) with pairs (2i, 2i+1), x = kv_in row or
 * W_kva*x_b, computed in float32 and rounded once to act_dtype. No other row changes.
 * Device errors: CACHE_FULL (position outside capacity), BAD_PAGE, POS_MISMATCH. */
mla_status mla_cache_append(const mla_config* cfg, const mla_cache* cache,
                            const void* kv_in, const void* w_kva, int32_t hidden,
                            const float* norm_w, const int32_t* positions,
                            const int32_t* seq_lens, int32_t B,
                            void* workspace, size_t ws_bytes, mla_stream_t stream);

/* One absorbed decode step for B sequences (async): the three stages below, in order.
 * moeflux mla_attn_forward.rs, folded SDPA chain; turbospark deepseek2 attn.rs, absorb ->
 * MQA attention over compressed rows -> v-combine.
 *   q          device [B, H, N+R] act_dtype; each head [q_nope (N) ; q_pe (R)].
 *   kv_b       device kv_b in kv_b_dtype (see mla_kv_b_bytes), 16-byte aligned.
 *   seq_lens   device [B] int32 rows to attend (1 <= seq_lens[b] <= capacity).
 *   positions  device [B] int32 RoPE position of each query's q_pe, or NULL when q_pe
 *              is already rotated.
 *   out        device [B, H, V] float32: out[b,h] = W_UV,h * sum_t p_t kv_lat_t.
 *   lse        device [B, H] float32 natural-log sum-exp of the scaled scores, or NULL.
 * Scores are s_t = softmax_scale * ([q' ; q_pe] . row_t) with q' = W_UK,h^T q_nope.
 * Launch order: when the cache capacity gives each attention CTA at least four 128-row tiles
 * (B * ceil(capacity / 128) >= 4 * the plan's splits, kernel 1) or each CTA pair at least eight
 * 64-row tiles (B * ceil(capacity / 64) >= 8 * splits, kernel 2), the first
 * kernel (the absorb) is launched in plain stream order: it starts only after all earlier
 * work on the stream, a cache append above all, has completed, and the attention kernel
 * after it streams cache rows while the absorb still runs, waiting only for the fused
 * queries. Otherwise every kernel is launched as described at the top. The three step calls
 * below always keep every kernel's wait in place; the results are bit-identical either way.
 * Tiny batches (mla_decode_plan reports kernel 3) run instead as one launch (absorb,
 * attention over 32-row chunks, merge and W_UV in one grid, float32 throughout): its results
 * agree with the three step calls within rounding, not bit for bit, and are the same from run
 * to run and for a sequence whatever the rest of the batch. It uses the workspace's header for
 * its barrier counters (left zero when it returns).
 * Device errors: BAD_SEQ_LEN, BAD_PAGE (that sequence's out/lse become NaN), TIMEOUT (one
 * launch: a grid-wide wait ran out; the outputs that CTA owns become NaN). */
mla_status mla_decode_attn(const mla_config* cfg, const void* q, const void* kv_b,
                           const mla_cache* cache, const int32_t* seq_lens,
                           const int32_t* positions, float* out, float* lse, int32_t B,
                           void* workspace, size_t ws_bytes, mla_stream_t stream);

/* Stage 1 of mla_decode_attn (async): RoPE of q_pe at positions[b] and the absorb
 * q'[b,h,:] = W_UK,h^T q_nope[b,h,:], written as the fused query rows [q' ; q_pe] in
 * act_dtype into the workspace (moeflux q_prime; turbospark encode_mla_absorb_q). */
mla_status mla_decode_absorb(const mla_config* cfg, const void* q, const void* kv_b,
                             const int32_t* positions, int32_t B,
                             void* workspace, size_t ws_bytes, mla_stream_t stream);

/* Stage 2 (async): split attention over the cache rows with all heads of a sequence
 * sharing each row. Each split writes its softmax-normalised latent sum O_s [H, C] and
 * its log-sum-exp lse_s [H] into the workspace (moeflux mla_sdpa_folded; turbospark
 * encode_mla_attention_decode, V = the row's first kv_lora values). */
mla_status mla_decode_partial(const mla_config* cfg, const mla_cache* cache,
                              const int32_t* seq_lens, int32_t B,
                              void* workspace, size_t ws_bytes, mla_stream_t stream);

/* Stage 3 (async): merge the splits (lse = log sum_s exp(lse_s), vc = sum_s
 * exp(lse_s - lse) O_s) and up-project out[b,h] = W_UV,h vc (moeflux out_per_head;
 * turbospark encode_mla_v_combine; the split + combine structure of turbospark
 * gptoss attn.rs). */
mla_status mla_decode_combine(const mla_config* cfg, const void* kv_b,
                              const int32_t* seq_lens, float* out, float* lse, int32_t B,
                              void* workspace, size_t ws_bytes, mla_stream_t stream);

/* ---- the projections around the step -------------------------------------------------------
 * moeflux mla_attn_forward.rs, mla_attn_layer_forward_gpu: Q chain (q_a_proj matvec ->
 * q_a_layernorm -> q_b_proj matvec), KV-A chain (kv_a_proj_with_mqa matvec), o_proj final
 * matvec; turbospark deepseek2 attn.rs, encode_mla_attention_block: Q_PROJ GEMV of the normed
 * hidden state (a model without a q rank), O_PROJ GEMV of the combined heads.
 * Every projection is y = W x per sequence, W row-major [out_dim, in_dim] in w_dtype (the
 * kv_b formats: F32, BF16, Q8_0 with blocks along in_dim, Q4_AFFINE with the codes, scales and
 * biases of the whole matrix in one buffer), accumulated in float32 in a fixed order
 * (run-to-run identical results). in_dim must be a multiple of 8 (32 for Q8_0, 64 for
 * Q4_AFFINE); every pointer 16-byte aligned. */
typedef struct mla_proj {
  int32_t hidden;          /* D: the layer's model width (in_dim of q_a / q, kv_a; out_dim of o) */
  int32_t q_lora;          /* 0: one q projection; else the Q chain's rank (in_dim of q_b) */
  int32_t w_dtype;         /* mla_dtype of all the weights below */
  float q_norm_eps;        /* RMSNorm epsilon of q_a_layernorm */
  const void* w_q_a;       /* device [q_lora, D] (q_lora > 0), else ignored */
  const float* q_a_norm_w; /* device [q_lora] float32 q_a_layernorm weight (q_lora > 0) */
  const void* w_q;         /* device q_b [H*(N+R), q_lora] when q_lora > 0, else q [H*(N+R), D] */
  const void* w_kva;       /* device [C+R, D], or NULL when no kv_a output is asked for */
  const void* w_o;         /* device [D, H*V], or NULL when mla_o_proj is not used */
} mla_proj;

/* Bytes of device workspace mla_front_end needs for B sequences. It holds a 256-byte header
 * (the device error word: clear it once, or zero-fill, before first use; read it with
 * mla_get_device_error) and, as needed, the float32 q_lat rows, the bf16 halves of the
 * normalised q_lat and the tensor-core path's split partials. Host-only (the split plan
 * depends on the device's SM count). */
mla_status mla_front_end_workspace_size(const mla_config* cfg, const mla_proj* pj, int32_t B,
                                        size_t* bytes);

/* The layer's front end for B sequences (async): the queries mla_decode_attn takes and the
 * kv_a rows mla_cache_append takes (with w_kva == NULL there).
 *   x    device [B, D] act_dtype: the layer's normed input (the caller owns that norm).
 *   q    device [B, H, N+R] act_dtype: q_lora > 0: q_full = W_q_b RMSNorm(W_q_a x) with the
 *        norm over all q_lora values (x / sqrt(mean(x^2) + q_norm_eps) * q_a_norm_w);
 *        q_lora == 0: q_full = W_q x. Head h is q_full[h*(N+R) : (h+1)*(N+R)], its q_nope
 *        first; q_pe is left unrotated (mla_decode_attn rotates it). Rounded once.
 *   kva  device [B, C+R] float32 = W_kva x, or NULL (then w_kva is not read).
 * Launches: one GEMV computing W_q_a x (or W_q x) and W_kva x together (one read of x), then,
 * for q_lora > 0, the norm of the q_lat rows and the q_b projection. Weights in BF16 run on
 * the tensor cores for 16 to 128 sequences (256 for a bf16 input), and for fewer sequences
 * when the matrix holds 64 MiB or more: a float32 input as bf16 hi + lo halves (about float32
 * accuracy), column slices summed in a fixed order. Every result is run-to-run identical and
 * q does not depend on whether kv_a is computed.
 * Errors: INVALID_ARG (null or misaligned pointer, bad dims, kva without w_kva),
 * UNSUPPORTED (w_dtype), WORKSPACE, CUDA; device: TIMEOUT (a bounded wait ran out: that
 * launch's outputs are NaN). */
mla_status mla_front_end(const mla_config* cfg, const mla_proj* pj, const void* x, void* q,
                         float* kva, int32_t B, void* workspace, size_t ws_bytes,
                         mla_stream_t stream);

/* Bytes of device workspace mla_o_proj needs for B sequences: the 256-byte header (as for
 * mla_front_end) and, on the tensor-core path, the bf16 halves of the input and the split
 * partials. Host-only. */
mla_status mla_o_proj_workspace_size(const mla_config* cfg, const mla_proj* pj, int32_t B,
                                     size_t* bytes);

/* Kernels one mla_front_end call (with or without kv_a) and one mla_o_proj call enqueue for
 * B sequences (they depend on the path and the column slices chosen). Host-only; either
 * pointer may be NULL. Errors: as mla_front_end_workspace_size. */
mla_status mla_proj_launches(const mla_config* cfg, const mla_proj* pj, int32_t B, int32_t* front_end,
                             int32_t* o_proj);

/* o_proj for B sequences (async): y[b] = W_o attn[b], attn [B, H, V] float32 read head after
 * head (head h's V values at h*V: the layout mla_decode_attn writes), y device [B, D] float32.
 * Paths and errors as mla_front_end (w_o must be set). */
mla_status mla_o_proj(const mla_config* cfg, const mla_proj* pj, const float* attn, float* y,
                      int32_t B, void* workspace, size_t ws_bytes, mla_stream_t stream);

/* ---- several query tokens per sequence ----------------------------------------------------
 * T new tokens of each sequence decoded at once (draft tokens of speculative decoding, a chunk
 * of a prompt), their rows already in the cache: token i of sequence b sits at position
 * positions[b] + i and attends the first seq_lens[b] - T + 1 + i rows (itself and every row
 * before it). The pages have no MLA prefill; this follows the causal decode of one token (moeflux
 * mla_attn_forward.rs, folded SDPA over cache_len = pos + 1 rows) applied to T stacked query
 * tokens, as moeflux gpu_matvec.rs's *_n_tokens encoders apply one weight matrix to N stacked
 * inputs. The T tokens run as T x H heads of one sequence (token-major), so every staged row
 * tile serves all of them; T = 1 is exactly mla_decode_attn (same kernels, bit-identical).
 *
 * Bytes of workspace mla_decode_attn_multi needs for (cfg, T, B); as
 * mla_decode_workspace_size for T = 1. INVALID_ARG for T < 1, T > 64 or T*H > 65536. */
mla_status mla_decode_multi_workspace_size(const mla_config* cfg, int32_t tokens, int32_t B,
                                           size_t* bytes);

/* Multi-token decode for B sequences (async).
 *   q          device [B, T, H, N+R] act_dtype (token i of sequence b at q[b][i]).
 *   seq_lens   device [B] int32: rows the last token attends (T <= seq_lens[b] <= capacity);
 *              the tokens' own rows are the last T of them.
 *   positions  device [B] int32 RoPE position of each sequence's first token, or NULL when
 *              q_pe is already rotated.
 *   out        device [B, T, H, V] float32; lse device [B, T, H] float32 or NULL.
 * Other arguments, launches and errors as mla_decode_attn; a seq_lens[b] below T is the device
 * error BAD_SEQ_LEN (that sequence's outputs NaN). */
mla_status mla_decode_attn_multi(const mla_config* cfg, int32_t tokens, const void* q,
                                 const void* kv_b, const mla_cache* cache, const int32_t* seq_lens,
                                 const int32_t* positions, float* out, float* lse, int32_t B,
                                 void* workspace, size_t ws_bytes, mla_stream_t stream);

/* ---- device error word ------------------------------------------------------------------ */

/* Synchronises `stream`, then reads the workspace's sticky error word: returns the first
 * device error any call using this workspace recorded since the last clear (MLA_OK if
 * none), and writes the sequence index it concerns to *seq_out when seq_out != NULL. */
mla_status mla_get_device_error(const void* workspace, int32_t* seq_out, mla_stream_t stream);

/* Clears the workspace's error word (async, on `stream`). A fresh workspace must be
 * cleared once (or zero-filled) before its first use. */
mla_status mla_clear_device_error(void* workspace, mla_stream_t stream);

/* ---- allocation-free decode --------------------------------------------------------------
 * An addition of this library: the papers and write-ups the method comes from have no
 * counterpart. It serves callers that may not allocate device memory when they decode (an
 * engine plugin whose host owns all device memory, a server whose memory budget was fixed
 * at start-up, a loop that cannot take the synchronisation an allocation implies).
 *
 * Bytes of the device array mla_decode_attn_noalloc uses as its workspace. */
#define MLA_NOALLOC_SCRATCH_BYTES (64ull * 1024ull * 1024ull)

/* mla_decode_attn (async) with the workspace taken from one array of
 * MLA_NOALLOC_SCRATCH_BYTES bytes of device memory that is part of the library
 * (a file-scope __device__ array, 256-byte aligned, one per device context), not from the
 * caller. It calls no allocator: no cudaMalloc/cudaFree, no allocating library.
 *   q, kv_b, cache, seq_lens, positions, out, lse, B, stream: as in mla_decode_attn.
 *   device_error  device int32[2] (4-byte aligned) or NULL: receives {status, sequence} of
 *                 the first device error of this call (MLA_OK = 0 when none), written on
 *                 `stream` after the decode.
 * Zero state: the array's first 256 bytes (the device error word) must be zero when the
 * kernels start; every call clears them on `stream` before its launches, and nothing else
 * in the array is read before it is written in the same call.
 * Address: every call looks the array's address up in the current device's context with
 * cudaGetSymbolAddress (no allocation), so a context torn down and recreated (e.g. after
 * cudaDeviceReset) is picked up. The first call on each device may load the library's
 * module for that device; make that first call before any stream capture.
 * Concurrency: every call on a device shares the one array. Calls that may overlap on the
 * GPU (different streams without ordering between them, or several host threads) race on
 * it and corrupt each other's results; order them on one stream or with events.
 * Errors: MLA_ERR_WORKSPACE when mla_decode_workspace_size(cfg, B) exceeds
 * MLA_NOALLOC_SCRATCH_BYTES (nothing enqueued); MLA_ERR_CUDA when the address lookup fails;
 * otherwise as mla_decode_attn. On an argument error found after the size check at most the
 * clearing of the array's error word has been enqueued. */
mla_status mla_decode_attn_noalloc(const mla_config* cfg, const void* q, const void* kv_b,
                                   const mla_cache* cache, const int32_t* seq_lens,
                                   const int32_t* positions, float* out, float* lse, int32_t B,
                                   int32_t* device_error, mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
