"""fp64 CPU oracle for one MLA decode step over a compressed latent KV cache.

TEST INFRASTRUCTURE. Only the tests, `__graft_entry__.smoke()` and the benchmark's CPU
baseline (and its `--impl reference` arm) may import or run this module. The product
path (the CUDA library and its Python binding) never imports it, and it imports
nothing from the product path: it shares no code, tables or helpers with it.

Everything is computed in float64 from inputs decoded exactly (bf16, fp16 and Q8_0 all
convert to float64 without rounding). The code is deliberately plain: one library
primitive (a matmul / einsum) per step, no blocking, no fusion.

Sources (docs.rs source pages):
  [moeflux-fwd]  moeflux 0.1.0-pre.3, src/riir/attn/mla_attn_forward.rs
  [ts-ds2]       turbospark-runtime 0.3.0, src/families/deepseek2/attn.rs
  [ts-gptoss]    turbospark-runtime 0.3.0, src/families/gptoss/attn.rs

Readings of points the pages leave open (each is listed with its reason in the design
notes): kv_b rows per head are the nope rows (W_UK) then the v rows (W_UV); RoPE pairs
consecutive elements and is a pure rotation (no magnitude scaling); the YaRN table
follows the YaRN paper's NTK-by-parts ramp; the softmax scale is
mscale^2 / sqrt(qk_nope + qk_rope); LSE is the natural log of the summed exponentials of
the scaled scores; Q8_0 blocks are an fp16 scale followed by 32 int8 codes.

Pins: tests/test_oracle_pins.py checks every function here against closed forms,
identities and the pages' own fixture (absorbed == unabsorbed MHA, T=1, softmax sums,
RoPE identities and pairing, YaRN limits, RMSNorm invariants, Q8_0 and 4-bit golden
blocks, the kv_b validation fixture, split/merge associativity, page addressing, and for
the projections rank-one closed forms, one-hot layout probes and the Q chain's scale
invariance).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

Q8_0_BLOCK_ELEMS = 32
Q8_0_BLOCK_BYTES = 34
DTYPE_Q8_0 = "q8_0"
Q4_GROUP = 64
DTYPE_Q4_AFFINE = "q4_affine"


# ---------------------------------------------------------------------------------------
# Exact decoding of stored formats
# ---------------------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64. A bf16 value is the top half of an fp32."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f32_to_f64(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def q8_0_to_f64(blob: np.ndarray, cols: int) -> np.ndarray:
    """Dequantise Q8_0 rows: each 34-byte block is an fp16 scale d then 32 int8 codes q,
    and the block's values are d*q (exact in float64). Blocks run along a row.

    [ts-ds2] `validate_q8_0_matrix`: 32-element blocks, a row holds kv_lora/32 blocks.
    """
    blob = np.asarray(blob, dtype=np.uint8)
    rows = blob.shape[0]
    nb = cols // Q8_0_BLOCK_ELEMS
    blocks = blob.reshape(rows, nb, Q8_0_BLOCK_BYTES)
    d = blocks[:, :, 0:2].copy().view("<f2").reshape(rows, nb).astype(np.float64)
    q = blocks[:, :, 2:].copy().view(np.int8).astype(np.float64)
    return (q * d[:, :, None]).reshape(rows, cols)


def q8_0_validate(dtype: str, shape: tuple, size_bytes: int, heads: int, nope: int,
                  kv_lora: int, v_dim: int) -> Optional[str]:
    """The kv_b contract for Q8_0: returns None when valid, else the reason.

    [ts-ds2] `validate_q8_0_matrix`: dtype must be Q8_0; shape must be
    (heads*(nope+v_dim), kv_lora); kv_lora must be a non-zero multiple of 32; the byte
    size must equal rows * (kv_lora/32) * block_bytes. Sizes use unbounded integers here.
    """
    if dtype != DTYPE_Q8_0:
        return f"kv_b requires Q8_0, got {dtype}"
    rows = heads * (nope + v_dim)
    if tuple(shape) != (rows, kv_lora):
        return f"shape {tuple(shape)} != {(rows, kv_lora)}"
    if kv_lora == 0 or kv_lora % Q8_0_BLOCK_ELEMS != 0:
        return f"width {kv_lora} does not tile Q8_0 blocks"
    expected = rows * (kv_lora // Q8_0_BLOCK_ELEMS) * Q8_0_BLOCK_BYTES
    if size_bytes != expected:
        return f"size {size_bytes} != {expected}"
    return None


def q4_affine_bytes(rows: int, cols: int) -> int:
    """Bytes of a 4-bit affine matrix: the packed codes (cols/2 bytes a row), then one bf16
    scale and one bf16 bias per 64-column group of every row."""
    return rows * (cols // 2) + 2 * rows * (cols // Q4_GROUP) * 2


def q4_affine_to_f64(blob: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Dequantise a 4-bit affine matrix [rows, cols]: w = scale * q + bias, with q an unsigned
    4-bit code and (scale, bias) shared by 64 consecutive columns of a row (exact in float64).

    [moeflux-fwd] `resolve_proj` (a 4-bit projection is three tensors: weight, scales, biases)
    and `encode_mla_q_prime_4bit` / `encode_mla_out_per_head_4bit` (group size 64);
    [moeflux-mv] `MatvecSpec` (packed weight, bf16 scales, bf16 biases). The byte layout is not
    on the pages; read as: the three tensors back to back in one buffer, codes first as
    little-endian 32-bit words of 8 codes each (code j of a word in bits 4j..4j+3, the lower
    column first), then scales [rows, cols/64] and biases [rows, cols/64], bf16, row-major.
    """
    blob = np.asarray(blob, dtype=np.uint8).reshape(-1)
    ng = cols // Q4_GROUP
    nc = rows * (cols // 2)
    words = blob[:nc].copy().view("<u4").reshape(rows, cols // 8)
    shifts = (4 * np.arange(8, dtype=np.uint32))[None, None, :]
    q = ((words[:, :, None] >> shifts) & np.uint32(15)).reshape(rows, cols).astype(np.float64)
    scales = bf16_to_f64(blob[nc:nc + 2 * rows * ng].copy().view("<u2").reshape(rows, ng))
    biases = bf16_to_f64(blob[nc + 2 * rows * ng:nc + 4 * rows * ng].copy().view("<u2").reshape(rows, ng))
    return q * np.repeat(scales, Q4_GROUP, axis=1) + np.repeat(biases, Q4_GROUP, axis=1)


# ---------------------------------------------------------------------------------------
# YaRN frequency table and magnitude scale
# ---------------------------------------------------------------------------------------

def yarn_inv_freq(rope_dim: int, theta: float, factor: float, orig_max_pos: int,
                  beta_fast: float, beta_slow: float) -> np.ndarray:
    """Per-pair inverse frequencies [rope_dim/2] with YaRN's NTK-by-parts blend.

    [moeflux-fwd] `MlaYarnTables::new` builds the table from (rope_dim, theta, factor,
    original max position, beta_fast, beta_slow); [ts-gptoss] module doc: YaRN ramps
    between two correction dimensions, so it needs a per-pair table. The formula itself
    is YaRN's (Peng et al. 2023): pair i has base frequency theta^(-2i/d); pairs below
    the fast correction dimension keep it, pairs above the slow one are divided by the
    factor, and a linear ramp blends in between.
    """
    d = rope_dim
    i = np.arange(d // 2, dtype=np.float64)
    base = theta ** (-2.0 * i / d)
    if factor <= 1.0:
        return base

    def corr_dim(n_rot: float) -> float:
        # the dimension whose wavelength completes n_rot turns over orig_max_pos
        return d * math.log(orig_max_pos / (n_rot * 2.0 * math.pi)) / (2.0 * math.log(theta))

    lo = max(math.floor(corr_dim(beta_fast)), 0)
    hi = min(math.ceil(corr_dim(beta_slow)), d - 1)
    if lo == hi:
        hi += 0.001
    ramp = np.clip((i - lo) / (hi - lo), 0.0, 1.0)
    return base / factor * ramp + base * (1.0 - ramp)


def yarn_mscale(factor: float, coeff: float = 1.0) -> float:
    """YaRN attention magnitude scale: 1 + 0.1*coeff*ln(factor) for factor > 1, else 1.

    [ts-ds2] `encode_mla_attention_block`, attention scale comment:
    (1 + 0.1*mscale*ln factor)^2 / sqrt(key_dim).
    """
    if factor <= 1.0:
        return 1.0
    return 1.0 + 0.1 * coeff * math.log(factor)


def softmax_scale(qk_nope: int, qk_rope: int, mscale: float) -> float:
    """[moeflux-fwd] folded SDPA chain: softmax_scale = mscale^2 / sqrt(qk_head_dim),
    qk_head_dim = nope + rope."""
    return mscale * mscale / math.sqrt(qk_nope + qk_rope)


# ---------------------------------------------------------------------------------------
# Interleaved RoPE and RMSNorm
# ---------------------------------------------------------------------------------------

def rope_pairs(x: np.ndarray, pos: int, inv_freq: np.ndarray) -> np.ndarray:
    """Rotate consecutive pairs (x[2i], x[2i+1]) of the last axis by angle pos*inv_freq[i].

    [ts-ds2] `encode_mla_attention_block`, pe-tail comment: the pairing is ggml's
    consecutive-element one, not (i, i + d/2). [moeflux-fwd] YaRN RoPE step: applied to
    q_pe (all heads) and to the shared k_pe at the token's position.
    """
    x = np.asarray(x, dtype=np.float64)
    a = float(pos) * np.asarray(inv_freq, dtype=np.float64)
    c, s = np.cos(a), np.sin(a)
    x0 = x[..., 0::2]
    x1 = x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * w over the last axis.

    [moeflux-fwd] KV chain: `kv_a_layernorm` over the latent half (kv_lora elements);
    [ts-ds2] the norm runs over kv_lora of the cache row only.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


# ---------------------------------------------------------------------------------------
# kv_b layout and cache addressing
# ---------------------------------------------------------------------------------------

def split_kv_b(kv_b: np.ndarray, heads: int, nope: int, v_dim: int):
    """kv_b [heads*(nope+v_dim), kv_lora] -> (W_UK [H, nope, C], W_UV [H, v_dim, C]).

    [moeflux-fwd] `kv_b_per_head = nope + v_head_dim`; out_per_head receives `nope` to
    skip the W_UK rows, so each head's block is its nope rows then its v rows.
    """
    C = kv_b.shape[1]
    blocks = np.asarray(kv_b, dtype=np.float64).reshape(heads, nope + v_dim, C)
    return blocks[:, :nope, :], blocks[:, nope:, :]


def physical_row(b: int, t, page_table: Optional[np.ndarray], page_size: int,
                 rows_per_seq: int):
    """Pool row holding logical row t of sequence b.

    Contiguous: b*rows_per_seq + t ([ts-ds2] `k_slot(layer, pos)` addresses one
    contiguous run of rows). Paged: page_table[b][t // page_size]*page_size + t % page_size.
    """
    t = np.asarray(t, dtype=np.int64)
    if page_table is None or page_size == 0:
        return b * rows_per_seq + t
    return page_table[b, t // page_size].astype(np.int64) * page_size + t % page_size


# ---------------------------------------------------------------------------------------
# Cache append
# ---------------------------------------------------------------------------------------

def kv_a_rows(x: np.ndarray, w_kva: np.ndarray) -> np.ndarray:
    """kv_a projection: row = W_kva x, [B, hidden] x [C+R, hidden] -> [B, C+R].

    [moeflux-fwd] KV-A chain (`kv_a_proj_with_mqa`, out_dim kv_lora+rope);
    [ts-ds2] kv_a writes its output straight into the cache row.
    """
    return np.asarray(x, dtype=np.float64) @ np.asarray(w_kva, dtype=np.float64).T


def append_rows(kva: np.ndarray, norm_w: np.ndarray, positions: Sequence[int],
                inv_freq: np.ndarray, kv_lora: int, eps: float) -> np.ndarray:
    """The finished cache rows [B, C+R]: RMSNorm over [0, C), RoPE over [C, C+R) at each
    sequence's position; nothing else changes.

    [ts-ds2] `encode_mla_attention_block`: kv_a into the row, in-place norm over kv_lora,
    then in-place RoPE of the pe tail (one head whose window starts at kv_lora).
    [moeflux-fwd] the same steps on separate buffers, then the append of (kv_lat, k_pe).
    """
    kva = np.asarray(kva, dtype=np.float64)
    out = np.empty_like(kva)
    for b in range(kva.shape[0]):
        out[b, :kv_lora] = rms_norm(kva[b, :kv_lora], norm_w, eps)
        out[b, kv_lora:] = rope_pairs(kva[b, kv_lora:], int(positions[b]), inv_freq)
    return out


# ---------------------------------------------------------------------------------------
# The projections around the step: the Q chain, a direct q projection, o_proj
# ---------------------------------------------------------------------------------------

def matvec(W: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y = W x for every input vector: W [out_dim, in_dim], x [..., in_dim] -> [..., out_dim].

    [moeflux-fwd] `encode_matvec` with `MatvecSpec { out_dim, in_dim }` (every projection
    of the layer is one); [ts-ds2] `encode_gemv_any(tensor, out, in)`.
    """
    return np.asarray(x, dtype=np.float64) @ np.asarray(W, dtype=np.float64).T


def heads_view(q_full: np.ndarray, heads: int, qk_head: int) -> np.ndarray:
    """[..., heads*qk_head] -> [..., heads, qk_head]: head h is the run of qk_head values
    starting at h*qk_head, its q_nope part first and its q_pe part last.

    [moeflux-fwd] `q_full: [num_heads, qk_head_dim]`, split per head into (q_nope, q_pe).
    """
    q_full = np.asarray(q_full, dtype=np.float64)
    return q_full.reshape(q_full.shape[:-1] + (heads, qk_head))


def q_chain(x: np.ndarray, W_qa: np.ndarray, q_norm_w: np.ndarray, eps: float,
            W_qb: np.ndarray, heads: int, qk_head: int) -> np.ndarray:
    """q [B, H, N+R] from the layer's normed input x [B, D] by the low-rank Q chain.

    [moeflux-fwd] Q chain: q_lat = matvec(x, q_a) with out_dim q_lora_rank and in_dim
    hidden_dim; the RMSNorm of q_lat over its q_lora_rank values with the q_a_layernorm
    weight and RMS_NORM_EPS; q_full = matvec(q_lat, q_b) with out_dim
    num_heads*qk_head_dim and in_dim q_lora_rank; then the per-head split.
    """
    q_lat = matvec(W_qa, x)
    return heads_view(matvec(W_qb, rms_norm(q_lat, q_norm_w, eps)), heads, qk_head)


def q_direct(x: np.ndarray, W_q: np.ndarray, heads: int, qk_head: int) -> np.ndarray:
    """q [B, H, N+R] = W_q x, the single q projection of a model without a q rank.

    [ts-ds2] `encode_mla_attention_block`: `Q_PROJ` GEMV of the normed hidden state into
    `[heads * head_dim]`, whose pe windows are then rotated before the absorb.
    """
    return heads_view(matvec(W_q, x), heads, qk_head)


def o_proj(out: np.ndarray, W_o: np.ndarray) -> np.ndarray:
    """y [B, D] = W_o . out[b] with out [B, H, V] read head after head (H*V values, head h
    at h*V), W_o [D, H*V].

    [moeflux-fwd] `o_proj` final matvec: input out_per_head, out_dim hidden_dim,
    in_dim num_heads*v_head_dim; [ts-ds2] `O_PROJ` GEMV from heads*v_dim to hidden.
    """
    out = np.asarray(out, dtype=np.float64)
    return matvec(W_o, out.reshape(out.shape[0], -1))


# ---------------------------------------------------------------------------------------
# Decode: absorbed (the method) and unabsorbed (plain MHA, the self-check)
# ---------------------------------------------------------------------------------------

def absorb_query(q_nope: np.ndarray, W_UK: np.ndarray) -> np.ndarray:
    """q'[h, c] = sum_n q_nope[h, n] W_UK[h, n, c]: the query moved into latent space.

    [moeflux-fwd] folded SDPA chain, `q_prime`; [ts-ds2] absorb into `[q' ; q_pe]` rows.
    """
    return np.einsum("hn,hnc->hc", q_nope, W_UK)


def scores(q_abs: np.ndarray, rows: np.ndarray, scale: float) -> np.ndarray:
    """s[h, t] = scale * ([q' ; q_pe_rot][h] . row_t): one dot over the whole compressed
    row [kv_lat ; k_pe].

    [ts-ds2] MQA attention over the compressed rows (key width = the cache row);
    [moeflux-fwd] `mla_sdpa_folded` over the latent and rope caches.
    """
    return scale * (q_abs @ rows.T)


def softmax_lse(s: np.ndarray):
    """Row-wise softmax probabilities and natural-log sum-exp, max-shifted."""
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    tot = e.sum(axis=-1, keepdims=True)
    return e / tot, (m + np.log(tot))[..., 0]


def decode_one(q: np.ndarray, W_UK: np.ndarray, W_UV: np.ndarray, rows: np.ndarray,
               pos: Optional[int], inv_freq: np.ndarray, scale: float, kv_lora: int):
    """Absorbed decode for one sequence.

    q [H, N+R] (each head [q_nope ; q_pe]), rows [L, C+R] the sequence's cache rows.
    Returns out [H, V] and lse [H].
    Steps: RoPE of q_pe at `pos` (None = already rotated); absorb q' = W_UK^T q_nope;
    scores over [q' ; q_pe] . row; softmax; v-combine vc = sum_t p_t kv_lat_t (V is the
    row's first kv_lora values); up-project out = W_UV vc.
    [moeflux-fwd] folded SDPA chain (q_prime -> sdpa -> out_per_head);
    [ts-ds2] absorb -> MQA attention -> v-combine.
    """
    N = W_UK.shape[1]
    q_nope = q[:, :N]
    q_pe = q[:, N:] if pos is None else rope_pairs(q[:, N:], pos, inv_freq)
    q_abs = np.concatenate([absorb_query(q_nope, W_UK), q_pe], axis=1)
    p, lse = softmax_lse(scores(q_abs, rows, scale))
    vc = p @ rows[:, :kv_lora]
    out = np.einsum("hvc,hc->hv", W_UV, vc)
    return out, lse


def decode_unabsorbed_one(q: np.ndarray, W_UK: np.ndarray, W_UV: np.ndarray,
                          rows: np.ndarray, pos: Optional[int], inv_freq: np.ndarray,
                          scale: float, kv_lora: int):
    """Plain multi-head attention over decompressed keys and values (the self-check).

    Per head h and row t: K_t = [W_UK,h kv_lat_t ; k_pe_t], V_t = W_UV,h kv_lat_t,
    s_t = scale * [q_nope ; q_pe_rot] . K_t, out = sum_t softmax(s)_t V_t.
    [moeflux-fwd] module doc: the folded path mirrors the unfolded CPU forward.
    """
    N = W_UK.shape[1]
    lat, pe = rows[:, :kv_lora], rows[:, kv_lora:]
    q_pe = q[:, N:] if pos is None else rope_pairs(q[:, N:], pos, inv_freq)
    H = q.shape[0]
    out = np.empty((H, W_UV.shape[1]))
    lse = np.empty(H)
    for h in range(H):
        K = np.concatenate([lat @ W_UK[h].T, pe], axis=1)      # [L, N+R]
        Vv = lat @ W_UV[h].T                                   # [L, V]
        s = scale * (K @ np.concatenate([q[h, :N], q_pe[h]]))
        m = s.max()
        e = np.exp(s - m)
        out[h] = (e @ Vv) / e.sum()
        lse[h] = m + math.log(e.sum())
    return out, lse


def partial_attention(q_abs: np.ndarray, rows: np.ndarray, scale: float, kv_lora: int):
    """One split of the rows: (O_s = softmax-normalised sum of kv_lat over the split,
    lse_s). Used to pin the split/merge structure ([ts-gptoss] split + COMBINE pass)."""
    p, lse = softmax_lse(scores(q_abs, rows, scale))
    return p @ rows[:, :kv_lora], lse


def lse_merge(parts):
    """Merge splits: lse = log sum_s exp(lse_s); O = sum_s exp(lse_s - lse) O_s."""
    lses = np.stack([l for _, l in parts])          # [S, H]
    m = lses.max(axis=0)
    w = np.exp(lses - m)
    tot = w.sum(axis=0)
    lse = m + np.log(tot)
    O = sum((w[s] / tot)[:, None] * parts[s][0] for s in range(len(parts)))
    return O, lse


# ---------------------------------------------------------------------------------------
# Several query tokens per sequence (speculative / chunked decode)
# ---------------------------------------------------------------------------------------

def decode_multi_one(q: np.ndarray, W_UK: np.ndarray, W_UV: np.ndarray, rows: np.ndarray,
                     pos0: Optional[int], inv_freq: np.ndarray, scale: float, kv_lora: int):
    """T query tokens of one sequence whose own rows are the last T of `rows`: token i sits at
    position pos0 + i (its q_pe is rotated there; pos0 None: already rotated) and attends the
    first L - T + 1 + i rows, i.e. itself and every row before it.

    q [T, H, N+R], rows [L, C+R]. Returns out [T, H, V], lse [T, H].
    Each token is one absorbed decode (decode_one); the tokens share the rows. [moeflux-fwd]
    folded SDPA over cache_len = pos + 1 rows, applied per stacked token as the `*_n_tokens`
    batched encoders of moeflux 0.1.0-pre.3, src/riir/backend/gpu/gpu_matvec.rs apply one
    weight matrix to N stacked inputs.
    """
    T, H = q.shape[0], q.shape[1]
    L = rows.shape[0]
    out = np.empty((T, H, W_UV.shape[1]))
    lse = np.empty((T, H))
    for i in range(T):
        pos = None if pos0 is None else pos0 + i
        out[i], lse[i] = decode_one(q[i], W_UK, W_UV, rows[:L - T + 1 + i], pos, inv_freq, scale, kv_lora)
    return out, lse


# ---------------------------------------------------------------------------------------
# Whole step on decoded inputs
# ---------------------------------------------------------------------------------------

def decode_step(q: np.ndarray, kv_b: np.ndarray, seq_rows, positions, inv_freq: np.ndarray,
                scale: float, heads: int, nope: int, v_dim: int, kv_lora: int,
                unabsorbed: bool = False):
    """out [B, H, V], lse [B, H] for all sequences.

    q [B, H, N+R] float64; kv_b [H(N+V), C] float64; seq_rows[b] = [L_b, C+R] float64 rows
    of sequence b in logical order; positions[b] = q RoPE position or None.
    """
    W_UK, W_UV = split_kv_b(kv_b, heads, nope, v_dim)
    one = decode_unabsorbed_one if unabsorbed else decode_one
    B = q.shape[0]
    out = np.empty((B, heads, v_dim))
    lse = np.empty((B, heads))
    for b in range(B):
        pos = None if positions is None else int(positions[b])
        out[b], lse[b] = one(q[b], W_UK, W_UV, seq_rows[b], pos, inv_freq, scale, kv_lora)
    return out, lse
