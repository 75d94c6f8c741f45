"""Seeded synthetic inputs for one MLA decode step (cache append + absorbed decode).

This module only draws random numbers and lays them out in the storage formats the
library reads (bf16 bit patterns, fp32, packed Q8_0 blocks, a paged pool with an int32
page table). It holds none of the method's arithmetic: no RoPE, no norm, no attention.
It is shared by the fp64 oracle's tests, the GPU parity tests and the benchmark, so both
sides of every comparison see the same bytes.

Value recipe (the pages fix shapes, not distributions; these are the workload
definitions' own):
  * q [B, H, nope+rope] ~ N(0, 1) (both the nope and the rope part).
  * latent cache entries ~ N(0, 1) * w[c], with w ~ U(0.5, 1.5) the per-channel weight
    that the append's RMSNorm also uses; k_pe cache entries ~ N(0, 1).
  * kv_b ~ N(0, 1/kv_lora). As Q8_0: int8 codes ~ U{-127..127}, one fp16 scale per
    32-element block ~ U(1e-3, 2e-3).
  * append input: a kv_a row [B, kv_lora+rope] ~ N(0, 1) in fp32, or, for the long-context
    workload, a hidden state x [B, 7168] ~ N(0, 1) and W_kva [kv_lora+rope, 7168] ~
    N(0, 1/7168), both bf16.
  * ragged lengths L_b ~ U{lo..hi}; 64-row pages; a seeded permutation of all physical
    pages handed out to the sequences in order; unused page-table entries are -1.
  * the layer's projections (front end and o_proj): x [B, hidden] ~ N(0, 1); every weight
    [out, in] ~ N(0, 1/in) (as Q8_0: codes ~ U{-127..127}, scales ~ U(0.5, 1.5)/(73.3 sqrt(in));
    4-bit: codes ~ U{0..15}, scales ~ U(0.5, 1.5)/(4.6 sqrt(in)), biases ~ -7.5 scale U(0.9, 1.1),
    so every format has about the same spread); the q_a_layernorm weight ~ U(0.5, 1.5); the
    attention output fed to o_proj [B, H, V] ~ N(0, 1) in fp32.
  * every cache row a step must not read (the append slot before the append, spare
    capacity, the unused tail of a last page) holds a NaN sentinel, so that a kernel
    that reads past a sequence's length shows up in the output.
Each tensor draws from its own PCG64 stream keyed by (seed, tensor tag), so the draw
order does not matter and a tensor can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass
from typing import Optional

import numpy as np

Q8_0_BLOCK_ELEMS = 32
Q8_0_BLOCK_BYTES = 34  # fp16 scale + 32 int8 codes

BF16_NAN_BITS = 0x7FC0

# stream tags: one independent PCG64 stream per tensor
_TAG = {
    "q": 1, "lat": 2, "pe": 3, "norm_w": 4, "kv_b": 5, "kv_b_d": 6, "kva": 7,
    "x": 8, "w_kva": 9, "pages": 10, "lengths": 11,
    "w_q_a": 12, "q_norm_w": 13, "w_q": 14, "w_o": 15, "attn": 16, "w_d": 17,
}


@dataclass(frozen=True)
class Workload:
    """One decode-step workload: dimensions, storage formats and the context recipe."""
    name: str
    B: int
    H: int
    C: int            # kv_lora
    N: int            # qk_nope
    R: int            # qk_rope
    V: int            # v_head
    act: str          # "f32" | "bf16": q and cache-row storage
    kv_b: str         # "f32" | "bf16" | "q8_0"
    # context: ("fixed", P) -> P rows pre-filled, append at position P, attend P+1 rows;
    #          ("uniform", lo, hi) -> L_b ~ U{lo..hi}, append at L_b-1, attend L_b rows
    context: tuple
    page_size: int = 0          # 0 = contiguous per-sequence rows, else rows per page
    append: str = "row"         # "row": kv_a row given; "gemv": x and W_kva given
    hidden: int = 0             # hidden size of x for append="gemv"
    rope_theta: float = 10000.0
    yarn_factor: float = 1.0
    yarn_mscale_coeff: float = 1.0
    yarn_orig_max_pos: int = 4096
    yarn_beta_fast: float = 32.0
    yarn_beta_slow: float = 1.0
    rms_eps: float = 1e-6
    seed: int = 0
    # query tokens per sequence (> 1: multi-token decode; the tokens' own rows are the last
    # `tokens` of the L_b rows, all pre-filled, q is [B, tokens, H, N+R], positions[b] = L_b -
    # tokens is the first token's position, and no row is appended)
    tokens: int = 1

    @property
    def row(self) -> int:
        return self.C + self.R

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads. Shapes follow DeepSeek-V2-Lite / V3-style MLA heads.
WORKLOADS = {
    "tiny_f32": Workload(
        name="tiny_f32", B=1, H=16, C=64, N=32, R=16, V=32, act="f32", kv_b="f32",
        context=("fixed", 64)),
    "v2lite_b1_t4096": Workload(
        name="v2lite_b1_t4096", B=1, H=16, C=512, N=128, R=64, V=128, act="bf16",
        kv_b="bf16", context=("fixed", 4095)),
    "v3_b32_t4096": Workload(
        name="v3_b32_t4096", B=32, H=128, C=512, N=128, R=64, V=128, act="bf16",
        kv_b="bf16", context=("fixed", 4095)),
    "ragged_paged_b64": Workload(
        name="ragged_paged_b64", B=64, H=128, C=512, N=128, R=64, V=128, act="bf16",
        kv_b="bf16", context=("uniform", 128, 32768), page_size=64),
    "long_q8_b4_t131072": Workload(
        name="long_q8_b4_t131072", B=4, H=128, C=512, N=128, R=64, V=128, act="bf16",
        kv_b="q8_0", context=("fixed", 131072), append="gemv", hidden=7168,
        yarn_factor=40.0, yarn_mscale_coeff=1.0),
}


@dataclass
class Problem:
    """Host-side inputs of one step, in the library's storage formats."""
    wl: Workload
    q: np.ndarray                 # [B,H,N+R] uint16 bf16 bits or float32
    pool: np.ndarray              # [n_phys_rows, C+R] uint16 bf16 bits or float32
    page_table: Optional[np.ndarray]  # [B, max_pages] int32, or None (contiguous)
    rows_per_seq: int             # contiguous capacity per sequence (0 when paged)
    max_pages: int                # page-table width (0 when contiguous)
    positions: np.ndarray         # [B] int32: append position = q RoPE position
    seq_lens: np.ndarray          # [B] int32: rows attended after the append (positions+1)
    norm_w: np.ndarray            # [C] float32
    kv_b: np.ndarray              # bf16 bits [H(N+V),C] | float32 [H(N+V),C] | uint8 Q8_0 [H(N+V), C/32*34]
    kva_rows: Optional[np.ndarray] = None   # [B, C+R] float32 (append="row")
    x: Optional[np.ndarray] = None          # [B, hidden] uint16 bf16 bits (append="gemv")
    w_kva: Optional[np.ndarray] = None      # [C+R, hidden] uint16 bf16 bits (append="gemv")

    @property
    def n_phys_rows(self) -> int:
        return self.pool.shape[0]


def _rng(seed: int, tag: str, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, _TAG[tag], sub]))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even storage encoding of float32 values as bf16 bit patterns."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _encode_act(a: np.ndarray, act: str) -> np.ndarray:
    return f32_to_bf16_bits(a) if act == "bf16" else np.ascontiguousarray(a, dtype=np.float32)


def lengths_for(wl: Workload) -> np.ndarray:
    """Rows attended by each sequence after the append (L_b)."""
    kind = wl.context[0]
    if kind == "fixed":
        return np.full(wl.B, wl.context[1] + 1, dtype=np.int32)
    if kind == "uniform":
        lo, hi = wl.context[1], wl.context[2]
        return _rng(wl.seed, "lengths").integers(lo, hi + 1, size=wl.B).astype(np.int32)
    raise ValueError(f"unknown context kind {kind!r}")


def _q8_0_pack(codes: np.ndarray, scales_f16: np.ndarray) -> np.ndarray:
    """Pack int8 codes [rows, cols] and fp16 scales [rows, cols/32] into 34-byte blocks."""
    rows, cols = codes.shape
    nb = cols // Q8_0_BLOCK_ELEMS
    out = np.empty((rows, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = scales_f16.astype("<f2").view(np.uint8).reshape(rows, nb, 2)
    out[:, :, 2:] = codes.astype(np.int8).view(np.uint8).reshape(rows, nb, Q8_0_BLOCK_ELEMS)
    return out.reshape(rows, nb * Q8_0_BLOCK_BYTES)


def q4_affine_pack(codes: np.ndarray, scales_bits: np.ndarray, biases_bits: np.ndarray) -> np.ndarray:
    """Storage of a 4-bit affine matrix as one byte buffer: codes [rows, cols] (0..15) as
    little-endian 32-bit words of 8 (code j of a word in bits 4j..4j+3), then the bf16 scale
    and bias bit patterns [rows, cols/64], row-major."""
    rows, cols = codes.shape
    c = codes.astype(np.uint32).reshape(rows, cols // 8, 8)
    words = np.zeros((rows, cols // 8), dtype=np.uint32)
    for j in range(8):
        words |= c[:, :, j] << np.uint32(4 * j)
    return np.concatenate([words.astype("<u4").view(np.uint8).reshape(-1),
                           np.ascontiguousarray(scales_bits, dtype="<u2").view(np.uint8).reshape(-1),
                           np.ascontiguousarray(biases_bits, dtype="<u2").view(np.uint8).reshape(-1)])


def make_kv_b(wl: Workload) -> np.ndarray:
    rows = wl.H * (wl.N + wl.V)
    if wl.kv_b == "q4_affine":
        # codes U{0..15}; per 64-column group a scale near 1/(4.6 sqrt(C)) (so values have about
        # the spread of the bf16 draw's N(0, 1/C)) and a bias near -7.5 * scale (centred codes)
        if wl.C % 64:
            raise ValueError("4-bit affine kv_b needs kv_lora % 64 == 0")
        g = wl.C // 64
        codes = _rng(wl.seed, "kv_b").integers(0, 16, size=(rows, wl.C), dtype=np.int16)
        s = _rng(wl.seed, "kv_b_d").uniform(0.5, 1.5, size=(rows, g)) / (4.6 * math.sqrt(wl.C))
        bias = -7.5 * s * _rng(wl.seed, "kv_b_d", 1).uniform(0.9, 1.1, size=(rows, g))
        return q4_affine_pack(codes, f32_to_bf16_bits(s.astype(np.float32)),
                              f32_to_bf16_bits(bias.astype(np.float32)))
    if wl.kv_b == "q8_0":
        if wl.C % Q8_0_BLOCK_ELEMS:
            raise ValueError("Q8_0 kv_b needs kv_lora % 32 == 0")
        codes = _rng(wl.seed, "kv_b").integers(-127, 128, size=(rows, wl.C), dtype=np.int16)
        d = _rng(wl.seed, "kv_b_d").uniform(1e-3, 2e-3, size=(rows, wl.C // Q8_0_BLOCK_ELEMS))
        return _q8_0_pack(codes, d.astype(np.float16))
    w = _rng(wl.seed, "kv_b").standard_normal((rows, wl.C), dtype=np.float32)
    w *= np.float32(1.0 / math.sqrt(wl.C))
    return _encode_act(w, wl.kv_b)


def make_weight(seed: int, tag: str, rows: int, cols: int, fmt: str) -> np.ndarray:
    """A projection weight [rows, cols] (out, in) in storage format `fmt`, drawn so that each
    element has about the spread of N(0, 1/cols) whatever the format."""
    sub = rows * 7919 + cols
    rng, rng_d = _rng(seed, tag, sub), _rng(seed, "w_d", sub)
    if fmt == "q8_0":
        if cols % Q8_0_BLOCK_ELEMS:
            raise ValueError("Q8_0 weights need in_dim % 32 == 0")
        codes = rng.integers(-127, 128, size=(rows, cols), dtype=np.int16)
        d = rng_d.uniform(0.5, 1.5, size=(rows, cols // Q8_0_BLOCK_ELEMS)) / (73.3 * math.sqrt(cols))
        return _q8_0_pack(codes, d.astype(np.float16))
    if fmt == "q4_affine":
        if cols % 64:
            raise ValueError("4-bit weights need in_dim % 64 == 0")
        codes = rng.integers(0, 16, size=(rows, cols), dtype=np.int16)
        sc = rng_d.uniform(0.5, 1.5, size=(rows, cols // 64)) / (4.6 * math.sqrt(cols))
        bias = -7.5 * sc * rng_d.uniform(0.9, 1.1, size=(rows, cols // 64))
        return q4_affine_pack(codes, f32_to_bf16_bits(sc.astype(np.float32)),
                              f32_to_bf16_bits(bias.astype(np.float32)))
    w = rng.standard_normal((rows, cols), dtype=np.float32)
    w *= np.float32(1.0 / math.sqrt(cols))
    return _encode_act(w, fmt)


@dataclass(frozen=True)
class ProjWorkload:
    """The layer's projections around one decode step: the front end (the Q chain or a direct
    q projection, plus kv_a) and o_proj, for B sequences."""
    name: str
    B: int
    H: int
    C: int
    N: int
    R: int
    V: int
    hidden: int
    q_lora: int       # 0: one direct q projection [H(N+R), hidden]
    act: str          # "f32" | "bf16": x and q storage
    w: str            # weight format of every projection: "f32" | "bf16" | "q8_0" | "q4_affine"
    eps: float = 1e-6
    seed: int = 0

    def with_(self, **kw) -> "ProjWorkload":
        return dataclasses.replace(self, **kw)


# V2-Lite-shaped (no q rank, hidden 2048, 16 heads) and V3-shaped (q rank 1536, hidden 7168,
# 128 heads) layers, plus a tiny fp32 one.
PROJ_WORKLOADS = {
    "tiny_proj_f32": ProjWorkload(name="tiny_proj_f32", B=3, H=4, C=64, N=32, R=16, V=32, hidden=256,
                                  q_lora=128, act="f32", w="f32"),
    "v2lite_proj_b1": ProjWorkload(name="v2lite_proj_b1", B=1, H=16, C=512, N=128, R=64, V=128, hidden=2048,
                                   q_lora=0, act="bf16", w="bf16"),
    "v3_proj_b4": ProjWorkload(name="v3_proj_b4", B=4, H=128, C=512, N=128, R=64, V=128, hidden=7168,
                               q_lora=1536, act="bf16", w="bf16"),
    "v3_proj_b64": ProjWorkload(name="v3_proj_b64", B=64, H=128, C=512, N=128, R=64, V=128, hidden=7168,
                                q_lora=1536, act="bf16", w="bf16"),
}


@dataclass
class ProjProblem:
    """Host-side inputs of the projections, in the library's storage formats."""
    wl: ProjWorkload
    x: np.ndarray                   # [B, hidden] act storage
    w_q_a: Optional[np.ndarray]     # [q_lora, hidden] (q_lora > 0)
    q_a_norm_w: Optional[np.ndarray]  # [q_lora] float32
    w_q: np.ndarray                 # [H(N+R), q_lora or hidden]
    w_kva: np.ndarray               # [C+R, hidden]
    w_o: np.ndarray                 # [hidden, H*V]
    attn: np.ndarray                # [B, H, V] float32: o_proj's input


def make_proj_problem(wl: ProjWorkload) -> ProjProblem:
    """Draw every input of the projections for workload `wl`."""
    x = _encode_act(_rng(wl.seed, "x").standard_normal((wl.B, wl.hidden), dtype=np.float32), wl.act)
    q_rows = wl.H * (wl.N + wl.R)
    if wl.q_lora > 0:
        w_q_a = make_weight(wl.seed, "w_q_a", wl.q_lora, wl.hidden, wl.w)
        q_a_norm_w = _rng(wl.seed, "q_norm_w").uniform(0.5, 1.5, size=wl.q_lora).astype(np.float32)
        w_q = make_weight(wl.seed, "w_q", q_rows, wl.q_lora, wl.w)
    else:
        w_q_a, q_a_norm_w = None, None
        w_q = make_weight(wl.seed, "w_q", q_rows, wl.hidden, wl.w)
    w_kva = make_weight(wl.seed, "w_kva", wl.C + wl.R, wl.hidden, wl.w)
    w_o = make_weight(wl.seed, "w_o", wl.hidden, wl.H * wl.V, wl.w)
    attn = _rng(wl.seed, "attn").standard_normal((wl.B, wl.H, wl.V), dtype=np.float32)
    return ProjProblem(wl=wl, x=x, w_q_a=w_q_a, q_a_norm_w=q_a_norm_w, w_q=w_q, w_kva=w_kva, w_o=w_o,
                       attn=attn)


def make_problem(wl: Workload, nan_fill: bool = True) -> Problem:
    """Draw every input of one step for workload `wl`."""
    B, H, C, N, R = wl.B, wl.H, wl.C, wl.N, wl.R
    row = C + R
    L = lengths_for(wl)
    T = wl.tokens
    if T > 1 and int(L.min()) < T:
        raise ValueError("every sequence needs at least one row per query token")
    positions = (L - T).astype(np.int32)
    norm_w = _rng(wl.seed, "norm_w").uniform(0.5, 1.5, size=C).astype(np.float32)

    q_shape = (B, H, N + R) if T == 1 else (B, T, H, N + R)
    q = _rng(wl.seed, "q").standard_normal(q_shape, dtype=np.float32)
    q = _encode_act(q, wl.act)

    # physical placement of logical row (b, t)
    if wl.page_size:
        ps = wl.page_size
        pages_per_seq = (L + ps - 1) // ps
        n_pages = int(pages_per_seq.sum())
        max_pages = int((int(L.max()) + ps - 1) // ps)
        if wl.context[0] == "uniform":
            max_pages = (wl.context[2] + ps - 1) // ps
        perm = _rng(wl.seed, "pages").permutation(n_pages).astype(np.int32)
        page_table = np.full((B, max_pages), -1, dtype=np.int32)
        k = 0
        for b in range(B):
            page_table[b, :pages_per_seq[b]] = perm[k:k + pages_per_seq[b]]
            k += pages_per_seq[b]
        n_phys = n_pages * ps
        rows_per_seq = 0
    else:
        page_table = None
        max_pages = 0
        rows_per_seq = int(L.max())
        n_phys = B * rows_per_seq

    dt = np.uint16 if wl.act == "bf16" else np.float32
    pool = np.empty((n_phys, row), dtype=dt)
    if wl.act == "bf16":
        pool.fill(BF16_NAN_BITS if nan_fill else 0)
    else:
        pool.fill(np.nan if nan_fill else 0.0)

    rng_lat = _rng(wl.seed, "lat")
    rng_pe = _rng(wl.seed, "pe")
    chunk = 1 << 14
    for b in range(B):
        # rows 0..P-1 pre-filled, row P the append slot; several tokens: every row pre-filled
        n_pre = int(positions[b]) if T == 1 else int(L[b])
        for t0 in range(0, n_pre, chunk):
            t1 = min(n_pre, t0 + chunk)
            lat = rng_lat.standard_normal((t1 - t0, C), dtype=np.float32) * norm_w[None, :]
            pe = rng_pe.standard_normal((t1 - t0, R), dtype=np.float32)
            vals = _encode_act(np.concatenate([lat, pe], axis=1), wl.act)
            t = np.arange(t0, t1)
            if page_table is not None:
                phys = page_table[b, t // wl.page_size].astype(np.int64) * wl.page_size + t % wl.page_size
            else:
                phys = b * rows_per_seq + t
            pool[phys] = vals

    kv_b = make_kv_b(wl)

    prob = Problem(wl=wl, q=q, pool=pool, page_table=page_table, rows_per_seq=rows_per_seq,
                   max_pages=max_pages, positions=positions, seq_lens=L.astype(np.int32),
                   norm_w=norm_w, kv_b=kv_b)
    if wl.append == "row":
        prob.kva_rows = _rng(wl.seed, "kva").standard_normal((B, row), dtype=np.float32)
    elif wl.append == "gemv":
        x = _rng(wl.seed, "x").standard_normal((B, wl.hidden), dtype=np.float32)
        w = _rng(wl.seed, "w_kva").standard_normal((row, wl.hidden), dtype=np.float32)
        w *= np.float32(1.0 / math.sqrt(wl.hidden))
        prob.x = f32_to_bf16_bits(x)
        prob.w_kva = f32_to_bf16_bits(w)
    else:
        raise ValueError(f"unknown append mode {wl.append!r}")
    return prob

