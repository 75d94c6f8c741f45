"""The whole step (append, then decode) on a synthetic problem, in fp64.

TEST INFRASTRUCTURE (same rule as mla_oracle): used by the tests, the smoke check and
the benchmark's CPU baseline only. It takes any object with the attributes the seeded
generator's `Problem` has (wl, q, pool, page_table, rows_per_seq, positions, seq_lens,
norm_w, kv_b, kva_rows | x, w_kva) and reads nothing but those arrays.
"""
from __future__ import annotations

import math

import numpy as np

from . import mla_oracle as O


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (8 significant bits), ties to even.
    Used once, where the cache stores the finished row in bf16."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def store(x: np.ndarray, act: str) -> np.ndarray:
    """The value a cache of dtype `act` holds for x (one rounding)."""
    if act == "bf16":
        return round_to_bf16(x)
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def decode_act(a: np.ndarray, act: str) -> np.ndarray:
    return O.bf16_to_f64(a) if act == "bf16" else O.f32_to_f64(a)


def kv_b_f64(prob) -> np.ndarray:
    wl = prob.wl
    if wl.kv_b == "q8_0":
        return O.q8_0_to_f64(prob.kv_b, wl.C)
    if wl.kv_b == "q4_affine":
        return O.q4_affine_to_f64(prob.kv_b, wl.H * (wl.N + wl.V), wl.C)
    return decode_act(prob.kv_b, wl.kv_b)


def tables(wl):
    """(inv_freq, softmax scale) for a workload's RoPE / YaRN parameters."""
    inv = O.yarn_inv_freq(wl.R, wl.rope_theta, wl.yarn_factor, wl.yarn_orig_max_pos,
                          wl.yarn_beta_fast, wl.yarn_beta_slow)
    ms = O.yarn_mscale(wl.yarn_factor, wl.yarn_mscale_coeff)
    return inv, O.softmax_scale(wl.N, wl.R, ms)


def appended_rows(prob) -> np.ndarray:
    """[B, C+R] float64: the finished rows the append writes, before storage rounding."""
    wl = prob.wl
    inv, _ = tables(wl)
    if prob.kva_rows is not None:
        kva = np.asarray(prob.kva_rows, dtype=np.float64)
    else:
        kva = O.kv_a_rows(O.bf16_to_f64(prob.x), O.bf16_to_f64(prob.w_kva))
    return O.append_rows(kva, prob.norm_w.astype(np.float64), prob.positions, inv,
                         wl.C, wl.rms_eps)


def sequence_rows(prob, b: int, new_row=None) -> np.ndarray:
    """[L_b, C+R] float64 rows sequence b attends, in logical order. With `new_row` the
    row at positions[b] is replaced by it (the cache state after the append)."""
    wl = prob.wl
    L = int(prob.seq_lens[b])
    phys = O.physical_row(b, np.arange(L), prob.page_table, wl.page_size, prob.rows_per_seq)
    rows = decode_act(prob.pool[phys], wl.act)
    if new_row is not None:
        rows[int(prob.positions[b])] = new_row
    return rows


def run_step(prob, seqs=None, heads=None, with_append: bool = True):
    """Append (when `with_append`) then decode. Returns (appended rows as stored
    [B, C+R] float64, out [nb, nh, V], lse [nb, nh]) over the chosen sequences/heads."""
    wl = prob.wl
    inv, scale = tables(wl)
    q = decode_act(prob.q, wl.act)
    kvb = kv_b_f64(prob)
    W_UK, W_UV = O.split_kv_b(kvb, wl.H, wl.N, wl.V)
    seqs = range(wl.B) if seqs is None else list(seqs)
    heads = np.arange(wl.H) if heads is None else np.asarray(heads)
    new = store(appended_rows(prob), wl.act) if with_append else None
    out = np.empty((len(seqs), len(heads), wl.V))
    lse = np.empty((len(seqs), len(heads)))
    for i, b in enumerate(seqs):
        rows = sequence_rows(prob, b, None if new is None else new[b])
        out[i], lse[i] = O.decode_one(q[b, heads], W_UK[heads], W_UV[heads], rows,
                                      int(prob.positions[b]), inv, scale, wl.C)
    return new, out, lse


def run_multi(prob, seqs=None, heads=None):
    """Multi-token decode of a problem whose workload has tokens > 1 (no append: every row is
    in the pool). Returns (out [nb, T, nh, V], lse [nb, T, nh]) over the chosen sequences/heads."""
    wl = prob.wl
    inv, scale = tables(wl)
    q = decode_act(prob.q, wl.act)
    W_UK, W_UV = O.split_kv_b(kv_b_f64(prob), wl.H, wl.N, wl.V)
    seqs = range(wl.B) if seqs is None else list(seqs)
    heads = np.arange(wl.H) if heads is None else np.asarray(heads)
    out = np.empty((len(seqs), wl.tokens, len(heads), wl.V))
    lse = np.empty((len(seqs), wl.tokens, len(heads)))
    for i, b in enumerate(seqs):
        out[i], lse[i] = O.decode_multi_one(q[b][:, heads], W_UK[heads], W_UV[heads], sequence_rows(prob, b),
                                            int(prob.positions[b]), inv, scale, wl.C)
    return out, lse


def rows_per_second_sample(prob, seconds: float = 10.0, heads=None):
    """Time the oracle on the host over a bounded sample of a workload: whole steps for one
    sequence at a time (all or `heads` of its heads), cycling through the sequences, until
    `seconds` elapse (at least one). Returns (rows per second, counting a row once per full
    set of heads; sequence-steps run; rows credited; elapsed seconds)."""
    import time
    H = prob.wl.H
    hs = None if heads is None else np.arange(min(int(heads), H))
    frac = 1.0 if hs is None else len(hs) / H
    t0 = time.perf_counter()
    n = 0
    rows = 0.0
    while True:
        b = n % prob.wl.B
        run_step(prob, seqs=[b], heads=hs)
        rows += float(prob.seq_lens[b]) * frac
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return rows / dt, n, rows, dt


# ---------------------------------------------------------------------------------------
# The layer's projections on a synthetic ProjProblem (x, w_q_a, q_a_norm_w, w_q, w_kva, w_o,
# attn and its workload's dims and formats)
# ---------------------------------------------------------------------------------------

def weight_f64(blob: np.ndarray, rows: int, cols: int, fmt: str) -> np.ndarray:
    """A stored [rows, cols] weight decoded exactly to float64."""
    if fmt == "q8_0":
        return O.q8_0_to_f64(blob, cols)
    if fmt == "q4_affine":
        return O.q4_affine_to_f64(blob, rows, cols)
    return decode_act(blob, fmt).reshape(rows, cols)


def front_end(pp):
    """(q [B, H, N+R], kva [B, C+R]) in float64: the Q chain (or the direct q projection) and
    the kv_a projection of the problem's x."""
    wl = pp.wl
    x = decode_act(pp.x, wl.act)
    qk = wl.N + wl.R
    if wl.q_lora > 0:
        q = O.q_chain(x, weight_f64(pp.w_q_a, wl.q_lora, wl.hidden, wl.w), pp.q_a_norm_w, wl.eps,
                      weight_f64(pp.w_q, wl.H * qk, wl.q_lora, wl.w), wl.H, qk)
    else:
        q = O.q_direct(x, weight_f64(pp.w_q, wl.H * qk, wl.hidden, wl.w), wl.H, qk)
    kva = O.kv_a_rows(x, weight_f64(pp.w_kva, wl.C + wl.R, wl.hidden, wl.w))
    return q, kva


def o_proj(pp, attn=None) -> np.ndarray:
    """y [B, hidden] in float64 = o_proj of `attn` (default: the problem's own input)."""
    wl = pp.wl
    a = O.f32_to_f64(pp.attn) if attn is None else np.asarray(attn, dtype=np.float64)
    return O.o_proj(a, weight_f64(pp.w_o, wl.hidden, wl.H * wl.V, wl.w))
