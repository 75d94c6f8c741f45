"""Pins for the fp64 oracle: each test checks it against something other than itself
(a closed form, an identity of the mathematics, or the pages' own fixture), chosen so
that a plausible slip (dropped term, wrong sign or index, transposed operand, swapped
kv_b blocks, wrong RoPE pairing, wrong ramp direction) fails at least one of them."""
import json
import math
import os

import numpy as np
import pytest

from oracle import mla_oracle as O
from oracle import step as OS

RNG = np.random.default_rng(12345)


def rand_problem(H, C, N, R, V, L, rng=RNG):
    q = rng.standard_normal((H, N + R))
    kv_b = rng.standard_normal((H * (N + V), C)) / math.sqrt(C)
    rows = rng.standard_normal((L, C + R))
    inv = O.yarn_inv_freq(R, 10000.0, 1.0, 4096, 32.0, 1.0)
    return q, kv_b, rows, inv


# ----------------------------------------------------------------------------------------
# absorbed == unabsorbed (plain MHA with decompressed K and V)
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("H,C,N,R,V,L,pos", [
    (1, 8, 4, 2, 3, 1, 0),
    (2, 16, 6, 4, 5, 7, 3),
    (3, 32, 8, 8, 12, 33, 100),
    (16, 64, 32, 16, 32, 65, 64),
    (4, 24, 10, 6, 7, 129, 5000),
])
def test_absorbed_equals_unabsorbed(H, C, N, R, V, L, pos):
    q, kv_b, rows, inv = rand_problem(H, C, N, R, V, L)
    W_UK, W_UV = O.split_kv_b(kv_b, H, N, V)
    scale = O.softmax_scale(N, R, 1.0)
    o1, l1 = O.decode_one(q, W_UK, W_UV, rows, pos, inv, scale, C)
    o2, l2 = O.decode_unabsorbed_one(q, W_UK, W_UV, rows, pos, inv, scale, C)
    assert np.max(np.abs(o1 - o2)) <= 1e-12 * max(1.0, np.max(np.abs(o2)))
    assert np.max(np.abs(l1 - l2)) <= 1e-12 * max(1.0, np.max(np.abs(l2)))


def test_scale_changes_result():
    # the scale enters the scores: a different scale must change out (guards a dropped scale)
    q, kv_b, rows, inv = rand_problem(2, 16, 6, 4, 5, 9)
    W_UK, W_UV = O.split_kv_b(kv_b, 2, 6, 5)
    o1, _ = O.decode_one(q, W_UK, W_UV, rows, 2, inv, 0.2, 16)
    o2, _ = O.decode_one(q, W_UK, W_UV, rows, 2, inv, 0.4, 16)
    assert np.max(np.abs(o1 - o2)) > 1e-6


# ----------------------------------------------------------------------------------------
# T = 1, identical rows, zero query: closed forms
# ----------------------------------------------------------------------------------------

def _kv_b_from_blocks(W_UK, W_UV):
    """Assemble kv_b from per-head blocks in the documented order (nope rows, then v rows)."""
    H = W_UK.shape[0]
    return np.concatenate([np.concatenate([W_UK[h], W_UV[h]], axis=0) for h in range(H)], axis=0)


def test_single_row_gives_up_projected_latent():
    rng = np.random.default_rng(1)
    H, C, N, R, V = 3, 16, 5, 4, 6
    W_UK = rng.standard_normal((H, N, C))
    W_UV = rng.standard_normal((H, V, C))
    kv_b = _kv_b_from_blocks(W_UK, W_UV)
    q = rng.standard_normal((H, N + R))
    rows = rng.standard_normal((1, C + R))
    inv = O.yarn_inv_freq(R, 10000.0, 1.0, 4096, 32.0, 1.0)
    uk, uv = O.split_kv_b(kv_b, H, N, V)
    out, _ = O.decode_one(q, uk, uv, rows, 7, inv, 0.3, C)
    for h in range(H):
        np.testing.assert_allclose(out[h], W_UV[h] @ rows[0, :C], rtol=1e-13, atol=1e-13)


def test_zero_query_gives_lse_zero_and_mean_value():
    # q = 0 -> all scores 0 -> lse = ln L, uniform weights -> out = W_UV mean(lat)
    rng = np.random.default_rng(2)
    H, C, N, R, V, L = 2, 8, 3, 2, 4, 11
    W_UK = rng.standard_normal((H, N, C))
    W_UV = rng.standard_normal((H, V, C))
    kv_b = _kv_b_from_blocks(W_UK, W_UV)
    uk, uv = O.split_kv_b(kv_b, H, N, V)
    rows = rng.standard_normal((L, C + R))
    inv = O.yarn_inv_freq(R, 10000.0, 1.0, 4096, 32.0, 1.0)
    out, lse = O.decode_one(np.zeros((H, N + R)), uk, uv, rows, 3, inv, 0.5, C)
    np.testing.assert_allclose(lse, np.full(H, math.log(L)), rtol=0, atol=1e-14)
    for h in range(H):
        np.testing.assert_allclose(out[h], W_UV[h] @ rows[:, :C].mean(axis=0), rtol=1e-12, atol=1e-13)


def test_identical_rows_lse_adds_log_count():
    rng = np.random.default_rng(3)
    H, C, N, R, V = 2, 8, 3, 2, 4
    q, kv_b, row, inv = rand_problem(H, C, N, R, V, 1, rng)
    uk, uv = O.split_kv_b(kv_b, H, N, V)
    o1, l1 = O.decode_one(q, uk, uv, row, 9, inv, 0.25, C)
    rows = np.repeat(row, 37, axis=0)
    o2, l2 = O.decode_one(q, uk, uv, rows, 9, inv, 0.25, C)
    np.testing.assert_allclose(o2, o1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1 + math.log(37), rtol=0, atol=1e-12)


def test_kv_b_block_order_pins_w_uk_rows():
    # zero W_UK (the nope rows of each head) and zero q_pe: scores are all zero, so out must
    # be W_UV applied to the mean latent. A split that took the v rows as W_UK would give
    # nonzero scores and a different out.
    rng = np.random.default_rng(4)
    H, C, N, R, V, L = 2, 8, 3, 2, 5, 13
    W_UK = np.zeros((H, N, C))
    W_UV = rng.standard_normal((H, V, C))
    kv_b = _kv_b_from_blocks(W_UK, W_UV)
    uk, uv = O.split_kv_b(kv_b, H, N, V)
    q = rng.standard_normal((H, N + R))
    q[:, N:] = 0.0
    rows = rng.standard_normal((L, C + R))
    inv = O.yarn_inv_freq(R, 10000.0, 1.0, 4096, 32.0, 1.0)
    out, lse = O.decode_one(q, uk, uv, rows, 3, inv, 0.7, C)
    np.testing.assert_allclose(lse, np.full(H, math.log(L)), atol=1e-14)
    for h in range(H):
        np.testing.assert_allclose(out[h], W_UV[h] @ rows[:, :C].mean(axis=0), rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------------------
# softmax and split / merge
# ----------------------------------------------------------------------------------------

def test_softmax_rows_sum_to_one_and_shift_invariant():
    s = RNG.standard_normal((5, 40)) * 3
    p, lse = O.softmax_lse(s)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-15)
    p2, lse2 = O.softmax_lse(s + 123.0)
    np.testing.assert_allclose(p2, p, atol=1e-15)
    np.testing.assert_allclose(lse2, lse + 123.0, atol=1e-12)
    # lse against the unshifted definition on small scores
    np.testing.assert_allclose(lse, np.log(np.exp(s).sum(axis=1)), rtol=1e-14)


@pytest.mark.parametrize("cuts", [[5], [1, 2, 3], [10, 11], [1, 30, 31, 60]])
def test_split_merge_equals_one_pass(cuts):
    H, C, R, L = 4, 16, 4, 64
    q_abs = RNG.standard_normal((H, C + R))
    rows = RNG.standard_normal((L, C + R))
    O1, l1 = O.partial_attention(q_abs, rows, 0.3, C)
    edges = [0] + cuts + [L]
    parts = [O.partial_attention(q_abs, rows[a:b], 0.3, C) for a, b in zip(edges[:-1], edges[1:])]
    O2, l2 = O.lse_merge(parts)
    np.testing.assert_allclose(O2, O1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-12)


# ----------------------------------------------------------------------------------------
# RoPE: consecutive pairs, pure rotation
# ----------------------------------------------------------------------------------------

INV16 = O.yarn_inv_freq(16, 10000.0, 1.0, 4096, 32.0, 1.0)


def test_rope_identity_at_position_zero():
    x = RNG.standard_normal((3, 16))
    np.testing.assert_array_equal(O.rope_pairs(x, 0, INV16), x)


def test_rope_preserves_each_pair_norm():
    x = RNG.standard_normal((5, 16))
    y = O.rope_pairs(x, 977, INV16)
    np.testing.assert_allclose(np.hypot(y[:, 0::2], y[:, 1::2]), np.hypot(x[:, 0::2], x[:, 1::2]),
                               rtol=1e-14)


@pytest.mark.parametrize("i", [0, 3, 7])
def test_rope_pairs_consecutive_elements(i):
    # e_{2i} rotates into index 2i+1 only: the (i, i + d/2) pairing would move it to i + d/2
    x = np.zeros(16)
    x[2 * i] = 1.0
    pos = 5
    y = O.rope_pairs(x, pos, INV16)
    a = pos * INV16[i]
    expect = np.zeros(16)
    expect[2 * i] = math.cos(a)
    expect[2 * i + 1] = math.sin(a)
    np.testing.assert_allclose(y, expect, atol=1e-15)


def test_rope_equals_complex_multiplication():
    # pair (x0, x1) as x0 + i x1, multiplied by exp(i * pos * inv_freq)
    x = RNG.standard_normal((4, 16))
    pos = 4097
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * pos * INV16)
    y = O.rope_pairs(x, pos, INV16)
    np.testing.assert_allclose(y[:, 0::2], z.real, atol=1e-12)
    np.testing.assert_allclose(y[:, 1::2], z.imag, atol=1e-12)


def test_rope_composition_and_relative_position():
    x = RNG.standard_normal(16)
    k = RNG.standard_normal(16)
    np.testing.assert_allclose(O.rope_pairs(O.rope_pairs(x, 30, INV16), 12, INV16),
                               O.rope_pairs(x, 42, INV16), atol=1e-12)
    d1 = O.rope_pairs(x, 100, INV16) @ O.rope_pairs(k, 60, INV16)
    d2 = O.rope_pairs(x, 40, INV16) @ k
    assert abs(d1 - d2) < 1e-12


# ----------------------------------------------------------------------------------------
# YaRN table and scales
# ----------------------------------------------------------------------------------------

def test_yarn_factor_one_is_plain_rope():
    for d in (16, 64):
        inv = O.yarn_inv_freq(d, 10000.0, 1.0, 4096, 32.0, 1.0)
        np.testing.assert_allclose(inv, [10000.0 ** (-2.0 * i / d) for i in range(d // 2)], rtol=1e-15)


def test_yarn_ramp_limits(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "yarn_rope64_theta1e4_factor40.json")))
    d = g["rope_dim"]
    inv = O.yarn_inv_freq(d, g["theta"], g["factor"], g["orig_max_pos"], g["beta_fast"], g["beta_slow"])
    base = np.array([g["theta"] ** (-2.0 * i / d) for i in range(d // 2)])
    lo, hi = g["ramp_lo"], g["ramp_hi"]
    # pairs at or below the fast correction dim keep the base frequency (high frequencies)
    np.testing.assert_allclose(inv[:lo + 1], base[:lo + 1], rtol=1e-15)
    # pairs at or above the slow correction dim are fully interpolated: base / factor
    np.testing.assert_allclose(inv[hi:], base[hi:] / g["factor"], rtol=1e-15)
    # in between, the interpolation weight rises linearly: ratio base/inv moves from 1 to factor
    ramp = (np.arange(lo, hi + 1) - lo) / (hi - lo)
    np.testing.assert_allclose(inv[lo:hi + 1] / base[lo:hi + 1], 1 - ramp + ramp / g["factor"], rtol=1e-14)


def test_mscale_and_softmax_scale(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "yarn_rope64_theta1e4_factor40.json")))
    assert abs(O.yarn_mscale(40.0, 1.0) - g["mscale"]) < 1e-15
    assert O.yarn_mscale(1.0, 1.0) == 1.0
    assert abs(O.softmax_scale(128, 64, O.yarn_mscale(40.0)) - g["softmax_scale_nope128_rope64"]) < 1e-13
    assert abs(O.softmax_scale(32, 16, 1.0) - g["softmax_scale_plain_nope32_rope16"]) < 1e-16
    assert abs(O.softmax_scale(128, 64, 1.0) - g["softmax_scale_plain_nope128_rope64"]) < 1e-16


# ----------------------------------------------------------------------------------------
# RMSNorm
# ----------------------------------------------------------------------------------------

def test_rms_norm_unit_rms_and_scale_invariance():
    x = RNG.standard_normal((3, 64)) * 5
    w = np.ones(64)
    y = O.rms_norm(x, w, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, rtol=1e-14)
    np.testing.assert_allclose(O.rms_norm(7.5 * x, w, 0.0), y, rtol=1e-14)
    wv = RNG.uniform(0.5, 1.5, 64)
    np.testing.assert_allclose(O.rms_norm(x, wv, 0.0) / wv, y, rtol=1e-14)


def test_rms_norm_eps_closed_form():
    # constant input c: mean square = c^2, so y = c / sqrt(c^2 + eps)
    c, eps = 1e-3, 1e-6
    y = O.rms_norm(np.full(8, c), np.full(8, 2.0), eps)
    np.testing.assert_allclose(y, 2.0 * c / math.sqrt(c * c + eps), rtol=1e-15)


# ----------------------------------------------------------------------------------------
# Q8_0
# ----------------------------------------------------------------------------------------

def test_q8_0_golden_blocks(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "q8_0_blocks.json")))
    raw = bytearray()
    expect = []
    for blk in g["blocks"]:
        raw += int(blk["d_f16_bits"]).to_bytes(2, "little")
        raw += bytes((c & 0xFF) for c in blk["codes"])
        expect += blk["values"]
    blob = np.frombuffer(bytes(raw), dtype=np.uint8).reshape(1, -1)
    got = O.q8_0_to_f64(blob, 64)
    np.testing.assert_array_equal(got[0], np.array(expect))


def test_q8_0_validation_fixture(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "q8_0_kv_b_validation.json")))
    args = (g["heads"], g["nope"], g["kv_lora"], g["v_dim"])
    v = g["valid"]
    assert O.q8_0_validate(v["dtype"], v["shape"], v["size_bytes"], *args) is None
    for r in g["rejects"]:
        assert O.q8_0_validate(r["dtype"], r["shape"], r["size_bytes"], *args) is not None, r["why"]
    # a width that does not tile 32-element blocks
    assert O.q8_0_validate("q8_0", (12, 48), 12 * 2 * 34, 4, 2, 48, 1) is not None


# ----------------------------------------------------------------------------------------
# cache addressing, append, storage rounding
# ----------------------------------------------------------------------------------------

def test_physical_row_paged_and_contiguous():
    pt = np.array([[3, 1, -1], [0, 2, 4]], dtype=np.int32)
    assert O.physical_row(0, 0, pt, 64, 0) == 192
    assert O.physical_row(0, 70, pt, 64, 0) == 70          # page 1 -> rows 64..127
    assert O.physical_row(1, 5, pt, 64, 0) == 5
    assert O.physical_row(1, 130, pt, 64, 0) == 4 * 64 + 2
    assert O.physical_row(2, 17, None, 0, 100) == 217


def test_append_rows_norm_and_rope_parts():
    rng = np.random.default_rng(5)
    C, R, B = 32, 8, 3
    kva = rng.standard_normal((B, C + R)) * 3
    w = rng.uniform(0.5, 1.5, C)
    inv = O.yarn_inv_freq(R, 10000.0, 1.0, 4096, 32.0, 1.0)
    pos = [0, 17, 4096]
    rows = O.append_rows(kva, w, pos, inv, C, 0.0)
    # latent: unit RMS once the weight is divided out
    np.testing.assert_allclose(np.sqrt(np.mean((rows[:, :C] / w) ** 2, axis=1)), 1.0, rtol=1e-14)
    # k_pe: untouched at position 0, rotated (not normed) elsewhere
    np.testing.assert_array_equal(rows[0, C:], kva[0, C:])
    for b in range(B):
        z = (kva[b, C::2] + 1j * kva[b, C + 1::2]) * np.exp(1j * pos[b] * inv)
        np.testing.assert_allclose(rows[b, C::2], z.real, atol=1e-12)
        np.testing.assert_allclose(rows[b, C + 1::2], z.imag, atol=1e-12)


def test_round_to_bf16_matches_ieee_rounding_on_float32_grid():
    # for values already on the fp32 grid, bf16 RNE rounding is the fp32->bf16 rounding
    import torch
    x = np.concatenate([RNG.standard_normal(5000).astype(np.float32),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0], np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(OS.round_to_bf16(x.astype(np.float64)), ref)


def test_kv_a_projection_is_matvec():
    x = RNG.standard_normal((2, 12))
    w = RNG.standard_normal((5, 12))
    np.testing.assert_allclose(O.kv_a_rows(x, w)[1], [sum(w[r, i] * x[1, i] for i in range(12)) for r in range(5)],
                               rtol=1e-13)


# ----------------------------------------------------------------------------------------
# bf16 decoding: hand-written bit patterns, the IEEE field formula, and torch's own cast
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("bits,value", [
    (0x3F80, 1.0), (0xBF80, -1.0), (0x4000, 2.0), (0xC000, -2.0), (0x4049, 3.140625),
    (0x3F00, 0.5), (0x0000, 0.0), (0x0080, 2.0 ** -126), (0x0001, 2.0 ** -133),
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127), (0x7F80, math.inf), (0xFF80, -math.inf),
])
def test_bf16_to_f64_hand_patterns(bits, value):
    got = O.bf16_to_f64(np.array([bits], dtype=np.uint16))[0]
    assert got == value and math.copysign(1.0, got) == math.copysign(1.0, value)


def test_bf16_to_f64_signed_zero_and_nan():
    z = O.bf16_to_f64(np.array([0x8000], dtype=np.uint16))[0]
    assert z == 0.0 and math.copysign(1.0, z) == -1.0
    assert np.isnan(O.bf16_to_f64(np.array([0x7FC0, 0xFFC1, 0x7F81], dtype=np.uint16))).all()


def _bf16_fields(bits: int) -> float:
    """bf16 value from its fields: sign 1 bit, exponent 8 bits (bias 127), fraction 7 bits."""
    s, e, m = bits >> 15, (bits >> 7) & 0xFF, bits & 0x7F
    if e == 0xFF:
        return math.nan if m else (-math.inf if s else math.inf)
    mag = math.ldexp(m, -126 - 7) if e == 0 else math.ldexp(128 + m, e - 127 - 7)
    return -mag if s else mag


def test_bf16_to_f64_matches_field_formula_on_every_pattern():
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = O.bf16_to_f64(allbits)
    want = np.array([_bf16_fields(int(b)) for b in allbits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(want[~nan]))


def test_bf16_to_f64_matches_torch_cast():
    torch = pytest.importorskip("torch")
    bits = np.random.default_rng(7).integers(0, 1 << 16, size=10000).astype(np.uint16)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_to_f64(bits)
    nan = np.isnan(t)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], t[~nan])


# ----------------------------------------------------------------------------------------
# 4-bit affine kv_b: hand-worked blocks (code order within a word, group boundaries)
# ----------------------------------------------------------------------------------------

def _q4_blob(case):
    words = np.array([int(w, 16) for w in case["words_row_major"]], dtype="<u4")
    sc = np.array([int(v, 16) for v in case["scales_bf16"]], dtype="<u2")
    bi = np.array([int(v, 16) for v in case["biases_bf16"]], dtype="<u2")
    return np.concatenate([words.view(np.uint8), sc.view(np.uint8), bi.view(np.uint8)])


def test_q4_affine_golden_blocks(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "q4_affine_blocks.json")))
    for case in g["cases"]:
        blob = _q4_blob(case)
        assert blob.size == O.q4_affine_bytes(case["rows"], case["cols"])
        w = O.q4_affine_to_f64(blob, case["rows"], case["cols"])
        for r, c, v in case["expect"]:
            assert w[r, c] == v, (r, c, w[r, c], v)


def test_q4_affine_code_order_within_a_word():
    # one word 0x87654321 in a 1 x 64 matrix with scale 1, bias 0: columns 0..7 hold 1..8
    words = np.zeros(8, dtype="<u4")
    words[0] = 0x87654321
    blob = np.concatenate([words.view(np.uint8), np.array([0x3F80], "<u2").view(np.uint8),
                           np.array([0x0000], "<u2").view(np.uint8)])
    w = O.q4_affine_to_f64(blob, 1, 64)
    assert list(w[0, :8]) == [1, 2, 3, 4, 5, 6, 7, 8] and not w[0, 8:].any()


# ----------------------------------------------------------------------------------------
# The layer's projections: matvec, the Q chain, the direct q projection, o_proj
# ----------------------------------------------------------------------------------------

def test_matvec_rank_one_closed_form():
    # W = u v^T maps x to u (v . x); a transposed W (or x on the wrong side) would give
    # v (u . x), a vector of another length
    u, v = RNG.standard_normal(7), RNG.standard_normal(11)
    x = RNG.standard_normal((3, 11))
    got = O.matvec(np.outer(u, v), x)
    assert got.shape == (3, 7)
    for b in range(3):
        np.testing.assert_allclose(got[b], u * float(np.dot(v, x[b])), rtol=1e-13, atol=1e-14)


def test_matvec_one_hot_input_picks_a_column():
    W = RNG.standard_normal((6, 9))
    for k in (0, 4, 8):
        e = np.zeros((1, 9))
        e[0, k] = 1.0
        np.testing.assert_array_equal(O.matvec(W, e)[0], W[:, k])


def test_heads_view_puts_each_head_in_one_run_nope_first():
    H, N, R = 3, 4, 2
    q = O.heads_view(np.arange(H * (N + R), dtype=np.float64)[None], H, N + R)[0]
    for h in range(H):
        np.testing.assert_array_equal(q[h, :N], np.arange(h * (N + R), h * (N + R) + N))
        np.testing.assert_array_equal(q[h, N:], np.arange(h * (N + R) + N, (h + 1) * (N + R)))


def test_q_direct_with_a_permutation_moves_input_values():
    # W_q = a permutation matrix P (row i has its 1 in column p[i]): q_full[i] = x[p[i]]
    H, qk, D = 2, 5, 10
    p = RNG.permutation(D)
    W = np.zeros((H * qk, D))
    W[np.arange(H * qk), p] = 1.0
    x = RNG.standard_normal((1, D))
    q = O.q_direct(x, W, H, qk)
    for h in range(H):
        for j in range(qk):
            assert q[0, h, j] == x[0, p[h * qk + j]]


def test_q_chain_normalises_between_the_two_projections():
    # identity q_a and rank-one q_b = u v^T: q_full = u * sum_k v_k w_k x_k / rms(x), which a
    # norm after q_b, a missing norm weight or a norm before q_a would all change
    D, H, qk = 16, 2, 3
    u, v = RNG.standard_normal(H * qk), RNG.standard_normal(D)
    w = RNG.uniform(0.5, 1.5, D)
    x = RNG.standard_normal((2, D)) * 3
    eps = 1e-6
    q = O.q_chain(x, np.eye(D), w, eps, np.outer(u, v), H, qk)
    for b in range(2):
        rms = math.sqrt(sum(t * t for t in x[b]) / D + eps)
        s = sum(v[k] * w[k] * x[b, k] for k in range(D)) / rms
        np.testing.assert_allclose(q[b].reshape(-1), u * s, rtol=1e-12)


def test_q_chain_is_invariant_to_input_scale():
    # the RMSNorm in the middle removes any positive scale of x (eps = 0), but not the sign
    D, L, H, qk = 24, 8, 2, 5
    Wa, Wb = RNG.standard_normal((L, D)), RNG.standard_normal((H * qk, L))
    w = RNG.uniform(0.5, 1.5, L)
    x = RNG.standard_normal((3, D))
    base = O.q_chain(x, Wa, w, 0.0, Wb, H, qk)
    np.testing.assert_allclose(O.q_chain(37.0 * x, Wa, w, 0.0, Wb, H, qk), base, rtol=1e-12)
    np.testing.assert_allclose(O.q_chain(-x, Wa, w, 0.0, Wb, H, qk), -base, rtol=1e-12)
    # and each sequence's q_lat has unit rms before the norm weight: with w = 1 and q_b = I
    q = O.q_chain(x, Wa, np.ones(L), 0.0, np.eye(L), 1, L)
    np.testing.assert_allclose(np.sqrt(np.mean(q[:, 0, :] ** 2, axis=1)), 1.0, rtol=1e-13)


def test_o_proj_reads_heads_in_order():
    # a one-hot input at (head h, value j) picks column h*V + j of W_o
    H, V, D = 3, 4, 5
    W = RNG.standard_normal((D, H * V))
    for h, j in ((0, 0), (1, 3), (2, 1)):
        a = np.zeros((1, H, V))
        a[0, h, j] = 1.0
        np.testing.assert_array_equal(O.o_proj(a, W)[0], W[:, h * V + j])


def test_o_proj_is_the_sum_of_per_head_blocks():
    H, V, D = 4, 3, 6
    W = RNG.standard_normal((D, H * V))
    a = RNG.standard_normal((2, H, V))
    want = sum(np.einsum("dv,bv->bd", W[:, h * V:(h + 1) * V], a[:, h, :]) for h in range(H))
    np.testing.assert_allclose(O.o_proj(a, W), want, rtol=1e-12, atol=1e-13)


def test_absorbed_layer_equals_mha_on_projected_inputs():
    # the whole layer on tiny shapes: x -> q (direct) -> absorbed decode over rows appended from
    # kv_a projections -> o_proj, against plain MHA built from the same projections
    H, C, N, R, V, D, L = 2, 8, 4, 4, 3, 16, 5
    Wq, Wkva = RNG.standard_normal((H * (N + R), D)), RNG.standard_normal((C + R, D))
    kv_b, Wo = RNG.standard_normal((H * (N + V), C)), RNG.standard_normal((D, H * V))
    xs = RNG.standard_normal((L, D))
    nw = RNG.uniform(0.5, 1.5, C)
    inv = O.yarn_inv_freq(R, 10000.0, 1.0, 4096, 32.0, 1.0)
    rows = O.append_rows(O.kv_a_rows(xs, Wkva), nw, list(range(L)), inv, C, 1e-6)
    q = O.q_direct(xs[-1:], Wq, H, N + R)
    W_UK, W_UV = O.split_kv_b(kv_b, H, N, V)
    out, _ = O.decode_one(q[0], W_UK, W_UV, rows, L - 1, inv, 0.3, C)
    ref, _ = O.decode_unabsorbed_one(q[0], W_UK, W_UV, rows, L - 1, inv, 0.3, C)
    np.testing.assert_allclose(O.o_proj(out[None], Wo), O.o_proj(ref[None], Wo), rtol=1e-11, atol=1e-12)


# ----------------------------------------------------------------------------------------
# Several query tokens per sequence
# ----------------------------------------------------------------------------------------

def _tiny_heads(H=3, C=8, N=4, R=4, V=5):
    kv_b = RNG.standard_normal((H * (N + V), C))
    W_UK, W_UV = O.split_kv_b(kv_b, H, N, V)
    return W_UK, W_UV


def test_multi_query_single_token_is_the_plain_decode():
    W_UK, W_UV = _tiny_heads()
    rows = RNG.standard_normal((7, 12))
    q = RNG.standard_normal((1, 3, 8))
    inv = O.yarn_inv_freq(4, 10000.0, 1.0, 4096, 32.0, 1.0)
    out, lse = O.decode_multi_one(q, W_UK, W_UV, rows, 6, inv, 0.4, 8)
    o1, l1 = O.decode_one(q[0], W_UK, W_UV, rows, 6, inv, 0.4, 8)
    np.testing.assert_array_equal(out[0], o1)
    np.testing.assert_array_equal(lse[0], l1)


def test_multi_query_is_causal():
    # token i must not see rows past L - T + i: changing them leaves token i alone and moves
    # the last token
    W_UK, W_UV = _tiny_heads()
    L, T = 9, 3
    rows = RNG.standard_normal((L, 12))
    q = RNG.standard_normal((T, 3, 8))
    inv = O.yarn_inv_freq(4, 10000.0, 1.0, 4096, 32.0, 1.0)
    out, lse = O.decode_multi_one(q, W_UK, W_UV, rows, L - T, inv, 0.4, 8)
    moved = rows.copy()
    moved[L - 1] += 5.0
    out2, lse2 = O.decode_multi_one(q, W_UK, W_UV, moved, L - T, inv, 0.4, 8)
    np.testing.assert_array_equal(out2[:T - 1], out[:T - 1])
    assert np.all(np.abs(lse2[T - 1] - lse[T - 1]) > 1e-6)


def test_multi_query_identical_rows_count_each_tokens_prefix():
    # all rows equal: token i averages to W_UV lat and its lse is s + ln(L - T + 1 + i)
    W_UK, W_UV = _tiny_heads()
    L, T = 10, 4
    row = RNG.standard_normal(12)
    rows = np.tile(row, (L, 1))
    q = RNG.standard_normal((T, 3, 8))
    q[:, :, 4:] = 0.0    # no rope part: the score does not depend on the position
    out, lse = O.decode_multi_one(q, W_UK, W_UV, rows, None, np.zeros(2), 0.4, 8)
    for i in range(T):
        for h in range(3):
            s = 0.4 * float(np.dot(np.einsum("n,nc->c", q[i, h, :4], W_UK[h]), row[:8]))
            assert abs(lse[i, h] - (s + math.log(L - T + 1 + i))) < 1e-12
            np.testing.assert_allclose(out[i, h], W_UV[h] @ row[:8], rtol=1e-12, atol=1e-12)


def test_multi_query_tokens_sit_at_consecutive_positions():
    # one rope pair (R = 2, frequency w), no latent: token i at position p0 + i scores row t,
    # whose pe is k rotated by t*w, as scale |q||k| cos((t - p0 - i) w + phi), phi the angle from
    # q to k; written out with numpy's cos, apart from the oracle's rotation
    H, C, N, R, V = 1, 4, 2, 2, 3
    kv_b = RNG.standard_normal((H * (N + V), C))
    W_UK, W_UV = O.split_kv_b(kv_b, H, N, V)
    w, scale, L, T, p0 = 0.37, 0.8, 11, 3, 8
    qp, k = np.array([0.6, -1.1]), np.array([1.3, 0.4])
    rows = np.zeros((L, C + R))
    for t in range(L):
        c, s_ = math.cos(t * w), math.sin(t * w)
        rows[t, C:] = [k[0] * c - k[1] * s_, k[0] * s_ + k[1] * c]
    q = np.zeros((T, H, N + R))
    q[:, 0, N:] = qp
    _, lse = O.decode_multi_one(q, W_UK, W_UV, rows, p0, np.array([w]), scale, C)
    phi = math.atan2(k[1], k[0]) - math.atan2(qp[1], qp[0])
    mag = math.hypot(*qp) * math.hypot(*k)
    for i in range(T):
        sc = [scale * mag * math.cos((t - p0 - i) * w + phi) for t in range(L - T + 1 + i)]
        assert abs(lse[i, 0] - math.log(sum(math.exp(x) for x in sc))) < 1e-12
