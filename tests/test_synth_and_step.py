"""Host-side checks of the seeded generator and the oracle's whole-step driver."""
import numpy as np
import pytest

from mla_latent_cache_absorb_gb300 import synth
from oracle import mla_oracle as O
from oracle import step as OS


def small(name, **kw):
    return synth.WORKLOADS[name].with_(**kw)


def test_generator_is_deterministic():
    wl = small("ragged_paged_b64", B=3, H=4, context=("uniform", 5, 200))
    a = synth.make_problem(wl)
    b = synth.make_problem(wl)
    for f in ("q", "pool", "page_table", "positions", "seq_lens", "norm_w", "kv_b", "kva_rows"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))


def test_paged_layout_is_a_permutation_with_sentinels():
    wl = small("ragged_paged_b64", B=5, H=2, context=("uniform", 1, 300))
    p = synth.make_problem(wl)
    used = p.page_table[p.page_table >= 0]
    assert sorted(used.tolist()) == list(range(p.n_phys_rows // 64))
    for b in range(wl.B):
        L = int(p.seq_lens[b])
        P = int(p.positions[b])
        assert P == L - 1
        rows = O.physical_row(b, np.arange(L), p.page_table, 64, 0)
        vals = p.pool[rows]
        # pre-filled rows are finite, the append slot holds the NaN sentinel
        assert np.all(vals[:P] != synth.BF16_NAN_BITS)
        assert np.all(vals[P] == synth.BF16_NAN_BITS)


def test_q8_0_kv_b_shape_and_validation():
    wl = small("long_q8_b4_t131072", B=1, H=4, context=("fixed", 10), hidden=64)
    kv_b = synth.make_kv_b(wl)
    rows = wl.H * (wl.N + wl.V)
    assert kv_b.shape == (rows, wl.C // 32 * 34)
    assert O.q8_0_validate("q8_0", (rows, wl.C), kv_b.size, wl.H, wl.N, wl.C, wl.V) is None
    w = O.q8_0_to_f64(kv_b, wl.C)
    # codes within +-127, scales within [1e-3, 2e-3] (fp16-rounded)
    d = np.abs(w).max()
    assert 0 < d <= 127 * 2.0e-3 * 1.001


@pytest.mark.parametrize("name", ["tiny_f32", "v2lite_b1_t4096"])
def test_step_absorbed_matches_unabsorbed(name):
    wl = synth.WORKLOADS[name]
    if name != "tiny_f32":
        wl = wl.with_(context=("fixed", 200))
    p = synth.make_problem(wl)
    new, out, lse = OS.run_step(p)
    inv, scale = OS.tables(wl)
    q = OS.decode_act(p.q, wl.act)
    rows = [OS.sequence_rows(p, b, new[b]) for b in range(wl.B)]
    out2, lse2 = O.decode_step(q, OS.kv_b_f64(p), rows, p.positions, inv, scale, wl.H, wl.N,
                               wl.V, wl.C, unabsorbed=True)
    np.testing.assert_allclose(out, out2, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse, lse2, rtol=0, atol=1e-10)
    assert np.all(np.isfinite(out))


def test_gemv_append_rows_are_finished_rows():
    wl = small("long_q8_b4_t131072", B=2, H=2, context=("fixed", 33), hidden=256)
    p = synth.make_problem(wl)
    rows = OS.appended_rows(p)
    inv, _ = OS.tables(wl)
    kva = O.bf16_to_f64(p.x) @ O.bf16_to_f64(p.w_kva).T
    w = p.norm_w.astype(np.float64)
    np.testing.assert_allclose(np.sqrt(np.mean((rows[:, :wl.C] / w) ** 2, axis=1)),
                               1.0 / np.sqrt(1 + wl.rms_eps / np.mean(kva[:, :wl.C] ** 2, axis=1)),
                               rtol=1e-12)
    np.testing.assert_allclose(np.hypot(rows[:, wl.C::2], rows[:, wl.C + 1::2]),
                               np.hypot(kva[:, wl.C::2], kva[:, wl.C + 1::2]), rtol=1e-12)
