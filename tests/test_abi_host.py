"""The C-ABI library on the host (no GPU): it loads, exports every symbol include/mla.h declares,
and its host-side helpers and validation follow the pages' definitions and fixture."""
import json
import os
import re

import numpy as np
import pytest

from oracle import mla_oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    lib = os.path.join(ROOT, "mla_latent_cache_absorb_gb300", "libmla.so")
    if not os.path.exists(lib):
        from mla_latent_cache_absorb_gb300 import build
        build.build()
    from mla_latent_cache_absorb_gb300 import binding
    return binding


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_symbol(L):
    import ctypes
    syms = declared_symbols()
    assert len(syms) >= 16
    lib = ctypes.CDLL(L.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), f"{s} declared in mla.h but not exported"
    assert set(syms) == set(L.EXPORTED), "binding and header disagree"


def test_status_strings_and_version(L):
    for code in L.STATUS:
        assert L.mla_status_string(code)
    assert L.mla_abi_version() == 1


@pytest.mark.parametrize("args", [
    (64, 10000.0, 1.0, 4096, 32.0, 1.0),
    (64, 10000.0, 40.0, 4096, 32.0, 1.0),
    (16, 10000.0, 1.0, 4096, 32.0, 1.0),
    (128, 50000.0, 8.0, 8192, 32.0, 1.0),
])
def test_yarn_table_matches_oracle(L, args):
    out = np.zeros(args[0] // 2)
    assert L.mla_yarn_inv_freq(*args, out) == 0
    np.testing.assert_allclose(out, O.yarn_inv_freq(*args), rtol=1e-14)


def test_yarn_table_rejects_bad_args(L):
    out = np.zeros(8)
    assert L.mla_yarn_inv_freq(15, 1e4, 1.0, 4096, 32.0, 1.0, out) == L.STATUS_CODE["MLA_ERR_INVALID_ARG"]
    assert L.mla_yarn_inv_freq(16, 1e4, 1.0, 4096, 32.0, 1.0, None) == L.STATUS_CODE["MLA_ERR_INVALID_ARG"]


def test_scales_match_golden(L, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "yarn_rope64_theta1e4_factor40.json")))
    assert abs(L.mla_yarn_mscale(40.0, 1.0) - g["mscale"]) < 1e-15
    assert L.mla_yarn_mscale(1.0, 1.0) == 1.0
    assert abs(L.mla_softmax_scale(128, 64, g["mscale"]) - g["softmax_scale_nope128_rope64"]) < 1e-8
    assert abs(L.mla_softmax_scale(32, 16, 1.0) - g["softmax_scale_plain_nope32_rope16"]) < 1e-8


def test_kv_b_validation_fixture(L, golden_dir):
    g = json.load(open(os.path.join(golden_dir, "q8_0_kv_b_validation.json")))
    H, N, C, V = g["heads"], g["nope"], g["kv_lora"], g["v_dim"]
    dt = {"q8_0": L.MLA_Q8_0, "dtype12": 12}
    ok = g["valid"]
    assert L.mla_validate_kv_b(dt[ok["dtype"]], *ok["shape"], ok["size_bytes"], H, N, C, V) == 0
    for r in g["rejects"]:
        assert L.mla_validate_kv_b(dt[r["dtype"]], *r["shape"], r["size_bytes"], H, N, C, V) != 0, r["why"]
    # width that does not tile 32-element blocks
    assert L.mla_validate_kv_b(L.MLA_Q8_0, 12, 48, 12 * 2 * 34, H, N, 48, V) != 0
    # other dtypes: plain element sizes
    assert L.mla_validate_kv_b(L.MLA_BF16, 12, 64, 12 * 64 * 2, H, N, C, V) == 0
    assert L.mla_validate_kv_b(L.MLA_F32, 12, 64, 12 * 64 * 4, H, N, C, V) == 0
    assert L.mla_validate_kv_b(L.MLA_F32, 12, 64, 12 * 64 * 2, H, N, C, V) != 0
    # overflow of heads * (nope + v) is rejected, not wrapped
    assert L.mla_validate_kv_b(L.MLA_BF16, 1, 64, 128, 2 ** 31 - 1, 2 ** 31 - 1, 64, 2) != 0


def _cfg(L, **kw):
    c = L.MlaConfig()
    c.n_heads, c.kv_lora, c.qk_nope, c.qk_rope, c.v_head = 16, 512, 128, 64, 128
    c.act_dtype, c.kv_b_dtype = L.MLA_BF16, L.MLA_BF16
    c.softmax_scale, c.rms_eps = 0.07, 1e-6
    c.page_size, c.max_pages_per_seq, c.rows_per_seq = 0, 0, 4096
    c.rope_inv_freq = 0x1000
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_kv_b_bytes(L):
    assert L.mla_kv_b_bytes(_cfg(L)) == 16 * 256 * 512 * 2
    assert L.mla_kv_b_bytes(_cfg(L, kv_b_dtype=L.MLA_Q8_0, n_heads=128)) == 128 * 256 * 16 * 34
    assert L.mla_kv_b_bytes(_cfg(L, kv_b_dtype=L.MLA_F32)) == 16 * 256 * 512 * 4


@pytest.mark.parametrize("bad", [
    dict(n_heads=0), dict(qk_rope=63), dict(qk_rope=0), dict(act_dtype=7), dict(kv_b_dtype=9),
    dict(rows_per_seq=0), dict(page_size=-1), dict(page_size=64, max_pages_per_seq=0),
    dict(softmax_scale=0.0), dict(softmax_scale=float("nan")),
])
def test_config_validation_before_any_device_call(L, bad):
    st, _ = L.mla_append_workspace_size(_cfg(L, **bad), 4)
    assert st == L.STATUS_CODE["MLA_ERR_INVALID_ARG"]


def test_q8_0_needs_tiling_width(L):
    st, _ = L.mla_append_workspace_size(_cfg(L, kv_b_dtype=L.MLA_Q8_0, kv_lora=48), 1)
    assert st == L.STATUS_CODE["MLA_ERR_BAD_KV_B"]


def test_append_workspace_size_and_null_args(L):
    # every call below must fail host validation: none of them may reach a kernel launch
    st, n = L.mla_append_workspace_size(_cfg(L), 4)
    assert st == 0 and n >= 256 + 4 * 576 * 4 and n % 256 == 0
    cache = L.MlaCache()
    cache.rows, cache.page_table, cache.n_physical_rows = 0x10000, None, 4 * 4096
    # null kv_in / norm_w / positions and B < 1 are rejected on the host
    args = dict(kv_in=0x2000, w_kva=None, hidden=0, norm_w=0x3000, positions=0x4000, seq_lens=None,
                B=4, workspace=0x5000, ws_bytes=n)
    for k in ("kv_in", "norm_w", "positions"):
        a = dict(args, **{k: None})
        assert L.mla_cache_append(_cfg(L), cache, *a.values()) == L.STATUS_CODE["MLA_ERR_INVALID_ARG"]
    assert L.mla_cache_append(_cfg(L), cache, *dict(args, B=0).values()) == L.STATUS_CODE["MLA_ERR_INVALID_ARG"]
    # the cache must hold B * rows_per_seq rows when contiguous
    small = L.MlaCache()
    small.rows, small.page_table, small.n_physical_rows = 0x10000, None, 4095
    assert L.mla_cache_append(_cfg(L), small, *args.values()) == L.STATUS_CODE["MLA_ERR_INVALID_ARG"]
    # workspace: too small or misaligned
    assert L.mla_cache_append(_cfg(L), cache, *dict(args, ws_bytes=n - 1).values()) == L.STATUS_CODE["MLA_ERR_WORKSPACE"]
    assert L.mla_cache_append(_cfg(L), cache, *dict(args, workspace=0x5010).values()) == L.STATUS_CODE["MLA_ERR_WORKSPACE"]
    # paged cache without a page table
    assert L.mla_cache_append(_cfg(L, page_size=64, max_pages_per_seq=64), cache, *args.values()) == \
        L.STATUS_CODE["MLA_ERR_INVALID_ARG"]
    # gemv append: hidden must keep 16-byte vectors
    assert L.mla_cache_append(_cfg(L), cache, *dict(args, w_kva=0x6000, hidden=7167).values()) == \
        L.STATUS_CODE["MLA_ERR_INVALID_ARG"]


def test_q4_affine_kv_b_contract(L):
    heads, nope, kv_lora, v = 4, 2, 128, 3
    rows = heads * (nope + v)
    size = rows * (kv_lora // 2) + rows * (kv_lora // 64) * 4
    assert size == O.q4_affine_bytes(rows, kv_lora)
    assert L.mla_validate_kv_b(L.MLA_Q4_AFFINE, rows, kv_lora, size, heads, nope, kv_lora, v) == 0
    bad = L.STATUS_CODE["MLA_ERR_BAD_KV_B"]
    assert L.mla_validate_kv_b(L.MLA_Q4_AFFINE, rows, kv_lora, size - 1, heads, nope, kv_lora, v) == bad
    assert L.mla_validate_kv_b(L.MLA_Q4_AFFINE, rows, 96, rows * 48 + rows * 4, heads, nope, 96, v) == bad
    cfg = L.MlaConfig()
    cfg.n_heads, cfg.kv_lora, cfg.qk_nope, cfg.qk_rope, cfg.v_head = heads, kv_lora, nope, 2, v
    cfg.act_dtype, cfg.kv_b_dtype = L.MLA_BF16, L.MLA_Q4_AFFINE
    assert L.mla_kv_b_bytes(cfg) == size
    cfg.kv_lora = 96
    assert L.mla_kv_b_bytes(cfg) == 0


def _proj(L, **kw):
    pj = L.MlaProj()
    pj.hidden, pj.q_lora, pj.w_dtype, pj.q_norm_eps = 7168, 1536, L.MLA_BF16, 1e-6
    pj.w_q_a, pj.q_a_norm_w, pj.w_q, pj.w_kva, pj.w_o = 0x10000, 0x20000, 0x30000, 0x40000, 0x50000
    for k, v in kw.items():
        setattr(pj, k, v)
    return pj


def test_projection_workspace_sizes(L):
    # a 256-byte error-word header, then (Q chain) the float32 q_lat rows, then the tensor-core
    # path's bf16 halves and split partials; sizes are whole 256-byte blocks
    st, n = L.mla_front_end_workspace_size(_cfg(L), _proj(L), 64)
    assert st == 0 and n >= 256 + 64 * 1536 * 4 + 2 * 64 * 1536 * 2 and n % 256 == 0
    # 4 sequences, 16 heads: every matrix under 64 MiB, CUDA cores: q_lat only
    st, small = L.mla_front_end_workspace_size(_cfg(L), _proj(L), 4)
    assert st == 0 and small == 256 + 4 * 1536 * 4
    st, n = L.mla_front_end_workspace_size(_cfg(L), _proj(L, q_lora=0), 4)
    assert st == 0 and n == 256
    st, n = L.mla_o_proj_workspace_size(_cfg(L), _proj(L), 4)
    assert st == 0 and n == 256
    # 4 sequences, 128 heads: q_b (75 MB) and W_o (235 MB) on the tensor cores, q_a + kv_a
    # (30 MB) on the CUDA cores: q_lat and the halves of the normalised q_lat / of attn
    st, n = L.mla_front_end_workspace_size(_cfg(L, n_heads=128), _proj(L), 4)
    assert st == 0 and n >= 256 + 4 * 1536 * 4 + 2 * 4 * 1536 * 2 and n % 256 == 0
    st, n = L.mla_o_proj_workspace_size(_cfg(L, n_heads=128), _proj(L), 4)
    assert st == 0 and n >= 256 + 2 * 4 * 128 * 128 * 2 and n % 256 == 0
    st, n = L.mla_o_proj_workspace_size(_cfg(L), _proj(L), 64)
    assert st == 0 and n >= 256 + 2 * 64 * 16 * 128 * 2 and n % 256 == 0
    st, n = L.mla_o_proj_workspace_size(_cfg(L), _proj(L, w_dtype=L.MLA_Q8_0), 64)   # CUDA cores
    assert st == 0 and n == 256


def test_projection_launch_counts(L):
    # 16 heads, 4 sequences: one GEMV each (q_a + kv_a, q_b, o_proj) and the norm
    assert L.mla_proj_launches(_cfg(L), _proj(L), 4) == (0, 3, 1)
    assert L.mla_proj_launches(_cfg(L), _proj(L, q_lora=0), 4) == (0, 1, 1)
    assert L.mla_proj_launches(_cfg(L), _proj(L, w_dtype=L.MLA_Q8_0), 64) == (0, 3, 1)
    # tensor cores: o_proj adds the halves of attn, and a slice reduction when the columns split
    st, fe, op = L.mla_proj_launches(_cfg(L, n_heads=128), _proj(L), 64)
    assert st == 0 and 3 <= fe <= 5 and op in (2, 3)
    st, _, _ = L.mla_proj_launches(_cfg(L), _proj(L, w_dtype=9), 4)
    assert st == L.STATUS_CODE["MLA_ERR_UNSUPPORTED"]


@pytest.mark.parametrize("bad,status", [
    (dict(hidden=7164), "MLA_ERR_INVALID_ARG"),                        # not a multiple of 8
    (dict(hidden=0), "MLA_ERR_INVALID_ARG"),
    (dict(q_lora=-1), "MLA_ERR_INVALID_ARG"),
    (dict(q_lora=1540), "MLA_ERR_INVALID_ARG"),
    (dict(w_dtype=2, hidden=7168 + 16), "MLA_ERR_INVALID_ARG"),  # Q8_0 blocks need % 32
    (dict(w_dtype=3, q_lora=1536 + 32), "MLA_ERR_INVALID_ARG"),        # 4-bit groups need % 64
    (dict(w_dtype=9), "MLA_ERR_UNSUPPORTED"),
])
def test_projection_contract_rejected_on_the_host(L, bad, status):
    st, _ = L.mla_front_end_workspace_size(_cfg(L), _proj(L, **bad), 4)
    assert st == L.STATUS_CODE[status]


def test_front_end_and_o_proj_null_and_misaligned_args(L):
    # every call below must fail host validation: none of them may reach a kernel launch
    cfg, pj = _cfg(L), _proj(L)
    INVALID = L.STATUS_CODE["MLA_ERR_INVALID_ARG"]
    ws, n = 0x70000, 4 * 1536 * 4
    assert L.mla_front_end(cfg, pj, None, 0x60000, 0x61000, 4, ws, n) == INVALID
    assert L.mla_front_end(cfg, pj, 0x60008, 0x60000, 0x61000, 4, ws, n) == INVALID
    assert L.mla_front_end(cfg, pj, 0x60000, None, 0x61000, 4, ws, n) == INVALID
    assert L.mla_front_end(cfg, _proj(L, w_kva=None), 0x60000, 0x61000, 0x62000, 4, ws, n) == INVALID
    assert L.mla_front_end(cfg, _proj(L, q_a_norm_w=None), 0x60000, 0x61000, None, 4, ws, n) == INVALID
    assert L.mla_front_end(cfg, pj, 0x60000, 0x61000, None, 0, ws, n) == INVALID
    assert L.mla_front_end(cfg, pj, 0x60000, 0x61000, None, 4, ws, n - 1) == L.STATUS_CODE["MLA_ERR_WORKSPACE"]
    assert L.mla_o_proj(cfg, _proj(L, w_o=None), 0x60000, 0x61000, 4, ws, n) == INVALID
    assert L.mla_o_proj(cfg, pj, 0x60004, 0x61000, 4, ws, n) == INVALID
    assert L.mla_o_proj(cfg, pj, 0x60000, 0x61000, 4, None, 0) == L.STATUS_CODE["MLA_ERR_WORKSPACE"]
    # o_proj's in_dim is H*V: 3 heads of 8 values (24) is no multiple of the 4-bit group of 64
    odd = _cfg(L)
    odd.n_heads, odd.v_head = 3, 8
    assert L.mla_o_proj(odd, _proj(L, w_dtype=3), 0x60000, 0x61000, 4, ws, n) == INVALID
