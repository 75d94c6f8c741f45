"""The layer's projections on the GPU against the fp64 oracle: the front end (Q chain or direct
q projection, with kv_a from the same input) and o_proj, in every weight format, at batch sizes
below, at and above one pass of 8 sequences; plus run-to-run determinism and a whole layer
(front end -> append -> decode -> o_proj) against the oracle's layer."""
import numpy as np
import pytest

from mla_latent_cache_absorb_gb300 import synth
from oracle import step as OS
from tests.gpu_util import max_rel, need_gpu

gpu = pytest.mark.gpu
PW = synth.PROJ_WORKLOADS

# float32 outputs (kva, o_proj): float32 sums of bf16 products, a few thousand terms
F32_TOL = 1e-4
# bf16 q: one rounding of a float32 result, so within one bf16 step of the exact value
Q_ELEM_REL = 2.0 ** -8

CASES = [
    ("tiny_f32", PW["tiny_proj_f32"]),
    ("v2lite_b1", PW["v2lite_proj_b1"]),
    ("v2lite_b9_q8", PW["v2lite_proj_b1"].with_(B=9, w="q8_0")),
    ("v2lite_b5_q4", PW["v2lite_proj_b1"].with_(B=5, w="q4_affine")),
    ("v3_b4", PW["v3_proj_b4"]),
    ("v3_b2_q8", PW["v3_proj_b4"].with_(B=2, w="q8_0")),
    ("v3_b3_q4", PW["v3_proj_b4"].with_(B=3, w="q4_affine")),
    # in_dim not a multiple of 256: the quantised GEMV without the ring (hidden 2112)
    ("v2lite_b3_q8_k2112", PW["v2lite_proj_b1"].with_(B=3, w="q8_0", hidden=2112)),
    ("v2lite_b3_q4_k2112", PW["v2lite_proj_b1"].with_(B=3, w="q4_affine", hidden=2112)),
    ("v3_b17_direct", PW["v3_proj_b4"].with_(B=17, q_lora=0)),
    # tensor-core path (bf16 weights, 16 or more sequences, or a matrix of 64 MiB or more, as
    # q_b and W_o in v3_b4 above): the smallest batch, the headline batch, the largest
    # float32-input batch, one past it (o_proj back on CUDA cores), a direct q projection with kv_a
    ("tc_v3_b16", PW["v3_proj_b4"].with_(B=16)),
    ("tc_v3_b64", PW["v3_proj_b64"]),
    ("tc_v3_b128", PW["v3_proj_b4"].with_(B=128)),
    ("tc_v3_b129", PW["v3_proj_b4"].with_(B=129)),
    ("tc_v2lite_b32_direct", PW["v2lite_proj_b1"].with_(B=32)),
]


def _check_q(got_bits, want, act, tag):
    got = OS.decode_act(got_bits, act)
    assert np.all(np.isfinite(got)), f"{tag}: non-finite q"
    r = max_rel(got, want)
    assert r <= 1e-2, f"{tag}: q max-rel {r}"
    if act == "bf16":
        scale = np.max(np.abs(want))
        ok = np.abs(got - want) <= Q_ELEM_REL * np.abs(want) + 1e-4 * scale
        assert ok.all(), f"{tag}: q elements off by more than a bf16 step at {np.argwhere(~ok)[:5]}"
    else:
        assert r <= F32_TOL, f"{tag}: q max-rel {r}"


@gpu
@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_front_end_and_o_proj_parity(name, wl):
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceProj
    pp = synth.make_proj_problem(wl)
    dp = DeviceProj(pp)
    L.check(dp.front_end(), "mla_front_end")
    L.check(dp.o_proj(), "mla_o_proj")
    torch.cuda.synchronize()
    q_want, kva_want = OS.front_end(pp)
    _check_q(dp.q_host(), q_want, wl.act, name)
    r = max_rel(dp.kva.cpu().numpy(), kva_want)
    assert r <= F32_TOL, f"{name}: kva max-rel {r}"
    r = max_rel(dp.y.cpu().numpy(), OS.o_proj(pp))
    assert r <= F32_TOL, f"{name}: o_proj max-rel {r}"


@gpu
def test_front_end_without_kva_and_repeatability():
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceProj
    pp = synth.make_proj_problem(PW["v3_proj_b4"].with_(B=11))
    with_kva, no_kva = DeviceProj(pp), DeviceProj(pp, with_kva=False)
    L.check(with_kva.front_end(), "front end")
    L.check(no_kva.front_end(), "front end without kv_a")
    q1 = with_kva.q.clone()
    L.check(with_kva.front_end(), "front end again")
    L.check(with_kva.o_proj(), "o_proj")
    y1 = with_kva.y.clone()
    L.check(with_kva.o_proj(), "o_proj again")
    torch.cuda.synchronize()
    assert torch.equal(q1, with_kva.q), "front end not run-to-run identical"
    assert torch.equal(q1, no_kva.q), "q depends on whether kv_a is computed"
    assert torch.equal(y1, with_kva.y), "o_proj not run-to-run identical"


@gpu
def test_tensor_core_path_is_repeatable():
    """The split-K partial sums are added in a fixed order: two runs are bit-identical."""
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceProj
    dp = DeviceProj(synth.make_proj_problem(PW["v3_proj_b64"].with_(B=48)))
    outs = []
    for _ in range(2):
        L.check(dp.front_end(), "front end")
        L.check(dp.o_proj(), "o_proj")
        torch.cuda.synchronize()
        outs.append((dp.q.clone(), dp.kva.clone(), dp.y.clone()))
    for u, v in zip(*outs):
        assert torch.equal(u, v)
    st, _ = L.mla_get_device_error(dp.ws)
    assert st == 0


@gpu
def test_front_end_argument_errors():
    need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceProj
    dp = DeviceProj(synth.make_proj_problem(PW["tiny_proj_f32"]))
    INVALID = L.STATUS_CODE["MLA_ERR_INVALID_ARG"]
    assert L.mla_front_end(dp.cfg, dp.pj, dp.x, dp.q, dp.kva, dp.wl.B, None, 0) == L.STATUS_CODE["MLA_ERR_WORKSPACE"]
    assert L.mla_front_end(dp.cfg, dp.pj, dp.x.data_ptr() + 4, dp.q, dp.kva, dp.wl.B, dp.ws, dp.ws.numel()) == INVALID
    saved = dp.pj.w_kva
    dp.pj.w_kva = None
    assert L.mla_front_end(dp.cfg, dp.pj, dp.x, dp.q, dp.kva, dp.wl.B, dp.ws, dp.ws.numel()) == INVALID
    dp.pj.w_kva = saved
    assert L.mla_o_proj(dp.cfg, dp.pj, dp.attn, dp.y, dp.wl.B, None, 0) == L.STATUS_CODE["MLA_ERR_WORKSPACE"]
    dp.pj.w_o = None
    assert L.mla_o_proj(dp.cfg, dp.pj, dp.attn, dp.y, dp.wl.B, dp.ws_o, dp.ws_o.numel()) == INVALID


@gpu
@pytest.mark.parametrize("q_lora", [0, 128])
def test_whole_layer_against_oracle(q_lora):
    """x -> mla_front_end -> mla_cache_append (the kv_a rows) -> mla_decode_attn -> mla_o_proj,
    against the oracle's layer on the same inputs, V2-Lite-sized heads over a short context."""
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceProj, DeviceStep
    from oracle import mla_oracle as O
    B = 3
    wl = synth.WORKLOADS["v2lite_b1_t4096"].with_(B=B, context=("uniform", 40, 300))
    prob = synth.make_problem(wl)
    pw = PW["v2lite_proj_b1"].with_(B=B, q_lora=q_lora)
    pp = synth.make_proj_problem(pw)
    dp = DeviceProj(pp)
    ds = DeviceStep(prob)
    L.check(dp.front_end(), "front end")
    ds.q.copy_(dp.q)
    L.check(L.mla_cache_append(ds.cfg, ds.cache, dp.kva, None, 0, ds.norm_w, ds.positions, ds.len_before, B,
                               ds.ws_append, ds.ws_append.numel(), ds.stream), "append")
    L.check(ds.decode(), "decode")
    L.check(dp.o_proj(ds.out), "o_proj")
    torch.cuda.synchronize()

    q, kva = OS.front_end(pp)
    q_stored = OS.store(q, wl.act)
    inv, scale = OS.tables(wl)
    new_rows = O.append_rows(kva, prob.norm_w, prob.positions, inv, wl.C, wl.rms_eps)
    seq_rows = [OS.sequence_rows(prob, b, OS.store(new_rows[b], wl.act)) for b in range(B)]
    out, _ = O.decode_step(q_stored, OS.kv_b_f64(prob), seq_rows, prob.positions, inv, scale, wl.H, wl.N, wl.V,
                           wl.C)
    y = OS.o_proj(pp, out)
    r = max_rel(dp.y.cpu().numpy(), y)
    assert r <= 1e-2, f"layer output max-rel {r}"
