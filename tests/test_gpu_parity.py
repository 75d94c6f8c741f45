"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the same seeded
inputs. Small cases span several row tiles and a ragged tail; the five workloads run at full
size with outputs compared on all (or sampled) sequences and heads."""
import numpy as np
import pytest

from mla_latent_cache_absorb_gb300 import synth
from tests.gpu_util import LSE_TOL, OUT_TOL, check_step, max_rel, need_gpu, run_gpu

W = synth.WORKLOADS
gpu = pytest.mark.gpu


# ---- small cases: several tiles and a ragged tail ---------------------------------------------

SMALL = [
    ("tiny_f32", W["tiny_f32"]),
    ("tiny_f32_long", W["tiny_f32"].with_(B=3, context=("fixed", 1000))),
    ("v2lite_small", W["v2lite_b1_t4096"].with_(context=("fixed", 1000))),
    ("v2lite_b3", W["v2lite_b1_t4096"].with_(B=3, context=("fixed", 300))),
    ("v3_b4_h128", W["v3_b32_t4096"].with_(B=4, context=("fixed", 777))),
    ("ragged_paged_small", W["ragged_paged_b64"].with_(B=6, context=("uniform", 1, 900))),
    ("ragged_contig_small", W["ragged_paged_b64"].with_(B=5, page_size=0, context=("uniform", 1, 700))),
    ("q8_gemv_small", W["long_q8_b4_t131072"].with_(B=2, context=("fixed", 1500))),
    ("q8_gemv_h16", W["long_q8_b4_t131072"].with_(B=3, H=16, context=("fixed", 129), hidden=1024)),
    # nine sequences: the kv_a projection's second register pass and a second combine block
    ("q8_gemv_b9", W["long_q8_b4_t131072"].with_(B=9, H=16, context=("fixed", 200), hidden=1024)),
    ("bf16_odd_heads", W["v3_b32_t4096"].with_(B=2, H=24, context=("fixed", 200))),
    # one 64-head group (two softmax warpgroups); 96 heads: a second group half filled, so its
    # second warpgroup owns no real head
    ("h64_one_group", W["v3_b32_t4096"].with_(B=3, H=64, context=("fixed", 500))),
    ("h96_partial_group", W["v3_b32_t4096"].with_(B=2, H=96, context=("uniform", 100, 600))),
]


@gpu
@pytest.mark.parametrize("name,wl", SMALL, ids=[s[0] for s in SMALL])
def test_small_parity(name, wl):
    need_gpu()
    check_step(synth.make_problem(wl), tag=name)


@gpu
def test_single_row_sequence():
    need_gpu()
    # L = 1: the sequence attends only its freshly appended row
    check_step(synth.make_problem(W["v3_b32_t4096"].with_(B=2, H=16, context=("fixed", 0))), tag="L1")


@gpu
def test_prerotated_q_pe_matches_positions_path():
    torch = need_gpu()
    from oracle import mla_oracle as O
    from oracle import step as OS
    wl = W["v2lite_b1_t4096"].with_(B=2, context=("fixed", 300))
    prob = synth.make_problem(wl)
    # rotate q_pe on the host with the oracle, store it, and decode with positions = NULL
    inv, _ = OS.tables(wl)
    q = OS.decode_act(prob.q, wl.act)
    for b in range(wl.B):
        q[b, :, wl.N:] = O.rope_pairs(q[b, :, wl.N:], int(prob.positions[b]), inv)
    prob.q = synth.f32_to_bf16_bits(q.astype(np.float32))
    _, out, lse, _ = run_gpu(prob, positions=False)
    # oracle with pos = None: q_pe is taken as already rotated
    W_UK, W_UV = O.split_kv_b(OS.kv_b_f64(prob), wl.H, wl.N, wl.V)
    new = OS.store(OS.appended_rows(prob), wl.act)
    for b in range(wl.B):
        rows = OS.sequence_rows(prob, b, new[b])
        ob, lb = O.decode_one(OS.decode_act(prob.q, wl.act)[b], W_UK, W_UV, rows, None, inv,
                              OS.tables(wl)[1], wl.C)
        assert max_rel(out[b], ob) <= OUT_TOL
        assert np.max(np.abs(lse[b] - lb)) <= LSE_TOL


@gpu
def test_large_query_positions_on_the_tensor_core_absorb():
    """The batched (tcgen05) absorb rotates q_pe with float-only angle arithmetic below 2^18 and
    the double path above it: query positions from 0 past that limit, against the oracle."""
    torch = need_gpu()
    from oracle import mla_oracle as O
    from oracle import step as OS
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    wl = W["v3_b32_t4096"].with_(B=8, context=("fixed", 160))
    prob = synth.make_problem(wl)
    qpos = np.array([0, 1, 4095, 65535, 131072, 200003, 262143, 262144 + 12345], dtype=np.int32)
    ds = DeviceStep(prob)
    st, plan = L.mla_decode_plan(ds.cfg, wl.B)
    L.check(st, "plan")
    L.check(ds.append(), "append")                 # the new rows at their own positions
    ds.positions = torch.from_numpy(qpos).to(ds.device)
    L.check(ds.decode(), "decode")
    torch.cuda.synchronize()
    out, lse = ds.out.cpu().numpy(), ds.lse.cpu().numpy()
    inv, scale = OS.tables(wl)
    W_UK, W_UV = O.split_kv_b(OS.kv_b_f64(prob), wl.H, wl.N, wl.V)
    new = OS.store(OS.appended_rows(prob), wl.act)
    q = OS.decode_act(prob.q, wl.act)
    for b in range(wl.B):
        ob, lb = O.decode_one(q[b], W_UK, W_UV, OS.sequence_rows(prob, b, new[b]), int(qpos[b]), inv, scale, wl.C)
        assert max_rel(out[b], ob) <= OUT_TOL, b
        assert np.max(np.abs(lse[b] - lb)) <= LSE_TOL, b


# ---- full-size workloads ------------------------------------------------------------------------

@gpu
def test_full_tiny_f32():
    need_gpu()
    check_step(synth.make_problem(W["tiny_f32"]), tag="tiny_f32")


@gpu
def test_full_v2lite_b1_t4096():
    need_gpu()
    check_step(synth.make_problem(W["v2lite_b1_t4096"]), tag="v2lite")


@gpu
def test_full_v3_b32_t4096():
    need_gpu()
    check_step(synth.make_problem(W["v3_b32_t4096"]), seqs=[0, 7, 31], tag="v3")


@gpu
def test_full_ragged_paged_b64():
    need_gpu()
    prob = synth.make_problem(W["ragged_paged_b64"])
    L = prob.seq_lens
    seqs = sorted({int(np.argmin(L)), int(np.argmax(L)), 0, 63})
    check_step(prob, seqs=seqs, heads=np.arange(0, 128, 9), tag="ragged")


@gpu
def test_full_long_q8_b4_t131072():
    need_gpu()
    check_step(synth.make_problem(W["long_q8_b4_t131072"]), seqs=[0, 3], heads=np.arange(0, 128, 17),
               tag="long_q8")


# ---- structural properties ------------------------------------------------------------------------

@gpu
def test_run_to_run_bit_identical():
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    prob = synth.make_problem(W["v3_b32_t4096"].with_(B=3, context=("fixed", 1000)))
    ds = DeviceStep(prob)
    L.check(ds.append(), "append")
    L.check(ds.decode(), "decode")
    torch.cuda.synchronize()
    o1, l1 = ds.out.clone(), ds.lse.clone()
    L.check(ds.decode(), "decode")
    torch.cuda.synchronize()
    assert torch.equal(o1, ds.out) and torch.equal(l1, ds.lse)


@gpu
def test_identity_page_table_equals_contiguous():
    torch = need_gpu()
    wl = W["v3_b32_t4096"].with_(B=3, H=32, context=("fixed", 255))
    prob_c = synth.make_problem(wl)
    # the same rows laid out as 64-row pages with an identity page table
    prob_p = synth.make_problem(wl)
    cap = prob_c.rows_per_seq
    pages = (cap + 63) // 64
    pool = np.full((wl.B * pages * 64, wl.row), synth.BF16_NAN_BITS, dtype=np.uint16)
    for b in range(wl.B):
        pool[b * pages * 64: b * pages * 64 + cap] = prob_c.pool[b * cap:(b + 1) * cap]
    prob_p.pool = pool
    prob_p.page_table = np.arange(wl.B * pages, dtype=np.int32).reshape(wl.B, pages)
    prob_p.max_pages = pages
    prob_p.rows_per_seq = 0
    prob_p.wl = wl.with_(page_size=64)
    _, oc, lc, _ = run_gpu(prob_c)
    _, op, lp, _ = run_gpu(prob_p)
    assert np.array_equal(oc, op) and np.array_equal(lc, lp)


@gpu
def test_batched_slice_equals_single_sequence():
    # each sequence of a batch of identical sequences matches the same sequence run alone
    # (the split plan depends on B, so agreement is to float32 reassociation, not bits; when the
    # planner hands the single sequence to the one-launch path and the batch to the staged
    # kernels, agreement is to the two paths' parity tolerance)
    need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    wl = W["v2lite_b1_t4096"].with_(B=1, context=("fixed", 500))
    prob1 = synth.make_problem(wl)
    _, o1, l1, _ = run_gpu(prob1)
    # batch of 3 copies of the same sequence
    prob3 = synth.make_problem(wl)
    rows = prob1.rows_per_seq
    prob3.wl = wl.with_(B=3)
    prob3.pool = np.concatenate([prob1.pool] * 3, axis=0)
    prob3.q = np.concatenate([prob1.q] * 3, axis=0)
    prob3.positions = np.repeat(prob1.positions, 3)
    prob3.seq_lens = np.repeat(prob1.seq_lens, 3)
    prob3.kva_rows = np.concatenate([prob1.kva_rows] * 3, axis=0)
    _, o3, l3, _ = run_gpu(prob3)
    k1 = L.mla_decode_plan(DeviceStep(prob1).cfg, 1)[1].kernel
    k3 = L.mla_decode_plan(DeviceStep(prob3).cfg, 3)[1].kernel
    to, tl = (1e-5, 1e-5) if (k1 == 3) == (k3 == 3) else (OUT_TOL, LSE_TOL)
    for b in range(3):
        assert max_rel(o3[b], o1[0]) <= to and np.max(np.abs(l3[b] - l1[0])) <= tl
    assert np.array_equal(o3[0], o3[1]) and np.array_equal(o3[1], o3[2])


STEP_CASES = [
    # short attentions: every kernel launched with programmatic serialization
    ("v2lite_b1", W["v2lite_b1_t4096"].with_(context=("fixed", 1500))),              # SIMT absorb + combine
    ("v3_b9_h128", W["v3_b32_t4096"].with_(B=9, context=("uniform", 100, 1200))),    # tensor-core absorb + combine
    ("ragged_paged_b6", W["ragged_paged_b64"].with_(B=6, context=("uniform", 1, 900))),
    ("tiny_f32", W["tiny_f32"]),                                                      # CUDA-core attention
    # long attentions (>= 4 tiles per CTA at capacity): absorb in plain order, early cache reads
    ("v3_b16_long", W["v3_b32_t4096"].with_(B=16, context=("uniform", 1500, 2500))),
    ("q8_b2_long", W["long_q8_b4_t131072"].with_(B=2, context=("fixed", 20000))),    # SIMT absorb + combine
    ("ragged_paged_b24_long", W["ragged_paged_b64"].with_(B=24, context=("uniform", 200, 3000))),
]


@gpu
@pytest.mark.parametrize("name,wl", STEP_CASES, ids=[c[0] for c in STEP_CASES])
def test_fused_call_equals_the_three_step_calls(name, wl):
    # for long attentions mla_decode_attn launches its absorb in plain stream order and lets
    # the attention read cache rows before waiting for it; the three step calls keep every wait
    # in place. Same kernels, same split plan: the results agree bit for bit. For tiny batches
    # (plan kernel 3) mla_decode_attn is one float32 launch instead: it agrees with the step
    # calls within the oracle's tolerances and is run-to-run identical.
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    ds = DeviceStep(synth.make_problem(wl))
    st, plan = L.mla_decode_plan(ds.cfg, wl.B)
    L.check(st, "plan")
    L.check(ds.append(), "mla_cache_append")
    L.check(ds.absorb(), "mla_decode_absorb")
    L.check(ds.partial(), "mla_decode_partial")
    L.check(ds.combine(), "mla_decode_combine")
    torch.cuda.synchronize()
    o_steps, l_steps = ds.out.clone(), ds.lse.clone()
    assert torch.isfinite(o_steps).all()
    ds.out.fill_(float("nan"))
    ds.lse.fill_(float("nan"))
    first = None
    for _ in range(2):   # twice: the second call follows the first call's combine, not an append
        L.check(ds.decode(), "mla_decode_attn")
        torch.cuda.synchronize()
        if plan.kernel == 3:
            assert max_rel(ds.out.cpu().numpy(), o_steps.cpu().numpy()) <= OUT_TOL
            assert float((ds.lse - l_steps).abs().max()) <= LSE_TOL
            if first is None:
                first = (ds.out.clone(), ds.lse.clone())
            else:
                assert torch.equal(ds.out, first[0]) and torch.equal(ds.lse, first[1])
        else:
            assert torch.equal(ds.out, o_steps) and torch.equal(ds.lse, l_steps)
    e, seq = L.mla_get_device_error(ds.ws_decode, ds.stream)
    assert e == 0, (e, seq)
