"""Multi-token decode (several query tokens per sequence, their rows already cached) on the GPU
against the fp64 oracle: each token attends its own causal prefix; the T tokens share every
staged row tile as T x H heads. Tensor-core and CUDA-core attention paths, contiguous and paged
caches, bf16 / Q8_0 / 4-bit kv_b, 16 and 128 heads; T = 1 is bit-identical to mla_decode_attn;
a sequence shorter than T is a device error."""
import dataclasses

import numpy as np
import pytest

from mla_latent_cache_absorb_gb300 import synth
from oracle import step as OS
from tests.gpu_util import LSE_TOL, OUT_TOL, max_rel, need_gpu

gpu = pytest.mark.gpu
W = synth.WORKLOADS

CASES = [
    ("h16_t2_b1", W["v2lite_b1_t4096"].with_(tokens=2)),
    ("h16_t4_b3_paged", W["v2lite_b1_t4096"].with_(B=3, tokens=4, page_size=64, context=("uniform", 4, 900))),
    ("h16_t8_ragged_tail", W["v2lite_b1_t4096"].with_(B=2, tokens=8, context=("uniform", 125, 131))),
    ("h128_t2_b4", W["v3_b32_t4096"].with_(B=4, tokens=2, context=("uniform", 300, 2000))),
    ("h128_t2_b8_tc_gemms", W["v3_b32_t4096"].with_(B=8, tokens=2, context=("uniform", 200, 1000))),
    ("h128_t3_paged_q8", W["ragged_paged_b64"].with_(B=5, tokens=3, kv_b="q8_0", context=("uniform", 3, 1500))),
    ("h128_t2_b9_q4", W["v3_b32_t4096"].with_(B=9, tokens=2, kv_b="q4_affine", context=("fixed", 700))),
    ("f32_t3", W["tiny_f32"].with_(B=2, tokens=3, context=("uniform", 3, 90))),
]


def _run(prob, positions=True):
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    ds = DeviceStep(prob)
    L.check(ds.decode_multi(positions=positions), "mla_decode_attn_multi")
    torch.cuda.synchronize()
    err, seq = L.mla_get_device_error(ds.ws_decode)
    return ds, err, seq


@gpu
@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_multi_token_parity(name, wl):
    prob = synth.make_problem(wl)
    ds, err, _ = _run(prob)
    assert err == 0, f"device error {err}"
    out, lse = ds.out.cpu().numpy(), ds.lse.cpu().numpy()
    o_out, o_lse = OS.run_multi(prob)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    r = max_rel(out, o_out)
    assert r <= OUT_TOL, f"{name}: out max-rel {r}"
    dl = float(np.max(np.abs(lse - o_lse)))
    assert dl <= LSE_TOL, f"{name}: lse max-abs {dl}"


@gpu
def test_single_token_is_bit_identical_to_decode_attn():
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    for wl in (W["v3_b32_t4096"].with_(B=3, context=("uniform", 100, 3000)), W["v2lite_b1_t4096"]):
        ds = DeviceStep(synth.make_problem(wl))
        L.check(ds.append(), "append")   # the one-token problems leave the new row to the append
        L.check(ds.decode(), "decode")
        torch.cuda.synchronize()
        o, l = ds.out.clone(), ds.lse.clone()
        assert bool(torch.isfinite(o).all())
        L.check(ds.decode_multi(), "decode_multi")
        torch.cuda.synchronize()
        assert torch.equal(o, ds.out) and torch.equal(l, ds.lse)


@gpu
def test_tokens_share_the_last_token_view():
    """The last token of a T-token call attends exactly the rows a one-token call with the same
    query and length would: its outputs agree within the tolerance (different head grouping)."""
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    wl = W["v2lite_b1_t4096"].with_(B=2, tokens=4, context=("uniform", 500, 1500))
    prob = synth.make_problem(wl)
    ds, err, _ = _run(prob)
    assert err == 0
    # the same cache and lengths, one query: the last token's, at its position
    single = dataclasses.replace(prob, wl=wl.with_(tokens=1), q=np.ascontiguousarray(prob.q[:, -1]),
                                 positions=(prob.positions + wl.tokens - 1).astype(np.int32))
    d1 = DeviceStep(single)
    L.check(d1.decode(), "decode")
    torch.cuda.synchronize()
    # a wrong row view would differ at O(1); the one-token call runs in float32 here (the
    # one-launch path for tiny batches) and the T-token call from bf16 latent queries, so they
    # agree to the oracle's output tolerance rather than to bf16 rounding of the same sums
    r = max_rel(ds.out[:, -1].cpu().numpy(), d1.out.cpu().numpy())
    assert r <= OUT_TOL, r


@gpu
def test_sequence_shorter_than_tokens_is_a_device_error():
    need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    wl = W["v2lite_b1_t4096"].with_(B=2, tokens=4, context=("uniform", 4, 50))
    prob = synth.make_problem(wl)
    prob.seq_lens = prob.seq_lens.copy()
    prob.seq_lens[1] = 3
    ds, err, seq = _run(prob)
    assert err == L.STATUS_CODE["MLA_ERR_BAD_SEQ_LEN"] and seq == 1
    out = ds.out.cpu().numpy()
    assert np.all(np.isnan(out[1])) and np.all(np.isfinite(out[0]))
