"""4-bit affine kv_b (groups of 64, bf16 scales and biases) on the GPU against the fp64 oracle:
the absorb reads W_UK and the combine reads W_UV through the same dequantisation, for 16 and
128 heads, contiguous and paged caches, and the fused call against the three step calls."""
import pytest

from mla_latent_cache_absorb_gb300 import synth
from tests.gpu_util import check_step, need_gpu

gpu = pytest.mark.gpu
W = synth.WORKLOADS

CASES = [
    ("h16_b2", W["v2lite_b1_t4096"].with_(B=2, kv_b="q4_affine", context=("fixed", 700))),
    ("h128_b3", W["v3_b32_t4096"].with_(B=3, kv_b="q4_affine", context=("uniform", 100, 1500))),
    ("h128_b9_paged", W["ragged_paged_b64"].with_(B=9, kv_b="q4_affine", context=("uniform", 1, 1200))),
    ("long_gemv_b2", W["long_q8_b4_t131072"].with_(B=2, kv_b="q4_affine", context=("fixed", 2000))),
]


@gpu
@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_q4_affine_kv_b_parity(name, wl):
    need_gpu()
    check_step(synth.make_problem(wl), tag=name)


@gpu
def test_q4_fused_call_equals_step_calls():
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    ds = DeviceStep(synth.make_problem(W["v3_b32_t4096"].with_(B=5, kv_b="q4_affine", context=("fixed", 900))))
    L.check(ds.append(), "append")
    L.check(ds.absorb(), "absorb")
    L.check(ds.partial(), "partial")
    L.check(ds.combine(), "combine")
    torch.cuda.synchronize()
    o, l = ds.out.clone(), ds.lse.clone()
    L.check(ds.decode(), "decode")
    torch.cuda.synchronize()
    assert torch.equal(o, ds.out) and torch.equal(l, ds.lse)
