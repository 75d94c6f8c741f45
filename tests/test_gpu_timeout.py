"""The timeout path of the bounded device waits, driven on purpose and without a fault: the
main-loop wait limit is set far below what a copy or an MMA takes (mla_set_wait_limit_ns), so
the tensor-core kernels' waits (and the one-launch path's grid-wide barriers) run out. Each such CTA records MLA_ERR_TIMEOUT, drains what it
issued, frees its tensor memory and writes NaN for the outputs it owns; the context stays
usable and the next call with the normal limit is bit-identical to a clean run."""
import numpy as np
import pytest

from mla_latent_cache_absorb_gb300 import synth
from tests.gpu_util import need_gpu

gpu = pytest.mark.gpu
W = synth.WORKLOADS

CASES = [
    # 128 heads, eight sequences: tcgen05 absorb, SM-pair attention and combine
    ("h128_b8", W["v3_b32_t4096"].with_(B=8, context=("fixed", 300))),
    # 16 heads, five sequences: tcgen05 attention (16-head group) between the CUDA-core kernels
    ("h16_b5", W["v2lite_b1_t4096"].with_(B=5, context=("fixed", 1000))),
    # 16 heads, one sequence: the one-launch path (its grid-wide barriers and row copies)
    ("h16_b1_one_launch", W["v2lite_b1_t4096"].with_(context=("fixed", 1000))),
]


@gpu
@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_waits_run_out_and_the_next_call_is_clean(name, wl):
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    ds = DeviceStep(synth.make_problem(wl))
    L.check(ds.append(), "append")
    L.check(ds.decode(), "decode")
    assert L.mla_get_device_error(ds.ws_decode, ds.stream)[0] == 0
    clean_out, clean_lse = ds.out.clone(), ds.lse.clone()
    assert torch.isfinite(clean_out).all()

    prev = L.mla_set_wait_limit_ns(1)
    try:
        L.check(ds.decode(), "decode with a 1 ns wait limit")
        st, _ = L.mla_get_device_error(ds.ws_decode, ds.stream)
    finally:
        assert L.mla_set_wait_limit_ns(0) == 1
    assert prev == 200_000_000
    assert st == L.STATUS_CODE["MLA_ERR_TIMEOUT"], L.STATUS.get(st, st)

    # every (sequence, head) output is either NaN (its CTA gave up) or exactly the clean value
    out, lse = ds.out.cpu().numpy(), ds.lse.cpu().numpy()
    co, cl = clean_out.cpu().numpy(), clean_lse.cpu().numpy()
    nan = np.isnan(out).all(axis=-1)
    assert nan.any(), "a timed-out run produced no NaN output"
    assert np.array_equal(out[~nan], co[~nan]) and np.array_equal(lse[~nan], cl[~nan])
    assert not np.isnan(out[~nan]).any()

    # the context is still usable: clear the error word, decode with the normal limit
    L.check(L.mla_clear_device_error(ds.ws_decode, ds.stream), "clear")
    L.check(ds.decode(), "decode")
    assert L.mla_get_device_error(ds.ws_decode, ds.stream)[0] == 0
    torch.cuda.synchronize()
    assert torch.equal(ds.out, clean_out) and torch.equal(ds.lse, clean_lse)


def test_wait_limit_setting_round_trips():
    pytest.importorskip("torch")
    from mla_latent_cache_absorb_gb300 import binding as L
    assert L.mla_set_wait_limit_ns(5_000) == 200_000_000
    assert L.mla_set_wait_limit_ns(0) == 5_000
    assert L.mla_set_wait_limit_ns(0) == 200_000_000
