"""The 128-head attention on SM pairs (a cluster of two CTAs, one latent half each, 64-row
tiles) against the fp64 oracle, on the shapes that exercise its exchange protocol: one-row and
one-tile sequences, many short sequences per pair (segment boundaries every tile or two), pairs
whose share starts or ends inside a sequence, ragged tails, paged caches, and more sequences
than pairs. The full-size workloads with 128 heads run through it in test_gpu_parity."""
import numpy as np
import pytest

from mla_latent_cache_absorb_gb300 import synth
from tests.gpu_util import check_step, need_gpu

gpu = pytest.mark.gpu
W = synth.WORKLOADS
V3 = W["v3_b32_t4096"]

CASES = [
    ("one_row", V3.with_(B=1, context=("fixed", 0))),
    ("one_tile_exact", V3.with_(B=2, context=("fixed", 63))),               # L = 64: one full tile
    ("two_tiles_ragged", V3.with_(B=1, context=("fixed", 100))),            # L = 101
    ("short_seqs_b40", V3.with_(B=40, context=("uniform", 1, 130))),        # 1-3 tiles each
    ("many_seqs_b200", V3.with_(B=200, context=("uniform", 1, 200))),       # more sequences than pairs
    ("long_b3", V3.with_(B=3, context=("uniform", 3000, 9000))),            # shares inside sequences
    ("paged_b12", W["ragged_paged_b64"].with_(B=12, context=("uniform", 1, 2500))),
    ("q8_b3", W["long_q8_b4_t131072"].with_(B=3, context=("fixed", 3000))),
]


@gpu
@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_pair_kernel_parity(name, wl):
    need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    prob = synth.make_problem(wl)
    st, plan = L.mla_decode_plan(DeviceStep(prob).cfg, wl.B)
    L.check(st, "plan")
    assert plan.kernel == 2 and plan.heads_per_cta == 128
    heads = None if wl.B <= 12 else np.arange(0, 128, 5)
    seqs = None if wl.B <= 40 else sorted({0, 1, 2, wl.B // 2, wl.B - 2, wl.B - 1})
    check_step(prob, seqs=seqs, heads=heads, tag=name)


@gpu
def test_pair_kernel_rescale_path():
    """Scores that grow along the sequence force the running maximum up tile after tile, so the
    output rows are rescaled in both CTAs of the pair (the factor sent with the probabilities)."""
    torch = need_gpu()
    wl = V3.with_(B=2, context=("fixed", 1000))
    prob = synth.make_problem(wl)
    # scale each cached row's latent part by a factor growing with its position: later rows score
    # higher, by far more than the rescale threshold over the sequence
    rows = prob.pool.astype(np.uint32) << 16
    f = rows.view(np.float32).reshape(prob.pool.shape).copy()
    for b in range(wl.B):
        base = b * prob.rows_per_seq
        ramp = np.linspace(0.2, 3.0, prob.rows_per_seq, dtype=np.float32)[:, None]
        f[base:base + prob.rows_per_seq, :wl.C] *= ramp
    prob.pool = synth.f32_to_bf16_bits(f)
    check_step(prob, tag="rescale")
