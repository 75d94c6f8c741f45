"""The one-launch decode for tiny batches (plan kernel 3: absorb, attention over 32-row chunks,
merge and W_UV in one grid with grid-wide barriers) against the fp64 oracle: ragged lengths
(chunks with fewer than 32 rows, one-row sequences), several sequences sharing the grid, CTAs
that take two chunks or two absorb / merge items, 32 heads (four heads per warp, two 16-head
tensor-core tiles), a 256-wide latent, paged caches. The full-size one-sequence workload runs
through it in test_gpu_parity. Each case is one the planner hands to the one-launch path."""
import numpy as np
import pytest

from mla_latent_cache_absorb_gb300 import synth
from tests.gpu_util import check_step, need_gpu, run_gpu

gpu = pytest.mark.gpu
W = synth.WORKLOADS
V2 = W["v2lite_b1_t4096"]

CASES = [
    ("b2_ragged", V2.with_(B=2, context=("uniform", 1, 700))),            # two rounds of items
    ("b4_h4", V2.with_(B=4, H=4, context=("uniform", 30, 2000))),         # two rounds of chunks
    ("one_row", V2.with_(B=1, context=("fixed", 0))),                     # L = 1: one short chunk
    ("exact_chunks", V2.with_(B=1, context=("fixed", 255))),              # L = 256: 8 full chunks
    ("h32", W["v3_b32_t4096"].with_(B=1, H=32, context=("fixed", 1000))),
    ("h32_c256", V2.with_(B=1, H=32, C=256, context=("fixed", 700))),
    ("paged_b3", W["ragged_paged_b64"].with_(B=3, H=8, context=("uniform", 1, 900))),
]


def _plan(ds, B):
    from mla_latent_cache_absorb_gb300 import binding as L
    st, plan = L.mla_decode_plan(ds.cfg, B)
    L.check(st, "plan")
    return plan


@gpu
@pytest.mark.parametrize("name,wl", CASES, ids=[c[0] for c in CASES])
def test_one_launch_decode_parity(name, wl):
    need_gpu()
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    prob = synth.make_problem(wl)
    plan = _plan(DeviceStep(prob), wl.B)
    assert plan.kernel == 3 and plan.rows_per_split == 32, (plan.kernel, plan.rows_per_split)
    check_step(prob, tag=name)


@gpu
def test_one_launch_batch_slice_equals_single_sequence():
    """Chunk boundaries depend on a sequence's own length only, so its result does not depend on
    the rest of the batch: each copy of a sequence in a batch of three equals it run alone, bit
    for bit."""
    need_gpu()
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    wl = V2.with_(B=1, H=8, context=("fixed", 777))
    prob1 = synth.make_problem(wl)
    assert _plan(DeviceStep(prob1), 1).kernel == 3
    _, o1, l1, _ = run_gpu(prob1)
    prob3 = synth.make_problem(wl)
    prob3.wl = wl.with_(B=3)
    prob3.pool = np.concatenate([prob1.pool] * 3, axis=0)
    prob3.q = np.concatenate([prob1.q] * 3, axis=0)
    prob3.positions = np.repeat(prob1.positions, 3)
    prob3.seq_lens = np.repeat(prob1.seq_lens, 3)
    prob3.kva_rows = np.concatenate([prob1.kva_rows] * 3, axis=0)
    assert _plan(DeviceStep(prob3), 3).kernel == 3
    _, o3, l3, _ = run_gpu(prob3)
    for b in range(3):
        assert np.array_equal(o3[b], o1[0]) and np.array_equal(l3[b], l1[0])
