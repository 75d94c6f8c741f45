"""Helpers for the GPU parity tests: run a synthetic problem through the C ABI and compare it
with the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest

from oracle import step as OS

# Tolerances of the method's statement: max|gpu - oracle| / max|oracle| <= 1e-2 on out and on
# the appended row; per-head |lse_gpu - lse_oracle| <= 1e-3 (absolute).
OUT_TOL = 1e-2
LSE_TOL = 1e-3
# each element of the appended row: within one bf16 step of the oracle's correctly rounded value
ROW_ELEM_REL = 2.0 ** -7


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def max_rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-30))


def run_gpu(prob, positions=True, stream=None):
    """Upload, run append + decode, return (DeviceStep, out, lse, pool after)."""
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300 import binding as L
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    ds = DeviceStep(prob, stream=stream)
    L.check(ds.append(), "append")
    L.check(ds.decode(positions=positions), "decode")
    torch.cuda.synchronize()
    return ds, ds.out.cpu().numpy(), ds.lse.cpu().numpy(), ds.pool_host()


def check_step(prob, seqs=None, heads=None, tag=""):
    """Full step on the GPU vs the oracle: cache rows (bit-exact placement, every untouched
    row byte-identical), appended row values, out and lse."""
    from mla_latent_cache_absorb_gb300 import binding as L
    from oracle import mla_oracle as O
    wl = prob.wl
    ds, out, lse, pool_after = run_gpu(prob)
    (ea, _), (ed, _) = ds.device_errors()
    assert ea == 0 and ed == 0, f"device errors append={L.STATUS[ea]} decode={L.STATUS[ed]}"
    seqs = list(range(wl.B)) if seqs is None else list(seqs)
    heads = np.arange(wl.H) if heads is None else np.asarray(heads)
    new_rows, o_out, o_lse = OS.run_step(prob, seqs=seqs, heads=heads)

    # cache: only the appended rows changed, each at its physical slot
    slots = np.array([int(O.physical_row(b, int(prob.positions[b]), prob.page_table, wl.page_size,
                                         prob.rows_per_seq)) for b in range(wl.B)])
    mask = np.ones(prob.pool.shape[0], dtype=bool)
    mask[slots] = False
    if wl.act == "bf16":
        assert np.array_equal(pool_after[mask], prob.pool[mask]), "rows other than the appended ones changed"
    else:
        assert np.array_equal(pool_after[mask].view(np.uint32), prob.pool[mask].view(np.uint32))
    got_rows = OS.decode_act(pool_after[slots], wl.act)
    assert max_rel(got_rows, new_rows) <= OUT_TOL, f"{tag} appended row max-rel {max_rel(got_rows, new_rows)}"
    elem = np.abs(got_rows - new_rows) <= ROW_ELEM_REL * np.abs(new_rows) + 1e-6
    assert elem.all(), f"{tag} appended row elements off by more than one bf16 step: {np.argwhere(~elem)[:5]}"

    g_out = out[seqs][:, heads]
    g_lse = lse[seqs][:, heads]
    assert np.all(np.isfinite(g_out)) and np.all(np.isfinite(g_lse)), f"{tag} non-finite output"
    r = max_rel(g_out, o_out)
    assert r <= OUT_TOL, f"{tag} out max-rel {r}"
    dl = float(np.max(np.abs(g_lse - o_lse)))
    assert dl <= LSE_TOL, f"{tag} lse max-abs {dl}"
    return ds, {"out_max_rel": r, "lse_max_abs": dl}
