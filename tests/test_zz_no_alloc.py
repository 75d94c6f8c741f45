"""mla_decode_attn_noalloc (the allocation-free decode call) against mla_decode_attn.

Both calls run the same kernels with the same split plan, so for the same inputs the outputs
must agree bit for bit; two calls in a row check that the array's state left by one call
does not leak into the next. The file sorts last so that it also runs after every other test
has used the library in the same process.
"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_scratch_size_constant_matches_header():
    src = open(os.path.join(ROOT, "include", "mla.h")).read()
    m = re.search(r"#define MLA_NOALLOC_SCRATCH_BYTES \((\d+)ull \* 1024ull \* 1024ull\)", src)
    assert m is not None
    from mla_latent_cache_absorb_gb300 import binding as L
    assert L.MLA_NOALLOC_SCRATCH_BYTES == int(m.group(1)) * 1024 * 1024


def _problem(name, **kw):
    from mla_latent_cache_absorb_gb300 import synth
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    wl = synth.WORKLOADS[name].with_(**kw)
    ds = DeviceStep(synth.make_problem(wl))
    return ds


def _noalloc(ds, out, lse, err, seq_lens=None):
    from mla_latent_cache_absorb_gb300 import binding as L
    return L.mla_decode_attn_noalloc(ds.cfg, ds.q, ds.kv_b, ds.cache,
                                     ds.seq_lens if seq_lens is None else seq_lens, ds.positions,
                                     out, lse, ds.wl.B, err, ds.stream)


CASES = [
    ("tiny_f32", "tiny_f32", {}),                                               # CUDA-core attention
    ("v2lite_tc", "v2lite_b1_t4096", dict(B=5, context=("uniform", 100, 900))),   # tcgen05, 16 heads
    ("v2lite_one_launch", "v2lite_b1_t4096", dict(B=2, context=("uniform", 100, 900))),  # tiny batch
    ("v3", "v3_b32_t4096", dict(B=5, context=("uniform", 200, 1500))),          # tcgen05, 128 heads
    ("ragged_paged", "ragged_paged_b64", dict(B=6, context=("uniform", 64, 2000))),  # paged cache
    # a long attention: the absorb launched in plain stream order, cache rows read early
    ("v3_long", "v3_b32_t4096", dict(B=16, context=("uniform", 1500, 2500))),
]


@pytest.mark.gpu
@pytest.mark.parametrize("name,kw", [c[1:] for c in CASES], ids=[c[0] for c in CASES])
def test_noalloc_matches_decode_attn_twice_in_a_row(name, kw):
    import torch
    from mla_latent_cache_absorb_gb300 import binding as L
    ds = _problem(name, **kw)
    L.check(ds.append(), "mla_cache_append")
    L.check(ds.decode(), "mla_decode_attn")
    torch.cuda.synchronize()
    ref_out, ref_lse = ds.out.clone(), ds.lse.clone()
    assert torch.isfinite(ref_out).all()
    for call in range(2):
        out = torch.full_like(ds.out, float("nan"))
        lse = torch.full_like(ds.lse, float("nan"))
        err = torch.full((2,), -7, dtype=torch.int32, device=ds.device)
        L.check(_noalloc(ds, out, lse, err), "mla_decode_attn_noalloc")
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out), f"call {call}: out differs from mla_decode_attn"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from mla_decode_attn"
        assert err.tolist() == [0, 0]


@pytest.mark.gpu
def test_noalloc_reports_each_calls_own_device_error():
    import torch
    from mla_latent_cache_absorb_gb300 import binding as L
    ds = _problem("v2lite_b1_t4096", B=4, context=("uniform", 100, 700))
    L.check(ds.append(), "mla_cache_append")
    L.check(ds.decode(), "mla_decode_attn")
    torch.cuda.synchronize()
    ref_out = ds.out.clone()
    bad = ds.seq_lens.clone()
    bad[2] = 0                                     # an empty sequence is a device error
    out, lse = torch.empty_like(ds.out), torch.empty_like(ds.lse)
    err = torch.zeros(2, dtype=torch.int32, device=ds.device)
    L.check(_noalloc(ds, out, lse, err, seq_lens=bad), "mla_decode_attn_noalloc")
    torch.cuda.synchronize()
    assert err.tolist() == [L.STATUS_CODE["MLA_ERR_BAD_SEQ_LEN"], 2]
    assert torch.isnan(out[2]).all() and torch.isnan(lse[2]).all()
    keep = [0, 1, 3]
    # unaffected up to float32 summation order (the invalid length can move split boundaries)
    ref = ref_out[keep]
    assert float((out[keep] - ref).abs().max()) <= 1e-5 * float(ref.abs().max())
    # the next call starts from a cleared error word
    L.check(_noalloc(ds, out, lse, err), "mla_decode_attn_noalloc")
    torch.cuda.synchronize()
    assert err.tolist() == [0, 0]
    assert torch.equal(out, ref_out)


@pytest.mark.gpu
def test_noalloc_refuses_a_batch_the_array_cannot_hold():
    import torch
    from mla_latent_cache_absorb_gb300 import binding as L
    ds = _problem("v3_b32_t4096", B=2, context=("fixed", 300))
    big_b = 256                                    # 128 heads x 256 sequences: > 64 MiB
    st, need = L.mla_decode_workspace_size(ds.cfg, big_b)
    L.check(st, "mla_decode_workspace_size")
    assert need > L.MLA_NOALLOC_SCRATCH_BYTES
    sentinel = torch.full((2,), 123, dtype=torch.int32, device=ds.device)
    st = L.mla_decode_attn_noalloc(ds.cfg, ds.q, ds.kv_b, ds.cache, ds.seq_lens, ds.positions,
                                   ds.out, ds.lse, big_b, sentinel, ds.stream)
    assert st == L.STATUS_CODE["MLA_ERR_WORKSPACE"]
    torch.cuda.synchronize()
    assert sentinel.tolist() == [123, 123]          # nothing was enqueued


@pytest.mark.gpu
def test_noalloc_allocates_no_device_memory():
    """The call's promise itself: after a first call (which may load the library's module on
    this device), further calls change neither the caching allocator's bytes in use nor the
    device's free memory."""
    import torch
    from mla_latent_cache_absorb_gb300 import binding as L
    ds = _problem("v3_b32_t4096", B=5, context=("uniform", 200, 1500))
    L.check(ds.append(), "mla_cache_append")
    out, lse = torch.empty_like(ds.out), torch.empty_like(ds.lse)
    err = torch.zeros(2, dtype=torch.int32, device=ds.device)
    L.check(_noalloc(ds, out, lse, err), "mla_decode_attn_noalloc")
    torch.cuda.synchronize()
    used0 = torch.cuda.memory_allocated(ds.device)
    free0, _ = torch.cuda.mem_get_info(ds.device)
    for _ in range(3):
        L.check(_noalloc(ds, out, lse, err), "mla_decode_attn_noalloc")
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(ds.device)
    assert torch.cuda.memory_allocated(ds.device) == used0
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
    assert err.tolist() == [0, 0]
