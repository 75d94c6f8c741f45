"""Device-detected conditions: each bad input here is one the kernels check before any memory
access (a length, a position, a page id), so the kernel records a status in the workspace and
skips the work; nothing faults. The other sequences of the batch must be unaffected."""
import numpy as np
import pytest

from mla_latent_cache_absorb_gb300 import synth
from tests.gpu_util import OUT_TOL, max_rel, need_gpu

gpu = pytest.mark.gpu
W = synth.WORKLOADS


def _setup(wl):
    torch = need_gpu()
    from mla_latent_cache_absorb_gb300.runner import DeviceStep
    prob = synth.make_problem(wl)
    return torch, prob, DeviceStep(prob)


@gpu
@pytest.mark.parametrize("bad_len", [0, -5, 10 ** 6])
def test_bad_seq_len_sets_error_and_nan_only_for_that_sequence(bad_len):
    from mla_latent_cache_absorb_gb300 import binding as L
    torch, prob, ds = _setup(W["v2lite_b1_t4096"].with_(B=3, context=("fixed", 200)))
    L.check(ds.append(), "append")
    L.check(ds.decode(), "decode")
    torch.cuda.synchronize()
    good = ds.out.clone()
    ds.seq_lens[1] = bad_len
    L.check(ds.decode(), "decode")
    st, seq = L.mla_get_device_error(ds.ws_decode, ds.stream)
    assert st == L.STATUS_CODE["MLA_ERR_BAD_SEQ_LEN"] and seq == 1
    out = ds.out.cpu().numpy()
    assert np.all(np.isnan(out[1])) and np.all(np.isnan(ds.lse[1].cpu().numpy()))
    # the other sequences are unaffected; an invalid length can move the split boundaries (one
    # sequence fewer in the tile list), which changes only float32 summation order
    assert max_rel(out[0], good[0].cpu().numpy()) <= 1e-5 and max_rel(out[2], good[2].cpu().numpy()) <= 1e-5
    # the error is sticky until cleared
    ds.seq_lens[1] = 201
    L.check(ds.decode(), "decode")
    assert L.mla_get_device_error(ds.ws_decode, ds.stream)[0] == L.STATUS_CODE["MLA_ERR_BAD_SEQ_LEN"]
    L.check(L.mla_clear_device_error(ds.ws_decode, ds.stream), "clear")
    L.check(ds.decode(), "decode")
    assert L.mla_get_device_error(ds.ws_decode, ds.stream)[0] == 0
    assert max_rel(ds.out.cpu().numpy(), good.cpu().numpy()) == 0.0


@gpu
# 2**31 - 1: the largest int32 page id, whose end row overflows 32-bit arithmetic
@pytest.mark.parametrize("bad_page", [-1, 10 ** 7, 2 ** 31 - 1])
def test_bad_page_id_sets_error(bad_page):
    from mla_latent_cache_absorb_gb300 import binding as L
    torch, prob, ds = _setup(W["ragged_paged_b64"].with_(B=3, H=16, context=("uniform", 200, 400)))
    L.check(ds.append(), "append")
    ds.page_table[2, 1] = bad_page
    L.check(ds.decode(), "decode")
    st, seq = L.mla_get_device_error(ds.ws_decode, ds.stream)
    assert st == L.STATUS_CODE["MLA_ERR_BAD_PAGE"] and seq == 2
    out = ds.out.cpu().numpy()
    assert np.all(np.isnan(out[2])) and np.all(np.isfinite(out[:2]))


@gpu
def test_bad_page_id_in_a_long_attention():
    # 128 heads, 24 sequences of up to 3000 rows: long enough (>= 4 tiles per CTA at capacity)
    # that mla_decode_attn reads cache rows before its dependency wait, where the producers
    # meet the bad page id. The split plan does not depend on page ids, so every other
    # sequence matches a clean run bit for bit.
    from mla_latent_cache_absorb_gb300 import binding as L
    torch, prob, ds = _setup(W["ragged_paged_b64"].with_(B=24, context=("uniform", 200, 3000)))
    L.check(ds.append(), "append")
    L.check(ds.decode(), "decode")
    torch.cuda.synchronize()
    assert L.mla_get_device_error(ds.ws_decode, ds.stream)[0] == 0
    clean_out, clean_lse = ds.out.clone(), ds.lse.clone()
    assert int(ds.seq_lens[5]) > 2 * 64          # the page below is one the sequence reads
    ds.page_table[5, 1] = -1
    L.check(ds.decode(), "decode")
    st, seq = L.mla_get_device_error(ds.ws_decode, ds.stream)
    assert st == L.STATUS_CODE["MLA_ERR_BAD_PAGE"] and seq == 5
    assert torch.isnan(ds.out[5]).all() and torch.isnan(ds.lse[5]).all()
    keep = [b for b in range(24) if b != 5]
    assert torch.equal(ds.out[keep], clean_out[keep]) and torch.equal(ds.lse[keep], clean_lse[keep])


@gpu
def test_append_position_mismatch_and_cache_full():
    from mla_latent_cache_absorb_gb300 import binding as L
    torch, prob, ds = _setup(W["v2lite_b1_t4096"].with_(B=2, context=("fixed", 100)))
    before = ds.pool.clone()
    ds.len_before[0] = 99          # caller's length disagrees with the append position
    L.check(ds.append(), "append")
    st, seq = L.mla_get_device_error(ds.ws_append, ds.stream)
    assert st == L.STATUS_CODE["MLA_ERR_POS_MISMATCH"] and seq == 0
    # sequence 0's slot untouched, sequence 1 appended
    rows = prob.rows_per_seq
    assert torch.equal(ds.pool[100], before[100])
    assert not torch.equal(ds.pool[rows + 100], before[rows + 100])
    L.check(L.mla_clear_device_error(ds.ws_append, ds.stream), "clear")
    ds.len_before.copy_(ds.positions)
    ds.positions[1] = rows            # one past the capacity of a contiguous sequence
    ds.len_before[1] = rows
    L.check(ds.append(), "append")
    st, seq = L.mla_get_device_error(ds.ws_append, ds.stream)
    assert st == L.STATUS_CODE["MLA_ERR_CACHE_FULL"] and seq == 1


@gpu
def test_host_validation_enqueues_nothing():
    from mla_latent_cache_absorb_gb300 import binding as L
    torch, prob, ds = _setup(W["v2lite_b1_t4096"].with_(B=1, context=("fixed", 100)))
    ds.out.fill_(7.0)
    n = ds.ws_decode.numel()
    assert L.mla_decode_attn(ds.cfg, ds.q, ds.kv_b, ds.cache, ds.seq_lens, ds.positions, ds.out, ds.lse, 1,
                             ds.ws_decode, n - 1, ds.stream) == L.STATUS_CODE["MLA_ERR_WORKSPACE"]
    assert L.mla_decode_attn(ds.cfg, None, ds.kv_b, ds.cache, ds.seq_lens, ds.positions, ds.out, ds.lse, 1,
                             ds.ws_decode, n, ds.stream) == L.STATUS_CODE["MLA_ERR_INVALID_ARG"]
    torch.cuda.synchronize()
    assert torch.all(ds.out == 7.0)
